"""The device epilogue over every fp32 bit pattern.

The epilogue (activation, then round to bf16 nearest-even) is a pure
function of one fp32 value, so it can be checked exhaustively: the library's
kda_epilogue_range runs the same device code as the conv kernel on all 2^32
patterns and the oracle computes bf16_rne(silu(f)) / bf16_rne(f) on the
host.  Bar: plain rounding bit-exact; SiLU within 1 bf16 ulp; NaN where the
oracle has NaN.
"""

from __future__ import annotations

import os
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import is_nan_bf16, ulp_diff

pytestmark = pytest.mark.gpu

SLAB = 1 << 28
PIECE = 1 << 24


def _host_piece(first: int, got: np.ndarray, activation: int) -> tuple[int, int, list]:
    n = got.size
    if activation == 1:
        want = oracle.silu_bf16_range(first, n)
    else:
        vals = np.arange(first, first + n, dtype=np.uint64).astype(np.uint32).view(np.float32)
        want = oracle.bf16_rne(vals)
    nan_w = is_nan_bf16(want)
    nan_g = is_nan_bf16(got)
    bad_nan = int(np.count_nonzero(nan_w != nan_g))
    d = ulp_diff(got, want)
    limit = 0 if activation == 0 else 1
    over = np.flatnonzero(d > limit)
    examples = [(first + int(i), int(want[i]), int(got[i])) for i in over[:4]]
    return bad_nan, int(over.size), examples


@pytest.mark.parametrize("activation", [0, 1], ids=["round", "silu"])
def test_epilogue_all_fp32_patterns(activation):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    oracle.load()
    t = time.time()
    dev = torch.empty(SLAB, dtype=torch.int16, device="cuda")
    host = torch.empty(SLAB, dtype=torch.int16, pin_memory=True)
    workers = max(1, min(32, os.cpu_count() or 1))
    bad_nan = over = 0
    examples = []
    with ThreadPoolExecutor(max_workers=workers) as pool:
        for slab in range(0, 1 << 32, SLAB):
            pkg.epilogue_range(slab, SLAB, activation, dev)
            host.copy_(dev)
            torch.cuda.synchronize()
            got = host.numpy().view(np.uint16).copy()
            jobs = [pool.submit(_host_piece, slab + o, got[o:o + PIECE], activation)
                    for o in range(0, SLAB, PIECE)]
            for j in jobs:
                bn, ov, ex = j.result()
                bad_nan += bn
                over += ov
                examples.extend(ex[: max(0, 8 - len(examples))])
    print(f"epilogue activation={activation}: {time.time() - t:.1f}s, "
          f"NaN-class mismatches {bad_nan}, beyond tolerance {over}, examples {examples}")
    assert bad_nan == 0, examples
    assert over == 0, [(hex(a), hex(w), hex(g)) for a, w, g in examples]
