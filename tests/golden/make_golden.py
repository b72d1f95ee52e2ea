"""Writes oracle_regression.json: digests of the oracle's results on small
seeded batches, so that any later change to the oracle's arithmetic shows up
as a failing CPU test (tests/test_golden.py) and has to be regenerated on
purpose.

The pages print no worked numerical example of the conv (only timings), so
no fixture here comes from them. Every value is written by this script, which
calls only the oracle package and the seeded input generators:

    python tests/golden/make_golden.py
"""

from __future__ import annotations

import hashlib
import json
import os
import platform
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402

DT = {"bf16": oracle.DTYPE_BF16, "f16": oracle.DTYPE_F16, "f32": oracle.DTYPE_F32}


def cases():
    """(name, batch, norm) -- norm None or (plane mask, head_dim, eps)."""
    yield "tiny", workloads.tiny(), None
    yield "varlen_small", workloads.make_batch("g_varlen", 7001, [1, 2, 3, 17, 40, 0, 5], 256, 128,
                                               264, 10, col_offset=8, his_p=0.5,
                                               null_count=1), None
    yield "f16_k5", workloads.make_batch("g_f16", 7002, [9, 1, 30], 192, 64, 200, 5,
                                         col_offset=8, x_dtype="f16", state_width=5), None
    yield "f32_nobias_none", workloads.make_batch("g_f32", 7003, [4, 12], 128, 64, 132, 4,
                                                  col_offset=4, x_dtype="f32", bias_std=None,
                                                  activation=0), None
    yield "bf16_state", workloads.make_batch("g_bst", 7004, [2, 7, 33], 256, 128, 264, 5,
                                             col_offset=8, state_dtype="bf16"), None
    yield "l2norm_h64", workloads.make_batch("g_l2", 7005, [3, 21, 1], 384, 128, 392, 5,
                                             col_offset=8), (0b011, 64, float(np.float32(1e-6)))


def run(b, norm):
    st = b.conv_states.copy()
    if norm is None:
        out = oracle.packed_conv1d_ex(b.x_buf, DT[b.x_dtype], b.col_offset, b.dim, b.part_dim,
                                      b.weight, b.bias, st, b.cache_indices,
                                      b.has_initial_state, b.query_start_loc, b.null_block_id,
                                      b.activation)["out"]
    else:
        out = oracle.packed_conv1d_l2norm(b.x_buf, DT[b.x_dtype], b.col_offset, b.dim,
                                          b.part_dim, b.weight, b.bias, st, b.cache_indices,
                                          b.has_initial_state, b.query_start_loc,
                                          b.null_block_id, b.activation, *norm)["out"]
    return out, st


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def record():
    res = {}
    for name, b, norm in cases():
        out, st = run(b, norm)
        flat = out.reshape(-1)
        res[name] = {"out_sha256": digest(out), "state_sha256": digest(st),
                     "out_shape": list(out.shape), "out_dtype": str(out.dtype),
                     "out_first8": [int(v) if out.dtype == np.uint16 else float(v)
                                    for v in flat[:8]]}
    return res


if __name__ == "__main__":
    path = os.path.join(HERE, "oracle_regression.json")
    with open(path, "w") as f:
        # expf (in the SiLU) comes from the host C library, whose last bit may
        # differ between architectures: the digests hold for this machine type
        json.dump({"written_by": "tests/golden/make_golden.py (oracle only)",
                   "machine": platform.machine(), "cases": record()}, f, indent=1)
    print("wrote", path)
