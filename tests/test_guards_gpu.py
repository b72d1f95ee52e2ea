"""Guard regions: every entry point writes only inside its outputs.

The output planes and the conv-state array are placed inside larger device
buffers whose margins (4 KB before, 4 KB after) hold a sentinel; after the
call the margins must be unchanged, for each entry point and x dtype."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

MARGIN = 4096  # bytes on each side


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


def _guarded(nbytes: int, dev) -> tuple[torch.Tensor, int]:
    buf = torch.full((MARGIN + nbytes + MARGIN,), 0xA5, dtype=torch.uint8, device=dev)
    return buf, buf.data_ptr() + MARGIN


def _margins_intact(buf: torch.Tensor, nbytes: int) -> bool:
    head = buf[:MARGIN]
    tail = buf[MARGIN + nbytes:]
    return bool(head.eq(0xA5).all().item() and tail.eq(0xA5).all().item())


@pytest.mark.parametrize("entry,x_dtype,width,state_dtype", [
    ("packed", "bf16", 3, "f32"), ("ex", "f16", 3, "f32"), ("ex", "f32", 5, "f32"),
    ("update", "bf16", 3, "f32"), ("update", "f32", 4, "f32"),
    ("ex", "bf16", 3, "bf16"), ("ex", "f16", 6, "bf16"), ("update", "bf16", 3, "bf16"),
    ("update", "f32", 5, "bf16"),
])
def test_writes_stay_inside_out_and_states(entry, x_dtype, width, state_dtype):
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    lengths = [1] * 40 if entry == "update" else [1, 2, 3, 70, 200, 5]
    b = workloads.make_batch(f"guard_{entry}", 901, lengths, 256, 128, 264, len(lengths) + 2,
                             col_offset=8, his_p=0.6, null_count=2, x_dtype=x_dtype,
                             state_width=width, state_dtype=state_dtype)
    if entry == "update":
        b.has_initial_state[:] = 1
    esz = 4 if x_dtype == "f32" else 2
    x = torch.from_numpy(b.x_buf if x_dtype == "f32" else b.x_buf.view(np.int16)).to(dev)
    out_bytes = (b.dim // b.part_dim) * b.tokens * b.part_dim * esz
    st_bytes = b.conv_states.nbytes
    obuf, optr = _guarded(out_bytes, dev)
    sbuf, sptr = _guarded(st_bytes, dev)
    sbuf[MARGIN:MARGIN + st_bytes].copy_(torch.from_numpy(b.conv_states.view(np.uint8).ravel()))
    w = torch.from_numpy(b.weight).to(dev)
    bias = torch.from_numpy(b.bias).to(dev)
    ci, his, qsl = (torch.from_numpy(a).to(dev) for a in
                    (b.cache_indices, b.has_initial_state, b.query_start_loc))
    dt = {"bf16": pkg.KDA_DTYPE_BF16, "f16": pkg.KDA_DTYPE_F16, "f32": pkg.KDA_DTYPE_F32}
    layout = pkg.make_layout(dt[x_dtype], width, (width * b.dim, width, 1), (4, 1),
                             dt[state_dtype])
    xp = x.data_ptr() + esz * b.col_offset
    if entry == "packed":
        pkg.kda_packed_conv1d(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, sptr, ci,
                              his, qsl, b.num_seqs, b.null_block_id, b.activation, optr)
    elif entry == "ex":
        pkg.kda_packed_conv1d_ex(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, sptr,
                                 ci, his, qsl, b.num_seqs, b.null_block_id, b.activation, optr,
                                 layout)
    else:
        pkg.kda_conv1d_update(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, sptr, ci,
                              b.null_block_id, b.activation, optr, layout)
    torch.cuda.synchronize()
    assert _margins_intact(obuf, out_bytes), "write outside the output planes"
    assert _margins_intact(sbuf, st_bytes), "write outside the conv-state array"
    # the null-block lines and unreferenced lines are untouched inside the array
    got = sbuf[MARGIN:MARGIN + st_bytes].cpu().numpy().view(b.conv_states.dtype).reshape(
        b.conv_states.shape)
    live = {int(c) for c in b.cache_indices if c != b.null_block_id}
    for line in range(b.conv_states.shape[0]):
        if line not in live:
            assert got[line].tobytes() == b.conv_states[line].tobytes()
