"""GPU parity of kda_packed_conv1d_ex (fp16 / fp32 x, conv state width K >= 3,
strided state and weight) against the general-layout oracle.

Bar: conv states bit-exact; outputs without activation bit-exact for every
dtype (they are the FP32 accumulator rounded to x's type, or the accumulator
itself for fp32); SiLU outputs within one ulp of x's type for bf16 / fp16
(the device SiLU is within about 2^-21 relative of a / (1 + expf(-a)), far
inside half an ulp of either 16-bit type) and within 2^-20 relative for fp32.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import pins
import workloads
from gpu_helpers import (assert_states_equal, state_dtype_of, state_to_device, state_to_host,
                         ulp_diff)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


def weight_to_device(b: workloads.Batch, form, dev):
    """The weight as a device tensor and its (channel, tap) strides and part
    stride.  form False / "channel_major": (dim, 4) contiguous; True /
    "tap_major": (4, dim) memory viewed as (dim, 4); "decode3": the kda_decode
    page's [qkv, width, channel] buffer, (dim / part_dim, 4, part_dim)."""
    if form == "decode3":
        parts = b.dim // b.part_dim
        w3 = np.ascontiguousarray(b.weight.reshape(parts, b.part_dim, 4).transpose(0, 2, 1))
        w = torch.from_numpy(w3).to(dev)
        return w, (w.stride(2), w.stride(1)), w.stride(0)
    if form is True or form == "tap_major":
        w = torch.from_numpy(np.ascontiguousarray(b.weight.T)).to(dev).t()
    else:
        w = torch.from_numpy(b.weight).to(dev)
    return w, w.stride(), 0


def strided_indices(ci: np.ndarray, stride: int, dev) -> torch.Tensor:
    """cache_indices as a view with `stride` elements between entries; the
    entries in between hold line 0, so reading one of them is caught."""
    if stride <= 1:
        return torch.from_numpy(ci).to(dev)
    buf = torch.zeros(max(len(ci) * stride, 1), dtype=torch.int32, device=dev)
    view = buf[::stride][:len(ci)]
    view.copy_(torch.from_numpy(ci))
    return view


def _run_device(b: workloads.Batch, state_mem_order: str = "dense", weight_tap_major=False,
                ci_stride: int = 1):
    """Runs kda_packed_conv1d_ex on b.  state_mem_order 'dense' keeps
    conv_states (lines, dim, K) contiguous; 'position_major' stores it as
    (lines, K, dim) memory viewed as (lines, dim, K).  weight_tap_major is a
    weight_to_device form; ci_stride > 1 passes cache_indices strided."""
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    if b.x_dtype == "f32":
        x = torch.from_numpy(b.x_buf).to(dev)
        out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), float("nan"),
                         dtype=torch.float32, device=dev)
    else:
        x = torch.from_numpy(b.x_buf.view(np.int16)).to(dev)
        out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), -1, dtype=torch.int16,
                         device=dev)
    if state_mem_order == "dense":
        st = state_to_device(b.conv_states, dev)
    else:
        st = state_to_device(np.ascontiguousarray(b.conv_states.transpose(0, 2, 1)), dev)
        st = st.transpose(1, 2)
    w, w_strides, w_part = weight_to_device(b, weight_tap_major, dev)
    bias = None if b.bias is None else torch.from_numpy(b.bias).to(dev)
    meta = [strided_indices(b.cache_indices, ci_stride, dev)] + [
        torch.from_numpy(a).to(dev) for a in (b.has_initial_state, b.query_start_loc)]
    dt = {"bf16": pkg.KDA_DTYPE_BF16, "f16": pkg.KDA_DTYPE_F16, "f32": pkg.KDA_DTYPE_F32}
    layout = pkg.make_layout(dt[b.x_dtype], st.size(2), st.stride(), w_strides,
                             state_dtype_of(st), w_part, ci_stride if ci_stride > 1 else 0)
    esz = 4 if b.x_dtype == "f32" else 2
    pkg.kda_packed_conv1d_ex(x.data_ptr() + esz * b.col_offset, b.row_stride, b.tokens, b.dim,
                             b.part_dim, w, bias, st, meta[0], meta[1], meta[2], b.num_seqs,
                             b.null_block_id, b.activation, out, layout)
    torch.cuda.synchronize()
    return out.cpu().numpy(), state_to_host(st)


def _ordered32(v: np.ndarray) -> np.ndarray:
    b = v.view(np.uint32).astype(np.int64)
    return np.where(b & 0x80000000, 0x80000000 - (b & 0x7FFFFFFF), 0x80000000 + (b & 0x7FFFFFFF))


def _compare(b: workloads.Batch, got: np.ndarray, want: np.ndarray) -> None:
    if b.x_dtype == "f32":
        unwritten = np.isnan(want)
        assert np.isnan(got[unwritten]).all(), "rows outside sequences written"
        g, w = got[~unwritten], want[~unwritten]
        if b.activation == 0:
            assert np.array_equal(g.view(np.uint32), w.view(np.uint32))
        else:
            rel = np.abs(g.astype(np.float64) - w) / np.maximum(np.abs(w.astype(np.float64)), 1e-30)
            assert (rel <= 2.0 ** -20).all(), float(rel.max())
    else:
        gb = got.view(np.uint16)
        untouched = want == 0xFFFF
        assert np.array_equal(gb[untouched], want[untouched]), "rows outside sequences written"
        d = ulp_diff(gb, want)
        assert d.max() <= (0 if b.activation == 0 else 1), int(d.max())


CASES = [
    # (name, seed, lengths, dim, part_dim, row_stride, col_offset, extra)
    ("f16_silu", 401, [1, 2, 3, 70, 150, 5], 256, 128, 264, 8, {"x_dtype": "f16"}),
    ("f16_none", 402, [33, 1, 200], 192, 64, 192, 0,
     {"x_dtype": "f16", "activation": 0, "bias_std": None}),
    ("f32_silu", 403, [9, 64, 65, 2], 128, 64, 132, 4, {"x_dtype": "f32"}),
    ("f32_none", 404, [300, 1], 256, 256, 256, 0, {"x_dtype": "f32", "activation": 0}),
    ("bf16_k4", 405, [1, 2, 5, 90], 128, 64, 136, 8, {"state_width": 4}),
    ("f16_k8", 406, [3, 7, 12, 40], 128, 128, 128, 0, {"x_dtype": "f16", "state_width": 8}),
    ("f32_k5_none", 407, [6, 1, 33], 64, 64, 68, 4,
     {"x_dtype": "f32", "state_width": 5, "activation": 0}),
    ("bf16_state", 408, [1, 2, 3, 70, 150, 5], 256, 128, 264, 8, {"state_dtype": "bf16"}),
    ("bf16_state_f16_none", 409, [33, 1, 2, 200], 192, 64, 192, 0,
     {"x_dtype": "f16", "state_dtype": "bf16", "activation": 0}),
    ("bf16_state_f32", 412, [9, 64, 65, 2], 128, 64, 132, 4,
     {"x_dtype": "f32", "state_dtype": "bf16"}),
    ("bf16_state_k6", 413, [1, 4, 7, 40], 128, 128, 128, 0,
     {"state_dtype": "bf16", "state_width": 6}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("mem", ["dense", "position_major"])
@pytest.mark.parametrize("tap_major", [False, True, "decode3"],
                         ids=["w_channel_major", "w_tap_major", "w_qkv_width_channel"])
def test_general_layout(case, mem, tap_major):
    name, seed, lengths, dim, part_dim, row_stride, col_offset, extra = case
    extra = dict(extra)
    b = workloads.make_batch(name, seed, lengths, dim, part_dim, row_stride, len(lengths) + 4,
                             col_offset=col_offset, his_p=0.6, null_count=1, **extra)
    st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=st)
    got, got_states = _run_device(b, mem, tap_major)
    assert_states_equal(got_states, st)
    _compare(b, got, ref["out"])


def test_general_layout_large_f16():
    """A full-width fp16 prefill batch (4 x 2048 tokens, 3 x 1536 channels)."""
    b = workloads.make_batch("f16_large", 410, [2048, 1, 2047, 4096], 4608, 1536, 6400, 64,
                             his_p=0.5, null_count=1, x_dtype="f16")
    st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=st)
    got, got_states = _run_device(b)
    assert_states_equal(got_states, st)
    _compare(b, got, ref["out"])


def test_page_style_wrapper_with_fp16_and_wide_state():
    """packed_causal_conv1d_fn with fp16 x, a (lines, dim, 4) state viewed from
    position-major memory and a tap-major weight view."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = workloads.make_batch("wrap", 411, [17, 3, 40], 384, 128, 384, 6, his_p=0.7,
                             x_dtype="f16", state_width=4)
    dev = torch.device("cuda")
    x = torch.from_numpy(b.x_buf.view(np.int16)).to(dev).view(torch.float16)
    st = state_to_device(np.ascontiguousarray(b.conv_states.transpose(0, 2, 1)), dev)
    st = st.transpose(1, 2)
    w = torch.from_numpy(np.ascontiguousarray(b.weight.T)).to(dev).t()
    assert pkg.packed_causal_conv1d_supported(x, w, st, b.part_dim)
    meta = [torch.from_numpy(a).to(dev) for a in
            (b.query_start_loc, b.cache_indices, b.has_initial_state)]
    out = pkg.packed_causal_conv1d_fn(x, w, torch.from_numpy(b.bias).to(dev), st, meta[0],
                                      meta[1], meta[2].bool(), b.part_dim, activation="silu",
                                      null_block_id=-1)
    torch.cuda.synchronize()
    ref_st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=ref_st)
    assert out.dtype == torch.float16
    assert np.array_equal(state_to_host(st).view(np.uint32), ref_st.view(np.uint32))
    _compare(b, out.view(torch.int16).cpu().numpy(), ref["out"])


@pytest.mark.parametrize("ci_stride", [2, 3, 7])
@pytest.mark.parametrize("weight", ["channel_major", "decode3"])
def test_strided_cache_indices(ci_stride, weight):
    """cache_indices passed as a strided view (the page's launch passes
    cache_indices.stride(0)): sequence s uses entry s * stride, and the
    entries in between (line 0) are never read."""
    b = workloads.make_batch(f"ci_stride{ci_stride}", 420 + ci_stride, [1, 5, 40, 2, 130, 3],
                             256, 128, 264, 12, col_offset=8, his_p=0.7, null_count=1)
    st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=st)
    got, got_states = _run_device(b, "dense", weight, ci_stride)
    assert_states_equal(got_states, st)
    _compare(b, got, ref["out"])


def test_page_wrapper_with_the_decode_weight_and_strided_indices():
    """packed_causal_conv1d_fn given the kda_decode page's (3, 4, part_dim)
    weight and a strided cache_indices view derives the layout from them."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = workloads.make_batch("wrap3", 431, [17, 3, 40, 1], 384, 128, 384, 9, his_p=0.7,
                             null_count=1)
    dev = torch.device("cuda")
    x = torch.from_numpy(b.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
    st = state_to_device(b.conv_states, dev)
    w, _, _ = weight_to_device(b, "decode3", dev)
    ci = strided_indices(b.cache_indices, 4, dev)
    assert pkg.packed_causal_conv1d_supported(x, w, st, b.part_dim)
    meta = [torch.from_numpy(a).to(dev) for a in (b.query_start_loc, b.has_initial_state)]
    out = pkg.packed_causal_conv1d_fn(x, w, torch.from_numpy(b.bias).to(dev), st, meta[0], ci,
                                      meta[1].bool(), b.part_dim, activation="silu",
                                      null_block_id=-1)
    torch.cuda.synchronize()
    ref_st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=ref_st)
    assert np.array_equal(state_to_host(st).view(np.uint32), ref_st.view(np.uint32))
    _compare(b, out.view(torch.int16).cpu().numpy(), ref["out"])
