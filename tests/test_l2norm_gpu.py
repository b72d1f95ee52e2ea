"""GPU parity of the q/k L2-norm epilogue (kda_packed_conv1d_l2norm,
kda_conv1d_update_l2norm) against the oracle's conv + norm.

Bar: conv states bit-exact (the norm does not touch them); planes outside
the mask bit-exact against the plain oracle conv when there is no
activation, within one ulp with SiLU; normed planes within one ulp of x's
type for bf16 / fp16. For fp32 the bound is 2^-19 relative: the device sums
squares in FP32 over the head and takes rsqrtf (about 2^-22 each), on top of
the SiLU's 2^-21, against the oracle's float64 norm.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import pins
import workloads
from gpu_helpers import assert_states_equal, state_dtype_of, state_to_device, state_to_host
from gpu_helpers import ulp_diff

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


DT = {"bf16": 0, "f16": 1, "f32": 2}


def _eps32(eps: float) -> float:
    """The eps the kernel sees (kda_l2norm_t holds a float)."""
    return float(np.float32(eps))


def _device_inputs(b: workloads.Batch, dev):
    f32 = b.x_dtype == "f32"
    x = torch.from_numpy(b.x_buf if f32 else b.x_buf.view(np.int16)).to(dev)
    out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), float("nan") if f32 else -1,
                     dtype=torch.float32 if f32 else torch.int16, device=dev)
    st = state_to_device(b.conv_states, dev)
    w = torch.from_numpy(b.weight).to(dev)
    bias = None if b.bias is None else torch.from_numpy(b.bias).to(dev)
    return x, out, st, w, bias


def _run(b: workloads.Batch, mask: int, head_dim: int, eps: float, entry: str = "packed"):
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    x, out, st, w, bias = _device_inputs(b, dev)
    layout = pkg.make_layout(DT[b.x_dtype], st.size(2), st.stride(), w.stride(),
                             state_dtype_of(st))
    norm = pkg.make_l2norm(mask, head_dim, eps)
    esz = 4 if b.x_dtype == "f32" else 2
    xp = x.data_ptr() + esz * b.col_offset
    ci = torch.from_numpy(b.cache_indices).to(dev)
    if entry == "packed":
        his = torch.from_numpy(b.has_initial_state).to(dev)
        qsl = torch.from_numpy(b.query_start_loc).to(dev)
        pkg.kda_packed_conv1d_l2norm(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, st,
                                     ci, his, qsl, b.num_seqs, b.null_block_id, b.activation,
                                     out, layout, norm)
    else:
        pkg.kda_conv1d_update_l2norm(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, st,
                                     ci, b.null_block_id, b.activation, out, layout, norm)
    torch.cuda.synchronize()
    return out.cpu().numpy(), state_to_host(st)


def _compare(b: workloads.Batch, got: np.ndarray, want: np.ndarray, mask: int) -> None:
    for plane in range(b.dim // b.part_dim):
        normed = bool((mask >> plane) & 1)
        g, w = got[plane], want[plane]
        if b.x_dtype == "f32":
            unwritten = np.isnan(w)
            assert np.isnan(g[unwritten]).all(), "rows outside sequences written"
            g64, w64 = g[~unwritten].astype(np.float64), w[~unwritten].astype(np.float64)
            if not normed and b.activation == 0:
                assert np.array_equal(g[~unwritten].view(np.uint32), w[~unwritten].view(np.uint32))
                continue
            bound = 2.0 ** -19 if normed else 2.0 ** -20
            rel = np.abs(g64 - w64) / np.maximum(np.abs(w64), 1e-30)
            assert (rel <= bound).all(), (plane, float(rel.max()))
        else:
            gb = g.view(np.uint16)
            untouched = w == 0xFFFF
            assert np.array_equal(gb[untouched], w[untouched]), "rows outside sequences written"
            d = ulp_diff(gb, w)
            limit = 0 if (not normed and b.activation == 0) else 1
            assert d.max() <= limit, (plane, int(d.max()))


CASES = [
    # (name, seed, lengths, dim, part_dim, row_stride, col_offset, mask, head_dim, extra)
    ("bf16_h128", 1101, [1, 2, 3, 70, 150, 5], 768, 256, 776, 8, 0b011, 128, {}),
    ("f16_h64_none", 1102, [33, 1, 200, 4], 384, 128, 392, 8, 0b101, 64,
     {"x_dtype": "f16", "activation": 0}),
    ("f32_h32", 1103, [9, 64, 65, 2], 256, 128, 260, 4, 0b01, 32, {"x_dtype": "f32"}),
    ("bf16_h64_straddle", 1104, [3, 40, 7], 3264, 1088, 3272, 8, 0b001, 64, {}),
    ("bf16_state_short", 1105, [1] * 30 + [2, 3, 5, 9], 384, 128, 392, 8, 0b011, 128,
     {"state_dtype": "bf16"}),
    ("bf16_h16_nobias", 1106, [12, 1, 33], 192, 64, 200, 8, 0b110, 16, {"bias_std": None}),
    ("f16_k5_h128", 1107, [2, 6, 20], 512, 256, 520, 8, 0b11, 128,
     {"x_dtype": "f16", "state_width": 5}),
    # at most one token per sequence: the looping short kernel with the norm
    ("bf16_h128_one_token", 1108, [1] * 40 + [0] * 6 + [2] * 3, 768, 256, 776, 8, 0b011, 128,
     {}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_packed_l2norm_matches_oracle(case):
    name, seed, lengths, dim, part_dim, row_stride, col_offset, mask, head_dim, extra = case
    b = workloads.make_batch(name, seed, lengths, dim, part_dim, row_stride, len(lengths) + 3,
                             col_offset=col_offset, his_p=0.6, null_count=1, **extra)
    eps = _eps32(1e-6)
    st = b.conv_states.copy()
    want = pins.run_oracle_l2norm(b, mask, head_dim, eps, states=st)["out"]
    got, got_st = _run(b, mask, head_dim, eps)
    assert_states_equal(got_st, st)
    _compare(b, got, want, mask)


@pytest.mark.parametrize("case", CASES[:4] + CASES[5:6], ids=[c[0] for c in CASES[:4] + CASES[5:6]])
def test_update_l2norm_matches_oracle(case):
    name, seed, _, dim, part_dim, row_stride, col_offset, mask, head_dim, extra = case
    batch = 77
    b = workloads.make_batch(name + "_dec", seed + 50, [1] * batch, dim, part_dim, row_stride,
                             2 * batch, col_offset=col_offset, his_p=1.0, null_count=2, **extra)
    b.has_initial_state[:] = 1
    eps = _eps32(1e-6)
    st = b.conv_states.copy()
    want = pins.run_oracle_l2norm(b, mask, head_dim, eps, states=st)["out"]
    got, got_st = _run(b, mask, head_dim, eps, entry="update")
    assert_states_equal(got_st, st)
    _compare(b, got, want, mask)


def test_l2norm_large_eps_and_zero_heads():
    """A large eps (0.25) and heads whose conv output is exactly zero (zero
    taps and bias on those channels): zeros out, no NaN."""
    b = workloads.make_batch("l2eps", 1110, [5, 17, 40], 256, 128, 264, 6, col_offset=8,
                             his_p=0.5, null_count=1)
    b.weight[32:64] = 0.0
    b.bias[32:64] = 0.0
    st = b.conv_states.copy()
    want = pins.run_oracle_l2norm(b, 0b11, 32, 0.25, states=st)["out"]
    got, got_st = _run(b, 0b11, 32, 0.25)
    assert_states_equal(got_st, st)
    _compare(b, got, want, 0b11)
    assert (got[0][:, 32:64].view(np.uint16) == 0).all()


def test_l2norm_tiny_heads_stay_finite():
    """Heads of tiny activations (taps and bias scaled by 2^-70, so that the
    head's sum of squares is far below FLT_MIN) with eps = 1e-6: the root of
    (sum + eps) is a normal number, the outputs are finite and match the
    float64 norm of the oracle."""
    b = workloads.make_batch("l2tiny", 1112, [5, 17, 40], 256, 128, 264, 6, col_offset=8,
                             his_p=0.5, null_count=1)
    b.weight[:64] *= np.float32(2.0 ** -70)
    b.bias[:64] *= np.float32(2.0 ** -70)
    b.conv_states[:, :64] = 0.0
    eps = _eps32(1e-6)
    st = b.conv_states.copy()
    want = pins.run_oracle_l2norm(b, 0b11, 32, eps, states=st)["out"]
    got, got_st = _run(b, 0b11, 32, eps)
    assert_states_equal(got_st, st)
    _compare(b, got, want, 0b11)
    g = got[0][:, :64].view(np.uint16)
    assert not (((g & 0x7F80) == 0x7F80) & (g != 0xFFFF)).any()  # no inf / NaN written


@pytest.mark.parametrize("name", ["long16k", "decode"])
def test_l2norm_full_size(name):
    """The 16K prefill chunk and the 1024-sequence decode step with q and k
    normalised per 128-channel head."""
    b = workloads.WORKLOADS[name]()
    eps = _eps32(1e-6)
    st = b.conv_states.copy()
    want = pins.run_oracle_l2norm(b, 0b011, 128, eps, states=st)["out"]
    got, got_st = _run(b, 0b011, 128, eps, entry="update" if name == "decode" else "packed")
    assert_states_equal(got_st, st)
    _compare(b, got, want, 0b011)


def test_empty_mask_is_the_plain_conv():
    import linear_attention_prefill_varlen_gb300 as pkg

    b = workloads.make_batch("l2none", 1111, [4, 30, 1], 384, 128, 392, 6, col_offset=8)
    st = b.conv_states.copy()
    want = pins.run_oracle_ex(b, states=st)["out"]
    got, got_st = _run(b, 0, 128, 1e-6)
    assert_states_equal(got_st, st)
    _compare(b, got, want, 0)
    assert pkg.make_l2norm(0).plane_mask == 0


def test_wrappers_with_qk_l2norm():
    """packed_causal_conv1d_fn then causal_conv1d_update with use_qk_l2norm on
    one conv-state tensor."""
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    dim, part, lines = 768, 256, 10
    pre = workloads.make_batch("l2flow", 1120, [40, 3, 1, 77], dim, part, 776, lines,
                               col_offset=8, his_p=0.5, null_count=1)
    st = torch.from_numpy(pre.conv_states).to(dev)
    w = torch.from_numpy(pre.weight).to(dev)
    bias = torch.from_numpy(pre.bias).to(dev)
    x = torch.from_numpy(pre.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
    xs = x[:, pre.col_offset:pre.col_offset + dim]
    meta = [torch.from_numpy(a).to(dev) for a in
            (pre.query_start_loc, pre.cache_indices, pre.has_initial_state)]
    out = pkg.packed_causal_conv1d_fn(xs, w, bias, st, meta[0], meta[1], meta[2].bool(), part,
                                      activation="silu", null_block_id=pre.null_block_id,
                                      use_qk_l2norm=True, head_dim=128, l2norm_eps=1e-6)
    ref_st = pre.conv_states.copy()
    want = pins.run_oracle_l2norm(pre, 0b011, 128, _eps32(1e-6), states=ref_st)["out"]
    torch.cuda.synchronize()
    assert_states_equal(st.cpu().numpy(), ref_st)
    _compare(pre, out.view(torch.int16).cpu().numpy(), want, 0b011)
    d = workloads.make_batch("l2flow_dec", 1121, [1] * 4, dim, part, 776, lines, col_offset=8)
    d.weight, d.bias, d.cache_indices = pre.weight, pre.bias, pre.cache_indices.copy()
    d.has_initial_state[:] = 1
    xd = torch.from_numpy(d.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
    ci = torch.from_numpy(d.cache_indices).to(dev)
    o = pkg.causal_conv1d_update(xd[:, d.col_offset:d.col_offset + dim], st, w, bias, ci, part,
                                 activation="silu", null_block_id=d.null_block_id,
                                 use_qk_l2norm=True, head_dim=128, l2norm_eps=1e-6)
    want = pins.run_oracle_l2norm(d, 0b011, 128, _eps32(1e-6), states=ref_st)["out"]
    torch.cuda.synchronize()
    assert_states_equal(st.cpu().numpy(), ref_st)
    _compare(d, o.view(torch.int16).cpu().numpy(), want, 0b011)
