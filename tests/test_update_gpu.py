"""GPU parity of kda_conv1d_update (one token per sequence) against the oracle
run with query_start_loc = 0..batch and every has_initial_state set.

Bar as for the packed path: conv states and activation-free outputs
bit-exact, SiLU outputs within one ulp of the 16-bit types (2^-20 relative
for fp32)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import pins
import workloads
from gpu_helpers import (assert_states_equal, state_dtype_of, state_to_device, state_to_host,
                         ulp_diff)
from test_general_layout_gpu import _compare, strided_indices, weight_to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


def _decode_batch(seed, batch, dim, part_dim, row_stride, lines, **kw):
    b = workloads.make_batch(f"dec{seed}", seed, [1] * batch, dim, part_dim, row_stride, lines,
                             his_p=1.0, **kw)
    b.has_initial_state[:] = 1  # the update continues every live sequence
    return b


def _run_update(b, position_major=False, tap_major=False, ci_stride=1):
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    f32 = b.x_dtype == "f32"
    x = torch.from_numpy(b.x_buf if f32 else b.x_buf.view(np.int16)).to(dev)
    out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), float("nan") if f32 else -1,
                     dtype=torch.float32 if f32 else torch.int16, device=dev)
    if position_major:
        st = state_to_device(np.ascontiguousarray(b.conv_states.transpose(0, 2, 1)), dev)
        st = st.transpose(1, 2)
    else:
        st = state_to_device(b.conv_states, dev)
    w, w_strides, w_part = weight_to_device(b, tap_major, dev)
    bias = None if b.bias is None else torch.from_numpy(b.bias).to(dev)
    ci = strided_indices(b.cache_indices, ci_stride, dev)
    dt = {"bf16": pkg.KDA_DTYPE_BF16, "f16": pkg.KDA_DTYPE_F16, "f32": pkg.KDA_DTYPE_F32}
    layout = pkg.make_layout(dt[b.x_dtype], st.size(2), st.stride(), w_strides,
                             state_dtype_of(st), w_part, ci_stride if ci_stride > 1 else 0)
    esz = 4 if f32 else 2
    pkg.kda_conv1d_update(x.data_ptr() + esz * b.col_offset, b.row_stride, b.tokens, b.dim,
                          b.part_dim, w, bias, st, ci, b.null_block_id, b.activation, out, layout)
    torch.cuda.synchronize()
    return out.cpu().numpy(), state_to_host(st)


CASES = [
    ("bf16_silu", 501, 300, 256, 128, 264, 8, {}),
    ("bf16_none", 502, 77, 128, 64, 128, 0, {"activation": 0, "bias_std": None}),
    ("f16_silu", 503, 129, 192, 64, 200, 8, {"x_dtype": "f16"}),
    ("f32_none", 504, 64, 128, 128, 132, 4, {"x_dtype": "f32", "activation": 0}),
    ("bf16_k4", 505, 90, 128, 64, 128, 0, {"state_width": 4}),
    ("f16_k6_silu", 506, 33, 256, 256, 256, 0, {"x_dtype": "f16", "state_width": 6}),
    ("bf16_state_bf16", 507, 300, 256, 128, 264, 8, {"state_dtype": "bf16"}),
    ("bf16_state_f16_none", 508, 96, 192, 64, 200, 8,
     {"x_dtype": "f16", "state_dtype": "bf16", "activation": 0}),
    ("bf16_state_f32", 509, 64, 128, 128, 132, 4, {"x_dtype": "f32", "state_dtype": "bf16"}),
    ("bf16_state_k5", 510, 50, 128, 64, 128, 0, {"state_dtype": "bf16", "state_width": 5}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("position_major", [False, True], ids=["dense", "position_major"])
@pytest.mark.parametrize("tap_major", [False, True, "decode3"],
                         ids=["w_channel_major", "w_tap_major", "w_qkv_width_channel"])
def test_update_matches_oracle(case, position_major, tap_major):
    name, seed, batch, dim, part_dim, row_stride, col_offset, extra = case
    b = _decode_batch(seed, batch, dim, part_dim, row_stride, 2 * batch, col_offset=col_offset,
                      null_count=3, **extra)
    st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=st)
    got, got_st = _run_update(b, position_major, tap_major)
    assert_states_equal(got_st, st)
    _compare(b, got, ref["out"])


@pytest.mark.parametrize("name", ["decode", "decode_bf16_state"])
def test_update_decode_workload_and_repeated_steps(name):
    """The 1024-sequence decode batch (fp32 or bf16 state), three steps in a
    row: each step's state feeds the next, as in generation."""
    b = workloads.WORKLOADS[name]()
    b.cache_indices[::97] = b.null_block_id
    dev_states = None
    st = b.conv_states.copy()
    for step in range(3):
        c = b.copy()
        c.x_buf = np.roll(b.x_buf, step, axis=1).copy()  # a different token row per step
        c.conv_states = st.copy() if dev_states is None else dev_states
        ref = pins.run_oracle_ex(c, states=st)
        got, dev_states = _run_update(c)
        assert_states_equal(dev_states, st)
        _compare(c, got, ref["out"])


def test_back_to_back_chain_on_one_state_buffer():
    """Calls that read the conv state the previous call wrote, issued back to
    back on one stream with nothing in between (all inputs uploaded and all
    outputs allocated first), so consecutive launches are adjacent and overlap
    their scheduling while each waits for its predecessor: a packed prefill,
    12 decode updates, another packed call; against the oracle in the same
    order."""
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    lines, dim, part = 40, 256, 128
    pre = workloads.make_batch("chain_pre", 601, [37, 5, 90, 1], dim, part, 264, lines,
                               col_offset=8, his_p=0.5)
    calls = [("packed", pre)]
    for step in range(12):
        d = workloads.make_batch(f"chain_dec{step}", 610 + step, [1] * 4, dim, part, 264, lines,
                                 col_offset=8)
        calls.append(("update", d))
    calls.append(("packed", workloads.make_batch("chain_post", 630, [3, 20, 2, 9], dim, part,
                                                 264, lines, col_offset=8)))
    for _, b in calls[1:]:
        b.weight, b.bias = pre.weight, pre.bias
        b.cache_indices = pre.cache_indices.copy()
        b.has_initial_state[:] = 1

    dev_st = torch.from_numpy(pre.conv_states).to(dev)
    w = torch.from_numpy(pre.weight).to(dev)
    bias = torch.from_numpy(pre.bias).to(dev)
    staged = []
    for kind, b in calls:
        staged.append(dict(
            x=torch.from_numpy(b.x_buf.view(np.int16)).to(dev),
            out=torch.full((dim // part, b.tokens, part), -1, dtype=torch.int16, device=dev),
            meta=[torch.from_numpy(a).to(dev) for a in
                  (b.cache_indices, b.has_initial_state, b.query_start_loc)]))
    torch.cuda.synchronize()
    for (kind, b), sd in zip(calls, staged):  # back to back
        xp = sd["x"].data_ptr() + 2 * b.col_offset
        ci, his, qsl = sd["meta"]
        if kind == "packed":
            pkg.kda_packed_conv1d(xp, b.row_stride, b.tokens, dim, part, w, bias, dev_st, ci,
                                  his, qsl, b.num_seqs, b.null_block_id, b.activation, sd["out"])
        else:
            pkg.kda_conv1d_update(xp, b.row_stride, b.tokens, dim, part, w, bias, dev_st, ci,
                                  b.null_block_id, b.activation, sd["out"])
    torch.cuda.synchronize()

    st_ref = pre.conv_states.copy()
    for (kind, b), sd in zip(calls, staged):
        want = pins.run_oracle_ex(b, states=st_ref)["out"]
        d = ulp_diff(sd["out"].cpu().numpy().view(np.uint16), want)
        assert d.max() <= 1, kind
    assert np.array_equal(dev_st.cpu().numpy().view(np.uint32), st_ref.view(np.uint32))


def test_update_in_cuda_graph_replays_with_new_metadata():
    """A captured decode update replays correctly after the x rows and cache
    indices change (same batch size)."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b1 = _decode_batch(801, 64, 256, 128, 256, 200, null_count=2)
    b2 = b1.copy()
    b2.x_buf = np.roll(b1.x_buf, 3, axis=0).copy()
    b2.cache_indices = np.random.default_rng(3).permutation(200)[:64].astype(np.int32)
    dev = torch.device("cuda")
    x = torch.from_numpy(b1.x_buf.view(np.int16)).to(dev)
    st = torch.from_numpy(b1.conv_states).to(dev)
    w = torch.from_numpy(b1.weight).to(dev)
    bias = torch.from_numpy(b1.bias).to(dev)
    ci = torch.from_numpy(b1.cache_indices).to(dev)
    out = torch.full((2, 64, 128), -1, dtype=torch.int16, device=dev)
    stream = torch.cuda.Stream()

    def step(s):
        pkg.kda_conv1d_update(x, b1.row_stride, 64, 256, 128, w, bias, st, ci, b1.null_block_id,
                              b1.activation, out, None, s)

    step(stream)  # outside capture: first-use set-up
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step(torch.cuda.current_stream())
    for b in (b1, b2):
        x.copy_(torch.from_numpy(b.x_buf.view(np.int16)))
        st.copy_(torch.from_numpy(b.conv_states))
        ci.copy_(torch.from_numpy(b.cache_indices))
        out.fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref_st = b.conv_states.copy()
        ref = pins.run_oracle_ex(b, states=ref_st)
        assert np.array_equal(st.cpu().numpy().view(np.uint32), ref_st.view(np.uint32))
        _compare(b, out.cpu().numpy(), ref["out"])


def test_wrappers_prefill_then_decode_on_a_bf16_state():
    """packed_causal_conv1d_fn then two causal_conv1d_update steps on one bf16
    conv-state tensor, as a serving loop runs them, against the oracle."""
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    dim, part, lines = 384, 128, 12
    pre = workloads.make_batch("bf16_flow_pre", 701, [40, 3, 1, 77], dim, part, 392, lines,
                               col_offset=8, his_p=0.5, null_count=1, state_dtype="bf16")
    st = state_to_device(pre.conv_states, dev)
    w = torch.from_numpy(pre.weight).to(dev)
    bias = torch.from_numpy(pre.bias).to(dev)
    x = torch.from_numpy(pre.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
    xs = x[:, pre.col_offset:pre.col_offset + dim]
    meta = [torch.from_numpy(a).to(dev) for a in
            (pre.query_start_loc, pre.cache_indices, pre.has_initial_state)]
    assert pkg.packed_causal_conv1d_supported(xs, w, st, part)
    out = pkg.packed_causal_conv1d_fn(xs, w, bias, st, meta[0], meta[1], meta[2].bool(), part,
                                      activation="silu", null_block_id=pre.null_block_id)
    ref_st = pre.conv_states.copy()
    ref = pins.run_oracle_ex(pre, states=ref_st)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    assert_states_equal(state_to_host(st), ref_st)
    _compare(pre, out.view(torch.int16).cpu().numpy(), ref["out"])
    for step in range(2):
        d = workloads.make_batch(f"bf16_flow_dec{step}", 710 + step, [1] * 4, dim, part, 392,
                                 lines, col_offset=8, state_dtype="bf16")
        d.weight, d.bias, d.cache_indices = pre.weight, pre.bias, pre.cache_indices.copy()
        d.has_initial_state[:] = 1
        xd = torch.from_numpy(d.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
        ci = torch.from_numpy(d.cache_indices).to(dev)
        o = pkg.causal_conv1d_update(xd[:, d.col_offset:d.col_offset + dim], st, w, bias, ci,
                                     part, activation="silu", null_block_id=d.null_block_id)
        ref = pins.run_oracle_ex(d, states=ref_st)
        torch.cuda.synchronize()
        assert_states_equal(state_to_host(st), ref_st)
        _compare(d, o.view(torch.int16).cpu().numpy(), ref["out"])


def test_update_position_major_state_at_an_unaligned_base():
    """A position-major state whose base is 4 bytes off a 16-byte boundary
    cannot move as vectors: the update must take the element path and still
    match the oracle."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = _decode_batch(531, 64, 256, 128, 256, 100, null_count=2, state_width=4)
    dev = torch.device("cuda")
    pm = np.ascontiguousarray(b.conv_states.transpose(0, 2, 1))  # (lines, K, dim)
    buf = torch.zeros(pm.size + 4, dtype=torch.float32, device=dev)
    buf[1:1 + pm.size].copy_(torch.from_numpy(pm.ravel()))
    st = buf[1:1 + pm.size].view(pm.shape).transpose(1, 2)  # (lines, dim, K) view
    assert st.data_ptr() % 16 == 4
    x = torch.from_numpy(b.x_buf.view(np.int16)).to(dev)
    out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), -1, dtype=torch.int16,
                     device=dev)
    w = torch.from_numpy(b.weight).to(dev)
    bias = torch.from_numpy(b.bias).to(dev)
    ci = torch.from_numpy(b.cache_indices).to(dev)
    layout = pkg.make_layout(pkg.KDA_DTYPE_BF16, 4, st.stride(), w.stride())
    pkg.kda_conv1d_update(x.data_ptr() + 2 * b.col_offset, b.row_stride, b.tokens, b.dim,
                          b.part_dim, w, bias, st, ci, b.null_block_id, b.activation, out, layout)
    torch.cuda.synchronize()
    ref_st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=ref_st)
    assert_states_equal(st.contiguous().cpu().numpy(), ref_st)
    _compare(b, out.cpu().numpy(), ref["out"])
    assert buf[0].item() == 0.0 and buf[-3:].abs().sum().item() == 0.0  # guards untouched


@pytest.mark.parametrize("ci_stride", [2, 5])
@pytest.mark.parametrize("state_dtype", ["f32", "bf16"])
def test_update_strided_indices_and_decode_weight(ci_stride, state_dtype):
    """The kda_decode page's pairing: a position-major conv state and the
    [qkv, width, channel] weight, with cache_indices as a strided view."""
    b = _decode_batch(540 + ci_stride, 200, 384, 128, 392, 300, col_offset=8, null_count=3,
                      state_dtype=state_dtype)
    st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=st)
    got, got_st = _run_update(b, True, "decode3", ci_stride)
    assert_states_equal(got_st, st)
    _compare(b, got, ref["out"])


def test_update_wrapper_with_the_decode_weight():
    """causal_conv1d_update with a bf16 position-major state and the
    (3, 4, part_dim) weight, the layout the kda_decode page's fused decode
    kernel takes."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = _decode_batch(550, 96, 384, 128, 384, 120, null_count=2, state_dtype="bf16")
    dev = torch.device("cuda")
    pm = state_to_device(np.ascontiguousarray(b.conv_states.transpose(0, 2, 1)), dev)
    st = pm.transpose(1, 2)
    w, _, _ = weight_to_device(b, "decode3", dev)
    x = torch.from_numpy(b.x_buf.view(np.int16)).to(dev).view(torch.bfloat16)
    ci = torch.from_numpy(b.cache_indices).to(dev)
    out = pkg.causal_conv1d_update(x, st, w, torch.from_numpy(b.bias).to(dev), ci, b.part_dim,
                                   activation="silu", null_block_id=b.null_block_id)
    torch.cuda.synchronize()
    ref_st = b.conv_states.copy()
    ref = pins.run_oracle_ex(b, states=ref_st)
    assert_states_equal(state_to_host(st.contiguous()), ref_st)
    _compare(b, out.view(torch.int16).cpu().numpy(), ref["out"])
