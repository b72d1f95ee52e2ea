"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded bytes, element by element.

Bar (from the method's arithmetic): pre-activations, activation=None outputs
and updated conv states bit-exact; SiLU outputs within 1 bf16 ulp (expf may
differ by a few fp32 ulp between host and device, which can move a bf16
rounding by one step and no more).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import pins
import workloads
from gpu_helpers import (DeviceBatch, assert_outputs_match, assert_states_equal, oracle_run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


def _sub(b: workloads.Batch, lo: int, hi: int, name: str) -> workloads.Batch:
    """Sequences lo..hi-1 of b as their own call (token rows kept in place)."""
    c = b.copy()
    c.name = name
    c.query_start_loc = b.query_start_loc[lo:hi + 1].copy()
    c.cache_indices = b.cache_indices[lo:hi].copy()
    c.has_initial_state = b.has_initial_state[lo:hi].copy()
    return c


def _cases():
    yield from workloads.WORKLOADS.keys()
    yield "short_only"
    yield "decode_only"


def _make(name: str) -> workloads.Batch:
    if name == "short_only":
        return _sub(workloads.short_decode(), 0, 256, name)
    if name == "decode_only":
        return _sub(workloads.short_decode(), 256, 1280, name)
    return workloads.WORKLOADS[name]()


@pytest.mark.parametrize("name", list(_cases()))
def test_workload_outputs_and_states(name):
    b = _make(name)
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)


@pytest.mark.parametrize("name", ["tiny", "varlen", "short_decode", "large_nobias"])
def test_workload_with_bf16_state(name):
    """The same draws with the conv state rounded to bf16 (through
    kda_packed_conv1d_ex): states bit-exact, outputs as above."""
    b = _make(name).copy()
    b.conv_states = workloads.bf16_bits(torch.from_numpy(b.conv_states))
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)


@pytest.mark.parametrize("name", ["tiny", "varlen", "long16k", "large_nobias", "spec_decode"])
def test_workload_preactivation_bit_exact(name):
    b = _make(name)
    ref, ref_states = oracle_run(b, want_preact=True)
    d = DeviceBatch(b, preact=True)
    d.run_preact()
    torch.cuda.synchronize()
    got = d.out.cpu().numpy()
    want = ref["preact"]
    written = ~np.isnan(want)
    assert np.array_equal(np.isnan(got), ~written)
    assert np.array_equal(got[written].view(np.uint32), want[written].view(np.uint32))
    assert_states_equal(d.states(), ref_states)


SWEEP = [
    # (seed, lengths, dim, part_dim, row_stride, col_offset, extra)
    (201, [1, 2, 3, 4, 5, 63, 64, 65, 129], 192, 64, 232, 8, {}),
    (202, [0, 7, 0, 130, 1], 256, 128, 1536 + 256, 1536, {}),
    (203, [300], 128, 64, 128, 0, {"activation": 0, "bias": False}),
    (204, [5, 9, 2], 512, 256, 520, 8, {"tokens": 40, "first_token": 7}),
    (205, [1] * 40, 128, 128, 136, 0, {"null_count": 5}),
    (206, [17, 250, 33, 64, 128, 3], 384, 192, 400, 16, {"his_p": 0.3, "null_count": 2}),
    (207, [1000, 1, 999], 64, 64, 72, 8, {"activation": 0}),
    (208, [2, 2, 2, 2], 1088, 1088, 1096, 8, {"bias": False}),
    # mean length below the queue depth: the short-sequence instantiation, with
    # programs both shorter and longer than the queue
    (209, [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 1, 1, 1, 1, 1, 1], 256, 128, 264, 8, {"his_p": 0.5}),
    (210, [0, 5, 0, 1, 2, 0, 4], 192, 64, 200, 8, {"activation": 0}),
    # at most one token per sequence (tokens <= num_seqs): the looping short
    # kernel.  Empty, one- and few-row sequences; one sequence longer than two
    # chunks beside empty ones; and a map of more blocks than one wave holds,
    # so that resident blocks loop over several
    (211, [0, 1, 0, 3, 1, 0, 1, 2, 0, 0, 1, 1, 0, 1], 256, 128, 264, 8,
     {"his_p": 0.5, "null_count": 2}),
    (212, [130] + [0] * 129 + [1] * 20, 192, 64, 200, 8, {"his_p": 0.7}),
    (213, ([1] * 25 + [0] * 4 + [2]) * 100, 256, 128, 264, 8, {"null_count": 40}),
]


@pytest.mark.parametrize("case", SWEEP, ids=[str(c[0]) for c in SWEEP])
def test_sweep(case):
    seed, lengths, dim, part_dim, row_stride, col_offset, extra = case
    extra = dict(extra)
    b = pins.small_batch(seed, lengths, dim=dim, part_dim=part_dim, row_stride=row_stride,
                         col_offset=col_offset, cache_lines=len(lengths) + 5,
                         null_count=extra.pop("null_count", 1), **extra)
    ref, ref_states = oracle_run(b, want_preact=True)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)
    p = DeviceBatch(b, preact=True)
    p.run_preact()
    torch.cuda.synchronize()
    got, want = p.out.cpu().numpy(), ref["preact"]
    written = ~np.isnan(want)
    assert np.array_equal(got[written].view(np.uint32), want[written].view(np.uint32))


def test_chunk_carry_on_device():
    """Two device calls with the state carried equal one device call."""
    base = pins.small_batch(301, [200, 5, 130, 4], dim=256, part_dim=128, null_count=0,
                            cache_lines=6, his_p=0.5)
    one = DeviceBatch(base)
    one.run()
    cut = [77, 2, 64, 3]
    qsl = base.query_start_loc
    first = [(int(qsl[s]), int(qsl[s]) + cut[s]) for s in range(base.num_seqs)]
    second = [(int(qsl[s]) + cut[s], int(qsl[s + 1])) for s in range(base.num_seqs)]
    c1 = pins._sub_batch(base, first, base.has_initial_state, base.conv_states.copy())
    d1 = DeviceBatch(c1)
    d1.run()
    c2 = pins._sub_batch(base, second, np.ones(base.num_seqs), c1.conv_states)
    d2 = DeviceBatch(c2)
    d2.conv_states.copy_(d1.conv_states)
    d2.run()
    torch.cuda.synchronize()
    assert_states_equal(d2.states(), one.states())
    full = pins.plane_view(one.out_bits(), base)
    o1, o2 = pins.plane_view(d1.out_bits(), c1), pins.plane_view(d2.out_bits(), c2)
    r1 = r2 = 0
    for s in range(base.num_seqs):
        (a1, b1), (a2, b2) = first[s], second[s]
        assert np.array_equal(o1[r1:r1 + b1 - a1], full[a1:b1])
        assert np.array_equal(o2[r2:r2 + b2 - a2], full[a2:b2])
        r1 += b1 - a1
        r2 += b2 - a2


def test_empty_calls_touch_nothing():
    import linear_attention_prefill_varlen_gb300 as pkg

    b = pins.small_batch(302, [4, 4], dim=128, part_dim=64, null_count=0, cache_lines=4)
    d = DeviceBatch(b)
    before = d.states().copy()
    args = list(d.args())
    args[2] = 0  # tokens
    pkg.kda_packed_conv1d(*args, b.activation, d.out)
    args = list(d.args())
    args[11] = 0  # num_seqs
    pkg.kda_packed_conv1d(*args, b.activation, d.out)
    torch.cuda.synchronize()
    assert (d.out_bits() == 0xFFFF).all()
    assert_states_equal(d.states(), before)


def test_cuda_graph_replay_with_new_metadata():
    """A captured launch replays correctly after the metadata buffers change
    (same tokens and num_seqs): the grid depends only on those two scalars."""
    b1 = pins.small_batch(303, [100, 3, 60, 1], dim=256, part_dim=128, null_count=1,
                          cache_lines=8)
    b2 = b1.copy()
    b2.query_start_loc = np.array([0, 1, 90, 150, 164], dtype=np.int32)
    b2.cache_indices = np.array([5, -1, 2, 7], dtype=np.int32)
    b2.has_initial_state = np.array([1, 1, 0, 1], dtype=np.uint8)
    d = DeviceBatch(b1)
    stream = torch.cuda.Stream()
    d.run(stream)  # warm-up outside capture
    stream.synchronize()
    d.conv_states.copy_(torch.from_numpy(b1.conv_states))
    d.out.fill_(-1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        d.run(torch.cuda.current_stream())
    for b in (b1, b2):
        d.conv_states.copy_(torch.from_numpy(b.conv_states))
        d.query_start_loc.copy_(torch.from_numpy(b.query_start_loc))
        d.cache_indices.copy_(torch.from_numpy(b.cache_indices))
        d.has_initial_state.copy_(torch.from_numpy(b.has_initial_state))
        d.out.fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref, ref_states = oracle_run(b)
        assert_states_equal(d.states(), ref_states)
        assert_outputs_match(d.out_bits(), ref["out"], b.activation)


def test_cuda_graph_replay_one_token_batch():
    """The looping short kernel (at most one token per sequence) captured once
    and replayed with new lengths, cache lines and initial-state flags."""
    b1 = pins.small_batch(305, [1] * 50 + [0] * 10, dim=256, part_dim=128, null_count=3,
                          cache_lines=70)
    assert b1.tokens <= b1.num_seqs
    b2 = b1.copy()
    lengths = np.array([2, 0, 3] + [1] * 45 + [0] * 12)  # same tokens (50), same num_seqs
    assert lengths.sum() == b1.tokens and lengths.size == b1.num_seqs
    b2.query_start_loc = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    b2.cache_indices = np.random.default_rng(11).permutation(70)[:60].astype(np.int32)
    b2.cache_indices[[4, 9]] = -1
    b2.has_initial_state = (np.arange(60) % 3 != 0).astype(np.uint8)
    d = DeviceBatch(b1)
    stream = torch.cuda.Stream()
    d.run(stream)  # warm-up outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        d.run(torch.cuda.current_stream())
    for b in (b1, b2, b1):
        d.conv_states.copy_(torch.from_numpy(b.conv_states))
        d.query_start_loc.copy_(torch.from_numpy(b.query_start_loc))
        d.cache_indices.copy_(torch.from_numpy(b.cache_indices))
        d.has_initial_state.copy_(torch.from_numpy(b.has_initial_state))
        d.out.fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ref, ref_states = oracle_run(b)
        assert_states_equal(d.states(), ref_states)
        assert_outputs_match(d.out_bits(), ref["out"], b.activation)


def test_nonzero_stream_and_null_block_none():
    """The page-style wrapper on a side stream, with null_block_id=None."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = pins.small_batch(304, [33, 70], dim=384, part_dim=128, null_count=0, cache_lines=4,
                         col_offset=0, row_stride=384)
    d = DeviceBatch(b)
    x = d.x_buf.view(torch.bfloat16)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        out = pkg.packed_causal_conv1d_fn(x, d.weight, d.bias, d.conv_states, d.query_start_loc,
                                          d.cache_indices, d.has_initial_state.bool(),
                                          b.part_dim, activation="silu", null_block_id=None)
    stream.synchronize()
    assert pkg.packed_causal_conv1d_supported(x, d.weight, d.conv_states, b.part_dim)
    ref, ref_states = oracle_run(b)
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"], 1)


def test_many_sequences_four_search_levels():
    """40,000 sequences (lengths 0..5, some null blocks): the program search
    needs four radix-32 levels (32^3 < 40,000)."""
    rng = np.random.default_rng(7)
    lengths = rng.integers(0, 6, size=40000).tolist()
    b = workloads.make_batch("many", 701, lengths, 64, 64, 64, 40010, his_p=0.5,
                             null_count=500)
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)


def test_many_one_token_sequences_radix_search_in_the_loop():
    """40,000 sequences of 0, 1 or 2 tokens with no more tokens than
    sequences: the looping short kernel, whose window would be too wide, so
    each block finds its sequence by the four-level radix search."""
    rng = np.random.default_rng(8)
    lengths = rng.integers(0, 3, size=40000)
    twos = np.flatnonzero(lengths == 2)
    excess = int(lengths.sum()) - lengths.size
    if excess > 0:
        lengths[rng.choice(twos, size=excess, replace=False)] = 1
    assert lengths.sum() <= lengths.size
    b = workloads.make_batch("many_one_token", 702, lengths.tolist(), 64, 64, 64, 40010,
                             his_p=0.5, null_count=500)
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)


def test_short_batch_prefetch_on_a_half_warp_segment():
    """A batch of short sequences (mean 14.3 rows: the short instantiation)
    large enough for 24-row chunks, so its steps issue the L2 prefetch of
    rows beyond the queue; dim 192, so each program's second warp covers 64
    channels and prefetches 128-byte row segments.  x is a column slice of
    a wider row (offset 8, stride 200)."""
    rng = np.random.default_rng(702)
    lengths = [1] * 2900 + [400] * 100
    rng.shuffle(lengths)
    b = workloads.make_batch("short_pf", 702, lengths, 192, 64, 200, 3010, col_offset=8,
                             his_p=0.5, null_count=20)
    assert b.tokens < 16 * b.num_seqs
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(d.out_bits(), ref["out"], b.activation)


def test_offsets_beyond_32_bits():
    """40M token rows x 64 channels: the output plane offset and the x row
    offset of the last rows exceed 2^31 elements.  One 100-token sequence
    at the very end (qsl[0] = 40M - 150, so thousands of leading programs own
    no rows and exit after the search); only its rows are compared."""
    T, D, start, L = 40_000_000, 64, 40_000_000 - 150, 100
    rng = np.random.default_rng(11)
    x_buf = np.zeros((T, D), dtype=np.uint16)
    vals = torch.from_numpy(rng.standard_normal((L, D)).astype(np.float32))
    x_buf[start:start + L] = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    b = workloads.Batch("offsets", x_buf, 0, D, D,
                        rng.uniform(-0.5, 0.5, (D, 4)).astype(np.float32),
                        (rng.standard_normal(D) * 0.1).astype(np.float32),
                        rng.standard_normal((2, D, 3)).astype(np.float32),
                        np.array([1], dtype=np.int32), np.array([1], dtype=np.uint8),
                        np.array([start, start + L], dtype=np.int32), -1, 1, 11)
    ref, ref_states = oracle_run(b)
    d = DeviceBatch(b)
    d.run()
    torch.cuda.synchronize()
    assert_states_equal(d.states(), ref_states)
    got = d.out[:, start - 50:].cpu().numpy().view(np.uint16)
    assert_outputs_match(got, ref["out"][:, start - 50:], 1)
    assert (d.out[:, :start].eq(-1)).all().item()  # rows before the sequence untouched


@pytest.mark.parametrize("activation,silu", [("silu", True), ("swish", True), (True, True),
                                             (None, False), ("none", False), (False, False)])
def test_page_wrapper_activation_names_and_out(activation, silu):
    """packed_causal_conv1d_fn selects SiLU for "silu", "swish" and True, as the
    page's wrapper does, and no activation otherwise; a caller-provided `out`
    receives the result."""
    import linear_attention_prefill_varlen_gb300 as pkg

    b = pins.small_batch(950, [20, 3, 41], dim=256, part_dim=128, null_count=0, cache_lines=5,
                         col_offset=0, row_stride=256, activation=1 if silu else 0)
    d = DeviceBatch(b)
    x = d.x_buf.view(torch.bfloat16)
    out = torch.full((2, b.tokens, 128), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    ret = pkg.packed_causal_conv1d_fn(x, d.weight, d.bias, d.conv_states, d.query_start_loc,
                                      d.cache_indices, d.has_initial_state, b.part_dim,
                                      activation=activation, null_block_id=-1, out=out)
    torch.cuda.synchronize()
    assert ret.data_ptr() == out.data_ptr()
    ref, ref_states = oracle_run(b)
    assert_states_equal(d.states(), ref_states)
    assert_outputs_match(out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"],
                         b.activation)
