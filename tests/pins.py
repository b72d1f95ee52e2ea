"""Independent checks that pin the CPU oracle to the pages and to mathematics.

Each ``pin_*`` function takes an oracle library handle (so that the same
checks can be run against deliberately broken copies of the oracle) and
raises AssertionError on a mismatch.  None of them re-types the oracle's
loop: they use a different formulation (a materialised padded column per
(sequence, channel) and exact rational arithmetic), a library routine
(torch's float64 conv1d and silu, torch's bf16 conversions), a closed form,
or an invariant that any correct implementation must satisfy.

What they follow: "vllm.models.kimi_k3.nvidia.ops.kda_conv" (docs.vllm.ai),
module docstring (exact bf16 widening, FP32 taps with FP32 weights and
state, SiLU, round to nearest even, dense planes; the state read once and
written back) and the packed_causal_conv1d_fn docstring (width-4 causal
depthwise conv as causal_conv1d_fn(x.T, ...).T, conv_states (lines, dim, 3)
updated in place, output (dim/part_dim, tokens, part_dim)).
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

import oracle
import workloads

U = 2.0 ** -24  # unit roundoff of fp32


# --------------------------------------------------------------------------
# Library conversions (torch CPU) used as independent references
# --------------------------------------------------------------------------

def torch_bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).float().numpy()


def torch_f32_to_bf16(vals: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def is_nan_bf16(bits: np.ndarray) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


# --------------------------------------------------------------------------
# Exact rational fp32 arithmetic
# --------------------------------------------------------------------------

_F32_MAX = Fraction((2 ** 24 - 1) * 2 ** 104)


def round_to_f32(q: Fraction) -> float:
    """Nearest fp32 to the exact rational q, ties to even (q != 0)."""
    sign = -1.0 if q < 0 else 1.0
    a = -q if q < 0 else q
    # e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if (Fraction(2) ** e) > a:
        e -= 1
    e = max(e, -126)  # below the normal range the quantum stays 2^-149
    qe = e - 23
    m = a / (Fraction(2) ** qe)
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = Fraction(n) * (Fraction(2) ** qe)
    if v > _F32_MAX:
        return sign * float("inf")
    return sign * float(v)


def fma_f32(a: float, b: float, c: float) -> float:
    """fp32 fused multiply-add of fp32-valued floats, one rounding, exact rationals."""
    exact = Fraction(a) * Fraction(b) + Fraction(c)
    if exact == 0:
        prod_neg = (np.signbit(a) != np.signbit(b))
        prod_zero = (a == 0.0 or b == 0.0)
        if prod_zero and c == 0.0 and prod_neg and np.signbit(c):
            return -0.0
        return 0.0
    return round_to_f32(exact)


# --------------------------------------------------------------------------
# Second formulation of the conv: a padded column per (sequence, channel)
# --------------------------------------------------------------------------

def padded_columns(b: workloads.Batch, s: int) -> tuple[np.ndarray, bool]:
    """(L+3, dim) float64 column [h0, h1, h2, x_a, ..., x_{a+L-1}] of sequence s
    (history rows first, oldest first) and whether its state line is live."""
    a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
    line = int(b.cache_indices[s])
    live = line != b.null_block_id
    hist = np.zeros((3, b.dim), dtype=np.float64)
    if live and b.has_initial_state[s]:
        hist = b.conv_states[line].T.astype(np.float64)  # (3, dim): row k = state index k
    xs = torch_bf16_to_f32(b.x_buf[a:e, b.col_offset:b.col_offset + b.dim]).astype(np.float64)
    return np.concatenate([hist, xs], axis=0), live


def run_oracle(b: workloads.Batch, lib=None, **kw) -> dict:
    return oracle.packed_conv1d(
        b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, b.conv_states,
        b.cache_indices, b.has_initial_state, b.query_start_loc, b.null_block_id,
        b.activation, lib=lib, **kw)


def plane_view(arr: np.ndarray, b: workloads.Batch) -> np.ndarray:
    """(planes, tokens, part_dim) -> (tokens, dim) with channel c at column c."""
    planes, tokens, p = arr.shape
    return np.ascontiguousarray(arr.transpose(1, 0, 2).reshape(tokens, planes * p))


def small_batch(seed: int, lengths, dim=128, part_dim=64, row_stride=None, col_offset=8,
                cache_lines=None, null_count=1, his_p=0.6, activation=1, bias=True,
                tokens=None, first_token=0, x_std=1.0, w_range=0.5) -> workloads.Batch:
    n = len(lengths)
    row_stride = row_stride or (dim + 24)
    cache_lines = cache_lines or (n + 3)
    return workloads.make_batch(
        f"small{seed}", seed, lengths, dim, part_dim, row_stride, cache_lines,
        col_offset=col_offset, x_std=x_std, w_range=w_range,
        bias_std=0.1 if bias else None, activation=activation, his_p=his_p,
        null_count=null_count, tokens=tokens, first_token=first_token)


# --------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------

def pin_bf16_widen(lib) -> None:
    """Every bf16 pattern widens to the value torch's conversion gives, and
    rounds back to itself (NaNs: stay NaN)."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f32(allb, lib)
    want = torch_bf16_to_f32(allb)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
    back = oracle.bf16_rne(got, lib)
    assert np.array_equal(back[~nan], allb[~nan])
    assert is_nan_bf16(back[nan]).all()


RNE_CASES = [  # (fp32 bits, bf16 bits) worked from the definition of round-half-even
    (0x3F808000, 0x3F80),  # tie, even below
    (0x3F818000, 0x3F82),  # tie, odd below -> up
    (0x3F808001, 0x3F81),  # just above the tie
    (0x3F807FFF, 0x3F80),  # just below the tie
    (0xBF808000, 0xBF80),  # negative tie, even
    (0xBF818000, 0xBF82),  # negative tie, odd
    (0x3FFF8000, 0x4000),  # tie that carries into the exponent
    (0x7F7FFFFF, 0x7F80),  # largest finite fp32 rounds to +inf
    (0x7F7F7FFF, 0x7F7F),  # stays finite
    (0x00008000, 0x0000),  # subnormal tie to even zero
    (0x00018000, 0x0002),  # subnormal tie up
    (0x80000000, 0x8000),  # -0
    (0x7F800000, 0x7F80),  # +inf
    (0xFF800000, 0xFF80),  # -inf
]


def pin_bf16_rne(lib, n_random: int = 1 << 20, seed: int = 7) -> None:
    """Hand-worked ties, then random patterns against torch's RNE conversion."""
    src = np.array([c[0] for c in RNE_CASES], dtype=np.uint32).view(np.float32)
    want = np.array([c[1] for c in RNE_CASES], dtype=np.uint16)
    got = oracle.bf16_rne(src, lib)
    assert np.array_equal(got, want), [hex(v) for v in got]
    rng = np.random.default_rng(seed)
    pats = rng.integers(0, 2 ** 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    vals = pats.view(np.float32)
    got = oracle.bf16_rne(vals, lib)
    ref = torch_f32_to_bf16(vals)
    nan = np.isnan(vals)
    assert np.array_equal(got[~nan], ref[~nan])
    assert is_nan_bf16(got[nan]).all()
    # NaN keeps its sign.
    assert np.array_equal(got[nan] >> 15, (pats[nan] >> 31).astype(np.uint16))


def _check_against_columns(b: workloads.Batch, res: dict, states_after: np.ndarray,
                           exact: bool) -> None:
    """Compares the oracle's preact / states with the padded-column formulation.

    exact=True: the fp32 chain acc=bias; acc=fma(v_j, w_j, acc), j oldest
    first, evaluated in exact rationals with one rounding per step; must be
    bit-identical.  exact=False: float64 window dot products within the
    error bound of four fp32 roundings."""
    pre = plane_view(res["preact"], b)
    w = b.weight.astype(np.float64)
    bias = np.zeros(b.dim) if b.bias is None else b.bias.astype(np.float64)
    expected_states = b.conv_states.copy()
    for s in range(b.num_seqs):
        a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
        L = e - a
        if L <= 0:
            continue
        col, live = padded_columns(b, s)
        if live:
            expected_states[int(b.cache_indices[s])] = col[L:L + 3].T.astype(np.float32)
        for t in range(L):
            win = col[t:t + 4]  # (4, dim), oldest first
            got = pre[a + t]
            if exact:
                for c in range(b.dim):
                    acc = float(np.float32(bias[c])) if b.bias is not None else 0.0
                    for j in range(4):
                        acc = fma_f32(float(win[j, c]), float(w[c, j]), acc)
                    assert np.float32(acc).view(np.uint32) == np.float32(got[c]).view(np.uint32), \
                        (s, t, c, acc, got[c])
            else:
                ref = bias + (win * w.T).sum(axis=0)
                mag = np.abs(bias) + (np.abs(win) * np.abs(w.T)).sum(axis=0)
                err = np.abs(got.astype(np.float64) - ref)
                assert (err <= 4 * U * mag + 1e-40).all(), (s, t, float(err.max()))
    assert np.array_equal(states_after.view(np.uint32), expected_states.view(np.uint32))


def pin_exact_rational(lib) -> None:
    """Brute force on tiny inputs: bit-identical pre-activations and states."""
    for seed, lengths in [(11, [1, 2, 3, 4, 5]), (12, [7, 0, 3, 9]), (13, [6, 2, 1, 5, 4])]:
        b = small_batch(seed, lengths, dim=64, part_dim=64, null_count=1)
        st = b.conv_states.copy()
        res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias,
                                   st, b.cache_indices, b.has_initial_state, b.query_start_loc,
                                   b.null_block_id, b.activation, want_preact=True, lib=lib)
        _check_against_columns(b, res, st, exact=True)
    b = small_batch(14, [3, 5], dim=128, part_dim=64, null_count=0, bias=False)
    st = b.conv_states.copy()
    res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, None, st,
                               b.cache_indices, b.has_initial_state, b.query_start_loc,
                               b.null_block_id, 0, want_preact=True, lib=lib)
    _check_against_columns(b, res, st, exact=True)


def pin_float64_windows(lib) -> None:
    """Window dot products in float64 (all lengths around the 3-row history and
    64-row chunk edges) within four fp32 roundings."""
    lengths = [1, 2, 3, 4, 5, 63, 64, 65, 129]
    b = small_batch(21, lengths, dim=192, part_dim=64, null_count=2, row_stride=232,
                    cache_lines=16)
    st = b.conv_states.copy()
    res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, st,
                               b.cache_indices, b.has_initial_state, b.query_start_loc,
                               b.null_block_id, b.activation, want_preact=True, lib=lib)
    _check_against_columns(b, res, st, exact=False)


def pin_torch_conv1d(lib, b: workloads.Batch | None = None) -> None:
    """torch.nn.functional.conv1d(groups=dim) in float64 over [history ; x_seq]^T,
    per sequence, against the oracle's pre-activation (library special case)."""
    if b is None:
        b = small_batch(31, [40, 1, 2, 77, 3, 130], dim=256, part_dim=128, null_count=1,
                        row_stride=320, col_offset=64, cache_lines=9)
    st = b.conv_states.copy()
    res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, st,
                               b.cache_indices, b.has_initial_state, b.query_start_loc,
                               b.null_block_id, b.activation, want_preact=True, lib=lib)
    pre = plane_view(res["preact"], b).astype(np.float64)
    w = torch.from_numpy(b.weight.astype(np.float64)).unsqueeze(1)  # (dim, 1, 4)
    bias_t = None if b.bias is None else torch.from_numpy(b.bias.astype(np.float64))
    for s in range(b.num_seqs):
        a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
        if e <= a:
            continue
        line = int(b.cache_indices[s])
        hist = np.zeros((3, b.dim))
        if line != b.null_block_id and b.has_initial_state[s]:
            hist = b.conv_states[line].T.astype(np.float64)
        xs = torch_bf16_to_f32(b.x_buf[a:e, b.col_offset:b.col_offset + b.dim]).astype(np.float64)
        inp = torch.from_numpy(np.concatenate([hist, xs]).T.copy()).unsqueeze(0)  # (1, dim, L+3)
        ref = torch.nn.functional.conv1d(inp, w, bias_t, groups=b.dim)[0].T.numpy()  # (L, dim)
        mag = torch.nn.functional.conv1d(inp.abs(), w.abs(), None if bias_t is None
                                         else bias_t.abs(), groups=b.dim)[0].T.numpy()
        err = np.abs(pre[a:e] - ref)
        assert (err <= 4 * U * mag + 1e-40).all(), (s, float(err.max()))


def pin_silu_and_rounding(lib) -> None:
    """SiLU against torch's float64 silu within a few fp32 ulp, and the stored
    bf16 against torch's RNE of the activated value."""
    b = small_batch(41, [50, 3, 90], dim=128, part_dim=64, null_count=0, cache_lines=5,
                    x_std=3.0, w_range=1.0)
    st = b.conv_states.copy()
    res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, st,
                               b.cache_indices, b.has_initial_state, b.query_start_loc,
                               b.null_block_id, 1, want_preact=True, want_act=True, lib=lib)
    live = ~np.isnan(res["preact"])
    pre = res["preact"][live].astype(np.float64)
    act = res["act"][live].astype(np.float64)
    ref = torch.nn.functional.silu(torch.from_numpy(pre)).numpy()
    assert (np.abs(act - ref) <= 8 * U * np.abs(ref) + 1e-44).all()
    assert np.array_equal(res["out"][live], torch_f32_to_bf16(res["act"][live]))
    # Values at the extremes of the SiLU, against float64 (denormal-free range).
    a = np.array([-80.0, -20.0, -3.5, -1e-3, 0.0, 1e-30, 0.5, 7.25, 30.0, 1e30], dtype=np.float32)
    got = oracle.silu(a, lib).astype(np.float64)
    ref = torch.nn.functional.silu(torch.from_numpy(a.astype(np.float64))).numpy()
    assert (np.abs(got - ref) <= 8 * U * np.abs(ref) + 1e-44).all()


def pin_closed_forms(lib) -> None:
    """Identity (w = e3), shift (w = e0) and bias-only (w = 0) kernels."""
    base = small_batch(51, [1, 2, 5, 40], dim=128, part_dim=64, null_count=1, his_p=1.0,
                       activation=0, bias=False, cache_lines=8)
    xv = base.x_buf[:, base.col_offset:base.col_offset + base.dim]
    qsl = base.query_start_loc

    # identity: out = x exactly (a -0 input gives +0, since the chain starts at +0)
    b = base.copy()
    b.weight[:] = 0
    b.weight[:, 3] = 1
    out = plane_view(run_oracle(b, lib)["out"], b)
    want = np.where((xv == 0x8000), 0, xv)
    assert np.array_equal(out[qsl[0]:qsl[-1]], want[qsl[0]:qsl[-1]])

    # shift by three rows: out[t] = x[t-3], or the rounded history for t < 3
    b = base.copy()
    b.weight[:] = 0
    b.weight[:, 0] = 1
    out = plane_view(run_oracle(b, lib)["out"], b)
    for s in range(b.num_seqs):
        a, e = int(qsl[s]), int(qsl[s + 1])
        line = int(b.cache_indices[s])
        hist = np.zeros((3, b.dim), dtype=np.float32)
        if line != b.null_block_id and b.has_initial_state[s]:
            hist = base.conv_states[line].T.copy()
        for t in range(e - a):
            want_row = xv[a + t - 3] if t >= 3 else torch_f32_to_bf16(hist[t] + np.float32(0))
            want_row = np.where(want_row == 0x8000, 0, want_row)
            assert np.array_equal(out[a + t], want_row), (s, t)

    # bias only: out = bf16(bias) on every sequence row
    b = base.copy()
    b.weight[:] = 0
    b.bias = np.linspace(-3, 3, b.dim).astype(np.float32)
    out = plane_view(run_oracle(b, lib)["out"], b)
    want = torch_f32_to_bf16(b.bias)
    for t in range(int(qsl[0]), int(qsl[-1])):
        assert np.array_equal(out[t], want)


def _sub_batch(b: workloads.Batch, ranges, his, states) -> workloads.Batch:
    """A batch holding, for each sequence, rows [lo, hi) of the original x."""
    rows = np.concatenate([np.arange(lo, hi) for lo, hi in ranges]).astype(np.int64)
    lens = [hi - lo for lo, hi in ranges]
    qsl = np.zeros(len(lens) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(lens)
    c = b.copy()
    c.x_buf = np.ascontiguousarray(b.x_buf[rows])
    c.query_start_loc = qsl
    c.has_initial_state = np.asarray(his, dtype=np.uint8)
    c.conv_states = states
    return c


def pin_chunk_carry(lib) -> None:
    """Splitting every sequence in two calls with the state carried equals one call."""
    lengths = [70, 5, 129, 4, 66]
    base = small_batch(61, lengths, dim=64, part_dim=64, null_count=0, his_p=0.5,
                       cache_lines=8)
    one = base.copy()
    full = run_oracle(one, lib)
    full_out = plane_view(full["out"], base)
    qsl = base.query_start_loc
    for m in [1, 2, 3, 17, 64, None]:
        first, second = [], []
        for s in range(base.num_seqs):
            a, e = int(qsl[s]), int(qsl[s + 1])
            cut = (e - a - 1) if m is None else min(m, e - a - 1)
            first.append((a, a + cut))
            second.append((a + cut, e))
        c1 = _sub_batch(base, first, base.has_initial_state, base.conv_states.copy())
        o1 = plane_view(run_oracle(c1, lib)["out"], c1)
        c2 = _sub_batch(base, second, np.ones(base.num_seqs), c1.conv_states)
        o2 = plane_view(run_oracle(c2, lib)["out"], c2)
        r1 = r2 = 0
        for s in range(base.num_seqs):
            (a1, b1), (a2, b2) = first[s], second[s]
            assert np.array_equal(o1[r1:r1 + b1 - a1], full_out[a1:b1]), (m, s)
            assert np.array_equal(o2[r2:r2 + b2 - a2], full_out[a2:b2]), (m, s)
            r1 += b1 - a1
            r2 += b2 - a2
        assert np.array_equal(c2.conv_states.view(np.uint32), one.conv_states.view(np.uint32)), m


def pin_zero_history(lib) -> None:
    """has_initial_state = 0 behaves as a zero state line with has_initial_state = 1,
    and a null-block sequence computes with zero history."""
    b = small_batch(71, [5, 2, 30], dim=128, part_dim=64, null_count=0, his_p=0.0,
                    cache_lines=6)
    r0 = run_oracle(b.copy(), lib)
    z = b.copy()
    z.has_initial_state[:] = 1
    for line in z.cache_indices:
        z.conv_states[line] = 0
    r1 = run_oracle(z, lib)
    assert np.array_equal(r0["out"], r1["out"])
    n = b.copy()
    n.cache_indices[:] = n.null_block_id
    n.has_initial_state[:] = 1
    r2 = run_oracle(n, lib)
    assert np.array_equal(r0["out"], r2["out"])


def pin_short_state_shift(lib) -> None:
    """Sequences shorter than 3 tokens shift the state: new = [old[L:], x rows]."""
    for his in (1, 0):
        b = small_batch(81 + his, [1, 2, 3], dim=64, part_dim=64, null_count=0,
                        his_p=float(his), cache_lines=5)
        st = b.conv_states.copy()
        run = b.copy()
        run.conv_states = st
        run_oracle(run, lib)
        for s, L in enumerate([1, 2, 3]):
            a = int(b.query_start_loc[s])
            line = int(b.cache_indices[s])
            old = b.conv_states[line] if his else np.zeros((b.dim, 3), dtype=np.float32)
            xs = torch_bf16_to_f32(b.x_buf[a:a + L, b.col_offset:b.col_offset + b.dim]).T
            want = np.concatenate([old[:, L:], xs], axis=1)
            assert np.array_equal(st[line].view(np.uint32), want.view(np.uint32)), (his, L)


def pin_permutation(lib) -> None:
    """Permuting the sequences permutes the outputs and leaves the states equal."""
    lengths = [9, 1, 33, 4, 17]
    b = small_batch(91, lengths, dim=128, part_dim=64, null_count=1, cache_lines=8)
    r = run_oracle(b.copy(), lib)
    perm = [3, 0, 4, 2, 1]
    qsl = b.query_start_loc
    ranges = [(int(qsl[s]), int(qsl[s + 1])) for s in perm]
    p = _sub_batch(b, ranges, b.has_initial_state[perm], b.conv_states.copy())
    p.cache_indices = b.cache_indices[perm].copy()
    rp = run_oracle(p, lib)
    want_states = b.copy()
    run_oracle(want_states, lib)
    assert np.array_equal(p.conv_states.view(np.uint32), want_states.conv_states.view(np.uint32))
    out, outp = plane_view(r["out"], b), plane_view(rp["out"], p)
    row = 0
    for lo, hi in ranges:
        assert np.array_equal(outp[row:row + hi - lo], out[lo:hi])
        row += hi - lo


def pin_untouched(lib) -> None:
    """Lines not referenced, the null block's sequence, rows outside
    [qsl[0], qsl[N]) and empty calls leave memory as it was."""
    b = small_batch(101, [4, 0, 9, 2], dim=128, part_dim=64, null_count=1, cache_lines=10,
                    tokens=30, first_token=5)
    # the empty sequence has no history: a state write for it would zero its line
    b.has_initial_state[1] = 0
    st = b.conv_states.copy()
    run = b.copy()
    run.conv_states = st
    out = run_oracle(run, lib)["out"]
    rows = plane_view(out, b)
    assert (rows[:5] == 0xFFFF).all() and (rows[5 + 15:] == 0xFFFF).all()
    live = {int(c) for c, L in zip(b.cache_indices, np.diff(b.query_start_loc))
            if c != b.null_block_id and L > 0}
    for line in range(b.cache_lines):
        if line not in live:
            assert np.array_equal(st[line].view(np.uint32), b.conv_states[line].view(np.uint32))
    # empty calls
    for qsl in (np.array([0], dtype=np.int32), np.array([0, 0, 0], dtype=np.int32)):
        e = b.copy()
        e.query_start_loc = qsl
        e.cache_indices = b.cache_indices[:qsl.size - 1].copy()
        e.has_initial_state = b.has_initial_state[:qsl.size - 1].copy()
        o = run_oracle(e, lib)["out"]
        assert (o == 0xFFFF).all()
        assert np.array_equal(e.conv_states.view(np.uint32), b.conv_states.view(np.uint32))


def pin_metadata_checks(lib) -> None:
    """Malformed metadata is rejected."""
    good = (np.array([0, 1], dtype=np.int32), np.array([0, 2, 5], dtype=np.int32))
    assert oracle.check_metadata(8, 4, *good, -1, lib=lib)[0] == oracle.REF_OK
    cases = [
        (np.array([0, 1]), np.array([0, 6, 5]), oracle.REF_BAD_QSL),  # decreasing
        (np.array([0, 1]), np.array([-1, 2, 5]), oracle.REF_BAD_QSL),  # negative start
        (np.array([0, 1]), np.array([0, 2, 9]), oracle.REF_BAD_QSL),  # past tokens
        (np.array([0, 4]), np.array([0, 2, 5]), oracle.REF_BAD_CACHE_INDEX),
        (np.array([-2, 1]), np.array([0, 2, 5]), oracle.REF_BAD_CACHE_INDEX),
        (np.array([1, 1]), np.array([0, 2, 5]), oracle.REF_DUP_CACHE_INDEX),
    ]
    for ci, qsl, rc in cases:
        assert oracle.check_metadata(8, 4, ci, qsl, -1, lib=lib)[0] == rc
    # two null-block sequences are not a duplicate
    assert oracle.check_metadata(8, 4, np.array([-1, -1]), good[1], -1, lib=lib)[0] == 0


ALL_PINS = [
    pin_bf16_widen, pin_bf16_rne, pin_exact_rational, pin_float64_windows, pin_torch_conv1d,
    pin_silu_and_rounding, pin_closed_forms, pin_chunk_carry, pin_zero_history,
    pin_short_state_shift, pin_permutation, pin_untouched, pin_metadata_checks,
]


# --------------------------------------------------------------------------
# The general-layout oracle: fp16 / fp32 x, state width K >= 3, strides
# --------------------------------------------------------------------------

def torch_f16_to_f32(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.float16).float().numpy()


def torch_f32_to_f16(vals: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def x_as_f32(b: workloads.Batch, rows) -> np.ndarray:
    """Input columns of b for the given rows, widened by torch's conversions."""
    xs = b.x_buf[rows, b.col_offset:b.col_offset + b.dim]
    if b.x_dtype == "bf16":
        return torch_bf16_to_f32(xs)
    if b.x_dtype == "f16":
        return torch_f16_to_f32(xs)
    return np.asarray(xs, dtype=np.float32)


DT = {"bf16": oracle.DTYPE_BF16, "f16": oracle.DTYPE_F16, "f32": oracle.DTYPE_F32}


def run_oracle_ex(b: workloads.Batch, lib=None, weight=None, states=None, **kw) -> dict:
    return oracle.packed_conv1d_ex(
        b.x_buf, DT[b.x_dtype], b.col_offset, b.dim, b.part_dim,
        b.weight if weight is None else weight, b.bias,
        b.conv_states if states is None else states, b.cache_indices, b.has_initial_state,
        b.query_start_loc, b.null_block_id, b.activation, lib=lib, **kw)


def pin_f16_widen(lib) -> None:
    """Every binary16 pattern widens to torch's value (NaN to NaN)."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got, want = oracle.f16_to_f32(allb, lib), torch_f16_to_f32(allb)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


F16_CASES = [  # (fp32 bits, binary16 bits) worked from round-half-even
    (0x3F801000, 0x3C00),  # 1 + 2^-11: tie, even below
    (0x3F803000, 0x3C02),  # 1 + 3*2^-11: tie, odd below -> up
    (0x3F801001, 0x3C01),  # just above the tie
    (0x477FE000, 0x7BFF),  # 65504, the largest finite half
    (0x477FEFFF, 0x7BFF),  # just below 65520
    (0x477FF000, 0x7C00),  # 65520: tie to the even neighbour 65536 = overflow
    (0x33800000, 0x0001),  # 2^-24, the smallest subnormal half
    (0x33000000, 0x0000),  # 2^-25: tie between 0 and 2^-24 -> 0
    (0x33000001, 0x0001),  # just above that tie
    (0x33C00000, 0x0002),  # 3 * 2^-25: tie between 1 and 2 quanta -> 2
    (0x387FE000, 0x0400),  # 1023.5 * 2^-24: tie -> the smallest normal 2^-14
    (0x387FC000, 0x03FF),  # 1023 * 2^-24, the largest subnormal half, exactly
    (0x80000000, 0x8000),  # -0
    (0x7F800000, 0x7C00),
    (0xFF800000, 0xFC00),
]


def pin_f16_rne(lib, seed: int = 9) -> None:
    """Hand-worked cases, every tie between neighbouring halves, dense samples
    of the half range and random patterns, against torch's fp32 -> fp16."""
    src = np.array([c[0] for c in F16_CASES], dtype=np.uint32).view(np.float32)
    want = np.array([c[1] for c in F16_CASES], dtype=np.uint16)
    got = oracle.f16_rne(src, lib)
    assert np.array_equal(got, want), [hex(v) for v in got]
    halves = torch_f16_to_f32(np.arange(0, 0x7C00, dtype=np.uint16)).astype(np.float64)
    ties = ((halves[:-1] + halves[1:]) / 2).astype(np.float32)  # exact in fp32
    rng = np.random.default_rng(seed)
    dense = (2.0 ** rng.uniform(-27, 17, size=1 << 20)).astype(np.float32)
    pats = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    for v in (ties, -ties, dense, -dense, pats.view(np.float32)):
        nan = np.isnan(v)
        g, w = oracle.f16_rne(v, lib), torch_f32_to_f16(v)
        assert np.array_equal(g[~nan], w[~nan])
        assert (((g[nan] & 0x7C00) == 0x7C00) & ((g[nan] & 0x3FF) != 0)).all()


def pin_ex_matches_basic(lib) -> None:
    """With bf16, width 3 and contiguous strides the general oracle computes
    bit for bit what the first one does (both pinned independently)."""
    for seed, lengths, act, bias in [(111, [5, 0, 70, 1, 2], 1, True), (112, [33, 3], 0, False)]:
        b = small_batch(seed, lengths, dim=128, part_dim=64, null_count=1, activation=act,
                        bias=bias, cache_lines=8)
        s1, s2 = b.conv_states.copy(), b.conv_states.copy()
        r1 = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, s1,
                                  b.cache_indices, b.has_initial_state, b.query_start_loc,
                                  b.null_block_id, act, lib=lib)
        r2 = run_oracle_ex(b, lib, states=s2)
        assert np.array_equal(r1["out"], r2["out"])
        assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


def pin_ex_typed_exact(lib) -> None:
    """fp16 and fp32 x: pre-activations bit-identical to the exact-rational
    FMA chain over the padded column; outputs = torch's rounding of them."""
    for x_dtype, seed in (("f16", 121), ("f32", 122)):
        b = workloads.make_batch(f"t{seed}", seed, [4, 1, 6], 64, 64, 80, 5, col_offset=8,
                                 activation=0, his_p=0.7, null_count=1, x_dtype=x_dtype)
        st = b.conv_states.copy()
        res = run_oracle_ex(b, lib, states=st, want_preact=True)
        pre = plane_view(res["preact"], b)
        w = b.weight.astype(np.float64)
        for s in range(b.num_seqs):
            a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
            line = int(b.cache_indices[s])
            hist = np.zeros((3, b.dim))
            if line != b.null_block_id and b.has_initial_state[s]:
                hist = b.conv_states[line].T.astype(np.float64)
            col = np.concatenate([hist, x_as_f32(b, slice(a, e)).astype(np.float64)])
            for t in range(e - a):
                for c in range(b.dim):
                    acc = float(np.float32(b.bias[c]))
                    for j in range(4):
                        acc = fma_f32(float(col[t + j, c]), float(w[c, j]), acc)
                    assert np.float32(acc).view(np.uint32) == pre[a + t, c].view(np.uint32)
        written = ~np.isnan(res["preact"])
        if x_dtype == "f16":
            assert np.array_equal(res["out"][written], torch_f32_to_f16(res["preact"][written]))
        else:
            assert np.array_equal(res["out"][written].view(np.uint32),
                                  res["preact"][written].view(np.uint32))


def pin_ex_state_width(lib) -> None:
    """Width K > 3: the taps read the K-3 .. K-1 positions (same outputs as a
    width-3 state holding them); afterwards the line holds the last K rows of
    [old line or zeros ; the sequence's rows]; splitting a sequence over two
    calls with the line carried equals one call."""
    for K in (4, 7):
        b = workloads.make_batch(f"k{K}", 130 + K, [1, 2, 5, 9, 20], 64, 64, 72, 8,
                                 col_offset=8, his_p=0.6, null_count=1, state_width=K)
        stK = b.conv_states.copy()
        rK = run_oracle_ex(b, lib, states=stK)
        b3 = b.copy()
        b3.conv_states = np.ascontiguousarray(b.conv_states[:, :, K - 3:])
        r3 = run_oracle_ex(b3, lib, states=b3.conv_states)
        assert np.array_equal(rK["out"], r3["out"])
        for s in range(b.num_seqs):
            line = int(b.cache_indices[s])
            if line == b.null_block_id:
                continue
            a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
            old = b.conv_states[line] if b.has_initial_state[s] else np.zeros((b.dim, K), np.float32)
            want = np.concatenate([old.T, x_as_f32(b, slice(a, e))])[-K:].T
            assert np.array_equal(stK[line].view(np.uint32), want.view(np.uint32)), (K, s)
    # chunk carry at width 5
    K = 5
    b = workloads.make_batch("carry5", 141, [30, 7, 2], 64, 64, 64, 4, his_p=0.5, state_width=K)
    full_st = b.conv_states.copy()
    full = plane_view(run_oracle_ex(b, lib, states=full_st)["out"], b)
    qsl = b.query_start_loc
    cut = [11, 3, 1]
    first = [(int(qsl[s]), int(qsl[s]) + cut[s]) for s in range(3)]
    second = [(int(qsl[s]) + cut[s], int(qsl[s + 1])) for s in range(3)]
    c1 = _sub_batch(b, first, b.has_initial_state, b.conv_states.copy())
    o1 = plane_view(run_oracle_ex(c1, lib, states=c1.conv_states)["out"], c1)
    c2 = _sub_batch(b, second, np.ones(3), c1.conv_states)
    o2 = plane_view(run_oracle_ex(c2, lib, states=c2.conv_states)["out"], c2)
    assert np.array_equal(c2.conv_states.view(np.uint32), full_st.view(np.uint32))
    r1 = r2 = 0
    for s in range(3):
        (a1, e1), (a2, e2) = first[s], second[s]
        assert np.array_equal(o1[r1:r1 + e1 - a1], full[a1:e1])
        assert np.array_equal(o2[r2:r2 + e2 - a2], full[a2:e2])
        r1, r2 = r1 + e1 - a1, r2 + e2 - a2


def pin_ex_strides(lib) -> None:
    """The same call with the state stored position-major and the weight
    tap-major (width-major), or the weight as the kda_decode page's
    [qkv, width, channel] buffer (packed or padded), gives the same outputs
    and the same state values."""
    K = 4
    b = workloads.make_batch("strides", 151, [3, 12, 1], 128, 64, 136, 6, col_offset=8,
                             his_p=0.7, null_count=1, state_width=K)
    st = b.conv_states.copy()
    ref = run_oracle_ex(b, lib, states=st)
    mem_s = np.ascontiguousarray(b.conv_states.transpose(0, 2, 1))  # (lines, K, dim)
    view_s = mem_s.transpose(0, 2, 1)  # (lines, dim, K) view, strides (K*dim, 1, dim)
    mem_w = np.ascontiguousarray(b.weight.T)  # (4, dim): tap-major
    got = run_oracle_ex(b, lib, weight=mem_w.T, states=view_s)
    assert np.array_equal(got["out"], ref["out"])
    assert np.array_equal(np.ascontiguousarray(view_s).view(np.uint32), st.view(np.uint32))
    # The kda_decode page's width-major decode weight, [qkv, width, channel]
    # with the channel contiguous (make_decode_conv1d_weight_loader): part i,
    # tap j, channel q of the part is weight[i * part_dim + q][j].
    parts = b.dim // b.part_dim
    w3 = np.ascontiguousarray(b.weight.reshape(parts, b.part_dim, 4).transpose(0, 2, 1))
    st3 = b.conv_states.copy()
    got3 = run_oracle_ex(b, lib, weight=w3, states=st3)
    assert np.array_equal(got3["out"], ref["out"])
    assert np.array_equal(st3.view(np.uint32), st.view(np.uint32))
    # the same buffer with padding between parts and between taps
    pad = np.zeros((parts, 5, b.part_dim + 8), dtype=np.float32)
    pad[:, :4, 4:4 + b.part_dim] = w3
    st4 = b.conv_states.copy()
    got4 = run_oracle_ex(b, lib, weight=pad[:, :4, 4:4 + b.part_dim], states=st4)
    assert np.array_equal(got4["out"], ref["out"])


ALL_PINS += [pin_f16_widen, pin_f16_rne, pin_ex_matches_basic, pin_ex_typed_exact,
             pin_ex_state_width, pin_ex_strides]


def pin_ex_bf16_state(lib) -> None:
    """A bf16 conv state: with bf16 x it holds exactly the values an fp32
    state would (the stored rows are input rows), so outputs and states match
    the fp32-state run bit for bit; with fp32 x the stored rows are torch's
    nearest-even rounding of the last K rows of [old line ; x rows]."""
    for K in (3, 4):
        b = workloads.make_batch(f"bst{K}", 161 + K, [1, 2, 9, 30], 128, 64, 136, 7,
                                 col_offset=8, his_p=0.6, null_count=1, state_width=K)
        b.conv_states = torch_bf16_to_f32(torch_f32_to_bf16(b.conv_states))  # bf16 values
        st32 = b.conv_states.copy()
        st16 = torch_f32_to_bf16(b.conv_states)
        r32 = run_oracle_ex(b, lib, states=st32)
        r16 = run_oracle_ex(b, lib, states=st16)
        assert np.array_equal(r32["out"], r16["out"])
        assert np.array_equal(torch_bf16_to_f32(st16).view(np.uint32), st32.view(np.uint32))
    b = workloads.make_batch("bst_f32x", 170, [1, 2, 5, 11], 64, 64, 68, 6, col_offset=4,
                             his_p=0.7, null_count=1, x_dtype="f32", state_width=4)
    st16 = torch_f32_to_bf16(b.conv_states)
    old = torch_bf16_to_f32(st16)
    run_oracle_ex(b, lib, states=st16)
    for s in range(b.num_seqs):
        line = int(b.cache_indices[s])
        if line == b.null_block_id:
            continue
        a, e = int(b.query_start_loc[s]), int(b.query_start_loc[s + 1])
        prev = old[line] if b.has_initial_state[s] else np.zeros_like(old[line])
        want = np.concatenate([prev.T, x_as_f32(b, slice(a, e))])[-4:].T
        assert np.array_equal(st16[line], torch_f32_to_bf16(np.ascontiguousarray(want))), s


ALL_PINS.append(pin_ex_bf16_state)


# --- the q/k L2 norm ("vllm.models.kimi_k3.amd.ops.kda_prefill": chunk_kda_prefill,
# use_qk_l2norm_in_kernel; q and k are [1, T, H, K], normed per token and head) ---

def pin_l2norm_closed_forms(lib) -> None:
    """Hand-worked heads: a 3-4-5 triangle, a lone entry with eps inside the
    root (1 / sqrt(1 + 3) = 1/2), a negative entry, an all-zero head."""
    y = np.array([[3, 4, 0, 0, 1, 0, 0, 0, -2, 0, 0, 0, 0, 0, 0, 0]], np.float32)
    got = oracle.l2norm_heads(y, 4, 0.0, lib)
    assert got[0, :4].tolist() == [3 / 5, 4 / 5, 0.0, 0.0]
    assert got[0, 4:8].tolist() == [1.0, 0.0, 0.0, 0.0]
    assert got[0, 8:12].tolist() == [-1.0, 0.0, 0.0, 0.0]
    got = oracle.l2norm_heads(y, 4, 3.0, lib)
    assert got[0, 4] == 0.5 and got[0, 8] == -2 / np.sqrt(7.0)
    assert got[0, 12:].tolist() == [0.0] * 4  # zero head, eps > 0: zeros


def pin_l2norm_invariants(lib) -> None:
    """On random heads: the squared norm of a result is ss / (ss + eps); every
    entry of a head is scaled by one positive factor; heads do not interact;
    scaling the input by 4 leaves an eps = 0 result bit-identical."""
    g = torch.Generator().manual_seed(71)
    y = (torch.randn(7, 192, generator=g) * torch.rand(7, 1, generator=g) * 3).numpy()
    y = y.astype(np.float32)
    eps = 1e-6
    got = oracle.l2norm_heads(y, 64, eps, lib)
    for h in range(3):
        yh = y[:, 64 * h:64 * (h + 1)].astype(np.float64)
        gh = got[:, 64 * h:64 * (h + 1)]
        ss = (yh * yh).sum(axis=1)
        assert np.allclose((gh * gh).sum(axis=1), ss / (ss + eps), rtol=1e-12, atol=0)
        ratio = gh / yh
        assert (ratio > 0).all()
        assert np.allclose(ratio, ratio[:, :1], rtol=1e-14, atol=0)
    y2 = y.copy()
    y2[:, 64:128] *= -7.5
    got2 = oracle.l2norm_heads(y2, 64, eps, lib)
    assert np.array_equal(got2[:, :64], got[:, :64]) and np.array_equal(got2[:, 128:], got[:, 128:])
    a = oracle.l2norm_heads(y, 64, 0.0, lib)
    assert np.array_equal(oracle.l2norm_heads(y * 4, 64, 0.0, lib), a)


def run_oracle_l2norm(b: workloads.Batch, norm_planes: int, head_dim: int, eps: float,
                      lib=None, states=None) -> dict:
    return oracle.packed_conv1d_l2norm(
        b.x_buf, DT[b.x_dtype], b.col_offset, b.dim, b.part_dim, b.weight, b.bias,
        b.conv_states if states is None else states, b.cache_indices, b.has_initial_state,
        b.query_start_loc, b.null_block_id, b.activation, norm_planes, head_dim, eps, lib=lib)


def pin_l2norm_conv(lib) -> None:
    """The conv with the norm folded in: planes outside the mask and the conv
    state are exactly the plain conv's; a normed plane's written rows have
    heads of unit length up to bf16 rounding, each pointing the way the same
    head of the plain (activated) conv output points, so the norm follows the
    activation; unwritten rows stay untouched; an empty mask is the plain
    conv."""
    b = workloads.make_batch("l2conv", 181, [1, 2, 7, 40], 192, 64, 200, 7, col_offset=8,
                             his_p=0.6, null_count=1, tokens=55)
    st_plain, st_norm = b.conv_states.copy(), b.conv_states.copy()
    plain = run_oracle_ex(b, lib, states=st_plain)["out"]
    normed = run_oracle_l2norm(b, 0b011, 32, 1e-6, lib, states=st_norm)["out"]
    assert np.array_equal(st_plain.view(np.uint32), st_norm.view(np.uint32))
    assert np.array_equal(normed[2], plain[2])
    written = plain[0][:, 0] != 0xFFFF
    assert (~written).sum() == 55 - 50
    for plane in (0, 1):
        assert (normed[plane][~written] == 0xFFFF).all()
        v = torch_bf16_to_f32(normed[plane][written]).astype(np.float64).reshape(-1, 2, 32)
        sq = (v * v).sum(axis=2)
        assert np.all(np.abs(sq - 1.0) < 2.0 ** -6), float(np.abs(sq - 1).max())
        p = torch_bf16_to_f32(plain[plane][written]).astype(np.float64).reshape(-1, 2, 32)
        unit = p / np.sqrt((p * p).sum(axis=2, keepdims=True))
        assert np.all(np.abs(v - unit) < 2.0 ** -6), float(np.abs(v - unit).max())
    st3 = b.conv_states.copy()
    assert np.array_equal(run_oracle_l2norm(b, 0, 32, 1e-6, lib, states=st3)["out"], plain)


ALL_PINS += [pin_l2norm_closed_forms, pin_l2norm_invariants, pin_l2norm_conv]


# --- the checker of the device epilogue over all 2^32 fp32 inputs ---

FLT_MAX = float(np.finfo(np.float32).max)


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers that step by one per representable value."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))


def pin_silu_bf16_range(lib) -> None:
    """kda_ref_silu_bf16_range, the host side of the exhaustive epilogue check
    (the kda_conv page's module docstring, 3rd paragraph: SiLU, then rounding
    to nearest even), over windows of 2^20 consecutive fp32 bit patterns:
    denormals upwards from +0, around 1.0, across the expf overflow near
    -88.72, up to +inf and into the NaNs, and one window that wraps from
    0xFFFFFFFF (negative NaNs) to 0x00000000.

    Element by element it is the rounding of the SiLU of the pattern at its
    own index (the two parts are pinned on their own above).  Against torch's
    float64 silu, rounded by torch to fp32 and then to bf16, it is within one
    bf16 ulp with the same NaN class.  Where e^-a overflows fp32 (a below
    -log(FLT_MAX)), the FP32 formula a / (1 + e^-a) is a / inf: -0."""
    n = 1 << 20
    thr = float(np.log(np.float64(FLT_MAX)))
    for first in (0x00000000, 0x3F800000 - n // 2, 0xC2B17218 - n // 2, 0x7F800000 - n // 2,
                  0xFFFFFFFF - n // 2 + 1):
        got = oracle.silu_bf16_range(first, n, lib)
        bits = ((np.arange(n, dtype=np.uint64) + np.uint64(first)) & np.uint64(0xFFFFFFFF))
        a32 = bits.astype(np.uint32).view(np.float32)
        assert np.array_equal(got, oracle.bf16_rne(oracle.silu(a32, lib), lib)), hex(first)
        with np.errstate(invalid="ignore"):  # NaN patterns widen to NaN
            a64 = a32.astype(np.float64)
        ref32 = torch.nn.functional.silu(torch.from_numpy(a64)).to(torch.float32).numpy()
        want = torch_f32_to_bf16(ref32)
        nan_got, nan_want = is_nan_bf16(got), is_nan_bf16(want)
        assert np.array_equal(nan_got, nan_want), hex(first)
        with np.errstate(invalid="ignore"):
            overflow = -a64 > thr * (1 + 1e-6)
            regular = ~nan_want & ~(-a64 > thr * (1 - 1e-6))
        assert (got[overflow] == 0x8000).all(), hex(first)
        d = np.abs(ordered_bf16(got[regular]) - ordered_bf16(want[regular]))
        assert d.size == 0 or d.max() <= 1, (hex(first), int(d.max()))


ALL_PINS.append(pin_silu_bf16_range)
