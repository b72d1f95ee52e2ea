"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it and runs the pins against it: at least
one pin has to fail.  The real oracle is never modified.
"""

import inspect
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_conv_ref.c")

# (name, text in the oracle, replacement).  Each text occurs exactly once.
MUTANTS = [
    ("taps_reversed", "acc = fmaf(v, weight[c * 4 + j], acc);",
     "acc = fmaf(v, weight[c * 4 + (3 - j)], acc);"),
    ("tap_dropped", "for (int j = 0; j < 4; ++j) {", "for (int j = 1; j < 4; ++j) {"),
    ("mul_then_add", "acc = fmaf(v, weight[c * 4 + j], acc);",
     "acc = v * weight[c * 4 + j] + acc;"),
    ("bias_dropped", "float acc = bias ? bias[c] : 0.0f;", "float acc = 0.0f;"),
    ("state_read_reversed", "h[k] = conv_states[(line * dim + c) * 3 + k];",
     "h[k] = conv_states[(line * dim + c) * 3 + (2 - k)];"),
    ("state_write_reversed", "conv_states[(line * dim + c) * 3 + k] = ns[k];",
     "conv_states[(line * dim + c) * 3 + k] = ns[2 - k];"),
    ("state_rows_off_by_one", "int64_t r = len - 3 + k;", "int64_t r = len - 4 + k;"),
    ("his_ignored", "int read_state = !is_null && has_initial_state[s];",
     "int read_state = !is_null;"),
    ("null_rejected", "if (line == null_block_id) continue;", ""),
    ("round_truncates", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) {", "if (0) {"),
    ("ties_away", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) {",
     "if (lo >= 0x8000u) {"),
    ("silu_sign", "float e = expf(-a);", "float e = expf(a);"),
    ("planes_row_major", "int64_t o = (plane * tokens + (a + t)) * part_dim + col;",
     "int64_t o = (a + t) * dim + c;"),
    ("widen_shift", "return f32_from_bits((uint32_t)h << 16);",
     "return f32_from_bits(((uint32_t)h << 16) | 1u);"),
    ("out_row_sequence_relative", "int64_t o = (plane * tokens + (a + t)) * part_dim + col;",
     "int64_t o = (plane * tokens + t) * part_dim + col;"),
    ("x_stride_is_dim",
     "float v = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * x_row_stride + c])",
     "float v = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * dim + c])"),
    ("short_state_not_shifted",
     "ns[k] = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * x_row_stride + c])\n"
     "                                     : h[r + 3];",
     "ns[k] = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * x_row_stride + c])\n"
     "                                     : h[k];"),
    ("empty_sequence_writes", "if (len <= 0) continue; /* an empty sequence",
     "if (len < 0) continue; /* an empty sequence"),
    ("silu_is_sigmoid", "return a / d;", "return 1.0f / d;"),
    ("bf16_nan_not_quieted", "return (uint16_t)(hi | 0x0040u);", "return (uint16_t)hi;"),
    # the metadata check (the pins hand it bad metadata; the conv never gets any)
    ("dup_not_detected", "for (int64_t r = 0; r < s; ++r) {", "for (int64_t r = 0; r < 0; ++r) {"),
    ("qsl_end_unchecked", "if ((int64_t)query_start_loc[num_seqs] > tokens) {", "if (0) {"),
    ("line_upper_unchecked", "if (line < 0 || line >= cache_lines) {", "if (line < 0) {"),
    ("qsl_start_unchecked", "if (query_start_loc[0] < 0) {", "if (0) {"),
    # the general-layout function and the binary16 conversions
    ("ex_taps_first3", ": h[K + r];", ": h[3 + r];"),
    ("ex_state_not_shifted", ": h[k + len];", ": h[k];"),
    ("ex_weight_stride_ignored", "acc = fmaf(v, weight[wbase + j * w_stride_j], acc);",
     "acc = fmaf(v, weight[c * 4 + j], acc);"),
    ("ex_weight_part_stride_ignored",
     "int64_t wbase = plane * w_stride_part + col * w_stride_c;",
     "int64_t wbase = c * w_stride_c;"),
    ("ex_weight_part_index_off", "int64_t wbase = plane * w_stride_part + col * w_stride_c;",
     "int64_t wbase = (dim / part_dim - 1 - plane) * w_stride_part + col * w_stride_c;"),
    ("f16_ties_away", "if (rem > halfway || (rem == halfway && (kept & 1u))) kept += 1u;",
     "if (rem >= halfway) kept += 1u;"),
    # 65504, the largest finite half, sent to infinity
    ("f16_overflow_boundary", "if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);",
     "if (a >= 0x477FE000u) return (uint16_t)(sign | 0x7C00u);"),
    ("f16_widen_no_specials",
     "if (exp == 0x1Fu) return f32_from_bits(sign | 0x7F800000u | (frac << 13));", ""),
    ("f16_no_subnormals", "int q = (e >= -14) ? e - 10 : -24;", "int q = e - 10;"),
    ("f16_widen_subnormal", "float v = ldexpf((float)frac, -24);",
     "float v = ldexpf((float)frac, -25);"),
    # stays in bounds: bf16 stores into an fp32 state only touch the array's own bytes
    ("state_stored_as_bf16_always", "ref_store(conv_states, state_dtype,",
     "ref_store(conv_states, REF_DTYPE_BF16,"),
    # the general-layout function's own copies of the basic steps
    ("ex_his_ignored", "int read_state = (!is_null) && (has_initial_state[s] != 0);",
     "int read_state = (!is_null);"),
    ("ex_bias_dropped", "float acc = (bias != NULL) ? bias[c] : 0.0f;", "float acc = 0.0f;"),
    ("ex_planes_row_major", "int64_t oi = (plane * tokens + (a + t)) * part_dim + col;",
     "int64_t oi = (a + t) * dim + c;"),
    ("ex_x_stride_ignored",
     "float v = (r >= 0) ? ref_load(x, dtype, (a + r) * x_row_stride + c) : h[K + r];",
     "float v = (r >= 0) ? ref_load(x, dtype, (a + r) * dim + c) : h[K + r];"),
    # bf16 outputs and bf16 state rows truncated instead of rounded
    ("bf16_store_truncates", "((uint16_t *)out)[i] = kda_ref_bf16_rne(y);",
     "((uint16_t *)out)[i] = (uint16_t)(bits_from_f32(y) >> 16);"),
    # the q/k L2 norm
    ("l2_first_head_only", "const float *v = y + r * width + h0;",
     "const float *v = y + r * width;"),
    ("l2_eps_outside_root", "double d = sqrt(ss + eps);", "double d = sqrt(ss) + eps;"),
    ("l2_no_root", "double d = sqrt(ss + eps);", "double d = ss + eps;"),
    ("l2_abs_not_square", "ss += (double)v[i] * (double)v[i];", "ss += fabs((double)v[i]);"),
    ("l2_last_channel_dropped", "for (int64_t i = 0; i < head_dim; ++i) ss +=",
     "for (int64_t i = 0; i + 1 < head_dim; ++i) ss +="),
    # the checker of the exhaustive epilogue test
    ("range_index_off_by_one", "float a = f32_from_bits((uint32_t)(first + i));",
     "float a = f32_from_bits((uint32_t)(first + i + 1));"),
    ("range_not_rounded", "out[i] = kda_ref_bf16_rne(kda_ref_silu(a));",
     "out[i] = (uint16_t)(bits_from_f32(kda_ref_silu(a)) >> 16);"),
    ("range_no_silu", "out[i] = kda_ref_bf16_rne(kda_ref_silu(a));",
     "out[i] = kda_ref_bf16_rne(a);"),
]


def test_real_oracle_has_every_mutation_site():
    text = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert text.count(old) == 1, name


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    text = open(SRC).read()
    assert text.count(old) == 1
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(src), out=str(tmp_path / f"{name}.so")))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError) as e:  # ValueError: the mutant rejected a call
            caught.append((pin.__name__, type(e).__name__))
            break
    assert caught, f"no pin caught mutant {name}"


# The norm's composition (which planes, which rows, after the activation) is
# Python in oracle/__init__.py; these mutants replace that function in the
# module for one test, and the L2-norm pins must catch each.
PY_MUTANTS = [
    ("l2_mask_shifted", "if not (norm_planes >> plane) & 1:",
     "if not (norm_planes >> (plane + 1)) & 1:"),
    ("l2_before_activation", "normed = l2norm_heads(post[plane][rows]",
     "normed = l2norm_heads(pre[plane][rows]"),
    ("l2_every_row", "rows = ~np.isnan(pre[plane][:, 0])",
     "rows = np.ones(pre.shape[1], dtype=bool)"),
]


@pytest.mark.parametrize("name,old,new", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_is_caught(name, old, new, monkeypatch, oracle_lib):
    src = inspect.getsource(oracle.packed_conv1d_l2norm)
    assert src.count(old) == 1, name
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    monkeypatch.setattr(oracle, "packed_conv1d_l2norm", ns["packed_conv1d_l2norm"])
    caught = []
    for pin in (pins.pin_l2norm_closed_forms, pins.pin_l2norm_invariants, pins.pin_l2norm_conv):
        try:
            pin(oracle_lib)
        except (AssertionError, ValueError) as e:
            caught.append((pin.__name__, type(e).__name__))
            break
    assert caught, f"no pin caught mutant {name}"
