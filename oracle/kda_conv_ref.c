/*
 * Test oracle for the packed varlen causal depthwise conv1d of the Kimi-K3 KDA
 * layer.  TEST INFRASTRUCTURE ONLY: the product path never links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.
 *
 * Plain, slow, single-threaded C.  It shares no code with the CUDA path.
 * Every number is computed the obvious way: one sequence, one channel, one
 * token at a time.
 *
 * What it computes follows "vllm.models.kimi_k3.nvidia.ops.kda_conv"
 * (docs.vllm.ai, module docstring and packed_causal_conv1d_fn):
 *   - module docstring, 3rd paragraph: bf16 input is widened to FP32 exactly,
 *     the taps use FP32 weights and an FP32 conv state, then SiLU, then the
 *     FP32 result is rounded to bf16 to nearest even and stored as dense
 *     (tokens, part_dim) planes, one per part;
 *   - module docstring, 4th paragraph: a sequence's conv state is read once
 *     and the updated state (the last 3 input rows) is written back;
 *   - packed_causal_conv1d_fn docstring: width-4 causal depthwise conv with
 *     the semantics of causal_conv1d_fn(x.T, ...).T, conv_states of shape
 *     (cache lines, dim, 3) updated in place, output (dim/part_dim, tokens,
 *     part_dim), plane i holding channels [i*part_dim, (i+1)*part_dim).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): the accumulator starts at bias[c] (+0.0f without bias) and the four
 * products are added with fused multiply-adds, oldest tap first; SiLU is
 * a / (1 + exp(-a)) in FP32; conv state index 2 is the most recent row;
 * a sequence whose cache index equals null_block_id is computed with a zero
 * history and its state is neither read nor written; token rows outside
 * [query_start_loc[0], query_start_loc[num_seqs]) are not written.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (no FMA
 * contraction: every fused multiply-add below is an explicit fmaf call).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Status codes returned by the oracle (not the library's codes). */
#define REF_OK 0
#define REF_BAD_SHAPE 1
#define REF_BAD_QSL 2
#define REF_BAD_CACHE_INDEX 3
#define REF_DUP_CACHE_INDEX 4

static float f32_from_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 -> fp32: a bf16 value is the upper half of an fp32 bit pattern, so the
 * widening is exact (module docstring: "bf16 -> FP32 is exact"). */
float kda_ref_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* fp32 -> bf16, round to nearest, ties to even, from the definition: keep the
 * upper 16 bits and round on the lower 16.  A carry out of the mantissa bumps
 * the exponent, which is what rounding up across a binade (or to infinity)
 * means.  A NaN stays a NaN with its sign: the quiet bit is set so that
 * truncating a payload that lives only in the lower half cannot make it an
 * infinity. */
uint16_t kda_ref_bf16_rne(float f) {
    uint32_t u = bits_from_f32(f);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) {
        return (uint16_t)(hi | 0x0040u);
    }
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) {
        hi += 1u;
    }
    return (uint16_t)hi;
}

/* SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a)), all in FP32. */
float kda_ref_silu(float a) {
    float e = expf(-a);
    float d = 1.0f + e;
    return a / d;
}

/* Elementwise array forms of the three functions above. */
void kda_ref_bf16_to_f32_n(const uint16_t *in, int64_t n, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kda_ref_bf16_to_f32(in[i]);
}

void kda_ref_bf16_rne_n(const float *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kda_ref_bf16_rne(in[i]);
}

void kda_ref_silu_n(const float *in, int64_t n, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kda_ref_silu(in[i]);
}

/* bf16_rne(silu(f)) for `count` consecutive fp32 bit patterns starting at
 * `first`.  Used to check a device epilogue over the whole fp32 range. */
void kda_ref_silu_bf16_range(uint32_t first, uint64_t count, uint16_t *out) {
    for (uint64_t i = 0; i < count; ++i) {
        float a = f32_from_bits((uint32_t)(first + i));
        out[i] = kda_ref_bf16_rne(kda_ref_silu(a));
    }
}

/* Checks the metadata of one call.  On failure *bad_index is the offending
 * sequence index (or -1).  Returns a REF_* code. */
int kda_ref_check_metadata(int64_t tokens, int64_t cache_lines, const int32_t *cache_indices,
                           const int32_t *query_start_loc, int64_t num_seqs,
                           int64_t null_block_id, int64_t *bad_index) {
    *bad_index = -1;
    if (tokens < 0 || num_seqs < 0 || cache_lines < 0) return REF_BAD_SHAPE;
    if (num_seqs == 0) return REF_OK;
    if (query_start_loc[0] < 0) {
        *bad_index = 0;
        return REF_BAD_QSL;
    }
    for (int64_t s = 0; s < num_seqs; ++s) {
        if (query_start_loc[s + 1] < query_start_loc[s]) {
            *bad_index = s;
            return REF_BAD_QSL;
        }
    }
    if ((int64_t)query_start_loc[num_seqs] > tokens) {
        *bad_index = num_seqs;
        return REF_BAD_QSL;
    }
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t line = cache_indices[s];
        if (line == null_block_id) continue;
        if (line < 0 || line >= cache_lines) {
            *bad_index = s;
            return REF_BAD_CACHE_INDEX;
        }
        for (int64_t r = 0; r < s; ++r) {
            if ((int64_t)cache_indices[r] == line) {
                *bad_index = s;
                return REF_DUP_CACHE_INDEX;
            }
        }
    }
    return REF_OK;
}

/*
 * The conv, one call.
 *
 * x           bf16 bits, token row t at x[t * x_row_stride], dim channels used.
 * weight      (dim, 4) fp32, weight[c*4 + j] multiplies row t-3+j.
 * bias        (dim) fp32 or NULL.
 * conv_states (cache_lines, dim, 3) fp32, updated in place.
 * out         (dim/part_dim, tokens, part_dim) bf16 bits.
 * preact      NULL or (dim/part_dim, tokens, part_dim) fp32: the accumulator
 *             before the activation.
 * act         NULL or the same layout: the fp32 value after the activation,
 *             before rounding.
 * activation  0 = none, 1 = SiLU.
 */
int kda_ref_packed_conv1d(const uint16_t *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                          int64_t part_dim, const float *weight, const float *bias,
                          float *conv_states, int64_t cache_lines, const int32_t *cache_indices,
                          const uint8_t *has_initial_state, const int32_t *query_start_loc,
                          int64_t num_seqs, int64_t null_block_id, int activation, uint16_t *out,
                          float *preact, float *act) {
    int64_t bad;
    if (tokens < 0 || dim < 0 || part_dim <= 0 || num_seqs < 0) return REF_BAD_SHAPE;
    if (dim % part_dim != 0 || x_row_stride < dim) return REF_BAD_SHAPE;
    if (activation != 0 && activation != 1) return REF_BAD_SHAPE;
    if (tokens == 0 || num_seqs == 0) return REF_OK;
    int rc = kda_ref_check_metadata(tokens, cache_lines, cache_indices, query_start_loc, num_seqs,
                                    null_block_id, &bad);
    if (rc != REF_OK) return rc;

    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t a = query_start_loc[s];
        int64_t len = (int64_t)query_start_loc[s + 1] - a;
        if (len <= 0) continue; /* an empty sequence: no output, state untouched */
        int64_t line = cache_indices[s];
        int is_null = (line == null_block_id);
        int read_state = !is_null && has_initial_state[s];

        for (int64_t c = 0; c < dim; ++c) {
            /* History rows -3, -2, -1 of the sequence: h[0] oldest, h[2] newest. */
            float h[3] = {0.0f, 0.0f, 0.0f};
            if (read_state) {
                for (int k = 0; k < 3; ++k) h[k] = conv_states[(line * dim + c) * 3 + k];
            }
            int64_t plane = c / part_dim;
            int64_t col = c % part_dim;

            for (int64_t t = 0; t < len; ++t) {
                float acc = bias ? bias[c] : 0.0f;
                for (int j = 0; j < 4; ++j) {
                    int64_t r = t - 3 + j; /* sequence-relative row of tap j */
                    float v = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * x_row_stride + c])
                                       : h[r + 3];
                    acc = fmaf(v, weight[c * 4 + j], acc);
                }
                float y = activation ? kda_ref_silu(acc) : acc;
                int64_t o = (plane * tokens + (a + t)) * part_dim + col;
                out[o] = kda_ref_bf16_rne(y);
                if (preact) preact[o] = acc;
                if (act) act[o] = y;
            }

            if (!is_null) {
                /* New state: the last 3 rows of [h ; x rows of the sequence]. */
                float ns[3];
                for (int k = 0; k < 3; ++k) {
                    int64_t r = len - 3 + k;
                    ns[k] = (r >= 0) ? kda_ref_bf16_to_f32(x[(a + r) * x_row_stride + c])
                                     : h[r + 3];
                }
                for (int k = 0; k < 3; ++k) conv_states[(line * dim + c) * 3 + k] = ns[k];
            }
        }
    }
    return REF_OK;
}

/* ------------------------------------------------------------------------ */
/* The general form: x / out in bf16, fp16 or fp32, a conv state of width     */
/* K >= 3 with arbitrary element strides, and a strided weight.               */
/* ------------------------------------------------------------------------ */

#define REF_DTYPE_BF16 0
#define REF_DTYPE_F16 1
#define REF_DTYPE_F32 2

/* IEEE binary16 -> fp32, exact, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 = zero/subnormal
 * (value fraction * 2^-24), exponent 31 = infinity/NaN. */
float kda_ref_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t exp = (h >> 10) & 0x1Fu;
    uint32_t frac = h & 0x3FFu;
    if (exp == 0x1Fu) return f32_from_bits(sign | 0x7F800000u | (frac << 13));
    if (exp != 0) return f32_from_bits(sign | ((exp + 112u) << 23) | (frac << 13));
    /* zero or subnormal: frac * 2^-24, exact in fp32 */
    float v = ldexpf((float)frac, -24);
    return sign ? -v : v;
}

/* fp32 -> IEEE binary16, round to nearest, ties to even, from the definition:
 * the result is the binary16 value nearest to f (the even one on a tie);
 * values at or beyond 65520 (the largest finite half plus half an ulp) go to
 * infinity.  NaN stays NaN with its sign (quiet bit set). */
uint16_t kda_ref_f16_rne(float f) {
    uint32_t u = bits_from_f32(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u | ((a >> 13) & 0x3FFu));
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520: inf */
    int e = (int)(a >> 23) - 127;                               /* unbiased exponent */
    uint32_t m = (a & 0x7FFFFFu) | (a >= 0x00800000u ? 0x800000u : 0u);
    if (a < 0x00800000u) e = -126;                               /* fp32 subnormal */
    /* the half quantum at this magnitude: 2^(e-10) for normal halves, 2^-24 below */
    int q = (e >= -14) ? e - 10 : -24;
    /* m * 2^(e-23) / 2^q = m >> (q - e + 23); round that shift to nearest even */
    int shift = q - e + 23;
    if (shift >= 32) return sign; /* far below the smallest subnormal half */
    uint32_t kept = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t halfway = 1u << (shift - 1);
    if (rem > halfway || (rem == halfway && (kept & 1u))) kept += 1u;
    /* kept counts quanta of 2^q: for normal halves it includes the implicit
     * 1024, and a carry to 2048 lands in the next binade */
    if (q == -24) return (uint16_t)(sign | kept); /* subnormal (or the smallest normal) */
    uint32_t biased = (uint32_t)(e + 15);
    if (kept >= 2048u) {
        kept >>= 1;
        biased += 1u;
    }
    if (biased >= 31u) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (biased << 10) | (kept & 0x3FFu));
}

void kda_ref_f16_to_f32_n(const uint16_t *in, int64_t n, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kda_ref_f16_to_f32(in[i]);
}

void kda_ref_f16_rne_n(const float *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kda_ref_f16_rne(in[i]);
}

static float ref_load(const void *x, int dtype, int64_t i) {
    if (dtype == REF_DTYPE_BF16) return kda_ref_bf16_to_f32(((const uint16_t *)x)[i]);
    if (dtype == REF_DTYPE_F16) return kda_ref_f16_to_f32(((const uint16_t *)x)[i]);
    return ((const float *)x)[i];
}

static void ref_store(void *out, int dtype, int64_t i, float y) {
    if (dtype == REF_DTYPE_BF16)
        ((uint16_t *)out)[i] = kda_ref_bf16_rne(y);
    else if (dtype == REF_DTYPE_F16)
        ((uint16_t *)out)[i] = kda_ref_f16_rne(y);
    else
        ((float *)out)[i] = y;
}

/*
 * The conv with the general layout.  Differences from kda_ref_packed_conv1d:
 *   x and out are of type `dtype` (bf16, fp16 or fp32; out has x's type, as
 *   packed_causal_conv1d_fn returns x.dtype); fp16 / bf16 outputs are rounded
 *   to nearest even, fp32 outputs are the FP32 result itself;
 *   weight[c][j] is at weight[(c / part_dim) * w_stride_part +
 *   (c % part_dim) * w_stride_c + j * w_stride_j]: a (dim, 4) weight with
 *   strides (s_c, s_j) is w_stride_part = part_dim * s_c; the width-major
 *   decode weight of "vllm.models.kimi_k3.amd.ops.kda_decode"
 *   (make_decode_conv1d_weight_loader: indexed [qkv, width, channel], the
 *   channel contiguous) is a (dim / part_dim, 4, part_dim) buffer with
 *   w_stride_part = 4 * part_dim, w_stride_j = part_dim, w_stride_c = 1;
 *   the conv state of a line holds the K = state_width most recent rows,
 *   position K-1 the newest, element (line, c, k) at
 *   conv_states[line * s_stride_line + c * s_stride_c + k * s_stride_k].
 *   The taps read its last 3 positions; afterwards the line holds the last K
 *   rows of [old state (or zeros) ; the sequence's rows].
 *   The state is stored as state_dtype: fp32, or bf16 (read exactly, written
 *   rounded to nearest even; with bf16 x the stored rows are exact).
 * With dtype bf16, K = 3 and contiguous strides this is kda_ref_packed_conv1d.
 */
int kda_ref_packed_conv1d_ex(const void *x, int dtype, int64_t x_row_stride, int64_t tokens,
                             int64_t dim, int64_t part_dim, const float *weight,
                             int64_t w_stride_c, int64_t w_stride_j, int64_t w_stride_part,
                             const float *bias,
                             void *conv_states, int state_dtype, int64_t cache_lines,
                             int64_t state_width,
                             int64_t s_stride_line, int64_t s_stride_c, int64_t s_stride_k,
                             const int32_t *cache_indices, const uint8_t *has_initial_state,
                             const int32_t *query_start_loc, int64_t num_seqs,
                             int64_t null_block_id, int activation, void *out, float *preact) {
    int64_t bad;
    if (tokens < 0 || dim < 0 || part_dim <= 0 || num_seqs < 0) return REF_BAD_SHAPE;
    if (dim % part_dim != 0 || x_row_stride < dim) return REF_BAD_SHAPE;
    if (activation != 0 && activation != 1) return REF_BAD_SHAPE;
    if (dtype != REF_DTYPE_BF16 && dtype != REF_DTYPE_F16 && dtype != REF_DTYPE_F32)
        return REF_BAD_SHAPE;
    if (state_width < 3 || state_width > 64) return REF_BAD_SHAPE;
    if (state_dtype != REF_DTYPE_F32 && state_dtype != REF_DTYPE_BF16) return REF_BAD_SHAPE;
    if (tokens == 0 || num_seqs == 0) return REF_OK;
    int rc = kda_ref_check_metadata(tokens, cache_lines, cache_indices, query_start_loc, num_seqs,
                                    null_block_id, &bad);
    if (rc != REF_OK) return rc;
    const int64_t K = state_width;

    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t a = query_start_loc[s];
        int64_t len = (int64_t)query_start_loc[s + 1] - a;
        if (len <= 0) continue;
        int64_t line = cache_indices[s];
        int is_null = (line == null_block_id);
        int read_state = (!is_null) && (has_initial_state[s] != 0);

        for (int64_t c = 0; c < dim; ++c) {
            float h[64];
            for (int64_t k = 0; k < K; ++k)
                h[k] = read_state ? ref_load(conv_states, state_dtype,
                                             line * s_stride_line + c * s_stride_c + k * s_stride_k)
                                  : 0.0f;
            int64_t plane = c / part_dim;
            int64_t col = c % part_dim;
            int64_t wbase = plane * w_stride_part + col * w_stride_c;

            for (int64_t t = 0; t < len; ++t) {
                float acc = (bias != NULL) ? bias[c] : 0.0f;
                for (int j = 0; j <= 3; ++j) {
                    int64_t r = t - 3 + j;
                    float v = (r >= 0) ? ref_load(x, dtype, (a + r) * x_row_stride + c) : h[K + r];
                    acc = fmaf(v, weight[wbase + j * w_stride_j], acc);
                }
                float y = activation ? kda_ref_silu(acc) : acc;
                int64_t oi = (plane * tokens + (a + t)) * part_dim + col;
                ref_store(out, dtype, oi, y);
                if (preact) preact[oi] = acc;
            }

            if (!is_null) {
                float ns[64];
                for (int64_t k = 0; k < K; ++k) {
                    int64_t r = len - K + k;
                    ns[k] = (r >= 0) ? ref_load(x, dtype, (a + r) * x_row_stride + c) : h[k + len];
                }
                for (int64_t k = 0; k < K; ++k)
                    ref_store(conv_states, state_dtype,
                              line * s_stride_line + c * s_stride_c + k * s_stride_k, ns[k]);
            }
        }
    }
    return REF_OK;
}

/*
 * The q/k L2 norm, per token and head.  "vllm.models.kimi_k3.amd.ops.
 * kda_prefill" (chunk_kda_prefill: q and k are [1, T, H, K]; its
 * use_qk_l2norm_in_kernel flag moves the normalisation of q and k into the
 * kernel that consumes them, and the fused path's comment gives it to that
 * kernel's prologue) norms each head's K channels of a token.  The pages print neither the formula's
 * epsilon nor its precision.  The reading: out = y / sqrt(sum over the head
 * of y^2 + eps), eps a caller argument, computed here in double from the FP32
 * conv outputs y (after the activation).
 *
 * y is rows x width floats (width = heads * head_dim, head h at columns
 * h*head_dim .. (h+1)*head_dim - 1); out receives rows x width doubles.
 */
int kda_ref_l2norm_heads(const float *y, int64_t rows, int64_t width, int64_t head_dim,
                         double eps, double *out) {
    if (rows < 0 || width < 0 || head_dim <= 0 || width % head_dim != 0) return REF_BAD_SHAPE;
    if (!(eps >= 0.0)) return REF_BAD_SHAPE;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t h0 = 0; h0 < width; h0 += head_dim) {
            const float *v = y + r * width + h0;
            double ss = 0.0;
            for (int64_t i = 0; i < head_dim; ++i) ss += (double)v[i] * (double)v[i];
            double d = sqrt(ss + eps);
            for (int64_t i = 0; i < head_dim; ++i) out[r * width + h0 + i] = (double)v[i] / d;
        }
    }
    return REF_OK;
}
