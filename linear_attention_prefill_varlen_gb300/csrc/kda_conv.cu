// Packed varlen causal depthwise conv1d (width 4) for GB300 / sm_103a.
//
// The operation is the one the vLLM page "vllm.models.kimi_k3.nvidia.ops.kda_conv"
// describes (module docstring and packed_causal_conv1d_fn): a row-strided bf16
// x (tokens, dim) is read in place, each channel is convolved causally over its
// sequence with 4 FP32 taps (history rows from an FP32 paged conv state), SiLU is
// optional, and the result is rounded to bf16 (nearest even) into dense
// (tokens, part_dim) planes.  The exact per-element arithmetic is spelled out in
// include/kda_conv.h.
//
// Design (memory-bound stencil, no contraction, so no tensor cores):
//   * grid = token programs x channel blocks, linearised with the channel block
//     fastest so that neighbouring CTAs stream neighbouring columns of the same
//     rows.  A token program p belongs to sequence s with f(s) <= p < f(s+1),
//     f(s) = floor(qsl[s] / chunk) + s; each sequence owns at least
//     ceil(len / chunk) programs and the total is at most ceil(tokens/chunk) +
//     num_seqs (the bound the page's launch uses).  Each warp finds s with a
//     radix-32 search over query_start_loc (one coalesced 32-candidate probe per
//     level), so there is no host-side chunk table and the grid depends only on
//     tokens and num_seqs (graph-safe).
//   * a thread owns VEC channels (one 16- or 8-byte vector of a row) and walks
//     the chunk's rows in order: 3 history rows stay in registers as FP32, the
//     next U rows are loaded one step ahead into a register queue, and every
//     row is 4 FMAs per channel in a fixed order, the activation, a packed RNE
//     conversion and one vector store into its plane.
//   * the first chunk of a sequence reads its conv state and, in the same
//     thread, writes the updated state (the sequence's last 3 rows, or the
//     shifted old history for sequences shorter than 3), so there is exactly
//     one reader and one writer per state line and no ordering between CTAs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <type_traits>

#include "kda_conv.h"

// Launch geometry (compile-time; the defaults are the measured choice on GB300).
#ifndef KDA_VEC
#define KDA_VEC 4  // channels per thread: one 8-byte bf16 vector
#endif
#ifndef KDA_QUEUE
#define KDA_QUEUE 6  // rows in flight per thread (a multiple of 3 keeps the history in place)
#endif
#ifndef KDA_CTA_THREADS
#define KDA_CTA_THREADS 128
#endif
#ifndef KDA_MIN_BLOCKS
#define KDA_MIN_BLOCKS 7  // resident CTAs per SM the register budget is sized for
#endif
#ifndef KDA_WAVES
#define KDA_WAVES 1  // waves of resident warps a long prefill is spread over
#endif
#ifndef KDA_LOAD_L2_256
#define KDA_LOAD_L2_256 0  // 1: x loads carry the L2::256B prefetch-size hint
#endif
#ifndef KDA_STORE_CS
#define KDA_STORE_CS 1  // 1: plane stores use the streaming (evict-first) cache hint
#endif

#ifndef KDA_LOAD_EVICT_FIRST
#define KDA_LOAD_EVICT_FIRST 0  // 1: x loads carry an L2 evict-first cache policy
#endif
#ifndef KDA_STORE_EVICT_FIRST
#define KDA_STORE_EVICT_FIRST 0  // 1: plane stores carry an L2 evict-first cache policy
#endif

#if KDA_LOAD_L2_256
#define KDA_LD_X "ld.global.nc.L1::no_allocate.L2::256B"
#else
#define KDA_LD_X "ld.global.nc.L1::no_allocate"
#endif
#if KDA_STORE_CS
#define KDA_ST_OUT "st.global.cs"
#else
#define KDA_ST_OUT "st.global"
#endif

namespace {

struct Params {
    const uint16_t *x;
    int64_t x_row_stride;  // elements
    int tokens;
    int dim;
    int part_dim;
    int num_seqs;
    const float *weight;
    const float *bias;
    float *conv_states;
    const int32_t *cache_indices;
    const uint8_t *has_initial_state;
    const int32_t *qsl;
    int64_t null_block_id;
    void *out;
    int64_t plane_stride;  // tokens * part_dim elements
    int chunk;             // tokens per program (>= 4)
    int warps_per_prog;    // warps covering one program's channel vectors
    int64_t total_warps;   // programs * warps_per_prog
    int search_steps;      // radix-32 levels: smallest s with 32^s >= num_seqs
    int search_top;        // 32^(search_steps - 1)
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// One row vector of VEC bf16 channels, as VEC/2 32-bit words (channel 2i in the
// low half of word i).  Streaming load: read once, keep out of L1.
template <int VEC>
__device__ __forceinline__ void load_row(const uint16_t *p, uint32_t (&w)[VEC / 2]) {
    static_assert(VEC == 4 || VEC == 8, "VEC must be 4 or 8");
#if KDA_LOAD_EVICT_FIRST
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    if constexpr (VEC == 8) {
        asm(KDA_LD_X ".L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
            : "l"(p), "l"(pol));
    } else {
        asm(KDA_LD_X ".L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
            : "=r"(w[0]), "=r"(w[1])
            : "l"(p), "l"(pol));
    }
#else
    if constexpr (VEC == 8) {
        asm(KDA_LD_X ".v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
            : "l"(p));
    } else {
        asm(KDA_LD_X ".v2.u32 {%0, %1}, [%2];"
            : "=r"(w[0]), "=r"(w[1])
            : "l"(p));
    }
#endif
}

template <int VEC>
__device__ __forceinline__ void zero_row(uint32_t (&w)[VEC / 2]) {
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) w[i] = 0u;
}

// bf16 -> fp32 is exact: a bf16 is the upper half of an fp32 bit pattern.
template <int VEC>
__device__ __forceinline__ void widen(const uint32_t (&w)[VEC / 2], float (&f)[VEC]) {
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Two fp32 -> one word of two bf16, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

// 2^x and 1/x on the special-function unit (PTX ex2.approx.ftz / rcp.approx.ftz:
// relative error about 2^-22; subnormal inputs and results are flushed to 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// SiLU in FP32: a / (1 + e^-a) with e^-a = 2^(-a log2 e), no branch.
//   r = 1 / (0.25 (1 + e)) keeps the reciprocal's input below 2^126 for every
//   finite e (e < 2^128), so r stays a normal number; y = a * (r * 0.25).
// Where e^-a overflows (a <= -88.7228, the threshold of an IEEE expf) r is 0
// and y is -0, as in the IEEE formula; a = -inf gives NaN, also as there.
// Relative error about 2^-21 elsewhere, far inside half a bf16 ulp (2^-9):
// after rounding, within one bf16 ulp of the IEEE formula (checked over all
// 2^32 inputs).
__device__ __forceinline__ float silu_f32(float a) {
    const float e = ex2_approx(a * -1.44269504088896341f);
    const float r = rcp_approx(__fmaf_rn(e, 0.25f, 0.25f));
    return a * (r * 0.25f);
}

template <int VEC>
__device__ __forceinline__ void silu_row(float (&y)[VEC]) {
#pragma unroll
    for (int v = 0; v < VEC; ++v) y[v] = silu_f32(y[v]);
}

template <int VEC>
__device__ __forceinline__ void store_bf16_row(uint16_t *p, const float (&y)[VEC]) {
    uint32_t w[VEC / 2];
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) w[i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
#if KDA_STORE_EVICT_FIRST
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    if constexpr (VEC == 8) {
        asm volatile(KDA_ST_OUT ".L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "l"(pol)
                     : "memory");
    } else {
        asm volatile(KDA_ST_OUT ".L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(w[0]),
                     "r"(w[1]), "l"(pol)
                     : "memory");
    }
#else
    if constexpr (VEC == 8) {
        asm volatile(KDA_ST_OUT ".v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3])
                     : "memory");
    } else {
        asm volatile(KDA_ST_OUT ".v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1])
                     : "memory");
    }
#endif
}

template <int VEC>
__device__ __forceinline__ void store_f32_row(float *p, const float (&y)[VEC]) {
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
        reinterpret_cast<float4 *>(p)[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2],
                                                       y[4 * i + 3]);
    }
}

// The sequence that owns token program `prog`, or -1 if the program is idle
// before the first sequence.  Must be called by all 32 lanes of a warp.
__device__ __forceinline__ int find_sequence(const Params &p, int prog, int lane) {
    int base = 0;
    int stride = p.search_top;
    for (int level = 0; level < p.search_steps; ++level) {
        const int idx = base + lane * stride;
        bool ok = false;
        if (idx < p.num_seqs) ok = (__ldg(p.qsl + idx) / p.chunk + idx) <= prog;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, ok);
        if (m == 0u) return -1;
        base += (__popc(m) - 1) * stride;
        stride >>= 5;
    }
    return base;
}

// ---------------------------------------------------------------------------
// The conv kernel
// ---------------------------------------------------------------------------

template <int VEC, int P, bool kPreact, bool kSilu, bool kBias>
__global__ void __launch_bounds__(KDA_CTA_THREADS, KDA_MIN_BLOCKS)
    kda_packed_conv1d_kernel(const Params p) {
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gwarp >= p.total_warps) return;  // whole warps only
    const int prog = (int)(gwarp / p.warps_per_prog);
    const int wv = (int)(gwarp - (int64_t)prog * p.warps_per_prog);

    const int s = find_sequence(p, prog, lane);
    if (s < 0) return;
    const int q0 = __ldg(p.qsl + s);
    const int f_s = q0 / p.chunk + s;
    if (f_s > prog) return;
    // Clamp the sequence to [0, tokens) so that malformed offsets never read or
    // write outside x / out.
    const int a = max(q0, 0);
    const int e = min(__ldg(p.qsl + s + 1), p.tokens);
    const int k = prog - f_s;
    const int64_t t0_wide = (int64_t)a + (int64_t)k * p.chunk;
    if (t0_wide >= e) return;
    const int t0 = (int)t0_wide;
    const int t1 = min(t0 + p.chunk, e);

    const int c = (wv * 32 + lane) * VEC;
    if (c >= p.dim) return;

    // Taps and bias of this thread's channels.
    float w[VEC][4];
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p.weight) + (c + v));
        w[v][0] = q.x;
        w[v][1] = q.y;
        w[v][2] = q.z;
        w[v][3] = q.w;
    }
    float bias[VEC];
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (kBias) q = __ldg(reinterpret_cast<const float4 *>(p.bias + c) + i);
        bias[4 * i] = q.x;
        bias[4 * i + 1] = q.y;
        bias[4 * i + 2] = q.z;
        bias[4 * i + 3] = q.w;
    }

    const uint16_t *xcol = p.x + c;
    const int64_t xs = p.x_row_stride;

    // Register queue: slot u holds row t+u; it is refilled with row t+P+u as
    // soon as row t+u has been widened, so P rows are always in flight.
    uint32_t q[P][VEC / 2];
#pragma unroll
    for (int u = 0; u < P; ++u) {
        if (t0 + u < t1)
            load_row<VEC>(xcol + (int64_t)(t0 + u) * xs, q[u]);
        else
            zero_row<VEC>(q[u]);
    }

    // History rows -3, -2, -1 relative to t0 (h0 oldest), in FP32.
    float h0[VEC], h1[VEC], h2[VEC];
    if (k == 0) {
        const int64_t line = __ldg(p.cache_indices + s);
        const bool live = line != p.null_block_id;
        float st[3 * VEC];
#pragma unroll
        for (int i = 0; i < 3 * VEC; ++i) st[i] = 0.0f;
        float4 *sp = reinterpret_cast<float4 *>(p.conv_states + (line * p.dim + c) * 3);
        if (live && __ldg(p.has_initial_state + s) != 0) {
#pragma unroll
            for (int i = 0; i < 3 * VEC / 4; ++i) {
                const float4 q = sp[i];
                st[4 * i] = q.x;
                st[4 * i + 1] = q.y;
                st[4 * i + 2] = q.z;
                st[4 * i + 3] = q.w;
            }
        }
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            h0[v] = st[3 * v];
            h1[v] = st[3 * v + 1];
            h2[v] = st[3 * v + 2];
        }
        if (live) {
            // The updated state: the last 3 rows of [history ; rows a .. e-1].
            const int len = e - a;
            float ns[3][VEC];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int row = len - 3 + r;
                if (row >= 0) {
                    uint32_t raw[VEC / 2];
                    load_row<VEC>(xcol + (int64_t)(a + row) * xs, raw);
                    widen<VEC>(raw, ns[r]);
                } else {
                    // history index row + 3 = len + r, which is 1 or 2 here
#pragma unroll
                    for (int v = 0; v < VEC; ++v) ns[r][v] = (len + r == 1) ? h1[v] : h2[v];
                }
            }
#pragma unroll
            for (int i = 0; i < 3 * VEC / 4; ++i) {
                float o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int flat = 4 * i + j;  // = 3 * channel + state index
                    o[j] = ns[flat % 3][flat / 3];
                }
                sp[i] = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        uint32_t raw[VEC / 2];
        load_row<VEC>(xcol + (int64_t)(t0 - 3) * xs, raw);
        widen<VEC>(raw, h0);
        load_row<VEC>(xcol + (int64_t)(t0 - 2) * xs, raw);
        widen<VEC>(raw, h1);
        load_row<VEC>(xcol + (int64_t)(t0 - 1) * xs, raw);
        widen<VEC>(raw, h2);
    }

    const int plane = c / p.part_dim;
    const int col = c - plane * p.part_dim;
    const int64_t out_row = p.part_dim;
    int64_t o = (int64_t)plane * p.plane_stride + col + (int64_t)t0 * out_row;
    const uint16_t *xnext = xcol + (int64_t)(t0 + P) * xs;

    // P rows per step.  Steps whose rows and refills all lie inside the chunk
    // run without per-row bounds checks; the last one or two steps check.
    int t = t0;
    auto rows = [&](auto checked_tag) {
        constexpr bool kChecked = decltype(checked_tag)::value;
#pragma unroll
        for (int u = 0; u < P; ++u) {
            float xv[VEC];
            widen<VEC>(q[u], xv);
            if (!kChecked || t + P + u < t1) load_row<VEC>(xnext + (int64_t)u * xs, q[u]);
            float y[VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                float acc = kBias ? bias[v] : 0.0f;
                acc = __fmaf_rn(h0[v], w[v][0], acc);
                acc = __fmaf_rn(h1[v], w[v][1], acc);
                acc = __fmaf_rn(h2[v], w[v][2], acc);
                acc = __fmaf_rn(xv[v], w[v][3], acc);
                y[v] = acc;
                h0[v] = h1[v];
                h1[v] = h2[v];
                h2[v] = xv[v];
            }
            if constexpr (kSilu) silu_row<VEC>(y);
            if (!kChecked || t + u < t1) {
                if constexpr (kPreact)
                    store_f32_row<VEC>(static_cast<float *>(p.out) + o + u * out_row, y);
                else
                    store_bf16_row<VEC>(static_cast<uint16_t *>(p.out) + o + u * out_row, y);
            }
        }
        xnext += P * xs;
        o += P * out_row;
    };
    for (; t + 2 * P <= t1; t += P) rows(std::false_type{});
    for (; t < t1; t += P) rows(std::true_type{});
}

// The epilogue alone, over consecutive fp32 bit patterns, VEC at a time
// through the same row functions as the conv kernel.  mode 0: rounding only;
// 1: SiLU, then rounding.
template <int VEC, int kMode>
__global__ void __launch_bounds__(256) kda_epilogue_range_kernel(uint32_t first, uint64_t count,
                                                                 uint16_t *out) {
    const uint64_t step = (uint64_t)VEC * gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)VEC * (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x);
         i < count; i += step) {
        float y[VEC];
#pragma unroll
        for (int v = 0; v < VEC; ++v) y[v] = __uint_as_float(first + (uint32_t)(i + v));
        if constexpr (kMode == 1) silu_row<VEC>(y);
        if (i + VEC <= count) {
            store_bf16_row<VEC>(out + i, y);
        } else {
            for (int v = 0; v < VEC && i + v < count; v += 2) {
                const uint32_t wd = pack_bf16x2(y[v], y[v + 1]);
                out[i + v] = (uint16_t)(wd & 0xFFFFu);
                if (i + v + 1 < count) out[i + v + 1] = (uint16_t)(wd >> 16);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

thread_local char g_last_error[256] = "";

constexpr int kVec = KDA_VEC;                 // channels per thread
constexpr int kQueue = KDA_QUEUE;             // rows in flight per thread
constexpr int kThreads = KDA_CTA_THREADS;
constexpr int kWarpsPerSm = KDA_CTA_THREADS / 32 * KDA_MIN_BLOCKS;
constexpr int kDefaultSms = 152;              // GB300, for shape queries without a device
constexpr int kMinChunk = 2 * KDA_QUEUE;
constexpr int kMaxChunk = 2048;

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

kda_status_t check_sizes(int64_t x_row_stride, int64_t tokens, int64_t dim, int64_t part_dim,
                         int64_t num_seqs) {
    if (tokens < 0 || dim < 0 || num_seqs < 0 || part_dim <= 0) return KDA_ERR_INVALID_ARG;
    if (tokens > INT32_MAX || dim > INT32_MAX / 4 || num_seqs > (int64_t(1) << 30))
        return KDA_ERR_INVALID_ARG;
    if (x_row_stride < dim) return KDA_ERR_INVALID_ARG;
    if (part_dim % 64 != 0 || dim % part_dim != 0) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

kda_status_t check_args(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                        int64_t part_dim, const float *weight, const float *bias,
                        const float *conv_states, const int32_t *cache_indices,
                        const uint8_t *has_initial_state, const int32_t *query_start_loc,
                        int64_t num_seqs, int activation, const void *out) {
    kda_status_t st = check_sizes(x_row_stride, tokens, dim, part_dim, num_seqs);
    if (st != KDA_OK) return st;
    if (activation != KDA_ACT_NONE && activation != KDA_ACT_SILU) return KDA_ERR_INVALID_ARG;
    if (tokens == 0 || num_seqs == 0 || dim == 0) return KDA_OK;  // nothing is touched
    if (!x || !weight || !conv_states || !cache_indices || !has_initial_state ||
        !query_start_loc || !out)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(x) || x_row_stride % 8 != 0 || !aligned16(weight) ||
        (bias && !aligned16(bias)) || !aligned16(conv_states) || !aligned16(out))
        return KDA_ERR_MISALIGNED;
    return KDA_OK;
}

struct Shape {
    int64_t ctas;
    int threads;
    int chunk;
    int64_t programs;
    int warps_per_prog;
    int64_t total_warps;
};

// Chunk length.  The resident-warp budget is waves x SMs x warps per SM.
// Preferred: the smallest multiple of the queue depth for which every program
// (ceil(tokens/chunk) + num_seqs of them, the slack ones included) fits in the
// budget at once, so no CTA waits for a later wave.  When num_seqs alone
// exceeds the budget, the chunk that spreads the tokens over the budget.
// Clamped to [kMinChunk, kMaxChunk].  It depends only on the scalar sizes and
// the SM count, so a captured launch stays valid for new metadata.
Shape launch_shape(int64_t tokens, int64_t dim, int64_t num_seqs, int sms) {
    Shape sh{};
    sh.threads = kThreads;
    const int64_t nvec = dim / kVec;
    sh.warps_per_prog = (int)((nvec + 31) / 32);
    const int64_t slots = (int64_t)KDA_WAVES * sms * kWarpsPerSm;
    const int64_t max_programs = slots / sh.warps_per_prog;
    int64_t chunk;
    if (max_programs > num_seqs) {
        chunk = (tokens + (max_programs - num_seqs) - 1) / (max_programs - num_seqs);
    } else {
        chunk = (tokens * sh.warps_per_prog + slots - 1) / slots;
    }
    chunk = (chunk + kQueue - 1) / kQueue * kQueue;
    if (chunk < kMinChunk) chunk = kMinChunk;
    if (chunk > kMaxChunk) chunk = kMaxChunk;
    sh.chunk = (int)chunk;
    sh.programs = (tokens + sh.chunk - 1) / sh.chunk + num_seqs;
    sh.total_warps = sh.programs * sh.warps_per_prog;
    const int64_t warps_per_cta = kThreads / 32;
    sh.ctas = (sh.total_warps + warps_per_cta - 1) / warps_per_cta;
    return sh;
}

// SM count of the current device, cached per device.
int current_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kDefaultSms;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = kDefaultSms;
        cache[dev] = n;
    }
    return cache[dev];
}

template <bool kPreact, bool kSilu, bool kBias>
void launch(const Params &p, const Shape &sh, cudaStream_t stream) {
    kda_packed_conv1d_kernel<kVec, kQueue, kPreact, kSilu, kBias>
        <<<(unsigned)sh.ctas, sh.threads, 0, stream>>>(p);
}

kda_status_t run(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                 int64_t part_dim, const float *weight, const float *bias, float *conv_states,
                 const int32_t *cache_indices, const uint8_t *has_initial_state,
                 const int32_t *query_start_loc, int64_t num_seqs, int64_t null_block_id,
                 int activation, void *out, bool preact, kda_stream_t stream) {
    kda_status_t st = check_args(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
                                 cache_indices, has_initial_state, query_start_loc, num_seqs,
                                 activation, out);
    if (st != KDA_OK) return st;
    if (tokens == 0 || num_seqs == 0 || dim == 0) return KDA_OK;

    const Shape sh = launch_shape(tokens, dim, num_seqs, current_sms());
    if (sh.ctas > INT32_MAX) return KDA_ERR_INVALID_ARG;
    Params p;
    p.x = static_cast<const uint16_t *>(x);
    p.x_row_stride = x_row_stride;
    p.tokens = (int)tokens;
    p.dim = (int)dim;
    p.part_dim = (int)part_dim;
    p.num_seqs = (int)num_seqs;
    p.weight = weight;
    p.bias = bias;
    p.conv_states = conv_states;
    p.cache_indices = cache_indices;
    p.has_initial_state = has_initial_state;
    p.qsl = query_start_loc;
    p.null_block_id = null_block_id;
    p.out = out;
    p.plane_stride = tokens * part_dim;
    p.chunk = sh.chunk;
    p.warps_per_prog = sh.warps_per_prog;
    p.total_warps = sh.total_warps;
    int steps = 0;
    int64_t reach = 1;
    while (reach < num_seqs) {
        reach *= 32;
        ++steps;
    }
    p.search_steps = steps;
    p.search_top = steps > 0 ? (int)(reach / 32) : 1;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool silu = activation == KDA_ACT_SILU;
    if (preact) {
        if (bias)
            launch<true, false, true>(p, sh, s);
        else
            launch<true, false, false>(p, sh, s);
    } else if (silu) {
        if (bias)
            launch<false, true, true>(p, sh, s);
        else
            launch<false, true, false>(p, sh, s);
    } else {
        if (bias)
            launch<false, false, true>(p, sh, s);
        else
            launch<false, false, false>(p, sh, s);
    }
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) {
        snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
                 cudaGetErrorString(err));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_packed_conv1d(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                               int64_t part_dim, const float *weight, const float *bias,
                               float *conv_states, const int32_t *cache_indices,
                               const uint8_t *has_initial_state, const int32_t *query_start_loc,
                               int64_t num_seqs, int64_t null_block_id, int activation, void *out,
                               kda_stream_t stream) {
    return run(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states, cache_indices,
               has_initial_state, query_start_loc, num_seqs, null_block_id, activation, out,
               false, stream);
}

kda_status_t kda_packed_conv1d_preact_f32(const void *x, int64_t x_row_stride, int64_t tokens,
                                          int64_t dim, int64_t part_dim, const float *weight,
                                          const float *bias, float *conv_states,
                                          const int32_t *cache_indices,
                                          const uint8_t *has_initial_state,
                                          const int32_t *query_start_loc, int64_t num_seqs,
                                          int64_t null_block_id, float *out, kda_stream_t stream) {
    return run(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states, cache_indices,
               has_initial_state, query_start_loc, num_seqs, null_block_id, KDA_ACT_NONE, out,
               true, stream);
}

kda_status_t kda_packed_conv1d_check_args(const void *x, int64_t x_row_stride, int64_t tokens,
                                          int64_t dim, int64_t part_dim, const float *weight,
                                          const float *bias, const float *conv_states,
                                          const int32_t *cache_indices,
                                          const uint8_t *has_initial_state,
                                          const int32_t *query_start_loc, int64_t num_seqs,
                                          int activation, const void *out) {
    return check_args(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
                      cache_indices, has_initial_state, query_start_loc, num_seqs, activation,
                      out);
}

kda_status_t kda_packed_conv1d_launch_shape(int64_t tokens, int64_t dim, int64_t part_dim,
                                            int64_t num_seqs, int32_t sm_count, int64_t *ctas,
                                            int32_t *threads, int32_t *chunk_tokens,
                                            int64_t *programs) {
    kda_status_t st = check_sizes(dim, tokens, dim, part_dim, num_seqs);
    if (st != KDA_OK) return st;
    Shape sh{};
    if (sm_count < 0) return KDA_ERR_INVALID_ARG;
    if (tokens > 0 && num_seqs > 0 && dim > 0)
        sh = launch_shape(tokens, dim, num_seqs, sm_count > 0 ? sm_count : current_sms());
    if (ctas) *ctas = sh.ctas;
    if (threads) *threads = sh.threads;
    if (chunk_tokens) *chunk_tokens = sh.chunk;
    if (programs) *programs = sh.programs;
    return KDA_OK;
}

kda_status_t kda_validate_metadata(const int32_t *query_start_loc, const int32_t *cache_indices,
                                   int64_t num_seqs, int64_t tokens, int64_t cache_lines,
                                   int64_t null_block_id, int64_t *bad_seq) {
    int64_t dummy;
    int64_t *bad = bad_seq ? bad_seq : &dummy;
    *bad = -1;
    if (num_seqs < 0 || tokens < 0 || cache_lines < 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;
    if (!query_start_loc || !cache_indices) return KDA_ERR_INVALID_ARG;
    if (query_start_loc[0] < 0) {
        *bad = 0;
        return KDA_ERR_METADATA;
    }
    for (int64_t s = 0; s < num_seqs; ++s) {
        if (query_start_loc[s + 1] < query_start_loc[s]) {
            *bad = s;
            return KDA_ERR_METADATA;
        }
    }
    if (query_start_loc[num_seqs] > tokens) {
        *bad = num_seqs;
        return KDA_ERR_METADATA;
    }
    // A line may serve one sequence only: mark lines in a byte map.
    unsigned char *seen = nullptr;
    if (cache_lines > 0) {
        seen = static_cast<unsigned char *>(calloc((size_t)cache_lines, 1));
        if (!seen) return KDA_ERR_INVALID_ARG;
    }
    kda_status_t st = KDA_OK;
    for (int64_t s = 0; s < num_seqs; ++s) {
        const int64_t line = cache_indices[s];
        if (line == null_block_id) continue;
        if (line < 0 || line >= cache_lines || seen[line]) {
            *bad = s;
            st = KDA_ERR_METADATA;
            break;
        }
        seen[line] = 1;
    }
    free(seen);
    return st;
}

kda_status_t kda_epilogue_range(uint32_t first, uint64_t count, int activation, uint16_t *out,
                                kda_stream_t stream) {
    if (activation != KDA_ACT_NONE && activation != KDA_ACT_SILU) return KDA_ERR_INVALID_ARG;
    if (count == 0) return KDA_OK;
    if (!out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(out)) return KDA_ERR_MISALIGNED;
    const uint64_t groups = (count + kVec - 1) / kVec;
    const unsigned threads = 256;
    const uint64_t want = (groups + threads - 1) / threads;
    const unsigned blocks = (unsigned)(want < 152ull * 64 ? want : 152ull * 64);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (activation == KDA_ACT_SILU)
        kda_epilogue_range_kernel<kVec, 1><<<blocks, threads, 0, s>>>(first, count, out);
    else
        kda_epilogue_range_kernel<kVec, 0><<<blocks, threads, 0, s>>>(first, count, out);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) {
        snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
                 cudaGetErrorString(err));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

const char *kda_status_string(kda_status_t status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape (part_dim % 64 or dim % part_dim)";
        case KDA_ERR_MISALIGNED: return "misaligned pointer or row stride (16-byte rule)";
        case KDA_ERR_CUDA: return "CUDA launch error";
        case KDA_ERR_METADATA: return "malformed metadata";
    }
    return "unknown status";
}

const char *kda_last_error_string(void) { return g_last_error; }

}  // extern "C"
