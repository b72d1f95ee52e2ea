// Packed varlen causal depthwise conv1d (width 4) for GB300 / sm_103a.
//
// The operation is the one the vLLM page "vllm.models.kimi_k3.nvidia.ops.kda_conv"
// describes (module docstring and packed_causal_conv1d_fn): a row-strided x
// (tokens, dim) is read in place, each channel is convolved causally over its
// sequence with 4 FP32 taps (history rows from a paged conv state, FP32 as on
// the page or optionally bf16), SiLU is optional, and the result is rounded to
// x's type (nearest even) into dense (tokens, part_dim) planes.  The exact per-element arithmetic is spelled out in
// include/kda_conv.h.
//
// Design (memory-bound stencil, no contraction, so no tensor cores):
//   * The grid is programs x warps-per-program warps, the warp index fastest,
//     so that neighbouring warps stream neighbouring columns of the same rows.
//     A program p belongs to sequence s with f(s) <= p < f(s+1),
//     f(s) = floor(qsl[s] / chunk) + s: each sequence owns at least
//     ceil(len / chunk) programs and there are ceil(tokens / chunk) + num_seqs
//     in all (the bound the page's launch uses).  Each warp finds s on the
//     device, by a radix-32 search over query_start_loc (one coalesced
//     32-candidate probe per level) or, for batches of more than 32 sequences,
//     by one round of loads over the window of query_start_loc that can hold
//     the owner, so there is no host-side chunk table and the grid depends only
//     on scalar sizes (graph-safe).
//   * Batches of short sequences (under 16 rows on average) launch a separate
//     instantiation with paths for programs shorter than the queue, one for
//     single-row sequences (decode tokens), and an L2 prefetch of rows beyond
//     the queue.  Batches of at most one token per sequence run that code as
//     one wave of resident blocks looping over the program map's blocks.
//   * A thread owns VEC channels of its program's rows and walks them in order:
//     3 history rows stay in registers as FP32, a rolling queue of P raw rows
//     keeps P loads in flight (a slot is refilled as soon as its row has been
//     widened), and every row is 4 FMAs per channel in a fixed order, the
//     activation, a packed round-to-nearest conversion and one vector store.
//   * The first chunk of a sequence reads its conv state and, in the same
//     thread, writes the updated state (the last rows of [old state ; the
//     sequence's rows]), so each state line has exactly one reader and one
//     writer and no ordering between CTAs is needed.
//   * The decode-shaped update (one token per sequence) is its own kernel with
//     no program search: one thread per (token, channel vector), or threads
//     that keep a channel vector and loop over the tokens.
//   * A device-side metadata check (two small kernels over the sequences)
//     serves callers that want their metadata checked where it lives.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <float.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <type_traits>

#include "kda_conv.h"

// Launch geometry (compile-time; the defaults are the measured choice on GB300).
#ifndef KDA_VEC
#define KDA_VEC 4  // channels per thread
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
#ifndef KDA_MIN_BLOCKS_F32
#define KDA_MIN_BLOCKS_F32 5  // the same for fp32 x (twice the queue registers)
#endif
#ifndef KDA_LOOP_MIN_BLOCKS
#define KDA_LOOP_MIN_BLOCKS 8  // the looping one-token kernel (16-bit x, no norm)
#endif
#ifndef KDA_LOOP_QUEUE
#define KDA_LOOP_QUEUE 3  // its queue depth for the rare programs of several rows
#endif
#ifndef KDA_WAVES
#define KDA_WAVES 1  // waves of resident warps a long prefill is spread over
#endif
#ifndef KDA_LOAD_L2_256
#define KDA_LOAD_L2_256 0  // 1: x loads carry the L2::256B prefetch-size hint
#endif
#ifndef KDA_SHORT_PREFETCH
#define KDA_SHORT_PREFETCH 6  // short-sequence kernel: rows beyond the queue fetched into L2 (0: off)
#endif
#ifndef KDA_STORE_CS
#define KDA_STORE_CS 1  // 1: plane stores use the streaming (evict-first) cache hint
#endif

#ifndef KDA_PDL
#define KDA_PDL 1  // 1: launch as a programmatic dependent of the preceding kernel (launch_kernel)
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

constexpr int kMaxStateWidth = 64;

// Division by a divisor fixed for a launch, as a multiply-high and two
// shifts (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): for 1 <= d < 2^31, l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, every n < 2^32 has
// n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0), t = umulhi(m, n).
struct FastDiv {
    uint32_t m;
    int s1, s2;
};

FastDiv make_fast_div(uint32_t d) {
    int l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    FastDiv f;
    f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1);
    f.s1 = l < 1 ? l : 1;
    f.s2 = l > 1 ? l - 1 : 0;
    return f;
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
    const uint32_t t = __umulhi(f.m, n);
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

struct Params {
    const void *x;
    int64_t x_row_stride;  // elements
    int tokens;
    int dim;
    int part_dim;
    int num_seqs;
    const float *weight;
    int64_t w_stride_c;  // weight[c][j] at weight[(c / part_dim) * w_stride_part +
    int64_t w_stride_j;  //   (c % part_dim) * w_stride_c + j * w_stride_j]
    int64_t w_stride_part;
    bool weight_dense;  // strides (4, 1): one float4 per channel
    const float *bias;
    void *conv_states;    // fp32, or bf16 when state_bf16
    int state_width;      // K >= 3; the taps read positions K-3 .. K-1
    int64_t s_stride[3];  // element strides of conv_states: line, channel, position
    bool state_dense;     // K == 3 and strides (3 * dim, 3, 1)
    bool state_bf16;      // stored as bf16: read exactly, written rounded to nearest even
    bool state_posvec;    // channels contiguous at each position (s_stride[1] == 1), line
                          // and position strides multiples of 4, base aligned: the four
                          // channels of a position move as one vector
    bool weight_tapvec;   // tap-major weight (w_stride_c == 1, w_stride_j % 4 == 0,
                          // 16-byte base): a tap's four channels are one float4
    const int32_t *cache_indices;
    int64_t ci_stride;  // sequence s uses cache_indices[s * ci_stride]
    const uint8_t *has_initial_state;
    const int32_t *qsl;
    int64_t null_block_id;
    void *out;
    int64_t plane_stride;  // tokens * part_dim elements
    int chunk;             // tokens per program (>= 4)
    int warps_per_prog;    // warps covering one program's channel vectors
    FastDiv chunk_div;     // division by chunk
    FastDiv wpp_div;       // division by warps_per_prog
    FastDiv part_div;      // division by part_dim
    FastDiv nvec_div;      // division by dim / VEC (the decode update's item index)
    int64_t total_warps;   // programs * warps_per_prog
    int search_steps;      // radix-32 levels: smallest s with 32^s >= num_seqs
    int search_top;        // 32^(search_steps - 1)
    int win_span;          // ceil(tokens / chunk): the owner of program p is >= p - win_span
    int win_rounds;        // 32-entry rounds of the window search (0: the radix search)
    uint32_t norm_mask;    // planes whose heads are L2-normalised (kNorm kernels)
    int norm_lanes;        // lanes per head: head_dim / VEC (a power of two <= 32)
    float norm_eps;        // added to the sum of squares inside the root
    unsigned map_ctas;     // blocks of the program map (total_warps / warps per block)
};

// ---------------------------------------------------------------------------
// Device helpers.  kDtype: KDA_DTYPE_BF16, KDA_DTYPE_F16 or KDA_DTYPE_F32 (the
// storage of x and out).  A row vector of VEC channels is kept raw, as
// VEC * bytes / 4 32-bit words.
// ---------------------------------------------------------------------------

template <int kDtype>
__host__ __device__ constexpr int elem_bytes() {
    return kDtype == KDA_DTYPE_F32 ? 4 : 2;
}

template <int VEC, int kDtype>
__host__ __device__ constexpr int row_words() {
    return VEC * elem_bytes<kDtype>() / 4;
}

// Streaming load of one raw row vector: read once, kept out of L1.
template <int W>
__device__ __forceinline__ void load_row(const void *p, uint32_t (&w)[W]) {
    static_assert(W == 2 || W % 4 == 0, "row vectors are 8 or 16*n bytes");
    if constexpr (W == 2) {
        asm(KDA_LD_X ".v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
    } else {
#pragma unroll
        for (int i = 0; i < W / 4; ++i) {
            asm(KDA_LD_X ".v4.u32 {%0, %1, %2, %3}, [%4];"
                : "=r"(w[4 * i]), "=r"(w[4 * i + 1]), "=r"(w[4 * i + 2]), "=r"(w[4 * i + 3])
                : "l"(static_cast<const char *>(p) + 16 * i));
        }
    }
}

template <int W>
__device__ __forceinline__ void zero_row(uint32_t (&w)[W]) {
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = 0u;
}

// Raw row -> FP32, exactly: a bf16 is the upper half of an fp32 bit pattern;
// every binary16 value is an fp32 value (hardware conversion); fp32 as is.
template <int VEC, int kDtype>
__device__ __forceinline__ void widen(const uint32_t (&w)[row_words<VEC, kDtype>()],
                                      float (&f)[VEC]) {
    if constexpr (kDtype == KDA_DTYPE_BF16) {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else if constexpr (kDtype == KDA_DTYPE_F16) {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) {
            __half2 h;
            memcpy(&h, &w[i], sizeof h);
            const float2 v = __half22float2(h);
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) f[i] = __uint_as_float(w[i]);
    }
}

// Two fp32 -> one word of two bf16, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

// Two fp32 -> one word of two binary16, round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    return u;
}

template <int W>
__device__ __forceinline__ void store_words(void *p, const uint32_t (&w)[W]) {
    if constexpr (W == 2) {
        asm volatile(KDA_ST_OUT ".v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1])
                     : "memory");
    } else {
#pragma unroll
        for (int i = 0; i < W / 4; ++i) {
            asm volatile(KDA_ST_OUT ".v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(
                             static_cast<char *>(p) + 16 * i),
                         "r"(w[4 * i]), "r"(w[4 * i + 1]), "r"(w[4 * i + 2]), "r"(w[4 * i + 3])
                         : "memory");
        }
    }
}

// FP32 row -> x's type (round to nearest even) -> one vector store.
template <int VEC, int kDtype>
__device__ __forceinline__ void store_out_row(void *p, const float (&y)[VEC]) {
    constexpr int W = row_words<VEC, kDtype>();
    uint32_t w[W];
    if constexpr (kDtype == KDA_DTYPE_BF16) {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) w[i] = pack_bf16x2(y[2 * i], y[2 * i + 1]);
    } else if constexpr (kDtype == KDA_DTYPE_F16) {
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) w[i] = pack_f16x2(y[2 * i], y[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) w[i] = __float_as_uint(y[i]);
    }
    store_words<W>(p, w);
}

template <int VEC>
__device__ __forceinline__ void store_f32_row(float *p, const float (&y)[VEC]) {
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
        reinterpret_cast<float4 *>(p)[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2],
                                                       y[4 * i + 3]);
    }
}

// Conv state, dense width 3: the 3 * VEC values of channels c .. c+VEC-1 of a
// line start at element (line * dim + c) * 3, address sp.  fp32: 12 * VEC bytes, 16-byte
// aligned (c is a multiple of 4).  bf16: 6 * VEC bytes, 8-byte aligned (dim is
// a multiple of 64 and c of 4), moved as 8-byte words of four values each.
__device__ __forceinline__ void *state_line_ptr(const Params &p, int64_t line, int c, bool bf16) {
    const int64_t off = (line * p.dim + c) * 3;
    return bf16 ? static_cast<void *>(static_cast<uint16_t *>(p.conv_states) + off)
                : static_cast<void *>(static_cast<float *>(p.conv_states) + off);
}

template <int VEC>
__device__ __forceinline__ void load_state3(const void *sp, bool bf16, float (&st)[3 * VEC]) {
    if (bf16) {
#pragma unroll
        for (int i = 0; i < 3 * VEC / 4; ++i) {
            const uint2 u = static_cast<const uint2 *>(sp)[i];
            st[4 * i] = __uint_as_float(u.x << 16);
            st[4 * i + 1] = __uint_as_float(u.x & 0xFFFF0000u);
            st[4 * i + 2] = __uint_as_float(u.y << 16);
            st[4 * i + 3] = __uint_as_float(u.y & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 3 * VEC / 4; ++i) {
            const float4 v4 = static_cast<const float4 *>(sp)[i];
            st[4 * i] = v4.x;
            st[4 * i + 1] = v4.y;
            st[4 * i + 2] = v4.z;
            st[4 * i + 3] = v4.w;
        }
    }
}

// Stores rows r = 0, 1, 2 of ns as state positions 0, 1, 2 (element 3 v + r).
template <int VEC>
__device__ __forceinline__ void store_state3(void *sp, bool bf16, const float (&ns)[3][VEC]) {
#define KDA_NS(flat) ns[(flat) % 3][(flat) / 3]
    if (bf16) {
#pragma unroll
        for (int i = 0; i < 3 * VEC / 4; ++i)
            static_cast<uint2 *>(sp)[i] = make_uint2(pack_bf16x2(KDA_NS(4 * i), KDA_NS(4 * i + 1)),
                               pack_bf16x2(KDA_NS(4 * i + 2), KDA_NS(4 * i + 3)));
    } else {
#pragma unroll
        for (int i = 0; i < 3 * VEC / 4; ++i)
            static_cast<float4 *>(sp)[i] = make_float4(KDA_NS(4 * i), KDA_NS(4 * i + 1), KDA_NS(4 * i + 2),
                                KDA_NS(4 * i + 3));
    }
#undef KDA_NS
}

// Four consecutive conv-state elements starting at element i (i a multiple of
// 4, the base aligned): one float4, or one 8-byte word of four bf16.
__device__ __forceinline__ void state_get4(const Params &p, int64_t i, bool bf16,
                                           float (&v)[4]) {
    if (bf16) {
        const uint2 u = *reinterpret_cast<const uint2 *>(
            static_cast<const uint16_t *>(p.conv_states) + i);
        v[0] = __uint_as_float(u.x << 16);
        v[1] = __uint_as_float(u.x & 0xFFFF0000u);
        v[2] = __uint_as_float(u.y << 16);
        v[3] = __uint_as_float(u.y & 0xFFFF0000u);
    } else {
        const float4 q = *reinterpret_cast<const float4 *>(static_cast<const float *>(p.conv_states) + i);
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    }
}

__device__ __forceinline__ void state_set4(const Params &p, int64_t i, bool bf16,
                                           const float (&v)[4]) {
    if (bf16)
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.conv_states) + i) =
            make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
    else
        *reinterpret_cast<float4 *>(static_cast<float *>(p.conv_states) + i) =
            make_float4(v[0], v[1], v[2], v[3]);
}

// Element offset of weight[c][0] (c's part, then c within the part).  A
// thread's VEC channels never straddle a part (part_dim % 64 == 0, c % VEC == 0).
__device__ __forceinline__ int64_t weight_base(const Params &p, int c) {
    const int part = (int)fast_div((uint32_t)c, p.part_div);
    return (int64_t)part * p.w_stride_part + (int64_t)(c - part * p.part_dim) * p.w_stride_c;
}

// Conv state element i (any layout), fp32 or bf16.
__device__ __forceinline__ float state_get(const Params &p, int64_t i) {
    if (p.state_bf16)
        return __uint_as_float((uint32_t)static_cast<const uint16_t *>(p.conv_states)[i] << 16);
    return static_cast<const float *>(p.conv_states)[i];
}

__device__ __forceinline__ void state_set(const Params &p, int64_t i, float v) {
    if (p.state_bf16)
        static_cast<uint16_t *>(p.conv_states)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else
        static_cast<float *>(p.conv_states)[i] = v;
}

// One row's four taps per channel, oldest first, from the accumulator's start
// value (the bias, or +0 without one) with fused multiply-adds; then the
// history moves up a row (h0 <- h1 <- h2 <- x).
template <int VEC, bool kBias>
__device__ __forceinline__ void taps_row(const float (&w)[VEC][4], const float (&bias)[VEC],
                                         float (&h0)[VEC], float (&h1)[VEC], float (&h2)[VEC],
                                         const float (&xv)[VEC], float (&y)[VEC]) {
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

// 1/sqrt(x) on the special-function unit (PTX rsqrt.approx.ftz: relative
// error about 2^-23; subnormal inputs are flushed to 0, giving +inf).
__device__ __forceinline__ float rsqrt_approx(float x) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The q/k L2 norm of G rows: a head is `lanes` consecutive lanes' VEC
// channels (lanes a power of two, the group aligned), all of which call this
// together with the group's lane mask.  Each row y *= 1 / sqrt(sum of y^2 +
// eps): the sum in FP32 (each lane's squares, then a butterfly over the
// group, unrolled for the 32-lane head of 128 channels), the root on the
// SFU.  The G butterflies are independent, so their shuffles overlap instead
// of waiting on one another.
template <int G, int VEC>
__device__ __forceinline__ void l2norm_rows(float (&y)[G][VEC], float eps, int lanes,
                                            unsigned mask) {
    float ss[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        ss[g] = 0.0f;
#pragma unroll
        for (int v = 0; v < VEC; ++v) ss[g] = __fmaf_rn(y[g][v], y[g][v], ss[g]);
    }
    if (lanes == 32) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) ss[g] += __shfl_xor_sync(0xFFFFFFFFu, ss[g], off);
        }
    } else {
        for (int off = lanes >> 1; off > 0; off >>= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) ss[g] += __shfl_xor_sync(mask, ss[g], off);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float r = rsqrt_approx(ss[g] + eps);
#pragma unroll
        for (int v = 0; v < VEC; ++v) y[g][v] *= r;
    }
}

// The same for up to 8 rows over a full-warp head (32 lanes), as a
// reduce-scatter: three halving levels leave each lane with one row's partial
// sum over 8 lanes (row 4*b4 + 2*b3 + b2 of its lane bits), two more levels
// complete it, one reciprocal root per lane, and each row's factor is then
// read from lane 4 * row.  Fewer shuffles and roots than G butterflies.
template <int G, int VEC>
__device__ __forceinline__ void l2norm_rows_warp(float (&y)[G][VEC], float eps, int lane) {
    static_assert(G <= 8, "up to eight rows");
    float s[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        s[g] = 0.0f;
        if (g < G) {
#pragma unroll
            for (int v = 0; v < VEC; ++v) s[g] = __fmaf_rn(y[g][v], y[g][v], s[g]);
        }
    }
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float k4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b4 ? s[4 + i] : s[i];
        const float send = b4 ? s[i] : s[4 + i];
        k4[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float k2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b3 ? k4[2 + i] : k4[i];
        const float send = b3 ? k4[i] : k4[2 + i];
        k2[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float k1 = (b2 ? k2[1] : k2[0]) + __shfl_xor_sync(0xFFFFFFFFu, b2 ? k2[0] : k2[1], 4);
    k1 += __shfl_xor_sync(0xFFFFFFFFu, k1, 2);
    k1 += __shfl_xor_sync(0xFFFFFFFFu, k1, 1);
    const float r = rsqrt_approx(k1 + eps);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float rg = __shfl_sync(0xFFFFFFFFu, r, 4 * g);
#pragma unroll
        for (int v = 0; v < VEC; ++v) y[g][v] *= rg;
    }
}

template <int VEC>
__device__ __forceinline__ void l2norm_row(float (&y)[VEC], float eps, int lanes,
                                           unsigned mask) {
    l2norm_rows<1, VEC>(reinterpret_cast<float (&)[1][VEC]>(y), eps, lanes, mask);
}

// The lane mask of this lane's head group (`lanes` a power of two <= 32).
__device__ __forceinline__ unsigned head_group_mask(int lane, int lanes) {
    if (lanes >= 32) return 0xFFFFFFFFu;
    return ((1u << lanes) - 1u) << (lane & ~(lanes - 1));
}

// The sequence that owns program `prog`, or -1 if the program is idle before
// the first sequence.  Must be called by all 32 lanes of a warp.
__device__ __forceinline__ int find_sequence(const Params &p, int prog, int lane) {
    int base = 0;
    int stride = p.search_top;
    for (int level = 0; level < p.search_steps; ++level) {
        const int idx = base + lane * stride;
        bool ok = false;
        if (idx < p.num_seqs) ok = (int)fast_div((uint32_t)__ldg(p.qsl + idx), p.chunk_div) + idx <= prog;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, ok);
        if (m == 0u) return -1;
        base += (__popc(m) - 1) * stride;
        stride >>= 5;
    }
    return base;
}

// Entry r of v for a warp-uniform r (a chain of selects, no local memory).
template <int N>
__device__ __forceinline__ int pick(const int (&v)[N], int r) {
    int x = v[0];
#pragma unroll
    for (int i = 1; i < N; ++i) x = (r == i) ? v[i] : x;
    return x;
}

// The same search in one round of loads.  With 0 <= qsl[s] <= tokens,
// f(s) <= prog < f(s+1) puts s in [prog - floor(tokens / chunk), prog], and
// the last sequence's programs end before ceil(tokens / chunk) + num_seqs, so
// s >= prog - ceil(tokens / chunk) holds for every owner s.  Hence
// the warp loads that window of query_start_loc (with the entry after it) at
// once, 32 entries per round and up to kMaxRounds rounds, all independent,
// instead of a chain of dependent levels.  floor(q / chunk) + j <= prog is
// tested as q < (prog - j + 1) * chunk (no division).  *q0 and *q1 receive
// qsl[s] and qsl[s+1] from the loaded window.  Returns -1 for an idle program.
template <int kMaxRounds>
__device__ __forceinline__ int find_sequence_window(const Params &p, int prog, int lane, int &q0,
                                                    int &q1) {
    const int lo = max(0, prog - p.win_span);
    const int hi = min(p.num_seqs, prog + 1);  // entries lo .. hi are loaded; s < hi
    int v[kMaxRounds];
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        const int j = lo + 32 * r + lane;
        v[r] = 0;
        if (r < p.win_rounds && j <= hi) v[r] = __ldg(p.qsl + j);
    }
    int count = 0;
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        if (r < p.win_rounds) {
            const int j = lo + 32 * r + lane;
            const bool ok = j < hi && (int64_t)v[r] < (int64_t)(prog - j + 1) * p.chunk;
            count += __popc(__ballot_sync(0xFFFFFFFFu, ok));
        }
    }
    if (count == 0) return -1;
    const int i0 = count - 1, i1 = count;  // window positions of s and s + 1
    q0 = __shfl_sync(0xFFFFFFFFu, pick(v, i0 >> 5), i0 & 31);
    q1 = __shfl_sync(0xFFFFFFFFu, pick(v, i1 >> 5), i1 & 31);
    return lo + i0;
}

constexpr int kWindowRounds = 4;  // the window search covers up to 128 entries

// A hint to the TMA unit: bring `bytes` of global memory (16-byte aligned, a
// multiple of 16 bytes) into L2.  It holds no register and nothing waits on it.
__device__ __forceinline__ void l2_prefetch(const void *ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(__cvta_generic_to_global(ptr)),
                 "r"(bytes)
                 : "memory");
}

// ---------------------------------------------------------------------------
// The conv kernel
// ---------------------------------------------------------------------------

// Resident CTAs per SM the register budget is sized for: fp32 rows are twice
// as wide, so their queue needs more registers.  The L2-norm epilogue holds a
// whole step's activations at once (its P head reductions run side by side,
// 24 more registers); it pays for them by keeping the thread's taps and bias
// in shared memory instead (reloaded per row, 20 registers fewer), so it runs
// at the plain kernel's occupancy.  Measured on GB300 for the 16K prefill with
// the norm: taps in registers at 5 CTAs 58.2 us, in shared memory at 7 CTAs
// 53.9 us (the plain kernel 52.6 us in the same process); 256 short prefills +
// 1024 decode tokens 94.5 -> 83.8 us; 64-channel heads (4 x 8192 tokens x
// 3 x 1088) 82.0 -> 73.8 us.
// fp32 x keeps two CTAs fewer with the norm: at the plain fp32 budget its
// norm variants spill.
template <int kDtype, bool kNorm = false>
__host__ __device__ constexpr int min_blocks() {
    return kDtype == KDA_DTYPE_F32 ? KDA_MIN_BLOCKS_F32 - (kNorm ? 2 : 0) : KDA_MIN_BLOCKS;
}

// This thread's taps (VEC float4) and bias (VEC / 4 float4) from shared
// address a, loaded afresh at each use (volatile: kept next to the use).
template <int VEC>
__device__ __forceinline__ void taps_from_shared(uint32_t a, float (&w)[VEC][4],
                                                 float (&b)[VEC]) {
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(w[v][0]), "=f"(w[v][1]), "=f"(w[v][2]), "=f"(w[v][3])
                     : "r"(a + 16u * v));
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(b[4 * i]), "=f"(b[4 * i + 1]), "=f"(b[4 * i + 2]), "=f"(b[4 * i + 3])
                     : "r"(a + 16u * (VEC + i)));
}

// kGeneral: the weight and the conv state may have any strides and the state
// any width K; otherwise both are dense (weight (dim, 4), state (lines, dim, 3)).
// kShort: programs with fewer rows than the queue take a path that computes
// only their rows.  It is a separate instantiation, chosen by the host for
// batches of short sequences: its mere presence costs the long-chunk path
// about 3 % on GB300 (register allocation and scheduling of the main loop
// shift), while it saves 10-15 % on batches of one- to five-token sequences.
// Its steps also prefetch the rows KDA_SHORT_PREFETCH beyond the queue's
// refill into L2 (16-bit x).  Such batches run many waves of warps, each
// exposing its start-up latency, and the prefetch hides part of it (4.5 % on
// 256 short prefills + 1024 decode tokens).  A single wave of long chunks
// already saturates DRAM: there the same prefetch cost 8-12 %.
// kNorm: planes in norm_mask get the per-head L2 norm after the activation.
// conv_block runs the warps of block `block` of the program map: map warp
// block * (blockDim.x / 32) + threadIdx.x / 32.
template <int VEC, int P, int kDtype, bool kGeneral, bool kPreact, bool kSilu, bool kBias,
          bool kShort, bool kNorm>
__device__ __forceinline__ void conv_block(const Params &p, const unsigned block) {
    constexpr int W = row_words<VEC, kDtype>();
    // x and out are addressed in elements of their storage type
    using XT = typename std::conditional<kDtype == KDA_DTYPE_F32, float, uint16_t>::type;
    using OT = typename std::conditional<kPreact, float, XT>::type;
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (int64_t)block * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gwarp >= p.total_warps) return;  // whole warps only
    const int prog = (int)fast_div((uint32_t)gwarp, p.wpp_div);  // total_warps < 2^32
    const int wv = (int)(gwarp - (int64_t)prog * p.warps_per_prog);

    int s, q0, q1;
    if (p.win_rounds > 0) {
        s = find_sequence_window<kWindowRounds>(p, prog, lane, q0, q1);
        if (s < 0) return;
    } else {
        s = find_sequence(p, prog, lane);
        if (s < 0) return;
        q0 = __ldg(p.qsl + s);
        q1 = __ldg(p.qsl + s + 1);
    }
    // A negative offset (malformed metadata) divides as a huge one: the
    // program is then idle, and nothing outside x and out is touched.
    const int64_t f_s = (int64_t)fast_div((uint32_t)q0, p.chunk_div) + s;
    if (f_s > prog) return;
    // Clamp the sequence to [0, tokens) so that malformed offsets never read or
    // write outside x / out.
    const int a = max(q0, 0);
    const int e = min(q1, p.tokens);
    const int k = (int)(prog - f_s);
    const int64_t t0_wide = (int64_t)a + (int64_t)k * p.chunk;
    if (t0_wide >= e) return;
    const int t0 = (int)t0_wide;
    const int t1 = min(t0 + p.chunk, e);

    const int c = (wv * 32 + lane) * VEC;
    if (c >= p.dim) return;

    // Taps and bias of this thread's channels.
    float w[VEC][4];
    if (!kGeneral || p.weight_dense) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(p.weight) + (c + v));
            w[v][0] = q.x;
            w[v][1] = q.y;
            w[v][2] = q.z;
            w[v][3] = q.w;
        }
    } else {
        const int64_t wb = weight_base(p, c);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[v][j] = __ldg(p.weight + wb + v * p.w_stride_c + j * p.w_stride_j);
        }
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

    const XT *xcol = static_cast<const XT *>(p.x) + c;
    const int64_t xs = p.x_row_stride;

    if constexpr (kShort && !kPreact) {
        // A one-row sequence (a decode token): one x row, the state line, one
        // output row and the line shifted by one row, as the decode update.
        if (k == 0 && t1 - t0 == 1 && e - a == 1 && (!kGeneral || p.state_dense)) {
            uint32_t raw[W];
            load_row<W>(xcol + (int64_t)t0 * xs, raw);
            const int64_t line = __ldg(p.cache_indices + (int64_t)s * p.ci_stride);
            const bool live = line != p.null_block_id;
            const bool read = live && __ldg(p.has_initial_state + s) != 0;
            const bool bf16 = kGeneral && p.state_bf16;
            void *sp = state_line_ptr(p, line, c, bf16);
            float st[3 * VEC];
#pragma unroll
            for (int i = 0; i < 3 * VEC; ++i) st[i] = 0.0f;
            if (read) load_state3<VEC>(sp, bf16, st);
            float xv[VEC], g0[VEC], g1[VEC], g2[VEC];
            widen<VEC, kDtype>(raw, xv);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                g0[v] = st[3 * v];
                g1[v] = st[3 * v + 1];
                g2[v] = st[3 * v + 2];
            }
            if (live) {
                float ns[3][VEC];
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    ns[0][v] = g1[v];
                    ns[1][v] = g2[v];
                    ns[2][v] = xv[v];
                }
                store_state3<VEC>(sp, bf16, ns);
            }
            float y[VEC];
            taps_row<VEC, kBias>(w, bias, g0, g1, g2, xv, y);
            if constexpr (kSilu) silu_row<VEC>(y);
            const int plane1 = (int)fast_div((uint32_t)c, p.part_div);
            if constexpr (kNorm) {
                if ((p.norm_mask >> plane1) & 1u)
                    l2norm_row<VEC>(y, p.norm_eps, p.norm_lanes, head_group_mask(lane, p.norm_lanes));
            }
            store_out_row<VEC, kDtype>(static_cast<XT *>(p.out) + (int64_t)plane1 * p.plane_stride +
                                           (c - plane1 * p.part_dim) + (int64_t)t0 * p.part_dim, y);
            return;
        }
    }
    // kNorm: the taps and bias move to this thread's slot of shared memory
    // and are reloaded for each row (see min_blocks).  Only the thread itself
    // reads its slot, so no barrier is needed.
    uint32_t tap_slot = 0;
    if constexpr (kNorm) {
        static_assert(VEC % 4 == 0, "taps and bias as float4s");
        __shared__ __align__(16) float4 taps_smem[KDA_CTA_THREADS][VEC + VEC / 4];
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            taps_smem[threadIdx.x][v] = make_float4(w[v][0], w[v][1], w[v][2], w[v][3]);
#pragma unroll
        for (int i = 0; i < VEC / 4; ++i)
            taps_smem[threadIdx.x][VEC + i] =
                make_float4(bias[4 * i], bias[4 * i + 1], bias[4 * i + 2], bias[4 * i + 3]);
        tap_slot = (uint32_t)__cvta_generic_to_shared(&taps_smem[threadIdx.x][0]);
        // the reloads are asm the compiler cannot see into: keep the stores
        // above them (a compiler-only barrier; one thread, one address, so
        // the hardware keeps the order)
        asm volatile("" ::: "memory");
    }
    // Register queue: slot u holds row t+u; it is refilled with row t+P+u as
    // soon as row t+u has been widened, so P rows are always in flight.
    uint32_t q[P][W];
#pragma unroll
    for (int u = 0; u < P; ++u) {
        if (t0 + u < t1)
            load_row<W>(xcol + (int64_t)(t0 + u) * xs, q[u]);
        else
            zero_row<W>(q[u]);
    }

    // History rows -3, -2, -1 relative to t0 (h0 oldest), in FP32.
    float h0[VEC], h1[VEC], h2[VEC];
    // kShort: a whole sequence shorter than the queue writes its new state
    // from the history registers after its rows (they then hold the last 3
    // rows of [old state ; its rows]) instead of loading those rows again.
    // Measured on GB300 with the one-row path above: 1024 one-token
    // sequences 32.5 -> 30.7 us, 1024 x 4 tokens 39.3 -> 38.8 us, 256 short
    // prefills + 1024 decode tokens 81.9 -> 79.8 us.
    bool defer = false;
    void *defer_sp = nullptr;
    bool defer_bf16 = false;
    if (k == 0) {
        const int64_t line = __ldg(p.cache_indices + (int64_t)s * p.ci_stride);
        const bool live = line != p.null_block_id;
        const bool read = live && __ldg(p.has_initial_state + s) != 0;
        const int len = e - a;
        if (!kGeneral || p.state_dense) {
            // Width 3, contiguous: a thread's VEC channels are 3*VEC values.
            const bool bf16 = kGeneral && p.state_bf16;
            void *sp = state_line_ptr(p, line, c, bf16);
            float st[3 * VEC];
#pragma unroll
            for (int i = 0; i < 3 * VEC; ++i) st[i] = 0.0f;
            if (read) load_state3<VEC>(sp, bf16, st);
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                h0[v] = st[3 * v];
                h1[v] = st[3 * v + 1];
                h2[v] = st[3 * v + 2];
            }
            if (kShort && live && t1 - t0 < P && t1 == e) {
                defer = true;
                defer_sp = sp;
                defer_bf16 = bf16;
            } else if (live) {
                // The updated state: the last 3 rows of [history ; rows a .. e-1].
                float ns[3][VEC];
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    const int row = len - 3 + r;
                    if (row >= 0) {
                        uint32_t raw[W];
                        load_row<W>(xcol + (int64_t)(a + row) * xs, raw);
                        widen<VEC, kDtype>(raw, ns[r]);
                    } else {
                        // history index row + 3 = len + r, which is 1 or 2 here
#pragma unroll
                        for (int v = 0; v < VEC; ++v) ns[r][v] = (len + r == 1) ? h1[v] : h2[v];
                    }
                }
                store_state3<VEC>(sp, bf16, ns);
            }
        } else {
            // Any width K and strides: positions K-3 .. K-1 feed the taps; the
            // update keeps the last K rows of [old line ; the sequence's rows].
            // Ascending positions read position kk + len before it is written.
            const int K = p.state_width;
            const int64_t s0 = p.s_stride[0], s1 = p.s_stride[1], s2 = p.s_stride[2];
            const int64_t base = line * s0 + (int64_t)c * s1;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                h0[v] = read ? state_get(p, base + v * s1 + (K - 3) * s2) : 0.0f;
                h1[v] = read ? state_get(p, base + v * s1 + (K - 2) * s2) : 0.0f;
                h2[v] = read ? state_get(p, base + v * s1 + (K - 1) * s2) : 0.0f;
            }
            if (live) {
                for (int kk = 0; kk < K; ++kk) {
                    const int row = len - K + kk;
                    float vals[VEC];
                    if (row >= 0) {
                        uint32_t raw[W];
                        load_row<W>(xcol + (int64_t)(a + row) * xs, raw);
                        widen<VEC, kDtype>(raw, vals);
                    } else {
#pragma unroll
                        for (int v = 0; v < VEC; ++v)
                            vals[v] = read ? state_get(p, base + v * s1 + (kk + len) * s2) : 0.0f;
                    }
#pragma unroll
                    for (int v = 0; v < VEC; ++v) state_set(p, base + v * s1 + kk * s2, vals[v]);
                }
            }
        }
    } else {
        uint32_t raw[W];
        load_row<W>(xcol + (int64_t)(t0 - 3) * xs, raw);
        widen<VEC, kDtype>(raw, h0);
        load_row<W>(xcol + (int64_t)(t0 - 2) * xs, raw);
        widen<VEC, kDtype>(raw, h1);
        load_row<W>(xcol + (int64_t)(t0 - 1) * xs, raw);
        widen<VEC, kDtype>(raw, h2);
    }

    // One row's taps, from registers or (kNorm) from the shared slot.
    auto row_taps = [&](const float (&xv)[VEC], float (&yy)[VEC]) {
        if constexpr (kNorm) {
            float wr[VEC][4], br[VEC];
            taps_from_shared<VEC>(tap_slot, wr, br);
            taps_row<VEC, kBias>(wr, br, h0, h1, h2, xv, yy);
        } else {
            taps_row<VEC, kBias>(w, bias, h0, h1, h2, xv, yy);
        }
    };

    const int plane = (int)fast_div((uint32_t)c, p.part_div);
    const int col = c - plane * p.part_dim;
    const int64_t out_row = p.part_dim;  // elements between output rows
    // Heads never straddle planes, so a head group agrees on norm_on.
    const bool norm_on = kNorm && ((p.norm_mask >> plane) & 1u);
    const unsigned norm_group = kNorm ? head_group_mask(lane, p.norm_lanes) : 0u;
    int64_t o = (int64_t)plane * p.plane_stride + col + (int64_t)t0 * out_row;
    const XT *xnext = xcol + (int64_t)(t0 + P) * xs;

    // P rows per step.  Steps whose rows and refills all lie inside the chunk
    // run without per-row bounds checks; the last one or two steps check.
    int t = t0;
    auto rows = [&](auto checked_tag) {
        constexpr bool kChecked = decltype(checked_tag)::value;
        if constexpr (kNorm) {
            // The step's P activations first, then their P head reductions
            // side by side, then the stores.
            float y[P][VEC];
#pragma unroll
            for (int u = 0; u < P; ++u) {
                float xv[VEC];
                widen<VEC, kDtype>(q[u], xv);
                if (!kChecked || t + P + u < t1) load_row<W>(xnext + (int64_t)u * xs, q[u]);
                row_taps(xv, y[u]);
                if constexpr (kSilu) silu_row<VEC>(y[u]);
            }
            if (norm_on) {
                if (p.norm_lanes == 32)  // a 128-channel head: one warp's row
                    l2norm_rows_warp<P, VEC>(y, p.norm_eps, lane);
                else
                    l2norm_rows<P, VEC>(y, p.norm_eps, p.norm_lanes, norm_group);
            }
#pragma unroll
            for (int u = 0; u < P; ++u) {
                if (!kChecked || t + u < t1)
                    store_out_row<VEC, kDtype>(static_cast<OT *>(p.out) + o + u * out_row, y[u]);
            }
        } else {
            if constexpr (kShort && !kPreact && kDtype != KDA_DTYPE_F32 && KDA_SHORT_PREFETCH > 0) {
                // Lane u < P: row t+P+D+u (D = KDA_SHORT_PREFETCH), the warp's
                // whole row segment, while inside the chunk.
                if (lane < P && t + (int64_t)(P + KDA_SHORT_PREFETCH) + lane < t1) {
                    const int seg = min(32 * VEC, p.dim - (c - lane * VEC));
                    l2_prefetch(xnext - lane * VEC + (int64_t)(KDA_SHORT_PREFETCH + lane) * xs,
                                (uint32_t)(seg * (int)sizeof(XT)));
                }
            }
#pragma unroll
            for (int u = 0; u < P; ++u) {
                float xv[VEC];
                widen<VEC, kDtype>(q[u], xv);
                if (!kChecked || t + P + u < t1) load_row<W>(xnext + (int64_t)u * xs, q[u]);
                float y[VEC];
                row_taps(xv, y);
                if constexpr (kSilu) silu_row<VEC>(y);
                if (!kChecked || t + u < t1) {
                    OT *dst = static_cast<OT *>(p.out) + o + u * out_row;
                    if constexpr (kPreact)
                        store_f32_row<VEC>(dst, y);
                    else
                        store_out_row<VEC, kDtype>(dst, y);
                }
            }
        }
        xnext += P * xs;
        o += P * out_row;
    };
    if constexpr (kShort) {
        if (t1 - t0 < P) {
            // Every row of the chunk is in the queue already: compute those
            // rows only (the checked step below computes all P).
            const int n = t1 - t0;
#pragma unroll
            for (int u = 0; u < P; ++u) {
                if (u >= n) break;
                float xv[VEC];
                widen<VEC, kDtype>(q[u], xv);
                float y[VEC];
                row_taps(xv, y);
                if constexpr (kSilu) silu_row<VEC>(y);
                if constexpr (kNorm) {
                    if (norm_on) l2norm_row<VEC>(y, p.norm_eps, p.norm_lanes, norm_group);
                }
                OT *dst = static_cast<OT *>(p.out) + o + u * out_row;
                if constexpr (kPreact)
                    store_f32_row<VEC>(dst, y);
                else
                    store_out_row<VEC, kDtype>(dst, y);
            }
            if (defer) {
                float ns[3][VEC];
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    ns[0][v] = h0[v];
                    ns[1][v] = h1[v];
                    ns[2][v] = h2[v];
                }
                store_state3<VEC>(defer_sp, defer_bf16, ns);
            }
            return;
        }
    }
    for (; t + 2 * P <= t1; t += P) rows(std::false_type{});
    for (; t < t1; t += P) rows(std::true_type{});
}

// Launched as a programmatic dependent: wait until the preceding grid in the
// stream has completed and its writes are visible (the same order a plain
// launch gives), and let the next grid be scheduled meanwhile.
__device__ __forceinline__ void pdl_prologue() {
#if KDA_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
#endif
}

template <int VEC, int P, int kDtype, bool kGeneral, bool kPreact, bool kSilu, bool kBias,
          bool kShort, bool kNorm>
__global__ void __launch_bounds__(KDA_CTA_THREADS, (min_blocks<kDtype, kNorm>()))
    kda_packed_conv1d_kernel(const Params p) {
    pdl_prologue();
    conv_block<VEC, P, kDtype, kGeneral, kPreact, kSilu, kBias, kShort, kNorm>(p, blockIdx.x);
}

// Batches of at most one token per sequence (decode steps): one wave of
// resident blocks, each looping over the blocks of the program map in
// round-robin order.  A warp starts its next one-token program as soon as it
// finishes, with no block launch or retirement in between (GB300, 1024
// one-token sequences: 29.9 -> 27.4 us).  A separate instantiation: compiled
// into the short kernel itself, the loop made its row path spill 12-16 bytes
// and cost 4 % on 1024 x 4 tokens; and for batches that mix 1-row and 48-row
// programs a round-robin assignment cannot balance the load as the block
// scheduler does (256 short prefills + 1024 decode tokens 78.9 -> 104.4 us).
// For 16-bit x without the norm it runs 8 blocks per SM, its programs of
// several rows (rare in such batches) taking a 3-row queue (P): against 7
// blocks and 6 rows, 1024 one-token sequences 27.3 -> 26.9 us, 4096 96.9 ->
// 94.4 us, 256 10.4 -> 9.3 us.
template <int kDtype, bool kNorm>
__host__ __device__ constexpr bool loop_lean() {
    return !kNorm && kDtype != KDA_DTYPE_F32;
}
template <int kDtype, bool kNorm>
__host__ __device__ constexpr int loop_blocks() {
    return loop_lean<kDtype, kNorm>() ? KDA_LOOP_MIN_BLOCKS : min_blocks<kDtype, kNorm>();
}
template <int VEC, int P, int kDtype, bool kSilu, bool kBias, bool kNorm>
__global__ void __launch_bounds__(KDA_CTA_THREADS, (loop_blocks<kDtype, kNorm>()))
    kda_packed_conv1d_loop_kernel(const Params p) {
    pdl_prologue();
    for (unsigned b = blockIdx.x; b < p.map_ctas; b += gridDim.x)
        conv_block<VEC, P, kDtype, false, false, kSilu, kBias, true, kNorm>(p, b);
}

// The epilogue alone, over consecutive fp32 bit patterns, VEC at a time
// through the same row functions as the conv kernel (bf16 output).
// kMode 0: rounding only; 1: SiLU, then rounding.
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
            store_out_row<VEC, KDA_DTYPE_BF16>(out + i, y);
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
// The decode-shaped update: token i is the next row of the sequence whose conv
// state is line cache_indices[i].  One thread per (token, channel vector): read
// the line's 3 newest rows, one row of x, write one output row and the line
// shifted by one row.  No program search: the grid is tokens x vectors.
// ---------------------------------------------------------------------------

// kLayout: 0 dense weight and dense fp32 state; 1 dense weight and dense bf16
// state; 2 any strides, width and state type (the element path); 3 a
// position-major fp32 state with a channel- or tap-major weight; 4 a bf16
// state, dense or position-major, with a channel- or tap-major weight; 5 a
// dense fp32 state with a tap-major weight.  3, 4 and 5 move every access as
// a vector (the flags weight_tapvec / state_posvec).  3 and 5 are separate
// instantiations because one holding both state branches spilled at the
// 64-register cap (24 bytes stored, 36 loaded per item).
//
// One (token, channel vector) of the decode update: the kernel below runs it
// once per thread (kLayout 0, 2) or over a grid-stride loop (kLayout 1, 3, 4).
// The taps and bias of channels c .. c+VEC-1.
template <int VEC, int kLayout, bool kBias>
__device__ __forceinline__ void update_weights(const Params &p, int c, float (&w)[VEC][4],
                                               float (&bias)[VEC]) {
    if (kLayout < 2 || (kLayout != 5 && p.weight_dense)) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const float4 q = __ldg(reinterpret_cast<const float4 *>(p.weight) + (c + v));
            w[v][0] = q.x;
            w[v][1] = q.y;
            w[v][2] = q.z;
            w[v][3] = q.w;
        }
    } else if (kLayout >= 3) {
        // tap-major: tap j of channels c .. c+3 is one float4
        const int64_t wb = weight_base(p, c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int i = 0; i < VEC / 4; ++i) {
                const float4 q = __ldg(reinterpret_cast<const float4 *>(
                    p.weight + wb + (int64_t)j * p.w_stride_j + 4 * i));
                w[4 * i][j] = q.x;
                w[4 * i + 1][j] = q.y;
                w[4 * i + 2][j] = q.z;
                w[4 * i + 3][j] = q.w;
            }
        }
    } else {
        const int64_t wb = weight_base(p, c);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[v][j] = __ldg(p.weight + wb + v * p.w_stride_c + j * p.w_stride_j);
        }
    }
#pragma unroll
    for (int i = 0; i < VEC / 4; ++i) {
        float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (kBias) q = __ldg(reinterpret_cast<const float4 *>(p.bias + c) + i);
        bias[4 * i] = q.x;
        bias[4 * i + 1] = q.y;
        bias[4 * i + 2] = q.z;
        bias[4 * i + 3] = q.w;
    }
}

// Token `token` of channels c .. c+VEC-1, given their taps and bias.
template <int VEC, int kDtype, int kLayout, bool kSilu, bool kBias, bool kNorm>
__device__ __forceinline__ void update_token(const Params &p, int64_t token, int c,
                                             const float (&w)[VEC][4], const float (&bias)[VEC]) {
    constexpr int W = row_words<VEC, kDtype>();
    using XT = typename std::conditional<kDtype == KDA_DTYPE_F32, float, uint16_t>::type;
    uint32_t raw[W];
    load_row<W>(static_cast<const XT *>(p.x) + token * p.x_row_stride + c, raw);
    float xv[VEC];
    widen<VEC, kDtype>(raw, xv);

    const int64_t line = __ldg(p.cache_indices + token * p.ci_stride);
    const bool live = line != p.null_block_id;
    float h0[VEC], h1[VEC], h2[VEC];
    if (kLayout < 2 || kLayout == 5 || (kLayout != 3 && p.state_dense)) {
        const bool bf16 = kLayout == 1 || kLayout == 4 || (kLayout == 2 && p.state_bf16);
        void *sp = state_line_ptr(p, line, c, bf16);
        float st[3 * VEC];
#pragma unroll
        for (int i = 0; i < 3 * VEC; ++i) st[i] = 0.0f;
        if (live) load_state3<VEC>(sp, bf16, st);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            h0[v] = st[3 * v];
            h1[v] = st[3 * v + 1];
            h2[v] = st[3 * v + 2];
        }
        if (live) {
            // new line: (h1, h2, x) per channel
            float ns[3][VEC];
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                ns[0][v] = h1[v];
                ns[1][v] = h2[v];
                ns[2][v] = xv[v];
            }
            store_state3<VEC>(sp, bf16, ns);
        }
    } else if (kLayout == 3 || kLayout == 4) {
        // Position-major: position k of channels c .. c+3 is one vector at
        // base + k * s2.  Read positions K-3 .. K-1; then move positions
        // 1 .. K-1 down by one (K-3 of them from registers) and write x at K-1.
        static_assert(VEC == 4, "one vector per position");
        constexpr bool bf16 = kLayout == 4;
        const int K = p.state_width;
        const int64_t s2 = p.s_stride[2];
        const int64_t base = line * p.s_stride[0] + c;
#pragma unroll
        for (int v = 0; v < VEC; ++v) h0[v] = h1[v] = h2[v] = 0.0f;
        if (live) {
            state_get4(p, base + (int64_t)(K - 3) * s2, bf16, h0);
            state_get4(p, base + (int64_t)(K - 2) * s2, bf16, h1);
            state_get4(p, base + (int64_t)(K - 1) * s2, bf16, h2);
            // positions 0 .. K-5 take positions 1 .. K-4 in ascending order
            // (each read before it is overwritten); none for K <= 4
#pragma unroll 1
            for (int k = 0; k + 4 < K; ++k) {
                float v4[4];
                state_get4(p, base + (int64_t)(k + 1) * s2, bf16, v4);
                state_set4(p, base + (int64_t)k * s2, bf16, v4);
            }
            if (K > 3) state_set4(p, base + (int64_t)(K - 4) * s2, bf16, h0);
            state_set4(p, base + (int64_t)(K - 3) * s2, bf16, h1);
            state_set4(p, base + (int64_t)(K - 2) * s2, bf16, h2);
            state_set4(p, base + (int64_t)(K - 1) * s2, bf16, xv);
        }
    } else {
        const int K = p.state_width;
        const int64_t s1 = p.s_stride[1], s2 = p.s_stride[2];
        const int64_t base = line * p.s_stride[0] + (int64_t)c * s1;
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            h0[v] = live ? state_get(p, base + v * s1 + (K - 3) * s2) : 0.0f;
            h1[v] = live ? state_get(p, base + v * s1 + (K - 2) * s2) : 0.0f;
            h2[v] = live ? state_get(p, base + v * s1 + (K - 1) * s2) : 0.0f;
        }
        if (live) {
            // shift by one row (ascending: position kk + 1 is read before it is
            // overwritten), then the new row at position K-1
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                for (int kk = 0; kk + 1 < K; ++kk)
                    state_set(p, base + v * s1 + (int64_t)kk * s2,
                              state_get(p, base + v * s1 + (int64_t)(kk + 1) * s2));
                state_set(p, base + v * s1 + (int64_t)(K - 1) * s2, xv[v]);
            }
        }
    }

    float y[VEC];
    taps_row<VEC, kBias>(w, bias, h0, h1, h2, xv, y);  // the history is not used after
    if constexpr (kSilu) silu_row<VEC>(y);
    const int plane = (int)fast_div((uint32_t)c, p.part_div);
    if constexpr (kNorm) {
        // A head group is `norm_lanes` consecutive threads of one token (dim is
        // a multiple of head_dim), so the group exits or stays together above.
        if ((p.norm_mask >> plane) & 1u)
            l2norm_row<VEC>(y, p.norm_eps, p.norm_lanes,
                            head_group_mask(threadIdx.x & 31, p.norm_lanes));
    }
    const int col = c - plane * p.part_dim;
    store_out_row<VEC, kDtype>(
        static_cast<XT *>(p.out) + (int64_t)plane * p.plane_stride + token * p.part_dim + col, y);
}

// One (token, channel vector) item, gid = token * (dim / VEC) + vector.
template <int VEC, int kDtype, int kLayout, bool kSilu, bool kBias, bool kNorm>
__device__ __forceinline__ void update_item(const Params &p, int64_t gid) {
    const int64_t nvec = p.dim / VEC;
    const int64_t token = fast_div((uint32_t)gid, p.nvec_div);  // items < 2^32
    if (token >= p.tokens) return;
    const int c = (int)(gid - token * nvec) * VEC;
    float w[VEC][4], bias[VEC];
    update_weights<VEC, kLayout, kBias>(p, c, w, bias);
    update_token<VEC, kDtype, kLayout, kSilu, kBias, kNorm>(p, token, c, w, bias);
}

// The layouts whose kernel keeps a channel vector per thread and loops over
// the tokens on a 2-D grid (the others take one item per thread, or a flat
// grid looping over the items).
__host__ __device__ constexpr bool token_loop_layout(int layout, bool norm) {
    return layout == 1 || layout == 5 || (!norm && (layout == 3 || layout == 4));
}

template <int VEC, int kDtype, int kLayout, bool kSilu, bool kBias, bool kNorm>
__global__ void __launch_bounds__(256, kLayout == 2 ? 2 : 4)
    kda_conv1d_update_kernel(const Params p) {
#if KDA_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
#endif
    constexpr bool kTokenLoop = token_loop_layout(kLayout, kNorm);
    if constexpr (kTokenLoop) {
        // A grid of about (resident CTAs per SM) x SMs whose threads keep one
        // channel vector (blockIdx.x, threadIdx.x) and loop over the tokens
        // (blockIdx.y, step gridDim.y): the taps and bias are loaded once per
        // thread.  GB300, 1024 x 4608, against a grid-stride loop over the
        // items that reloads them: bf16 dense state 16.3 -> 15.8 us (17.0 ->
        // 16.7 us with the norm), bf16 position-major 19.1 -> 18.7 us, a dense
        // fp32 state with a tap-major weight 24.4 -> 23.7 us (24.1 -> 23.6 us
        // with the norm); the fp32 position-major state with a channel-major
        // weight 25.0 -> 25.3 us.
        const int v = blockIdx.x * blockDim.x + threadIdx.x;
        if (v >= p.dim / VEC) return;
        const int c = v * VEC;
        float w[VEC][4], bias[VEC];
        update_weights<VEC, kLayout, kBias>(p, c, w, bias);
        for (int64_t token = blockIdx.y; token < p.tokens; token += gridDim.y)
            update_token<VEC, kDtype, kLayout, kSilu, kBias, kNorm>(p, token, c, w, bias);
    } else if constexpr (kLayout == 1 || kLayout >= 3) {
        // With the L2 norm the taps held across the loop made the
        // position-major variants spill or slow down (fp32: 25.8 -> 27.3 us),
        // so these keep a grid of (resident CTAs per SM) x SMs looping over
        // the items.  Lanes advance together, so head groups stay whole.
        const int64_t total = (int64_t)p.tokens * (p.dim / VEC);
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride)
            update_item<VEC, kDtype, kLayout, kSilu, kBias, kNorm>(p, g);
    } else {
        const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        update_item<VEC, kDtype, kLayout, kSilu, kBias, kNorm>(p, gid);
    }
}

// ---------------------------------------------------------------------------
// Metadata checks on the device (kda_validate_metadata_device)
// ---------------------------------------------------------------------------

// Pass 1 over the sequences: offsets that go backwards, a negative first or a
// too-large last offset (res[0] = the smallest offending index, as the host
// check reports it), cache indices outside [0, lines) (res[1]), and for every
// live line the first sequence that uses it (claim[line] = the smallest s).
// claim and res start at 0xFFFFFFFF.
__global__ void __launch_bounds__(256) kda_validate_claim_kernel(
    const int32_t *qsl, const int32_t *ci, int64_t ci_stride, int num_seqs, int64_t tokens,
    int64_t lines, int64_t null_block_id, uint32_t *claim, uint32_t *res) {
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < num_seqs; s += step) {
        const int q0 = qsl[s], q1 = qsl[s + 1];
        if (s == 0 && q0 < 0) atomicMin(&res[0], 0u);
        if (q1 < q0) atomicMin(&res[0], (uint32_t)s);
        if (s == num_seqs - 1 && (int64_t)q1 > tokens) atomicMin(&res[0], (uint32_t)num_seqs);
        const int64_t line = ci[s * ci_stride];
        if (line == null_block_id) continue;
        if (line < 0 || line >= lines)
            atomicMin(&res[1], (uint32_t)s);
        else
            atomicMin(&claim[line], (uint32_t)s);
    }
}

// Pass 2: a live sequence whose line an earlier sequence claimed is a duplicate.
__global__ void __launch_bounds__(256) kda_validate_dup_kernel(
    const int32_t *ci, int64_t ci_stride, int num_seqs, int64_t lines, int64_t null_block_id,
    const uint32_t *claim, uint32_t *res) {
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < num_seqs; s += step) {
        const int64_t line = ci[s * ci_stride];
        if (line == null_block_id || line < 0 || line >= lines) continue;
        if (claim[line] < (uint32_t)s) atomicMin(&res[1], (uint32_t)s);
    }
}

// Scratch for kda_validate_metadata_device_noalloc: the claim array of up to
// kNoAllocLines cache lines, then the two result words.  Every GPU that loads
// the library holds it (1 MiB) until the process exits; every call of that
// entry point shares it.
constexpr int64_t kNoAllocLines = int64_t(1) << 18;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocLines + 64];

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

thread_local char g_last_error[256] = "";
thread_local cudaError_t g_launch_status = cudaSuccess;  // of the last cudaLaunchKernelEx

constexpr int kVec = KDA_VEC;                 // channels per thread
constexpr int kQueue = KDA_QUEUE;             // rows in flight per thread
constexpr int kThreads = KDA_CTA_THREADS;
constexpr int kDefaultSms = 152;              // GB300, for shape queries without a device
constexpr int kMinChunk = 2 * KDA_QUEUE;
constexpr int kMaxChunk = 2048;
// Mean sequence length below which the kShort instantiation is launched.
// Measured on GB300 (1024-sequence batches): one-token sequences mixed with
// longer ones gain 3-5 % at 16, a batch of uniform 12-token sequences loses
// 1.7 %, and long sequences keep the plain instantiation.
constexpr int kShortMean = 16;

bool aligned(const void *ptr, uintptr_t bytes) {
    return (reinterpret_cast<uintptr_t>(ptr) & (bytes - 1)) == 0;
}

// The layout a NULL layout pointer stands for: bf16, width 3, contiguous.
kda_conv_layout_t default_layout(int64_t dim) {
    kda_conv_layout_t l;
    l.x_dtype = KDA_DTYPE_BF16;
    l.state_width = 3;
    l.state_stride[0] = 3 * dim;
    l.state_stride[1] = 3;
    l.state_stride[2] = 1;
    l.weight_stride[0] = 4;
    l.weight_stride[1] = 1;
    l.state_dtype = KDA_DTYPE_F32;
    l.version = 0;
    l.weight_part_stride = 0;
    l.cache_index_stride = 0;
    return l;
}

// The caller's layout (NULL: the default).  A version-0 struct may be the
// shorter struct of earlier releases, so the version-1 fields are read only
// when the caller says they are there.
kda_conv_layout_t read_layout(const kda_conv_layout_t *in, int64_t dim) {
    if (!in) return default_layout(dim);
    kda_conv_layout_t l;
    memcpy(&l, in, offsetof(kda_conv_layout_t, weight_part_stride));
    l.weight_part_stride = 0;
    l.cache_index_stride = 0;
    if (l.version == 1) {
        l.weight_part_stride = in->weight_part_stride;
        l.cache_index_stride = in->cache_index_stride;
    }
    return l;
}

// Element stride between weight parts: the layout's, or that of one (dim, 4) array.
int64_t weight_part_stride(const kda_conv_layout_t &l, int64_t part_dim) {
    return l.weight_part_stride != 0 ? l.weight_part_stride : part_dim * l.weight_stride[0];
}

kda_status_t check_sizes(int64_t x_row_stride, int64_t tokens, int64_t dim, int64_t part_dim,
                         int64_t num_seqs) {
    if (tokens < 0 || dim < 0 || num_seqs < 0 || part_dim <= 0) return KDA_ERR_INVALID_ARG;
    if (tokens > INT32_MAX || dim > INT32_MAX / 4 || num_seqs > (int64_t(1) << 30))
        return KDA_ERR_INVALID_ARG;
    if (x_row_stride < dim) return KDA_ERR_INVALID_ARG;
    if (part_dim % 64 != 0 || dim % part_dim != 0) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// Width 3 and strides (3 * dim, 3, 1), whatever the state's storage type.
bool state_is_dense(const kda_conv_layout_t &l, int64_t dim) {
    return l.state_width == 3 && l.state_stride[0] == 3 * dim && l.state_stride[1] == 3 &&
           l.state_stride[2] == 1;
}

// Position-major state whose four-channel groups are aligned vectors.
bool state_is_posvec(const kda_conv_layout_t &l, const void *conv_states) {
    const uintptr_t vec_bytes = l.state_dtype == KDA_DTYPE_BF16 ? 8 : 16;
    return l.state_stride[1] == 1 && l.state_stride[0] % 4 == 0 && l.state_stride[2] % 4 == 0 &&
           aligned(conv_states, vec_bytes);
}

// Tap-major weight whose four-channel groups of a tap are aligned float4s
// (also a [part, tap, channel] weight with such strides).
bool weight_is_tapvec(const kda_conv_layout_t &l, const float *weight, int64_t part_dim) {
    return l.weight_stride[0] == 1 && l.weight_stride[1] % 4 == 0 &&
           weight_part_stride(l, part_dim) % 4 == 0 && aligned(weight, 16);
}

// One (dim, 4) contiguous array: one float4 per channel.
bool weight_is_dense(const kda_conv_layout_t &l, int64_t part_dim) {
    return l.weight_stride[0] == 4 && l.weight_stride[1] == 1 &&
           weight_part_stride(l, part_dim) == 4 * part_dim;
}

kda_status_t check_args(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                        int64_t part_dim, const float *weight, const float *bias,
                        const void *conv_states, const int32_t *cache_indices,
                        const uint8_t *has_initial_state, const int32_t *query_start_loc,
                        int64_t num_seqs, int activation, const void *out,
                        const kda_conv_layout_t &l, bool need_ranges = true) {
    kda_status_t st = check_sizes(x_row_stride, tokens, dim, part_dim, num_seqs);
    if (st != KDA_OK) return st;
    if (activation != KDA_ACT_NONE && activation != KDA_ACT_SILU) return KDA_ERR_INVALID_ARG;
    if (l.x_dtype != KDA_DTYPE_BF16 && l.x_dtype != KDA_DTYPE_F16 && l.x_dtype != KDA_DTYPE_F32)
        return KDA_ERR_INVALID_ARG;
    if ((l.state_dtype != KDA_DTYPE_F32 && l.state_dtype != KDA_DTYPE_BF16) ||
        (l.version != 0 && l.version != 1) || l.cache_index_stride < 0)
        return KDA_ERR_INVALID_ARG;
    if (l.state_width < 3) return KDA_ERR_INVALID_ARG;
    if (l.state_width > kMaxStateWidth) return KDA_ERR_UNSUPPORTED;
    if (tokens == 0 || num_seqs == 0 || dim == 0) return KDA_OK;  // nothing is touched
    if (!x || !weight || !conv_states || !cache_indices || !out) return KDA_ERR_INVALID_ARG;
    if (need_ranges && (!has_initial_state || !query_start_loc)) return KDA_ERR_INVALID_ARG;
    // rows of x must start on 16-byte boundaries: 8 elements of 2 bytes, 4 of 4
    const int64_t row_quantum = l.x_dtype == KDA_DTYPE_F32 ? 4 : 8;
    if (!aligned(x, 16) || x_row_stride % row_quantum != 0 || !aligned(out, 16) ||
        (bias && !aligned(bias, 16)))
        return KDA_ERR_MISALIGNED;
    if (weight_is_dense(l, part_dim) ? !aligned(weight, 16) : !aligned(weight, 4))
        return KDA_ERR_MISALIGNED;
    const uintptr_t state_elem = l.state_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    if (!aligned(conv_states, state_is_dense(l, dim) ? 16 : state_elem)) return KDA_ERR_MISALIGNED;
    return KDA_OK;
}

struct Shape {
    int64_t ctas;
    int threads;
    int chunk;
    int64_t programs;
    int warps_per_prog;
    int64_t total_warps;
    bool short_seqs;  // mean sequence length below kShortMean: the kShort kernel
};

// Chunk length (rows per program), rounded up to a multiple of the queue
// depth and clamped to [kMinChunk, kMaxChunk].  The resident-warp budget
// (slots) is waves x SMs x warps per SM.
//   * One sequence: the smallest chunk for which every program fits in the
//     budget at once, so no CTA waits for a later wave.
//   * num_seqs at or above the budget's program count: the even spread of the
//     tokens over the budget, no less than kSpreadFloor rows.
//   * In between: the one-wave fit, but at most the even spread over two
//     waves (no less than kSpreadFloor rows).  The one-wave fit alone gives
//     tokens / (budget - num_seqs) rows, which grows without bound as num_seqs
//     nears the budget: one long prompt among ~100 short ones then streamed
//     through a few latency-bound warps (GB300, 16K tokens: one 8192-token
//     prompt among 99 of 80 tokens took 152 us with 900-row chunks and 58 us
//     with 72-row ones; batches of uniform sequences keep their time).
// It depends only on the scalar sizes and the SM count, so a captured launch
// stays valid for new metadata.
constexpr int64_t kSpreadFloor = 48;

Shape launch_shape(int64_t tokens, int64_t dim, int64_t num_seqs, int sms,
                   int blocks_per_sm = KDA_MIN_BLOCKS) {
    Shape sh{};
    sh.threads = kThreads;
    const int64_t nvec = dim / kVec;
    sh.warps_per_prog = (int)((nvec + 31) / 32);
    const int64_t slots = (int64_t)KDA_WAVES * sms * (kThreads / 32) * blocks_per_sm;
    const int64_t max_programs = slots / sh.warps_per_prog;
    int64_t chunk;
    if (max_programs > num_seqs) {
        chunk = (tokens + (max_programs - num_seqs) - 1) / (max_programs - num_seqs);
        if (num_seqs > 1) {
            int64_t spread2 = (tokens * sh.warps_per_prog + 2 * slots - 1) / (2 * slots);
            if (spread2 < kSpreadFloor) spread2 = kSpreadFloor;
            if (chunk > spread2) chunk = spread2;
        }
    } else {
        chunk = (tokens * sh.warps_per_prog + slots - 1) / slots;
        // no less than kSpreadFloor rows: fewer idle programs and a narrower
        // search window for decode-sized batches (GB300: 1024 one-token
        // sequences 29.7 -> 29.5 us, 1024 x 4 tokens 37.6 -> 37.3 us)
        if (chunk < kSpreadFloor) chunk = kSpreadFloor;
    }
    chunk = (chunk + kQueue - 1) / kQueue * kQueue;
    if (chunk < kMinChunk) chunk = kMinChunk;
    if (chunk > kMaxChunk) chunk = kMaxChunk;
    sh.chunk = (int)chunk;
    sh.programs = (tokens + sh.chunk - 1) / sh.chunk + num_seqs;
    sh.total_warps = sh.programs * sh.warps_per_prog;
    sh.short_seqs = tokens < (int64_t)kShortMean * num_seqs;
    const int64_t warps_per_cta = kThreads / 32;
    sh.ctas = (sh.total_warps + warps_per_cta - 1) / warps_per_cta;
    return sh;
}

// SM count of the current device, cached per device (host threads may race to
// fill an entry; they store the same value).
int current_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kDefaultSms;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = kDefaultSms;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Launches a conv kernel.  With KDA_PDL the launch carries the programmatic
// stream serialization attribute: the grid may be scheduled while the
// preceding kernel in the stream drains (when that kernel signals
// griddepcontrol.launch_dependents, as these kernels do), and the kernel's
// first instruction, griddepcontrol.wait, holds every thread until that
// kernel has completed and its writes are visible.  Stream order is exactly
// that of a plain launch; what overlaps is the launch and the block
// scheduling, not any memory access.  After any other kind of predecessor
// the launch behaves as a plain one.
void launch_kernel(void (*kernel)(Params), dim3 blocks, unsigned threads, const Params &p,
                   cudaStream_t stream) {
#if KDA_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = blocks;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    g_launch_status = cudaLaunchKernelEx(&cfg, kernel, p);
#else
    kernel<<<blocks, threads, 0, stream>>>(p);
#endif
}

template <int kDtype, bool kGeneral, bool kPreact, bool kSilu, bool kBias, bool kNorm>
void launch_norm(const Params &p, const Shape &sh, cudaStream_t stream) {
    if (sh.short_seqs) {
        if constexpr (!kGeneral && !kPreact) {
            if (p.tokens <= p.num_seqs) {  // at most one token per sequence on average
                const int64_t resident = (int64_t)current_sms() * loop_blocks<kDtype, kNorm>();
                constexpr int kLoopP = loop_lean<kDtype, kNorm>() ? KDA_LOOP_QUEUE : kQueue;
                launch_kernel(kda_packed_conv1d_loop_kernel<kVec, kLoopP, kDtype, kSilu, kBias, kNorm>,
                              dim3((unsigned)std::min(sh.ctas, resident)), (unsigned)sh.threads, p,
                              stream);
                return;
            }
        }
        launch_kernel(kda_packed_conv1d_kernel<kVec, kQueue, kDtype, kGeneral, kPreact, kSilu,
                                               kBias, true, kNorm>,
                      dim3((unsigned)sh.ctas), (unsigned)sh.threads, p, stream);
    } else {
        launch_kernel(kda_packed_conv1d_kernel<kVec, kQueue, kDtype, kGeneral, kPreact, kSilu,
                                               kBias, false, kNorm>,
                      dim3((unsigned)sh.ctas), (unsigned)sh.threads, p, stream);
    }
}

template <int kDtype, bool kGeneral, bool kPreact, bool kSilu, bool kBias>
void launch(const Params &p, const Shape &sh, cudaStream_t stream) {
    if constexpr (!kPreact) {
        if (p.norm_mask != 0u) {
            launch_norm<kDtype, kGeneral, kPreact, kSilu, kBias, true>(p, sh, stream);
            return;
        }
    }
    launch_norm<kDtype, kGeneral, kPreact, kSilu, kBias, false>(p, sh, stream);
}

template <int kDtype, bool kGeneral>
void dispatch_act(const Params &p, const Shape &sh, bool silu, cudaStream_t s) {
    if (silu) {
        if (p.bias)
            launch<kDtype, kGeneral, false, true, true>(p, sh, s);
        else
            launch<kDtype, kGeneral, false, true, false>(p, sh, s);
    } else {
        if (p.bias)
            launch<kDtype, kGeneral, false, false, true>(p, sh, s);
        else
            launch<kDtype, kGeneral, false, false, false>(p, sh, s);
    }
}

template <int kDtype>
void dispatch(const Params &p, const Shape &sh, bool silu, cudaStream_t s) {
    if (p.weight_dense && p.state_dense && !p.state_bf16)
        dispatch_act<kDtype, false>(p, sh, silu, s);
    else
        dispatch_act<kDtype, true>(p, sh, silu, s);
}

// KDA_ERR_CUDA with CUDA's text for `err` (a failed runtime call).
kda_status_t cuda_failure(cudaError_t err) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
             cudaGetErrorString(err));
    return KDA_ERR_CUDA;
}

kda_status_t record_cuda_error() {
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) err = g_launch_status;
    g_launch_status = cudaSuccess;
    if (err != cudaSuccess) {
        snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(err),
                 cudaGetErrorString(err));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

// The L2-norm options: NULL or an empty mask is no norm.  A head is head_dim
// channels, head_dim / kVec lanes: a power of two up to a warp, dividing
// part_dim so that heads never straddle planes.
kda_status_t check_norm(const kda_l2norm_t *norm, int64_t dim, int64_t part_dim) {
    if (!norm || norm->plane_mask == 0u) return KDA_OK;
    if (norm->reserved != 0) return KDA_ERR_INVALID_ARG;
    if (!(norm->eps >= 0.0f) || norm->eps > 3.0e38f) return KDA_ERR_INVALID_ARG;  // NaN too
    // A subnormal eps would be flushed by the SFU root (rsqrt.approx.ftz) and
    // leave a head of tiny activations inf or NaN: 0 or a normal number only.
    if (norm->eps > 0.0f && norm->eps < FLT_MIN) return KDA_ERR_INVALID_ARG;
    const int64_t planes = dim / part_dim;
    if (planes < 32 && (norm->plane_mask >> planes) != 0u) return KDA_ERR_INVALID_ARG;
    const int64_t hd = norm->head_dim;
    if (hd < kVec || hd % kVec != 0) return KDA_ERR_UNSUPPORTED;
    const int64_t lanes = hd / kVec;
    if (lanes > 32 || (lanes & (lanes - 1)) != 0) return KDA_ERR_UNSUPPORTED;
    if (part_dim % hd != 0) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

void set_norm(Params &p, const kda_l2norm_t *norm) {
    const bool on = norm && norm->plane_mask != 0u;
    p.norm_mask = on ? norm->plane_mask : 0u;
    p.norm_lanes = on ? norm->head_dim / kVec : 1;
    p.norm_eps = on ? norm->eps : 0.0f;
}

kda_status_t run(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                 int64_t part_dim, const float *weight, const float *bias, void *conv_states,
                 const int32_t *cache_indices, const uint8_t *has_initial_state,
                 const int32_t *query_start_loc, int64_t num_seqs, int64_t null_block_id,
                 int activation, void *out, bool preact, const kda_conv_layout_t *layout,
                 const kda_l2norm_t *norm, kda_stream_t stream) {
    const kda_conv_layout_t l = read_layout(layout, dim);
    kda_status_t st = check_args(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
                                 cache_indices, has_initial_state, query_start_loc, num_seqs,
                                 activation, out, l);
    if (st != KDA_OK) return st;
    if (part_dim > 0 && (st = check_norm(norm, dim, part_dim)) != KDA_OK) return st;
    if (tokens == 0 || num_seqs == 0 || dim == 0) return KDA_OK;

    const bool norm_on = !preact && norm && norm->plane_mask != 0u;
    const int blocks_per_sm = l.x_dtype == KDA_DTYPE_F32
                                  ? (norm_on ? min_blocks<KDA_DTYPE_F32, true>()
                                             : min_blocks<KDA_DTYPE_F32>())
                                  : min_blocks<KDA_DTYPE_BF16>();
    const Shape sh = launch_shape(tokens, dim, num_seqs, current_sms(), blocks_per_sm);
    // warp and program indices are divided in 32 bits on the device
    if (sh.ctas > INT32_MAX || sh.total_warps >= (int64_t(1) << 32)) return KDA_ERR_INVALID_ARG;
    Params p;
    p.x = x;
    p.x_row_stride = x_row_stride;
    p.tokens = (int)tokens;
    p.dim = (int)dim;
    p.part_dim = (int)part_dim;
    p.num_seqs = (int)num_seqs;
    p.weight = weight;
    p.w_stride_c = l.weight_stride[0];
    p.w_stride_j = l.weight_stride[1];
    p.w_stride_part = weight_part_stride(l, part_dim);
    p.weight_dense = weight_is_dense(l, part_dim);
    p.bias = bias;
    p.conv_states = conv_states;
    p.state_width = l.state_width;
    for (int i = 0; i < 3; ++i) p.s_stride[i] = l.state_stride[i];
    p.state_dense = state_is_dense(l, dim);
    p.state_bf16 = l.state_dtype == KDA_DTYPE_BF16;
    p.state_posvec = state_is_posvec(l, conv_states);
    p.weight_tapvec = weight_is_tapvec(l, weight, part_dim);
    p.cache_indices = cache_indices;
    p.ci_stride = l.cache_index_stride > 0 ? l.cache_index_stride : 1;
    p.has_initial_state = has_initial_state;
    p.qsl = query_start_loc;
    p.null_block_id = null_block_id;
    p.out = out;
    p.plane_stride = tokens * part_dim;
    p.chunk = sh.chunk;
    p.warps_per_prog = sh.warps_per_prog;
    p.chunk_div = make_fast_div((uint32_t)sh.chunk);
    p.wpp_div = make_fast_div((uint32_t)sh.warps_per_prog);
    p.part_div = make_fast_div((uint32_t)part_dim);
    p.total_warps = sh.total_warps;
    p.map_ctas = (unsigned)sh.ctas;
    int steps = 0;
    int64_t reach = 1;
    while (reach < num_seqs) {
        reach *= 32;
        ++steps;
    }
    p.search_steps = steps;
    p.search_top = steps > 0 ? (int)(reach / 32) : 1;
    // The window search replaces two or more radix levels when its entries
    // (ceil(tokens / chunk) + 2 at most) fit in kWindowRounds rounds.  Measured
    // on GB300: 256 short prefills + 1024 decode tokens 82.8 against 85.1 us,
    // 1024 decode tokens 33.3 against 33.8 us; with 8 rounds it was slower
    // than the radix search, and with one level to replace no faster.
    p.win_span = (int)((tokens + sh.chunk - 1) / sh.chunk);
    const int64_t win_entries = p.win_span + 2;
    p.win_rounds = (num_seqs > 32 && win_entries <= 32 * kWindowRounds)
                       ? (int)((win_entries + 31) / 32)
                       : 0;
    set_norm(p, preact ? nullptr : norm);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (preact) {  // bf16 x and the default layout only
        if (bias)
            launch<KDA_DTYPE_BF16, false, true, false, true>(p, sh, s);
        else
            launch<KDA_DTYPE_BF16, false, true, false, false>(p, sh, s);
    } else if (l.x_dtype == KDA_DTYPE_F16) {
        dispatch<KDA_DTYPE_F16>(p, sh, activation == KDA_ACT_SILU, s);
    } else if (l.x_dtype == KDA_DTYPE_F32) {
        dispatch<KDA_DTYPE_F32>(p, sh, activation == KDA_ACT_SILU, s);
    } else {
        dispatch<KDA_DTYPE_BF16>(p, sh, activation == KDA_ACT_SILU, s);
    }
    return record_cuda_error();
}

// blocks: the grid of the layout's token loop (or one item per thread);
// norm_blocks: the flat grid the norm variant takes where it has no token loop.
template <int kDtype, int kLayout, bool kSilu, bool kBias>
void launch_update(const Params &p, dim3 blocks, dim3 norm_blocks, cudaStream_t stream) {
    if (p.norm_mask != 0u)
        launch_kernel(kda_conv1d_update_kernel<kVec, kDtype, kLayout, kSilu, kBias, true>,
                      token_loop_layout(kLayout, true) ? blocks : norm_blocks, 256, p, stream);
    else
        launch_kernel(kda_conv1d_update_kernel<kVec, kDtype, kLayout, kSilu, kBias, false>, blocks,
                      256, p, stream);
}

template <int kDtype, int kLayout>
void dispatch_update_act(const Params &p, dim3 blocks, dim3 norm_blocks, bool silu,
                         cudaStream_t s) {
    if (silu) {
        if (p.bias)
            launch_update<kDtype, kLayout, true, true>(p, blocks, norm_blocks, s);
        else
            launch_update<kDtype, kLayout, true, false>(p, blocks, norm_blocks, s);
    } else {
        if (p.bias)
            launch_update<kDtype, kLayout, false, true>(p, blocks, norm_blocks, s);
        else
            launch_update<kDtype, kLayout, false, false>(p, blocks, norm_blocks, s);
    }
}

// The decode step moves little besides the state lines, so a dense bf16 state
// has its own lean variant (the general one holds about twice the registers).
// Layouts 1, 3, 4 and 5 run a grid of about 4 CTAs per SM: in the token loop
// blockIdx.x picks 256 channel vectors and blockIdx.y the first token, which
// then steps by gridDim.y; otherwise a flat grid loops over the items.
template <int kDtype>
void dispatch_update(const Params &p, int64_t blocks, bool silu, cudaStream_t s) {
    const int64_t nvec = p.dim / kVec;
    const unsigned gx = (unsigned)((nvec + 255) / 256);
    const int64_t resident = 4 * (int64_t)current_sms();
    const int64_t want_y = resident / gx;
    const unsigned gy = (unsigned)(want_y < 1 ? 1 : (want_y < p.tokens ? want_y : p.tokens));
    const dim3 loop_grid(gx, gy);
    const dim3 flat_loop((unsigned)(blocks < resident ? blocks : resident));
    const dim3 flat((unsigned)blocks);
    if (p.weight_dense && p.state_dense)
        if (p.state_bf16)
            dispatch_update_act<kDtype, 1>(p, loop_grid, flat_loop, silu, s);
        else
            dispatch_update_act<kDtype, 0>(p, flat, flat, silu, s);
    else if ((p.weight_dense || p.weight_tapvec) && (p.state_dense || p.state_posvec))
        if (p.state_bf16)
            dispatch_update_act<kDtype, 4>(p, loop_grid, flat_loop, silu, s);
        else if (p.state_posvec)
            dispatch_update_act<kDtype, 3>(p, loop_grid, flat_loop, silu, s);
        else  // a dense fp32 state: the weight is tap-major (both dense is layout 0)
            dispatch_update_act<kDtype, 5>(p, loop_grid, flat_loop, silu, s);
    else
        dispatch_update_act<kDtype, 2>(p, flat, flat, silu, s);
}

kda_status_t run_update(const void *x, int64_t x_row_stride, int64_t batch, int64_t dim,
                        int64_t part_dim, const float *weight, const float *bias,
                        void *conv_states, const int32_t *cache_indices, int64_t null_block_id,
                        int activation, void *out, const kda_conv_layout_t *layout,
                        const kda_l2norm_t *norm, kda_stream_t stream) {
    const kda_conv_layout_t l = read_layout(layout, dim);
    kda_status_t st = check_args(x, x_row_stride, batch, dim, part_dim, weight, bias, conv_states,
                                 cache_indices, nullptr, nullptr, batch, activation, out, l,
                                 false);
    if (st != KDA_OK) return st;
    if (part_dim > 0 && (st = check_norm(norm, dim, part_dim)) != KDA_OK) return st;
    if (batch == 0 || dim == 0) return KDA_OK;
    const int64_t threads_total = batch * (dim / kVec);
    const int64_t blocks = (threads_total + 255) / 256;
    // item indices are divided in 32 bits on the device
    if (blocks > INT32_MAX || threads_total >= (int64_t(1) << 32)) return KDA_ERR_INVALID_ARG;
    Params p{};
    p.x = x;
    p.x_row_stride = x_row_stride;
    p.tokens = (int)batch;
    p.dim = (int)dim;
    p.part_dim = (int)part_dim;
    p.num_seqs = (int)batch;
    p.weight = weight;
    p.w_stride_c = l.weight_stride[0];
    p.w_stride_j = l.weight_stride[1];
    p.w_stride_part = weight_part_stride(l, part_dim);
    p.weight_dense = weight_is_dense(l, part_dim);
    p.bias = bias;
    p.conv_states = conv_states;
    p.state_width = l.state_width;
    for (int i = 0; i < 3; ++i) p.s_stride[i] = l.state_stride[i];
    p.state_dense = state_is_dense(l, dim);
    p.state_bf16 = l.state_dtype == KDA_DTYPE_BF16;
    p.state_posvec = state_is_posvec(l, conv_states);
    p.weight_tapvec = weight_is_tapvec(l, weight, part_dim);
    p.cache_indices = cache_indices;
    p.ci_stride = l.cache_index_stride > 0 ? l.cache_index_stride : 1;
    p.null_block_id = null_block_id;
    p.out = out;
    p.plane_stride = batch * part_dim;
    p.part_div = make_fast_div((uint32_t)part_dim);
    p.nvec_div = make_fast_div((uint32_t)(dim / kVec));
    set_norm(p, norm);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool silu = activation == KDA_ACT_SILU;
    if (l.x_dtype == KDA_DTYPE_F16)
        dispatch_update<KDA_DTYPE_F16>(p, blocks, silu, s);
    else if (l.x_dtype == KDA_DTYPE_F32)
        dispatch_update<KDA_DTYPE_F32>(p, blocks, silu, s);
    else
        dispatch_update<KDA_DTYPE_BF16>(p, blocks, silu, s);
    return record_cuda_error();
}

// The device checks with caller-provided scratch: claim (lines entries) and
// res (2 entries), both device memory.  Enqueues on `s`, copies the two
// results back and synchronises `s`.
kda_status_t validate_on_device(const int32_t *qsl, const int32_t *ci, int64_t ci_stride,
                                int64_t num_seqs, int64_t tokens, int64_t lines,
                                int64_t null_block_id, uint32_t *claim, uint32_t *res,
                                int64_t *bad, cudaStream_t s) {
    cudaError_t err = cudaMemsetAsync(res, 0xFF, 2 * sizeof(uint32_t), s);
    if (err == cudaSuccess && lines > 0)
        err = cudaMemsetAsync(claim, 0xFF, (size_t)lines * sizeof(uint32_t), s);
    if (err != cudaSuccess) return cuda_failure(err);
    const int threads = 256;
    const int64_t want = (num_seqs + threads - 1) / threads;
    const int blocks = (int)(want < 4 * 152 ? want : 4 * 152);
    kda_validate_claim_kernel<<<blocks, threads, 0, s>>>(qsl, ci, ci_stride, (int)num_seqs, tokens,
                                                         lines, null_block_id, claim, res);
    kda_validate_dup_kernel<<<blocks, threads, 0, s>>>(ci, ci_stride, (int)num_seqs, lines,
                                                       null_block_id, claim, res);
    kda_status_t st = record_cuda_error();
    if (st != KDA_OK) return st;
    uint32_t host_res[2] = {0xFFFFFFFFu, 0xFFFFFFFFu};
    err = cudaMemcpyAsync(host_res, res, sizeof host_res, cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess) err = cudaStreamSynchronize(s);
    if (err != cudaSuccess) return cuda_failure(err);
    if (host_res[0] != 0xFFFFFFFFu) {
        *bad = host_res[0];
        return KDA_ERR_METADATA;
    }
    if (host_res[1] != 0xFFFFFFFFu) {
        *bad = host_res[1];
        return KDA_ERR_METADATA;
    }
    return KDA_OK;
}

// The device address of g_noalloc_scratch on the current device, looked up
// once per device with that device current (in host code the symbol's name
// is a host-side stand-in, not a device address).  Returns nullptr and sets
// *err if the lookup fails.
uint32_t *noalloc_scratch(cudaError_t *err) {
    static std::atomic<uint32_t *> cache[64];
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    uint32_t *ptr = cache[dev].load(std::memory_order_acquire);
    if (ptr == nullptr) {
        void *addr = nullptr;
        *err = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        ptr = static_cast<uint32_t *>(addr);
        cache[dev].store(ptr, std::memory_order_release);  // racing threads store the same value
    }
    return ptr;
}

kda_status_t check_validate_args(const int32_t *qsl, const int32_t *ci, int64_t ci_stride,
                                 int64_t num_seqs, int64_t tokens, int64_t lines) {
    if (num_seqs < 0 || tokens < 0 || lines < 0 || ci_stride < 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs > (int64_t(1) << 30) || lines > (int64_t(1) << 31)) return KDA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!qsl || !ci)) return KDA_ERR_INVALID_ARG;
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
               false, nullptr, nullptr, stream);
}

kda_status_t kda_packed_conv1d_ex(const void *x, int64_t x_row_stride, int64_t tokens,
                                  int64_t dim, int64_t part_dim, const float *weight,
                                  const float *bias, void *conv_states,
                                  const int32_t *cache_indices, const uint8_t *has_initial_state,
                                  const int32_t *query_start_loc, int64_t num_seqs,
                                  int64_t null_block_id, int activation, void *out,
                                  const kda_conv_layout_t *layout, kda_stream_t stream) {
    return run(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states, cache_indices,
               has_initial_state, query_start_loc, num_seqs, null_block_id, activation, out,
               false, layout, nullptr, stream);
}

kda_status_t kda_packed_conv1d_l2norm(const void *x, int64_t x_row_stride, int64_t tokens,
                                      int64_t dim, int64_t part_dim, const float *weight,
                                      const float *bias, void *conv_states,
                                      const int32_t *cache_indices,
                                      const uint8_t *has_initial_state,
                                      const int32_t *query_start_loc, int64_t num_seqs,
                                      int64_t null_block_id, int activation, void *out,
                                      const kda_conv_layout_t *layout, const kda_l2norm_t *norm,
                                      kda_stream_t stream) {
    return run(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states, cache_indices,
               has_initial_state, query_start_loc, num_seqs, null_block_id, activation, out,
               false, layout, norm, stream);
}

kda_status_t kda_conv1d_update(const void *x, int64_t x_row_stride, int64_t batch, int64_t dim,
                              int64_t part_dim, const float *weight, const float *bias,
                              void *conv_states, const int32_t *cache_indices,
                              int64_t null_block_id, int activation, void *out,
                              const kda_conv_layout_t *layout, kda_stream_t stream) {
    return run_update(x, x_row_stride, batch, dim, part_dim, weight, bias, conv_states,
                      cache_indices, null_block_id, activation, out, layout, nullptr, stream);
}

kda_status_t kda_conv1d_update_l2norm(const void *x, int64_t x_row_stride, int64_t batch,
                                      int64_t dim, int64_t part_dim, const float *weight,
                                      const float *bias, void *conv_states,
                                      const int32_t *cache_indices, int64_t null_block_id,
                                      int activation, void *out, const kda_conv_layout_t *layout,
                                      const kda_l2norm_t *norm, kda_stream_t stream) {
    return run_update(x, x_row_stride, batch, dim, part_dim, weight, bias, conv_states,
                      cache_indices, null_block_id, activation, out, layout, norm, stream);
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
               true, nullptr, nullptr, stream);
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
                      out, default_layout(dim));
}

kda_status_t kda_packed_conv1d_ex_check_args(
    const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim, int64_t part_dim,
    const float *weight, const float *bias, const void *conv_states,
    const int32_t *cache_indices, const uint8_t *has_initial_state,
    const int32_t *query_start_loc, int64_t num_seqs, int activation, const void *out,
    const kda_conv_layout_t *layout) {
    return check_args(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
                      cache_indices, has_initial_state, query_start_loc, num_seqs, activation,
                      out, read_layout(layout, dim));
}

kda_status_t kda_l2norm_check(const kda_l2norm_t *norm, int64_t dim, int64_t part_dim) {
    kda_status_t st = check_sizes(dim, 0, dim, part_dim, 0);
    if (st != KDA_OK) return st;
    return check_norm(norm, dim, part_dim);
}

kda_status_t kda_packed_conv1d_launch_shape(int64_t tokens, int64_t dim, int64_t part_dim,
                                            int64_t num_seqs, int32_t sm_count, int64_t *ctas,
                                            int32_t *threads, int32_t *chunk_tokens,
                                            int64_t *programs) {
    kda_status_t st = check_sizes(dim, tokens, dim, part_dim, num_seqs);
    if (st != KDA_OK) return st;
    if (sm_count < 0) return KDA_ERR_INVALID_ARG;
    Shape sh{};
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

kda_status_t kda_validate_metadata_device(const int32_t *query_start_loc,
                                          const int32_t *cache_indices,
                                          int64_t cache_index_stride, int64_t num_seqs,
                                          int64_t tokens, int64_t cache_lines,
                                          int64_t null_block_id, int64_t *bad_seq,
                                          kda_stream_t stream) {
    int64_t dummy;
    int64_t *bad = bad_seq ? bad_seq : &dummy;
    *bad = -1;
    kda_status_t st = check_validate_args(query_start_loc, cache_indices, cache_index_stride,
                                          num_seqs, tokens, cache_lines);
    if (st != KDA_OK || num_seqs == 0) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // scratch: the claim array, then the two result words (256-byte aligned)
    const size_t claim_bytes = ((size_t)cache_lines * sizeof(uint32_t) + 255) / 256 * 256;
    void *scratch = nullptr;
    cudaError_t err = cudaMallocAsync(&scratch, claim_bytes + 256, s);
    if (err != cudaSuccess) return cuda_failure(err);
    uint32_t *claim = static_cast<uint32_t *>(scratch);
    uint32_t *res = reinterpret_cast<uint32_t *>(static_cast<char *>(scratch) + claim_bytes);
    st = validate_on_device(query_start_loc, cache_indices,
                            cache_index_stride > 0 ? cache_index_stride : 1, num_seqs, tokens,
                            cache_lines, null_block_id, claim, res, bad, s);
    err = cudaFreeAsync(scratch, s);
    if (st != KDA_ERR_CUDA && err != cudaSuccess) return cuda_failure(err);
    return st;
}

kda_status_t kda_validate_metadata_device_noalloc(const int32_t *query_start_loc,
                                                  const int32_t *cache_indices,
                                                  int64_t cache_index_stride, int64_t num_seqs,
                                                  int64_t tokens, int64_t cache_lines,
                                                  int64_t null_block_id, int64_t *bad_seq,
                                                  kda_stream_t stream) {
    int64_t dummy;
    int64_t *bad = bad_seq ? bad_seq : &dummy;
    *bad = -1;
    kda_status_t st = check_validate_args(query_start_loc, cache_indices, cache_index_stride,
                                          num_seqs, tokens, cache_lines);
    if (st != KDA_OK || num_seqs == 0) return st;
    if (cache_lines > kNoAllocLines) {
        snprintf(g_last_error, sizeof g_last_error,
                 "cache_lines %lld exceeds the %lld lines of the static scratch",
                 (long long)cache_lines, (long long)kNoAllocLines);
        return KDA_ERR_UNSUPPORTED;
    }
    cudaError_t err = cudaSuccess;
    uint32_t *scratch = noalloc_scratch(&err);
    if (scratch == nullptr) return cuda_failure(err);
    // validate_on_device clears the claim words it uses and the two result
    // words before its kernels run, whatever an earlier call left there.
    return validate_on_device(query_start_loc, cache_indices,
                              cache_index_stride > 0 ? cache_index_stride : 1, num_seqs, tokens,
                              cache_lines, null_block_id, scratch, scratch + kNoAllocLines, bad,
                              static_cast<cudaStream_t>(stream));
}

kda_status_t kda_epilogue_range(uint32_t first, uint64_t count, int activation, uint16_t *out,
                                kda_stream_t stream) {
    if (activation != KDA_ACT_NONE && activation != KDA_ACT_SILU) return KDA_ERR_INVALID_ARG;
    if (count == 0) return KDA_OK;
    if (!out) return KDA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return KDA_ERR_MISALIGNED;
    const uint64_t groups = (count + kVec - 1) / kVec;
    const unsigned threads = 256;
    const uint64_t want = (groups + threads - 1) / threads;
    const unsigned blocks = (unsigned)(want < 152ull * 64 ? want : 152ull * 64);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (activation == KDA_ACT_SILU)
        kda_epilogue_range_kernel<kVec, 1><<<blocks, threads, 0, s>>>(first, count, out);
    else
        kda_epilogue_range_kernel<kVec, 0><<<blocks, threads, 0, s>>>(first, count, out);
    return record_cuda_error();
}

const char *kda_status_string(kda_status_t status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape or layout";
        case KDA_ERR_MISALIGNED: return "misaligned pointer or row stride";
        case KDA_ERR_CUDA: return "CUDA launch error";
        case KDA_ERR_METADATA: return "malformed metadata";
    }
    return "unknown status";
}

const char *kda_last_error_string(void) { return g_last_error; }

}  // extern "C"
