/*
 * kda_conv.h -- C ABI of the GB300 (sm_103a) packed varlen causal depthwise
 * conv1d that the Kimi-K3 KDA layer runs over the Q|K|V columns of its
 * in_proj output before the delta-rule recurrence.
 *
 * The operation is the one the vLLM page "vllm.models.kimi_k3.nvidia.ops.
 * kda_conv" (docs.vllm.ai) describes:
 *   - module docstring, 3rd paragraph: bf16 Q|K|V columns are read in place,
 *     widened exactly to FP32, convolved with FP32 weights and an FP32 conv
 *     state, passed through SiLU, rounded to bf16 to nearest even and stored
 *     as dense (tokens, part_dim) planes of one buffer;
 *   - module docstring, 4th paragraph: programs find their (sequence, token
 *     chunk) on the device from query_start_loc, so a launch needs no host
 *     table and can be captured in a CUDA graph; only a sequence's first
 *     chunk reads its conv state and that same program writes the update;
 *   - packed_causal_conv1d_fn and its docstring: the argument set (x, weight,
 *     bias, conv_states, query_start_loc, cache_indices, has_initial_state,
 *     part_dim, activation, null_block_id), width-4 taps, conv_states
 *     (cache lines, dim, 3) updated in place, result (dim/part_dim, tokens,
 *     part_dim), and the early return when there are no tokens or sequences;
 *   - packed_causal_conv1d_supported: what inputs the method accepts
 *     (unit channel stride, FP32 weight (dim, 4) and state, part_dim a
 *     multiple of 64 that divides dim).
 *
 * For token t of sequence s (rows query_start_loc[s] .. query_start_loc[s+1]-1)
 * and channel c, with v(j) the FP32 value of input row t-3+j (history rows
 * -3, -2, -1 come from the conv state, index 0 oldest):
 *     acc = bias ? bias[c] : +0.0f
 *     acc = fmaf(v(j), weight[c][j], acc)      for j = 0, 1, 2, 3 in that order
 *     y   = activation == SiLU ? acc / (1 + exp(-acc)) : acc
 *     out[c / part_dim][t][c % part_dim] = bf16_round_nearest_even(y)
 * and afterwards conv_states[cache_indices[s]][c][k] = v of row L-3+k
 * (k = 0, 1, 2; L = the sequence length), i.e. the last three rows of
 * [history ; the sequence's input rows].
 *
 * All entry points are synchronous with respect to the host only where
 * stated; the conv calls are asynchronous on the given stream, allocate
 * nothing, never synchronise, and launch a kernel and grid that depend only on
 * the scalar arguments (so a captured launch replays correctly for new
 * metadata values of the same tokens / num_seqs). When tokens < 16 * num_seqs
 * (sequences averaging under 16 rows, such as decode tokens mixed into a
 * prefill batch, or speculative-decoding verification) the packed entry
 * points launch an instantiation with a short-chunk path. Its results are the
 * same bit for bit. The conv kernels are launched as
 * programmatic dependents of the preceding kernel in the stream: they may be
 * scheduled while it drains, but every thread first waits until it has
 * completed and its writes are visible, so ordering is that of a plain launch.
 */
#ifndef KDA_CONV_H_
#define KDA_CONV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef void *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* NULL required pointer, negative size, bad activation, ... */
    KDA_ERR_UNSUPPORTED = 2, /* shape the method does not cover (part_dim % 64, dim % part_dim) */
    KDA_ERR_MISALIGNED = 3,  /* a pointer or the row stride breaks the 16-byte rule below */
    KDA_ERR_CUDA = 4,        /* the launch failed; kda_last_error_string() has CUDA's message */
    KDA_ERR_METADATA = 5     /* kda_validate_metadata found malformed metadata */
} kda_status_t;

typedef enum { KDA_ACT_NONE = 0, KDA_ACT_SILU = 1 } kda_activation_t;

/* Storage type of x and out, and of the conv state (kda_conv_layout_t). */
typedef enum { KDA_DTYPE_BF16 = 0, KDA_DTYPE_F16 = 1, KDA_DTYPE_F32 = 2 } kda_dtype_t;

/*
 * The general layout of kda_packed_conv1d_ex, after packed_causal_conv1d_supported
 * on the kda_conv page: x may be bf16, fp16 or fp32 (out has x's type, as
 * packed_causal_conv1d_fn returns x.dtype), the FP32 weight and the conv state are
 * passed with their strides, and the conv state may be wider than 3 or stored
 * as bf16.
 *   x_dtype        kda_dtype_t of x and out.
 *   state_width    K = conv_states size(2), 3..64. A line holds the K most recent
 *                  rows (position K-1 the newest); the taps read positions K-3..K-1;
 *                  afterwards the line holds the last K rows of [old line (or zeros
 *                  without an initial state) ; the sequence's rows].
 *   state_stride   element strides of conv_states: line, channel, position.
 *   weight_stride  element strides of weight: channel, tap (4, 1 is channel-major;
 *                  1, dim is the tap-major layout of a width-major weight copy).
 *   state_dtype    KDA_DTYPE_F32 or KDA_DTYPE_BF16 (any other value is
 *                  KDA_ERR_INVALID_ARG); set it explicitly: a zero-filled struct
 *                  means bf16. A bf16 state is read exactly (a bf16 is an fp32
 *                  value) and each value written to it is the FP32 value rounded
 *                  to nearest even; the accumulation stays FP32 either way. The
 *                  kda_conv page keeps the state in FP32; the kda_decode page's
 *                  fused decode kernel (is_fused_kda_decode_supported) takes a
 *                  bf16 conv state only. bf16 halves a decode step's state traffic.
 *   version        0 or 1 (any other value is KDA_ERR_INVALID_ARG). With 0 the
 *                  struct ends here: the library reads none of the fields below,
 *                  so a caller may pass the shorter struct of earlier releases.
 *                  With 1 the two fields below are read as well.
 *   weight_part_stride   (version 1) element stride between the parts of the
 *                  weight, for a weight that is not one (dim, 4) array: weight[c][j]
 *                  is at (c / part_dim) * weight_part_stride + (c % part_dim) *
 *                  weight_stride[0] + j * weight_stride[1]. 0 means part_dim *
 *                  weight_stride[0], i.e. the (dim, 4) form above. The width-major
 *                  decode weight of the vLLM page "vllm.models.kimi_k3.amd.ops.
 *                  kda_decode" (make_decode_conv1d_weight_loader: indexed
 *                  [qkv, width, channel], the channel contiguous) is a
 *                  (dim / part_dim, 4, part_dim) buffer: weight_stride = (1,
 *                  part_dim), weight_part_stride = 4 * part_dim.
 *   cache_index_stride   (version 1) elements between consecutive cache_indices
 *                  entries (sequence s uses cache_indices[s * stride]), as the
 *                  kda_conv page's packed_causal_conv1d_fn passes
 *                  cache_indices.stride(0) to its kernel; 0 means 1. Must be >= 0.
 */
typedef struct kda_conv_layout {
    int32_t x_dtype;
    int32_t state_width;
    int64_t state_stride[3];
    int64_t weight_stride[2];
    int32_t state_dtype;
    int32_t version;
    int64_t weight_part_stride; /* read only when version >= 1 */
    int64_t cache_index_stride; /* read only when version >= 1 */
} kda_conv_layout_t;

/*
 * kda_packed_conv1d -- the conv, one launch.
 *
 * Device pointers, all owned by the caller:
 *   x                 bf16 (tokens rows, x_row_stride elements apart); channels
 *                     0..dim-1 of each row are the input (a column slice of the
 *                     in_proj output, read in place). 16-byte aligned.
 *   weight            fp32 (dim, 4), contiguous, weight[c*4 + j] multiplies row
 *                     t-3+j. 16-byte aligned.
 *   bias              fp32 (dim) or NULL for no bias. 16-byte aligned.
 *   conv_states       fp32 (cache_lines, dim, 3), contiguous; index 2 is the most
 *                     recent row. Read and updated in place. 16-byte aligned.
 *   cache_indices     int32 [num_seqs]: the conv-state line of each sequence, or
 *                     null_block_id for a padding sequence (computed with a zero
 *                     history; its state is neither read nor written).
 *   has_initial_state uint8/bool [num_seqs]: 0 = start from a zero history.
 *   query_start_loc   int32 [num_seqs+1], non-decreasing, query_start_loc[num_seqs]
 *                     <= tokens: sequence s owns token rows [qsl[s], qsl[s+1]).
 *   out               bf16 (dim/part_dim, tokens, part_dim), dense; plane i holds
 *                     channels [i*part_dim, (i+1)*part_dim). Rows no sequence owns
 *                     are left as they were. 16-byte aligned.
 * Scalars: x_row_stride >= dim and a multiple of 8 elements; part_dim a positive
 * multiple of 64 dividing dim; activation a kda_activation_t; tokens and
 * num_seqs >= 0.
 *
 * Returns KDA_OK after enqueueing the launch on `stream` (or without a launch when
 * tokens == 0 or num_seqs == 0). Argument errors return without touching memory;
 * sizes whose launch would need 2^32 warps or more (program and warp indices are
 * divided in 32 bits on the device) return KDA_ERR_INVALID_ARG.
 * The metadata (query_start_loc, cache_indices) is the caller's contract and is
 * not checked on the device beyond clamping token rows to [0, tokens): a cache
 * index outside [0, cache_lines) other than null_block_id, or two live sequences
 * sharing a line, is undefined behaviour (kda_validate_metadata checks both).
 * `out` must not overlap x or conv_states.
 */
kda_status_t kda_packed_conv1d(const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim,
                               int64_t part_dim, const float *weight, const float *bias,
                               float *conv_states, const int32_t *cache_indices,
                               const uint8_t *has_initial_state, const int32_t *query_start_loc,
                               int64_t num_seqs, int64_t null_block_id, int activation, void *out,
                               kda_stream_t stream);

/*
 * kda_packed_conv1d_ex -- kda_packed_conv1d with the general layout above; layout
 * NULL means bf16 x, an fp32 state of width 3 and contiguous strides
 * (kda_packed_conv1d itself). conv_states points to elements of the layout's
 * state_dtype. Rounding of out: bf16 and fp16 to nearest even, fp32 none.
 * Alignment: x and out 16-byte aligned and x_row_stride a multiple of 16 bytes
 * (8 elements of bf16 / fp16, 4 of fp32); weight 16-byte aligned when its strides
 * are (4, 1) (and the part stride 4 * part_dim), else 4-byte; conv_states
 * 16-byte aligned when it is width 3 and
 * contiguous, else aligned to its element; bias 16-byte aligned. Everything else
 * as for kda_packed_conv1d.
 */
kda_status_t kda_packed_conv1d_ex(const void *x, int64_t x_row_stride, int64_t tokens,
                                  int64_t dim, int64_t part_dim, const float *weight,
                                  const float *bias, void *conv_states,
                                  const int32_t *cache_indices, const uint8_t *has_initial_state,
                                  const int32_t *query_start_loc, int64_t num_seqs,
                                  int64_t null_block_id, int activation, void *out,
                                  const kda_conv_layout_t *layout, kda_stream_t stream);

/*
 * kda_conv1d_update -- the decode-shaped case: token i (row i of x, i < batch) is
 * the next row of the sequence whose conv state is line cache_indices[i]. It is
 * kda_packed_conv1d with query_start_loc = 0, 1, ..., batch and every
 * has_initial_state set, computed without the program search: one thread per
 * (token, channel vector) reads the line's 3 newest rows, writes one output row
 * out[c / part_dim][i][c % part_dim] and the line shifted by one row (the oldest
 * dropped, x appended). A token whose cache index is null_block_id is computed
 * with a zero history and its line is not touched. The decode-step counterpart of
 * the conv update the kda_decode page's fused decode kernel performs. Layout as
 * for kda_packed_conv1d_ex (NULL: bf16 x, fp32 state, width 3, contiguous); with a
 * bf16 state the line is 6 bytes per channel instead of 12. Besides the
 * contiguous layout, two others move as vectors. One is a position-major state
 * (channel stride 1, as a width-first (lines, K, dim) cache viewed as
 * (lines, dim, K)) whose line and position strides are multiples of 4 and
 * whose base is 16-byte (fp32) or 8-byte (bf16) aligned. The other is a
 * tap-major weight (strides (1, a multiple of 4), 16-byte aligned). Other
 * strides are read and written element by element. Cache indices must
 * be distinct (or null); out must not overlap x or conv_states. batch * dim / 4
 * must be below 2^32 (KDA_ERR_INVALID_ARG otherwise). Asynchronous on `stream`;
 * allocates nothing.
 */
kda_status_t kda_conv1d_update(const void *x, int64_t x_row_stride, int64_t batch, int64_t dim,
                              int64_t part_dim, const float *weight, const float *bias,
                              void *conv_states, const int32_t *cache_indices,
                              int64_t null_block_id, int activation, void *out,
                              const kda_conv_layout_t *layout, kda_stream_t stream);

/*
 * The q/k L2 norm folded into the conv's epilogue, after the vLLM page
 * "vllm.models.kimi_k3.amd.ops.kda_prefill": chunk_kda_prefill takes q and k
 * as [1, T, H, K], and its use_qk_l2norm_in_kernel parameter and the fused
 * path's comment have the kernel that consumes them norm each token's heads
 * itself. Done here instead, the Q and K planes leave the conv normalised.
 * The norm costs no extra pass over memory.
 * The pages print neither the epsilon nor the precision. This library's
 * reading: for each token and each head of head_dim consecutive channels of a
 * selected plane, with y the FP32 conv output after the activation,
 *     y = y / sqrt(sum over the head of y^2 + eps)
 * computed in FP32 (the sum over lanes in a butterfly, the reciprocal root on
 * the special-function unit, relative error about 2^-23) before the rounding
 * to x's type.
 *   plane_mask  bit i: normalise output plane i (Q|K|V packing: 0x3 for q, k).
 *               0 = no norm. Bits at or above dim / part_dim are an error.
 *   head_dim    channels per head: 4, 8, 16, 32, 64 or 128, dividing part_dim.
 *   eps         0, or a normal finite number (>= FLT_MIN, about 1.18e-38); a
 *               subnormal eps is KDA_ERR_INVALID_ARG, because the reciprocal root
 *               flushes subnormal inputs to zero. With eps = 0 a head whose sum of
 *               squares is zero or subnormal comes out NaN or inf.
 *   reserved    must be 0.
 */
typedef struct kda_l2norm {
    uint32_t plane_mask;
    int32_t head_dim;
    float eps;
    int32_t reserved;
} kda_l2norm_t;

/*
 * kda_packed_conv1d_l2norm -- kda_packed_conv1d_ex, then the L2 norm above on
 * the planes norm->plane_mask selects. norm NULL or plane_mask 0 is
 * kda_packed_conv1d_ex itself. The conv state is updated exactly as without
 * the norm. Invalid norm options return KDA_ERR_INVALID_ARG (mask, eps,
 * reserved) or KDA_ERR_UNSUPPORTED (head_dim) before any launch.
 */
kda_status_t kda_packed_conv1d_l2norm(const void *x, int64_t x_row_stride, int64_t tokens,
                                      int64_t dim, int64_t part_dim, const float *weight,
                                      const float *bias, void *conv_states,
                                      const int32_t *cache_indices,
                                      const uint8_t *has_initial_state,
                                      const int32_t *query_start_loc, int64_t num_seqs,
                                      int64_t null_block_id, int activation, void *out,
                                      const kda_conv_layout_t *layout, const kda_l2norm_t *norm,
                                      kda_stream_t stream);

/*
 * kda_conv1d_update_l2norm -- kda_conv1d_update with the same L2 norm: the
 * decode step's q and k rows leave normalised, as in the fused decode kernel
 * of the vLLM page "vllm.models.kimi_k3.amd.ops.kda_decode".
 */
kda_status_t kda_conv1d_update_l2norm(const void *x, int64_t x_row_stride, int64_t batch,
                                      int64_t dim, int64_t part_dim, const float *weight,
                                      const float *bias, void *conv_states,
                                      const int32_t *cache_indices, int64_t null_block_id,
                                      int activation, void *out, const kda_conv_layout_t *layout,
                                      const kda_l2norm_t *norm, kda_stream_t stream);

/* kda_l2norm_check -- host only: the status the *_l2norm entry points return
 * for these norm options with this dim and part_dim. No CUDA call is made. */
kda_status_t kda_l2norm_check(const kda_l2norm_t *norm, int64_t dim, int64_t part_dim);

/*
 * kda_packed_conv1d_preact_f32 -- the same conv without activation or rounding:
 * `out` receives the FP32 accumulator (dim/part_dim, tokens, part_dim) and the conv
 * state is updated exactly as by kda_packed_conv1d. Same arguments and rules as
 * kda_packed_conv1d (there is no activation argument). For checking the FP32
 * arithmetic bit for bit; not a hot path.
 */
kda_status_t kda_packed_conv1d_preact_f32(const void *x, int64_t x_row_stride, int64_t tokens,
                                          int64_t dim, int64_t part_dim, const float *weight,
                                          const float *bias, float *conv_states,
                                          const int32_t *cache_indices,
                                          const uint8_t *has_initial_state,
                                          const int32_t *query_start_loc, int64_t num_seqs,
                                          int64_t null_block_id, float *out, kda_stream_t stream);

/*
 * kda_packed_conv1d_check_args -- host only: the status kda_packed_conv1d would
 * return for these arguments before launching (pointers are inspected for NULL and
 * alignment only, never dereferenced). No CUDA call is made.
 */
kda_status_t kda_packed_conv1d_check_args(const void *x, int64_t x_row_stride, int64_t tokens,
                                          int64_t dim, int64_t part_dim, const float *weight,
                                          const float *bias, const float *conv_states,
                                          const int32_t *cache_indices,
                                          const uint8_t *has_initial_state,
                                          const int32_t *query_start_loc, int64_t num_seqs,
                                          int activation, const void *out);

/* kda_packed_conv1d_ex_check_args -- host only: the argument check of
 * kda_packed_conv1d_ex (as kda_packed_conv1d_check_args, with a layout). */
kda_status_t kda_packed_conv1d_ex_check_args(
    const void *x, int64_t x_row_stride, int64_t tokens, int64_t dim, int64_t part_dim,
    const float *weight, const float *bias, const void *conv_states,
    const int32_t *cache_indices, const uint8_t *has_initial_state,
    const int32_t *query_start_loc, int64_t num_seqs, int activation, const void *out,
    const kda_conv_layout_t *layout);

/*
 * kda_packed_conv1d_launch_shape -- the launch kda_packed_conv1d makes for these
 * sizes on a GPU with sm_count SMs (sm_count = 0: the current device, which makes
 * one CUDA attribute query; a positive sm_count makes no CUDA call). *ctas = thread
 * blocks of the program map, *threads = threads per block, *chunk_tokens = tokens
 * per program, *programs = token programs (ceil(tokens/chunk) + num_seqs). A batch
 * of at most one token per sequence (tokens <= num_seqs) in the default layout runs
 * the map's blocks on at most one wave of resident blocks that loop over them; the
 * launched grid is then min(*ctas, resident blocks). Returns KDA_OK, or
 * KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED for bad sizes. When tokens == 0 or
 * num_seqs == 0 all outputs are 0 (no launch). Output pointers may be NULL.
 */
kda_status_t kda_packed_conv1d_launch_shape(int64_t tokens, int64_t dim, int64_t part_dim,
                                            int64_t num_seqs, int32_t sm_count, int64_t *ctas,
                                            int32_t *threads, int32_t *chunk_tokens,
                                            int64_t *programs);

/*
 * kda_validate_metadata -- host only, HOST pointers: checks query_start_loc
 * (qsl[0] >= 0, non-decreasing, qsl[num_seqs] <= tokens) and cache_indices
 * (each in [0, cache_lines) or equal to null_block_id; no line used by two
 * sequences). Returns KDA_OK or KDA_ERR_METADATA with *bad_seq set to the first
 * offending sequence (num_seqs for a bad final offset), or KDA_ERR_INVALID_ARG.
 * bad_seq may be NULL.
 */
kda_status_t kda_validate_metadata(const int32_t *query_start_loc, const int32_t *cache_indices,
                                   int64_t num_seqs, int64_t tokens, int64_t cache_lines,
                                   int64_t null_block_id, int64_t *bad_seq);

/*
 * kda_validate_metadata_device -- the checks of kda_validate_metadata on DEVICE
 * metadata, without copying it to the host: query_start_loc (num_seqs + 1 entries)
 * and cache_indices (num_seqs entries, cache_index_stride elements apart; 0 means
 * 1) are device pointers. The kda_conv page leaves the metadata to the caller
 * (packed_causal_conv1d_fn checks nothing on the device); this is the check a
 * caller can run on the metadata it is about to pass, on the stream it will use.
 * Two small kernels run on `stream`: the first records, for every cache line, the
 * first sequence that uses it (an atomic minimum in a scratch array of
 * cache_lines words) and the offset and range failures; the second marks a
 * sequence whose line an earlier sequence holds. The library takes the scratch
 * (cache_lines * 4 bytes + 256) with cudaMallocAsync on `stream` and returns it
 * with cudaFreeAsync.
 * Synchronous: the call copies the result back and synchronises `stream` before
 * it returns, so it cannot be captured in a CUDA graph. Returns KDA_OK,
 * KDA_ERR_METADATA with *bad_seq set exactly as kda_validate_metadata sets it
 * (the first offending sequence in the same order of checks; num_seqs for a bad
 * final offset), KDA_ERR_INVALID_ARG (negative sizes or stride, NULL pointers,
 * num_seqs > 2^30, cache_lines > 2^31), or KDA_ERR_CUDA (allocation, launch or
 * copy failure; kda_last_error_string() has CUDA's text). bad_seq may be NULL.
 */
kda_status_t kda_validate_metadata_device(const int32_t *query_start_loc,
                                          const int32_t *cache_indices,
                                          int64_t cache_index_stride, int64_t num_seqs,
                                          int64_t tokens, int64_t cache_lines,
                                          int64_t null_block_id, int64_t *bad_seq,
                                          kda_stream_t stream);

/*
 * kda_validate_metadata_device_noalloc -- kda_validate_metadata_device for callers
 * that cannot allocate device memory. The pages have no counterpart: this entry
 * point exists for callers such as a serving engine that has reserved all of the
 * GPU's memory up front for its own pool (so a cudaMalloc or cudaMallocAsync of
 * its own would fail or take memory the engine has promised elsewhere), or a
 * host thread that must not make the driver calls, and their possible
 * synchronisation, that allocating and freeing involve.
 * Same arguments, checks, results and synchronisation as
 * kda_validate_metadata_device, but the scratch is a fixed array inside the
 * library, 1 MiB of device memory on every GPU that loads the library, held until
 * the process exits: cache_lines may be at most 262144 (2^18); a larger value
 * returns KDA_ERR_UNSUPPORTED (kda_last_error_string() says why) before any CUDA
 * call. The call allocates nothing and frees nothing. The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress, with that device
 * current) and keeps it; make that first call before any stream capture begins.
 * Every call shares the one array: the call clears the words it uses before its
 * kernels run, so an earlier call's leftovers do not matter, but two calls whose
 * work overlaps on the GPU (other streams, other host threads, the same device)
 * race on it and may both report wrong results. Serialise them.
 */
kda_status_t kda_validate_metadata_device_noalloc(const int32_t *query_start_loc,
                                                  const int32_t *cache_indices,
                                                  int64_t cache_index_stride, int64_t num_seqs,
                                                  int64_t tokens, int64_t cache_lines,
                                                  int64_t null_block_id, int64_t *bad_seq,
                                                  kda_stream_t stream);

/*
 * kda_epilogue_range -- the device epilogue of kda_packed_conv1d on its own, for
 * checking it over all fp32 inputs. out[i] = bf16_round_nearest_even(act(f)), where
 * f is the fp32 value whose bit pattern is first + i (wrapping mod 2^32), for
 * i < count, through the same device functions as the conv kernel.
 * activation: KDA_ACT_NONE or KDA_ACT_SILU. Device `out` (uint16, count
 * elements, 16-byte aligned), asynchronous on `stream`.
 */
kda_status_t kda_epilogue_range(uint32_t first, uint64_t count, int activation, uint16_t *out,
                                kda_stream_t stream);

/* Static text for a status code. */
const char *kda_status_string(kda_status_t status);

/* The CUDA error text behind the calling thread's last KDA_ERR_CUDA ("" if none). */
const char *kda_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_CONV_H_ */
