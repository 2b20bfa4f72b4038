/*
 * mla.h -- C ABI of libmla: decode of multi-head latent attention (MLA) over a
 * compressed latent||rope KV cache, on NVIDIA GB300 (sm_103a).
 *
 * The operations follow the page "mlx-bun 0.0.11 -> 0.0.13,
 * package/src/model/glm52-mla.ts" (the MLA page):
 *   - partialInterleavedRopeMlx         -> mla_rope_partial_interleaved
 *   - Glm52Mla.attendAbsorbed, q_nope @ Wk      -> mla_absorb_q
 *   - Glm52Mla.attendAbsorbed, scores, softmax, p @ latent, with the per-row
 *     windows of Glm52Mla.forward and the selected-position gather
 *                                        -> mla_decode_attend
 *   - Glm52Mla.attendAbsorbed, latentContext @ Wv^T, heads concatenated
 *                                        -> mla_project_v
 *   - rmsNormF32Mlx and the append of Glm52Mla.project / forward
 *                                        -> mla_append_compressed
 *   - the composition of the four decode operations -> mla_decode_step
 *   - Glm52Mla.attendReconstructed (prefill: per-head K/V materialised)
 *                                        -> mla_reconstruct_kv + mla_prefill_attend
 * and "mlx-bun ... glm52-dsa.ts", selectGlm52DsaDevice -> mla_select_topk,
 * and "mlx-bun 0.2.0 -> 0.4.0, glm52-cache.ts", Glm52Cache.specRoundRollback,
 * filter and mergeRows -> mla_plan_rollback / mla_plan_filter /
 * mla_plan_merge + mla_cache_shift_rows, and mla_rollback_lengths,
 * and the causal verify window of "mlx-bun 0.4.0 -> 1.0.0, glm52.ts",
 * Glm52DecoderLayer.attend (token i of a block sees the prefix up to itself).
 *
 * Conventions shared by every entry point
 *   - Ownership: the caller allocates and owns every buffer (device memory
 *     unless stated).  The library never allocates device memory, frees or
 *     synchronises; scratch memory is a caller-provided workspace.
 *   - Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Nothing is launched when a call returns an
 *     error, and outputs are then left untouched.
 *   - Errors: every function returns an mla_status.  Host-side checks of
 *     scalars, pointers, strides and alignment run before any launch; on
 *     failure a detail string is kept per thread (mla_last_error_detail).
 *     A failed launch returns MLA_ERR_CUDA.  Values that only exist on the
 *     device (lengths, selections) are checked by the kernels, which OR the
 *     MLA_DEVICE_* bits into *device_status (if non-NULL) and skip the bad
 *     entry instead of dereferencing it.
 *   - Layout: strides are in elements; the feature (last) axis is always
 *     contiguous.  dtype values are mla_dtype.
 *   - Threads: calls are thread-safe; distinct streams may run concurrently
 *     as long as their workspaces do not overlap.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (same type, declared without the CUDA headers). */
typedef struct CUstream_st* mla_stream_t;

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARGUMENT = 1, /* bad scalar, NULL pointer, bad stride or size */
  MLA_ERR_UNSUPPORTED = 2,      /* valid request that no kernel here serves     */
  MLA_ERR_CUDA = 3,             /* a CUDA runtime / launch error                */
  MLA_ERR_INDEX_OUT_OF_RANGE = 4,
  MLA_ERR_DEVICE_TIMEOUT = 5
} mla_status;

typedef enum mla_dtype { MLA_DTYPE_F32 = 0, MLA_DTYPE_BF16 = 1 } mla_dtype;

/* Bits the kernels OR into *device_status. */
#define MLA_DEVICE_BAD_SELECTION_COUNT (1 << 1) /* a count of 0, < -1 or > k_max   */
#define MLA_DEVICE_INDEX_OUT_OF_RANGE (1 << 4)  /* a position outside its window    */
#define MLA_DEVICE_TIMEOUT (1 << 5)             /* a bounded device wait gave up    */
#define MLA_DEVICE_LAYOUT (1 << 6)              /* shared memory not laid out as the
                                                   kernel expects; nothing computed */
#define MLA_DEVICE_SCORE_RANGE (1 << 7)         /* a bf16 decode score half exceeded
                                                   MLA_FP16_SCORE_LIMIT (see
                                                   mla_decode_attend)               */
#define MLA_DEVICE_VALUE_RANGE (1 << 8)         /* a split piece's context (an average
                                                   of latent rows) left the fp16
                                                   range of the bf16 decode's
                                                   partials; saturated               */
/* Largest |half score| (unscaled q . k over one CTA's 288 features) that the
 * bf16 decode's fp16 score exchange carries within the bf16 tolerance. */
#define MLA_FP16_SCORE_LIMIT 256.0f

/* Static, never NULL. */
const char* mla_status_string(int status);
/* Thread-local detail of the last failed call on this thread ("" if none). */
const char* mla_last_error_detail(void);
/* ABI version, (major << 16) | minor. */
int mla_version(void);

/* The page's softmax scale, 1/sqrt(qk_nope + qk_rope) (MLA page,
 * attendReconstructed and attendAbsorbed: scores divided by the square root of
 * qkHeadDim = qk_nope_head_dim + qk_rope_head_dim), rounded once to f32; pass
 * it as `softmax_scale`.  0 for negative dims or a zero sum. */
float mla_default_softmax_scale(int32_t nope, int32_t rope_dim);

/*
 * Partial interleaved RoPE (MLA page, partialInterleavedRopeMlx).
 *
 * Logical tensor [rows, tokens, inner, width]; element (r, t, i, f) sits at
 * base + r*strides[0] + t*strides[1] + i*strides[2] + f.  The first
 * `rotary_dims` features enter pair-interleaved [a0,b0,a1,b1,...] and leave
 * as split halves [r0..r_{h-1}, i0..i_{h-1}] with r_j = a_j cos - b_j sin and
 * i_j = b_j cos + a_j sin; features >= rotary_dims are copied.  Position of
 * token t of row r is p = offset_r + t with offset_r = row_offsets[r] (device
 * int32 [rows], values must be >= 0) or `position_offset` when row_offsets is
 * NULL.  Angle of pair j: f32(p * invf_j), invf_j = f32(pow(f32(theta),
 * f32(-2j / rotary_dims))) -- the page's f32 roundings -- then sincos in f32.
 * Math is f32; `in` and `out` share `dtype`.  in == out with equal strides
 * (in place) is allowed; other overlaps are not.
 * Errors: INVALID_ARGUMENT for NULL pointers, non-positive sizes, odd / zero /
 * too large rotary_dims (> width or > 256), theta <= 0 or not finite, a
 * negative position_offset.
 */
int mla_rope_partial_interleaved(const void* in, void* out, int dtype, int64_t rows,
                                 int64_t tokens, int64_t inner, int64_t width,
                                 const int64_t* in_strides /* host [3] */,
                                 const int64_t* out_strides /* host [3] */,
                                 int32_t rotary_dims, float theta,
                                 const int32_t* row_offsets, int64_t position_offset,
                                 mla_stream_t stream);

/*
 * Query absorption (MLA page, attendAbsorbed: "q_nope @ Wk produces latent-space q").
 *
 * q_out[n, h, 0:rank] = q_nope[n, h, 0:nope] @ W_UK_h, where W_UK_h is rows
 * [h*(nope+v_dim), h*(nope+v_dim)+nope) of kv_b_proj ([heads*(nope+v_dim),
 * rank], row-major, the linear layer's weight).  q_nope[n, h, k] sits at
 * q_nope + n*q_nope_row_stride + h*q_nope_head_stride + k; q_out likewise.
 * Only columns [0, rank) of each q_out head row are written, so q_out may be
 * the packed [n_q, H, rank+rope] query that mla_decode_attend reads.
 * fp32 accumulation; all three tensors have `dtype`.
 * bf16 is served for heads 64 or 128, nope = 128 and rank = 512 (other bf16
 * shapes: MLA_ERR_UNSUPPORTED), with q_nope and kv_b_proj 16-byte aligned
 * and q_nope strides multiples of 16 bytes (else MLA_ERR_INVALID_ARGUMENT),
 * at most 2^20 rows: 1..4 query rows are a matrix-vector product bound by the
 * weight read and run on the CUDA cores (one CTA per head), 5 rows and more
 * on the tensor cores (tcgen05, blocks of 256 rows).  f32 (any shape) runs
 * on the CUDA cores.
 */
int mla_absorb_q(const void* q_nope, int64_t q_nope_row_stride, int64_t q_nope_head_stride,
                 const void* kv_b_proj, void* q_out, int64_t q_out_row_stride,
                 int64_t q_out_head_stride, int dtype, int32_t n_q, int32_t heads, int32_t nope,
                 int32_t v_dim, int32_t rank, mla_stream_t stream);

/*
 * Latent-space decode attention (MLA page, attendAbsorbed: combined scores,
 * scale, softmax, p @ latent; with Glm52Mla.forward's per-row windows and
 * selected positions, and the verify window of Glm52DecoderLayer.attend).
 *
 * Query rows n = b*s_q + i (batch row b, token i < s_q).  q[n, h, 0:rank] is
 * the absorbed query and q[n, h, rank:rank+rope_dim] the rotated q_rope
 * (mla_absorb_q and mla_rope_partial_interleaved write exactly this).
 * Cache: row t of batch row b is latent[b*latent_batch_stride +
 * (kv_start[b]+t)*latent_row_stride + 0:rank] and rope[...] likewise, for
 * t < kv_len[b]; kv_start == NULL means 0.  Rows may be packed (batch stride
 * 0, kv_start = prefix sums) or padded (kv_start = the page's left pad);
 * kv_start[b] + kv_len[b] <= t_max is the caller's promise.  Token i of row
 * b sees window keys t <= kv_len[b] - s_q + i (causal among the s_q tokens).
 * Selection: if selected_positions != NULL, row n attends to the window keys
 * selected_positions[n*k_max + 0 .. count-1] (a multiset, any order), with
 * count = selected_counts[n]; count == -1 means dense.  A count of 0, < -1
 * or > k_max sets MLA_DEVICE_BAD_SELECTION_COUNT and the row attends to
 * nothing; a position outside the token's visible window sets
 * MLA_DEVICE_INDEX_OUT_OF_RANGE and is skipped.
 * s = (q_lat . latent_t + q_rope . rope_t) * softmax_scale (the page's scale
 * is 1/sqrt(qk_nope + qk_rope)); p = softmax(s); ctx = sum_t p_t latent_t.
 * Outputs: ctx_out[n*ctx_row_stride + h*ctx_head_stride + 0:rank] in
 * out_dtype, and lse_out[n*heads + h] = log(sum_t exp(s_t)) (f32, may be
 * NULL).  A row with no visible key gets ctx = 0 and lse = -inf.
 * q, latent and rope have `dtype`.  workspace must hold
 * mla_decode_workspace_size(...) bytes (256-byte aligned) and may be NULL
 * when that size is 0.
 * bf16 with heads 64 or 128, rank = 512, rope_dim = 64 runs the tensor-core
 * flash-decode kernel (tcgen05 + TMA, split-K over SM pairs; 64 heads are
 * padded to the MMA's 128 rows inside the kernel); it needs q, latent, rope
 * and ctx_out 16-byte aligned, strides that are multiples of 16 bytes, equal
 * zero-ness of the two batch strides and at most 2^20 query rows (else
 * MLA_ERR_INVALID_ARGUMENT).  Other bf16 shapes return MLA_ERR_UNSUPPORTED
 * and launch nothing.  f32 (any shape) runs a CUDA-core kernel.
 * Score range: each SM pair exchanges its two halves of a score (the
 * unscaled q . k over 288 of the 576 features) as fp16, so each half is
 * clamped to +-65504 and carries a rounding error of 2^-11 of its size; a
 * half whose magnitude exceeds MLA_FP16_SCORE_LIMIT sets
 * MLA_DEVICE_SCORE_RANGE (the result is still written, with that error).
 */
int mla_decode_attend(const void* q, int64_t q_row_stride, int64_t q_head_stride,
                      const void* latent, int64_t latent_row_stride, int64_t latent_batch_stride,
                      const void* rope, int64_t rope_row_stride, int64_t rope_batch_stride,
                      int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                      int32_t s_q, int32_t heads, int32_t rank, int32_t rope_dim, int64_t t_max,
                      const int32_t* selected_positions, const int32_t* selected_counts,
                      int32_t k_max, float softmax_scale, void* ctx_out, int64_t ctx_row_stride,
                      int64_t ctx_head_stride, int out_dtype, float* lse_out, void* workspace,
                      size_t workspace_bytes, int32_t* device_status, mla_stream_t stream);

/*
 * Decode attention for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for users of the library.
 *
 * Same arguments, results, checks and device-status bits as
 * mla_decode_attend, without `workspace` / `workspace_bytes`: the split-K
 * scratch is a fixed array of MLA_NO_ALLOC_SCRATCH_BYTES that the library
 * reserves on every GPU that loads it, held until the process exits.  Meant
 * for callers that cannot call cudaMalloc when they decode: a serving process
 * whose memory pool has already claimed the free device memory, a plugin or
 * foreign-language host that passes tensors in but has no allocator to hand,
 * or a latency-bound loop in which an allocation (and the device-wide
 * synchronisation it may cause) is not acceptable.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 * Set-up: the first call on a device looks up the array's device address with
 * that device current; make that first call before any stream capture.
 * Limit: a request whose mla_decode_workspace_size(...) exceeds
 * MLA_NO_ALLOC_SCRATCH_BYTES returns MLA_ERR_UNSUPPORTED and launches nothing
 * (at H = 128, rank 512 on a 152-SM GB300 this allows about 430 query rows).
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; nothing in it has to start at zero (each call writes what
 * it later reads).  Calls whose work overlaps on the GPU -- unordered streams,
 * or several host threads at once -- race on the array and give undefined
 * results; order them on one stream.
 */
#define MLA_NO_ALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int mla_decode_attend_no_alloc(const void* q, int64_t q_row_stride, int64_t q_head_stride,
                               const void* latent, int64_t latent_row_stride,
                               int64_t latent_batch_stride, const void* rope,
                               int64_t rope_row_stride, int64_t rope_batch_stride, int dtype,
                               const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                               int32_t s_q, int32_t heads, int32_t rank, int32_t rope_dim,
                               int64_t t_max, const int32_t* selected_positions,
                               const int32_t* selected_counts, int32_t k_max, float softmax_scale,
                               void* ctx_out, int64_t ctx_row_stride, int64_t ctx_head_stride,
                               int out_dtype, float* lse_out, int32_t* device_status,
                               mla_stream_t stream);

/* Workspace bytes mla_decode_attend needs for these sizes on the current
 * device (0 on an invalid request).  `selected` is non-zero when a selection
 * will be passed. */
size_t mla_decode_workspace_size(int32_t batch, int32_t s_q, int32_t heads, int32_t rank,
                                 int32_t rope_dim, int64_t t_max, int32_t k_max, int selected,
                                 int dtype);

/* 1 if mla_decode_attend runs the tensor-core kernel for these sizes, 0 if the
 * CUDA-core kernel (f32), -1 if the request is invalid or not served. */
int mla_decode_kernel_kind(int32_t heads, int32_t rank, int32_t rope_dim, int dtype, int out_dtype);

/*
 * Value projection (MLA page, attendAbsorbed: "the latent context multiplies
 * Wv^T", heads concatenated along the feature axis).
 *
 * out[n*out_row_stride + h*v_dim + j] = ctx[n, h, 0:rank] . W_UV_h[j, 0:rank],
 * W_UV_h = rows [h*(nope+v_dim)+nope, (h+1)*(nope+v_dim)) of kv_b_proj.
 * ctx[n, h, c] sits at ctx + n*ctx_row_stride + h*ctx_head_stride + c.  The
 * output stops before o_proj.  fp32 accumulation.  ctx and kv_b_proj have
 * `dtype`; out has out_dtype.  bf16 is served for heads 64 or 128, rank =
 * 512 and v_dim = 128 (other bf16 shapes: MLA_ERR_UNSUPPORTED) on the tensor
 * cores (tcgen05, blocks of 64 query rows, at most 2^20 rows), with ctx and
 * kv_b_proj 16-byte aligned and ctx strides multiples of 16 bytes (else
 * MLA_ERR_INVALID_ARGUMENT).  f32 (any shape) runs on the CUDA cores.
 */
int mla_project_v(const void* ctx, int64_t ctx_row_stride, int64_t ctx_head_stride,
                  const void* kv_b_proj, int dtype, void* out, int64_t out_row_stride,
                  int out_dtype, int32_t n_q, int32_t heads, int32_t nope, int32_t v_dim,
                  int32_t rank, mla_stream_t stream);

/*
 * Append of new tokens' compressed state (MLA page: rmsNormF32Mlx, and
 * Glm52Mla.project / Glm52Mla.forward, which normalise the latent part of the
 * new tokens' kv_a projection, rotate its rope part at the row's position
 * offset and append both to the cache before attending).
 *
 * Inputs: latent_raw[b*latent_raw_row_stride + t*latent_raw_token_stride +
 * 0:rank] and the pair-interleaved rope_raw[b*.. + t*.. + 0:rope_dim] of new
 * token t < s_new of batch row b, in `dtype`; norm_weight[rank] in `dtype`;
 * eps >= 0.  Token t is written to buffer row r = kv_start[b] + kv_len[b] + t
 * of the cache (layout as in mla_decode_attend; kv_start NULL means 0):
 * latent[r] = x * (mean(x^2) + eps)^(-1/2) * weight, computed in f32, and
 * rope[r] = the RoPE of mla_rope_partial_interleaved at position
 * row_offsets[b] + t (row_offsets NULL: the row's current length kv_len[b]),
 * in cache_dtype.  kv_len_out[b] (may be NULL, may alias kv_len) receives
 * kv_len[b] + s_new.  A row whose new tokens would pass t_max (or with a
 * negative length, start or offset) is left unchanged, keeps its length and
 * sets MLA_DEVICE_INDEX_OUT_OF_RANGE.  Rows of a packed buffer must leave
 * room after their windows: the call writes where it is told.
 * rank <= 1024, rope_dim even and <= 256.
 */
int mla_append_compressed(const void* latent_raw, int64_t latent_raw_row_stride, int64_t latent_raw_token_stride,
                          const void* rope_raw, int64_t rope_raw_row_stride, int64_t rope_raw_token_stride,
                          int dtype, const void* norm_weight, float eps, float theta, const int32_t* row_offsets,
                          void* latent, int64_t latent_row_stride, int64_t latent_batch_stride, void* rope,
                          int64_t rope_row_stride, int64_t rope_batch_stride, int cache_dtype,
                          const int32_t* kv_start, const int32_t* kv_len, int32_t* kv_len_out, int32_t batch,
                          int32_t s_new, int32_t rank, int32_t rope_dim, int64_t t_max, int32_t* device_status,
                          mla_stream_t stream);

/*
 * Deterministic DSA top-k selection ("mlx-bun ... glm52-dsa.ts",
 * selectGlm52DsaDevice): the positions that mla_decode_attend's selected mode
 * reads, from per-row f32 indexer scores (the score function itself is not
 * on the pages).
 *
 * Row n has lengths[n] (device) scores at scores[n*score_row_stride + 0..);
 * the caller promises lengths[n] <= score_row_stride.  A row with
 * lengths[n] <= top_k is dense: counts[n] = -1 and its selection row is left
 * as it was (a negative length also sets MLA_DEVICE_BAD_SELECTION_COUNT).
 * Otherwise counts[n] = top_k and selected[n*selected_row_stride + 0..top_k)
 * holds the top_k positions under the order (score descending, equal scores
 * by ascending position) -- equal means equal f32 bits, with the order of
 * the bits' monotone map to uint32 (+0 above -0; positive NaN above +inf,
 * negative NaN below -inf) -- listed as: the selected positions whose score
 * is above the threshold (the minimum selected score; NaN if any selected
 * score is NaN) in ascending order, then the others in ascending order.
 * The output is bit-exact and deterministic.
 */
int mla_select_topk(const float* scores, int64_t score_row_stride, const int32_t* lengths, int32_t n_rows,
                    int32_t top_k, int32_t* selected, int64_t selected_row_stride, int32_t* counts,
                    int32_t* device_status, mla_stream_t stream);

/*
 * One whole decode step of the attention layer in three launches: the four
 * operations above composed as the MLA page's attendAbsorbed composes them,
 * with RoPE folded into the absorb launch and the split combine folded into
 * the W_UV projection launch.
 *
 * Inputs: q_nope[n*q_nope_row_stride + h*q_nope_head_stride + 0:nope] and the
 * raw (pair-interleaved, unrotated) q_rope[n*q_rope_row_stride +
 * h*q_rope_head_stride + 0:rope_dim] of query row n = b*s_q + i, rotated at
 * position offset_b + i (offset_b = q_row_offsets[b], device, or
 * q_position_offset when q_row_offsets is NULL) with base `theta`, as
 * mla_rope_partial_interleaved does; kv_b_proj, the cache, the windows and
 * the selection exactly as mla_absorb_q and mla_decode_attend take them.
 * Output: out[n*out_row_stride + h*v_dim + j] as mla_project_v writes it, in
 * out_dtype, and lse_out[n*heads + h] as mla_decode_attend writes it (may be
 * NULL).  The absorbed query and the context stay in `workspace`, which must
 * hold mla_decode_step_workspace_size(...) bytes (256-byte aligned).
 * Served: bf16 with heads 128, nope 128, v_dim 128, rank 512, rope_dim 64 and
 * at most 64 query rows (16-byte aligned q_nope, q_rope, kv_b_proj and cache;
 * q_nope and cache strides multiples of 16 bytes); other requests return
 * MLA_ERR_UNSUPPORTED and launch nothing -- compose the four entry points.
 * Device-side checks and status bits are those of mla_decode_attend.
 */
int mla_decode_step(const void* q_nope, int64_t q_nope_row_stride, int64_t q_nope_head_stride,
                    const void* q_rope, int64_t q_rope_row_stride, int64_t q_rope_head_stride,
                    const int32_t* q_row_offsets, int64_t q_position_offset, float theta,
                    const void* kv_b_proj, const void* latent, int64_t latent_row_stride,
                    int64_t latent_batch_stride, const void* rope, int64_t rope_row_stride,
                    int64_t rope_batch_stride, int dtype, const int32_t* kv_start, const int32_t* kv_len,
                    int32_t batch, int32_t s_q, int32_t heads, int32_t nope, int32_t v_dim, int32_t rank,
                    int32_t rope_dim, int64_t t_max, const int32_t* selected_positions,
                    const int32_t* selected_counts, int32_t k_max, float softmax_scale, void* out,
                    int64_t out_row_stride, int out_dtype, float* lse_out, void* workspace,
                    size_t workspace_bytes, int32_t* device_status, mla_stream_t stream);

/* Workspace bytes mla_decode_step needs (0 if the request is invalid or not
 * served by the fused step). */
size_t mla_decode_step_workspace_size(int32_t batch, int32_t s_q, int32_t heads, int32_t nope, int32_t v_dim,
                                      int32_t rank, int32_t rope_dim, int64_t t_max, int32_t k_max,
                                      int selected, int dtype);

/*
 * Failure-detection self-test (no counterpart on the pages).  Every device
 * wait of the library is bounded: a wait that gives up sets
 * MLA_DEVICE_TIMEOUT, the kernel drains what it started and returns, and the
 * CUDA context stays usable.  This call launches one warp that waits on a
 * barrier nothing ever completes, through the same bounded wait, for at most
 * limit_cycles SM clock cycles (0 < limit <= 2^32; the kernels use 2^32,
 * about 2 s): afterwards *device_status has MLA_DEVICE_TIMEOUT set and
 * *waited_cycles (device, may be NULL) holds the cycles waited.
 */
int mla_selftest_bounded_wait(int64_t limit_cycles, int32_t* device_status, int64_t* waited_cycles,
                              mla_stream_t stream);

/*
 * Row operations of the compressed cache ("mlx-bun 0.2.0 -> 0.4.0,
 * package/src/model/glm52-cache.ts": Glm52Cache.specRoundRollback, filter and
 * mergeRows).
 *
 * Right-aligned layout (the pages' own): every state array (latent, rope, an
 * indexer key cache, ...) is [B, width, features]; row b holds row_offsets[b]
 * valid tokens in columns left_pad[b] .. width-1, so left_pad[b] +
 * row_offsets[b] == width.  Each operation is a host plan (integer
 * bookkeeping on host arrays, no device work) plus one mla_cache_shift_rows
 * call per state array, which writes a new array of the planned width:
 *   - rollback (specRoundRollback): row b began the round with
 *     before_offsets[b] tokens and keeps keep[b] of the tokens appended
 *     since.  Each row is rotated right by its rejected count (column c takes
 *     column (c - rejected + width) mod width) and the columns that are pad in
 *     every row afterwards are cut: shift[b] = removable - rejected[b] with
 *     removable = min_b(left_pad[b] + rejected[b]); the new width is width -
 *     removable.  The uniform case (the page hands it to trim) is the same
 *     rotation.
 *   - filter: the rows keep_rows[0..n_keep) in that order, less the leading
 *     columns that are pad in every kept row; src_row = keep_rows, shift[i] =
 *     that common pad.
 *   - merge (mergeRows): the rows of several caches, listed in merge order,
 *     right-aligned in a width equal to the largest row offset; pad columns
 *     are zero (zero_below[i] = the row's new pad).  Call mla_cache_shift_rows
 *     once per source cache, with dst advanced to that source's first row and
 *     the plan arrays sliced to its rows (src_row = the row's index in its
 *     source).
 * The plans take and return HOST int32 arrays of the row count, return
 * MLA_ERR_INVALID_ARGUMENT (writing nothing) for a row that is not
 * right-aligned, a kept row outside [0, batch) or a rollback that keeps more
 * tokens than the round appended, and never touch the device.
 *
 * Per-row window layout (kv_start, kv_len; the decode entry points'): no data
 * moves in a rollback; mla_rollback_lengths sets each row's length back to
 * its accepted prefix, and the rejected tokens are overwritten by the next
 * append.
 */
int mla_plan_rollback(int32_t batch, int32_t width, const int32_t* left_pad, const int32_t* row_offsets,
                      const int32_t* before_offsets, const int32_t* keep, int32_t* shift, int32_t* new_left_pad,
                      int32_t* new_row_offsets, int32_t* new_width);
int mla_plan_filter(int32_t batch, int32_t width, const int32_t* left_pad, const int32_t* row_offsets,
                    const int32_t* keep_rows, int32_t n_keep, int32_t* shift, int32_t* new_left_pad,
                    int32_t* new_row_offsets, int32_t* new_width);
int mla_plan_merge(int32_t n_rows, const int32_t* source_width, const int32_t* left_pad,
                   const int32_t* row_offsets, int32_t* shift, int32_t* zero_below, int32_t* new_left_pad,
                   int32_t* new_width);

/*
 * The gather behind the three row operations, bit-exact for any dtype:
 *   dst[i, c, :] = c < zero_below[i] ? 0
 *                : src[src_row[i], (c + shift[i]) mod src_width, :]
 * for rows i < n_rows (<= 65535) and columns c < dst_width.  src is [src_batch,
 * src_width, features] and dst [n_rows, dst_width, features], strides in
 * elements (token stride >= features; feature axis contiguous).  src_row,
 * shift and zero_below are DEVICE int32 arrays of n_rows (NULL: row i, 0, 0);
 * shift may be negative.  dst must not overlap src (MLA_ERR_INVALID_ARGUMENT:
 * the rotation is not done in place) and its rows must not overlap each
 * other.  dst_width 0 launches nothing.  A src_row outside [0, src_batch) or
 * a zero_below outside [0, dst_width] sets MLA_DEVICE_INDEX_OUT_OF_RANGE and
 * leaves that destination row unwritten.  src_width may be 0 (an empty
 * cache; src may then be NULL) when every row is all zero (zero_below[i] ==
 * dst_width); a row that would read it is flagged the same way.
 */
int mla_cache_shift_rows(const void* src, int64_t src_token_stride, int64_t src_batch_stride, int32_t src_batch,
                         int32_t src_width, void* dst, int64_t dst_token_stride, int64_t dst_batch_stride,
                         int32_t dst_width, int32_t features, int dtype, const int32_t* src_row,
                         const int32_t* shift, const int32_t* zero_below, int32_t n_rows, int32_t* device_status,
                         mla_stream_t stream);

/*
 * Rollback in the per-row window layout: kv_len_out[b] = kv_len_before[b] +
 * keep[b] (device int32 arrays of batch; kv_len_out may alias kv_len).  A row
 * with a negative entry or that would keep more than kv_len[b] tokens keeps
 * kv_len[b] and sets MLA_DEVICE_INDEX_OUT_OF_RANGE.
 */
int mla_rollback_lengths(const int32_t* kv_len_before, const int32_t* keep, const int32_t* kv_len,
                         int32_t* kv_len_out, int32_t batch, int32_t* device_status, mla_stream_t stream);

/*
 * Reconstructed prefill (the MLA page, Glm52Mla.attendReconstructed, with the
 * left-pad mask of the "mlx-bun 0.2.0 -> 0.4.0" hunk).  For a long block of
 * new tokens the per-head keys and values are materialised once and
 * attention runs in its plain form.
 *
 * mla_reconstruct_kv: for rows t < n_rows of latent [n_rows, rank] (row
 * stride in elements) and head h < heads,
 *   k_nope[t, h, :] = latent[t, :] . W_UK_h^T   (W_UK_h = kv_b_proj rows
 *                                                h*(nope+v_dim) .. +nope)
 *   v[t, h, :]      = latent[t, :] . W_UV_h^T   (the next v_dim rows)
 * kv_b_proj is [heads*(nope+v_dim), rank] contiguous.  k_nope / v element
 * (t, h, d) sits at t*row_stride + h*head_stride + d, rows and heads not
 * overlapping (row-major or head-major; else MLA_ERR_INVALID_ARGUMENT).
 * bf16 in and out, f32
 * accumulation.  Served: bf16, nope = v_dim = 128, rank a multiple of 64 up
 * to 1024, 16-byte aligned pointers and strides; other requests return
 * MLA_ERR_UNSUPPORTED.  The rope part of the keys is not materialised: it is
 * the cache's rope key, shared by all heads.
 *
 * mla_prefill_attend: query token i < s_q of batch row b (query row n =
 * b*s_q + i) attends, for every head, to the window keys t <= kv_len[b] -
 * s_q + i of buffer rows kv_start[b] + t (the block's own tokens are the
 * window's last s_q keys; kv_start is the page's left pad), with
 *   score = (q_nope[n,h,:] . k_nope[row,h,:] + q_rope[n,h,:] . rope[row,:]) * softmax_scale
 * and writes out[n, h*v_dim + d] = sum_t softmax(score)_t v[row, h, d]
 * (heads concatenated, out_dtype) and lse_out[n*heads + h] (natural log of
 * the softmax denominator, may be NULL).  q_rope must already be rotated
 * (mla_rope_partial_interleaved).  Buffer rows of batch row b start at
 * b*t_max, or all batch rows share rows 0..t_max-1 when `packed` is
 * non-zero; k_nope, v and rope are indexed by the same buffer row.  A query
 * token with no visible key (kv_len < s_q) gets zeros and lse = -inf.  A
 * window outside [0, t_max) sets MLA_DEVICE_INDEX_OUT_OF_RANGE and that
 * batch row is skipped.  Served: bf16 with nope 128, rope 64, v_dim 128,
 * 16-byte aligned pointers and strides (out_row_stride a multiple of 8);
 * other requests return MLA_ERR_UNSUPPORTED.
 */
int mla_reconstruct_kv(const void* latent, int64_t latent_row_stride, int64_t n_rows, const void* kv_b_proj,
                       int32_t heads, int32_t nope, int32_t v_dim, int32_t rank, void* k_nope,
                       int64_t k_row_stride, int64_t k_head_stride, void* v, int64_t v_row_stride,
                       int64_t v_head_stride, int dtype, int32_t* device_status, mla_stream_t stream);

int mla_prefill_attend(const void* q_nope, int64_t q_nope_row_stride, int64_t q_nope_head_stride,
                       const void* q_rope, int64_t q_rope_row_stride, int64_t q_rope_head_stride,
                       const void* k_nope, int64_t k_row_stride, int64_t k_head_stride, const void* v,
                       int64_t v_row_stride, int64_t v_head_stride, const void* rope, int64_t rope_row_stride,
                       int packed, int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                       int32_t s_q, int32_t heads, int32_t nope, int32_t rope_dim, int32_t v_dim, int64_t t_max,
                       float softmax_scale, void* out, int64_t out_row_stride, int out_dtype, float* lse_out,
                       int32_t* device_status, mla_stream_t stream);

/*
 * Test hook: the selected-position gather of attendAbsorbed (takeAxis on
 * latent and rope), bit-exact.  out[n, j, 0:rank+rope_dim] = latent || rope of
 * window key selected_positions[n*k_max + j] of query row n, for j < count;
 * the remaining slots, and slots whose position is outside the token's
 * visible window (flagged like mla_decode_attend), are zero.  A count of -1
 * gathers the visible window keys 0, 1, ... (at most k_max).
 */
int mla_gather_selected(const void* latent, int64_t latent_row_stride,
                        int64_t latent_batch_stride, const void* rope, int64_t rope_row_stride,
                        int64_t rope_batch_stride, int dtype, const int32_t* kv_start,
                        const int32_t* kv_len, int32_t batch, int32_t s_q, int32_t rank,
                        int32_t rope_dim, int64_t t_max, const int32_t* selected_positions,
                        const int32_t* selected_counts, int32_t k_max, void* out,
                        int32_t* device_status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
