// Internal declarations shared by the host API and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// Per-thread detail of the last error (set by the host API).
void set_error_detail(const char* fmt, ...);

constexpr int kMaxRotaryDims = 256;

struct RopeParams {
  const void* in;
  void* out;
  int64_t rows, tokens, inner, width;
  int64_t in_stride[3];
  int64_t out_stride[3];
  int32_t rotary_dims;
  const int32_t* row_offsets;
  int64_t position_offset;
  float inv_freq[kMaxRotaryDims / 2];
};
cudaError_t launch_rope(const RopeParams& p, int dtype, cudaStream_t stream);

// Geometry of a decode call (all strides in elements).
struct DecodeGeometry {
  const void* q;
  int64_t q_row_stride, q_head_stride;
  const void* latent;
  int64_t latent_row_stride, latent_batch_stride;
  const void* rope;
  int64_t rope_row_stride, rope_batch_stride;
  const int32_t* kv_start;
  const int32_t* kv_len;
  int32_t batch, s_q, heads, rank, rope_dim;
  int64_t t_max;
  const int32_t* sel;
  const int32_t* sel_count;
  int32_t k_max;
  float scale_log2;  // softmax_scale * log2(e)
  void* ctx_out;
  int64_t ctx_row_stride, ctx_head_stride;
  float* lse_out;
  int32_t* device_status;
};

// CUDA-core decode of the f32 path (any shape; f32 q and cache).
size_t simt_decode_workspace(const DecodeGeometry& g, int* splits_out);
cudaError_t launch_simt_decode(const DecodeGeometry& g, int dtype, int out_dtype, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

// Tensor-core decode (bf16, heads 64 or 128, rank 512, rope 64).  With a tail, the
// split combine is fused with the W_UV projection (bf16 context in
// g.ctx_out, n_q <= 64, v_dim 128) and `tail->out` receives [n_q, H*v].
struct DecodeTail {
  const void* w;  // kv_b_proj [heads*(nope+v_dim), rank] bf16
  void* out;
  int64_t out_row_stride;
  int out_dtype;
  int32_t heads, nope, v_dim, rank;
};
size_t tc_decode_workspace(int32_t n_q);
cudaError_t launch_tc_decode(const DecodeGeometry& g, int out_dtype, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream, const DecodeTail* tail = nullptr);

struct AbsorbParams {
  const void* q_nope;
  int64_t q_row_stride, q_head_stride;
  const void* w;
  void* out;
  int64_t out_row_stride, out_head_stride;
  int32_t n_q, heads, nope, v_dim, rank;
};
// RoPE of the query's rope part folded into the tensor-core absorb launch
// (bf16, 64 rotary dims = the whole rope part): q_rope[n, h, 0:64] enters
// pair-interleaved and leaves rotated at q_out[n, h, out_col : out_col+64].
// Position of query row n = b*s_q + i is offset_b + i.
struct AbsorbRope {
  const void* q_rope;
  int64_t row_stride, head_stride;
  int32_t s_q;
  const int32_t* row_offsets;  // device [batch] or NULL
  int64_t position_offset;     // used when row_offsets is NULL
  int32_t out_col;
  float inv_freq[32];
};
// The page's f32 roundings of the inverse frequencies:
// invf_j = f32(pow(f32 theta, f32(f32(-2j) / d))).
void rope_inverse_frequencies(float theta, int rotary_dims, float* inv_freq);

cudaError_t launch_simt_absorb(const AbsorbParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_tc_absorb(const AbsorbParams& p, cudaStream_t stream, const AbsorbRope* rope = nullptr);
// CUDA-core matrix-vector absorb for 1..4 query rows (bf16, rank 512, nope 128).
bool gemv_absorb_serves(const AbsorbParams& p);
cudaError_t launch_gemv_absorb(const AbsorbParams& p, cudaStream_t stream, const AbsorbRope* rope = nullptr);

struct ProjectParams {
  const void* ctx;
  int64_t ctx_row_stride, ctx_head_stride;
  const void* w;
  void* out;
  int64_t out_row_stride;
  int32_t n_q, heads, nope, v_dim, rank;
};
cudaError_t launch_simt_project(const ProjectParams& p, int dtype, int out_dtype,
                                cudaStream_t stream);
cudaError_t launch_tc_project(const ProjectParams& p, int out_dtype, cudaStream_t stream);

cudaError_t launch_gather(const DecodeGeometry& g, int dtype, void* out, cudaStream_t stream);

// Append of S new tokens per batch row (RMSNorm of the latent, RoPE of the key).
constexpr int kMaxAppendRank = 1024;
struct AppendParams {
  const void* latent_raw;
  int64_t lr_row_stride, lr_tok_stride;
  const void* rope_raw;
  int64_t rr_row_stride, rr_tok_stride;
  const void* weight;
  float eps;
  const int32_t* row_offsets;
  void* cache_latent;
  int64_t cl_row_stride, cl_batch_stride;
  void* cache_rope;
  int64_t cr_row_stride, cr_batch_stride;
  const int32_t* kv_start;
  const int32_t* kv_len;
  int32_t* kv_len_out;
  int32_t batch, s_new, rank, rope_dim;
  int64_t t_max;
  int32_t* status;
  float inv_freq[kMaxRotaryDims / 2];
};
cudaError_t launch_append(const AppendParams& p, int in_dtype, int cache_dtype, cudaStream_t stream);

// Deterministic top-k selection of positions from per-row f32 scores.
struct SelectParams {
  const float* scores;
  int64_t row_stride;
  const int32_t* lengths;
  int32_t n_rows, top_k;
  int32_t* selected;
  int64_t out_stride;
  int32_t* counts;
  int32_t* status;
};
cudaError_t launch_select_topk(const SelectParams& p, cudaStream_t stream);

// Row gather of a right-aligned cache state array (rollback, filter, merge):
// dst[i, c] = c < zero_below[i] ? 0 : src[src_row[i], (c + shift[i]) mod src_width].
// Sizes and strides in bytes.
struct ShiftRowsParams {
  const void* src;
  int64_t src_col_bytes, src_batch_bytes;
  int32_t src_batch, src_width;
  void* dst;
  int64_t dst_col_bytes, dst_batch_bytes;
  int32_t dst_width, n_rows;
  int64_t row_bytes;
  const int32_t* src_row;     // NULL: row i
  const int32_t* shift;       // NULL: 0
  const int32_t* zero_below;  // NULL: 0
  int32_t* status;
  int32_t units_per_col, cols_per_cta;  // set by the launcher
};
cudaError_t launch_shift_rows(const ShiftRowsParams& p, int vec_bytes, cudaStream_t stream);
cudaError_t launch_rollback_lengths(const int32_t* before, const int32_t* keep, const int32_t* kv_len,
                                    int32_t* kv_len_out, int32_t batch, int32_t* status, cudaStream_t stream);

// Reconstruction of per-head keys and values from latent rows (prefill).
struct ReconstructParams {
  const void* latent;
  int64_t latent_row_stride, n_rows;
  const void* kv_b_proj;
  int32_t heads, nope, v_dim, rank;
  void* k_nope;
  int64_t k_row_stride, k_head_stride;
  void* v;
  int64_t v_row_stride, v_head_stride;
  int32_t* status;
};
cudaError_t launch_tc_reconstruct(const ReconstructParams& p, cudaStream_t stream);

// Causal prefill attention over materialised per-head keys / values.
struct PrefillParams {
  const void* q_nope;
  int64_t qn_row_stride, qn_head_stride;
  const void* q_rope;
  int64_t qr_row_stride, qr_head_stride;
  const void* k_nope;
  int64_t k_row_stride, k_head_stride;
  const void* v;
  int64_t v_row_stride, v_head_stride;
  const void* rope;
  int64_t rope_row_stride;
  const int32_t* kv_start;
  const int32_t* kv_len;
  int64_t t_max;
  int32_t packed;
  int32_t batch, s_q, heads, nope, rope_dim, v_dim;
  float softmax_scale;
  void* out;
  int64_t out_row_stride;
  int32_t out_dtype;
  float* lse;
  int32_t* status;
};
cudaError_t launch_tc_prefill(const PrefillParams& p, cudaStream_t stream);

// Failure-detection self-test (a bounded wait on a barrier that never completes).
cudaError_t launch_bounded_wait(long long limit_cycles, int32_t* status, long long* waited, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace mla
