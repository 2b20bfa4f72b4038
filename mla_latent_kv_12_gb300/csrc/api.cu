// Host side of the C ABI: argument validation, kernel selection, launches.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <stdint.h>

#include "mla_internal.h"

namespace mla {

namespace {
thread_local char g_detail[512] = "";

bool valid_dtype(int d) { return d == MLA_DTYPE_F32 || d == MLA_DTYPE_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return status;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MLA_OK;
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MLA_CHECK(cond, ...) \
  do {                       \
    if (!(cond)) return fail(MLA_ERR_INVALID_ARGUMENT, __VA_ARGS__); \
  } while (0)

}  // namespace

void set_error_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
}

void rope_inverse_frequencies(float theta, int rotary_dims, float* inv_freq) {
  // The page's f32 roundings: exponent f32(f32(-2j)/d), invf f32(pow(f32 theta, exponent)).
  const double theta32 = (double)(float)theta;
  for (int j = 0; j < rotary_dims / 2; ++j) {
    const float exponent = (float)((double)(float)(-2.0 * j) / (double)rotary_dims);
    inv_freq[j] = (float)pow(theta32, (double)exponent);
  }
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  if (dev < 64) cache[dev] = n;
  return n;
}

// The bf16 shapes the tensor-core kernels serve (the GLM / DeepSeek MLA
// shape with 64 or 128 heads).  Other bf16 shapes are refused.
static bool served_heads(int32_t heads) { return heads == 64 || heads == 128; }
static bool tc_decode_shape(int32_t heads, int32_t rank, int32_t rope_dim, int dtype) {
  return dtype == MLA_DTYPE_BF16 && served_heads(heads) && rank == 512 && rope_dim == 64;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_INDEX_OUT_OF_RANGE: return "index out of range";
    case MLA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* mla_last_error_detail(void) { return g_detail; }

float mla_default_softmax_scale(int32_t nope, int32_t rope_dim) {
  if (nope < 0 || rope_dim < 0 || nope + rope_dim <= 0) return 0.f;
  return (float)(1.0 / sqrt((double)nope + (double)rope_dim));
}

int mla_version(void) { return (1 << 16) | 0; }

int mla_rope_partial_interleaved(const void* in, void* out, int dtype, int64_t rows, int64_t tokens,
                                 int64_t inner, int64_t width, const int64_t* in_strides,
                                 const int64_t* out_strides, int32_t rotary_dims, float theta,
                                 const int32_t* row_offsets, int64_t position_offset,
                                 mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(in && out && in_strides && out_strides, "rope: NULL pointer");
  MLA_CHECK(valid_dtype(dtype), "rope: bad dtype %d", dtype);
  MLA_CHECK(rows > 0 && tokens > 0 && inner > 0 && width > 0, "rope: sizes must be positive");
  MLA_CHECK(rotary_dims > 0 && (rotary_dims & 1) == 0 && rotary_dims <= width &&
                rotary_dims <= kMaxRotaryDims,
            "rope: rotary_dims %d must be positive, even, <= width %lld and <= %d", rotary_dims,
            (long long)width, kMaxRotaryDims);
  MLA_CHECK(width - rotary_dims <= 256, "rope: the kept tail may hold at most 256 features");
  MLA_CHECK(isfinite(theta) && theta > 0.f, "rope: theta must be positive and finite");
  MLA_CHECK(row_offsets || position_offset >= 0, "rope: position offset must be non-negative");
  for (int k = 0; k < 3; ++k)
    MLA_CHECK(in_strides[k] >= 0 && out_strides[k] >= 0, "rope: strides must be non-negative");
  RopeParams p;
  memset(&p, 0, sizeof(p));
  p.in = in;
  p.out = out;
  p.rows = rows;
  p.tokens = tokens;
  p.inner = inner;
  p.width = width;
  for (int k = 0; k < 3; ++k) {
    p.in_stride[k] = in_strides[k];
    p.out_stride[k] = out_strides[k];
  }
  p.rotary_dims = rotary_dims;
  p.row_offsets = row_offsets;
  p.position_offset = position_offset;
  rope_inverse_frequencies(theta, rotary_dims, p.inv_freq);
  return cuda_status(launch_rope(p, dtype, (cudaStream_t)stream), "rope launch");
}

int mla_absorb_q(const void* q_nope, int64_t q_nope_row_stride, int64_t q_nope_head_stride,
                 const void* kv_b_proj, void* q_out, int64_t q_out_row_stride,
                 int64_t q_out_head_stride, int dtype, int32_t n_q, int32_t heads, int32_t nope,
                 int32_t v_dim, int32_t rank, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(q_nope && kv_b_proj && q_out, "absorb: NULL pointer");
  MLA_CHECK(valid_dtype(dtype), "absorb: bad dtype %d", dtype);
  MLA_CHECK(n_q > 0 && heads > 0 && nope > 0 && v_dim > 0 && rank > 0, "absorb: sizes must be positive");
  MLA_CHECK(nope <= 256, "absorb: nope %d > 256", nope);
  MLA_CHECK(q_nope_head_stride >= nope && q_nope_row_stride >= 0 && q_out_head_stride >= rank &&
                q_out_row_stride >= 0,
            "absorb: strides too small for the head widths");
  AbsorbParams p{q_nope, q_nope_row_stride, q_nope_head_stride, kv_b_proj, q_out,
                 q_out_row_stride, q_out_head_stride, n_q, heads, nope, v_dim, rank};
  if (dtype == MLA_DTYPE_F32)
    return cuda_status(launch_simt_absorb(p, dtype, (cudaStream_t)stream), "absorb launch");
  if (!(served_heads(heads) && nope == 128 && rank == 512))
    return fail(MLA_ERR_UNSUPPORTED, "absorb: bf16 is served for heads 64 or 128, nope 128, rank 512 "
                                     "(got heads %d, nope %d, rank %d)", heads, nope, rank);
  MLA_CHECK(n_q <= (1 << 20), "absorb: at most 2^20 query rows");
  MLA_CHECK(aligned16(q_nope) && aligned16(kv_b_proj) && q_nope_head_stride % 8 == 0 &&
                q_nope_row_stride % 8 == 0,
            "absorb: q_nope and kv_b_proj must be 16-byte aligned, q_nope strides multiples of 16 bytes");
  // Up to four rows the product is a matrix-vector product bound by the
  // weight read: CUDA cores stream it (no MMA tile to fill).
  if (gemv_absorb_serves(p))
    return cuda_status(launch_gemv_absorb(p, (cudaStream_t)stream), "absorb (matrix-vector) launch");
  return cuda_status(launch_tc_absorb(p, (cudaStream_t)stream), "absorb (tensor core) launch");
}

int mla_decode_kernel_kind(int32_t heads, int32_t rank, int32_t rope_dim, int dtype, int out_dtype) {
  if (heads <= 0 || rank <= 0 || rope_dim < 0 || !valid_dtype(dtype) || !valid_dtype(out_dtype)) return -1;
  if (dtype == MLA_DTYPE_F32) return 0;
  return tc_decode_shape(heads, rank, rope_dim, dtype) ? 1 : -1;
}

static int decode_geometry(DecodeGeometry& g, const void* q, int64_t q_row_stride,
                           int64_t q_head_stride, const void* latent, int64_t latent_row_stride,
                           int64_t latent_batch_stride, const void* rope, int64_t rope_row_stride,
                           int64_t rope_batch_stride, int dtype, const int32_t* kv_start,
                           const int32_t* kv_len, int32_t batch, int32_t s_q, int32_t heads,
                           int32_t rank, int32_t rope_dim, int64_t t_max,
                           const int32_t* selected_positions, const int32_t* selected_counts,
                           int32_t k_max, float softmax_scale, void* ctx_out,
                           int64_t ctx_row_stride, int64_t ctx_head_stride, float* lse_out,
                           int32_t* device_status, bool need_q) {
  MLA_CHECK(valid_dtype(dtype), "decode: bad dtype %d", dtype);
  MLA_CHECK(batch > 0 && s_q > 0 && heads > 0 && rank > 0 && rope_dim >= 0 && t_max > 0,
            "decode: sizes must be positive");
  MLA_CHECK((int64_t)batch * s_q <= (1 << 24), "decode: too many query rows");
  MLA_CHECK(t_max < (1LL << 31), "decode: t_max must fit int32");
  MLA_CHECK(rank <= 1024 && rope_dim <= 256, "decode: rank <= 1024 and rope <= 256 are served");
  MLA_CHECK(latent && kv_len && (rope || rope_dim == 0), "decode: NULL cache pointer");
  MLA_CHECK(!need_q || (q && ctx_out), "decode: NULL q or ctx_out");
  MLA_CHECK(latent_row_stride >= rank && latent_batch_stride >= 0 &&
                (rope_dim == 0 || rope_row_stride >= rope_dim) && rope_batch_stride >= 0,
            "decode: cache strides too small");
  if (need_q)
    MLA_CHECK(q_head_stride >= rank + rope_dim && q_row_stride >= 0 && ctx_head_stride >= rank &&
                  ctx_row_stride >= 0,
              "decode: q / ctx strides too small");
  MLA_CHECK(!need_q || (isfinite(softmax_scale) && softmax_scale > 0.f),
            "decode: softmax_scale must be positive");
  if (selected_positions) {
    MLA_CHECK(selected_counts && k_max > 0, "decode: a selection needs counts and k_max > 0");
  }
  memset(&g, 0, sizeof(g));
  g.q = q;
  g.q_row_stride = q_row_stride;
  g.q_head_stride = q_head_stride;
  g.latent = latent;
  g.latent_row_stride = latent_row_stride;
  g.latent_batch_stride = latent_batch_stride;
  g.rope = rope;
  g.rope_row_stride = rope_row_stride;
  g.rope_batch_stride = rope_batch_stride;
  g.kv_start = kv_start;
  g.kv_len = kv_len;
  g.batch = batch;
  g.s_q = s_q;
  g.heads = heads;
  g.rank = rank;
  g.rope_dim = rope_dim;
  g.t_max = t_max;
  g.sel = selected_positions;
  g.sel_count = selected_positions ? selected_counts : nullptr;
  g.k_max = selected_positions ? k_max : 0;
  g.scale_log2 = softmax_scale * 1.4426950408889634f;
  g.ctx_out = ctx_out;
  g.ctx_row_stride = ctx_row_stride;
  g.ctx_head_stride = ctx_head_stride;
  g.lse_out = lse_out;
  g.device_status = device_status;
  return MLA_OK;
}

size_t mla_decode_workspace_size(int32_t batch, int32_t s_q, int32_t heads, int32_t rank,
                                 int32_t rope_dim, int64_t t_max, int32_t k_max, int selected,
                                 int dtype) {
  if (batch <= 0 || s_q <= 0 || heads <= 0 || rank <= 0 || rope_dim < 0 || t_max <= 0 ||
      !valid_dtype(dtype) || (selected && k_max <= 0))
    return 0;
  const int64_t n_q = (int64_t)batch * s_q;   // 64-bit: no overflow before the limits below
  if (dtype == MLA_DTYPE_BF16) {
    if (!tc_decode_shape(heads, rank, rope_dim, dtype) || n_q > (1 << 20)) return 0;
    return (tc_decode_workspace((int32_t)n_q) + 255) & ~(size_t)255;
  }
  if (n_q > (1 << 24)) return 0;
  DecodeGeometry g;
  memset(&g, 0, sizeof(g));
  g.batch = batch;
  g.s_q = s_q;
  g.heads = heads;
  g.rank = rank;
  g.rope_dim = rope_dim;
  g.t_max = t_max;
  g.k_max = selected ? k_max : 0;
  g.sel = selected ? reinterpret_cast<const int32_t*>(16) : nullptr;
  const size_t need = simt_decode_workspace(g, nullptr);
  return (need + 255) & ~(size_t)255;
}

int mla_decode_attend(const void* q, int64_t q_row_stride, int64_t q_head_stride,
                      const void* latent, int64_t latent_row_stride, int64_t latent_batch_stride,
                      const void* rope, int64_t rope_row_stride, int64_t rope_batch_stride,
                      int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                      int32_t s_q, int32_t heads, int32_t rank, int32_t rope_dim, int64_t t_max,
                      const int32_t* selected_positions, const int32_t* selected_counts,
                      int32_t k_max, float softmax_scale, void* ctx_out, int64_t ctx_row_stride,
                      int64_t ctx_head_stride, int out_dtype, float* lse_out, void* workspace,
                      size_t workspace_bytes, int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  DecodeGeometry g;
  int st = decode_geometry(g, q, q_row_stride, q_head_stride, latent, latent_row_stride,
                           latent_batch_stride, rope, rope_row_stride, rope_batch_stride, dtype,
                           kv_start, kv_len, batch, s_q, heads, rank, rope_dim, t_max,
                           selected_positions, selected_counts, k_max, softmax_scale, ctx_out,
                           ctx_row_stride, ctx_head_stride, lse_out, device_status, true);
  if (st != MLA_OK) return st;
  MLA_CHECK(valid_dtype(out_dtype), "decode: bad out_dtype %d", out_dtype);
  if (dtype == MLA_DTYPE_BF16 && !tc_decode_shape(heads, rank, rope_dim, dtype))
    return fail(MLA_ERR_UNSUPPORTED, "decode: bf16 is served for heads 64 or 128, rank 512, rope_dim 64 "
                                     "(got heads %d, rank %d, rope_dim %d)", heads, rank, rope_dim);
  const size_t need = mla_decode_workspace_size(batch, s_q, heads, rank, rope_dim, t_max, k_max,
                                                selected_positions != nullptr, dtype);
  MLA_CHECK(workspace_bytes >= need && (need == 0 || workspace),
            "decode: workspace of %zu bytes < %zu needed", workspace_bytes, need);
  MLA_CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
            "decode: workspace must be 256-byte aligned");
  if (tc_decode_shape(heads, rank, rope_dim, dtype)) {
    // The tensor-core kernel moves 16-byte vectors and TMA boxes: every base
    // pointer 16-byte aligned, every stride a multiple of 16 bytes.
    const int64_t ovec = out_dtype == MLA_DTYPE_F32 ? 4 : 8;
    MLA_CHECK(aligned16(q) && aligned16(latent) && aligned16(rope) && aligned16(ctx_out),
              "decode: q, latent, rope and ctx_out must be 16-byte aligned");
    MLA_CHECK(q_row_stride % 8 == 0 && q_head_stride % 8 == 0 && latent_row_stride % 8 == 0 &&
                  latent_batch_stride % 8 == 0 && rope_row_stride % 8 == 0 &&
                  rope_batch_stride % 8 == 0 && ctx_row_stride % ovec == 0 && ctx_head_stride % ovec == 0,
              "decode: strides must be multiples of 16 bytes");
    MLA_CHECK((int64_t)batch * s_q <= (1 << 20), "decode: at most 2^20 query rows");
    MLA_CHECK((latent_batch_stride == 0) == (rope_batch_stride == 0),
              "decode: latent and rope batch strides must both be zero (packed rows) or both non-zero");
    return cuda_status(launch_tc_decode(g, out_dtype, workspace, workspace_bytes, (cudaStream_t)stream),
                       "decode (tensor core) launch");
  }
  return cuda_status(launch_simt_decode(g, dtype, out_dtype, workspace, workspace_bytes,
                                        (cudaStream_t)stream),
                     "decode launch");
}

static size_t step_q_bytes(int32_t n_q, int32_t heads) {
  return ((size_t)n_q * heads * 576 * 2 + 255) & ~(size_t)255;
}
static size_t step_ctx_bytes(int32_t n_q, int32_t heads) {
  return ((size_t)n_q * heads * 512 * 2 + 255) & ~(size_t)255;
}
static bool step_shape(int dtype, int32_t heads, int32_t nope, int32_t v_dim, int32_t rank, int32_t rope_dim,
                       int64_t n_q) {
  return dtype == MLA_DTYPE_BF16 && served_heads(heads) && nope == 128 && v_dim == 128 && rank == 512 &&
         rope_dim == 64 && n_q > 0 && n_q <= 64;
}

size_t mla_decode_step_workspace_size(int32_t batch, int32_t s_q, int32_t heads, int32_t nope, int32_t v_dim,
                                      int32_t rank, int32_t rope_dim, int64_t t_max, int32_t k_max,
                                      int selected, int dtype) {
  if (batch <= 0 || s_q <= 0 || t_max <= 0 || (selected && k_max <= 0) ||
      !step_shape(dtype, heads, nope, v_dim, rank, rope_dim, (int64_t)batch * s_q))
    return 0;
  const int32_t n_q = batch * s_q;
  return step_q_bytes(n_q, heads) + step_ctx_bytes(n_q, heads) + ((tc_decode_workspace(n_q) + 255) & ~(size_t)255);
}

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
                    size_t workspace_bytes, int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(q_nope && q_rope && kv_b_proj && out && workspace, "decode_step: NULL pointer");
  MLA_CHECK(valid_dtype(dtype) && valid_dtype(out_dtype), "decode_step: bad dtype");
  MLA_CHECK(batch > 0 && s_q > 0 && heads > 0 && nope > 0 && v_dim > 0 && rank > 0 && rope_dim > 0,
            "decode_step: sizes must be positive");
  MLA_CHECK(isfinite(theta) && theta > 0.f, "decode_step: theta must be positive and finite");
  MLA_CHECK(q_row_offsets || q_position_offset >= 0, "decode_step: position offset must be non-negative");
  const int64_t n_q = (int64_t)batch * s_q;
  if (!step_shape(dtype, heads, nope, v_dim, rank, rope_dim, n_q))
    return fail(MLA_ERR_UNSUPPORTED,
                "decode_step: the fused step serves bf16, heads 64 or 128, nope 128, v 128, rank 512, rope 64 "
                "and at most 64 query rows; compose the four entry points for other requests");
  MLA_CHECK(aligned16(q_nope) && aligned16(q_rope) && aligned16(kv_b_proj) && aligned16(latent) &&
                aligned16(rope),
            "decode_step: q_nope, q_rope, kv_b_proj, latent and rope must be 16-byte aligned");
  MLA_CHECK(q_nope_head_stride >= nope && q_nope_row_stride >= 0 && q_nope_head_stride % 8 == 0 &&
                q_nope_row_stride % 8 == 0,
            "decode_step: q_nope strides must cover nope and be multiples of 16 bytes");
  MLA_CHECK(q_rope_head_stride >= rope_dim && q_rope_row_stride >= 0 && q_rope_head_stride % 2 == 0 &&
                q_rope_row_stride % 2 == 0,
            "decode_step: q_rope strides must cover rope_dim and be even");
  MLA_CHECK(out_row_stride >= (int64_t)heads * v_dim, "decode_step: out_row_stride < heads * v_dim");
  MLA_CHECK(latent_row_stride % 8 == 0 && latent_batch_stride % 8 == 0 && rope_row_stride % 8 == 0 &&
                rope_batch_stride % 8 == 0,
            "decode_step: cache strides must be multiples of 16 bytes");
  MLA_CHECK((latent_batch_stride == 0) == (rope_batch_stride == 0),
            "decode_step: latent and rope batch strides must both be zero (packed rows) or both non-zero");
  const size_t need = mla_decode_step_workspace_size(batch, s_q, heads, nope, v_dim, rank, rope_dim, t_max, k_max,
                                                     selected_positions != nullptr, dtype);
  MLA_CHECK(need > 0 && workspace_bytes >= need, "decode_step: workspace of %zu bytes < %zu needed",
            workspace_bytes, need);
  MLA_CHECK((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
            "decode_step: workspace must be 256-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qbuf = ws;
  void* ctxbuf = ws + step_q_bytes((int32_t)n_q, heads);
  uint8_t* dws = ws + step_q_bytes((int32_t)n_q, heads) + step_ctx_bytes((int32_t)n_q, heads);
  const size_t dws_bytes = workspace_bytes - (size_t)(dws - ws);
  const int64_t D = rank + rope_dim;
  DecodeGeometry g;
  int st = decode_geometry(g, qbuf, heads * D, D, latent, latent_row_stride, latent_batch_stride, rope,
                           rope_row_stride, rope_batch_stride, dtype, kv_start, kv_len, batch, s_q, heads, rank,
                           rope_dim, t_max, selected_positions, selected_counts, k_max, softmax_scale, ctxbuf,
                           (int64_t)heads * rank, rank, lse_out, device_status, true);
  if (st != MLA_OK) return st;
  AbsorbParams ap{q_nope, q_nope_row_stride, q_nope_head_stride, kv_b_proj, qbuf, heads * D, D,
                  (int32_t)n_q, heads, nope, v_dim, rank};
  AbsorbRope rp;
  memset(&rp, 0, sizeof(rp));
  rp.q_rope = q_rope;
  rp.row_stride = q_rope_row_stride;
  rp.head_stride = q_rope_head_stride;
  rp.s_q = s_q;
  rp.row_offsets = q_row_offsets;
  rp.position_offset = q_position_offset;
  rp.out_col = rank;
  rope_inverse_frequencies(theta, rope_dim, rp.inv_freq);
  st = cuda_status(gemv_absorb_serves(ap) ? launch_gemv_absorb(ap, (cudaStream_t)stream, &rp)
                                           : launch_tc_absorb(ap, (cudaStream_t)stream, &rp),
                   "decode_step: absorb + rope launch");
  if (st != MLA_OK) return st;
  DecodeTail tail{kv_b_proj, out, out_row_stride, out_dtype, heads, nope, v_dim, rank};
  return cuda_status(launch_tc_decode(g, MLA_DTYPE_BF16, dws, dws_bytes, (cudaStream_t)stream, &tail),
                     "decode_step: decode + combine/projection launch");
}

int mla_append_compressed(const void* latent_raw, int64_t latent_raw_row_stride, int64_t latent_raw_token_stride,
                          const void* rope_raw, int64_t rope_raw_row_stride, int64_t rope_raw_token_stride,
                          int dtype, const void* norm_weight, float eps, float theta, const int32_t* row_offsets,
                          void* latent, int64_t latent_row_stride, int64_t latent_batch_stride, void* rope,
                          int64_t rope_row_stride, int64_t rope_batch_stride, int cache_dtype,
                          const int32_t* kv_start, const int32_t* kv_len, int32_t* kv_len_out, int32_t batch,
                          int32_t s_new, int32_t rank, int32_t rope_dim, int64_t t_max, int32_t* device_status,
                          mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(latent_raw && norm_weight && latent && kv_len && (rope_dim == 0 || (rope_raw && rope)),
            "append: NULL pointer");
  MLA_CHECK(valid_dtype(dtype) && valid_dtype(cache_dtype), "append: bad dtype");
  MLA_CHECK(batch > 0 && s_new > 0 && rank > 0 && rope_dim >= 0 && t_max > 0, "append: sizes must be positive");
  MLA_CHECK(rank <= kMaxAppendRank, "append: rank %d > %d", rank, kMaxAppendRank);
  MLA_CHECK((rope_dim & 1) == 0 && rope_dim <= kMaxRotaryDims, "append: rope_dim must be even and <= %d",
            kMaxRotaryDims);
  MLA_CHECK(isfinite(eps) && eps >= 0.f, "append: RMSNorm epsilon must be non-negative");
  MLA_CHECK(isfinite(theta) && theta > 0.f, "append: theta must be positive and finite");
  MLA_CHECK(latent_raw_token_stride >= rank && latent_raw_row_stride >= 0 && latent_row_stride >= rank &&
                latent_batch_stride >= 0,
            "append: latent strides too small");
  MLA_CHECK(rope_dim == 0 || (rope_raw_token_stride >= rope_dim && rope_raw_row_stride >= 0 &&
                              rope_row_stride >= rope_dim && rope_batch_stride >= 0),
            "append: rope strides too small");
  AppendParams p;
  memset(&p, 0, sizeof(p));
  p.latent_raw = latent_raw;
  p.lr_row_stride = latent_raw_row_stride;
  p.lr_tok_stride = latent_raw_token_stride;
  p.rope_raw = rope_raw;
  p.rr_row_stride = rope_raw_row_stride;
  p.rr_tok_stride = rope_raw_token_stride;
  p.weight = norm_weight;
  p.eps = eps;
  p.row_offsets = row_offsets;
  p.cache_latent = latent;
  p.cl_row_stride = latent_row_stride;
  p.cl_batch_stride = latent_batch_stride;
  p.cache_rope = rope;
  p.cr_row_stride = rope_row_stride;
  p.cr_batch_stride = rope_batch_stride;
  p.kv_start = kv_start;
  p.kv_len = kv_len;
  p.kv_len_out = kv_len_out;
  p.batch = batch;
  p.s_new = s_new;
  p.rank = rank;
  p.rope_dim = rope_dim;
  p.t_max = t_max;
  p.status = device_status;
  if (rope_dim > 0) rope_inverse_frequencies(theta, rope_dim, p.inv_freq);
  return cuda_status(launch_append(p, dtype, cache_dtype, (cudaStream_t)stream), "append launch");
}

int mla_select_topk(const float* scores, int64_t score_row_stride, const int32_t* lengths, int32_t n_rows,
                    int32_t top_k, int32_t* selected, int64_t selected_row_stride, int32_t* counts,
                    int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(scores && lengths && selected && counts, "select_topk: NULL pointer");
  MLA_CHECK(n_rows > 0 && top_k > 0, "select_topk: n_rows and top_k must be positive");
  MLA_CHECK(score_row_stride >= 0 && selected_row_stride >= top_k, "select_topk: strides too small");
  SelectParams p{scores, score_row_stride, lengths, n_rows, top_k, selected, selected_row_stride, counts,
                 device_status};
  return cuda_status(launch_select_topk(p, (cudaStream_t)stream), "select_topk launch");
}

int mla_selftest_bounded_wait(int64_t limit_cycles, int32_t* device_status, int64_t* waited_cycles,
                              mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(device_status, "selftest: NULL device_status");
  MLA_CHECK(limit_cycles > 0 && limit_cycles <= ((int64_t)1 << 32),
            "selftest: limit must be in (0, 2^32] cycles");
  return cuda_status(launch_bounded_wait((long long)limit_cycles, device_status,
                                         reinterpret_cast<long long*>(waited_cycles), (cudaStream_t)stream),
                     "selftest launch");
}

int mla_project_v(const void* ctx, int64_t ctx_row_stride, int64_t ctx_head_stride,
                  const void* kv_b_proj, int dtype, void* out, int64_t out_row_stride,
                  int out_dtype, int32_t n_q, int32_t heads, int32_t nope, int32_t v_dim,
                  int32_t rank, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(ctx && kv_b_proj && out, "project_v: NULL pointer");
  MLA_CHECK(valid_dtype(dtype) && valid_dtype(out_dtype), "project_v: bad dtype");
  MLA_CHECK(n_q > 0 && heads > 0 && nope > 0 && v_dim > 0 && rank > 0, "project_v: sizes must be positive");
  MLA_CHECK(rank <= 1024, "project_v: rank %d > 1024", rank);
  MLA_CHECK(ctx_head_stride >= rank && ctx_row_stride >= 0 && out_row_stride >= (int64_t)heads * v_dim,
            "project_v: strides too small");
  ProjectParams p{ctx, ctx_row_stride, ctx_head_stride, kv_b_proj, out, out_row_stride,
                  n_q, heads, nope, v_dim, rank};
  if (dtype == MLA_DTYPE_F32)
    return cuda_status(launch_simt_project(p, dtype, out_dtype, (cudaStream_t)stream), "project_v launch");
  if (!(served_heads(heads) && rank == 512 && v_dim == 128))
    return fail(MLA_ERR_UNSUPPORTED, "project_v: bf16 is served for heads 64 or 128, rank 512, v_dim 128 "
                                     "(got heads %d, rank %d, v_dim %d)", heads, rank, v_dim);
  MLA_CHECK(n_q <= (1 << 20), "project_v: at most 2^20 query rows");
  MLA_CHECK(aligned16(ctx) && aligned16(kv_b_proj) && ctx_head_stride % 8 == 0 && ctx_row_stride % 8 == 0,
            "project_v: ctx and kv_b_proj must be 16-byte aligned, ctx strides multiples of 16 bytes");
  return cuda_status(launch_tc_project(p, out_dtype, (cudaStream_t)stream), "project_v (tensor core) launch");
}

int mla_gather_selected(const void* latent, int64_t latent_row_stride, int64_t latent_batch_stride,
                        const void* rope, int64_t rope_row_stride, int64_t rope_batch_stride,
                        int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                        int32_t s_q, int32_t rank, int32_t rope_dim, int64_t t_max,
                        const int32_t* selected_positions, const int32_t* selected_counts,
                        int32_t k_max, void* out, int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(out && selected_counts && k_max > 0, "gather: NULL output, counts, or k_max <= 0");
  DecodeGeometry g;
  int st = decode_geometry(g, nullptr, 0, 0, latent, latent_row_stride, latent_batch_stride, rope,
                           rope_row_stride, rope_batch_stride, dtype, kv_start, kv_len, batch, s_q,
                           1, rank, rope_dim, t_max, selected_positions, selected_counts, k_max, 1.f,
                           nullptr, 0, 0, nullptr, device_status, false);
  if (st != MLA_OK) return st;
  g.sel_count = selected_counts;
  g.k_max = k_max;
  return cuda_status(launch_gather(g, dtype, out, (cudaStream_t)stream), "gather launch");
}

// ------------------------------------------------------------ cache row operations

int mla_plan_rollback(int32_t batch, int32_t width, const int32_t* left_pad, const int32_t* row_offsets,
                      const int32_t* before_offsets, const int32_t* keep, int32_t* shift, int32_t* new_left_pad,
                      int32_t* new_row_offsets, int32_t* new_width) {
  g_detail[0] = 0;
  MLA_CHECK(left_pad && row_offsets && before_offsets && keep && shift && new_left_pad && new_row_offsets &&
                new_width,
            "plan_rollback: NULL pointer");
  MLA_CHECK(batch > 0 && width >= 0, "plan_rollback: batch must be positive and width non-negative");
  int64_t removable = INT64_MAX;
  for (int32_t b = 0; b < batch; ++b) {
    MLA_CHECK(left_pad[b] >= 0 && row_offsets[b] >= 0 && (int64_t)left_pad[b] + row_offsets[b] == width,
              "plan_rollback: row %d is not right-aligned (pad %d + offset %d != width %d)", b, left_pad[b],
              row_offsets[b], width);
    const int64_t next = (int64_t)before_offsets[b] + keep[b];
    MLA_CHECK(before_offsets[b] >= 0 && keep[b] >= 0 && next <= row_offsets[b],
              "plan_rollback: row %d keeps %lld tokens of %d", b, (long long)next, row_offsets[b]);
    const int64_t pad = (int64_t)left_pad[b] + (row_offsets[b] - next);
    if (pad < removable) removable = pad;
  }
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t next = before_offsets[b] + keep[b];
    const int32_t rejected = row_offsets[b] - next;
    shift[b] = (int32_t)(removable - rejected);
    new_left_pad[b] = (int32_t)(left_pad[b] + rejected - removable);
    new_row_offsets[b] = next;
  }
  *new_width = (int32_t)(width - removable);
  return MLA_OK;
}

int mla_plan_filter(int32_t batch, int32_t width, const int32_t* left_pad, const int32_t* row_offsets,
                    const int32_t* keep_rows, int32_t n_keep, int32_t* shift, int32_t* new_left_pad,
                    int32_t* new_row_offsets, int32_t* new_width) {
  g_detail[0] = 0;
  MLA_CHECK(left_pad && row_offsets && keep_rows && shift && new_left_pad && new_row_offsets && new_width,
            "plan_filter: NULL pointer");
  MLA_CHECK(batch > 0 && width >= 0 && n_keep > 0, "plan_filter: batch and n_keep must be positive");
  int32_t removable = INT32_MAX;
  for (int32_t i = 0; i < n_keep; ++i) {
    const int32_t b = keep_rows[i];
    MLA_CHECK(b >= 0 && b < batch, "plan_filter: kept row %d outside [0, %d)", b, batch);
    MLA_CHECK(left_pad[b] >= 0 && row_offsets[b] >= 0 && (int64_t)left_pad[b] + row_offsets[b] == width,
              "plan_filter: row %d is not right-aligned", b);
    if (left_pad[b] < removable) removable = left_pad[b];
  }
  for (int32_t i = 0; i < n_keep; ++i) {
    shift[i] = removable;
    new_left_pad[i] = left_pad[keep_rows[i]] - removable;
    new_row_offsets[i] = row_offsets[keep_rows[i]];
  }
  *new_width = width - removable;
  return MLA_OK;
}

int mla_plan_merge(int32_t n_rows, const int32_t* source_width, const int32_t* left_pad,
                   const int32_t* row_offsets, int32_t* shift, int32_t* zero_below, int32_t* new_left_pad,
                   int32_t* new_width) {
  g_detail[0] = 0;
  MLA_CHECK(source_width && left_pad && row_offsets && shift && zero_below && new_left_pad && new_width,
            "plan_merge: NULL pointer");
  MLA_CHECK(n_rows > 0, "plan_merge: n_rows must be positive");
  int32_t width = 0;
  for (int32_t i = 0; i < n_rows; ++i) {
    MLA_CHECK(left_pad[i] >= 0 && row_offsets[i] >= 0 &&
                  (int64_t)left_pad[i] + row_offsets[i] == source_width[i],
              "plan_merge: row %d is not right-aligned in its source", i);
    if (row_offsets[i] > width) width = row_offsets[i];
  }
  for (int32_t i = 0; i < n_rows; ++i) {
    const int32_t pad = width - row_offsets[i];
    shift[i] = left_pad[i] - pad;
    zero_below[i] = pad;
    new_left_pad[i] = pad;
  }
  *new_width = width;
  return MLA_OK;
}

int mla_cache_shift_rows(const void* src, int64_t src_token_stride, int64_t src_batch_stride, int32_t src_batch,
                         int32_t src_width, void* dst, int64_t dst_token_stride, int64_t dst_batch_stride,
                         int32_t dst_width, int32_t features, int dtype, const int32_t* src_row,
                         const int32_t* shift, const int32_t* zero_below, int32_t n_rows, int32_t* device_status,
                         mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(dst && (src || src_width == 0), "shift_rows: NULL pointer");
  MLA_CHECK(valid_dtype(dtype), "shift_rows: bad dtype %d", dtype);
  MLA_CHECK(features > 0 && src_batch > 0 && src_width >= 0 && dst_width >= 0 && n_rows > 0,
            "shift_rows: sizes must be positive (widths non-negative)");
  MLA_CHECK(n_rows <= 65535, "shift_rows: at most 65535 rows per call");
  MLA_CHECK(src_token_stride >= features && dst_token_stride >= features && src_batch_stride >= 0 &&
                dst_batch_stride >= 0,
            "shift_rows: strides too small");
  MLA_CHECK(n_rows == 1 || dst_batch_stride >= (int64_t)dst_width * dst_token_stride,
            "shift_rows: destination rows overlap");
  if (dst_width == 0) return MLA_OK;
  const int64_t elem = dtype == MLA_DTYPE_F32 ? 4 : 2;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t s1 = s0 + (uintptr_t)(((int64_t)(src_batch - 1) * src_batch_stride +
                                         (int64_t)(src_width - 1) * src_token_stride + features) * elem);
  const uintptr_t d1 = d0 + (uintptr_t)(((int64_t)(n_rows - 1) * dst_batch_stride +
                                         (int64_t)(dst_width - 1) * dst_token_stride + features) * elem);
  MLA_CHECK(src_width == 0 || d1 <= s0 || s1 <= d0,
            "shift_rows: source and destination overlap (the gather is not in place)");
  ShiftRowsParams p;
  memset(&p, 0, sizeof(p));
  p.src = src;
  p.src_col_bytes = src_token_stride * elem;
  p.src_batch_bytes = src_batch_stride * elem;
  p.src_batch = src_batch;
  p.src_width = src_width;
  p.dst = dst;
  p.dst_col_bytes = dst_token_stride * elem;
  p.dst_batch_bytes = dst_batch_stride * elem;
  p.dst_width = dst_width;
  p.n_rows = n_rows;
  p.row_bytes = (int64_t)features * elem;
  p.src_row = src_row;
  p.shift = shift;
  p.zero_below = zero_below;
  p.status = device_status;
  int vec = 16;
  while (vec > 2 && ((s0 | d0) % vec || p.src_col_bytes % vec || p.dst_col_bytes % vec ||
                     p.src_batch_bytes % vec || p.dst_batch_bytes % vec || p.row_bytes % vec))
    vec >>= 1;
  return cuda_status(launch_shift_rows(p, vec, (cudaStream_t)stream), "shift_rows launch");
}

int mla_rollback_lengths(const int32_t* kv_len_before, const int32_t* keep, const int32_t* kv_len,
                         int32_t* kv_len_out, int32_t batch, int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(kv_len_before && keep && kv_len && kv_len_out, "rollback_lengths: NULL pointer");
  MLA_CHECK(batch > 0, "rollback_lengths: batch must be positive");
  return cuda_status(launch_rollback_lengths(kv_len_before, keep, kv_len, kv_len_out, batch, device_status,
                                             (cudaStream_t)stream),
                     "rollback_lengths launch");
}

// ------------------------------------------------------------ reconstructed prefill

int mla_reconstruct_kv(const void* latent, int64_t latent_row_stride, int64_t n_rows, const void* kv_b_proj,
                       int32_t heads, int32_t nope, int32_t v_dim, int32_t rank, void* k_nope,
                       int64_t k_row_stride, int64_t k_head_stride, void* v, int64_t v_row_stride,
                       int64_t v_head_stride, int dtype, int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(latent && kv_b_proj && k_nope && v, "reconstruct: NULL pointer");
  MLA_CHECK(valid_dtype(dtype), "reconstruct: bad dtype %d", dtype);
  MLA_CHECK(n_rows > 0 && heads > 0 && nope > 0 && v_dim > 0 && rank > 0, "reconstruct: sizes must be positive");
  MLA_CHECK(n_rows < ((int64_t)1 << 31), "reconstruct: at most 2^31 - 1 rows");
  MLA_CHECK(latent_row_stride >= rank && k_head_stride >= nope && v_head_stride >= v_dim && k_row_stride >= 0 &&
                v_row_stride >= 0,
            "reconstruct: strides too small");
  // The outputs are written: their (row, head) vectors must not overlap, in a
  // row-major ([rows, heads, d]) or head-major ([heads, rows, d]) layout.
  auto disjoint = [&](int64_t row_stride, int64_t head_stride, int64_t d) {
    return (row_stride >= (int64_t)heads * head_stride && head_stride >= d) ||
           (head_stride >= n_rows * row_stride && row_stride >= d);
  };
  MLA_CHECK(disjoint(k_row_stride, k_head_stride, nope) && disjoint(v_row_stride, v_head_stride, v_dim),
            "reconstruct: output rows or heads overlap");
  if (!(dtype == MLA_DTYPE_BF16 && nope == 128 && v_dim == 128 && rank % 64 == 0 && rank <= 1024 &&
        heads <= 65535))
    return fail(MLA_ERR_UNSUPPORTED, "reconstruct: served for bf16, nope = v = 128, rank a multiple of 64 "
                                     "up to 1024");
  MLA_CHECK(aligned16(latent) && aligned16(kv_b_proj) && aligned16(k_nope) && aligned16(v) &&
                latent_row_stride % 8 == 0 && k_row_stride % 8 == 0 && k_head_stride % 8 == 0 &&
                v_row_stride % 8 == 0 && v_head_stride % 8 == 0,
            "reconstruct: pointers and strides must be 16-byte aligned");
  ReconstructParams p{latent, latent_row_stride, n_rows, kv_b_proj, heads, nope, v_dim, rank, k_nope,
                      k_row_stride, k_head_stride, v, v_row_stride, v_head_stride, device_status};
  return cuda_status(launch_tc_reconstruct(p, (cudaStream_t)stream), "reconstruct launch");
}

int mla_prefill_attend(const void* q_nope, int64_t q_nope_row_stride, int64_t q_nope_head_stride,
                       const void* q_rope, int64_t q_rope_row_stride, int64_t q_rope_head_stride,
                       const void* k_nope, int64_t k_row_stride, int64_t k_head_stride, const void* v,
                       int64_t v_row_stride, int64_t v_head_stride, const void* rope, int64_t rope_row_stride,
                       int packed, int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
                       int32_t s_q, int32_t heads, int32_t nope, int32_t rope_dim, int32_t v_dim, int64_t t_max,
                       float softmax_scale, void* out, int64_t out_row_stride, int out_dtype, float* lse_out,
                       int32_t* device_status, mla_stream_t stream) {
  g_detail[0] = 0;
  MLA_CHECK(q_nope && q_rope && k_nope && v && rope && kv_start && kv_len && out, "prefill: NULL pointer");
  MLA_CHECK(valid_dtype(dtype) && valid_dtype(out_dtype), "prefill: bad dtype");
  MLA_CHECK(batch > 0 && s_q > 0 && heads > 0 && nope > 0 && rope_dim > 0 && v_dim > 0 && t_max > 0,
            "prefill: sizes must be positive");
  MLA_CHECK(isfinite(softmax_scale) && softmax_scale > 0.f, "prefill: softmax scale must be positive and finite");
  MLA_CHECK(q_nope_head_stride >= nope && q_rope_head_stride >= rope_dim && k_head_stride >= nope &&
                v_head_stride >= v_dim && rope_row_stride >= rope_dim && q_nope_row_stride >= 0 &&
                q_rope_row_stride >= 0 && k_row_stride >= 0 && v_row_stride >= 0 &&
                out_row_stride >= (int64_t)heads * v_dim,
            "prefill: strides too small");
  const int64_t buf_rows = packed ? t_max : (int64_t)batch * t_max;
  MLA_CHECK(buf_rows < ((int64_t)1 << 31) && (int64_t)batch * s_q < ((int64_t)1 << 31),
            "prefill: at most 2^31 - 1 buffer rows and query rows");
  if (!(dtype == MLA_DTYPE_BF16 && nope == 128 && rope_dim == 64 && v_dim == 128 && heads <= 65535 &&
        batch <= 65535))
    return fail(MLA_ERR_UNSUPPORTED, "prefill: served for bf16 with nope 128, rope 64, v 128");
  MLA_CHECK(aligned16(q_nope) && aligned16(q_rope) && aligned16(k_nope) && aligned16(v) && aligned16(rope) &&
                aligned16(out) && q_nope_row_stride % 8 == 0 && q_nope_head_stride % 8 == 0 &&
                q_rope_row_stride % 8 == 0 && q_rope_head_stride % 8 == 0 && k_row_stride % 8 == 0 &&
                k_head_stride % 8 == 0 && v_row_stride % 8 == 0 && v_head_stride % 8 == 0 &&
                rope_row_stride % 8 == 0 && out_row_stride % 8 == 0,
            "prefill: pointers and strides must be 16-byte aligned");
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  p.q_nope = q_nope;
  p.qn_row_stride = q_nope_row_stride;
  p.qn_head_stride = q_nope_head_stride;
  p.q_rope = q_rope;
  p.qr_row_stride = q_rope_row_stride;
  p.qr_head_stride = q_rope_head_stride;
  p.k_nope = k_nope;
  p.k_row_stride = k_row_stride;
  p.k_head_stride = k_head_stride;
  p.v = v;
  p.v_row_stride = v_row_stride;
  p.v_head_stride = v_head_stride;
  p.rope = rope;
  p.rope_row_stride = rope_row_stride;
  p.kv_start = kv_start;
  p.kv_len = kv_len;
  p.t_max = t_max;
  p.packed = packed ? 1 : 0;
  p.batch = batch;
  p.s_q = s_q;
  p.heads = heads;
  p.nope = nope;
  p.rope_dim = rope_dim;
  p.v_dim = v_dim;
  p.softmax_scale = softmax_scale;
  p.out = out;
  p.out_row_stride = out_row_stride;
  p.out_dtype = out_dtype;
  p.lse = lse_out;
  p.status = device_status;
  return cuda_status(launch_tc_prefill(p, (cudaStream_t)stream), "prefill launch");
}

}  // extern "C"
