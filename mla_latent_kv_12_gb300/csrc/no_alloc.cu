// mla_decode_attend_no_alloc: the decode entry point for callers that cannot
// allocate device memory when they decode.  Its split-K scratch is a
// file-scope device array that the library reserves on every GPU it is loaded
// on; the caller still passes every input and output buffer.
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

// The scratch array.  In host code this name is only a host-side stand-in: its
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[MLA_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up on the
// first call for that device, with that device current).
int scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error_detail("decode (no alloc): cudaGetDevice failed: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error_detail("decode (no alloc): device %d beyond the %d this library tracks", dev, kMaxDevices);
    return MLA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_error_detail("decode (no alloc): cudaGetSymbolAddress of the scratch array failed: %s",
                       cudaGetErrorString(e));
      return MLA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" int mla_decode_attend_no_alloc(
    const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* latent,
    int64_t latent_row_stride, int64_t latent_batch_stride, const void* rope, int64_t rope_row_stride,
    int64_t rope_batch_stride, int dtype, const int32_t* kv_start, const int32_t* kv_len, int32_t batch,
    int32_t s_q, int32_t heads, int32_t rank, int32_t rope_dim, int64_t t_max,
    const int32_t* selected_positions, const int32_t* selected_counts, int32_t k_max, float softmax_scale,
    void* ctx_out, int64_t ctx_row_stride, int64_t ctx_head_stride, int out_dtype, float* lse_out,
    int32_t* device_status, mla_stream_t stream) {
  const size_t need = mla_decode_workspace_size(batch, s_q, heads, rank, rope_dim, t_max, k_max,
                                                selected_positions != nullptr, dtype);
  if (need > MLA_NO_ALLOC_SCRATCH_BYTES) {
    mla::set_error_detail(
        "decode (no alloc): this request needs %zu bytes of scratch, more than the %zu-byte built-in "
        "array; use mla_decode_attend with a workspace",
        need, (size_t)MLA_NO_ALLOC_SCRATCH_BYTES);
    return MLA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  const int st = mla::scratch_on_current_device(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode_attend(q, q_row_stride, q_head_stride, latent, latent_row_stride, latent_batch_stride,
                           rope, rope_row_stride, rope_batch_stride, dtype, kv_start, kv_len, batch, s_q,
                           heads, rank, rope_dim, t_max, selected_positions, selected_counts, k_max,
                           softmax_scale, ctx_out, ctx_row_stride, ctx_head_stride, out_dtype, lse_out,
                           scratch, (size_t)MLA_NO_ALLOC_SCRATCH_BYTES, device_status, stream);
}
