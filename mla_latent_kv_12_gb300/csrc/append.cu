// Append of new tokens' compressed state to the latent||rope cache
// ("glm52-mla.ts": rmsNormF32Mlx; Glm52Mla.project, which RMS-normalises the
// latent part of kv_a_proj's output and rotates its rope part at the row's
// position offset; Glm52Mla.forward, which appends both to the cache before
// attending).
//
// One CTA per batch row, one warp per new token: the warp reads the token's
// raw latent (up to 1024 values, 32 per lane), reduces the sum of squares with
// shuffles, scales by rsqrt(mean + eps) and the norm weight in f32 and stores
// to buffer row kv_start + kv_len + t; then it rotates the token's rope key at
// position offset + t (rope_rotate_pair, the RoPE kernel's arithmetic).  The
// row's new length is written after a block barrier, so the output may alias
// the input lengths.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "rope_math.cuh"
#include "tc_host.h"

namespace mla {
namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void st_f(T* p, float x);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kAppendWarps = 8;
constexpr int kMaxPerLane = kMaxAppendRank / 32;

template <typename TI, typename TC>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const __grid_constant__ AppendParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int len = p.kv_len[b];
  const int start = p.kv_start ? p.kv_start[b] : 0;
  const int64_t pos0 = p.row_offsets ? (int64_t)p.row_offsets[b] : (int64_t)len;
  const bool fits = len >= 0 && start >= 0 && pos0 >= 0 && (int64_t)start + len + p.s_new <= p.t_max;
  if (!fits) {
    if (threadIdx.x == 0 && p.status) atomicOr(p.status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
  } else {
    const TI* w = static_cast<const TI*>(p.weight);
    for (int t = warp; t < p.s_new; t += kAppendWarps) {
      const int64_t row = (int64_t)start + len + t;
      // ---- RMSNorm of the latent, f32
      const TI* x = static_cast<const TI*>(p.latent_raw) + b * p.lr_row_stride + t * p.lr_tok_stride;
      float v[kMaxPerLane];
      float sq = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxPerLane; ++k) {
        const int i = lane + 32 * k;
        v[k] = i < p.rank ? ld_f(x + i) : 0.f;
        sq = fmaf(v[k], v[k], sq);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      const float inv = rsqrtf(sq / (float)p.rank + p.eps);
      TC* dl = static_cast<TC*>(p.cache_latent) + b * p.cl_batch_stride + row * p.cl_row_stride;
#pragma unroll
      for (int k = 0; k < kMaxPerLane; ++k) {
        const int i = lane + 32 * k;
        if (i < p.rank) st_f(dl + i, v[k] * inv * ld_f(w + i));
      }
      // ---- RoPE of the rope key at position pos0 + t
      const TI* rr = static_cast<const TI*>(p.rope_raw) + b * p.rr_row_stride + t * p.rr_tok_stride;
      TC* dr = static_cast<TC*>(p.cache_rope) + b * p.cr_batch_stride + row * p.cr_row_stride;
      const int half = p.rope_dim >> 1;
      for (int j = lane; j < half; j += 32) {
        float re, im;
        rope_rotate_pair(ld_f(rr + 2 * j), ld_f(rr + 2 * j + 1), pos0 + t, p.inv_freq[j], re, im);
        st_f(dr + j, re);
        st_f(dr + half + j, im);
      }
    }
  }
  __syncthreads();   // every thread has read kv_len[b] before it may be overwritten
  if (threadIdx.x == 0 && p.kv_len_out) p.kv_len_out[b] = fits ? len + p.s_new : len;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int in_dtype, int cache_dtype, cudaStream_t stream) {
  const dim3 grid((unsigned)p.batch), block(kAppendWarps * 32);
  cudaError_t e;
  if (in_dtype == MLA_DTYPE_F32 && cache_dtype == MLA_DTYPE_F32)
    e = launch_pdl(append_kernel<float, float>, grid, block, 0, stream, p);
  else if (in_dtype == MLA_DTYPE_F32)
    e = launch_pdl(append_kernel<float, __nv_bfloat16>, grid, block, 0, stream, p);
  else if (cache_dtype == MLA_DTYPE_F32)
    e = launch_pdl(append_kernel<__nv_bfloat16, float>, grid, block, 0, stream, p);
  else
    e = launch_pdl(append_kernel<__nv_bfloat16, __nv_bfloat16>, grid, block, 0, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
