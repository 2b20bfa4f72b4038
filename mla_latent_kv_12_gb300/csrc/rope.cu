// Partial interleaved RoPE ("glm52-mla.ts", partialInterleavedRopeMlx).
//
// One warp per feature vector (r, t, i): every lane first reads its pairs and
// tail elements into registers, the warp synchronises, then writes -- so the
// call may run in place.  The per-pair arithmetic is rope_rotate_pair.
#include <cuda_bf16.h>

#include "mla_internal.h"
#include "rope_math.cuh"
#include "tc_host.h"

namespace mla {
namespace {

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxPairsPerLane = kMaxRotaryDims / 2 / 32;  // 4
constexpr int kMaxTailPerLane = 8;                          // tail <= 256

template <typename T>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) rope_kernel(const __grid_constant__ RopeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t vec = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t nvec = p.rows * p.tokens * p.inner;
  if (vec >= nvec) return;
  const int64_t i = vec % p.inner;
  const int64_t t = (vec / p.inner) % p.tokens;
  const int64_t r = vec / (p.inner * p.tokens);
  const T* src = static_cast<const T*>(p.in) + r * p.in_stride[0] + t * p.in_stride[1] +
                 i * p.in_stride[2];
  T* dst = static_cast<T*>(p.out) + r * p.out_stride[0] + t * p.out_stride[1] +
           i * p.out_stride[2];
  const int half = p.rotary_dims >> 1;
  const int64_t pos = (p.row_offsets ? (int64_t)p.row_offsets[r] : p.position_offset) + t;

  float re[kMaxPairsPerLane], im[kMaxPairsPerLane];
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    const int j = lane + 32 * k;
    re[k] = 0.f;
    im[k] = 0.f;
    if (j < half) {
      rope_rotate_pair(load_f(src + 2 * j), load_f(src + 2 * j + 1), pos, p.inv_freq[j], re[k], im[k]);
    }
  }
  const int tail = (int)(p.width - p.rotary_dims);
  T tv[kMaxTailPerLane];
#pragma unroll
  for (int k = 0; k < kMaxTailPerLane; ++k) {
    const int e = lane + 32 * k;
    if (e < tail) tv[k] = src[p.rotary_dims + e];
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < kMaxPairsPerLane; ++k) {
    const int j = lane + 32 * k;
    if (j < half) {
      dst[j] = from_f<T>(re[k]);
      dst[half + j] = from_f<T>(im[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxTailPerLane; ++k) {
    const int e = lane + 32 * k;
    if (e < tail) dst[p.rotary_dims + e] = tv[k];
  }
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int dtype, cudaStream_t stream) {
  const int64_t nvec = p.rows * p.tokens * p.inner;
  const int64_t blocks = (nvec + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const cudaError_t e =
      dtype == MLA_DTYPE_F32
          ? launch_pdl(rope_kernel<float>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, stream, p)
          : launch_pdl(rope_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
