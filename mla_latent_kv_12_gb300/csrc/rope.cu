// Partial interleaved RoPE ("glm52-mla.ts", partialInterleavedRopeMlx).
//
// One warp per (r, t) and up to eight consecutive inner vectors i: the
// angles depend on the position only, so each lane takes one sincos per pair
// and applies it to all of the warp's vectors.  Every lane first reads its
// pairs of all those vectors into registers, the warp synchronises, then
// writes -- so the call may run in place.  The angle is rope_angle, the
// rotation the one of rope_rotate_pair.
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
constexpr int kVecPerWarp = 8;  // consecutive inner vectors of one (r, t): they share every angle

template <typename T, int PPL>  // PPL: rotary pairs per lane (rotary_dims <= 64 * PPL)
__global__ void __launch_bounds__(kWarpsPerBlock * 32) rope_kernel(const __grid_constant__ RopeParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t n_ic = (p.inner + kVecPerWarp - 1) / kVecPerWarp;
  const int64_t wv = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t n_wv = p.rows * p.tokens * n_ic;
  if (wv >= n_wv) return;
  int64_t ic, t, r;
  if (n_wv < (1LL << 31)) {
    // 32-bit division (a 64-bit one costs about a hundred instructions)
    const uint32_t w = (uint32_t)wv, nic = (uint32_t)n_ic, tok = (uint32_t)p.tokens;
    const uint32_t rt = w / nic;
    ic = w - rt * nic;
    r = rt / tok;
    t = rt - (uint32_t)r * tok;
  } else {
    ic = wv % n_ic;
    t = (wv / n_ic) % p.tokens;
    r = wv / (n_ic * p.tokens);
  }
  const int half = p.rotary_dims >> 1;
  const int64_t i0 = ic * kVecPerWarp;
  const int nv = (int)min((int64_t)kVecPerWarp, p.inner - i0);
  const T* src0 = static_cast<const T*>(p.in) + r * p.in_stride[0] + t * p.in_stride[1] + i0 * p.in_stride[2];
  T* dst0 = static_cast<T*>(p.out) + r * p.out_stride[0] + t * p.out_stride[1] + i0 * p.out_stride[2];

  // Every rotary pair of the warp's vectors is read before any is written, so
  // the call may run in place; the loads are issued before the angles are
  // formed so that their latency overlaps the sincos.
  float av[kVecPerWarp][PPL], bv[kVecPerWarp][PPL];
#pragma unroll
  for (int v = 0; v < kVecPerWarp; ++v)
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
      const int j = lane + 32 * k;
      av[v][k] = 0.f;
      bv[v][k] = 0.f;
      if (v < nv && j < half) {
        const T* src = src0 + v * p.in_stride[2];
        av[v][k] = load_f(src + 2 * j);
        bv[v][k] = load_f(src + 2 * j + 1);
      }
    }
  // Angles depend on (position, pair) only: one sincos per pair for the warp's vectors.
  const int64_t pos = (p.row_offsets ? (int64_t)p.row_offsets[r] : p.position_offset) + t;
  float sn[PPL], cs[PPL];
#pragma unroll
  for (int k = 0; k < PPL; ++k) {
    const int j = lane + 32 * k;
    sn[k] = 0.f;
    cs[k] = 1.f;
    if (j < half) sincosf(rope_angle(pos, p.inv_freq[j]), &sn[k], &cs[k]);
  }
  __syncwarp();
#pragma unroll
  for (int v = 0; v < kVecPerWarp; ++v)
#pragma unroll
    for (int k = 0; k < PPL; ++k) {
      const int j = lane + 32 * k;
      if (v < nv && j < half) {
        T* dst = dst0 + v * p.out_stride[2];
        dst[j] = from_f<T>(av[v][k] * cs[k] - bv[v][k] * sn[k]);
        dst[half + j] = from_f<T>(bv[v][k] * cs[k] + av[v][k] * sn[k]);
      }
    }
  // The kept tail is copied element for element (same position in and out).
  const int tail = (int)(p.width - p.rotary_dims);
  for (int v = 0; v < nv; ++v)
    for (int e = lane; e < tail; e += 32)
      dst0[v * p.out_stride[2] + p.rotary_dims + e] = src0[v * p.in_stride[2] + p.rotary_dims + e];
}

template <typename T>
cudaError_t launch_rope_t(const RopeParams& p, dim3 grid, cudaStream_t stream) {
  const int ppl = (p.rotary_dims + 63) / 64;
  if (ppl <= 1) return launch_pdl(rope_kernel<T, 1>, grid, dim3(kWarpsPerBlock * 32), 0, stream, p);
  if (ppl <= 2) return launch_pdl(rope_kernel<T, 2>, grid, dim3(kWarpsPerBlock * 32), 0, stream, p);
  return launch_pdl(rope_kernel<T, kMaxPairsPerLane>, grid, dim3(kWarpsPerBlock * 32), 0, stream, p);
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int dtype, cudaStream_t stream) {
  const int64_t nvec = p.rows * p.tokens * ((p.inner + kVecPerWarp - 1) / kVecPerWarp);
  const int64_t blocks = (nvec + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks);
  const cudaError_t e = dtype == MLA_DTYPE_F32 ? launch_rope_t<float>(p, grid, stream)
                                               : launch_rope_t<__nv_bfloat16>(p, grid, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
