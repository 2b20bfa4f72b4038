// Absorption for a handful of query rows ("glm52-mla.ts", Glm52Mla.attendAbsorbed,
// q_nope @ W_UK_h), with the query RoPE folded in like the tensor-core launch.
//
// At up to four query rows the product is a matrix-vector product bound by
// reading W_UK (16.8 MB at H=128): one CTA per head streams its [128 x 512]
// slice with every byte in flight at once (512 threads x 16 loads of 16 B),
// multiplies on the CUDA cores in f32 and sums the eight partial products of
// the nope axis through shared memory.  128 CTAs leave the remaining SMs to
// the decode launch that follows (it may start as soon as this grid has
// waited for its own inputs).
#include <cuda_bf16.h>
#include <string.h>

#include "mla_internal.h"
#include "rope_math.cuh"
#include "tc_host.h"

namespace mla {
namespace {

constexpr int kGemvThreads = 512;
constexpr int kGemvRank = 512;   // latent dims: 64 groups of 8
constexpr int kGemvNope = 128;   // nope rows: 8 groups of 16

struct GemvArgs {
  AbsorbParams p;
  int32_t with_rope;
  AbsorbRope rope;
};

template <int NQ>
__global__ void __launch_bounds__(kGemvThreads) absorb_gemv_kernel(const __grid_constant__ GemvArgs g) {
  extern __shared__ float red[];   // [8 nope groups][NQ][512]
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const AbsorbParams& p = g.p;
  const int h = blockIdx.x, t = threadIdx.x;
  const int dg = t & 63, kg = t >> 6;   // dims 8dg .. 8dg+7, nope rows 16kg .. 16kg+15
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(p.w) +
                           ((int64_t)h * (p.nope + p.v_dim) + 16 * kg) * kGemvRank + 8 * dg;
  uint4 wv[16];
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) wv[kk] = __ldg(reinterpret_cast<const uint4*>(w + kk * kGemvRank));
  float acc[NQ][8];
#pragma unroll
  for (int n = 0; n < NQ; ++n) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[n][e] = 0.f;
    if (n < p.n_q) {
      const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q_nope) + (int64_t)n * p.q_row_stride +
                               (int64_t)h * p.q_head_stride + 16 * kg;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float qv = __bfloat162float(q[kk]);
        const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv[kk]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 wf = __bfloat1622float2(wp[e]);
          acc[n][2 * e] = fmaf(qv, wf.x, acc[n][2 * e]);
          acc[n][2 * e + 1] = fmaf(qv, wf.y, acc[n][2 * e + 1]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; e += 4)
      *reinterpret_cast<float4*>(&red[(kg * NQ + n) * kGemvRank + 8 * dg + e]) =
          make_float4(acc[n][e], acc[n][e + 1], acc[n][e + 2], acc[n][e + 3]);
  }
  __syncthreads();
  for (int o = t; o < NQ * kGemvRank; o += kGemvThreads) {
    const int n = o / kGemvRank, d = o % kGemvRank;
    if (n >= p.n_q) continue;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) s += red[(k * NQ + n) * kGemvRank + d];
    static_cast<__nv_bfloat16*>(p.out)[(int64_t)n * p.out_row_stride + (int64_t)h * p.out_head_stride + d] =
        __float2bfloat16_rn(s);
  }
  if (g.with_rope && t < 32) {
    // RoPE of head h's rope part: lane j = rotary pair j.
    const AbsorbRope& r = g.rope;
    for (int n = 0; n < p.n_q; ++n) {
      const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(r.q_rope) + (int64_t)n * r.row_stride +
                                 (int64_t)h * r.head_stride;
      const __nv_bfloat162 ab = reinterpret_cast<const __nv_bfloat162*>(src)[t];
      const int b = n / r.s_q, i = n % r.s_q;
      const int64_t pos = (r.row_offsets ? (int64_t)r.row_offsets[b] : r.position_offset) + i;
      float re, im;
      rope_rotate_pair(__low2float(ab), __high2float(ab), pos, r.inv_freq[t], re, im);
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (int64_t)n * p.out_row_stride +
                           (int64_t)h * p.out_head_stride + r.out_col;
      dst[t] = __float2bfloat16_rn(re);
      dst[32 + t] = __float2bfloat16_rn(im);
    }
  }
}

template <int NQ>
cudaError_t launch_nq(const GemvArgs& g, cudaStream_t stream) {
  const size_t smem = (size_t)8 * NQ * kGemvRank * sizeof(float);
  {
    const cudaError_t ea = set_max_dynamic_smem(absorb_gemv_kernel<NQ>, (int)smem);
    if (ea != cudaSuccess) return ea;
  }
  return launch_pdl(absorb_gemv_kernel<NQ>, dim3(g.p.heads), dim3(kGemvThreads), smem, stream, g);
}

}  // namespace

bool gemv_absorb_serves(const AbsorbParams& p) {
  return p.n_q >= 1 && p.n_q <= 4 && p.rank == kGemvRank && p.nope == kGemvNope &&
         (reinterpret_cast<uintptr_t>(p.w) & 15u) == 0;
}

cudaError_t launch_gemv_absorb(const AbsorbParams& p, cudaStream_t stream, const AbsorbRope* rope) {
  GemvArgs g;
  memset(&g, 0, sizeof(g));
  g.p = p;
  g.with_rope = rope != nullptr;
  if (rope) g.rope = *rope;
  cudaError_t e;
  switch (p.n_q) {
    case 1: e = launch_nq<1>(g, stream); break;
    case 2: e = launch_nq<2>(g, stream); break;
    default: e = launch_nq<4>(g, stream); break;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
