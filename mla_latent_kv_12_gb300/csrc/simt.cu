// CUDA-core kernels of the f32 path: the general-shape decode (any heads /
// rank / rope over an f32 cache), its split combine, query absorption and value
// projection, plus the selected-position gather (f32 or bf16 rows, a bit-exact
// copy).  f32 arithmetic throughout: TF32 tensor cores would miss the f32
// path's 1e-4 relative bound.  bf16 caches are served by the tensor-core
// kernels only (other bf16 shapes are refused by the host API).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {
namespace {

__device__ __forceinline__ float to_f(float x) { return x; }
template <typename T>
__device__ __forceinline__ T cvt(float x);
template <>
__device__ __forceinline__ float cvt<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Number of keys query row n may attend to, and whether they come from a
// selection.  Dense rows see window keys 0 .. kv_len - s_q + i.
struct RowKeys {
  int32_t start;   // kv_start[b]
  int32_t limit;   // keys visible to this token (window prefix length)
  int32_t count;   // entries to visit
  const int32_t* list;  // selection list or nullptr (dense)
  int64_t batch_off_lat, batch_off_rope;
};

__device__ __forceinline__ RowKeys row_keys(const DecodeGeometry& g, int n) {
  RowKeys k;
  const int b = n / g.s_q, i = n % g.s_q;
  k.start = g.kv_start ? g.kv_start[b] : 0;
  const int32_t len = g.kv_len[b];
  k.limit = len - g.s_q + i + 1;
  if (k.limit < 0) k.limit = 0;
  if (k.limit > len) k.limit = len;
  k.list = nullptr;
  k.count = k.limit;
  if (g.sel != nullptr) {
    const int32_t c = g.sel_count[n];
    if (c != -1) {
      if (c <= 0 || c > g.k_max) {
        k.count = 0;
        if (g.device_status) atomicOr(g.device_status, MLA_DEVICE_BAD_SELECTION_COUNT);
      } else {
        k.count = c;
        k.list = g.sel + (int64_t)n * g.k_max;
      }
    }
  }
  k.batch_off_lat = (int64_t)b * g.latent_batch_stride;
  k.batch_off_rope = (int64_t)b * g.rope_batch_stride;
  return k;
}

constexpr int kDecodeWarps = 4;
constexpr int kMaxD = 1280;            // rank + rope
constexpr int kMaxRank = 1024;
constexpr int kMaxRankPerLane = kMaxRank / 32;

// grid (splits, heads, n_q); 4 warps.  Split s of row n covers entries
// [s*chunk, (s+1)*chunk) of that row's key list, chunk = ceil(count/splits).
template <typename T, typename TO>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    simt_decode_kernel(const __grid_constant__ DecodeGeometry g, float* __restrict__ ws, int splits) {
  const int split = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int D = g.rank + g.rope_dim;
  __shared__ float q_s[kMaxD];
  __shared__ float m_s[kDecodeWarps], l_s[kDecodeWarps];
  __shared__ float acc_s[kDecodeWarps][kMaxRank];

  const T* qrow = static_cast<const T*>(g.q) + (int64_t)n * g.q_row_stride + (int64_t)h * g.q_head_stride;
  for (int d = threadIdx.x; d < D; d += blockDim.x) q_s[d] = to_f(qrow[d]);
  __syncthreads();

  const RowKeys rk = row_keys(g, n);
  const int chunk = (rk.count + splits - 1) / splits;
  const int lo = split * chunk;
  const int hi = min(rk.count, lo + chunk);

  const T* lat = static_cast<const T*>(g.latent) + rk.batch_off_lat;
  const T* rop = static_cast<const T*>(g.rope) + rk.batch_off_rope;

  float m = -CUDART_INF_F, l = 0.f;
  float acc[kMaxRankPerLane];
#pragma unroll
  for (int j = 0; j < kMaxRankPerLane; ++j) acc[j] = 0.f;

  for (int e = lo + warp; e < hi; e += kDecodeWarps) {
    int32_t t = e;
    if (rk.list) {
      t = rk.list[e];
      if (t < 0 || t >= rk.limit) {
        if (lane == 0 && g.device_status) atomicOr(g.device_status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
        continue;
      }
    }
    const int64_t row = (int64_t)rk.start + t;
    const T* lrow = lat + row * g.latent_row_stride;
    const T* rrow = rop + row * g.rope_row_stride;
    float c[kMaxRankPerLane];
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxRankPerLane; ++j) {
      const int d = lane + 32 * j;
      c[j] = 0.f;
      if (d < g.rank) {
        c[j] = to_f(lrow[d]);
        part = fmaf(q_s[d], c[j], part);
      }
    }
    for (int d = lane; d < g.rope_dim; d += 32) part = fmaf(q_s[g.rank + d], to_f(rrow[d]), part);
    const float s = warp_sum(part) * g.scale_log2;
    const float m_new = fmaxf(m, s);
    const float alpha = exp2f(m - m_new);
    const float pr = exp2f(s - m_new);
    l = l * alpha + pr;
#pragma unroll
    for (int j = 0; j < kMaxRankPerLane; ++j) acc[j] = fmaf(acc[j], alpha, pr * c[j]);
    m = m_new;
  }

  // Merge the warps.
  if (lane == 0) {
    m_s[warp] = m;
    l_s[warp] = l;
  }
#pragma unroll
  for (int j = 0; j < kMaxRankPerLane; ++j) {
    const int d = lane + 32 * j;
    if (d < g.rank) acc_s[warp][d] = acc[j];
  }
  __syncthreads();
  float M = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, m_s[w]);
  float wgt[kDecodeWarps];
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < kDecodeWarps; ++w) {
    wgt[w] = (m_s[w] == -CUDART_INF_F) ? 0.f : exp2f(m_s[w] - M);
    L += wgt[w] * l_s[w];
  }
  const int64_t slot = ((int64_t)n * splits + split) * g.heads + h;
  if (splits == 1) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    TO* out = static_cast<TO*>(g.ctx_out) + (int64_t)n * g.ctx_row_stride + (int64_t)h * g.ctx_head_stride;
    for (int d = threadIdx.x; d < g.rank; d += blockDim.x) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) o = fmaf(wgt[w], acc_s[w][d], o);
      out[d] = cvt<TO>(o * inv);
    }
    if (threadIdx.x == 0 && g.lse_out)
      g.lse_out[(int64_t)n * g.heads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
  } else {
    float* o_ws = ws + slot * g.rank;
    for (int d = threadIdx.x; d < g.rank; d += blockDim.x) {
      float o = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) o = fmaf(wgt[w], acc_s[w][d], o);
      o_ws[d] = o;
    }
    const int64_t nslots = (int64_t)gridDim.z * splits * g.heads;
    if (threadIdx.x == 0) {
      float* ml = ws + nslots * g.rank;
      ml[2 * slot] = (L > 0.f) ? M : -CUDART_INF_F;
      ml[2 * slot + 1] = L;
    }
  }
}

// grid (heads, n_q); merges the splits of one (row, head).
template <typename TO>
__global__ void __launch_bounds__(128)
    simt_combine_kernel(const __grid_constant__ DecodeGeometry g, const float* __restrict__ ws, int splits) {
  const int h = blockIdx.x, n = blockIdx.y;
  const int64_t nslots = (int64_t)gridDim.y * splits * g.heads;
  const float* ml = ws + nslots * g.rank;
  float M = -CUDART_INF_F;
  for (int s = 0; s < splits; ++s) {
    const int64_t slot = ((int64_t)n * splits + s) * g.heads + h;
    M = fmaxf(M, ml[2 * slot]);
  }
  float L = 0.f;
  for (int s = 0; s < splits; ++s) {
    const int64_t slot = ((int64_t)n * splits + s) * g.heads + h;
    const float ms = ml[2 * slot];
    if (ms != -CUDART_INF_F) L += exp2f(ms - M) * ml[2 * slot + 1];
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  TO* out = static_cast<TO*>(g.ctx_out) + (int64_t)n * g.ctx_row_stride + (int64_t)h * g.ctx_head_stride;
  for (int d = threadIdx.x; d < g.rank; d += blockDim.x) {
    float o = 0.f;
    for (int s = 0; s < splits; ++s) {
      const int64_t slot = ((int64_t)n * splits + s) * g.heads + h;
      const float ms = ml[2 * slot];
      if (ms != -CUDART_INF_F) o = fmaf(exp2f(ms - M), ws[slot * g.rank + d], o);
    }
    out[d] = cvt<TO>(o * inv);
  }
  if (threadIdx.x == 0 && g.lse_out)
    g.lse_out[(int64_t)n * g.heads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
}

// ---------------------------------------------------------------- absorption
// grid (ceil(rank/128), heads, ceil(n_q/32)); thread = latent column.
template <typename T>
__global__ void __launch_bounds__(128) simt_absorb_kernel(const __grid_constant__ AbsorbParams p) {
  constexpr int kRows = 32;
  const int r = blockIdx.x * 128 + threadIdx.x;
  const int h = blockIdx.y;
  const int n0 = blockIdx.z * kRows;
  const int nr = min(kRows, p.n_q - n0);
  extern __shared__ float qs[];  // [kRows][nope]
  const T* q = static_cast<const T*>(p.q_nope);
  for (int e = threadIdx.x; e < nr * p.nope; e += blockDim.x) {
    const int nn = e / p.nope, k = e % p.nope;
    qs[nn * p.nope + k] = to_f(q[(int64_t)(n0 + nn) * p.q_row_stride + (int64_t)h * p.q_head_stride + k]);
  }
  __syncthreads();
  if (r >= p.rank) return;
  float acc[kRows];
#pragma unroll
  for (int j = 0; j < kRows; ++j) acc[j] = 0.f;
  const T* w = static_cast<const T*>(p.w) + (int64_t)h * (p.nope + p.v_dim) * p.rank + r;
  for (int k = 0; k < p.nope; ++k) {
    const float wk = to_f(w[(int64_t)k * p.rank]);
#pragma unroll
    for (int j = 0; j < kRows; ++j) acc[j] = fmaf(qs[j * p.nope + k], wk, acc[j]);
  }
  T* out = static_cast<T*>(p.out);
#pragma unroll
  for (int j = 0; j < kRows; ++j)
    if (j < nr) out[(int64_t)(n0 + j) * p.out_row_stride + (int64_t)h * p.out_head_stride + r] = cvt<T>(acc[j]);
}

// ---------------------------------------------------------------- value projection
// grid (heads, ceil(n_q/8)); 8 warps; warp = output column j (strided), lanes over rank.
template <typename T, typename TO>
__global__ void __launch_bounds__(256) simt_project_kernel(const __grid_constant__ ProjectParams p) {
  constexpr int kRows = 8;
  const int h = blockIdx.x;
  const int n0 = blockIdx.y * kRows;
  const int nr = min(kRows, p.n_q - n0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  extern __shared__ float cs[];  // [kRows][rank]
  const T* ctx = static_cast<const T*>(p.ctx);
  for (int e = threadIdx.x; e < nr * p.rank; e += blockDim.x) {
    const int nn = e / p.rank, c = e % p.rank;
    cs[nn * p.rank + c] = to_f(ctx[(int64_t)(n0 + nn) * p.ctx_row_stride + (int64_t)h * p.ctx_head_stride + c]);
  }
  __syncthreads();
  const T* wv = static_cast<const T*>(p.w) + ((int64_t)h * (p.nope + p.v_dim) + p.nope) * p.rank;
  TO* out = static_cast<TO*>(p.out);
  for (int j = warp; j < p.v_dim; j += 8) {
    float acc[kRows];
#pragma unroll
    for (int t = 0; t < kRows; ++t) acc[t] = 0.f;
    for (int c = lane; c < p.rank; c += 32) {
      const float wc = to_f(wv[(int64_t)j * p.rank + c]);
#pragma unroll
      for (int t = 0; t < kRows; ++t) acc[t] = fmaf(cs[t * p.rank + c], wc, acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kRows; ++t) {
      const float s = warp_sum(acc[t]);
      if (lane == 0 && t < nr) out[(int64_t)(n0 + t) * p.out_row_stride + (int64_t)h * p.v_dim + j] = cvt<TO>(s);
    }
  }
}

// ---------------------------------------------------------------- gather hook
// grid (ceil(k_max/8), n_q); warp per output slot; raw element copies.
template <typename T>
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ DecodeGeometry g, T* __restrict__ out) {
  const int n = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (j >= g.k_max) return;
  const RowKeys rk = row_keys(g, n);
  const int D = g.rank + g.rope_dim;
  T* dst = out + ((int64_t)n * g.k_max + j) * D;
  bool ok = j < rk.count;
  int32_t t = j;
  if (ok && rk.list) {
    t = rk.list[j];
    if (t < 0 || t >= rk.limit) {
      ok = false;
      if (lane == 0 && g.device_status) atomicOr(g.device_status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
    }
  }
  if (!ok) {
    for (int d = lane; d < D; d += 32) dst[d] = T();
    return;
  }
  const int64_t row = (int64_t)rk.start + t;
  const T* lrow = static_cast<const T*>(g.latent) + rk.batch_off_lat + row * g.latent_row_stride;
  const T* rrow = static_cast<const T*>(g.rope) + rk.batch_off_rope + row * g.rope_row_stride;
  for (int d = lane; d < g.rank; d += 32) dst[d] = lrow[d];
  for (int d = lane; d < g.rope_dim; d += 32) dst[g.rank + d] = rrow[d];
}

int simt_splits(const DecodeGeometry& g) {
  // Enough blocks to fill the GPU a few times over, at least ~128 keys each.
  const int64_t keys = g.sel ? (int64_t)g.k_max : g.t_max;
  const int64_t blocks = (int64_t)g.batch * g.s_q * g.heads;
  const int64_t want = (4LL * device_sm_count() + blocks - 1) / blocks;
  int64_t by_len = (keys + 127) / 128;
  int64_t s = want < by_len ? want : by_len;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return (int)s;
}

}  // namespace

size_t simt_decode_workspace(const DecodeGeometry& g, int* splits_out) {
  const int s = simt_splits(g);
  if (splits_out) *splits_out = s;
  if (s == 1) return 0;
  const size_t slots = (size_t)g.batch * g.s_q * s * g.heads;
  return slots * ((size_t)g.rank + 2) * sizeof(float);
}

cudaError_t launch_simt_decode(const DecodeGeometry& g, int dtype, int out_dtype, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  int splits = 1;
  const size_t need = simt_decode_workspace(g, &splits);
  if (workspace_bytes < need) return cudaErrorInvalidValue;
  const int n_q = g.batch * g.s_q;
  dim3 grid(splits, g.heads, n_q);
  float* ws = static_cast<float*>(workspace);
#define MLA_SIMT_DECODE(T, TO)                                                       \
  simt_decode_kernel<T, TO><<<grid, kDecodeWarps * 32, 0, stream>>>(g, ws, splits); \
  if (splits > 1) simt_combine_kernel<TO><<<dim3(g.heads, n_q), 128, 0, stream>>>(g, ws, splits);
  if (dtype != MLA_DTYPE_F32) return cudaErrorInvalidValue;
  if (out_dtype == MLA_DTYPE_F32) { MLA_SIMT_DECODE(float, float) } else { MLA_SIMT_DECODE(float, __nv_bfloat16) }
#undef MLA_SIMT_DECODE
  return cudaGetLastError();
}

cudaError_t launch_simt_absorb(const AbsorbParams& p, int dtype, cudaStream_t stream) {
  dim3 grid((p.rank + 127) / 128, p.heads, (p.n_q + 31) / 32);
  const size_t smem = 32 * (size_t)p.nope * sizeof(float);
  if (dtype != MLA_DTYPE_F32) return cudaErrorInvalidValue;
  simt_absorb_kernel<float><<<grid, 128, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_simt_project(const ProjectParams& p, int dtype, int out_dtype, cudaStream_t stream) {
  dim3 grid(p.heads, (p.n_q + 7) / 8);
  const size_t smem = 8 * (size_t)p.rank * sizeof(float);
  if (dtype != MLA_DTYPE_F32) return cudaErrorInvalidValue;
  if (out_dtype == MLA_DTYPE_F32)
    simt_project_kernel<float, float><<<grid, 256, smem, stream>>>(p);
  else
    simt_project_kernel<float, __nv_bfloat16><<<grid, 256, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const DecodeGeometry& g, int dtype, void* out, cudaStream_t stream) {
  dim3 grid((g.k_max + 7) / 8, g.batch * g.s_q);
  if (dtype == MLA_DTYPE_F32)
    gather_kernel<float><<<grid, 256, 0, stream>>>(g, static_cast<float*>(out));
  else
    gather_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(g, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace mla
