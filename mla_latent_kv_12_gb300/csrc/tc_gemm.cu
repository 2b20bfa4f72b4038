// Tensor-core (tcgen05) kernels of the two per-head projections around the
// latent attention ("glm52-mla.ts", Glm52Mla.attendAbsorbed):
//
//   absorb:  q_lat[n, h, :]  = q_nope[n, h, :] @ W_UK_h        ([n_q,128] x [128,512])
//   project: out[n, h*v + j] = ctx[n, h, :] . W_UV_h[j, :]     ([n_q,512] x [512,128])
//
// Both are weight-read bound at decode sizes (n_q <= 64): each CTA streams one
// head's weight slice once with TMA and puts the weight on the MMA's M side
// (swap-AB), so the few query rows become the N dimension (padded to 16).
// Larger batches are cut into blocks of query rows (256 for the absorb, 64
// for the projection), one more grid dimension; each block re-reads the
// weight slice, from L2 after the first.
// Accumulation is f32 in TMEM; one warp quarter reads back 32 rows each.
#include <cuda_bf16.h>
#include <string.h>

#include "mla_internal.h"
#include "rope_math.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mla {
namespace {

using namespace tc;

constexpr long long kWaitLimit = 1LL << 32;  // clock cycles (~2 s)

__device__ __forceinline__ void flag_timeout(int32_t* status) {
  if (status) atomicOr(status, MLA_DEVICE_TIMEOUT);
}

// ------------------------------------------------------------------ absorb
// grid (rank/128, heads, row blocks); 128 threads.  A = W_UK_h^T tile [128 latent x 128 nope]
// (MN-major: latent contiguous in kv_b_proj rows), B = q_nope rows of head h
// [npad x 128] (K-major).  D [128 latent x npad] f32 in TMEM.
struct AbsorbArgs {
  void* out;
  int64_t out_row_stride, out_head_stride;
  int32_t n_q, npad;     // npad: query rows per block (the MMA's N), a multiple of 16
  int32_t w_head_rows;  // W_UK_h starts at row h*w_head_rows
  int32_t* status;
  int32_t with_rope;    // CTAs of blockIdx.x == 0 also rotate q_rope of head h
  AbsorbRope rope;
};

__global__ void __launch_bounds__(128) tc_absorb_kernel(const __grid_constant__ CUtensorMap wmap,
                                                        const __grid_constant__ CUtensorMap qmap,
                                                        const __grid_constant__ AbsorbArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                       // 2 boxes x [128 k][64 m] = 32 KB
  uint8_t* sB = smem + 32768;               // 2 boxes x [npad n][64 k]
  __shared__ __align__(8) uint64_t bar_full, bar_mma;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * 128, h = blockIdx.y;
  const int npad = a.npad;
  const int row0 = blockIdx.z * npad;   // first query row of this block
  const uint32_t ncols = npad <= 32 ? 32 : (npad <= 64 ? 64 : (npad <= 128 ? 128 : 256));

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&qmap);
    mbar_init(&bar_full, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  bool ok = true;
  pdl_wait();
  // Dependants may launch now: they wait for this grid before reading its
  // output, and the decode kernel's CTAs (a whole SM each) start on the SMs
  // these CTAs leave, overlapping their prologue with this grid's tail.
  pdl_trigger();

  if (threadIdx.x == 0) {
    const uint32_t bytes = 2 * 16384 + 2 * npad * 128;
    mbar_arrive_expect_tx(&bar_full, bytes);
    tma_load_2d(sA, &wmap, &bar_full, m0, h * a.w_head_rows);
    tma_load_2d(sA + 16384, &wmap, &bar_full, m0 + 64, h * a.w_head_rows);
    tma_load_3d(sB, &qmap, &bar_full, 0, h, row0);               // rows past n_q load as zeros
    tma_load_3d(sB + npad * 128, &qmap, &bar_full, 64, h, row0);
    ok = mbar_wait(&bar_full, 0, kWaitLimit);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, npad, 1, 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t ad = smem_desc(a0 + k * 2048, 16384, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(b0 + (k >> 2) * npad * 128 + (k & 3) * 32, 16, 1024, kSwizzle128B);
        mma_ss(tmem, ad, bd, idesc, k > 0);
      }
      mma_commit(&bar_mma);
    } else {
      flag_timeout(a.status);
      mma_commit(&bar_mma);
    }
  }
  __syncwarp();
  if (a.with_rope && blockIdx.x == 0) {
    // While the MMAs run: RoPE of head h's rope part, lane j = rotary pair j,
    // warp w = query rows w, w+4, ...
    const AbsorbRope& r = a.rope;
    const int row_end = min(a.n_q, row0 + npad);
    for (int n = row0 + warp; n < row_end; n += 4) {
      const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(r.q_rope) + (int64_t)n * r.row_stride +
                                 (int64_t)h * r.head_stride;
      const __nv_bfloat162 ab = reinterpret_cast<const __nv_bfloat162*>(src)[lane];
      const int b = n / r.s_q, i = n % r.s_q;
      const int64_t pos = (r.row_offsets ? (int64_t)r.row_offsets[b] : r.position_offset) + i;
      float re, im;
      rope_rotate_pair(__low2float(ab), __high2float(ab), pos, r.inv_freq[lane], re, im);
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (int64_t)n * a.out_row_stride +
                           (int64_t)h * a.out_head_stride + r.out_col;
      dst[lane] = __float2bfloat16_rn(re);
      dst[32 + lane] = __float2bfloat16_rn(im);
    }
  }
  ok = mbar_wait_warp(&bar_mma, 0, kWaitLimit);   // warp-uniform: the epilogue's TMEM loads are collective
  if (!ok && lane == 0) flag_timeout(a.status);
  tc_fence_after();
  if (ok) {
    const uint32_t row_addr = tmem + ((uint32_t)(32 * warp) << 16);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)h * a.out_head_stride + m0 + 32 * warp + lane;
    for (int c0 = 0; c0 < npad; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = row0 + c0 + j;
        if (n < a.n_q) out[(int64_t)n * a.out_row_stride] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

// ------------------------------------------------------------------ project
// grid (heads, row blocks); 128 threads.  A = W_UV_h [128 v x 512 latent] (K-major),
// B = ctx rows of head h [npad x 512] (K-major).  8 K-boxes of 64, one
// barrier each so the MMAs start as soon as the first box lands.
struct ProjectArgs {
  void* out;
  int64_t out_row_stride;
  int32_t n_q, npad, v_dim;
  int32_t w_row0, w_head_rows;  // W_UV_h starts at row h*w_head_rows + w_row0
  int32_t out_f32;
  int32_t* status;
};

__global__ void __launch_bounds__(128) tc_project_kernel(const __grid_constant__ CUtensorMap wmap,
                                                         const __grid_constant__ CUtensorMap cmap,
                                                         const __grid_constant__ ProjectArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                 // 8 x [128 rows][64] = 128 KB
  uint8_t* sB = smem + 8 * 16384;     // 8 x [npad rows][64]
  __shared__ __align__(8) uint64_t bar_full[8];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int npad = a.npad;
  const int qrow0 = blockIdx.y * npad;   // first query row of this block
  const uint32_t ncols = npad <= 32 ? 32 : 64;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&cmap);
    for (int i = 0; i < 8; ++i) mbar_init(&bar_full[i], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  bool ok = true;
  pdl_wait();

  if (threadIdx.x == 0) {
    const int row0 = h * a.w_head_rows + a.w_row0;  // first row of W_UV_h in kv_b_proj
    for (int i = 0; i < 8; ++i) {
      mbar_arrive_expect_tx(&bar_full[i], 16384 + npad * 128);
      tma_load_2d(sA + i * 16384, &wmap, &bar_full[i], 64 * i, row0);
      tma_load_3d(sB + i * npad * 128, &cmap, &bar_full[i], 64 * i, h, qrow0);   // rows past n_q: zeros
    }
    const uint32_t idesc = idesc_bf16_f32(128, npad, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int i = 0; i < 8 && ok; ++i) {
      ok = mbar_wait(&bar_full[i], 0, kWaitLimit);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = smem_desc(a0 + i * 16384 + k * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(b0 + i * npad * 128 + k * 32, 16, 1024, kSwizzle128B);
        mma_ss(tmem, ad, bd, idesc, (i | k) != 0);
      }
    }
    if (!ok) {
      flag_timeout(a.status);
      for (int i = 0; i < 8; ++i) mbar_wait(&bar_full[i], 0, kWaitLimit);  // drain in-flight copies
    }
    mma_commit(&bar_mma);
  }
  __syncwarp();
  // warp-uniform (the epilogue's TMEM loads are collective); thread 0's own
  // result joins through the barrier wait of warp 0
  ok = __all_sync(0xffffffffu, mbar_wait(&bar_mma, 0, kWaitLimit) && ok);
  tc_fence_after();
  if (ok) {
    const uint32_t row_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const int j = 32 * warp + lane;
    for (int c0 = 0; c0 < npad; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int n = qrow0 + c0 + t;
        if (n >= a.n_q) continue;
        const float v = __uint_as_float(r[t]);
        const int64_t off = (int64_t)n * a.out_row_stride + (int64_t)h * a.v_dim + j;
        if (a.out_f32)
          static_cast<float*>(a.out)[off] = v;
        else
          static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(v);
      }
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

int pad16(int n) { return (n + 15) & ~15; }

}  // namespace

constexpr int kAbsorbBlockRows = 256, kProjectBlockRows = 64;

cudaError_t launch_tc_absorb(const AbsorbParams& p, cudaStream_t stream, const AbsorbRope* rope) {
  const int npad = p.n_q > kAbsorbBlockRows ? kAbsorbBlockRows : pad16(p.n_q);
  const int nblk = (p.n_q + npad - 1) / npad;
  CUtensorMap wmap, qmap;
  {
    const uint64_t dims[2] = {(uint64_t)p.rank, (uint64_t)p.heads * (p.nope + p.v_dim)};
    const uint64_t strides[1] = {(uint64_t)p.rank * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap_bf16(&wmap, p.w, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.nope, (uint64_t)p.heads, (uint64_t)p.n_q};
    const uint64_t strides[2] = {(uint64_t)p.q_head_stride * 2, (uint64_t)(p.q_row_stride ? p.q_row_stride : 8) * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)npad};
    if (!encode_tmap_bf16(&qmap, p.q_nope, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  AbsorbArgs a;
  memset(&a, 0, sizeof(a));
  a.out = p.out;
  a.out_row_stride = p.out_row_stride;
  a.out_head_stride = p.out_head_stride;
  a.n_q = p.n_q;
  a.npad = npad;
  a.w_head_rows = p.nope + p.v_dim;
  if (rope) {
    a.with_rope = 1;
    a.rope = *rope;
  }
  const size_t smem = 1024 + 32768 + 2 * (size_t)npad * 128;
  {
    const cudaError_t ea = set_max_dynamic_smem(tc_absorb_kernel, (int)(1024 + 32768 + 2 * 256 * 128));
    if (ea != cudaSuccess) return ea;
  }
  const cudaError_t e =
      launch_pdl(tc_absorb_kernel, dim3(p.rank / 128, p.heads, nblk), dim3(128), smem, stream, wmap, qmap, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_tc_project(const ProjectParams& p, int out_dtype, cudaStream_t stream) {
  const int npad = p.n_q > kProjectBlockRows ? kProjectBlockRows : pad16(p.n_q);
  const int nblk = (p.n_q + npad - 1) / npad;
  CUtensorMap wmap, cmap;
  {
    const uint64_t dims[2] = {(uint64_t)p.rank, (uint64_t)p.heads * (p.nope + p.v_dim)};
    const uint64_t strides[1] = {(uint64_t)p.rank * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap_bf16(&wmap, p.w, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.rank, (uint64_t)p.heads, (uint64_t)p.n_q};
    const uint64_t strides[2] = {(uint64_t)p.ctx_head_stride * 2,
                                 (uint64_t)(p.ctx_row_stride ? p.ctx_row_stride : 8) * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)npad};
    if (!encode_tmap_bf16(&cmap, p.ctx, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  ProjectArgs a{p.out, p.out_row_stride, p.n_q, npad, p.v_dim, p.nope, p.nope + p.v_dim,
                out_dtype == MLA_DTYPE_F32 ? 1 : 0, nullptr};
  const size_t smem = 1024 + 8 * 16384 + 8 * (size_t)npad * 128;
  {
    const cudaError_t ea = set_max_dynamic_smem(tc_project_kernel, (int)(1024 + 8 * 16384 + 8 * 64 * 128));
    if (ea != cudaSuccess) return ea;
  }
  const cudaError_t e = launch_pdl(tc_project_kernel, dim3(p.heads, nblk), dim3(128), smem, stream, wmap, cmap, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
