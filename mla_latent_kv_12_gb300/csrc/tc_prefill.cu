// Reconstructed prefill attention on tcgen05 ("glm52-mla.ts",
// Glm52Mla.attendReconstructed, with the left-pad mask of the 0.2.0 -> 0.4.0
// hunk): for a long block of new tokens the per-head keys and values are
// materialised once and attention runs in its plain form, which costs
// 2*H*(nope+rope+v) flops per (query, key) pair instead of the absorbed
// form's 2*H*(2*rank+rope).
//
//   tc_reconstruct_kernel  K_nope[t,h,:] = latent[t,:] . W_UK_h^T,
//                          V[t,h,:]      = latent[t,:] . W_UV_h^T
//     persistent (one CTA per SM over (128-row tile, head) tiles): per tile
//     one tcgen05 MMA chain M=128 tokens x N=256 (head h's 256 rows of
//     kv_b_proj) x K=rank, fed by a 4-stage TMA ring, into one of two TMEM
//     accumulators; the epilogue warps round the other accumulator to bf16
//     into swizzled shared memory (half a tile at a time) and write it with
//     TMA tensor stores.
//
//   tc_prefill_kernel      causal flash attention, one CTA per (128 query
//     rows, head, batch row).  Q (nope || rotated rope, 192 features) stays
//     in shared memory; each 128-key tile brings K_nope and the cache's
//     shared rope key (one ring, freed when the tile's scores are done) and V
//     (a second ring, freed when its P.V is done) by TMA.  Warp 1 issues
//     S(j+1) = Q.K^T into one of two TMEM score buffers while eight softmax
//     warps (two per quarter of the query rows, 64 score columns each) turn
//     S(j) into bf16 P (two TMEM buffers of their own); then it issues
//     O += P.V with P read from TMEM.  The running maximum is only moved when
//     it grows by more than 2^8 (the accumulated O and sum are then rescaled
//     in TMEM), so most tiles skip the correction.
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include "mla_internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mla {
namespace {

using namespace tc;

constexpr long long kWaitLimit = 1LL << 32;  // clock cycles (~2 s)
constexpr int kChunk = 128 * 128;            // 128 rows x 64 bf16 (one 128-byte swizzle atom column)

__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Offset of 16-byte unit u of row r in a 128-byte-swizzled chunk.
__device__ __forceinline__ uint32_t sw128(int r, int u) { return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4)); }

// ------------------------------------------------------------------ reconstruct

constexpr int RC_STAGES = 4;
constexpr int RC_A_BYTES = kChunk;          // 128 tokens x 64 latent features
constexpr int RC_B_BYTES = 2 * kChunk;      // 256 weight rows x 64 latent features
constexpr int RC_STAGE_BYTES = RC_A_BYTES + RC_B_BYTES;
constexpr int RC_OUT_BYTES = 2 * kChunk;    // half a tile's bf16 output (K_nope, then V): 2 chunks
constexpr int RC_SMEM = 1024 + RC_STAGES * RC_STAGE_BYTES + RC_OUT_BYTES;
constexpr int RC_THREADS = 192;             // producer, MMA issuer, 4 epilogue warps

struct ReconArgs {
  int32_t k_chunks;     // rank / 64
  int32_t head_rows;    // nope + v rows of kv_b_proj per head
  int32_t row_tiles;    // 128-row tiles
  int32_t n_tiles;      // row_tiles * heads (tile = row tile fastest, then head)
  int32_t* status;
};

// Persistent: CTA c takes tiles c, c + grid, ...  Two TMEM accumulators of
// 256 columns: the epilogue of one tile runs under the MMAs of the next.
__global__ void __launch_bounds__(RC_THREADS, 1)
    tc_reconstruct_kernel(const __grid_constant__ CUtensorMap lat_map, const __grid_constant__ CUtensorMap w_map,
                          const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                          const __grid_constant__ ReconArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_s = smem + RC_STAGES * RC_STAGE_BYTES;
  __shared__ __align__(8) uint64_t full_bar[RC_STAGES], empty_bar[RC_STAGES], acc_full[2], acc_empty[2], mma_drain;
  __shared__ uint32_t tmem_s;
  __shared__ volatile int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&lat_map);
    tma_prefetch_desc(&w_map);
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&v_map);
    for (int s = 0; s < RC_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&acc_full[q], 1);
      mbar_init(&acc_empty[q], 128);
    }
    mbar_init(&mma_drain, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  auto fail = [&]() {
    abort_s = 1;
    if (a.status) atomicOr(a.status, MLA_DEVICE_TIMEOUT);
  };
  const int n_mine = a.n_tiles > (int)blockIdx.x ? (a.n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: every k-chunk of every tile
    bool issued[RC_STAGES] = {};
    uint32_t issued_phase[RC_STAGES] = {};
    if (lane == 0) {
      int q = 0;
      for (int it = 0; it < n_mine && !abort_s; ++it) {
        const int tile = (int)blockIdx.x + it * (int)gridDim.x;
        const int row0 = (tile % a.row_tiles) * 128, h = tile / a.row_tiles;
        for (int kc = 0; kc < a.k_chunks && !abort_s; ++kc, ++q) {
          const int s = q % RC_STAGES;
          const uint32_t ph = (uint32_t)(q / RC_STAGES) & 1u;
          if (q >= RC_STAGES && !mbar_wait(&empty_bar[s], ph ^ 1u, kWaitLimit)) { fail(); break; }
          uint8_t* st = smem + s * RC_STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[s], RC_STAGE_BYTES);
          tma_load_2d(st, &lat_map, &full_bar[s], kc * 64, row0);
          tma_load_2d(st + RC_A_BYTES, &w_map, &full_bar[s], kc * 64, h * a.head_rows);
          issued[s] = true;
          issued_phase[s] = ph;
        }
      }
      for (int s = 0; s < RC_STAGES; ++s)
        if (issued[s]) mbar_wait(&full_bar[s], issued_phase[s], kWaitLimit);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, 256, 0, 0);
    const uint64_t desc0 = smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
    bool ok = true;
    int q = 0;
    for (int it = 0; ok && it < n_mine; ++it) {
      const int acc = it & 1;
      // The epilogue has read this accumulator's previous tile.
      if (it >= 2 && !mbar_wait_warp(&acc_empty[acc], (uint32_t)((it >> 1) - 1) & 1u, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      for (int kc = 0; kc < a.k_chunks; ++kc, ++q) {
        const int s = q % RC_STAGES;
        if (!mbar_wait_warp(&full_bar[s], (uint32_t)(q / RC_STAGES) & 1u, kWaitLimit)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = desc0 + (uint64_t)(s * (RC_STAGE_BYTES >> 4));
        const uint64_t bd = ad + (uint64_t)(RC_A_BYTES >> 4);
        const uint32_t first = kc == 0 ? 0u : 1u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + (uint32_t)(acc * 256), ad + (uint64_t)((k * 32) >> 4), bd + (uint64_t)((k * 32) >> 4),
                   idesc, k == 0 ? first : 1u);
          mma_commit(&empty_bar[s]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&acc_full[acc]);
      __syncwarp();
      if (abort_s) ok = false;
    }
    if (!ok) fail();
    if (elect_one()) mma_commit(&mma_drain);
    __syncwarp();
    mbar_wait_warp(&mma_drain, 0, kWaitLimit);
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;                     // token row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool issuer = warp == 2 && lane == 0;
    for (int it = 0; it < n_mine; ++it) {
      const int acc = it & 1;
      const int tile = (int)blockIdx.x + it * (int)gridDim.x;
      const int row0 = (tile % a.row_tiles) * 128, h = tile / a.row_tiles;
      const bool ok = mbar_wait_warp(&acc_full[acc], (uint32_t)(it >> 1) & 1u, kWaitLimit);
      if (!ok) fail();
      // The previous tile's stores have read the staging buffer.
      if (issuer) bulk_wait_read();
      // One decision for all four warps, so that none waits at a barrier the
      // others have left.
      if (named_sync_or(1, 128, !ok || abort_s)) break;
      tc_fence_after();
      // Two halves through one 32 KB staging buffer: K_nope (accumulator
      // columns 0..127), then V (128..255), each as two 64-feature chunks.
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        if (half == 1) {
          if (issuer) bulk_wait_read();       // the K_nope stores have read the buffer
          named_sync(1, 128);
        }
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
          uint32_t v[32];
          tmem_ld32(tmem + (uint32_t)(acc * 256 + half * 128 + p * 32) + lane_off, v);
          tmem_wait_ld_regs(v);
          uint8_t* chunk = out_s + (p >> 1) * kChunk;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
            w.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
            w.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
            w.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
            *reinterpret_cast<uint4*>(chunk + sw128(r, (p & 1) * 4 + u)) = w;
          }
        }
        if (half == 1) {
          // The accumulator may take the next tile once every lane's loads are done.
          tc_fence_before();
          mbar_arrive(&acc_empty[acc]);
        }
        fence_proxy_async_smem();
        named_sync(1, 128);
        if (issuer) {
          const CUtensorMap* map = half == 0 ? &k_map : &v_map;
          tma_store_3d(map, out_s, 0, h, row0);
          tma_store_3d(map, out_s + kChunk, 64, h, row0);
          bulk_commit();
        }
      }
    }
    if (issuer) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ prefill attention

constexpr int PF_STAGES = 2;                  // per ring
constexpr int PF_Q_BYTES = 3 * kChunk;        // Q tile: nope 0..63 | nope 64..127 | rope
constexpr int PF_K_BYTES = 3 * kChunk;        // K_nope x2 | rope  (freed when S completes)
constexpr int PF_V_BYTES = 2 * kChunk;        // V x2              (freed when P.V completes)
constexpr int PF_SMEM = 1024 + PF_Q_BYTES + PF_STAGES * (PF_K_BYTES + PF_V_BYTES);
constexpr int PF_THREADS = 352;               // K producer, MMA, 8 softmax warps, V producer
constexpr uint32_t PF_TM_O = 256;             // TMEM: S0 at 0, S1 at 128, O at 256, P0 at 384, P1 at 448
constexpr uint32_t PF_TM_P = 384;             // 128 keys of bf16 P = 64 columns per buffer
constexpr float kRescaleLog2 = 8.f;

struct PrefillArgs {
  const int32_t* kv_start;
  const int32_t* kv_len;
  int64_t t_max;         // buffer rows of one batch row (the packed buffer's rows when packed)
  int32_t packed;        // all batch rows share one buffer row range
  int32_t batch, s_q, n_qtiles;
  float scale_log2;      // softmax scale * log2(e)
  void* out;
  int64_t out_row_stride;
  int32_t v_dim, out_f32;
  float* lse;
  int32_t* status;
};

__global__ void __launch_bounds__(PF_THREADS, 1)
    tc_prefill_kernel(const __grid_constant__ CUtensorMap qn_map, const __grid_constant__ CUtensorMap qr_map,
                      const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap r_map,
                      const __grid_constant__ CUtensorMap v_map, const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;
  uint8_t* k_ring = smem + PF_Q_BYTES;
  uint8_t* v_ring = k_ring + PF_STAGES * PF_K_BYTES;
  __shared__ __align__(8) uint64_t q_full, k_full[PF_STAGES], k_empty[PF_STAGES], v_full[PF_STAGES],
      v_empty[PF_STAGES], s_full[2], p_full, pv_done, mma_drain, xbar[2][4], lbar[4];
  __shared__ float red_max[2][2][128], red_sum[2][128];
  __shared__ uint32_t tmem_s;
  __shared__ volatile int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = a.n_qtiles - 1 - (int)blockIdx.x;       // longest causal rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int i0 = qt * 128;

  const int64_t start = a.kv_start[b], len = a.kv_len[b];
  if (start < 0 || len < 0 || start + len > a.t_max) {
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
    return;
  }
  // Token i of the block sits at window position len - s_q + i and sees the
  // keys at or before it.
  const int64_t offs = len - a.s_q;
  const int64_t i_hi = min((int64_t)i0 + 127, (int64_t)a.s_q - 1);
  const int64_t key_end = min(len, offs + i_hi + 1);
  const int n_kt = key_end > 0 ? (int)((key_end + 127) / 128) : 0;
  const int64_t ybase = (a.packed ? 0 : (int64_t)b * a.t_max) + start;
  const int q_row0 = b * a.s_q + i0;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&qn_map);
    tma_prefetch_desc(&qr_map);
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&r_map);
    tma_prefetch_desc(&v_map);
    mbar_init(&q_full, 1);
    for (int s = 0; s < PF_STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&p_full, 256);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&xbar[0][q], 64);
      mbar_init(&xbar[1][q], 64);
      mbar_init(&lbar[q], 64);
    }
    mbar_init(&pv_done, 1);
    mbar_init(&mma_drain, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  auto fail = [&]() {
    abort_s = 1;
    if (a.status) atomicOr(a.status, MLA_DEVICE_TIMEOUT);
  };
  auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, abort_s != 0); };

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------ TMA producers: warp 0 Q and the
    // K ring (K_nope, rope), warp 10 the V ring; each stage is refilled as soon as
    // its consumer MMA completes.
    const bool kside = warp == 0;
    uint64_t* fullb = kside ? k_full : v_full;
    uint64_t* emptyb = kside ? k_empty : v_empty;
    bool issued[PF_STAGES] = {};
    uint32_t issued_phase[PF_STAGES] = {};
    bool q_issued = false;
    if (lane == 0 && n_kt > 0) {
      if (kside) {
        mbar_arrive_expect_tx(&q_full, PF_Q_BYTES);
        tma_load_3d(q_s, &qn_map, &q_full, 0, h, q_row0);
        tma_load_3d(q_s + kChunk, &qn_map, &q_full, 64, h, q_row0);
        tma_load_3d(q_s + 2 * kChunk, &qr_map, &q_full, 0, h, q_row0);
        q_issued = true;
      }
      for (int kt = 0; kt < n_kt && !abort_s; ++kt) {
        const int s = kt % PF_STAGES;
        const uint32_t ph = (uint32_t)(kt / PF_STAGES) & 1u;
        if (kt >= PF_STAGES && !mbar_wait(&emptyb[s], ph ^ 1u, kWaitLimit)) { fail(); break; }
        const int y = (int)(ybase + (int64_t)kt * 128);
        if (kside) {
          uint8_t* st = k_ring + s * PF_K_BYTES;
          mbar_arrive_expect_tx(&fullb[s], PF_K_BYTES);
          tma_load_3d(st, &k_map, &fullb[s], 0, h, y);
          tma_load_3d(st + kChunk, &k_map, &fullb[s], 64, h, y);
          tma_load_2d(st + 2 * kChunk, &r_map, &fullb[s], 0, y);
        } else {
          uint8_t* st = v_ring + s * PF_V_BYTES;
          mbar_arrive_expect_tx(&fullb[s], PF_V_BYTES);
          tma_load_3d(st, &v_map, &fullb[s], 0, h, y);
          tma_load_3d(st + kChunk, &v_map, &fullb[s], 64, h, y);
        }
        issued[s] = true;
        issued_phase[s] = ph;
      }
      // Every issued copy lands before the CTA may exit.
      if (q_issued) mbar_wait(&q_full, 0, kWaitLimit);
      for (int s = 0; s < PF_STAGES; ++s)
        if (issued[s]) mbar_wait(&fullb[s], issued_phase[s], kWaitLimit);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
    const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);
    // Stage s's descriptors are the base's plus s stage sizes (16-byte units).
    const uint64_t kdesc0 = smem_desc(smem_u32(k_ring), 16, 1024, kSwizzle128B);
    const uint64_t qdesc = smem_desc(smem_u32(q_s), 16, 1024, kSwizzle128B);
    const uint64_t vdesc0 = smem_desc(smem_u32(v_ring), kChunk, 1024, kSwizzle128B);
    auto issue_s = [&](int j) -> bool {
      const int s = j % PF_STAGES;
      if (!mbar_wait_warp(&k_full[s], (uint32_t)(j / PF_STAGES) & 1u, kWaitLimit)) return false;
      tc_fence_after();
      // A = the Q tile, B = the K tile, both in shared memory.  Issued by one
      // elected lane of the converged warp with descriptors that differ from
      // a base by constants: the tensor core then accepts an M=128 N=128 MMA
      // about every 68 cycles (a lane-0 branch with per-MMA descriptor
      // arithmetic issues at roughly half that rate).
      const uint64_t kd = kdesc0 + (uint64_t)(s * (PF_K_BYTES >> 4));
      const uint32_t d_s = tmem + (uint32_t)((j & 1) * 128);
      if (elect_one()) {
#pragma unroll
        for (int c = 0; c < 3; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(d_s, qdesc + (uint64_t)((c * kChunk + k * 32) >> 4),
                   kd + (uint64_t)((c * kChunk + k * 32) >> 4), idesc_s, (c | k) != 0);
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[s]);
      }
      __syncwarp();
      return true;
    };
    bool ok = n_kt == 0 || mbar_wait_warp(&q_full, 0, kWaitLimit);
    if (ok && n_kt > 0) ok = issue_s(0);
    for (int j = 0; ok && j < n_kt; ++j) {
      if (j + 1 < n_kt && !issue_s(j + 1)) { ok = false; break; }
      const int s = j % PF_STAGES;
      if (!mbar_wait_warp(&v_full[s], (uint32_t)(j / PF_STAGES) & 1u, kWaitLimit)) { ok = false; break; }
      uint8_t* st = v_ring + s * PF_V_BYTES;
      const int64_t valid = len - (int64_t)j * 128;
      if (valid < 128) {
        // Tail tile: clear the V rows past the window, so that P = 0 never
        // meets a non-finite value of rows this call does not own.
        const int v0 = valid < 0 ? 0 : (int)valid;
        for (int q = lane; q < (128 - v0) * 16; q += 32) {
          const int c = q / ((128 - v0) * 8), rem = q % ((128 - v0) * 8);
          *reinterpret_cast<uint4*>(st + c * kChunk + (v0 + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!mbar_wait_warp(&p_full, (uint32_t)j & 1u, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      const uint64_t vd = vdesc0 + (uint64_t)(s * (PF_V_BYTES >> 4));
      const uint32_t p_src = tmem + PF_TM_P + (uint32_t)((j & 1) * 64);
      const uint32_t first = j == 0 ? 0u : 1u;
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ts(tmem + PF_TM_O, p_src + (uint32_t)(k * 8), vd + (uint64_t)((k * 2048) >> 4), idesc_pv,
                 k == 0 ? first : 1u);
        mma_commit(&v_empty[s]);
        mma_commit(&pv_done);
      }
      __syncwarp();
      if (aborted()) { ok = false; break; }
    }
    if (!ok) fail();
    // No MMA may be in flight when TMEM is released.
    if (lane == 0) mma_commit(&mma_drain);
    __syncwarp();
    mbar_wait_warp(&mma_drain, 0, kWaitLimit);
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 2..9)
    // Warp w owns TMEM lanes 32*(w%4).. (its query rows) and score columns
    // 64*half.. of them, half = (w-2)/4: two warps per SM sub-partition share
    // the exponentials of a tile.  The two warps of a row quarter combine their
    // row maxima through shared memory (double-buffered, an mbarrier per tile
    // parity), so both take the same running-maximum decisions; each keeps its
    // own partial sum, added once at the end.
    const int quarter = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = 32 * quarter + lane;
    const int i = i0 + r;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t col0 = 64u * (uint32_t)hf;
    const int64_t limit = i < a.s_q ? offs + i : -1;       // last visible window position
    const int64_t min_limit = offs + i0;                   // the tile's first row
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      if (!mbar_wait_warp(&s_full[j & 1], (uint32_t)(j >> 1) & 1u, kWaitLimit)) { ok = false; break; }
      tc_fence_after();
      // This thread's 64 raw scores in two 32-column loads behind one wait.
      uint32_t v[2][32];
      tmem_ld32(tmem + lane_off + (uint32_t)((j & 1) * 128) + col0, v[0]);
      tmem_ld32(tmem + lane_off + (uint32_t)((j & 1) * 128) + col0 + 32, v[1]);
      tmem_wait_ld_regs(v[0]);
      reg_fence32(v[1]);
      const int64_t kbase = (int64_t)j * 128 + col0;
      const bool full = ((int64_t)j * 128 + 127 <= min_limit) && ((int64_t)j * 128 + 127 < len);
      if (!full) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kbase + c * 32 + e > limit) v[c][e] = __float_as_uint(-INFINITY);
      }
      // Partial row maximum with eight independent chains.
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) m8[e & 7] = fmaxf(m8[e & 7], __uint_as_float(v[c][e]));
      const float mpart = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      red_max[j & 1][hf][r] = mpart;
      mbar_arrive(&xbar[j & 1][quarter]);
      if (!mbar_wait_warp(&xbar[j & 1][quarter], (uint32_t)(j >> 1) & 1u, kWaitLimit)) { ok = false; break; }
      const float mraw = fmaxf(mpart, red_max[j & 1][hf ^ 1][r]);
      const float mx = mraw * a.scale_log2;          // log2 units (the scale is positive)
      // Move the running maximum only when it grows by more than 2^8.
      const bool move = mx > m_used + kRescaleLog2;
      float alpha = 1.f;
      if (move) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2_approx(m_used - mx);
        m_used = mx;
        l *= alpha;
      }
      uint32_t pk[32];
      float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (m_used == -INFINITY) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pk[e] = 0u;
      } else {
        const float neg_m = -m_used;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(v[c][2 * e]), a.scale_log2, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(v[c][2 * e + 1]), a.scale_log2, neg_m));
            s8[e & 7] += p0 + p1;
            pk[c * 16 + e] = pack_bf16x2(p0, p1);
          }
      }
      l += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
      // O holds P(0..j-1).V once the previous P.V is done; correct this
      // thread's 64 columns in place (warp-uniform: tcgen05.ld/st are collective).
      if (j > 0) {
        if (!mbar_wait_warp(&pv_done, (uint32_t)(j - 1) & 1u, kWaitLimit)) { ok = false; break; }
        if (__any_sync(0xffffffffu, move)) {
          tc_fence_after();
          const float f = move ? alpha : 1.f;
          uint32_t o[32];
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            tmem_ld32(tmem + lane_off + PF_TM_O + col0 + c * 32, o);
            tmem_wait_ld_regs(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(tmem + lane_off + PF_TM_O + col0 + c * 32, o);
          }
        }
      }
      // P (bf16 pairs) into its own buffer: the buffer last held P(j-2),
      // whose P.V is complete (P.V(j-1), waited for above, accumulates into
      // the same O after it).  The score buffer is left to the next scores:
      // MMAs into different accumulators are not ordered, so P must not
      // share columns with a later score MMA.
      tmem_st32(tmem + lane_off + PF_TM_P + (uint32_t)((j & 1) * 64) + 32u * (uint32_t)hf, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full);
      if (aborted()) { ok = false; break; }
    }
    if (ok && n_kt > 0) {
      ok = mbar_wait_warp(&pv_done, (uint32_t)(n_kt - 1) & 1u, kWaitLimit);
      if (!ok) fail();
    } else if (!ok) {
      fail();
    }
    // The row's sum: this half's plus the partner's.
    if (ok) {
      red_sum[hf][r] = l;
      mbar_arrive(&lbar[quarter]);
      ok = mbar_wait_warp(&lbar[quarter], 0, kWaitLimit);
      if (ok) l += red_sum[hf ^ 1][r];
      else fail();
    }
    // Epilogue: O / l, heads concatenated; lse in natural log.
    const bool visible = l > 0.f;
    const float inv = visible ? 1.f / l : 0.f;
    const bool write = i < a.s_q;
    const int64_t n = (int64_t)b * a.s_q + i;
    const int64_t ocol = (int64_t)h * a.v_dim + col0;
    if (ok && n_kt > 0) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + PF_TM_O + col0 + c * 32, o);
        tmem_wait_ld_regs(o);
        if (write) {
          if (a.out_f32) {
            float* dst = static_cast<float*>(a.out) + n * a.out_row_stride + ocol + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              *reinterpret_cast<float4*>(dst + e) =
                  make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                              __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + n * a.out_row_stride + ocol + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
              w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
              w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
              w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
              *reinterpret_cast<uint4*>(dst + e) = w;
            }
          }
        }
      }
    } else if (ok && write) {
      // No visible key (a row shorter than its block): zeros.
      for (int d = 0; d < 64; ++d) {
        if (a.out_f32) static_cast<float*>(a.out)[n * a.out_row_stride + ocol + d] = 0.f;
        else static_cast<__nv_bfloat16*>(a.out)[n * a.out_row_stride + ocol + d] = __float2bfloat16_rn(0.f);
      }
    }
    if (ok && write && hf == 0 && a.lse)
      a.lse[n * gridDim.y + h] = visible ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_tc_reconstruct(const ReconstructParams& p, cudaStream_t stream) {
  CUtensorMap lat_map, w_map, k_map, v_map;
  {
    const uint64_t dims[2] = {(uint64_t)p.rank, (uint64_t)p.n_rows};
    const uint64_t strides[1] = {(uint64_t)p.latent_row_stride * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap_bf16(&lat_map, p.latent, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.rank, (uint64_t)p.heads * (p.nope + p.v_dim)};
    const uint64_t strides[1] = {(uint64_t)p.rank * 2};
    const uint32_t box[2] = {64, 256};
    if (!encode_tmap_bf16(&w_map, p.kv_b_proj, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.nope, (uint64_t)p.heads, (uint64_t)p.n_rows};
    const uint64_t strides[2] = {(uint64_t)p.k_head_stride * 2, (uint64_t)p.k_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&k_map, p.k_nope, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.v_dim, (uint64_t)p.heads, (uint64_t)p.n_rows};
    const uint64_t strides[2] = {(uint64_t)p.v_head_stride * 2, (uint64_t)p.v_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&v_map, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cudaError_t ea = set_max_dynamic_smem(tc_reconstruct_kernel, RC_SMEM);
    if (ea != cudaSuccess) return ea;
  }
  const int row_tiles = (int)((p.n_rows + 127) / 128);
  const int64_t n_tiles = (int64_t)row_tiles * p.heads;
  if (n_tiles >= (1LL << 31)) return cudaErrorInvalidValue;
  ReconArgs a{p.rank / 64, p.nope + p.v_dim, row_tiles, (int32_t)n_tiles, p.status};
  const int sms = device_sm_count();
  const unsigned grid = (unsigned)(n_tiles < sms ? n_tiles : sms);
  tc_reconstruct_kernel<<<grid, RC_THREADS, RC_SMEM, stream>>>(lat_map, w_map, k_map, v_map, a);
  return cudaGetLastError();
}

cudaError_t launch_tc_prefill(const PrefillParams& p, cudaStream_t stream) {
  CUtensorMap qn_map, qr_map, k_map, r_map, v_map;
  const uint64_t n_q = (uint64_t)p.batch * p.s_q;
  const uint64_t buf_rows = p.packed ? (uint64_t)p.t_max : (uint64_t)p.batch * p.t_max;
  {
    const uint64_t dims[3] = {(uint64_t)p.nope, (uint64_t)p.heads, n_q};
    const uint64_t strides[2] = {(uint64_t)p.qn_head_stride * 2, (uint64_t)p.qn_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&qn_map, p.q_nope, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.rope_dim, (uint64_t)p.heads, n_q};
    const uint64_t strides[2] = {(uint64_t)p.qr_head_stride * 2, (uint64_t)p.qr_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&qr_map, p.q_rope, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.nope, (uint64_t)p.heads, buf_rows};
    const uint64_t strides[2] = {(uint64_t)p.k_head_stride * 2, (uint64_t)p.k_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&k_map, p.k_nope, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.rope_dim, buf_rows};
    const uint64_t strides[1] = {(uint64_t)p.rope_row_stride * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap_bf16(&r_map, p.rope, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)p.v_dim, (uint64_t)p.heads, buf_rows};
    const uint64_t strides[2] = {(uint64_t)p.v_head_stride * 2, (uint64_t)p.v_row_stride * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!encode_tmap_bf16(&v_map, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cudaError_t ea = set_max_dynamic_smem(tc_prefill_kernel, PF_SMEM);
    if (ea != cudaSuccess) return ea;
  }
  PrefillArgs a;
  memset(&a, 0, sizeof(a));
  a.kv_start = p.kv_start;
  a.kv_len = p.kv_len;
  a.t_max = p.t_max;
  a.packed = p.packed;
  a.batch = p.batch;
  a.s_q = p.s_q;
  a.n_qtiles = (p.s_q + 127) / 128;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  a.out = p.out;
  a.out_row_stride = p.out_row_stride;
  a.v_dim = p.v_dim;
  a.out_f32 = p.out_dtype == MLA_DTYPE_F32 ? 1 : 0;
  a.lse = p.lse;
  a.status = p.status;
  const dim3 grid((unsigned)a.n_qtiles, (unsigned)p.heads, (unsigned)p.batch);
  tc_prefill_kernel<<<grid, PF_THREADS, PF_SMEM, stream>>>(qn_map, qr_map, k_map, r_map, v_map, a);
  return cudaGetLastError();
}

}  // namespace mla
