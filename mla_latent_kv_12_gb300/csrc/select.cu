// Deterministic DSA top-k selection ("glm52-dsa.ts", selectGlm52DsaDevice and
// its rank-key / order-key kernels): per row, the top_k positions under the
// order (score descending, equal scores by ascending position); threshold =
// the minimum selected score; output = selected positions above the
// threshold in ascending order, then the threshold ties in ascending order.
// Rows with at most top_k scores are dense (count -1, the decode's marker).
//
// A cluster of up to 8 CTAs (1024 threads each) per row, each owning a slice
// of it.  The rank key is the order-preserving map of the f32 bits to uint32,
// complemented (ascending key = descending score).  A 3-pass radix select
// (digits of 11, 11 and 10 bits; per-CTA shared-memory histograms with one
// atomic per distinct digit per warp, summed across the cluster through
// distributed shared memory) finds the top_k-th smallest key K and how many
// entries equal to K are taken (the lowest positions).  The compaction gives
// each warp a contiguous range of positions, walked 32 at a time: a counting
// pass, a scan of the per-warp counts plus the earlier CTAs' totals, and an
// ordered write pass with in-warp ranks from ballots (nothing is above the
// threshold when a selected score is NaN: the minimum is then NaN, as the
// page's min is).
#include <math.h>
#include <stdint.h>

#include "mla_internal.h"
#include "tc_host.h"

namespace mla {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBins = 2048;   // 11-bit digits
constexpr int kUnroll = 8;    // independent loads in flight per thread
constexpr int kSelCluster = 8; // CTAs per row

__device__ __forceinline__ uint32_t rank_key(float s) {
  const uint32_t bits = __float_as_uint(s);
  const uint32_t ascending = (bits & 0x80000000u) ? ~bits : (bits ^ 0x80000000u);
  return ~ascending;
}
__device__ __forceinline__ float key_score(uint32_t key) {
  const uint32_t ascending = ~key;
  const uint32_t bits = (ascending & 0x80000000u) ? (ascending ^ 0x80000000u) : ~ascending;
  return __uint_as_float(bits);
}

// Block-wide exclusive scan of up to three counters per thread (all threads
// call it); returns the exclusive prefixes and writes the block totals.
__device__ __forceinline__ void block_scan3(int (&v)[3], int (&excl)[3], int (&total)[3], int (*warp_sums)[3]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc[3] = {v[0], v[1], v[2]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      const int x = __shfl_up_sync(0xffffffffu, inc[c], o);
      if (lane >= o) inc[c] += x;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int c = 0; c < 3; ++c) warp_sums[warp][c] = inc[c];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      int w = warp_sums[lane][c];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += x;
      }
      warp_sums[lane][c] = w;   // inclusive over warps
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    excl[c] = (warp ? warp_sums[warp - 1][c] : 0) + inc[c] - v[c];
    total[c] = warp_sums[kSelWarps - 1][c];
  }
  __syncthreads();   // warp_sums is reused by the next call
}

__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t ctas_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 32-bit load from the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ int ld_peer(const int* local, uint32_t rank) {
  uint32_t a, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return (int)v;
}

// A cluster of 1..kSelCluster CTAs per row (chosen at launch); CTA c owns the
// slice [c*span, (c+1)*span) of the row.  Every CTA sums all the CTAs' histograms
// through distributed shared memory and takes the same digit, so the radix
// state stays identical across the cluster without a broadcast.
__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const __grid_constant__ SelectParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ int hist[kBins];       // this CTA's histogram (read by the whole cluster)
  __shared__ int total[kBins];      // the cluster's histogram
  __shared__ int warp_sums[kSelWarps][3];
  __shared__ int cta_tot[4];        // this CTA's above / other-smaller / ties / NaN-selected counts
  __shared__ uint32_t prefix_s;
  __shared__ int remaining_s;
  const uint32_t crank = cta_rank_in_cluster();
  const int ncta = (int)ctas_in_cluster();
  const int row = blockIdx.x / ncta;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = p.lengths[row];
  const int k = p.top_k;
  const float* sc = p.scores + (int64_t)row * p.row_stride;
  if (L <= k) {                     // the same in every CTA of the cluster
    if (threadIdx.x == 0 && crank == 0) {
      p.counts[row] = -1;           // dense: every visible key
      if (L < 0 && p.status) atomicOr(p.status, MLA_DEVICE_BAD_SELECTION_COUNT);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
  const int span = ((L + ncta - 1) / ncta + 31) & ~31;
  const int clo = min(L, (int)crank * span), chi = min(L, clo + span);
  // ---- radix select of the k-th smallest key (1-based): digits of 11, 11 and
  // 10 bits from the top; lanes of a warp holding the same digit add once
  if (threadIdx.x == 0) {
    prefix_s = 0;
    remaining_s = k;
  }
  int hi_bits = 0;   // key bits fixed by earlier passes
  for (int pass = 0; pass < 3; ++pass) {
    const int width = pass < 2 ? 11 : 10;
    const int shift = 32 - hi_bits - width;
    const uint32_t mask = (1u << width) - 1u;
    for (int i = threadIdx.x; i < kBins; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = prefix_s;
    for (int base = clo; base < chi; base += kSelThreads * kUnroll) {
      float v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {   // kUnroll independent loads in flight
        const int i = base + u * kSelThreads + threadIdx.x;
        v[u] = i < chi ? sc[i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kSelThreads + threadIdx.x;
        const uint32_t key = rank_key(v[u]);
        const bool match = i < chi && (hi_bits == 0 || (key >> (32 - hi_bits)) == prefix);
        const uint32_t digit = (key >> shift) & mask;
        const uint32_t active = __ballot_sync(0xffffffffu, match);
        if (match) {
          const uint32_t same = __match_any_sync(active, digit);
          if ((__ffs(same) - 1) == lane) atomicAdd(&hist[digit], __popc(same));
        }
      }
    }
    cluster_barrier();   // every CTA's histogram is complete
    for (int i = threadIdx.x; i < (1 << width); i += kSelThreads) {
      int t = 0;
      for (int c = 0; c < ncta; ++c) t += ld_peer(&hist[i], (uint32_t)c);
      total[i] = t;
    }
    __syncthreads();
    {
      // the bin holding the remaining rank: thread t owns bins 2t, 2t+1; a
      // block scan of the pair sums locates it
      const int nb = 1 << width;
      const int b0 = 2 * threadIdx.x;
      const int h0 = b0 < nb ? total[b0] : 0, h1 = b0 + 1 < nb ? total[b0 + 1] : 0;
      const int rem = remaining_s;   // read by every thread before the scan's barriers
      int vb[3] = {h0 + h1, 0, 0}, exb[3], totb[3];
      block_scan3(vb, exb, totb, warp_sums);
      const int before = exb[0];
      if (before < rem && rem <= before + h0 + h1) {   // exactly one thread
        const int in_first = rem <= before + h0;
        prefix_s = (prefix << width) | (uint32_t)(in_first ? b0 : b0 + 1);
        remaining_s = in_first ? rem - before : rem - before - h0;
      }
    }
    cluster_barrier();   // every CTA has read the histograms (they are cleared next pass)
    hi_bits += width;
  }
  const uint32_t kth = prefix_s;        // the k-th smallest key (the same in every CTA)
  const int take_ties = remaining_s;    // entries equal to kth that are taken (lowest positions)
  const float thr = key_score(kth);
  // ---- compaction: warp w of this CTA owns positions [lo, hi) of its slice,
  // walked 32 at a time (coalesced).  Pass 1 counts the entries above the
  // threshold, the other smaller keys and the ties, and whether a selected
  // score is NaN (then the threshold -- the minimum selected score -- is NaN
  // and nothing is above it).
  const int wspan = ((chi - clo + kSelWarps - 1) / kSelWarps + 31) & ~31;
  const int lo = min(chi, clo + warp * wspan), hi = min(chi, lo + wspan);
  const uint32_t lt = (1u << lane) - 1u;
  int c_above = 0, c_less = 0, c_tie = 0;
  bool nan_sel = isnan(thr);
  for (int base0 = lo; base0 < hi; base0 += 32 * kUnroll) {
    float vv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base0 + 32 * u + lane;
      vv[u] = i < hi ? sc[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base0 + 32 * u + lane;
      const bool in = i < hi;
      const float s = vv[u];
      const uint32_t key = in ? rank_key(s) : 0xffffffffu;
      c_above += __popc(__ballot_sync(0xffffffffu, in && s > thr));
      c_less += __popc(__ballot_sync(0xffffffffu, in && key < kth && !(s > thr)));
      c_tie += __popc(__ballot_sync(0xffffffffu, in && key == kth));
      nan_sel |= __any_sync(0xffffffffu, in && isnan(s) && key < kth);
    }
  }
  if (threadIdx.x < 4) cta_tot[threadIdx.x] = 0;
  __syncthreads();
  if (lane == 0) {
    atomicAdd(&cta_tot[0], c_above);
    atomicAdd(&cta_tot[1], c_less);
    atomicAdd(&cta_tot[2], c_tie);
    if (nan_sel) atomicOr(&cta_tot[3], 1);
  }
  // exclusive prefix of the per-warp counts inside this CTA
  int v[3] = {lane == 0 ? c_above : 0, lane == 0 ? c_less : 0, lane == 0 ? c_tie : 0}, ex[3], tot[3];
  block_scan3(v, ex, tot, warp_sums);   // its barriers also complete cta_tot
  cluster_barrier();                    // every CTA's totals are complete
  int n_above = 0, pre[3] = {0, 0, 0};
  bool thr_nan = false;
  for (int c = 0; c < ncta; ++c) {
    const int a = ld_peer(&cta_tot[0], (uint32_t)c), l = ld_peer(&cta_tot[1], (uint32_t)c),
              t = ld_peer(&cta_tot[2], (uint32_t)c), nn = ld_peer(&cta_tot[3], (uint32_t)c);
    n_above += a;
    thr_nan |= nn != 0;
    if (c < (int)crank) pre[0] += a, pre[1] += l, pre[2] += t;
  }
  if (thr_nan) n_above = 0;
  const int ex_above = pre[0] + __shfl_sync(0xffffffffu, ex[0], 0);
  const int ex_less = pre[1] + __shfl_sync(0xffffffffu, ex[1], 0);
  const int ex_tie = pre[2] + __shfl_sync(0xffffffffu, ex[2], 0);
  // Pass 2 writes: above-threshold entries at [0, n_above) in position order,
  // the other selected ones (smaller keys not above it, then the first
  // take_ties ties) after them in position order.  With a NaN threshold every
  // selected entry is in the second list.  (The ties taken before this range
  // are the first min(ties before, take_ties).)
  int o_above = ex_above, o_rest = ex_less + min(ex_tie, take_ties) + (thr_nan ? ex_above : 0), t_seen = ex_tie;
  int32_t* out = p.selected + (int64_t)row * p.out_stride;
  for (int base0 = lo; base0 < hi; base0 += 32 * kUnroll) {
    float vv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base0 + 32 * u + lane;
      vv[u] = i < hi ? sc[i] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base0 + 32 * u + lane;
      const bool in = i < hi;
      const float s = vv[u];
      const uint32_t key = in ? rank_key(s) : 0xffffffffu;
      const uint32_t tie_mask = __ballot_sync(0xffffffffu, in && key == kth);
      const bool sel = in && (key < kth || (key == kth && t_seen + __popc(tie_mask & lt) < take_ties));
      t_seen += __popc(tie_mask);
      const bool above = sel && !thr_nan && s > thr;
      const uint32_t a_mask = __ballot_sync(0xffffffffu, above);
      const uint32_t r_mask = __ballot_sync(0xffffffffu, sel && !above);
      if (sel) {
        const int slot = above ? o_above + __popc(a_mask & lt) : n_above + o_rest + __popc(r_mask & lt);
        if (slot < k) out[slot] = i;
      }
      o_above += __popc(a_mask);
      o_rest += __popc(r_mask);
    }
  }
  if (threadIdx.x == 0 && crank == 0) p.counts[row] = k;
  cluster_barrier();   // no CTA leaves while another may still read its totals
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  // CTAs per row: one per 16k scores of the row stride (an upper bound of the
  // lengths), at most kSelCluster, and few enough that all rows fit one wave.
  const int64_t by_len = (p.row_stride + 16383) / 16384;
  const int64_t by_rows = device_sm_count() / (int64_t)p.n_rows;
  int ncta = 1;
  while (ncta * 2 <= kSelCluster && ncta * 2 <= by_len && ncta * 2 <= by_rows) ncta *= 2;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)ncta;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.n_rows * ncta));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
