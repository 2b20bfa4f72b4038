// Deterministic DSA top-k selection ("glm52-dsa.ts", selectGlm52DsaDevice and
// its rank-key / order-key kernels): per row, the top_k positions under the
// order (score descending, equal scores by ascending position); threshold =
// the minimum selected score; output = selected positions above the
// threshold in ascending order, then the threshold ties in ascending order.
// Rows with at most top_k scores are dense (count -1, the decode's marker).
//
// One CTA (1024 threads) per row.  The rank key is the order-preserving map
// of the f32 bits to uint32, complemented (ascending key = descending score).
// A 3-pass radix select (digits of 11, 11 and 10 bits, shared-memory
// histograms with one atomic per distinct digit per warp) finds the top_k-th
// smallest key K and how many entries equal to K are taken (the lowest
// positions).  The compaction gives each warp a contiguous range of positions,
// walked 32 at a time: a counting pass, one block-wide scan of the per-warp
// counts, and an ordered write pass with in-warp ranks from ballots (nothing
// is above the threshold when a selected score is NaN: the minimum is then
// NaN, as the page's min is).
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

__global__ void __launch_bounds__(kSelThreads, 1) select_topk_kernel(const __grid_constant__ SelectParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ int hist[kBins];
  __shared__ int warp_sums[kSelWarps][3];
  __shared__ uint32_t prefix_s;
  __shared__ int remaining_s;
  __shared__ int count_gt_s, nan_sel_s;
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = p.lengths[row];
  const int k = p.top_k;
  const float* sc = p.scores + (int64_t)row * p.row_stride;
  if (L <= k) {
    if (threadIdx.x == 0) {
      p.counts[row] = -1;                 // dense: every visible key
      if (L < 0 && p.status) atomicOr(p.status, MLA_DEVICE_BAD_SELECTION_COUNT);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    return;
  }
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
    for (int base = 0; base < L; base += kSelThreads * kUnroll) {
      float v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {   // kUnroll independent loads in flight
        const int i = base + u * kSelThreads + threadIdx.x;
        v[u] = i < L ? sc[i] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * kSelThreads + threadIdx.x;
        const uint32_t key = rank_key(v[u]);
        const bool match = i < L && (hi_bits == 0 || (key >> (32 - hi_bits)) == prefix);
        const uint32_t digit = (key >> shift) & mask;
        const uint32_t active = __ballot_sync(0xffffffffu, match);
        if (match) {
          const uint32_t same = __match_any_sync(active, digit);
          if ((__ffs(same) - 1) == lane) atomicAdd(&hist[digit], __popc(same));
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane j owns bins [64j, 64j+64): local sums, a warp scan, then the bin
      const int nb = 1 << width;
      const int per = nb / 32;
      int sum = 0;
      for (int q = 0; q < per; ++q) sum += hist[per * lane + q];
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      const int before = incl - sum;
      const int rem = remaining_s;
      if (before < rem && rem <= incl) {  // exactly one lane
        int cum = before;
        for (int q = 0; q < per; ++q) {
          const int c = hist[per * lane + q];
          if (rem <= cum + c) {
            prefix_s = (prefix << width) | (uint32_t)(per * lane + q);
            remaining_s = rem - cum;
            break;
          }
          cum += c;
        }
      }
    }
    __syncthreads();
    hi_bits += width;
  }
  const uint32_t kth = prefix_s;        // the k-th smallest key
  const int take_ties = remaining_s;    // entries equal to kth that are taken (lowest positions)
  const float thr = key_score(kth);
  // ---- compaction: warp w owns positions [w*span, (w+1)*span), walked 32 at a
  // time (coalesced).  Pass 1 counts, per warp, the entries above the
  // threshold, the other smaller keys and the ties, and whether a selected
  // score is NaN (then the threshold -- the minimum selected score -- is NaN
  // and nothing is above it).
  const int span = ((L + kSelWarps - 1) / kSelWarps + 31) & ~31;
  const int lo = min(L, warp * span), hi = min(L, lo + span);
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
  if (threadIdx.x == 0) count_gt_s = 0, nan_sel_s = 0;
  __syncthreads();
  if (lane == 0) {
    atomicAdd(&count_gt_s, c_above);
    if (nan_sel) atomicOr(&nan_sel_s, 1);
  }
  // exclusive prefix of the per-warp counts (one value per warp: lanes > 0 add 0)
  int v[3] = {lane == 0 ? c_above : 0, lane == 0 ? c_less : 0, lane == 0 ? c_tie : 0}, ex[3], tot[3];
  block_scan3(v, ex, tot, warp_sums);   // its barriers also publish count_gt_s / nan_sel_s
  ex[0] = __shfl_sync(0xffffffffu, ex[0], 0);
  ex[1] = __shfl_sync(0xffffffffu, ex[1], 0);
  ex[2] = __shfl_sync(0xffffffffu, ex[2], 0);
  const bool thr_nan = nan_sel_s != 0;
  const int n_above = thr_nan ? 0 : count_gt_s;
  // Pass 2 writes: above-threshold entries at [0, n_above) in position order,
  // the other selected ones (smaller keys not above it, then the first
  // take_ties ties) after them in position order.  With a NaN threshold every
  // selected entry is in the second list.  (The ties taken before this range
  // are the first min(ties before, take_ties).)
  int o_above = ex[0], o_rest = ex[1] + min(ex[2], take_ties) + (thr_nan ? ex[0] : 0), t_seen = ex[2];
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
  if (threadIdx.x == 0) p.counts[row] = k;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t launch_select_topk(const SelectParams& p, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(select_topk_kernel, dim3((unsigned)p.n_rows), dim3(kSelThreads), 0, stream, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
