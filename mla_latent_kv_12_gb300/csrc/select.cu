// Deterministic DSA top-k selection ("glm52-dsa.ts", selectGlm52DsaDevice and
// its rank-key / order-key kernels): per row, the top_k positions under the
// order (score descending, equal scores by ascending position); threshold =
// the minimum selected score; output = selected positions above the
// threshold in ascending order, then the threshold ties in ascending order.
// Rows with at most top_k scores are dense (count -1, the decode's marker).
//
// One CTA (1024 threads) per row.  The rank key is the order-preserving map
// of the f32 bits to uint32, complemented (ascending key = descending score).
// A 4-pass radix select (8 bits per pass, shared-memory histograms) finds the
// top_k-th smallest key K and how many entries equal to K are taken (the
// lowest positions).  A counting pass gives the number of entries above the
// threshold (0 when a selected score is NaN: the minimum is then NaN, as the
// page's min is), and an ordered pass compacts the selection with block-wide
// prefix sums, chunk by chunk in position order.
#include <math.h>
#include <stdint.h>

#include "mla_internal.h"
#include "tc_host.h"

namespace mla {
namespace {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

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

__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(const __grid_constant__ SelectParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ int hist[256];
  __shared__ int warp_sums[kSelWarps][3];
  __shared__ uint32_t prefix_s;
  __shared__ int remaining_s;
  __shared__ int count_gt_s, nan_sel_s;
  const int row = blockIdx.x;
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
  // ---- radix select of the k-th smallest key (1-based), 8 bits per pass
  if (threadIdx.x == 0) {
    prefix_s = 0;
    remaining_s = k;
  }
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = prefix_s;
    for (int i = threadIdx.x; i < L; i += kSelThreads) {
      const uint32_t key = rank_key(sc[i]);
      const bool match = pass == 0 || (key >> (shift + 8)) == prefix;
      if (match) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane j owns bins 8j..8j+7: local sums, a warp scan, then the bin
      const int lane = threadIdx.x;
      int local[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) local[q] = hist[8 * lane + q], sum += local[q];
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
        for (int q = 0; q < 8; ++q) {
          if (rem <= cum + local[q]) {
            prefix_s = (prefix << 8) | (uint32_t)(8 * lane + q);
            remaining_s = rem - cum;
            break;
          }
          cum += local[q];
        }
      }
    }
    __syncthreads();
  }
  const uint32_t kth = prefix_s;        // the k-th smallest key
  const int take_ties = remaining_s;    // entries equal to kth that are taken (lowest positions)
  const float thr = key_score(kth);
  // ---- entries above the threshold; a NaN among the selected makes the
  // threshold NaN (nothing is above it)
  if (threadIdx.x == 0) count_gt_s = 0, nan_sel_s = isnan(thr) ? 1 : 0;
  __syncthreads();
  int gt = 0, nan_sel = 0;
  for (int i = threadIdx.x; i < L; i += kSelThreads) {
    const float s = sc[i];
    gt += s > thr ? 1 : 0;
    nan_sel |= (isnan(s) && rank_key(s) < kth) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    nan_sel |= __shfl_xor_sync(0xffffffffu, nan_sel, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&count_gt_s, gt);
    if (nan_sel) atomicOr(&nan_sel_s, 1);
  }
  __syncthreads();
  const bool thr_nan = nan_sel_s != 0;
  const int n_above = thr_nan ? 0 : count_gt_s;
  // ---- ordered compaction: above-threshold positions, then the rest, ascending
  int carry[3] = {0, 0, 0};   // above, other selected, ties seen (key == kth)
  int32_t* out = p.selected + (int64_t)row * p.out_stride;
  for (int base = 0; base < L; base += kSelThreads) {
    const int i = base + threadIdx.x;
    int v[3] = {0, 0, 0};
    bool sel = false, above = false;
    uint32_t key = 0;
    float s = 0.f;
    if (i < L) {
      s = sc[i];
      key = rank_key(s);
      v[2] = key == kth ? 1 : 0;
    }
    int ex[3], tot[3];
    // first the tie ranks (a tie is taken if fewer than take_ties ties precede it)
    int vt[3] = {0, 0, v[2]};
    block_scan3(vt, ex, tot, warp_sums);
    if (i < L) {
      sel = key < kth || (key == kth && carry[2] + ex[2] < take_ties);
      above = !thr_nan && s > thr;
      v[0] = (sel && above) ? 1 : 0;
      v[1] = (sel && !above) ? 1 : 0;
    }
    const int tie_total = tot[2];
    int vs[3] = {v[0], v[1], 0};
    block_scan3(vs, ex, tot, warp_sums);
    if (sel) {
      const int slot = above ? carry[0] + ex[0] : n_above + carry[1] + ex[1];
      if (slot < k) out[slot] = i;
    }
    carry[0] += tot[0];
    carry[1] += tot[1];
    carry[2] += tie_total;
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
