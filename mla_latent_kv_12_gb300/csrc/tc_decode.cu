// Tensor-core flash-decode over the latent||rope cache ("glm52-mla.ts",
// Glm52Mla.attendAbsorbed: s = q_lat.latent + q_rope.rope, scaled, softmax,
// ctx = p @ latent; with the per-row windows / selections of Glm52Mla.forward
// and the causal verify window of Glm52DecoderLayer.attend).
//
// Design (bf16, H = 128 or 64 heads, rank 512, rope 64):
//  * All 128 heads of one query row form the M = 128 side of every tcgen05 MMA
//    (64 heads are padded to 128 with zero query rows, whose results are
//    dropped: at one query row the kernel is bound by the cache read, which
//    the padding does not change);
//    keys come in tiles of 64 (the N side of the score MMA, the K side of P.V).
//  * A cluster of two CTAs (an SM pair) owns one stream of work.  The f32
//    context accumulator [128 x 512] would fill a whole SM's TMEM, so the pair
//    splits the feature axis evenly: CTA r scores latent dims [256r, 256r+256)
//    and rope dims [32r, 32r+32) (18 MMA K-steps each).  Each CTA scales its
//    partial scores to the log2 domain, rounds them to fp16 and stores them
//    straight into the peer's shared memory with asynchronous remote stores
//    (st.async, counted as transactions on the receiving barrier); each CTA
//    then adds its own and the peer's halves in f32, runs the online softmax,
//    and accumulates O[:, own 256 latent dims] += P . latent[:, own dims],
//    normalised by its own sum.  No MMA work is repeated and every cache byte
//    is read by exactly one CTA of the pair.
//  * Q (the CTA's dims) and P live in TMEM as the MMA A operand; cache tiles
//    are TMA-loaded into a 4-stage ring (latent dims with 128-byte swizzle,
//    the CTA's rope dims with 64-byte swizzle); one tile serves the score MMA
//    (K-major B) and the P.V MMA (MN-major B) through two descriptors.
//  * Warp roles: warp 0 loads (TMA tiles, or TMA gather4 / cp.async row
//    gathers for selected positions, plus L2 prefetch ahead); warp 1 issues the
//    score MMAs; warps 6..9 read the scores from TMEM and run the exchange;
//    warps 2..5 (one thread per head) run the online softmax (log2 domain,
//    lazy rescale) and the epilogue; warp 10 issues the P.V MMAs.  The
//    instance for TMA row gathers adds warps 11..13, which issue their share
//    of each tile's gather4 copies.
//  * Split-K: each query row's tiles are counted (by every CTA in its prologue
//    for up to 128 rows, else by a planner kernel); the flattened tile
//    sequence, in which each row start is charged a few tiles when the ranges
//    are long, is cut into equal ranges, one per cluster group.  A row wholly
//    inside one range is finished in place; otherwise each piece writes its
//    normalised context O / l in fp16 with (m, l) in f32, and a combine kernel
//    merges them.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mla {
namespace {

using namespace tc;

constexpr int BN = 64;                    // keys per tile
constexpr int STAGES = 4;
// A stage holds one tile of this CTA's features: four [64 keys x 64 latent
// dims] boxes (128-byte rows, 128-byte swizzle) and its 32 rope dims
// ([64 keys x 32 dims], 64-byte rows, 64-byte swizzle).
constexpr int CHUNK_BYTES = BN * 128;
constexpr int ROPE_BYTES = BN * 64;
constexpr int STAGE_BYTES = 4 * CHUNK_BYTES + ROPE_BYTES;
constexpr int STAGE_TX = STAGE_BYTES;     // bytes one tile's loads deliver into a stage
constexpr int XH_BYTES = 128 * BN * 2;    // fp16 partial scores of one tile (one send / receive buffer)
constexpr int HEADS = 128, RANK = 512, DV = 256;  // DV: latent dims per CTA
// producer, score MMA, 4 softmax, 4 exchange and P.V MMA warps; the kernel
// instance for TMA row gathers of selected positions adds three warps that
// share each tile's gathers with the producer (its own instance: compiled for
// more threads the dense kernel gets fewer registers and ran 3 % slower)
constexpr int THREADS = 352, THREADS_GATHER = THREADS + 96;
constexpr int kGatherWarp = 11;   // first extra gather warp
// Dynamic shared memory: the stage ring, then send[2] and receive[2].  The
// 1024-byte alignment of the extern declaration places it on a 1024-byte
// boundary after the static variables (checked at run time).
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 4 * XH_BYTES;
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 400, TM_P = 464;  // TMEM columns (Q: 128 + 16)
constexpr long long kWaitLimit = 1LL << 32;  // clock cycles (~2 s)
constexpr float kRescaleThreshold = 8.0f;    // log2 units
// A group's tile range is at least this long: each split writes a 256 KB f32
// partial, worth it only against a few 72 KB tiles of cache read.
constexpr int kMinTilesPerGroup = 4;
// Each work unit with tiles is charged this many tiles' worth of time for
// its start: a segment boundary drains the pair's pipeline (the next query
// enters TMEM only once the previous segment's last scores are read, then
// its first scores and exchange run before the softmax resumes), which costs
// several tiles of streaming.  The charge sits in the split plan ahead of the
// unit's tiles, so a group whose range holds more unit starts gets fewer
// tiles.  It applies when the groups stream at least kChargeMinSpan tiles
// each: with a few tiles per group (a short or selected-position batch) every
// group pays one start anyway, and a charge would only idle groups.
constexpr int kUnitStartCharge = 10;
constexpr int kChargeMinSpan = 32;
// Tiles of the current row pulled into L2 ahead of their load (the decode
// kernel's template parameter): farther for a lockstep group (the group's
// pairs all read each tile, three of them from L2), nearer for a single row,
// whose early prefetches the streamed cache evicts again before use.  A
// compile-time distance: with a run-time one the lockstep verify decode ran
// 3 % slower.
constexpr int kPrefetchAheadGroup = 8, kPrefetchAheadRow = 3;
constexpr int kQueryPrefetchTiles = 4;   // the next segment's query is pulled into L2 this many tiles before
// Up to this many query rows, every CTA plans the split itself in its prologue
// (no planner launch); larger batches use the planner kernel.
constexpr int kMaxRowsInKernelPlan = 128;

struct TcDecodeArgs {
  const __nv_bfloat16* q;
  int64_t q_row_stride, q_head_stride;
  const __nv_bfloat16* latent;
  int64_t latent_row_stride, latent_batch_stride;
  const __nv_bfloat16* rope;
  int64_t rope_row_stride, rope_batch_stride;
  const int32_t* kv_start;
  const int32_t* kv_len;
  int32_t s_q, n_q;
  int32_t heads;       // 64 or 128; rows h >= heads of the MMA's M side are zero padding
  const int32_t* sel;
  const int32_t* sel_count;
  int32_t k_max;
  float scale_log2;
  void* ctx;
  int64_t ctx_row_stride, ctx_head_stride;
  int32_t out_f32;
  float* lse;
  int32_t* status;
  int32_t* prefix;     // [n_units + 2] the split plan: prefix over work units, then the start charge
  int32_t* keys;       // [n_q] visible entries per query row (planner)
  uint4* ws_o;         // [slots][RANK/8][H] partial context, 8 fp16 dims per entry (O / l of the piece)
  float* ws_ml;        // [slots][2][H] partial (m, l), log2 domain
  int32_t num_clusters;
  int32_t width;       // query rows per work unit = clusters per group
  int32_t n_units;     // n_q / width
  int32_t min_tiles;   // smallest tile range given to a group
  int32_t batch_in_map;  // 1: use batch coordinate b in the tensor maps
  int32_t gather_tma;    // 1: selected rows come by TMA gather4 (else cp.async)
  int32_t lat_rows_per_batch, rope_rows_per_batch;  // batch stride in rows (gather maps)
  int32_t plan_in_kernel;  // 1: n_q <= kMaxRowsInKernelPlan, each CTA plans (CTA 0 also stores the plan)
  // 1 inside a fused step: the launch before the decode kernel is the absorb
  // kernel, which writes only the query and lets its dependants start only
  // after its own wait, so every other input is complete when this grid starts.
  int32_t early_inputs;
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ int row_limit(const TcDecodeArgs& a, int n) {
  const int b = n / a.s_q, i = n % a.s_q;
  const int len = a.kv_len[b];
  int lim = len - a.s_q + i + 1;
  lim = lim < 0 ? 0 : (lim > len ? len : lim);
  return lim;
}

// Work units are query rows, or -- for a dense multi-token verify -- whole
// batch rows whose `width` = s_q tokens are served by a group of `width`
// clusters in lockstep (member i takes token i), so the tokens of a batch row
// read each cache tile at the same time and three of four reads hit L2.
// The units' tiles form one flattened sequence cut into equal ranges, one per
// group (at least `min_tiles` each, so a short sequence uses fewer groups).
// In that sequence each unit with tiles occupies charge + tiles positions,
// its tiles at the end: prefix[0..n_units] holds these extents' exclusive
// prefix and prefix[n_units + 1] the charge, so unit u's tile j sits at
// position prefix[u] + charge + j.
__device__ __forceinline__ int group_span(const TcDecodeArgs& a, int total) {
  const int ngroups = a.num_clusters / a.width;
  const int per = (total + ngroups - 1) / ngroups;
  return per > a.min_tiles ? per : a.min_tiles;
}

// The start charge of a plan whose units hold `raw` tiles in all.
__device__ __forceinline__ int unit_start_charge(const TcDecodeArgs& a, int raw) {
  const int ngroups = a.num_clusters / a.width;
  return (raw + ngroups - 1) / ngroups >= kChargeMinSpan ? kUnitStartCharge : 0;
}

struct WorkIter {
  const int32_t* prefix;
  int n, t, t_begin, t_end, charge;
  __device__ void init(const TcDecodeArgs& a, const int32_t* unit_prefix, int group) {
    prefix = unit_prefix;
    charge = prefix[a.n_units + 1];
    const int total = prefix[a.n_units];
    const int per = group_span(a, total);
    const int ngroups = a.num_clusters / a.width;
    const long long b0 = group < ngroups ? (long long)group * per : total;
    t_begin = (int)min((long long)total, b0);
    t_end = (int)min((long long)total, (long long)t_begin + per);
    // first unit with prefix[n+1] > t_begin
    int lo = 0, hi = a.n_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid + 1] > t_begin) hi = mid; else lo = mid + 1;
    }
    n = lo;
    t = t_begin;
  }
  // Next segment: unit u, unit-local tiles [t0, t1); `whole` if all of the
  // unit's tiles lie inside this group's range.  A unit whose start charge
  // alone falls in the range is no segment.
  __device__ bool next(int& u, int& t0, int& t1, bool& whole) {
    while (t < t_end) {
      while (prefix[n + 1] <= t) ++n;
      const int rs = prefix[n] + charge, re = prefix[n + 1];   // the unit's tiles
      const int s = max(t, rs), e = min(t_end, re);
      t = e;
      if (s >= e) continue;
      u = n;
      t0 = s - rs;
      t1 = e - rs;
      whole = rs >= t_begin && re <= t_end;
      return true;
    }
    return false;
  }
};

// The groups whose ranges hold unit u's tiles: [first, last] (a unit with
// tiles; `charge` = prefix[n_units + 1]).
__device__ __forceinline__ int first_group_of(const int32_t* prefix, int u, int per, int charge) {
  return (prefix[u] + charge) / per;
}
__device__ __forceinline__ int last_group_of(const int32_t* prefix, int u, int per) {
  return (prefix[u + 1] - 1) / per;
}

// A member's share of a unit segment: its query row n and the segment's tiles
// clipped to that row's own tiles (a verify token sees a shorter prefix than
// the last token).  False if nothing is left.
__device__ __forceinline__ bool member_segment(const TcDecodeArgs& a, const int32_t* keys, int u, int member,
                                               int& n, int& t0, int& t1) {
  n = u * a.width + member;
  const int tiles = (keys[n] + BN - 1) / BN;
  if (t1 > tiles) t1 = tiles;
  return t0 < t1;
}

// TMA row gather of key group g (keys 4g..4g+3) of tile t into a stage: one
// gather4 per 64-dim latent chunk and one for this CTA's 32 rope dims.
// Entries past the count or out of range load the window's first row
// (finite data; the softmax gives them p = 0).
__device__ __forceinline__ void gather_key_group(const TcDecodeArgs& a, const CUtensorMap* lat_rows_map,
                                                 const CUtensorMap* rope_rows_map, uint8_t* dst, uint64_t* bar,
                                                 int g, int t, int b, int start, int limit, int keys,
                                                 const int32_t* list, uint32_t rank, int dim_base) {
  int lr[4], rr[4], pos[4];
  // the four positions are read before any is checked: one round trip (a
  // status update between reads would order them)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = t * BN + 4 * g + j;
    pos[j] = (list && e < keys) ? __ldg(list + e) : e;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = t * BN + 4 * g + j;
    bool v = e < keys;
    int p = pos[j];
    if (v && list) {
      if (p < 0 || p >= limit) {
        v = false;
        if (a.status && rank == 0) atomicOr(a.status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
      }
    }
    const int w = start + (v ? p : 0);
    lr[j] = b * a.lat_rows_per_batch + w;
    rr[j] = b * a.rope_rows_per_batch + w;
  }
  for (int c = 0; c < 4; ++c)
    tma_gather4(dst + c * CHUNK_BYTES + g * 4 * 128, lat_rows_map, bar, dim_base + 64 * c, lr[0], lr[1], lr[2], lr[3]);
  tma_gather4(dst + 4 * CHUNK_BYTES + g * 4 * 64, rope_rows_map, bar, 32 * (int)rank, rr[0], rr[1], rr[2], rr[3]);
}

// ------------------------------------------------------------------ planner
// Per query row the number of visible entries; the planner (or the decode
// prologue) turns them into tiles and the exclusive prefix of tiles over work
// units.  Bad selection counts give 0 and are flagged where `flag` is set.
__device__ __forceinline__ int row_keys(const TcDecodeArgs& a, int n, bool flag) {
  int keys = row_limit(a, n);
  if (a.sel) {
    const int c = a.sel_count[n];
    if (c != -1) {
      if (c <= 0 || c > a.k_max) {
        keys = 0;
        if (flag && a.status) atomicOr(a.status, MLA_DEVICE_BAD_SELECTION_COUNT);
      } else {
        keys = c;
      }
    }
  }
  return keys;
}

// The split plan inside a kernel (n_q <= kMaxRowsInKernelPlan; called by every
// thread of the block, blockDim >= n_q): visible entries per query row, then per
// unit its tiles (the longest of its `width` rows) and their exclusive prefix,
// scanned by warp 0 (four units per lane, in unit order).
// With start_s / limit_s, also each row's first cache row and window limit.
__device__ __forceinline__ void plan_rows(const TcDecodeArgs& a, int32_t* keys_s, int32_t* prefix_s, bool flag,
                                          int32_t* start_s = nullptr, int32_t* limit_s = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < a.n_q) {
    const int n = threadIdx.x;
    keys_s[n] = row_keys(a, n, flag);
    if (start_s) {
      start_s[n] = a.kv_start ? a.kv_start[n / a.s_q] : 0;
      limit_s[n] = row_limit(a, n);
    }
  }
  __syncthreads();
  if (warp == 0) {
    int tl[kMaxRowsInKernelPlan / 32];
    int raw = 0;
#pragma unroll
    for (int j = 0; j < kMaxRowsInKernelPlan / 32; ++j) {
      const int u = 32 * j + lane;
      int tiles = 0;
      if (u < a.n_units)
        for (int i = 0; i < a.width; ++i) tiles = max(tiles, (keys_s[u * a.width + i] + BN - 1) / BN);
      tl[j] = tiles;
      raw += tiles;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) raw += __shfl_xor_sync(0xffffffffu, raw, o);
    const int charge = unit_start_charge(a, raw);
    int carry = 0;
#pragma unroll
    for (int j = 0; j < kMaxRowsInKernelPlan / 32; ++j) {
      const int u = 32 * j + lane;
      const int ext = tl[j] > 0 ? tl[j] + charge : 0;   // the unit's extent in the plan
      int v = ext;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += x;
      }
      if (u < a.n_units) prefix_s[u] = carry + v - ext;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
      prefix_s[a.n_units] = carry;
      prefix_s[a.n_units + 1] = charge;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(1024) tc_plan_kernel(const __grid_constant__ TcDecodeArgs a) {
  pdl_wait();
  __shared__ int warp_sums[32];
  __shared__ int carry_s, raw_s;
  if (threadIdx.x == 0) carry_s = 0, raw_s = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // pass 1: visible entries per row (stored) and the units' tiles in all
  int raw = 0;
  for (int u = threadIdx.x; u < a.n_units; u += 1024) {
    int tiles = 0;
    for (int i = 0; i < a.width; ++i) {
      const int n = u * a.width + i;
      const int keys = row_keys(a, n, true);
      a.keys[n] = keys;
      const int t = (keys + BN - 1) / BN;
      tiles = t > tiles ? t : tiles;
    }
    raw += tiles;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) raw += __shfl_xor_sync(0xffffffffu, raw, o);
  if (lane == 0) atomicAdd(&raw_s, raw);
  __syncthreads();
  const int charge = unit_start_charge(a, raw_s);
  // pass 2: the units' extents (each thread rereads the rows it stored) and
  // their exclusive prefix
  for (int base = 0; base < a.n_units; base += 1024) {
    const int u = base + threadIdx.x;
    int ext = 0;
    if (u < a.n_units) {
      int tiles = 0;
      for (int i = 0; i < a.width; ++i) {
        const int t = (a.keys[u * a.width + i] + BN - 1) / BN;
        tiles = t > tiles ? t : tiles;
      }
      ext = tiles > 0 ? tiles + charge : 0;
    }
    int v = ext;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += x;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += x;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int excl = carry_s + (warp ? warp_sums[warp - 1] : 0) + v - ext;
    if (u < a.n_units) a.prefix[u] = excl;
    __syncthreads();
    if (threadIdx.x == 1023) carry_s = excl + ext;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    a.prefix[a.n_units] = carry_s;
    a.prefix[a.n_units + 1] = charge;
  }
  pdl_trigger();
}

// ------------------------------------------------------------------ decode

// kLateP: a tile's P is announced to the P.V issuer only once the next tile's
// score halves have arrived (for the lockstep verify groups, whose tensor work
// per tile is four tokens' worth: each P.V then follows the next tile's score
// MMAs instead of delaying them; single rows lose by the added P.V latency).
// Without deadlock: the next tile's scores wait on the P.V STAGES tiles back
// (its stage) and on the exchange of this tile's, in both CTAs, never on this P.V.
template <int kPrefetchAhead, int kThreads, bool kLateP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap lat_map, const __grid_constant__ CUtensorMap rope_map,
                     const __grid_constant__ CUtensorMap lat_rows_map, const __grid_constant__ CUtensorMap rope_rows_map,
                     const __grid_constant__ TcDecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {   // the same in every CTA: nothing waits on anything yet
    if (threadIdx.x == 0 && a.status) atomicOr(a.status, MLA_DEVICE_LAYOUT);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* stages = smem;
  // Exchange buffers, each [8][128 heads][16 B] of fp16 scores: xin[b] is written
  // by the peer's remote stores, xout[b] holds this CTA's own half for its
  // softmax warps.
  uint8_t* xin = smem + STAGES * STAGE_BYTES;        // 2 x XH_BYTES
  uint8_t* xout = xin + 2 * XH_BYTES;                // 2 x XH_BYTES

  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t s_full, s_free, p_full, q_full, o_free, mma_drain, pv_drain;
  __shared__ __align__(8) uint64_t x_full[2], x_free[2], xo_free[2];  // per exchange buffer
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int32_t plan_keys_s[kMaxRowsInKernelPlan];
  __shared__ int32_t plan_prefix_s[kMaxRowsInKernelPlan + 2];
  __shared__ int32_t row_start_s[kMaxRowsInKernelPlan], row_limit_s[kMaxRowsInKernelPlan];
  auto aborted = [&]() -> bool { return __any_sync(0xffffffffu, abort_s != 0); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int dim_base = 256 * (int)rank;     // first latent dim of this CTA
  const int cluster = blockIdx.x >> 1;
  const int group = cluster / a.width, member = cluster % a.width;
  const bool gather = a.sel != nullptr;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&lat_map);
    tma_prefetch_desc(&rope_map);
    if (gather && a.gather_tma) {
      tma_prefetch_desc(&lat_rows_map);
      tma_prefetch_desc(&rope_rows_map);
    }
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], (gather && !a.gather_tma) ? 32 : 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 4);      // the exchange warps have read S
    mbar_init(&p_full, 4);      // one arrival per softmax warp
    mbar_init(&q_full, 4);      // the exchange warps have written this segment's query into TMEM
    mbar_init(&o_free, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&x_full[b], 4);   // our exchange warps have staged xout[b] (one arrival carries the
                                  // expected bytes) + the peer's remote-store bytes into xin[b]
      mbar_init(&x_free[b], 4);   // the peer's softmax warps have read xin[b] (so our copy is done)
      mbar_init(&xo_free[b], 4);  // our softmax warps have read xout[b]
    }
    mbar_init(&mma_drain, 1);
    mbar_init(&pv_drain, 1);
    abort_s = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  // Only the query is written by the launch before a fused step's decode: there
  // the softmax warps alone wait (before their first query load), and the plan
  // and the first cache loads start at once.
  if (!a.early_inputs) pdl_wait();

  const int32_t* keys_p = a.keys;
  const int32_t* prefix_p = a.prefix;
  if (a.plan_in_kernel) {
    plan_rows(a, plan_keys_s, plan_prefix_s, blockIdx.x == 0, row_start_s, row_limit_s);
    keys_p = plan_keys_s;
    prefix_p = plan_prefix_s;
    if (blockIdx.x == 0) {   // a copy in the workspace, where the planner launch puts it above 128 rows
      for (int i = threadIdx.x; i < a.n_q; i += blockDim.x) a.keys[i] = plan_keys_s[i];
      for (int i = threadIdx.x; i <= a.n_units + 1; i += blockDim.x) a.prefix[i] = plan_prefix_s[i];
    }
  }
  WorkIter it;
  it.init(a, prefix_p, group);

  auto fail = [&]() {
    abort_s = 1;
    if (a.status) atomicOr(a.status, MLA_DEVICE_TIMEOUT);
  };

  if (warp == 0) {
    // ============================================================ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_phase[STAGES];
    bool issued[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued[s] = false, issued_phase[s] = 0;
    int fills = 0;   // the ring's first STAGES fills need no free slot
    int u, n, t0, t1;
    bool whole;
    while (!aborted() && it.next(u, t0, t1, whole)) {
      if (!member_segment(a, keys_p, u, member, n, t0, t1)) continue;
      const int b = n / a.s_q;
      const int start = a.plan_in_kernel ? row_start_s[n] : (a.kv_start ? a.kv_start[b] : 0);
      const int limit = a.plan_in_kernel ? row_limit_s[n] : row_limit(a, n);
      const int keys = keys_p[n];
      const int zb = a.batch_in_map ? b : 0;
      const int32_t* list = (gather && a.sel_count[n] != -1) ? a.sel + (int64_t)n * a.k_max : nullptr;
      if (!gather && lane == 0) {
        // the segment's first tiles that the loop's look-ahead will not cover
        for (int t = t0 + STAGES; t < t0 + kPrefetchAhead && t < t1; ++t) {
          for (int c = 0; c < 4; ++c) tma_prefetch_l2_3d(&lat_map, dim_base + 64 * c, start + t * BN, zb);
          tma_prefetch_l2_3d(&rope_map, 32 * (int)rank, start + t * BN, zb);
        }
      }
      for (int t = t0; t < t1 && !aborted(); ++t) {
        if (fills++ >= STAGES && !mbar_wait_warp(&empty_bar[stage], phase ^ 1u, kWaitLimit)) { fail(); break; }
        if (!gather) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&full_bar[stage], STAGE_TX);
            uint8_t* dst = stages + stage * STAGE_BYTES;
            const int y = start + t * BN;
            for (int c = 0; c < 4; ++c)
              tma_load_3d(dst + c * CHUNK_BYTES, &lat_map, &full_bar[stage], dim_base + 64 * c, y, zb);
            tma_load_3d(dst + 4 * CHUNK_BYTES, &rope_map, &full_bar[stage], 32 * (int)rank, y, zb);
            // Pull a tile a few steps ahead into L2, so that refilling a stage
            // once it frees costs an L2 rather than an HBM round trip.
            if (t + kPrefetchAhead < t1) {
              const int yp = y + kPrefetchAhead * BN;
              for (int c = 0; c < 4; ++c) tma_prefetch_l2_3d(&lat_map, dim_base + 64 * c, yp, zb);
              tma_prefetch_l2_3d(&rope_map, 32 * (int)rank, yp, zb);
            }
          }
        } else if (a.gather_tma) {
          // Row gather by TMA: 16 groups of four keys, one gather4 per 64-dim
          // chunk, shared by this warp and the extra gather warps (a warp
          // issues them one lane at a time, ~100 cycles each): issuer i takes
          // groups i, i + issuers, ...  The other issuers' copies complete on
          // the same barrier, whose expected bytes this warp announces for
          // the whole stage.
          if (lane == 0) mbar_arrive_expect_tx(&full_bar[stage], STAGE_TX);
          __syncwarp();
          constexpr int kIssuers = 1 + (kThreads - THREADS) / 32;
          if (kIssuers * lane < BN / 4)
            gather_key_group(a, &lat_rows_map, &rope_rows_map, stages + stage * STAGE_BYTES, &full_bar[stage],
                             kIssuers * lane, t, b, start, limit, keys, list, rank, dim_base);
        } else {
          // Row gather: lane L owns keys L and L+32 of the tile.
          const int e0 = t * BN + lane, e1 = e0 + 32;
          int p0 = e0, p1 = e1;
          bool v0 = e0 < keys, v1 = e1 < keys;
          if (list) {
            p0 = v0 ? list[e0] : 0;
            p1 = v1 ? list[e1] : 0;
            const bool b0 = v0 && (p0 < 0 || p0 >= limit), b1 = v1 && (p1 < 0 || p1 >= limit);
            if ((b0 || b1) && a.status && rank == 0) atomicOr(a.status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
            v0 = v0 && !b0;
            v1 = v1 && !b1;
          }
          const uint32_t dst0 = smem_u32(stages + stage * STAGE_BYTES);
          const int64_t lat_b = (int64_t)b * a.latent_batch_stride, rope_b = (int64_t)b * a.rope_batch_stride;
          for (int r = 0; r < BN; ++r) {
            const int src_lane = r & 31;
            const int pr = __shfl_sync(0xffffffffu, r < 32 ? p0 : p1, src_lane);
            const bool vr = __shfl_sync(0xffffffffu, r < 32 ? v0 : v1, src_lane);
            const int64_t row = (int64_t)start + (vr ? pr : 0);
            const __nv_bfloat16* lrow = a.latent + lat_b + row * a.latent_row_stride + dim_base;
            const __nv_bfloat16* rrow = a.rope + rope_b + row * a.rope_row_stride + 32 * (int)rank;
            // 32 16-byte pieces of the latent dims (128-byte swizzle: piece u
            // of row r at u ^ (r % 8)), then 4 of the rope dims (64-byte
            // swizzle: piece u of row r at u ^ ((r / 2) % 4))
            for (int q16 = lane; q16 < 36; q16 += 32) {
              const __nv_bfloat16* src;
              uint32_t dst;
              if (q16 < 32) {
                const int c = q16 >> 3, uu = q16 & 7;
                src = lrow + c * 64 + uu * 8;
                dst = dst0 + c * CHUNK_BYTES + r * 128 + ((uu ^ (r & 7)) << 4);
              } else {
                const int uu = q16 - 32;
                src = rrow + uu * 8;
                dst = dst0 + 4 * CHUNK_BYTES + r * 64 + ((uu ^ ((r >> 1) & 3)) << 4);
              }
              cp_async_16(dst, src, vr ? 16u : 0u);
            }
          }
          cp_async_arrive_noinc(&full_bar[stage]);
        }
        issued[stage] = true;
        issued_phase[stage] = phase;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
    }
    // Drain: every issued fill must land before this CTA may exit.
    for (int s = 0; s < STAGES; ++s)
      if (issued[s]) mbar_wait(&full_bar[s], issued_phase[s], kWaitLimit);
  } else if (warp == 1) {
    // ============================================================ score MMA issuer
    // S(t) as soon as tile t has landed and the exchange warps have read S(t-1);
    // the P.V issuer (warp 10) runs independently, so scores run ahead.
    const uint32_t idesc_s = idesc_bf16_f32(128, BN, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t tile = 0;      // global tile counter (S phases)
    uint32_t seg = 0;       // segment counter (q_full phases)
    int u, n, t0, t1;
    bool whole;
    while (!aborted() && it.next(u, t0, t1, whole)) {
      if (!member_segment(a, keys_p, u, member, n, t0, t1)) continue;
      const int keys = keys_p[n];
      if (!mbar_wait_warp(&q_full, seg & 1u, kWaitLimit)) { fail(); break; }
      for (int t = t0; t < t1; ++t) {
        if (!mbar_wait_warp(&full_bar[stage], phase, kWaitLimit)) { fail(); break; }
        if (!gather && t == (keys - 1) / BN && (keys % BN) != 0) {
          // Tail tile: clear the rows past the window so that P = 0 never meets
          // a non-finite value left in the caller's buffer.
          const int valid = keys % BN;
          uint8_t* st = stages + stage * STAGE_BYTES;
          for (int q16 = lane; q16 < (BN - valid) * 4 * 8; q16 += 32) {
            const int c = q16 / ((BN - valid) * 8), rem = q16 % ((BN - valid) * 8);
            const int r = valid + rem / 8, uu = rem % 8;
            *reinterpret_cast<uint4*>(st + c * CHUNK_BYTES + r * 128 + uu * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (gather && !a.gather_tma) fence_proxy_async_smem();
        if (tile > 0 && !mbar_wait_warp(&s_free, (tile - 1) & 1u, kWaitLimit)) { fail(); break; }
        tc_fence_after();
        // 16 latent K-steps, then this CTA's two rope K-steps.  Descriptors
        // differ only in the start address (16-byte units, low bits); one
        // elected lane of the converged warp issues them with constant
        // offsets (a lane-0 branch with per-MMA descriptor arithmetic issues
        // the N=64 MMAs at about half the rate).
        const uint64_t d0 = smem_desc(smem_u32(stages + stage * STAGE_BYTES), 16, 1024, kSwizzle128B);
        // this CTA's 32 rope dims: 64-byte rows, 8-row groups 512 bytes apart
        const uint64_t d_rope =
            smem_desc(smem_u32(stages + stage * STAGE_BYTES + 4 * CHUNK_BYTES), 16, 512, kSwizzle64B);
        if (elect_one()) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ts(tmem + TM_S, tmem + TM_Q + c * 32 + k * 8, d0 + (uint64_t)((c * CHUNK_BYTES + k * 32) >> 4),
                     idesc_s, (c | k) != 0);
          }
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_ts(tmem + TM_S, tmem + TM_Q + 128 + k * 8, d_rope + (uint64_t)((k * 32) >> 4), idesc_s, 1u);
          mma_commit(&s_full);
        }
        __syncwarp();
        ++tile;
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
      if (aborted()) break;
      ++seg;
    }
    // All score MMAs complete before TMEM is released.
    if (lane == 0) mma_commit(&mma_drain);
    __syncwarp();
    mbar_wait_warp(&mma_drain, 0, kWaitLimit);
  } else if (warp == 10) {
    // ============================================================ P.V MMA issuer
    const uint32_t idesc_pv = idesc_bf16_f32(128, DV, 0, 1);
    int stage = 0;
    uint32_t tile = 0, seg = 0;
    int u, n, t0, t1;
    bool whole;
    while (!aborted() && it.next(u, t0, t1, whole)) {
      if (!member_segment(a, keys_p, u, member, n, t0, t1)) continue;
      for (int t = t0; t < t1; ++t) {
        const bool first = (t == t0);
        // O is overwritten by a segment's first P.V: the previous segment's
        // epilogue must have read it.
        if (first && seg > 0 && !mbar_wait_warp(&o_free, (seg - 1) & 1u, kWaitLimit)) { fail(); break; }
        if (!mbar_wait_warp(&p_full, tile & 1u, kWaitLimit)) { fail(); break; }
        tc_fence_after();
        const uint64_t d0 = smem_desc(smem_u32(stages + stage * STAGE_BYTES), CHUNK_BYTES, 1024, kSwizzle128B);
        const uint32_t acc0 = first ? 0u : 1u;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < BN / 16; ++k)
            mma_ts(tmem + TM_O, tmem + TM_P + k * 8, d0 + (uint64_t)((k * 2048) >> 4), idesc_pv,
                   k == 0 ? acc0 : 1u);
          // one commit: the stage barrier also tells the softmax warps that
          // this P.V has completed (a second commit costs its own latency)
          mma_commit(&empty_bar[stage]);
        }
        __syncwarp();
        ++tile;
        if (++stage == STAGES) stage = 0;
      }
      if (aborted()) break;
      ++seg;
    }
    if (lane == 0) mma_commit(&pv_drain);
    __syncwarp();
    mbar_wait_warp(&pv_drain, 0, kWaitLimit);
  } else if (kThreads > THREADS && warp >= kGatherWarp) {
    // ============================================================ extra gather warps
    // Their share of the TMA row gathers of every tile (selected positions
    // only), following the producer's tiles, stages and stage waits.
    constexpr int kIssuers = 1 + (kThreads - THREADS) / 32;
    const int issuer = 1 + (warp - kGatherWarp);
    if (gather && a.gather_tma) {
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      int u, n, t0, t1;
      bool whole;
      while (!aborted() && it.next(u, t0, t1, whole)) {
        if (!member_segment(a, keys_p, u, member, n, t0, t1)) continue;
        const int b = n / a.s_q;
        const int start = a.plan_in_kernel ? row_start_s[n] : (a.kv_start ? a.kv_start[b] : 0);
        const int limit = a.plan_in_kernel ? row_limit_s[n] : row_limit(a, n);
        const int keys = keys_p[n];
        const int32_t* list = a.sel_count[n] != -1 ? a.sel + (int64_t)n * a.k_max : nullptr;
        for (int t = t0; t < t1 && !aborted(); ++t) {
          if (fills++ >= STAGES && !mbar_wait_warp(&empty_bar[stage], phase ^ 1u, kWaitLimit)) { fail(); break; }
          const int g = issuer + kIssuers * lane;
          if (g < BN / 4)
            gather_key_group(a, &lat_rows_map, &rope_rows_map, stages + stage * STAGE_BYTES, &full_bar[stage], g, t,
                             b, start, limit, keys, list, rank, dim_base);
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ============================================================ exchange warps
    // Read this CTA's partial scores from TMEM, round them to fp16 (saturating)
    // and send them to the peer with remote stores, one tile ahead of the
    // softmax warps (two send and two receive buffers).
    const int quarter = warp & 3;
    const int h = 32 * quarter + lane;
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const bool issuer = (h == 0);
    const uint32_t xin_peer = mapa(smem_u32(xin), peer);
    uint32_t x_full_peer[2];
    x_full_peer[0] = mapa(smem_u32(&x_full[0]), peer);
    x_full_peer[1] = mapa(smem_u32(&x_full[1]), peer);
    if (a.early_inputs) pdl_wait();   // the query comes from the launch before this one
    uint32_t tile = 0;
    float half_max = 0.f;   // largest |half score| sent (checked against the fp16 exchange's range)
    int u, n, t0, t1;
    bool whole;
    while (!aborted() && it.next(u, t0, t1, whole)) {
      if (!member_segment(a, keys_p, u, member, n, t0, t1)) continue;
      {
        // This head's query (this CTA's latent dims [dim_base, dim_base+256)
        // into TMEM columns 0..127 of Q, its rope dims [32*rank, 32*rank+32)
        // into columns 128..143).  Every score MMA of the previous segment has
        // completed (its last scores were read here), so Q is free; the
        // softmax warps may still be finishing that segment meanwhile.
        const __nv_bfloat16* qrow = a.q + (int64_t)n * a.q_row_stride + (int64_t)h * a.q_head_stride;
        const bool real = h < a.heads;   // rows past the head count stay zero
        {
          // all 36 loads in flight at once: 256 latent dims, then the 32 rope dims
          uint4 qv[36];
          const uint4* qlat = reinterpret_cast<const uint4*>(qrow + dim_base);
          const uint4* qrope = reinterpret_cast<const uint4*>(qrow + RANK + 32 * (int)rank);
#pragma unroll
          for (int v = 0; v < 32; ++v) qv[v] = real ? __ldg(qlat + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int v = 0; v < 4; ++v) qv[32 + v] = real ? __ldg(qrope + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
#pragma unroll
            for (int v = 0; v < 8; ++v)
              r[4 * v] = qv[8 * c + v].x, r[4 * v + 1] = qv[8 * c + v].y, r[4 * v + 2] = qv[8 * c + v].z,
              r[4 * v + 3] = qv[8 * c + v].w;
            tmem_st32(tmem + TM_Q + c * 32 + lane_off, r);
          }
          uint32_t r[16];
#pragma unroll
          for (int v = 0; v < 4; ++v)
            r[4 * v] = qv[32 + v].x, r[4 * v + 1] = qv[32 + v].y, r[4 * v + 2] = qv[32 + v].z, r[4 * v + 3] = qv[32 + v].w;
          tmem_st16(tmem + TM_Q + 128 + lane_off, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full);
      }
      // A few tiles before this segment ends, the next segment's query row
      // (this head's 512 + 64 bytes) is pulled into L2 -- and its address
      // translation warmed -- so that loading it at the boundary is an L2 hit.
      // Earlier would not do: the cache tiles streamed meanwhile evict it.
      const int t_pf = t1 - kQueryPrefetchTiles > t0 ? t1 - kQueryPrefetchTiles : t0;
      for (int t = t0; t < t1; ++t) {
        if (t == t_pf) {
          WorkIter peek = it;
          int un, nn, tn0, tn1;
          bool wn;
          while (peek.next(un, tn0, tn1, wn)) {
            if (!member_segment(a, keys_p, un, member, nn, tn0, tn1)) continue;
            if (h < a.heads) {
              const __nv_bfloat16* qnext = a.q + (int64_t)nn * a.q_row_stride + (int64_t)h * a.q_head_stride;
#pragma unroll
              for (int l = 0; l < 4; ++l) prefetch_l2(qnext + dim_base + 64 * l);
              prefetch_l2(qnext + RANK + 32 * (int)rank);
            }
            break;
          }
        }
        const uint32_t b = tile & 1u, use = tile >> 1;
        if (tile >= 2) {
          // the peer has read our copy of tile-2 (so xout[b] is read too), and
          // our softmax warps have read their own half of it
          // (a signal only: the peer's reads of that buffer completed before its
          // arrive, so a CTA-scope wait suffices)
          if (!mbar_wait_warp(&x_free[b], (use - 1) & 1u, kWaitLimit)) { fail(); break; }
          if (!mbar_wait_warp(&xo_free[b], (use - 1) & 1u, kWaitLimit)) { fail(); break; }
        }
        if (!mbar_wait_warp(&s_full, tile & 1u, kWaitLimit)) { fail(); break; }
        tc_fence_after();
        uint32_t sa[32], sb[32];
        tmem_ld32(tmem + TM_S + lane_off, sa);
        tmem_ld32(tmem + TM_S + 32 + lane_off, sb);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free);
        // Each 16-byte piece goes to our own softmax warps (xout) and, as an
        // asynchronous remote store that completes on the peer's x_full, into
        // the peer's receive buffer: no staging round trip, no bulk copy.
        uint8_t* xo = xout + b * XH_BYTES;
        const uint32_t xi = xin_peer + b * XH_BYTES;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int k = 8 * c + 2 * q;   // scores k, k+1
            const float lo_raw = __uint_as_float(k < 32 ? sa[k] : sb[k - 32]);
            const float hi_raw = __uint_as_float(k < 32 ? sa[k + 1] : sb[k - 31]);
            half_max = fmax3(half_max, fabsf(lo_raw), fabsf(hi_raw));
            // sent already scaled (log2 units): the softmax then only adds
            const float2 sc = mul_f32x2(make_float2(lo_raw, hi_raw), make_float2(a.scale_log2, a.scale_log2));
            const __half2 hv = __floats2half2_rn(fminf(fmaxf(sc.x, -65504.f), 65504.f), fminf(fmaxf(sc.y, -65504.f), 65504.f));
            w[q] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          *reinterpret_cast<uint4*>(xo + (c * 128 + h) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          st_async_v4(xi + (uint32_t)((c * 128 + h) * 16), w[0], w[1], w[2], w[3], x_full_peer[b]);
        }
        __syncwarp();
        // xout[b] is written by this warp; receive buffer b expects the peer's
        // XH_BYTES for this tile (announced by one of the four arrivals).
        if (issuer)
          mbar_arrive_expect_tx_u32(smem_u32(&x_full[b]), XH_BYTES);
        else if (lane == 0)
          mbar_arrive(&x_full[b]);
        ++tile;
      }
    }
    // Padding rows (heads >= a.heads) score 0; a key row past the window
    // holds zeros.  So any half beyond the limit is a real score.
    if (__any_sync(0xffffffffu, !(half_max <= MLA_FP16_SCORE_LIMIT)) && lane == 0 && a.status)
      atomicOr(a.status, MLA_DEVICE_SCORE_RANGE);
  } else {
    // ============================================================ softmax / epilogue
    if (a.early_inputs) pdl_wait();   // the query comes from the launch before this one
    const int quarter = warp & 3;
    const int h = 32 * quarter + lane;                    // head = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    uint32_t x_free_peer[2];
    x_free_peer[0] = mapa(smem_u32(&x_free[0]), peer);
    x_free_peer[1] = mapa(smem_u32(&x_free[1]), peer);
    uint32_t tile = 0, seg = 0;
    // P.V(k) has completed once its commit arrives on the stage barrier
    // empty_bar[k % STAGES] (that barrier's (k / STAGES)-th completion).  P.V's
    // complete in order, and when P.V(k) is waited for, P.V(k - STAGES) has
    // been waited for already and P.V(k + STAGES) cannot have started, so the
    // phase parity identifies the completion.
    auto wait_pv = [&](uint32_t k) -> bool {
      return mbar_wait_warp(&empty_bar[k % STAGES], (k / STAGES) & 1u, kWaitLimit);
    };
    int u, n, t0, t1;
    bool whole;
    while (!aborted() && it.next(u, t0, t1, whole)) {
      const bool any = member_segment(a, keys_p, u, member, n, t0, t1);
      const int64_t slot = ((int64_t)u + group) * a.width + member;
      if (!any) {
        // Nothing of this row in the group's range: an empty partial (weight 0).
        if (!whole && rank == 0 && h < a.heads) {
          a.ws_ml[(slot * 2) * HEADS + h] = -CUDART_INF_F;
          a.ws_ml[(slot * 2 + 1) * HEADS + h] = 0.f;
        }
        continue;
      }
      const int keys = keys_p[n];
      const int limit = a.plan_in_kernel ? row_limit_s[n] : row_limit(a, n);
      const int32_t* list = (gather && a.sel_count[n] != -1) ? a.sel + (int64_t)n * a.k_max : nullptr;
      float m_used = -CUDART_INF_F, l = 0.f;
      bool first_tile = true;
      bool p_pending = false;   // kLateP: the previous tile's P is not yet announced
      // Selected positions of the lane's two entries of the next tile, read a
      // tile ahead so that their load is not on the path of the tile's scores.
      int pos0 = 0, pos1 = 0;
      if (list) {
        const int e0 = t0 * BN + lane, e1 = e0 + 32;
        if (e0 < keys) pos0 = __ldg(list + e0);
        if (e1 < keys) pos1 = __ldg(list + e1);
      }
      for (int t = t0; t < t1; ++t) {
        // ---- validity of this tile's 64 entries (lane L: entries L, L+32);
        // a whole tile of a dense row needs no check (warp-uniform test)
        uint64_t valid = ~0ull;
        if (list != nullptr || (t + 1) * BN > keys) {
          const int e0 = t * BN + lane, e1 = e0 + 32;
          bool v0 = e0 < keys, v1 = e1 < keys;
          if (list) {
            v0 = v0 && pos0 >= 0 && pos0 < limit;
            v1 = v1 && pos1 >= 0 && pos1 < limit;
            if (t + 1 < t1) {
              if (e0 + BN < keys) pos0 = __ldg(list + e0 + BN);
              if (e1 + BN < keys) pos1 = __ldg(list + e1 + BN);
            }
          }
          valid = (uint64_t)__ballot_sync(0xffffffffu, v0) | ((uint64_t)__ballot_sync(0xffffffffu, v1) << 32);
        }
        // ---- both halves present: our own (staged by the exchange warps) and
        // the peer's (its remote stores complete as transaction bytes on this
        // local barrier, which makes them visible to the threads that observe
        // the phase: a CTA-scope acquire, as for a TMA load)
        const uint32_t b = tile & 1u, use = tile >> 1;
        if (!mbar_wait_warp(&x_full[b], use & 1u, kWaitLimit)) { fail(); break; }
        if (kLateP && p_pending) {
          if (lane == 0) mbar_arrive(&p_full);
          p_pending = false;
        }
        // ---- x = own + peer - m_ref in the log2 domain (both halves arrive
        // already scaled), as two fp16-operand additions per score (exact
        // conversions, f32 arithmetic), relative to the running maximum m_ref
        // (0 before any entry was seen).
        // The two CTAs of a pair may round x differently (they take the halves
        // in opposite order); each normalises its own half of the context by
        // its own sum, so the results stay consistent.
        const float m_ref = (m_used == -CUDART_INF_F) ? 0.f : m_used;
        if (valid != ~0ull) {
          // Entries past the window or out of range: this head's own half in
          // xout[b] becomes fp16 -inf, so that x = -inf whatever the peer's
          // (finite) half.  A rolled loop with computed addresses: it runs at a
          // row's last tile only, where an unrolled masking pass would be
          // fetched cold into the instruction cache.
          const uint32_t row = smem_u32(xout + b * XH_BYTES) + (uint32_t)h * 16u;
          uint64_t inv = ~valid;
#pragma unroll 1
          while (inv != 0ull) {
            const int k = __ffsll((long long)inv) - 1;
            inv &= inv - 1ull;
            st_shared_u16(row + (uint32_t)((k >> 3) * 128 * 16 + (k & 7) * 2), 0xFC00u);
          }
        }
        float x[BN];
        {
          const uint8_t* xo = xout + b * XH_BYTES;
          const uint8_t* xi = xin + b * XH_BYTES;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 o4 = *reinterpret_cast<const uint4*>(xo + (c * 128 + h) * 16);
            const uint4 i4 = *reinterpret_cast<const uint4*>(xi + (c * 128 + h) * 16);
            const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, iw[4] = {i4.x, i4.y, i4.z, i4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              x[8 * c + 2 * q] = add_f16lo(iw[q], add_f16lo(ow[q], -m_ref));
              x[8 * c + 2 * q + 1] = add_f16hi(iw[q], add_f16hi(ow[q], -m_ref));
            }
          }
        }
        // ---- tile maximum (three-input max tree), relative to m_ref
        float mx;
        {
          float m21[22];
#pragma unroll
          for (int k = 0; k < 21; ++k) m21[k] = fmax3(x[3 * k], x[3 * k + 1], x[3 * k + 2]);
          m21[21] = x[63];
          float m7[8];
#pragma unroll
          for (int k = 0; k < 7; ++k) m7[k] = fmax3(m21[3 * k], m21[3 * k + 1], m21[3 * k + 2]);
          m7[7] = m21[21];
          mx = fmax3(fmax3(m7[0], m7[1], m7[2]), fmax3(m7[3], m7[4], m7[5]), fmaxf(m7[6], m7[7]));
        }
        // Every score above fed mx, so the warp holds all of this tile's send
        // and receive data: free both buffers with relaxed arrives ordered by
        // that dependency (a release arrive costs a cluster-scope fence per tile).
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_relaxed_dep(&xo_free[b], __float_as_uint(mx));
          mbar_arrive_remote_relaxed_dep(x_free_peer[b], __float_as_uint(mx));
        }
        // ---- online softmax with lazy rescaling: the reference moves only
        // when the tile maximum exceeds it by more than the threshold (or on
        // the first visible entry); p = 2^(x - shift).
        float alpha = 1.f, shift = 0.f;
        bool rescale = false;
        if (mx != -CUDART_INF_F && (mx > kRescaleThreshold || m_used == -CUDART_INF_F)) {
          alpha = (m_used == -CUDART_INF_F) ? 0.f : ex2_approx(-mx);
          rescale = !first_tile && m_used != -CUDART_INF_F;
          m_used = m_ref + mx;
          shift = mx;
        }
        uint32_t pk[32];
        float2 ps2[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ps2[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < BN; k += 2) {
          const float2 xs = add_f32x2(make_float2(x[k], x[k + 1]), make_float2(-shift, -shift));
          const float p0 = ex2_approx(xs.x);
          const float p1 = ex2_approx(xs.y);
          ps2[(k >> 1) & 7] = add_f32x2(ps2[(k >> 1) & 7], make_float2(p0, p1));
          const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
          pk[k >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
        }
        ps2[0] = add_f32x2(add_f32x2(ps2[0], ps2[1]), add_f32x2(ps2[2], ps2[3]));
        ps2[4] = add_f32x2(add_f32x2(ps2[4], ps2[5]), add_f32x2(ps2[6], ps2[7]));
        ps2[0] = add_f32x2(ps2[0], ps2[4]);
        const float psum = ps2[0].x + ps2[0].y;
        l = l * alpha + psum;
        // ---- P into TMEM once the previous P.V has consumed it (and O is stable)
        if (tile > 0 && !wait_pv(tile - 1)) { fail(); break; }
        tc_fence_after();
        // tcgen05.ld / st are warp-collective: the whole warp takes the
        // rescale pass when any of its heads needs it, the others with factor 1.
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + TM_O + c * 32 + lane_off, o);
            tmem_wait_ld_regs(o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
            tmem_st32(tmem + TM_O + c * 32 + lane_off, o);
          }
        }
        tmem_st32(tmem + TM_P + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (kLateP && t + 1 < t1)
          p_pending = true;
        else if (lane == 0)
          mbar_arrive(&p_full);
        first_tile = false;
        ++tile;
      }
      if (aborted()) break;
      // ---- epilogue: wait for the segment's last P.V
      if (!wait_pv(tile - 1)) { fail(); break; }
      tc_fence_after();
      // O leaves TMEM 32 columns at a time, the next chunk's load in flight
      // while the current one is stored.
      auto drain_o = [&](auto&& store_chunk) {
        uint32_t oa[32], ob[32];
        tmem_ld32(tmem + TM_O + lane_off, oa);
        // rolled: the epilogue runs once per segment, so its code is fetched
        // cold; four copies of the chunk stores would cost more than the loop
#pragma unroll 1
        for (int c = 0; c < DV / 32; c += 2) {
          tmem_wait_ld_regs(oa);
          tmem_ld32(tmem + TM_O + (c + 1) * 32 + lane_off, ob);
          store_chunk(c, oa);
          tmem_wait_ld_regs(ob);
          if (c + 2 < DV / 32) tmem_ld32(tmem + TM_O + (c + 2) * 32 + lane_off, oa);
          store_chunk(c + 1, ob);
        }
      };
      if (h >= a.heads) {
        // a padding row: nothing to store
      } else if (whole) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int64_t off = (int64_t)n * a.ctx_row_stride + (int64_t)h * a.ctx_head_stride + dim_base;
        if (a.out_f32) {
          drain_o([&](int c, const uint32_t(&o)[32]) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.ctx) + off + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                   __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
          });
        } else {
          drain_o([&](int c, const uint32_t(&o)[32]) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.ctx) + off + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                                  pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          });
        }
        if (rank == 0 && a.lse)
          a.lse[(int64_t)n * a.heads + h] = l > 0.f ? (m_used + log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      } else {
        // Partial as [slot][RANK/8][H] entries of 8 fp16 dims: this piece's
        // context normalised by its own sum (O / l, an average of latent
        // rows, so within the range of the cache's values), with (m, l) in
        // f32 beside it.  A thread stores 8 dims of its head as one 16-byte
        // vector, a warp 512 B contiguous.  Stored with an evict-last L2
        // policy: the combine reads them after the whole decode, and the
        // cache stream would otherwise push the early pieces out to DRAM.
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const uint64_t keep = l2_policy_evict_last();
        uint4* dst = a.ws_o + (slot * (RANK / 8) + dim_base / 8) * HEADS + h;
        float vmax = 0.f;
        drain_o([&](int c, const uint32_t(&o)[32]) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float x0 = __uint_as_float(o[8 * q + 2 * j]) * inv, x1 = __uint_as_float(o[8 * q + 2 * j + 1]) * inv;
              vmax = fmaxf(vmax, fmaxf(fabsf(x0), fabsf(x1)));   // beyond 65504 the fp16 value is infinite
              const __half2 hv = __floats2half2_rn(x0, x1);
              w[j] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            st_global_v4_policy(dst + (int64_t)(4 * c + q) * HEADS, make_uint4(w[0], w[1], w[2], w[3]), keep);
          }
        });
        if (!(vmax <= 65504.f) && a.status) atomicOr(a.status, MLA_DEVICE_VALUE_RANGE);
        if (rank == 0) {
          st_global_f32_policy(a.ws_ml + (slot * 2) * HEADS + h, l > 0.f ? m_used : -CUDART_INF_F, keep);
          st_global_f32_policy(a.ws_ml + (slot * 2 + 1) * HEADS + h, l, keep);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free);
      ++seg;
    }
  }

  // ---------------------------------------------------------------- teardown
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // the peer no longer writes into this CTA's shared memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ combine
// 8 fp16 dims of a stored partial (loaded as one 16-byte vector), as f32.
__device__ __forceinline__ uint4 ld_partial(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ void unpack_partial(const uint4 r, float (&x)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
    x[2 * j] = f.x;
    x[2 * j + 1] = f.y;
  }
}

// grid (n_q, RANK / CDIMS); 128 threads, thread h < heads merges dims
// [d0, d0 + CDIMS) of head h over the row's pieces.  Partials are stored as
// [slot][RANK/8][H] entries of 8 fp16 dims, so a warp's 16-byte loads per
// piece read 512 B.  The loads of up to kCombineBatch pieces are issued
// together, and batches are merged online.  Few rows have many pieces each
// (one row of 4096 keys: 16) and a small grid, many rows a few pieces each and
// a grid of several thousand CTAs: the batch is chosen per launch, since its
// registers bound the CTAs resident per SM.
constexpr int CDIMS = 8;
constexpr int kCombineWideRows = 8;   // rows up to which the combine loads 16 pieces at once

template <int kCombineBatch>
__global__ void __launch_bounds__(128) tc_combine_kernel(const __grid_constant__ TcDecodeArgs a) {
  __shared__ int32_t keys_s[kMaxRowsInKernelPlan];
  __shared__ int32_t prefix_s[kMaxRowsInKernelPlan + 2];
  const int n = blockIdx.x;
  const int d0 = blockIdx.y * CDIMS;
  const int h = threadIdx.x;
  const int u = n / a.width, member = n % a.width;
  // The row's pieces, before the wait.  The plan depends only on the call's
  // inputs and, above kMaxRowsInKernelPlan rows, on the planner launch: every
  // decode CTA passes its own dependency wait before it lets this grid start,
  // so all of those launches have completed.  (The copy of an in-kernel plan
  // that the decode kernel stores is not read: it is visible only after the
  // wait.)
  int keys;
  const int32_t* prefix;
  if (a.plan_in_kernel) {
    plan_rows(a, keys_s, prefix_s, false);   // 128 threads >= n_q
    keys = keys_s[n];
    prefix = prefix_s;
  } else {
    keys = a.keys[n];
    prefix = a.prefix;
  }
  int c0 = 0, c1 = 0;
  if (keys != 0) {
    const int per = group_span(a, prefix[a.n_units]);
    c0 = first_group_of(prefix, u, per, prefix[a.n_units + 1]);
    c1 = last_group_of(prefix, u, per);
  }
  pdl_wait();
  if (h >= a.heads) return;
  const int64_t orow = (int64_t)n * a.ctx_row_stride + (int64_t)h * a.ctx_head_stride + d0;
  float acc[CDIMS];
#pragma unroll
  for (int j = 0; j < CDIMS; ++j) acc[j] = 0.f;
  float M = -CUDART_INF_F, L = 0.f;
  static_assert(CDIMS == 8, "one 8-dim group of the partial layout per thread");
  bool write = true;
  if (keys != 0) {
    if (c0 == c1) {
      write = false;                       // finished in place by its group
    } else {
      auto slot_of = [&](int g) -> int64_t { return ((int64_t)u + g) * a.width + member; };
      for (int cb = c0; cb <= c1; cb += kCombineBatch) {
        float mq[kCombineBatch], lq[kCombineBatch];
        uint4 raw[kCombineBatch];
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
          mq[q] = -CUDART_INF_F;
          lq[q] = 0.f;
          raw[q] = make_uint4(0, 0, 0, 0);
          if (cb + q <= c1) {
            const int64_t sl = slot_of(cb + q);
            mq[q] = a.ws_ml[(sl * 2) * HEADS + h];
            lq[q] = a.ws_ml[(sl * 2 + 1) * HEADS + h];
            raw[q] = ld_partial(a.ws_o + (sl * (RANK / 8) + d0 / 8) * HEADS + h);
          }
        }
        float mb = M;
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) mb = fmaxf(mb, mq[q]);
        if (mb == -CUDART_INF_F) continue;   // every piece so far is empty
        const float f = exp2f(M - mb);       // 0 while M is still -inf
        L *= f;
#pragma unroll
        for (int j = 0; j < CDIMS; ++j) acc[j] *= f;
        M = mb;
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
          // the piece's weight e^(m - M) l; an empty piece (m = -inf) has weight
          // 0 and its context, never written, is not read into the sum
          const float w = mq[q] != -CUDART_INF_F ? exp2f(mq[q] - M) * lq[q] : 0.f;
          L += w;
          float x[CDIMS];
          unpack_partial(raw[q], x);
#pragma unroll
          for (int j = 0; j < CDIMS; ++j) acc[j] = (w != 0.f) ? fmaf(w, x[j], acc[j]) : acc[j];
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int j = 0; j < CDIMS; ++j) acc[j] *= inv;
    }
  }
  if (write) {
    if (a.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.ctx) + orow);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.ctx) + orow) =
          make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                     pack_bf16x2(acc[6], acc[7]));
    }
    if (blockIdx.y == 0 && a.lse)
      a.lse[(int64_t)n * a.heads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
  }
}

// ------------------------------------------------------------------ combine + W_UV projection
// The fused tail of a decode step: grid (heads), 512 threads.  CTA h merges
// the split partials of head h for every query row into the bf16 context rows
// (the rows finished in place are read back from the context buffer), lays
// them out as the K-major B operand [npad rows x 512] of a tcgen05 MMA in
// shared memory, and multiplies by W_UV_h [128 x 512] (A, TMA-loaded) into
// out[n, h*128 + j] -- the same contraction as mla_project_v.
struct ProjectTail {
  void* out;
  int64_t out_row_stride;
  int32_t out_f32;
  int32_t npad;               // n_q rounded up to 16 (the MMA's N)
  int32_t v_dim;
  int32_t w_row0, w_head_rows;  // W_UV_h starts at row h*w_head_rows + w_row0
};

constexpr int PROJ_THREADS = 512;   // 8 groups of 64 threads (one 8-dim group of a row each)
constexpr int PROJ_GROUPS = PROJ_THREADS / 64;
constexpr int PROJ_UNROLL = 8;      // pieces whose loads are in flight together
constexpr int PROJ_BOX_BYTES = 128 * 128;                  // [128 v rows][64 dims] bf16
constexpr int PROJ_MERGE_BYTES = PROJ_THREADS * 10 * 4;    // per thread (M, L, acc[8])
constexpr int PROJ_SMEM_MAX = 1024 + 8 * PROJ_BOX_BYTES + 8 * 64 * 128 + PROJ_MERGE_BYTES;

// Online merge of one stored split piece (m, l, O / l [8 dims]) into a running (M, L, acc).
__device__ __forceinline__ void merge_stored_piece(float& M, float& L, float (&acc)[8], float m, float l,
                                                   const float (&xn)[8]) {
  if (m == -CUDART_INF_F) return;       // an empty piece (weight 0; its context was never written)
  if (m > M) {
    const float f = exp2f(M - m);       // 0 while M is still -inf
    L *= f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] *= f;
    M = m;
  }
  const float w = exp2f(m - M) * l;
  L += w;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, xn[j], acc[j]);
}

// Online merge of one running state (m, l, O[8 dims], O unnormalised) into another (M, L, acc).
__device__ __forceinline__ void merge_piece(float& M, float& L, float (&acc)[8], float m, float l,
                                            const float (&x)[8]) {
  if (m == -CUDART_INF_F) return;       // an empty piece (weight 0; its O was never written)
  if (m > M) {
    const float f = exp2f(M - m);       // 0 while M is still -inf
    L *= f;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] *= f;
    M = m;
  }
  const float w = exp2f(m - M);
  L = fmaf(w, l, L);
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, x[j], acc[j]);
}

__global__ void __launch_bounds__(PROJ_THREADS) tc_combine_project_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                          const __grid_constant__ TcDecodeArgs a,
                                                                          const __grid_constant__ ProjectTail p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                       // 8 K-boxes of W_UV_h
  uint8_t* sB = smem + 8 * PROJ_BOX_BYTES;  // 8 K-boxes of [npad rows][64 dims] context
  __shared__ __align__(8) uint64_t bar_full[8];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base_s;
  __shared__ int mma_ok_s;
  __shared__ int32_t keys_s[kMaxRowsInKernelPlan];
  __shared__ int32_t prefix_s[kMaxRowsInKernelPlan + 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int npad = p.npad;
  const uint32_t ncols = npad <= 32 ? 32 : 64;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&wmap);
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
  // W_UV_h is not written by the decode kernel this one depends on, and every
  // launch before that kernel has completed by the time this grid starts (each
  // launch of the step lets its dependants start only after its own wait), so
  // the weight loads are issued before the wait and overlap the decode's tail.
  if (threadIdx.x == 0) {
    const int row0 = h * p.w_head_rows + p.w_row0;
    for (int i = 0; i < 8; ++i) {
      mbar_arrive_expect_tx(&bar_full[i], PROJ_BOX_BYTES);
      tma_load_2d(sA + i * PROJ_BOX_BYTES, &wmap, &bar_full[i], 64 * i, row0);
    }
  }
  // The split plan depends only on the step's inputs (complete, as above):
  // recomputed here, the same way the decode kernel computes it, before the
  // wait; the pieces' partial buffers are touched (L2 prefetch: address
  // translation and lines) so that the loads after the wait hit.
  plan_rows(a, keys_s, prefix_s, false);
  {
    const int per = group_span(a, prefix_s[a.n_units]);
    for (int n = threadIdx.x >> 5; n < a.n_q; n += PROJ_THREADS / 32) {
      if (keys_s[n] == 0) continue;
      const int u = n / a.width, member = n % a.width;
      const int c0 = first_group_of(prefix_s, u, per, prefix_s[a.n_units + 1]), c1 = last_group_of(prefix_s, u, per);
      if (c0 == c1) continue;
      for (int c = c0 + lane; c <= c1; c += 32) {
        const int64_t sl = ((int64_t)u + c) * a.width + member;
        prefetch_l2(a.ws_ml + sl * 2 * HEADS + h);
        prefetch_l2(a.ws_o + sl * (RANK / 8) * HEADS);
      }
    }
  }
  pdl_wait();

  // ---- context rows of head h into sB (bf16, 128-byte swizzle: the 16-byte
  // chunk c of row n sits at chunk c ^ (n & 7)).  Thread = (group k, 8-dim
  // group g).  With fewer than 8 query rows, `nsplit` groups share a row, each
  // merging every nsplit-th piece, and their states are merged in shared memory.
  {
    float* merge_s = reinterpret_cast<float*>(sB + 8 * npad * 128);
    const int g = threadIdx.x & 63, k = threadIdx.x >> 6;
    int rows_pow2 = 1;
    while (rows_pow2 < a.n_q && rows_pow2 < PROJ_GROUPS) rows_pow2 <<= 1;
    const int nsplit = PROJ_GROUPS / rows_pow2;        // 1, 2, 4 or 8
    const int rows_per_pass = PROJ_GROUPS / nsplit;
    const int rsub = k % nsplit;
    const int per = group_span(a, prefix_s[a.n_units]);
    // the padding rows n_q .. npad-1 of the MMA's N are zero
    for (int i = a.n_q * 64 + threadIdx.x; i < npad * 64; i += PROJ_THREADS) {
      const int n = i >> 6, gg = i & 63;
      *reinterpret_cast<uint4*>(sB + (gg >> 3) * (npad * 128) + n * 128 + (((gg & 7) ^ (n & 7)) << 4)) =
          make_uint4(0, 0, 0, 0);
    }
    // rows in passes of rows_per_pass: the same trip count in every group
    const int n_real = (a.n_q + rows_per_pass - 1) / rows_per_pass * rows_per_pass;
    for (int n = k / nsplit; n < n_real; n += rows_per_pass) {
      int kind = 0, u = 0, member = 0, c0 = 0, c1 = -1;         // 0: padding row, 1: no key, 2: whole, 3: split
      if (n < a.n_q) {
        kind = 1;
        if (keys_s[n] != 0) {
          u = n / a.width;
          member = n % a.width;
          c0 = first_group_of(prefix_s, u, per, prefix_s[a.n_units + 1]);
          c1 = last_group_of(prefix_s, u, per);
          kind = c0 == c1 ? 2 : 3;
        }
      }
      float M = -CUDART_INF_F, L = 0.f, acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
      if (kind == 3) {
        for (int c = c0 + rsub; c <= c1; c += PROJ_UNROLL * nsplit) {
          float mq[PROJ_UNROLL], lq[PROJ_UNROLL];
          uint4 raw[PROJ_UNROLL];
#pragma unroll
          for (int q = 0; q < PROJ_UNROLL; ++q) {
            mq[q] = -CUDART_INF_F;
            raw[q] = make_uint4(0, 0, 0, 0);
            const int cq = c + q * nsplit;
            if (cq <= c1) {
              const int64_t sl = ((int64_t)u + cq) * a.width + member;
              mq[q] = a.ws_ml[(sl * 2) * HEADS + h];
              lq[q] = a.ws_ml[(sl * 2 + 1) * HEADS + h];
              raw[q] = ld_partial(a.ws_o + (sl * (RANK / 8) + g) * HEADS + h);
            }
          }
#pragma unroll
          for (int q = 0; q < PROJ_UNROLL; ++q) {
            float x[8];
            unpack_partial(raw[q], x);
            merge_stored_piece(M, L, acc, mq[q], lq[q], x);
          }
        }
      }
      if (nsplit > 1) {   // uniform over the block: every thread reaches both barriers
        float* mine = merge_s + (size_t)threadIdx.x * 10;
        mine[0] = M;
        mine[1] = L;
#pragma unroll
        for (int j = 0; j < 8; ++j) mine[2 + j] = acc[j];
        __syncthreads();
        if (rsub == 0 && kind == 3) {
          for (int o = 1; o < nsplit; ++o) {
            const float* other = merge_s + (size_t)(threadIdx.x + 64 * o) * 10;
            float xo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) xo[j] = other[2 + j];
            merge_piece(M, L, acc, other[0], other[1], xo);
          }
        }
        __syncthreads();
      }
      if (rsub == 0) {
        uint4 packed = make_uint4(0, 0, 0, 0);
        if (kind == 2) {
          // finished in place by its group: bf16 context (and lse) already written
          packed = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.ctx) +
                                                   (int64_t)n * a.ctx_row_stride + (int64_t)h * a.ctx_head_stride +
                                                   8 * g);
        } else if (kind == 3) {
          const float inv = L > 0.f ? 1.f / L : 0.f;
          packed = make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                              pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
        }
        if (g == 0 && a.lse && (kind == 1 || kind == 3))
          a.lse[(int64_t)n * a.heads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
        *reinterpret_cast<uint4*>(sB + (g >> 3) * (npad * 128) + n * 128 + (((g & 7) ^ (n & 7)) << 4)) = packed;
      }
    }
  }
  fence_proxy_async_smem();   // generic-proxy writes of sB, read by the MMA
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool ok = true;
  if (warp == 0) {
    // One elected lane of the converged warp issues, descriptors = base + constants.
    const uint32_t idesc = idesc_bf16_f32(128, npad, 0, 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int i = 0; i < 8 && ok; ++i) {
      ok = mbar_wait_warp(&bar_full[i], 0, kWaitLimit);
      if (!ok) break;
      tc_fence_after();
      const uint64_t ad = smem_desc(a0 + i * PROJ_BOX_BYTES, 16, 1024, kSwizzle128B);
      const uint64_t bd = smem_desc(b0 + i * npad * 128, 16, 1024, kSwizzle128B);
      if (elect_one()) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tmem, ad + (uint64_t)((k * 32) >> 4), bd + (uint64_t)((k * 32) >> 4), idesc, (i | k) != 0);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) {
      if (a.status) atomicOr(a.status, MLA_DEVICE_TIMEOUT);
      for (int i = 0; i < 8; ++i) mbar_wait(&bar_full[i], 0, kWaitLimit);  // drain in-flight copies
    }
    if (lane == 0) mma_ok_s = ok ? 1 : 0;
    if (elect_one()) mma_commit(&bar_mma);
    __syncwarp();
  }
  __syncthreads();
  ok = mbar_wait_warp(&bar_mma, 0, kWaitLimit) && mma_ok_s != 0;
  tc_fence_after();
  if (ok) {
    // warp w reads TMEM lanes 32 (w % 4) .. +31 (v rows) and columns
    // (query rows) [16 (w / 4), +16), the blocks repeating every 64 columns
    const int lq = warp & 3;
    const uint32_t row_addr = tmem + ((uint32_t)(32 * lq) << 16);
    const int j = 32 * lq + lane;
    for (int c0 = 16 * (warp >> 2); c0 < npad; c0 += 16 * (PROJ_THREADS / 128)) {
      uint32_t r[16];
      tmem_ld16(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int n = c0 + t;
        if (n >= a.n_q) continue;
        const float v = __uint_as_float(r[t]);
        const int64_t off = (int64_t)n * p.out_row_stride + (int64_t)h * p.v_dim + j;
        if (p.out_f32)
          static_cast<float*>(p.out)[off] = v;
        else
          static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(v);
      }
    }
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

int tc_decode_clusters() { return device_sm_count() / 2; }

// The partials are laid out for the MMA's 128 rows whatever the head count.
size_t tc_decode_workspace(int32_t n_q) {
  const size_t slots = (size_t)n_q + tc_decode_clusters();
  return align256((size_t)(n_q + 2) * 4) + align256((size_t)n_q * 4) +
         align256(slots * HEADS * RANK * 2) + align256(slots * HEADS * 2 * 4);
}

cudaError_t launch_tc_decode(const DecodeGeometry& g, int out_dtype, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream, const DecodeTail* tail) {
  const int n_q = g.batch * g.s_q;
  const int nclusters = tc_decode_clusters();
  if (workspace_bytes < tc_decode_workspace(n_q)) return cudaErrorInvalidValue;
  if (g.heads != 64 && g.heads != HEADS) return cudaErrorInvalidValue;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  TcDecodeArgs a;
  a.q = static_cast<const __nv_bfloat16*>(g.q);
  a.q_row_stride = g.q_row_stride;
  a.q_head_stride = g.q_head_stride;
  a.latent = static_cast<const __nv_bfloat16*>(g.latent);
  a.latent_row_stride = g.latent_row_stride;
  a.latent_batch_stride = g.latent_batch_stride;
  a.rope = static_cast<const __nv_bfloat16*>(g.rope);
  a.rope_row_stride = g.rope_row_stride;
  a.rope_batch_stride = g.rope_batch_stride;
  a.kv_start = g.kv_start;
  a.kv_len = g.kv_len;
  a.s_q = g.s_q;
  a.n_q = n_q;
  a.heads = g.heads;
  a.sel = g.sel;
  a.sel_count = g.sel_count;
  a.k_max = g.k_max;
  a.scale_log2 = g.scale_log2;
  a.ctx = g.ctx_out;
  a.ctx_row_stride = g.ctx_row_stride;
  a.ctx_head_stride = g.ctx_head_stride;
  a.out_f32 = out_dtype == MLA_DTYPE_F32;
  a.lse = g.lse_out;
  a.status = g.device_status;
  size_t off = 0;
  a.prefix = reinterpret_cast<int32_t*>(ws + off);
  off += align256((size_t)(n_q + 2) * 4);
  a.keys = reinterpret_cast<int32_t*>(ws + off);
  off += align256((size_t)n_q * 4);
  const size_t slots = (size_t)n_q + nclusters;
  a.ws_o = reinterpret_cast<uint4*>(ws + off);
  off += align256(slots * HEADS * RANK * 2);
  a.ws_ml = reinterpret_cast<float*>(ws + off);
  a.num_clusters = nclusters;
  // A dense multi-token verify serves each batch row's tokens with a group of
  // clusters in lockstep; everything else is one query row per unit.
  a.width = (g.sel == nullptr && g.s_q > 1 && g.s_q <= 8) ? g.s_q : 1;
  a.n_units = n_q / a.width;
  a.min_tiles = kMinTilesPerGroup;
  a.batch_in_map = (g.latent_batch_stride != 0 || g.rope_batch_stride != 0) ? 1 : 0;
  a.plan_in_kernel = n_q <= kMaxRowsInKernelPlan ? 1 : 0;
  a.early_inputs = (tail != nullptr && a.plan_in_kernel) ? 1 : 0;

  // Tensor maps over [B_buf, t_max, dims] (the batch axis has extent 1 for a
  // packed-flat cache whose batch stride is 0).
  const uint64_t bmap = a.batch_in_map ? (uint64_t)g.batch : 1;
  CUtensorMap lat_map, rope_map;
  {
    const uint64_t dims[3] = {(uint64_t)g.rank, (uint64_t)g.t_max, bmap};
    const uint64_t bstride = a.batch_in_map ? (uint64_t)g.latent_batch_stride * 2
                                            : (uint64_t)g.t_max * g.latent_row_stride * 2;
    const uint64_t strides[2] = {(uint64_t)g.latent_row_stride * 2, bstride};
    const uint32_t box[3] = {64, BN, 1};
    if (!encode_tmap_bf16(&lat_map, g.latent, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {(uint64_t)g.rope_dim, (uint64_t)g.t_max, bmap};
    const uint64_t bstride = a.batch_in_map ? (uint64_t)g.rope_batch_stride * 2
                                            : (uint64_t)g.t_max * g.rope_row_stride * 2;
    const uint64_t strides[2] = {(uint64_t)g.rope_row_stride * 2, bstride};
    const uint32_t box[3] = {32, BN, 1};   // one CTA's 32 rope dims: 64-byte rows
    if (!encode_tmap_bf16(&rope_map, g.rope, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  // Row maps for gathers: the cache as [rows, dims] with one-row boxes; a
  // batch row's rows start at b * (batch stride / row stride).
  CUtensorMap lat_rows_map = lat_map, rope_rows_map = rope_map;
  a.gather_tma = 0;
  a.lat_rows_per_batch = a.rope_rows_per_batch = 0;
  if (g.sel != nullptr && g.latent_batch_stride % g.latent_row_stride == 0 &&
      g.rope_batch_stride % g.rope_row_stride == 0) {
    a.lat_rows_per_batch = a.batch_in_map ? (int32_t)(g.latent_batch_stride / g.latent_row_stride) : 0;
    a.rope_rows_per_batch = a.batch_in_map ? (int32_t)(g.rope_batch_stride / g.rope_row_stride) : 0;
    const uint64_t lrows = (uint64_t)(a.batch_in_map ? g.batch - 1 : 0) * a.lat_rows_per_batch + g.t_max;
    const uint64_t rrows = (uint64_t)(a.batch_in_map ? g.batch - 1 : 0) * a.rope_rows_per_batch + g.t_max;
    const uint64_t ld[2] = {(uint64_t)g.rank, lrows}, rd[2] = {(uint64_t)g.rope_dim, rrows};
    const uint64_t ls[1] = {(uint64_t)g.latent_row_stride * 2}, rs[1] = {(uint64_t)g.rope_row_stride * 2};
    const uint32_t box[2] = {64, 1}, rbox[2] = {32, 1};
    if (lrows < (1ull << 31) && rrows < (1ull << 31) && encode_tmap_bf16(&lat_rows_map, g.latent, 2, ld, ls, box) &&
        encode_tmap_bf16(&rope_rows_map, g.rope, 2, rd, rs, rbox, CU_TENSOR_MAP_SWIZZLE_64B))
      a.gather_tma = 1;
  }
  const bool lockstep = a.width > 1;
  // (the prefetch distance only serves the dense path; gathers take the
  // instance with the extra gather warps)
  auto* const decode_kernel = a.gather_tma ? tc_decode_kernel<kPrefetchAheadRow, THREADS_GATHER, false>
                              : lockstep   ? tc_decode_kernel<kPrefetchAheadGroup, THREADS, true>
                                           : tc_decode_kernel<kPrefetchAheadRow, THREADS, false>;
  {
    const cudaError_t ea = set_max_dynamic_smem(decode_kernel, SMEM_BYTES);
    if (ea != cudaSuccess) return ea;
  }
  cudaError_t e = cudaSuccess;
  if (!a.plan_in_kernel) {
    e = launch_pdl(tc_plan_kernel, dim3(1), dim3(1024), 0, stream, a);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(decode_kernel, dim3(2 * nclusters), dim3(a.gather_tma ? THREADS_GATHER : THREADS), SMEM_BYTES, stream,
                 lat_map, rope_map, lat_rows_map, rope_rows_map, a);
  if (e != cudaSuccess) return e;
  if (tail == nullptr) {
    // batch 16 (128 registers, 4 CTAs per SM) while the grid fits one wave
    // at that occupancy, else 4
    auto* const combine = n_q <= kCombineWideRows ? tc_combine_kernel<16> : tc_combine_kernel<4>;
    e = launch_pdl(combine, dim3(n_q, RANK / CDIMS), dim3(HEADS), 0, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // Fused tail: combine + W_UV projection (bf16 context, n_q <= 64).
  CUtensorMap wmap;
  {
    const uint64_t dims[2] = {(uint64_t)tail->rank, (uint64_t)tail->heads * (tail->nope + tail->v_dim)};
    const uint64_t strides[1] = {(uint64_t)tail->rank * 2};
    const uint32_t box[2] = {64, 128};
    if (!encode_tmap_bf16(&wmap, tail->w, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  ProjectTail p;
  p.out = tail->out;
  p.out_row_stride = tail->out_row_stride;
  p.out_f32 = tail->out_dtype == MLA_DTYPE_F32 ? 1 : 0;
  p.npad = (n_q + 15) & ~15;
  p.v_dim = tail->v_dim;
  p.w_row0 = tail->nope;
  p.w_head_rows = tail->nope + tail->v_dim;
  {
    const cudaError_t ea = set_max_dynamic_smem(tc_combine_project_kernel, PROJ_SMEM_MAX);
    if (ea != cudaSuccess) return ea;
  }
  const size_t smem = 1024 + 8 * PROJ_BOX_BYTES + 8 * (size_t)p.npad * 128 + PROJ_MERGE_BYTES;
  e = launch_pdl(tc_combine_project_kernel, dim3(tail->heads), dim3(PROJ_THREADS), smem, stream, wmap, a, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
