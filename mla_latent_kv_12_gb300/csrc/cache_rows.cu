// Row operations of the compressed cache ("mlx-bun 0.2.0 -> 0.4.0,
// package/src/model/glm52-cache.ts": Glm52Cache.specRoundRollback, filter
// and mergeRows).
//
// In the right-aligned layout every row of a state array [B, width, F] ends at
// the last column, so a rollback, a filter or a merge moves whole rows of
// tokens.  All three are one gather: destination column c of row i takes
// source column (c + shift[i]) mod src_width of source row src_row[i], or is
// zero below zero_below[i].  The kernel copies bytes (any dtype, bit-exact),
// grid (column blocks, rows), each CTA moving about 32 KB with 16-byte
// vectors when every address and stride allows, four loads in flight per
// thread before their stores.
//
// In the per-row window layout (kv_start, kv_len) nothing moves: a rollback
// only sets each row's length back to its accepted prefix
// (rollback_lengths_kernel).
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowUnroll = 4;

template <typename V>
__global__ void __launch_bounds__(kRowThreads) shift_rows_kernel(ShiftRowsParams p) {
  const int32_t row = blockIdx.y;
  const int32_t src_row = p.src_row ? p.src_row[row] : row;
  const int32_t zero_below = p.zero_below ? p.zero_below[row] : 0;
  // An empty source (width 0) can only feed rows that are all zero.
  if (src_row < 0 || src_row >= p.src_batch || zero_below < 0 || zero_below > p.dst_width ||
      (p.src_width == 0 && zero_below < p.dst_width)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicOr(p.status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
    return;
  }
  int64_t shift = (p.shift && p.src_width > 0) ? (int64_t)p.shift[row] % p.src_width : 0;
  if (shift < 0) shift += p.src_width;

  const int64_t c0 = (int64_t)blockIdx.x * p.cols_per_cta;
  const int64_t n_cols = min((int64_t)p.cols_per_cta, (int64_t)p.dst_width - c0);
  const int units = p.units_per_col;  // V-sized units in one column's features
  const int64_t total = n_cols * units;
  const char* src = static_cast<const char*>(p.src) + (int64_t)src_row * p.src_batch_bytes;
  char* dst = static_cast<char*>(p.dst) + (int64_t)row * p.dst_batch_bytes;

  for (int64_t base = threadIdx.x; base < total; base += (int64_t)kRowThreads * kRowUnroll) {
    V v[kRowUnroll];
    char* out[kRowUnroll];
#pragma unroll
    for (int k = 0; k < kRowUnroll; ++k) {
      const int64_t u = base + (int64_t)k * kRowThreads;
      out[k] = nullptr;
      if (u < total) {
        const int64_t col = c0 + u / units;
        const int64_t part = u % units;
        out[k] = dst + col * p.dst_col_bytes + part * (int64_t)sizeof(V);
        if (col < zero_below) {
          v[k] = V{};
        } else {
          int64_t sc = col + shift;
          if (sc >= p.src_width) sc %= p.src_width;
          v[k] = *reinterpret_cast<const V*>(src + sc * p.src_col_bytes + part * (int64_t)sizeof(V));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kRowUnroll; ++k)
      if (out[k]) *reinterpret_cast<V*>(out[k]) = v[k];
  }
}

__global__ void rollback_lengths_kernel(const int32_t* before, const int32_t* keep, const int32_t* kv_len,
                                        int32_t* kv_len_out, int32_t batch, int32_t* status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int32_t len = kv_len[b];
  const int64_t next = (int64_t)before[b] + keep[b];
  if (before[b] < 0 || keep[b] < 0 || next > len) {
    if (status) atomicOr(status, MLA_DEVICE_INDEX_OUT_OF_RANGE);
    kv_len_out[b] = len;
    return;
  }
  kv_len_out[b] = (int32_t)next;
}

}  // namespace

cudaError_t launch_shift_rows(const ShiftRowsParams& p_in, int vec_bytes, cudaStream_t stream) {
  ShiftRowsParams p = p_in;
  p.units_per_col = (int32_t)(p.row_bytes / vec_bytes);
  const int64_t per_cta = (32 * 1024) / (p.row_bytes > 0 ? p.row_bytes : 1);
  p.cols_per_cta = (int32_t)(per_cta < 1 ? 1 : (per_cta > 1024 ? 1024 : per_cta));
  const dim3 grid((unsigned)((p.dst_width + p.cols_per_cta - 1) / p.cols_per_cta), (unsigned)p.n_rows);
  switch (vec_bytes) {
    case 16: shift_rows_kernel<uint4><<<grid, kRowThreads, 0, stream>>>(p); break;
    case 8: shift_rows_kernel<uint2><<<grid, kRowThreads, 0, stream>>>(p); break;
    case 4: shift_rows_kernel<uint32_t><<<grid, kRowThreads, 0, stream>>>(p); break;
    default: shift_rows_kernel<uint16_t><<<grid, kRowThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_rollback_lengths(const int32_t* before, const int32_t* keep, const int32_t* kv_len,
                                    int32_t* kv_len_out, int32_t batch, int32_t* status, cudaStream_t stream) {
  rollback_lengths_kernel<<<(batch + 127) / 128, 128, 0, stream>>>(before, keep, kv_len, kv_len_out, batch,
                                                                    status);
  return cudaGetLastError();
}

}  // namespace mla
