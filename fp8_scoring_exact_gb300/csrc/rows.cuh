// rows.cuh -- row pairing, index remapping, the remapping path and the
// group-wide radix select used by every selection stage.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dsa {

// Query rows of work pair `pair`: dense rows 2p, 2p+1; paged rows of one
// sequence b taken two at a time.  Returns the number of rows (1 or 2).
__device__ __forceinline__ int pair_rows(const RowSpace& rs, int pair, int* rows) {
  if (!rs.paged) {
    rows[0] = 2 * pair;
    rows[1] = 2 * pair + 1;
    return (2 * pair + 1 < rs.R) ? 2 : 1;
  }
  const int per = (rs.next_n + 1) / 2;
  const int b = pair / per;
  const int i0 = 2 * (pair % per);
  rows[0] = b * rs.next_n + i0;
  rows[1] = rows[0] + 1;
  return (i0 + 1 < rs.next_n) ? 2 : 1;
}

__device__ __forceinline__ int row_seq(const RowSpace& rs, int row) { return rs.paged ? row / rs.next_n : -1; }

// Output index of logical key s of `row`: dense s; paged physical slot.
__device__ __forceinline__ int32_t out_index(const RowSpace& rs, int row, int s) {
  if (!rs.paged) return s;
  const int b = row / rs.next_n;
  const int page = __ldg(&rs.block_table[(int64_t)b * rs.max_pages + (s >> 6)]);
  return page * PAGE + (s & (PAGE - 1));
}

// Remapping path (L <= K): every valid index, then -1 padding.  All threads
// of the calling group stride over the K outputs.
__device__ __forceinline__ void write_all_valid(const RowSpace& rs, int row, int b, int e, int K, int32_t* out,
                                                int tid, int nthr) {
  int32_t* o = out + (int64_t)row * K;
  const int L = e - b;
  for (int i = tid; i < K; i += nthr) o[i] = (i < L) ? out_index(rs, row, b + i) : -1;
}

__device__ __forceinline__ void group_sync(int bar_id, int nthr) {
  if (bar_id == 0)
    __syncthreads();
  else
    named_bar_sync(bar_id, nthr);
}

// Four 8-bit radix passes, most significant byte first, over n keys given by
// key_at(i): returns theta = the K-th largest key and r = how many keys equal
// to theta belong to the top K.  Called by all nthr threads of a group whose
// first warp is full (tid 0..31); hist[256] and sdig[2] are shared memory.
template <class KeyAt>
__device__ __forceinline__ void group_radix_select(KeyAt key_at, int n, int K, int* hist, int* sdig, int tid,
                                                   int nthr, int bar_id, uint32_t& theta, int& r) {
  uint32_t prefix = 0, mask = 0;
  int rem = K;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = tid; b < 256; b += nthr) hist[b] = 0;
    group_sync(bar_id, nthr);
    for (int i = tid; i < n; i += nthr) {
      const uint32_t k = key_at(i);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFFu], 1);
    }
    group_sync(bar_id, nthr);
    if (tid < 32) radix_pick_digit(hist, rem, sdig);
    group_sync(bar_id, nthr);
    const int digit = sdig[0];
    rem = sdig[1];
    prefix |= (uint32_t)digit << shift;
    mask |= 0xFFu << shift;
    group_sync(bar_id, nthr);  // sdig / hist reused by the next pass
  }
  theta = prefix;
  r = rem;
}

// Sample grid of a key range [lo, hi): keys congruent to SAMPLE_OFFSET modulo
// the stride (SAMPLE_STRIDE, widened so that at most MAX_SAMPLES fall in the
// range).  Returns first position and count; stride in *S.
__device__ __forceinline__ void sample_grid(int lo, int hi, int* first, int* count, int* S) {
  const int L = hi - lo;
  const int widen = max(1, ceil_div(L, SAMPLE_STRIDE * MAX_SAMPLES));
  const int st = SAMPLE_STRIDE * widen;
  const int off = SAMPLE_OFFSET % st;
  int f = lo + ((off - lo) % st + st) % st;
  *first = f;
  *S = st;
  *count = (f < hi) ? ceil_div(hi - f, st) : 0;
}

// Descending rank of the threshold among m samples of an L-key row.
__device__ __forceinline__ int sample_rank(int m, int L, int target) {
  if (L <= 0) return 0;
  return (int)(((int64_t)m * target + L - 1) / L);
}

}  // namespace dsa
