// rows.cuh -- row pairing, index remapping, the remapping path and the
// group-wide radix select used by every selection stage.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dsa {

// Query rows of work group `g` of G rows each: dense rows G*g .. G*g+G-1;
// paged rows of one sequence b taken G at a time.  Returns the row count.
template <int G>
__device__ __forceinline__ int rows_of_group(const RowSpace& rs, int g, int* rows) {
  int first, count;
  if (!rs.paged) {
    first = G * g;
    count = min(G, rs.R - first);
  } else {
    const int per = (rs.next_n + G - 1) / G;
    const int b = g / per;
    const int i0 = G * (g % per);
    first = b * rs.next_n + i0;
    count = min(G, rs.next_n - i0);
  }
  for (int i = 0; i < G; ++i) rows[i] = first + i;
  return count;
}

__device__ __forceinline__ int row_seq(const RowSpace& rs, int row) { return rs.paged ? row / rs.next_n : -1; }

// Output index of logical key s of `row`: dense s; paged physical slot.  A
// block-table entry outside [0, num_pages) gives -1 and sets ST_RANGE.
__device__ __forceinline__ int32_t out_index(const RowSpace& rs, int row, int s) {
  if (!rs.paged) return s;
  const int b = row / rs.next_n;
  const int page = __ldg(&rs.block_table[(int64_t)b * rs.max_pages + (s >> 6)]);
  if (page < 0 || page >= rs.num_pages) {
    if (rs.status) atomicOr(rs.status, ST_RANGE);
    return -1;
  }
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

// Histogram of the current byte over keys matching (prefix, mask), one warp
// iteration at a time: the bucket most lanes share (that of the first live
// lane) is added once per warp, the others lane by lane.  Candidate keys
// crowd into few buckets, so this removes most shared-atomic conflicts.
__device__ __forceinline__ void hist_add(bool live, uint32_t bin, int lane, int* hist) {
  const unsigned lv = __ballot_sync(0xffffffffu, live);
  if (!lv) return;
  const int first = __ffs(lv) - 1;
  const uint32_t lead = __shfl_sync(0xffffffffu, bin, first);
  const unsigned same = __ballot_sync(0xffffffffu, live && bin == lead);
  if (lane == first) atomicAdd(&hist[lead], __popc(same));
  if (live && bin != lead) atomicAdd(&hist[bin], 1);
}

// Four 8-bit radix passes, most significant byte first, over n keys given by
// key_at(i): returns theta = the K-th largest key and r = how many keys equal
// to theta belong to the top K.  Called by all nthr threads (a multiple of 32)
// of a group whose first warp is full (tid 0..31); hist[256] and sdig[4] are
// shared memory.  When the bucket that holds the K-th key has at most
// `ccap` keys, they are compacted into cbuf (shared memory) and the remaining
// passes scan only them.
template <class KeyAt>
__device__ __forceinline__ void group_radix_select(KeyAt key_at, int n, int K, int* hist, int* sdig, int tid,
                                                   int nthr, int bar_id, uint32_t& theta, int& r,
                                                   uint32_t* cbuf = nullptr, int ccap = 0) {
  uint32_t prefix = 0, mask = 0;
  int rem = K;
  const int lane = tid & 31;
  int nc = -1;  // >= 0: live keys are compacted in cbuf[0, nc)
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int b = tid; b < 256; b += nthr) hist[b] = 0;
    group_sync(bar_id, nthr);
    const int m = nc >= 0 ? nc : n;
    for (int base = 0; base < m; base += nthr) {
      const int i = base + tid;
      uint32_t k = 0;
      bool live = false;
      if (i < m) {
        k = nc >= 0 ? cbuf[i] : key_at(i);
        live = (k & mask) == prefix;
      }
      hist_add(live, (k >> shift) & 0xFFu, lane, hist);
    }
    group_sync(bar_id, nthr);
    if (tid < 32) radix_pick_digit(hist, rem, sdig);
    group_sync(bar_id, nthr);
    const int digit = sdig[0];
    rem = sdig[1];
    const int in_bucket = sdig[2];
    prefix |= (uint32_t)digit << shift;
    mask |= 0xFFu << shift;
    group_sync(bar_id, nthr);  // sdig / hist reused below
    if (pass < 3 && nc < 0 && cbuf && in_bucket <= ccap && in_bucket < n / 2) {
      // compact the live bucket: later passes scan in_bucket keys, not n
      if (tid == 0) sdig[3] = 0;
      group_sync(bar_id, nthr);
      for (int base = 0; base < n; base += nthr) {
        const int i = base + tid;
        uint32_t k = 0;
        bool live = false;
        if (i < n) {
          k = key_at(i);
          live = (k & mask) == prefix;
        }
        const unsigned lv = __ballot_sync(0xffffffffu, live);
        int pos = 0;
        if (lane == 0 && lv) pos = atomicAdd(&sdig[3], __popc(lv));
        pos = __shfl_sync(0xffffffffu, pos, 0);
        if (live) cbuf[pos + __popc(lv & ((1u << lane) - 1u))] = k;
      }
      group_sync(bar_id, nthr);
      nc = in_bucket;
    }
  }
  theta = prefix;
  r = rem;
}

// Emission after the select: every key above theta and the first rr keys
// equal to theta go to o[] (the above ones to [0, K - rr), the equal ones to
// [K - rr, K)); slots are reserved once per warp.  All nthr threads call it
// with the same n; counters[0..1] are shared memory zeroed beforehand.
template <class KeyAt, class IdAt>
__device__ __forceinline__ void group_emit(KeyAt key_at, IdAt id_at, int n, uint32_t theta, int rr, int K,
                                           int32_t* o, int* counters, int tid, int nthr) {
  const int lane = tid & 31;
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  for (int base = 0; base < n; base += nthr) {
    const int i = base + tid;
    uint32_t k = 0;
    int32_t id = 0;
    if (i < n) {
      k = key_at(i);
      if (k >= theta) id = id_at(i);
    }
    const bool gt = (i < n) && k > theta;
    const bool eq = (i < n) && k == theta;
    const unsigned mg = __ballot_sync(0xffffffffu, gt);
    const unsigned me = __ballot_sync(0xffffffffu, eq);
    int bg = 0, be = 0;
    if (lane == 0) {
      if (mg) bg = atomicAdd(&counters[0], __popc(mg));
      if (me) be = atomicAdd(&counters[1], __popc(me));
    }
    bg = __shfl_sync(0xffffffffu, bg, 0);
    be = __shfl_sync(0xffffffffu, be, 0);
    if (gt) o[bg + __popc(mg & lt)] = id;
    if (eq) {
      const int e = be + __popc(me & lt);
      if (e < rr) o[K - rr + e] = id;
    }
  }
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

// ------------------------------------------- whole-CTA selection (256 threads)
// Descending scan of nb (<= 1024) bin counts by the NT threads of a CTA
// (1024 / NT bins each, thread t owning the t-th run from the top): the
// bin that holds the rem-th largest key goes to sc[2], the rank inside it
// to sc[3], its count to sc[4]; with `slots`, every bin's count is
// replaced by the number of keys in the bins above it (its first slot in a
// descending counting sort).  sc[32..63]: warp sums.  Ends with a CTA
// barrier.
template <int NT>
__device__ __forceinline__ void desc_scan_pick(int* hist, int nb, int rem, int* sc, bool slots) {
  constexpr int BPT = 1024 / NT;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c[BPT], s = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int b = nb - 1 - BPT * tid - j;
    c[j] = b >= 0 ? hist[b] : 0;
    s += c[j];
  }
  int incl = s;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) sc[32 + warp] = incl;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) incl += w < warp ? sc[32 + w] : 0;
  int e = incl - s;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int b = nb - 1 - BPT * tid - j;
    if (e < rem && rem <= e + c[j]) {
      sc[2] = b;
      sc[3] = rem - e;
      sc[4] = c[j];
    }
    if (slots && b >= 0) hist[b] = e;
    e += c[j];
  }
  __syncthreads();
}

}  // namespace dsa
