// select_kernels.cu -- device-side plan, sampled thresholds (with the
// remapping path) and the standalone exact top-K over fp32 score rows.
//
// Method: "Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2",
// section 3.2 (sampled threshold aiming at ~2K candidates, compare-and-append,
// four 8-bit radix passes over order-preserving keys, certificate, exact
// repair) and section 3.4 (one shared-memory reservation per batch of items,
// vector loads); remapping path for rows with at most K keys from the
// contest write-up ("DSA TopK Indexer").
#include "common.cuh"
#include "kernels.h"
#include "rows.cuh"

namespace dsa {

// ===================================================================== plan ==
// One CTA of 1024 threads.  Main plan: validate every row's range, zero the
// per-call counters, form the row groups and the unit prefix sum.  Repair
// plan: one group per queued row.  Sample plan (dense): the same groups over
// each row's sample-grid range (rows with L <= K left out), written to
// rb / re in grid-index space.
constexpr int PLAN_THREADS = 1024;

__device__ __forceinline__ int block_inclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;  // inclusive prefix over warps
  }
  __syncthreads();
  const int res = x + (wid > 0 ? warp_sums[wid - 1] : 0);
  __syncthreads();
  return res;
}

__device__ __forceinline__ int group_units(int lo, int hi, int chunk) {
  if (hi <= lo) return 0;
  const int tiles = ceil_div(hi, TILE) - lo / TILE;
  return ceil_div(tiles, chunk);
}

// A row's range for the main plan (validated input range, or the paged
// row's causal range; an invalid one becomes empty and sets *bad) or for the
// sample plan (the grid keys SAMPLE_OFFSET + j * S inside the row's main
// range: j in [j0, j1)).
__device__ __forceinline__ void plan_row_range(const PlanParams& p, int row, int& b, int& e, bool& bad) {
  const RowSpace& rs = p.rs;
  b = e = 0;
  if (p.plan == PLAN_SAMPLE) {
    const int S = p.sample_stride;
    const int rb = p.row_begin_in[row], re = p.row_end_in[row];
    b = rb > SAMPLE_OFFSET ? ceil_div(rb - SAMPLE_OFFSET, S) : 0;
    e = max(b, re > SAMPLE_OFFSET ? ceil_div(re - SAMPLE_OFFSET, S) : 0);
  } else if (!rs.paged) {
    b = p.row_begin_in[row];
    e = p.row_end_in[row];
    if (b < 0 || e > rs.N || b > e) {
      bad = true;
      b = e = 0;
    }
  } else {
    const int sq = row / rs.next_n, i = row % rs.next_n;
    const int sl = rs.seq_lens[sq];
    if (sl < 0 || sl > rs.max_pages * PAGE)
      bad = true;
    else
      e = max(0, sl - rs.next_n + i + 1);
  }
}

// Groups of a plan and their work-unit prefix (unit_start), by every thread
// of the calling CTA (any multiple of 32 threads); G groups.  warp_sums: 32
// ints and s_carry: one int of shared memory.  The main and sample plans
// form their rows' ranges here (written to rb / re; *bad: an invalid main
// range).  Failed-row entries are read through L2: the repair plan may run in
// the CTA that finishes the candidate selection, whose other CTAs queued
// them.
__device__ void plan_groups(const PlanParams& p, int G, int* warp_sums, int* s_carry, bool* bad = nullptr) {
  const RowSpace& rs = p.rs;
  const int tid = threadIdx.x;
  if (tid == 0) *s_carry = 0;
  __syncthreads();
  for (int base = 0; base < G; base += (int)blockDim.x) {
    const int g = base + tid;
    int units = 0;
    if (g < G) {
      Group grp;
      grp.nrows = 0;
      grp.lo = 0x7fffffff;
      grp.hi = 0;
      for (int i = 0; i < GROUP_ROWS; ++i) grp.row[i] = grp.slot[i] = 0;
      if (p.plan != PLAN_REPAIR) {
        int rows[GROUP_ROWS];
        const int nr = rows_of_group<GROUP_ROWS>(rs, g, rows);
        grp.seq = rs.paged ? rows[0] / rs.next_n : -1;
        for (int i = 0; i < nr; ++i) {
          int b, e;
          bool rbad = false;
          plan_row_range(p, rows[i], b, e, rbad);
          if (rbad && bad) *bad = true;
          p.rb[rows[i]] = b;
          p.re[rows[i]] = e;
          // the sample plan leaves out the rows the main plan calls trivial
          const int len = p.plan == PLAN_SAMPLE ? p.row_end_in[rows[i]] - p.row_begin_in[rows[i]] : e - b;
          if (len > p.trivial_len && e > b) {
            grp.row[grp.nrows] = rows[i];
            grp.slot[grp.nrows] = rows[i];
            ++grp.nrows;
            grp.lo = min(grp.lo, b);
            grp.hi = max(grp.hi, e);
          }
        }
      } else if (rs.paged) {
        const int row = __ldcg(&p.failed_rows[g]);
        grp.nrows = 1;
        grp.row[0] = row;
        grp.slot[0] = g;
        grp.seq = row / rs.next_n;
        grp.lo = p.rb[row];
        grp.hi = p.re[row];
      } else {
        // failed-list entries 4g .. 4g + 3; slot = the entry (its score row)
        const int nf = __ldcg(&p.stats->fail_count);
        grp.seq = -1;
        for (int i = 0; i < GROUP_ROWS && GROUP_ROWS * g + i < nf; ++i) {
          const int f = GROUP_ROWS * g + i, row = __ldcg(&p.failed_rows[f]);
          grp.row[grp.nrows] = row;
          grp.slot[grp.nrows] = f;
          ++grp.nrows;
          grp.lo = min(grp.lo, p.rb[row]);
          grp.hi = max(grp.hi, p.re[row]);
        }
      }
      if (grp.nrows == 0) grp.lo = grp.hi = 0;
      units = group_units(grp.lo, grp.hi, p.chunk_tiles);
      p.groups[g] = grp;
    }
    const int incl = block_inclusive_scan(units, warp_sums);
    const int carry = *s_carry;
    if (g < G) p.unit_start[g + 1] = carry + incl;
    __syncthreads();
    if (tid == (int)blockDim.x - 1) *s_carry = carry + incl;
    __syncthreads();
  }
  if (tid == 0) {
    p.unit_start[0] = 0;
    p.stats->next_unit[p.plan] = 0;
    if (p.plan == PLAN_MAIN) {
      p.stats->n_groups = G;
      p.stats->total_units = *s_carry;
    } else if (p.plan == PLAN_REPAIR) {
      p.stats->r_groups = G;
      p.stats->r_units = *s_carry;
    } else {
      p.stats->s_groups = G;
      p.stats->s_units = *s_carry;
    }
  }
}

// Groups of the repair plan: dense rows all read one key array, so four
// failed rows share a group (scored over the union of their ranges); paged
// rows, one per group.
__device__ __forceinline__ int repair_groups(const PlanParams& p) {
  const int nf = __ldcg(&p.stats->fail_count);
  return p.rs.paged ? nf : ceil_div(nf, GROUP_ROWS);
}

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(const PlanParams p) {
  pdl_enter();
  __shared__ int warp_sums[32];
  __shared__ int s_carry;
  const RowSpace& rs = p.rs;
  // main and sample plans: one thread per group forms its rows' ranges and
  // the group (no pass over the rows before); the main plan's status block
  // is written whole at the end (the call's other kernels start after)
  const int G = p.plan == PLAN_REPAIR ? repair_groups(p) : n_groups(rs);
  bool bad = false;
  plan_groups(p, G, warp_sums, &s_carry, &bad);
  if (p.plan == PLAN_MAIN) {
    if (p.pair_cnt)
      for (int i = threadIdx.x; i < p.n_pairs; i += blockDim.x) p.pair_cnt[i] = 0;
    const bool any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
      Stats z = {};
      z.wait_ns = p.wait_ns;
      z.status = any_bad ? ST_RANGE : 0;
      z.n_groups = G;
      z.total_units = s_carry;
      *p.stats = z;
    }
  }
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t s) {
  return launch_pdl(plan_kernel, dim3(1), dim3(PLAN_THREADS), 0, s, p);
}

// The rank-th largest (1 <= rank <= m) of a warp's m keys, key[q] of lane l
// being key q * 32 + l (positions >= m ignored): radix passes in a per-warp
// histogram (hist: 256 ints, pick: 4 ints of shared memory), with no CTA
// barrier.  Every key agrees above the highest bit where the smallest and
// largest differ, so the first digit is the 8 bits just below and at that
// bit (a row's samples spread over its bins instead of crowding into one or
// two of a byte-aligned digit, whose shared-memory atomics then serialize);
// the later digits are the next 8 bits down, and a digit whose bucket holds
// a single key ends the search.
template <int KPL>
__device__ __forceinline__ uint32_t warp_select_rank(const uint32_t (&key)[KPL], int m, int rank, int* hist,
                                                     int* pick) {
  const int lane = threadIdx.x & 31;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < KPL; ++q) {
    if (q * 32 + lane < m) {
      kmin = min(kmin, key[q]);
      kmax = max(kmax, key[q]);
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  const uint32_t diff = kmin ^ kmax;
  if (diff == 0u) return kmin;  // every key the same
  int top = 31 - __clz(diff);   // the digit's highest bit
  uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
  uint32_t prefix = kmin & mask;
  int rem = rank;
#pragma unroll 1
  while (true) {
    const int lo = max(0, top - 7);
    const uint32_t dmask = (2u << (top - lo)) - 1u;  // the digit's bits, at bit 0
#pragma unroll
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
      const int i = q * 32 + lane;
      if (i < m && (key[q] & mask) == prefix) atomicAdd(&hist[(key[q] >> lo) & dmask], 1);
    }
    __syncwarp();
    radix_pick_digit(hist, rem, pick);
    __syncwarp();
    prefix |= (uint32_t)pick[0] << lo;
    mask |= dmask << lo;
    rem = pick[1];
    const int cnt = pick[2];
    __syncwarp();
    if (cnt == 1) {
      // the answer is the only key in its bucket: read it whole
      uint32_t found = 0u;
      bool have = false;
#pragma unroll
      for (int q = 0; q < KPL; ++q) {
        const int i = q * 32 + lane;
        if (i < m && (key[q] & mask) == prefix) {
          found = key[q];
          have = true;
        }
      }
      const unsigned b = __ballot_sync(0xffffffffu, have);
      return __shfl_sync(0xffffffffu, found, __ffs(b) - 1);
    }
    if (lo == 0) return prefix;
    top = lo - 1;
  }
}

// ================================================================== sample ==
// One CTA (4 warps) per query-row pair: rows with at most K keys take the
// remapping path; the other rows score the keys on a 1-in-200 grid with
// tcgen05 (keys gathered into a swizzled shared tile by the threads) and take
// as threshold the sample of descending rank ceil(m * target / L), one warp
// per row once the scores are out of tensor memory (which is released first,
// so the next CTA on the SM can start its MMA).
// Split mode (paged rows, whose grids span several tiles): one CTA per (pair,
// 128-key sample tile), so the tiles' gathers run side by side; each writes
// its fp32 sample scores (and the tile-0 CTA the rows' sample ranges and
// the trivial rows), and sample_tau_kernel selects the thresholds.
constexpr int SAMPLE_THREADS = 128;
constexpr uint32_t SM_OFF_Q = 0;
constexpr uint32_t SM_OFF_K = SM_OFF_Q + SAMPLE_ROWS * H * D;       // 16384
constexpr uint32_t SM_OFF_SAMP = SM_OFF_K + TILE * D;               // 32768
constexpr uint32_t SM_OFF_W = SM_OFF_SAMP + SAMPLE_ROWS * MAX_SAMPLES * 4;  // 40960
constexpr uint32_t SM_OFF_SC = SM_OFF_W + SAMPLE_ROWS * H * 4;
constexpr uint32_t SM_OFF_HIST = SM_OFF_SC + TILE * 4;                   // a 256-bin histogram per warp
constexpr uint32_t SM_OFF_PICK = SM_OFF_HIST + (SAMPLE_THREADS / 32) * 256 * 4;  // and its pick words
constexpr uint32_t SM_OFF_MISC = SM_OFF_PICK + (SAMPLE_THREADS / 32) * 4 * 4;
// 52 KB per CTA: 4 CTAs (4 x 128 TMEM columns, all 512) fit on an SM, and
// the launch bounds hold the registers to 128 so that 4 CTAs fit there too
constexpr uint32_t SAMPLE_SMEM = 52 * 1024;
static_assert(SM_OFF_MISC + 64 + 1024 <= SAMPLE_SMEM, "sample smem");

__global__ void __launch_bounds__(SAMPLE_THREADS, 4) sample_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                const SampleParams p) {
  pdl_enter();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* samp = (uint32_t*)(smem + SM_OFF_SAMP);
  float* wsm = (float*)(smem + SM_OFF_W);
  float* scs = (float*)(smem + SM_OFF_SC);
  int* misc = (int*)(smem + SM_OFF_MISC);  // [0] tmem base, [5] abort, [6] wait result
  const uint32_t bar = sbase + SM_OFF_MISC + 32;
  const RowSpace& rs = p.rs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = p.K;

  int rows[SAMPLE_ROWS];
  const int nr = rows_of_group<SAMPLE_ROWS>(rs, blockIdx.x, rows);
  const bool split = p.split != 0;
  const int tile0 = split ? (int)blockIdx.y : 0;  // split: this CTA's sample tile
  int act[2], nact = 0, lo = 0x7fffffff, hi = 0, ntriv = 0;
  for (int i = 0; i < nr; ++i) {
    const int b = p.rb[rows[i]], e = p.re[rows[i]];
    if (e - b <= K) {
      if (tile0 == 0) write_all_valid(rs, rows[i], b, e, K, p.out, tid, SAMPLE_THREADS);
      ++ntriv;
    } else {
      act[nact++] = rows[i];
      lo = min(lo, b);
      hi = max(hi, e);
    }
  }
  if (tid == 0 && ntriv && tile0 == 0) atomicAdd(&p.stats->trivial, ntriv);
  if (nact == 0) return;
  int first, m_u, S;
  sample_grid(lo, hi, &first, &m_u, &S);
  const int target = (int)(((int64_t)p.target16 * K) / 16);
  if (split) {
    if (m_u == 0) {  // no grid key in the pair's ranges: every key passes
      if (tile0 == 0 && tid < nact) p.tau[act[tid]] = 0u;
      return;
    }
    // each active row's samples: pair-grid indices [j0, j1) inside its range
    if (tile0 == 0 && tid < nact) {
      const int row = act[tid];
      const int b = p.rb[row], e = p.re[row];
      p.srb[row] = max(0, ceil_div(b - first, S));
      p.sre[row] = min(m_u, max(0, ceil_div(e - first, S)));
    }
    if (tile0 * TILE >= m_u) return;
  } else if (m_u == 0) {
    if (tid < nact) p.tau[act[tid]] = 0u;
    return;
  }

  if (warp == 0) {
    tmem_alloc(sbase + SM_OFF_MISC, TILE);
    tmem_relinquish();
  }
  if (tid == 0) {
    misc[5] = 0;
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < nact * H; i += SAMPLE_THREADS) {
    const int a = i / H, j = i % H;
    wsm[i] = p.w[(int64_t)act[a] * H + j] * p.q_scale[act[a]];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)misc[0];
  volatile int* abort_flag = (volatile int*)&misc[5];
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, nact * H * D);
    for (int a = 0; a < nact; ++a) tma_load_2d(sbase + SM_OFF_Q + a * H * D, &tm_q, 0, act[a] * H, bar);
  }
  // tiles [tt_begin, tt_end) of the pair's grid: all of them, or this
  // CTA's one in split mode
  const int tt_begin = tile0;
  const int tt_end = split ? tile0 + 1 : ceil_div(m_u, TILE);
  // one sample key per thread: its 128 bytes and scale; the next tile's are
  // loaded while the current tile is multiplied and reduced
  uint4 chunk[8];
  float ks = 0.f;
  auto fetch = [&](int tt) {
    const int j = tt * TILE + tid;
    const int s = first + j * S;
    int64_t slot = s;
    bool in_cache = j < m_u;
    if (in_cache && rs.paged) {
      const int page = __ldg(&rs.block_table[(int64_t)(act[0] / rs.next_n) * rs.max_pages + (s >> 6)]);
      in_cache = page >= 0 && page < rs.num_pages;  // a bad page id reads as a zero key
      slot = (int64_t)page * PAGE + (s & (PAGE - 1));
    }
    ks = 0.f;
    if (in_cache) {
      const uint4* src = (const uint4*)(p.k + slot * D);
#pragma unroll
      for (int c = 0; c < 8; ++c) chunk[c] = __ldg(&src[c]);
      ks = __ldg(&p.k_scale[slot]);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) chunk[c] = make_uint4(0, 0, 0, 0);
    }
  };
  fetch(tt_begin);
  // thread 0 waits (bounded) and the CTA follows its result; pend = the
  // parity of the phase whose copy or MMA is outstanding (at most one)
  uint32_t pend = 0;
  if (tid == 0) misc[6] = mbar_wait(bar, 0, abort_flag, p.stats) ? 1 : 0;
  __syncwarp();
  __syncthreads();
  bool ok = misc[6] != 0;
  const uint32_t idesc = idesc_e4m3_f32(TILE, H * nact);
  for (int tt = tt_begin; tt < tt_end && ok; ++tt) {
    const int j = tt * TILE + tid;
    const bool vj = j < m_u;
    // the fetched key into the 128-byte-swizzled tile
    uint8_t* krow = smem + SM_OFF_K + tid * D;
#pragma unroll
    for (int c = 0; c < 8; ++c) *(uint4*)(krow + ((c ^ (tid & 7)) << 4)) = chunk[c];
    scs[tid] = ks;
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 32; ++k)
        mma_e4m3(tmem, sw128_kmajor_desc(sbase + SM_OFF_K + 32 * k), sw128_kmajor_desc(sbase + SM_OFF_Q + 32 * k),
                 idesc, k > 0);
      mma_commit(bar);
    }
    if (tt + 1 < tt_end) fetch(tt + 1);
    // phase 0 was the q load; this CTA's i-th MMA commit completes phase i + 1
    pend = (tt - tt_begin + 1) & 1;
    if (tid == 0) misc[6] = mbar_wait(bar, pend, abort_flag, p.stats) ? 1 : 0;
    __syncwarp();
    __syncthreads();
    ok = misc[6] != 0;
    if (!ok) break;
    tc_fence_after();
    for (int a = 0; a < nact; ++a) {
      const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + a * H;
      // four interleaved sums (a 64-long chain of dependent FMAs would set
      // the epilogue's latency), 32 heads per TMEM load
      float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < H; hh += 32) {
        uint32_t v[32];
        tmem_ld32(ta + hh, v);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h)
          a4[h & 3] = fmaf(wsm[a * H + hh + h], fmaxf(__uint_as_float(v[h]), 0.f), a4[h & 3]);
      }
      const float acc = (a4[0] + a4[1]) + (a4[2] + a4[3]);
      if (vj) {
        if (split)
          p.sscores[(int64_t)act[a] * p.sld + j] = acc * scs[tid];
        else
          samp[a * MAX_SAMPLES + j] = ordered_key(acc * scs[tid]);
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  // a wait gave up: the copy or MMA it waited for lands before the shared
  // memory and TMEM are released
  if (!ok && tid == 0) mbar_drain(bar, pend);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TILE);
  }
  if (split) {
    // the pair's last tile CTA to finish selects its thresholds from the
    // sample scores the pair's CTAs wrote (each thread fenced its own)
    __threadfence();
    __syncthreads();
    if (tid == 0) misc[7] = atomicAdd(&p.pair_cnt[blockIdx.x], 1) == ceil_div(m_u, TILE) - 1;
    __syncthreads();
    if (!misc[7]) return;
    __threadfence();
  }
  // threshold of active row a (by warp a) from the samples inside its own
  // range (a larger m than the selection holds would leave the threshold at
  // 0, every key a candidate, and the certificate would send the row to
  // repair)
  if (warp < nact) {
    const int row = act[warp];
    uint32_t tau = 0u;
    if (ok) {
      const int b = p.rb[row], e = p.re[row];
      const int j0 = max(0, ceil_div(b - first, S));
      const int j1 = min(m_u, ceil_div(e - first, S));
      const int m = max(0, j1 - j0);
      const int rank = sample_rank(m, e - b, target);
      int* whist = (int*)(smem + SM_OFF_HIST) + warp * 256;
      int* wpick = (int*)(smem + SM_OFF_PICK) + warp * 4;
      if (split && m > 0 && m <= MAX_SAMPLES && rank >= 1 && rank <= m) {
        // the pair's tiles: sample scores in global memory, up to 8 tiles
        uint32_t key[MAX_SAMPLES / 32];
        const float* sr = p.sscores + (int64_t)row * p.sld + j0;
#pragma unroll
        for (int q = 0; q < MAX_SAMPLES / 32; ++q) {
          const int i = q * 32 + lane;
          key[q] = i < m ? ordered_key(__ldcg(&sr[i])) : 0u;
        }
        tau = warp_select_rank<MAX_SAMPLES / 32>(key, m, rank, whist, wpick);
      } else if (!split && m > 0 && m <= 4 * 32 && rank >= 1 && rank <= m) {
        // one tile: the sample keys in shared memory
        uint32_t key[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = q * 32 + lane;
          key[q] = i < m ? samp[warp * MAX_SAMPLES + j0 + i] : 0u;
        }
        tau = warp_select_rank<4>(key, m, rank, whist, wpick);
      }
      if (tau != 0u && p.tau_bias != 0) {
        const int64_t t = (int64_t)tau + p.tau_bias;
        tau = (uint32_t)(t < 0 ? 0 : (t > 0xffffffffll ? 0xffffffffll : t));
      }
    }
    if (lane == 0) p.tau[row] = tau;
  }
}

cudaError_t launch_sample(const CUtensorMap& tm_q, const SampleParams& p, int n_pairs_, cudaStream_t s) {
  const dim3 grid(n_pairs_, p.split ? ceil_div(MAX_SAMPLES, TILE) : 1);
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_attr_once(sample_kernel, SAMPLE_SMEM, attr_set);
  if (e != cudaSuccess) return e;
  if (n_pairs_ <= 0) return cudaSuccess;
  return launch_pdl(sample_kernel, grid, dim3(SAMPLE_THREADS), SAMPLE_SMEM, s, tm_q, p);
}

// ============================================================ sample (dense) ==
// Dense rows sample one global grid of keys (SAMPLE_OFFSET + j * stride, the
// same keys for every row; a row uses the grid keys inside its range), so
// the grid is gathered once into a contiguous key set and scored by the
// persistent scorer like any key set.  This kernel gathers it, builds the
// sample plan and writes the rows with L <= K (their output is every valid
// index).
constexpr int PREP_THREADS = 256;

__global__ void __launch_bounds__(PREP_THREADS) sample_prep_kernel(const SamplePrepParams p) {
  pdl_enter();
  // the first CTA builds the sample plan (the groups over the rows' grid
  // ranges) while the others gather: one launch fewer
  if (blockIdx.x == 0) {
    __shared__ int warp_sums[32];
    __shared__ int s_carry;
    plan_groups(p.plan, n_groups(p.rs), warp_sums, &s_carry);
  }
  const int gt = blockIdx.x * PREP_THREADS + threadIdx.x;
  const int nthreads = gridDim.x * PREP_THREADS;
  // 8 threads per grid key: 16 bytes each
  for (int i = gt; i < p.n_samples * 8; i += nthreads) {
    const int j = i >> 3, c = i & 7;
    const int64_t src = (int64_t)SAMPLE_OFFSET + (int64_t)j * p.stride;
    reinterpret_cast<uint4*>(p.sk + (int64_t)j * D)[c] = __ldg(reinterpret_cast<const uint4*>(p.k + src * D) + c);
    if (c == 0) p.sks[j] = __ldg(&p.k_scale[src]);
  }
  // trivial rows: one warp per row
  const int warp = gt >> 5, nwarps = nthreads >> 5, lane = threadIdx.x & 31;
  int ntriv = 0;
  for (int row = warp; row < p.rs.R; row += nwarps) {
    const int b = p.rb[row], e = p.re[row];
    if (e - b > p.K) continue;
    int32_t* o = p.out + (int64_t)row * p.K;
    for (int i = lane; i < p.K; i += 32) o[i] = i < e - b ? b + i : -1;
    ++ntriv;
  }
  if (lane == 0 && ntriv) atomicAdd(&p.stats->trivial, ntriv);
}

// One warp per row with L > K: the threshold is the sample of descending rank
// ceil(m * target / L) among the row's m grid-key scores (radix select in a
// per-warp histogram), plus the test bias; 0 (every key passes) when the
// rank falls outside the sample.
constexpr int TAU_THREADS = 256;
// two builds: up to 672 samples per row (rows of up to ~134K keys: 64
// registers, 4 blocks per SM, so 4096 rows take one wave) and up to
// MAX_SAMPLES (127 registers, 2 blocks per SM)
constexpr int TAU_KPL_SHORT = 21;
template <int KPL>
__global__ void __launch_bounds__(TAU_THREADS, KPL <= TAU_KPL_SHORT ? 4 : 2) sample_tau_kernel(const SampleTauParams p) {
  pdl_enter();
  __shared__ int hist_all[TAU_THREADS / 32][256];
  __shared__ int pick_all[TAU_THREADS / 32][4];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int* hist = hist_all[wid];
  int* pick = pick_all[wid];
  const int warp = blockIdx.x * (TAU_THREADS / 32) + wid, nwarps = gridDim.x * (TAU_THREADS / 32);
  const int target = (int)(((int64_t)p.target16 * p.K) / 16);
  int ntriv = 0;
  for (int row = warp; row < p.rs.R; row += nwarps) {
    const int b = p.rb[row], L = p.re[row] - b;
    if (L <= p.K) {
      if (p.from_matrix) {  // trivial path: every valid index, then -1
        int32_t* o = p.out + (int64_t)row * p.K;
        for (int i = lane; i < p.K; i += 32) o[i] = i < L ? b + i : -1;
        ++ntriv;
      }
      continue;
    }
    int j0, m, stride = 1;
    const float* sr;
    if (p.from_matrix) {  // the row's own grid keys in the score matrix
      int first;
      sample_grid(b, b + L, &first, &m, &stride);
      j0 = 0;
      sr = p.sscores + (int64_t)row * p.sld + first;
    } else {
      j0 = p.srb[row];
      m = p.sre[row] - j0;
      sr = p.sscores + (int64_t)row * p.sld + j0;
    }
    m = min(m, MAX_SAMPLES);
    const int rank = sample_rank(m, L, target);
    uint32_t tau = 0u;
    // (more samples than this build holds cannot occur: the launch picks
    // the build from the longest row; a threshold of 0 would only send the
    // row to repair)
    if (m > 0 && m <= 32 * KPL && rank >= 1 && rank <= m) {
      uint32_t key[KPL];
#pragma unroll
      for (int q = 0; q < KPL; ++q) {
        const int i = q * 32 + lane;
        key[q] = i < m ? ordered_key(__ldcg(&sr[(int64_t)i * stride])) : 0u;
      }
      const uint32_t prefix = warp_select_rank<KPL>(key, m, rank, hist, pick);
      tau = prefix;
      if (p.tau_bias != 0) {
        const int64_t t = (int64_t)tau + p.tau_bias;
        tau = (uint32_t)(t < 0 ? 0 : (t > 0xffffffffll ? 0xffffffffll : t));
      }
    }
    if (lane == 0) p.tau[row] = tau;
  }
  if (lane == 0 && ntriv) atomicAdd(&p.stats->trivial, ntriv);
}

cudaError_t launch_sample_prep(const SamplePrepParams& p, cudaStream_t s) {
  return launch_pdl(sample_prep_kernel, dim3(64), dim3(PREP_THREADS), 0, s, p);
}
cudaError_t launch_sample_tau(const SampleTauParams& p, cudaStream_t s) {
  const int blocks = max(1, min(1024, ceil_div(p.rs.R, TAU_THREADS / 32)));
  // a row of L keys has at most L / SAMPLE_STRIDE + 1 grid samples (the
  // stride widens for longer rows, up to MAX_SAMPLES)
  const int64_t max_m = std::min<int64_t>(MAX_SAMPLES, (int64_t)p.rs.N / SAMPLE_STRIDE + 2);
  if (max_m <= 32 * TAU_KPL_SHORT)
    return launch_pdl(sample_tau_kernel<TAU_KPL_SHORT>, dim3(blocks), dim3(TAU_THREADS), 0, s, p);
  return launch_pdl(sample_tau_kernel<MAX_SAMPLES / 32>, dim3(blocks), dim3(TAU_THREADS), 0, s, p);
}

// ================================================================== select ==
// Standalone exact top-K of fp32 score rows, one CTA per row at a time:
// sampled threshold -> filter into shared memory (float4 loads, one shared
// reservation per warp) -> radix select on the candidates.  The certificate
// holds for any threshold, so a failed filter (fewer than K or more than
// SELECT_CAP candidates) retries with a relaxed threshold; when no threshold
// separates the top K (massive ties) the radix select runs over the row.
constexpr uint32_t SEL_OFF_KEY = 0;
constexpr uint32_t SEL_OFF_IDX = SEL_OFF_KEY + SELECT_CAP * 4;
constexpr uint32_t SEL_OFF_SAMP = SEL_OFF_IDX + SELECT_CAP * 4;
constexpr uint32_t SEL_OFF_CMP = SEL_OFF_SAMP + MAX_SAMPLES * 4;
constexpr int SEL_CMP_CAP = 2048;
constexpr uint32_t SEL_OFF_HIST = SEL_OFF_CMP + SEL_CMP_CAP * 4;
constexpr uint32_t SEL_OFF_MISC = SEL_OFF_HIST + 256 * 4;
constexpr uint32_t SELECT_SMEM = SEL_OFF_MISC + 64;

__global__ void __launch_bounds__(SELECT_THREADS) select_kernel(const SelectParams p) {
  pdl_enter();
  extern __shared__ uint8_t smem[];
  uint32_t* ckey = (uint32_t*)(smem + SEL_OFF_KEY);
  int32_t* cidx = (int32_t*)(smem + SEL_OFF_IDX);
  uint32_t* samp = (uint32_t*)(smem + SEL_OFF_SAMP);
  uint32_t* cmp = (uint32_t*)(smem + SEL_OFF_CMP);
  int* hist = (int*)(smem + SEL_OFF_HIST);
  int* misc = (int*)(smem + SEL_OFF_MISC);  // [0..3] digit block, [4] count, [5..6] emit counters
  const RowSpace& rs = p.rs;
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.K;
  const int count = rs.R;
  const int target = (int)(((int64_t)p.target16 * K) / 16);

  for (int f = blockIdx.x; f < count; f += gridDim.x) {
    const int row = f;
    const int b = p.rb[row], e = p.re[row];
    const int L = e - b;
    int32_t* o = p.out + (int64_t)row * K;
    if (tid == 0) {
      misc[4] = 0;
      misc[5] = 0;
      misc[6] = 0;
    }
    if (L <= K) {
      write_all_valid(rs, row, b, e, K, p.out, tid, SELECT_THREADS);
      continue;
    }
    const float* srow = p.scores + (int64_t)row * p.ld;

    // sampled threshold: the sample of descending rank `rk` (0 = every key)
    int first, m, S;
    sample_grid(b, e, &first, &m, &S);
    for (int j = tid; j < m; j += SELECT_THREADS) samp[j] = ordered_key(srow[first + j * S]);
    __syncthreads();
    auto tau_at_rank = [&](int rk) -> uint32_t {
      if (m <= 0 || rk < 1 || rk > m) return 0u;
      uint32_t t;
      int rr;
      group_radix_select([&](int i) { return samp[i]; }, m, rk, hist, misc, tid, SELECT_THREADS, 0, t, rr);
      return t;
    };

    // compare-and-append: 4 items per thread per step, one shared atomic per warp
    const int a0 = min(e, (b + 3) & ~3);   // first 16-byte aligned index
    const int a1 = max(a0, e & ~3);        // end of the aligned body
    const int nh = (a0 - b) + (e - a1);    // scalar head + tail (<= 6)
    const int nvec = (a1 - a0) >> 2;
    const float4* v4 = (const float4*)(srow + a0);
    const int rounds = ceil_div(nvec, SELECT_THREADS);
    // every key of [b, e) once: f(key, index, valid) on all lanes of a warp
    auto visit_row = [&](auto&& f) {
      if (tid < 32) {
        const bool v = lane < nh;
        const int i = !v ? b : (lane < (a0 - b) ? b + lane : a1 + (lane - (a0 - b)));
        f(v ? ordered_key(srow[i]) : 0u, i, v);
      }
      for (int rd = 0; rd < rounds; ++rd) {
        const int vi = rd * SELECT_THREADS + tid;
        const bool v = vi < nvec;
        const float4 x = v ? __ldcs(&v4[vi]) : make_float4(0.f, 0.f, 0.f, 0.f);
        f(ordered_key(x.x), a0 + vi * 4 + 0, v);
        f(ordered_key(x.y), a0 + vi * 4 + 1, v);
        f(ordered_key(x.z), a0 + vi * 4 + 2, v);
        f(ordered_key(x.w), a0 + vi * 4 + 3, v);
      }
    };
    uint32_t lt;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
    auto filter = [&](uint32_t tau) -> int {
      if (tid == 0) misc[4] = 0;
      __syncthreads();
      // the unaligned head and tail (at most 6 keys): warp 0
      if (tid < 32) {
        const bool v = lane < nh;
        const int i = !v ? b : (lane < (a0 - b) ? b + lane : a1 + (lane - (a0 - b)));
        const uint32_t k = v ? ordered_key(srow[i]) : 0u;
        const bool pass = v && k >= tau;
        const unsigned mp = __ballot_sync(0xffffffffu, pass);
        if (mp) {
          int base = 0;
          if (lane == 0) base = atomicAdd(&misc[4], __popc(mp));
          base = __shfl_sync(0xffffffffu, base, 0) + __popc(mp & lt);
          if (pass && base < SELECT_CAP) {
            ckey[base] = k;
            cidx[base] = i;
          }
        }
      }
      // the aligned body: SEL_UNROLL float4 loads in flight per thread, its
      // passing keys counted, a warp scan, one reservation per warp and
      // round (a ballot and a shared atomic per key slot serialised the
      // warps on one counter)
      for (int base4 = 0; base4 < nvec; base4 += SELECT_THREADS * SEL_UNROLL) {
        uint32_t kk[4 * SEL_UNROLL];
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) {
          const int vi = base4 + u * SELECT_THREADS + tid;
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (vi < nvec) x = __ldcs(&v4[vi]);
          kk[4 * u + 0] = vi < nvec ? ordered_key(x.x) : 0u;
          kk[4 * u + 1] = vi < nvec ? ordered_key(x.y) : 0u;
          kk[4 * u + 2] = vi < nvec ? ordered_key(x.z) : 0u;
          kk[4 * u + 3] = vi < nvec ? ordered_key(x.w) : 0u;
        }
        // key 0 never passes a threshold above 0, and tau 0 admits every
        // valid key: padding counts only when tau is 0, so test vi again
        int c = 0;
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) {
          const bool vv = base4 + u * SELECT_THREADS + tid < nvec;
#pragma unroll
          for (int q = 0; q < 4; ++q) c += vv && kk[4 * u + q] >= tau;
        }
        int incl = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += t;
        }
        int wb = 0;
        if (lane == 31 && incl) wb = atomicAdd(&misc[4], incl);
        int pos = __shfl_sync(0xffffffffu, wb, 31) + incl - c;
        if (c) {
#pragma unroll
          for (int u = 0; u < SEL_UNROLL; ++u) {
            const int vi = base4 + u * SELECT_THREADS + tid;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (vi < nvec && kk[4 * u + q] >= tau) {
                if (pos < SELECT_CAP) {
                  ckey[pos] = kk[4 * u + q];
                  cidx[pos] = a0 + vi * 4 + q;
                }
                ++pos;
              }
            }
          }
        }
      }
      // every thread reads the count before the barrier that lets the next
      // filter (after a threshold lookup that may take no barrier) reset it
      __syncthreads();
      const int count = misc[4];
      __syncthreads();
      return count;
    };

    // the certificate holds for any threshold: retry with a relaxed one when
    // the first leaves fewer than K candidates or more than fit
    int rk = sample_rank(m, L, target);
    uint32_t tau = tau_at_rank(rk);
    int n = filter(tau);
    for (int att = 0; att < 3 && !(n >= K && n <= SELECT_CAP); ++att) {
      if (n < K) {
        if (tau == 0u) break;
        rk *= 4;
      } else {
        if (rk <= 1) break;
        rk = max(1, rk / 4);
      }
      tau = tau_at_rank(rk);
      n = filter(tau);
    }
    uint32_t theta;
    int rr;
    if (n >= K && n <= SELECT_CAP) {
      group_radix_select([&](int i) { return ckey[i]; }, n, K, hist, misc, tid, SELECT_THREADS, 0, theta, rr, cmp,
                         SEL_CMP_CAP);
      group_emit([&](int i) { return ckey[i]; },
                 [&](int i) { return rs.paged ? out_index(rs, row, cidx[i]) : cidx[i]; }, n, theta, rr, K, o,
                 misc + 5, tid, SELECT_THREADS);
    } else {
      // no threshold separates the top K (massive ties): four radix passes
      // over the whole row, then emission
      uint32_t prefix = 0, mask = 0;
      int rem = K;
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int bb = tid; bb < 256; bb += SELECT_THREADS) hist[bb] = 0;
        __syncthreads();
        visit_row([&](uint32_t k, int, bool v) {
          hist_add(v && (k & mask) == prefix, (k >> shift) & 0xFFu, lane, hist);
        });
        __syncthreads();
        if (tid < 32) radix_pick_digit(hist, rem, misc);
        __syncthreads();
        prefix |= (uint32_t)misc[0] << shift;
        mask |= 0xFFu << shift;
        rem = misc[1];
        __syncthreads();
      }
      theta = prefix;
      rr = rem;
      visit_row([&](uint32_t k, int i, bool v) {
        const bool gt = v && k > theta, eq = v && k == theta;
        const unsigned mg = __ballot_sync(0xffffffffu, gt), me = __ballot_sync(0xffffffffu, eq);
        int bg = 0, be = 0;
        if (lane == 0) {
          if (mg) bg = atomicAdd(&misc[5], __popc(mg));
          if (me) be = atomicAdd(&misc[6], __popc(me));
        }
        bg = __shfl_sync(0xffffffffu, bg, 0);
        be = __shfl_sync(0xffffffffu, be, 0);
        if (gt) o[bg + __popc(mg & lt)] = rs.paged ? out_index(rs, row, i) : i;
        if (eq) {
          const int q2 = be + __popc(me & lt);
          if (q2 < rr) o[K - rr + q2] = rs.paged ? out_index(rs, row, i) : i;
        }
      });
    }
    __syncthreads();
  }
}

// ======================================================== candidate select ==
// Exact top-K of each planned row from the candidates the filter left
// ("Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2", section 3.2:
// every key at or above the threshold is a candidate, and when there are at
// least K of them the top K of the candidates are the top K of the row).
// The candidates stay in their regions in global memory (the scorer has
// just written them, mostly to L2) and each row reads them twice instead of
// staging them in shared memory.  Every candidate is at or above the row's
// threshold key tau, so the first pass histograms (key - tau) in CS_BINS
// bins of 2^CS_SHIFT0 key units (1/512 of a binade for normal floats; the
// last bin takes everything beyond) and places the K-th key in one bin b0;
// the histogram's descending exclusive prefix gives each bin above b0 its
// first output slot (a counting sort of those bins).  A bin b0 holding more
// than CS_STAGE keys is narrowed to a sub-interval by further CS_BINS-bin
// passes over its key interval (each divides the interval by CS_BINS, down
// to a single key value).  The last pass writes every key of the bins above
// b0 to its bin's next slot and the keys of b0 above the interval after
// them, and stages the interval's keys, whose rank-rem key (theta) is found
// by counting ranks.  One CTA per (group, row) item at a time with ~14 KB
// of shared memory, so many rows are in flight per SM.
constexpr int CS_BINS = 1024;
constexpr int CS_SHIFT0 = 14;
constexpr int CS_STAGE = 128;
// Two builds of the selector (measured on GB300): many rows (more than
// CS_FEW_PER_SM per SM), CTAs of 256 threads, 6 per SM, two 16-byte loads
// in flight per thread and pass (throughput); few rows, larger CTAs so that
// a row's loads take fewer rounds (its latency is the kernel's).
#ifndef DSA_CS_FEW_NT
#define DSA_CS_FEW_NT 512
#endif
#ifndef DSA_CS_FEW_CTAS
#define DSA_CS_FEW_CTAS 2
#endif
#ifndef DSA_CS_FEW_UNROLL
#define DSA_CS_FEW_UNROLL 4
#endif
constexpr int CS_MANY_NT = 256, CS_MANY_CTAS = 6, CS_MANY_UNROLL = 2;
constexpr int CS_FEW_NT = DSA_CS_FEW_NT, CS_FEW_CTAS = DSA_CS_FEW_CTAS, CS_FEW_UNROLL = DSA_CS_FEW_UNROLL;
constexpr int CS_FEW_PER_SM = 4;
constexpr uint32_t CS_OFF_HIST = 0;                                  // level-0 histogram, then slots
constexpr uint32_t CS_OFF_HIST2 = CS_OFF_HIST + CS_BINS * 4;         // narrowing passes
constexpr uint32_t CS_OFF_CNT = CS_OFF_HIST2 + CS_BINS * 4;          // per-region candidate counts
constexpr uint32_t CS_OFF_SKEY = CS_OFF_CNT + CAND_MAX_REGIONS * 4;  // the interval's keys
constexpr uint32_t CS_OFF_SIDX = CS_OFF_SKEY + CS_STAGE * 4;         // and ids
constexpr uint32_t CS_OFF_OUT = CS_OFF_SIDX + CS_STAGE * 4;          // the row's output, written out at the end
constexpr uint32_t CS_OFF_MISC = CS_OFF_OUT + MAX_K * 4;
constexpr uint32_t CAND_SMEM = CS_OFF_MISC + 64 * 4;
static_assert(CS_STAGE <= CS_MANY_NT && CS_STAGE <= CS_FEW_NT, "one staged key per thread");
static_assert(CS_MANY_CTAS * (CAND_SMEM + 1024) <= 228 * 1024 && CS_FEW_CTAS * (CAND_SMEM + 1024) <= 228 * 1024,
              "candidate-selector CTAs per SM");
static_assert(CS_MANY_CTAS * CS_MANY_NT <= 2048 && CS_FEW_CTAS * CS_FEW_NT <= 2048, "threads per SM");

template <int NT, int CTAS, int CS_UNROLL>
__global__ void __launch_bounds__(NT, CTAS) cand_select_kernel(const CandParams p) {
  constexpr int CS_PER_THREAD = CAND_MAX_REGIONS / NT;  // regions scanned per thread
  static_assert(CAND_MAX_REGIONS % NT == 0 && CS_BINS % NT == 0, "region scan, bins per thread");
  pdl_enter();
  extern __shared__ __align__(16) uint8_t smem[];
  int* hist = (int*)(smem + CS_OFF_HIST);
  int* hist2 = (int*)(smem + CS_OFF_HIST2);
  int* cnts = (int*)(smem + CS_OFF_CNT);
  uint32_t* skey = (uint32_t*)(smem + CS_OFF_SKEY);
  int32_t* sidx = (int32_t*)(smem + CS_OFF_SIDX);
  int32_t* so = (int32_t*)(smem + CS_OFF_OUT);
  // [0..7] bin pick, [17] staged count, [21] theta, [22] rr, [23..25]
  // emission counters (staged above / staged equal / single-value equal),
  // [26] last-CTA flag, [27] next item, [32..63] warp sums
  int* misc = (int*)(smem + CS_OFF_MISC);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NWARPS = NT / 32;
  const int K = p.K;
  const int items = p.stats->n_groups * GROUP_ROWS;
  // items: the CTA's own first, then (the many-row build) the next from a
  // counter: rows differ in cost, and a static split left SMs idle at the
  // end; the few-row build has at most one item per CTA
  constexpr bool dynamic = NT == CS_MANY_NT && CTAS == CS_MANY_CTAS;
  auto next_item = [&](int cur) {
    if (!dynamic) return cur + (int)gridDim.x;
    if (tid == 0) misc[27] = (int)gridDim.x + atomicAdd(&p.stats->cs_next, 1);
    __syncthreads();
    const int v = misc[27];
    __syncthreads();
    return v;
  };
  for (int it = blockIdx.x; it < items; it = next_item(it)) {
    const int g = it / GROUP_ROWS, r = it % GROUP_ROWS;
    const Group* gp = p.groups + g;
    if (r >= gp->nrows) continue;  // uniform over the CTA
    const int row = gp->row[r];
    // a paged group of at most two rows has two candidate teams per unit
    // (the scorer's virtual units 2 c and 2 c + 1)
    const int nu = (p.rs.paged && gp->nrows <= 2 ? 2 : 1) * (p.unit_start[g + 1] - p.unit_start[g]);
    const int nreg = nu * UNIT_REGIONS;
    const int wcap = region_cap(max(nu, 1));
    const int32_t* cnt = p.unit_count + (int64_t)row * p.max_units * UNIT_REGIONS;
    const uint32_t tau = __ldcg(&p.tau[row]);
    // certificate over the region counts (wcap + 1 = candidates were lost):
    // n >= K and no region lost any (the regions hold at most ROW_SLOTS, and
    // the candidates are read in place, so that bounds n)
    int tsum = 0;
    bool lost = nreg > CAND_MAX_REGIONS;
#pragma unroll
    for (int i = 0; i < CS_PER_THREAD; ++i) {
      const int j = tid * CS_PER_THREAD + i;
      // (a count is in [0, wcap + 1] unless the scorer gave up before
      // writing it: clamped, so a stale word cannot move a read out of
      // the row's slots)
      const int x = j < nreg ? max(__ldcg(&cnt[j]), 0) : 0;
      lost |= x > wcap;
      const int c = min(x, wcap);
      cnts[j] = c;
      tsum += c;
    }
    tsum = __reduce_add_sync(0xffffffffu, tsum);
    if (lane == 0) misc[32 + warp] = tsum;
#pragma unroll
    for (int j = 0; j < CS_BINS / NT; ++j) hist[tid + NT * j] = 0;
    if (tid == 0) misc[17] = misc[23] = misc[24] = misc[25] = 0;
    const bool any_lost = __syncthreads_or(lost);
    int n = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) n += misc[32 + w];
    if (n < K || any_lost) {
      if (tid == 0) {
        const int f = atomicAdd(&p.stats->fail_count, 1);
        p.failed_rows[f] = row;
        atomicAdd(n < K ? &p.stats->underflow : &p.stats->overflow, 1);
      }
      __syncthreads();
      continue;
    }
    if (tid == 0) atomicAdd(&p.stats->cand_total, n);
    const uint32_t* ck = p.cand_key + (int64_t)row * ROW_SLOTS;
    const int32_t* ci = p.cand_idx + (int64_t)row * ROW_SLOTS;
    // tpr threads per region, enough for one round of CS_UNROLL 16-byte
    // loads each over an average region (many short regions: one thread
    // each, so that all of a row's loads are in flight at once); a region
    // starts on a 4-entry boundary and holds a multiple of 4 slots, so its
    // last load stays inside it
    const int avg4 = ceil_div(n, 4 * nreg);
    int tpr = 1;
    while (tpr < 32 && tpr * CS_UNROLL < avg4) tpr *= 2;
    const int rstep = NT / tpr, sub = tid % tpr;

    // pass 1: histogram of (key - tau) >> CS_SHIFT0, and a check that no
    // candidate is below tau
    bool below = false;
    for (int jb = 0; jb < nreg; jb += rstep) {
      const int j = jb + tid / tpr;
      const int x = j < nreg ? cnts[j] : 0;
      const uint4* sk4 = reinterpret_cast<const uint4*>(ck + (int64_t)j * wcap);
      const int x4 = (x + 3) >> 2;
      for (int e = sub; e < x4; e += CS_UNROLL * tpr) {
        uint4 v[CS_UNROLL];
#pragma unroll
        for (int u = 0; u < CS_UNROLL; ++u) {
          const int eu = e + u * tpr;
          v[u] = eu < x4 ? __ldcg(&sk4[eu]) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < CS_UNROLL; ++u) {
          const uint32_t kk[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (4 * (e + u * tpr) + c < x) {
              below |= kk[c] < tau;
              atomicAdd(&hist[min((kk[c] - tau) >> CS_SHIFT0, (uint32_t)(CS_BINS - 1))], 1);
            }
          }
        }
      }
    }
    if (__syncthreads_or(below)) {
      // (the filter keeps keys at or above tau only: never taken; a row
      // that broke it is rescored exactly)
      if (tid == 0) {
        const int f = atomicAdd(&p.stats->fail_count, 1);
        p.failed_rows[f] = row;
        atomicAdd(&p.stats->overflow, 1);
      }
      __syncthreads();
      continue;
    }
    desc_scan_pick<NT>(hist, CS_BINS, K, misc, true);  // hist now holds each bin's first slot
    const uint32_t b0 = (uint32_t)misc[2];
    int rem = misc[3], bc = misc[4];
    // the K-th key's interval [lo, hi)
    unsigned long long lo = (unsigned long long)tau + ((unsigned long long)b0 << CS_SHIFT0);
    unsigned long long hi = 1ull << 32;
    if (b0 < CS_BINS - 1) hi = min(hi, lo + (1ull << CS_SHIFT0));
    // narrowing passes while the interval holds more keys than the stage
#pragma unroll 1
    while (bc > CS_STAGE && hi - lo > 1) {
      const int s = max(0, 64 - __clzll((long long)(hi - lo - 1)) - 10);
      const uint32_t lo32 = (uint32_t)lo, hin = (uint32_t)(hi - 1);
#pragma unroll
      for (int j = 0; j < CS_BINS / NT; ++j) hist2[tid + NT * j] = 0;
      __syncthreads();
      for (int jb = 0; jb < nreg; jb += rstep) {
        const int j = jb + tid / tpr;
        const int x = j < nreg ? cnts[j] : 0;
        const uint4* sk4 = reinterpret_cast<const uint4*>(ck + (int64_t)j * wcap);
        const int x4 = (x + 3) >> 2;
        for (int e = sub; e < x4; e += tpr) {
          const uint4 v = __ldcg(&sk4[e]);
          const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (4 * e + c < x && kk[c] >= lo32 && kk[c] <= hin) atomicAdd(&hist2[(kk[c] - lo32) >> s], 1);
        }
      }
      __syncthreads();
      desc_scan_pick<NT>(hist2, CS_BINS, rem, misc, false);
      rem = misc[3];
      bc = misc[4];
      lo += (unsigned long long)misc[2] << s;
      hi = min(hi, lo + (1ull << s));
    }
    const bool single = hi - lo == 1;  // the interval is one key value: theta
    const uint32_t lo32 = (uint32_t)lo, hin = (uint32_t)(hi - 1);
    int32_t* o = p.out + (int64_t)row * K;

    // last pass (slots in the shared copy of the row's output): the bins
    // above b0 to their slots ([0, A0)), the keys of b0 above the interval
    // next (to K - rem), the interval's keys staged (or, for a single value,
    // its first rem keys to [K - rem, K))
    for (int jb = 0; jb < nreg; jb += rstep) {
      const int j = jb + tid / tpr;
      const int x = j < nreg ? cnts[j] : 0;
      const uint4* sk4 = reinterpret_cast<const uint4*>(ck + (int64_t)j * wcap);
      const int4* si4 = reinterpret_cast<const int4*>(ci + (int64_t)j * wcap);
      const int x4 = (x + 3) >> 2;
      for (int e = sub; e < x4; e += CS_UNROLL * tpr) {
        uint4 v[CS_UNROLL];
        int4 d[CS_UNROLL];
#pragma unroll
        for (int u = 0; u < CS_UNROLL; ++u) {
          const int eu = e + u * tpr;
          v[u] = eu < x4 ? __ldcg(&sk4[eu]) : make_uint4(0, 0, 0, 0);
          d[u] = eu < x4 ? __ldcg(&si4[eu]) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < 4 * CS_UNROLL; ++c) {
          const uint4 vu = v[c >> 2];
          const int4 du = d[c >> 2];
          const uint32_t kq[4] = {vu.x, vu.y, vu.z, vu.w};
          const int32_t iq[4] = {du.x, du.y, du.z, du.w};
          if (4 * (e + (c >> 2) * tpr) + (c & 3) < x) {
            const uint32_t k = kq[c & 3];
            const int32_t idc = iq[c & 3];
            const uint32_t bin = min((k - tau) >> CS_SHIFT0, (uint32_t)(CS_BINS - 1));
            if (bin > b0) {
              so[atomicAdd(&hist[bin], 1)] = idc;
            } else if (bin == b0) {
              if (k > hin) {
                so[atomicAdd(&hist[b0], 1)] = idc;
              } else if (k >= lo32) {
                if (single) {
                  const int q = atomicAdd(&misc[25], 1);
                  if (q < rem) so[K - rem + q] = idc;
                } else {
                  const int q = atomicAdd(&misc[17], 1);
                  skey[q] = k;
                  sidx[q] = idc;
                }
              }
            }
          }
        }
      }
    }
    __syncthreads();
    if (!single) {
      // the rem-th largest of the bc staged keys: the first of its equal
      // keys whose count of larger keys is below rem and reaches rem with
      // its equals
      const bool mine = tid < bc;
      const uint32_t me = mine ? skey[tid] : 0u;
      if (mine) {
        int gt = 0, eq = 0, eqb = 0;
        for (int j = 0; j < bc; ++j) {
          const uint32_t y = skey[j];
          gt += y > me;
          eq += y == me;
          eqb += (y == me) & (j < tid);
        }
        if (eqb == 0 && gt < rem && rem <= gt + eq) {
          misc[21] = (int)me;
          misc[22] = rem - gt;
        }
      }
      __syncthreads();
      const uint32_t theta = (uint32_t)misc[21];
      const int rr = misc[22];
      if (mine) {
        if (me > theta) {
          so[K - rem + atomicAdd(&misc[23], 1)] = sidx[tid];
        } else if (me == theta) {
          const int q = atomicAdd(&misc[24], 1);
          if (q < rr) so[K - rr + q] = sidx[tid];
        }
      }
    }
    // the row out, coalesced (the slots above scatter)
    __syncthreads();
    for (int i = tid; i < K; i += NT) o[i] = so[i];
    __syncthreads();
  }
  // the CTA that finishes last writes the repair plan (the rows queued
  // above), which the repair scorer launched next reads
  if (p.plan_repair) {
    // (thread 0 wrote this CTA's failed-row entries: its fence orders them
    // before its ticket)
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      misc[26] = atomicAdd(&p.stats->cs_done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    const bool last = misc[26] != 0;
    if (last) {
      __threadfence();
      plan_groups(p.repair, repair_groups(p.repair), misc, hist);
    }
  }
}

cudaError_t launch_cand_select(const CandParams& p, int sms, cudaStream_t s) {
  static DeviceFlags attr_many, attr_few;
  if (p.rs.R > CS_FEW_PER_SM * sms) {
    auto k = cand_select_kernel<CS_MANY_NT, CS_MANY_CTAS, CS_MANY_UNROLL>;
    cudaError_t e = set_smem_attr_once(k, CAND_SMEM, attr_many);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(CS_MANY_CTAS * sms), dim3(CS_MANY_NT), CAND_SMEM, s, p);
  }
  auto k = cand_select_kernel<CS_FEW_NT, CS_FEW_CTAS, CS_FEW_UNROLL>;
  cudaError_t e = set_smem_attr_once(k, CAND_SMEM, attr_few);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(CS_FEW_CTAS * sms), dim3(CS_FEW_NT), CAND_SMEM, s, p);
}

// ============================================================ wide select ==
// The rows whose certificate failed are few and long: each is selected by a
// cluster of WIDE_CLUSTER CTAs (thread-block cluster), one slice of the row
// per CTA.  Keys are the order-preserving images of the repaired fp32
// scores; each radix pass fixes one byte of the K-th largest key: every CTA
// histograms its slice, rank 0 sums the cluster's histograms through
// distributed shared memory and picks the digit, and every CTA reads it
// back; hardware cluster barriers separate the phases.  One launch for all
// rows, which exits at once when no row failed.
constexpr int WIDE_CLUSTER = 8;
constexpr int WIDE_THREADS = 512;
constexpr int WIDE_UNROLL = 4;  // float4 loads in flight per thread

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// all threads of all CTAs of the cluster; orders shared and global memory
// at cluster scope
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// 32-bit load from the shared memory of CTA `rank` of the cluster, at the
// offset `p` has in this CTA
__device__ __forceinline__ int ld_dsmem(const int* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

__global__ void __cluster_dims__(WIDE_CLUSTER, 1, 1) __launch_bounds__(WIDE_THREADS)
    wide_cluster_kernel(const WideParams p) {
  pdl_enter();
  __shared__ int hist[256];
  __shared__ int tot[256];
  __shared__ int ctl[4];  // rank 0: digit, remaining rank; every rank: [2], [3] its emission totals
  __shared__ int wsum[2][WIDE_THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int nf = p.stats->fail_count;
  const int K = p.K;
  for (int f = (int)cluster_id_x(); f < nf; f += (int)cluster_count_x()) {
    const int row = p.list[f];
    const int b = p.rb[row], e = p.re[row];
    const float* srow = p.scores + (int64_t)(p.by_row ? row : f) * p.ld;
    // this CTA's slice: float4s covering [a, e) split in WIDE_CLUSTER parts
    const int a = b & ~3;
    const int n4 = ((e + 3) >> 2) - (a >> 2);
    const int per = ceil_div(n4, WIDE_CLUSTER);
    const int v0 = (int)rank * per, v1 = min(n4, v0 + per);
    const float4* v4 = reinterpret_cast<const float4*>(srow + a);
    // fn(key, index, valid) on all lanes, 4 keys per float4, WIDE_UNROLL
    // float4 loads in flight per thread (one at a time left every pass
    // waiting on the L2 latency); the order of a thread's keys is fixed
    auto visit = [&](auto&& fn) {
      for (int base = v0; base < v1; base += WIDE_THREADS * WIDE_UNROLL) {
        float4 x[WIDE_UNROLL];
#pragma unroll
        for (int u = 0; u < WIDE_UNROLL; ++u) {
          const int vi = base + u * WIDE_THREADS + tid;
          x[u] = vi < v1 ? __ldcg(&v4[vi]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < WIDE_UNROLL; ++u) {
          const int vi = base + u * WIDE_THREADS + tid;
          const bool in = vi < v1;
          const int i0 = a + 4 * vi;
          fn(ordered_key(x[u].x), i0 + 0, in && i0 + 0 >= b && i0 + 0 < e);
          fn(ordered_key(x[u].y), i0 + 1, in && i0 + 1 >= b && i0 + 1 < e);
          fn(ordered_key(x[u].z), i0 + 2, in && i0 + 2 >= b && i0 + 2 < e);
          fn(ordered_key(x[u].w), i0 + 3, in && i0 + 3 >= b && i0 + 3 < e);
        }
      }
    };
    uint32_t prefix = 0, mask = 0;
    int rem = K;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += WIDE_THREADS) hist[i] = 0;
      __syncthreads();
      visit([&](uint32_t k, int, bool v) { hist_add(v && (k & mask) == prefix, (k >> shift) & 0xFFu, lane, hist); });
      cluster_sync_all();  // every CTA's histogram is complete
      if (rank == 0) {
        for (int i = tid; i < 256; i += WIDE_THREADS) {
          int sum = 0;
#pragma unroll
          for (int r = 0; r < WIDE_CLUSTER; ++r) sum += ld_dsmem(&hist[i], (uint32_t)r);
          tot[i] = sum;
        }
        __syncthreads();
        if (tid < 32) radix_pick_digit(tot, rem, ctl);
      }
      cluster_sync_all();  // the digit is in rank 0's ctl
      const uint32_t digit = (uint32_t)ld_dsmem(&ctl[0], 0);
      rem = ld_dsmem(&ctl[1], 0);
      prefix |= digit << shift;
      mask |= 0xFFu << shift;
      cluster_sync_all();  // everyone read the digit before the next pass rewrites it
    }
    // every key above the K-th key and the first `rem` keys equal to it, in
    // the cluster's slice order: each thread counts its keys, a CTA scan
    // gives its offsets, the 8 CTA totals are exchanged through distributed
    // shared memory, then every thread writes its keys (no global atomics:
    // reservations on two counters shared by the cluster serialised it)
    const uint32_t theta = prefix;
    const int rr = rem;
    int32_t* o = p.out + (int64_t)row * K;
    int cg = 0, ce = 0;
    visit([&](uint32_t k, int, bool v) {
      cg += v && k > theta;
      ce += v && k == theta;
    });
    int ig = cg, ie = ce;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int tg = __shfl_up_sync(0xffffffffu, ig, d), te = __shfl_up_sync(0xffffffffu, ie, d);
      if (lane >= d) {
        ig += tg;
        ie += te;
      }
    }
    const int warp = tid >> 5;
    if (lane == 31) {
      wsum[0][warp] = ig;
      wsum[1][warp] = ie;
    }
    __syncthreads();
    int og = ig - cg, oe = ie - ce, cta_g = 0, cta_e = 0;
#pragma unroll
    for (int w = 0; w < WIDE_THREADS / 32; ++w) {
      og += w < warp ? wsum[0][w] : 0;
      oe += w < warp ? wsum[1][w] : 0;
      cta_g += wsum[0][w];
      cta_e += wsum[1][w];
    }
    if (tid == 0) {
      ctl[2] = cta_g;
      ctl[3] = cta_e;
    }
    cluster_sync_all();  // every CTA's totals are published
    for (uint32_t r = 0; r < rank; ++r) {
      og += ld_dsmem(&ctl[2], r);
      oe += ld_dsmem(&ctl[3], r);
    }
    visit([&](uint32_t k, int i, bool v) {
      if (v && k > theta) {
        if (og < K - rr) o[og] = p.rs.paged ? out_index(p.rs, row, i) : i;
        ++og;
      } else if (v && k == theta) {
        if (oe < rr) o[K - rr + oe] = p.rs.paged ? out_index(p.rs, row, i) : i;
        ++oe;
      }
    });
    cluster_sync_all();  // the row is done (and ctl read) before the cluster moves on
  }
}

cudaError_t launch_wide_select(const WideParams& p, int clusters, cudaStream_t s) {
  return launch_pdl(wide_cluster_kernel, dim3(clusters * WIDE_CLUSTER), dim3(WIDE_THREADS), 0, s, p);
}

cudaError_t launch_select(const SelectParams& p, int grid, cudaStream_t s) {
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_attr_once(select_kernel, SELECT_SMEM, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_kernel, dim3(grid), dim3(SELECT_THREADS), SELECT_SMEM, s, p);
}

// ======================================================== matrix filter ==
// Compare-and-append over a given fp32 score matrix ("Fusing Indexer Scoring
// and Exact Top-k for DeepSeek-V3.2", section 3.2, applied to a stored
// matrix): warp w of a 512-thread CTA takes row slot w / 4 of the unit's
// group and every 4th 128-key tile of the unit from tile w % 4 on, reading
// each tile as one float4 per lane, MF_UNROLL tiles in flight (the HBM
// latency needs about 64 KB in flight per SM, and two CTAs fit one); the
// scores that reach the row's threshold go to the warp's region of the row
// with a ballot and a register counter, and the count to unit_count at the
// end of the unit: the layout the candidate selector reads after the
// scorer's filter epilogue (any split of a unit's keys over its 4 regions
// serves it).
constexpr int MF_THREADS = 512;
constexpr int MF_UNROLL = 4;
// Compaction of the kept scores (measured on the standalone top-K): rows
// shorter than MF_SHORT_ROW keep a large share (~K of L) and use a ballot per
// score; in longer rows a warp step keeping at most MF_SCAN_MAX of its 512
// scores uses per-lane masks and one warp scan (4096 x 131072, ~3% kept:
// 0.773 -> 0.647 ms), a step keeping more (ties at the threshold) ballots
// over the mask bits.
constexpr int MF_SHORT_ROW = 32768;
constexpr int MF_SCAN_MAX = 48;
static_assert(MF_UNROLL == 4, "the kept-score mask and its selects are written for four float4s");

__global__ void __launch_bounds__(MF_THREADS) matrix_filter_kernel(const MatrixFilterParams p) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp >> 2, quarter = warp & 3;
  const int n_groups = p.stats->n_groups, total = p.stats->total_units;
  const uint32_t lt = lanemask_lt();
  // a contiguous range of units per CTA: the group is found once by binary
  // search and then advanced (a search per unit left the loads idle for as
  // long as the unit's own streaming took)
  const int per = ceil_div(total, (int)gridDim.x);
  const int u_begin = (int)blockIdx.x * per, u_end = min(total, u_begin + per);
  int g = 0;
  if (u_begin < u_end) {
    int lo = 0, hi = n_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(&p.unit_start[mid]) <= u_begin)
        lo = mid;
      else
        hi = mid - 1;
    }
    g = lo;
  }
  int g_start = u_begin < u_end ? __ldg(&p.unit_start[g]) : 0;
  int g_next = u_begin < u_end ? __ldg(&p.unit_start[g + 1]) : 0;
  for (int u = u_begin; u < u_end; ++u) {
    while (u >= g_next) {
      ++g;
      g_start = g_next;
      g_next = __ldg(&p.unit_start[g + 1]);
    }
    const int c = u - g_start;
    const int nunits = g_next - g_start;
    const Group* gp = p.groups + g;
    if (r >= gp->nrows) continue;  // uniform over the warp
    const int t0 = gp->lo / TILE + c * p.chunk_tiles;
    const int t1 = (int)min((int64_t)t0 + p.chunk_tiles, (int64_t)ceil_div(gp->hi, TILE));
    const int row = gp->row[r];
    const int b = p.rb[row], e = p.re[row];
    // the threshold as a float: score >= tauf <=> its key >= the threshold
    // key (non-NaN scores), so a key is formed only for the scores that pass
    const float tauf = key_threshold_float(p.tau[row]);
    const int wcap = region_cap(nunits);
    const int64_t region = (int64_t)row * ROW_SLOTS + (int64_t)(c * UNIT_REGIONS + quarter) * wcap;
    uint32_t* ck = p.cand_key + region;
    int32_t* ci = p.cand_idx + region;
    const float* srow = p.scores + (int64_t)row * p.ld;
    const bool short_row = e - b < MF_SHORT_ROW;
    int wcnt = 0;
    for (int t = t0 + quarter; t < t1; t += 4 * MF_UNROLL) {
      float4 x[MF_UNROLL];
#pragma unroll
      for (int v = 0; v < MF_UNROLL; ++v) {
        const int s = (t + 4 * v) * TILE + 4 * lane;  // first of the lane's 4 keys
        // a float4 wholly inside [b, e) (ld is a multiple of 4 and the row
        // range lies in [0, N]: a float4 that reaches into it stays inside
        // the row), zero when none of its keys is in range
        x[v] = (t + 4 * v < t1 && s + 3 >= b && s < e) ? __ldcs(reinterpret_cast<const float4*>(srow + s))
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (short_row) {
        // short rows keep a large share (~K of L): a ballot per score and
        // key position keeps the warp's stores in runs
#pragma unroll
        for (int v = 0; v < MF_UNROLL; ++v) {
          const int s0 = (t + 4 * v) * TILE + 4 * lane;
          const bool tile_in = t + 4 * v < t1;
          const float xs[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
          bool pr[4];
          if (tile_in && s0 >= b && s0 + 4 <= e) {
#pragma unroll
            for (int j = 0; j < 4; ++j) pr[j] = xs[j] >= tauf;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) pr[j] = tile_in && s0 + j >= b && s0 + j < e && xs[j] >= tauf;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t m = __ballot_sync(0xffffffffu, pr[j]);
            if (m) {  // warp-uniform: nothing to do when no lane keeps a score
              const int pos = wcnt + __popc(m & lt);
              if (pr[j] && pos < wcap) {
                ck[pos] = ordered_key(xs[j]);
                ci[pos] = s0 + j;
              }
              wcnt += __popc(m);
            }
          }
        }
        continue;
      }
      // long rows: the lane's kept scores as a 16-bit mask
      uint32_t mask = 0u;
#pragma unroll
      for (int v = 0; v < MF_UNROLL; ++v) {
        const int s0 = (t + 4 * v) * TILE + 4 * lane;
        const bool tile_in = t + 4 * v < t1;
        const float xs[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
        if (tile_in && s0 >= b && s0 + 4 <= e) {  // the common case: the whole float4 in range
#pragma unroll
          for (int j = 0; j < 4; ++j) mask |= (xs[j] >= tauf ? 1u : 0u) << (4 * v + j);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mask |= (tile_in && s0 + j >= b && s0 + j < e && xs[j] >= tauf ? 1u : 0u) << (4 * v + j);
        }
      }
      const int cnt = __popc(mask);
      const int tot = __reduce_add_sync(0xffffffffu, cnt);
      if (tot == 0) continue;  // warp-uniform
      if (tot <= MF_SCAN_MAX) {
        // few kept (long rows keep ~2K of L): one warp scan of the counts,
        // then each lane writes its own (a ballot per score costs four
        // times the instructions, and nearly every warp step keeps some)
        int incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += y;
        }
        int pos = wcnt + incl - cnt;
        while (mask) {
          const int q = __ffs(mask) - 1;
          mask &= mask - 1u;
          const int v = q >> 2, j = q & 3;
          const float4 xv = v == 0 ? x[0] : v == 1 ? x[1] : v == 2 ? x[2] : x[MF_UNROLL - 1];
          const float val = j == 0 ? xv.x : j == 1 ? xv.y : j == 2 ? xv.z : xv.w;
          if (pos < wcap) {
            ck[pos] = ordered_key(val);
            ci[pos] = (t + 4 * v) * TILE + 4 * lane + j;
          }
          ++pos;
        }
      } else {
        // many kept (ties at the threshold): a ballot per key position
        // keeps the warp's stores in runs
#pragma unroll
        for (int q = 0; q < 4 * MF_UNROLL; ++q) {
          const bool pr = (mask >> q) & 1u;
          const uint32_t m = __ballot_sync(0xffffffffu, pr);
          if (m) {  // warp-uniform
            const int pos = wcnt + __popc(m & lt);
            if (pr && pos < wcap) {
              const float4 xv = x[q >> 2];
              const float val = (q & 3) == 0 ? xv.x : (q & 3) == 1 ? xv.y : (q & 3) == 2 ? xv.z : xv.w;
              ck[pos] = ordered_key(val);
              ci[pos] = (t + 4 * (q >> 2)) * TILE + 4 * lane + (q & 3);
            }
            wcnt += __popc(m);
          }
        }
        continue;
      }
      wcnt += tot;
    }
    if (lane == 0) p.unit_count[(int64_t)row * p.max_units * UNIT_REGIONS + c * UNIT_REGIONS + quarter] = min(wcnt, wcap + 1);
  }
}

cudaError_t launch_matrix_filter(const MatrixFilterParams& p, int grid, cudaStream_t s) {
  return launch_pdl(matrix_filter_kernel, dim3(grid), dim3(MF_THREADS), 0, s, p);
}

// ============================================================== row top-K ==
// Exact top-K over a given fp32 score matrix ("Fusing Indexer Scoring and
// Exact Top-k for DeepSeek-V3.2", sections 3.2 and 3.3, over a stored
// matrix) in items of a whole row or, for many long rows, half a row.
// Eight warps per CTA: seven stream an item while the eighth takes the next
// item and its row's threshold from that row's own sample grid (the
// threshold kernel's grid, rank and per-warp radix select, so both halves
// of a row get the same threshold).  The stream compares each score with
// the threshold's float image and appends the scores at or above it to the
// item's candidate slots (one list per item, a shared counter), the next
// step's loads in flight while a step is compared.  The CTA that finishes a
// row (the second of its halves: a ticket per row) selects the row's top K
// from its lists with the candidate selector's passes (histogram over
// key - tau, narrowing, counting-sort emission, rank counting of the
// interval).  With half rows the selections fall at scattered times, so
// while some CTAs select the others keep the stream going (whole rows of
// equal length keep the CTAs in step: they all select at once), and the
// last items are short.
#ifndef DSA_RT_U
#define DSA_RT_U 4
#endif
constexpr int RT_SW = 7;                // stream warps
constexpr int RT_NS = RT_SW * 32;       // stream threads
constexpr int RT_NT = RT_NS + 32;       // and the threshold warp: the selection's threads
constexpr int RT_THREADS = RT_NT;
constexpr int RT_CTAS = MATRIX_TOPK_CTAS_PER_SM;
constexpr int RT_U = DSA_RT_U;          // float4s per thread and stream step (two steps in registers)
constexpr int RT_HALF = ROW_SLOTS / 2;  // candidate slots of each half of a row (items of half rows)
constexpr int RT_SU = 2;                // 16-byte candidate loads per thread and selection round
constexpr uint32_t RT_OFF_HIST = 0;
constexpr uint32_t RT_OFF_HIST2 = RT_OFF_HIST + CS_BINS * 4;
constexpr uint32_t RT_OFF_SKEY = RT_OFF_HIST2 + CS_BINS * 4;
constexpr uint32_t RT_OFF_SIDX = RT_OFF_SKEY + CS_STAGE * 4;
constexpr uint32_t RT_OFF_OUT = RT_OFF_SIDX + CS_STAGE * 4;
constexpr uint32_t RT_OFF_WHIST = RT_OFF_OUT + MAX_K * 4;
constexpr uint32_t RT_OFF_WPICK = RT_OFF_WHIST + 256 * 4;
constexpr uint32_t RT_OFF_MISC = RT_OFF_WPICK + 4 * 4;
constexpr uint32_t RT_OFF_STAGE = RT_OFF_MISC + 64 * 4;                   // per stream warp: a step's scores
constexpr uint32_t RT_OFF_LIST = RT_OFF_STAGE + RT_SW * RT_U * 32 * 16;  // and the offsets of its kept ones
constexpr uint32_t RT_SMEM = RT_OFF_LIST + RT_SW * RT_U * 32 * 4 * 2;
static_assert(RT_CTAS * (RT_SMEM + 1024) <= 228 * 1024 && RT_CTAS * RT_THREADS <= 2048, "row top-K CTAs per SM");
static_assert(CS_STAGE <= RT_NT && 1024 % RT_NT == 0 && 4 * RT_U <= 32, "staging, bins per thread, step mask");

// The threshold key of row `row` over [b, e) (L > K) from its grid scores in
// the matrix: the sample of descending rank ceil(m * target / L), plus the
// test bias; 0 (every key passes) when the rank falls outside the sample.
template <int KPL>
__device__ __forceinline__ uint32_t rt_threshold(const MatrixTopkParams& p, int row, int b, int e, int target,
                                                 int* whist, int* wpick) {
  const int lane = threadIdx.x & 31;
  int first, m, stride;
  sample_grid(b, e, &first, &m, &stride);
  m = min(m, MAX_SAMPLES);
  const int rank = sample_rank(m, e - b, target);
  uint32_t tau = 0u;
  if (m > 0 && m <= 32 * KPL && rank >= 1 && rank <= m) {
    const float* sr = p.scores + (int64_t)row * p.ld + first;
    uint32_t key[KPL];
#pragma unroll
    for (int q = 0; q < KPL; ++q) {
      const int i = q * 32 + lane;
      key[q] = i < m ? ordered_key(__ldcg(&sr[(int64_t)i * stride])) : 0u;
    }
    tau = warp_select_rank<KPL>(key, m, rank, whist, wpick);
    if (p.tau_bias != 0) {
      const int64_t t = (int64_t)tau + p.tau_bias;
      tau = (uint32_t)(t < 0 ? 0 : (t > 0xffffffffll ? 0xffffffffll : t));
    }
  }
  return tau;
}

// 0xffffffff when x >= t, else 0 (false for NaN)
__device__ __forceinline__ uint32_t ge_mask(float x, float t) {
  uint32_t r;
  asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(r) : "f"(x), "f"(t));
  return r;
}

// A stream thread's share of a row's whole float4s [fi0, fi1): float4
// fi0 + t, then every RT_NS-th, RT_U per step, the next step's loads in
// flight while a step is compared.  The warp's kept scores of a step go to
// ck / ci (cap slots) at consecutive positions from the shared counter
// *count: each lane stages its step in shared memory (stage: RT_U x 32
// float4s, position v, lane l at v * 32 + l) and lists the offsets of its
// kept scores there (list, in lane order: a warp scan of the counts), then
// lane j writes the list's j-th score.  With TIES, a score whose key equals
// the threshold key tau is kept only while the item holds fewer than K
// such (the shared counter *ties): a top K takes at most K keys equal to
// its K-th, and the keys at tau are below it unless tau is the K-th, so a
// row whose threshold falls on a heavily tied value (zeros) does not fill
// its slots with them (the second pass over an item whose list overflowed;
// the first places the warp's run before it forms the keys).  Steps whose
// every float4 lies inside the range (all but a row's last) take no
// per-lane range tests.
template <bool TIES>
__device__ __forceinline__ void rt_stream(const float4* s4, int fi0, int fi1, float tauf, uint32_t tau, int K,
                                          uint32_t* ck, int32_t* ci, int cap, int* count, int* ties, float4* stage,
                                          uint16_t* list) {
  constexpr int U = RT_U, NS = RT_NS;
  const int lane = threadIdx.x & 31;
  const int wt = (int)threadIdx.x - lane;  // the warp's first stream thread
  const float* stagef = reinterpret_cast<const float*>(stage);
  int fw = fi0 + wt;                       // lane 0's first float4 of the step
  float4 x[U];
#pragma unroll
  for (int v = 0; v < U; ++v) {
    const int f = fw + lane + v * NS;
    x[v] = f < fi1 ? __ldcs(&s4[f]) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll 1
  for (; fw < fi1; fw += U * NS) {  // (warp-uniform)
    const int fn = fw + U * NS;     // the next step
    float4 y[U];
    if (fn + 31 + (U - 1) * NS < fi1) {
#pragma unroll
      for (int v = 0; v < U; ++v) y[v] = __ldcs(&s4[fn + lane + v * NS]);
    } else {
#pragma unroll
      for (int v = 0; v < U; ++v) {
        const int f = fn + lane + v * NS;
        y[v] = f < fi1 ? __ldcs(&s4[f]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    uint32_t mask = 0u;
    if (fw + 31 + (U - 1) * NS < fi1) {
#pragma unroll
      for (int v = 0; v < U; ++v) {
        mask |= ge_mask(x[v].x, tauf) & (1u << (4 * v));
        mask |= ge_mask(x[v].y, tauf) & (1u << (4 * v + 1));
        mask |= ge_mask(x[v].z, tauf) & (1u << (4 * v + 2));
        mask |= ge_mask(x[v].w, tauf) & (1u << (4 * v + 3));
      }
    } else {
#pragma unroll
      for (int v = 0; v < U; ++v) {
        if (fw + lane + v * NS < fi1) {
          mask |= ge_mask(x[v].x, tauf) & (1u << (4 * v));
          mask |= ge_mask(x[v].y, tauf) & (1u << (4 * v + 1));
          mask |= ge_mask(x[v].z, tauf) & (1u << (4 * v + 2));
          mask |= ge_mask(x[v].w, tauf) & (1u << (4 * v + 3));
        }
      }
    }
    const int cnt = __popc(mask);
    int incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += t;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (tot != 0) {  // warp-uniform
      int base = 0;
      if (!TIES && lane == 31) base = atomicAdd(count, tot);
#pragma unroll
      for (int v = 0; v < U; ++v) stage[v * 32 + lane] = x[v];
      int p = incl - cnt;
      while (mask) {
        const int q = __ffs(mask) - 1;
        mask &= mask - 1u;
        list[p++] = (uint16_t)(((q >> 2) * 32 + lane) * 4 + (q & 3));
      }
      __syncwarp();
      if (!TIES) {
        base = __shfl_sync(0xffffffffu, base, 31);
        for (int j = lane; j < tot; j += 32) {
          const int code = list[j];
          const int pos = base + j;
          if (pos < cap) {
            ck[pos] = ordered_key(stagef[code]);
            ci[pos] = 4 * (fw + ((code >> 2) & 31) + (code >> 7) * NS) + (code & 3);
          }
        }
      }
      for (int jb = 0; TIES && jb < tot; jb += 32) {  // (warp-uniform)
        const int j = jb + lane;
        const bool active = j < tot;
        const int code = active ? list[j] : 0;
        const uint32_t key = ordered_key(stagef[code]);
        const bool tie = active && key == tau;
        bool keep = active && !tie;
        const uint32_t tb = __ballot_sync(0xffffffffu, tie);
        if (tb) {
          int t0 = 0;
          if (lane == 0) t0 = atomicAdd(ties, __popc(tb));
          t0 = __shfl_sync(0xffffffffu, t0, 0);
          keep |= tie && t0 + __popc(tb & lanemask_lt()) < K;
        }
        const uint32_t kb = __ballot_sync(0xffffffffu, keep);
        if (lane == 0 && kb) base = atomicAdd(count, __popc(kb));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(kb & lanemask_lt());
        if (keep && pos < cap) {
          ck[pos] = key;
          ci[pos] = 4 * (fw + ((code >> 2) & 31) + (code >> 7) * NS) + (code & 3);
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int v = 0; v < U; ++v) x[v] = y[v];
  }
}

// The exact top K of a row's candidates into o, by every thread of the CTA:
// the two halves' lists, slots [0, na) and [RT_HALF, RT_HALF + nb) of the
// row's (a whole row's list: nb = 0; K <= na + nb, every key at or above
// tau); false when a candidate lies below tau.  The lists are read as one sequence of 16-byte groups
// (a half's last group holds fewer than 4 of its keys).
template <bool TWO>
__device__ __forceinline__ bool rt_select(const uint32_t* ck, const int32_t* ci, int na, int nb, uint32_t tau,
                                          int K, int32_t* o, uint8_t* smem, int* misc) {
  constexpr int NT = RT_NT, SU = RT_SU;
  int* hist = (int*)(smem + RT_OFF_HIST);
  int* hist2 = (int*)(smem + RT_OFF_HIST2);
  uint32_t* skey = (uint32_t*)(smem + RT_OFF_SKEY);
  int32_t* sidx = (int32_t*)(smem + RT_OFF_SIDX);
  int32_t* so = (int32_t*)(smem + RT_OFF_OUT);
  const int tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < CS_BINS / NT; ++j) hist[tid + NT * j] = 0;
  if (tid == 0) misc[17] = misc[23] = misc[24] = misc[25] = 0;
  __syncthreads();
  const uint4* ck4 = reinterpret_cast<const uint4*>(ck);
  const int4* ci4 = reinterpret_cast<const int4*>(ci);
  const int na4 = (na + 3) >> 2, n4 = na4 + ((nb + 3) >> 2);
  // group e4 of the sequence: its place in the slots (in groups) and how
  // many of its 4 keys are candidates (the slots past a list's end up to a
  // multiple of 4 are read, not used)
  auto group = [&](int e4, int& lim) {
    if (!TWO || e4 < na4) {
      lim = na - 4 * e4;
      return e4;
    }
    lim = nb - 4 * (e4 - na4);
    return RT_HALF / 4 + (e4 - na4);
  };
  // pass 1: histogram of (key - tau) >> CS_SHIFT0, and a check that no
  // candidate is below tau
  bool below = false;
#pragma unroll 1
  for (int e4 = tid; e4 < n4; e4 += SU * NT) {
    uint4 v[SU];
    int lim[SU];
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      lim[u] = 0;
      v[u] = e4 + u * NT < n4 ? __ldcg(&ck4[group(e4 + u * NT, lim[u])]) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      const uint32_t kk[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c < lim[u]) {
          below |= kk[c] < tau;
          atomicAdd(&hist[min((kk[c] - tau) >> CS_SHIFT0, (uint32_t)(CS_BINS - 1))], 1);
        }
      }
    }
  }
  if (__syncthreads_or(below)) return false;  // (never: the stream keeps keys at or above tau)
  desc_scan_pick<NT>(hist, CS_BINS, K, misc, true);  // hist now holds each bin's first slot
  const uint32_t b0 = (uint32_t)misc[2];
  int rem = misc[3], bc = misc[4];
  unsigned long long lo = (unsigned long long)tau + ((unsigned long long)b0 << CS_SHIFT0);
  unsigned long long hi = 1ull << 32;
  if (b0 < CS_BINS - 1) hi = min(hi, lo + (1ull << CS_SHIFT0));
  // narrowing passes while the K-th key's interval holds more keys than the
  // stage
#pragma unroll 1
  while (bc > CS_STAGE && hi - lo > 1) {
    const int sh = max(0, 64 - __clzll((long long)(hi - lo - 1)) - 10);
    const uint32_t lo32 = (uint32_t)lo, hin = (uint32_t)(hi - 1);
#pragma unroll
    for (int j = 0; j < CS_BINS / NT; ++j) hist2[tid + NT * j] = 0;
    __syncthreads();
#pragma unroll 1
    for (int e4 = tid; e4 < n4; e4 += NT) {
      int lim;
      const uint4 v = __ldcg(&ck4[group(e4, lim)]);
      const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < lim && kk[c] >= lo32 && kk[c] <= hin) atomicAdd(&hist2[(kk[c] - lo32) >> sh], 1);
    }
    __syncthreads();
    desc_scan_pick<NT>(hist2, CS_BINS, rem, misc, false);
    rem = misc[3];
    bc = misc[4];
    lo += (unsigned long long)misc[2] << sh;
    hi = min(hi, lo + (1ull << sh));
  }
  const bool single = hi - lo == 1;  // the interval is one key value: theta
  const uint32_t lo32 = (uint32_t)lo, hin = (uint32_t)(hi - 1);
  // last pass (slots in the shared copy of the row's output): the bins above
  // b0 to their slots, the keys of b0 above the interval next, the
  // interval's keys staged (or, for a single value, its first rem keys to
  // [K - rem, K))
#pragma unroll 1
  for (int e4 = tid; e4 < n4; e4 += SU * NT) {
    uint4 v[SU];
    int4 d[SU];
    int lim[SU];
#pragma unroll
    for (int u = 0; u < SU; ++u) {
      lim[u] = 0;
      const bool ok = e4 + u * NT < n4;
      const int g = ok ? group(e4 + u * NT, lim[u]) : 0;
      v[u] = ok ? __ldcg(&ck4[g]) : make_uint4(0, 0, 0, 0);
      d[u] = ok ? __ldcg(&ci4[g]) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < 4 * SU; ++c) {
      const uint4 vu = v[c >> 2];
      const int4 du = d[c >> 2];
      const uint32_t k = (c & 3) == 0 ? vu.x : (c & 3) == 1 ? vu.y : (c & 3) == 2 ? vu.z : vu.w;
      const int32_t idc = (c & 3) == 0 ? du.x : (c & 3) == 1 ? du.y : (c & 3) == 2 ? du.z : du.w;
      if ((c & 3) < lim[c >> 2]) {
        const uint32_t bin = min((k - tau) >> CS_SHIFT0, (uint32_t)(CS_BINS - 1));
        if (bin > b0) {
          so[atomicAdd(&hist[bin], 1)] = idc;
        } else if (bin == b0) {
          if (k > hin) {
            so[atomicAdd(&hist[b0], 1)] = idc;
          } else if (k >= lo32) {
            if (single) {
              const int q = atomicAdd(&misc[25], 1);
              if (q < rem) so[K - rem + q] = idc;
            } else {
              const int q = atomicAdd(&misc[17], 1);
              skey[q] = k;
              sidx[q] = idc;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (!single) {
    // the rem-th largest of the bc staged keys and its ties
    const bool mine = tid < bc;
    const uint32_t me = mine ? skey[tid] : 0u;
    if (mine) {
      int gt = 0, eq = 0, eqb = 0;
      for (int j = 0; j < bc; ++j) {
        const uint32_t y = skey[j];
        gt += y > me;
        eq += y == me;
        eqb += (y == me) & (j < tid);
      }
      if (eqb == 0 && gt < rem && rem <= gt + eq) {
        misc[21] = (int)me;
        misc[22] = rem - gt;
      }
    }
    __syncthreads();
    const uint32_t theta = (uint32_t)misc[21];
    const int rr = misc[22];
    if (mine) {
      if (me > theta) {
        so[K - rem + atomicAdd(&misc[23], 1)] = sidx[tid];
      } else if (me == theta) {
        const int q = atomicAdd(&misc[24], 1);
        if (q < rr) so[K - rr + q] = sidx[tid];
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < K; i += NT) o[i] = so[i];
  return true;
}

// A stream warp's part of item `half` (of `parts`) of row `row` over [b, e):
// the item's share of the row's float4s wholly inside [b, e) into the
// item's slots (misc[12]: the count, misc[15]: keys at the threshold); the
// keys before and after them (fewer than 4 at each end) one by one, with
// the row's first and last item.
template <bool TIES>
__device__ __forceinline__ void rt_item(const MatrixTopkParams& p, int row, int b, int e, int half, int parts,
                                        uint32_t tau, int K, int* misc) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cap = ROW_SLOTS / parts;
  const int fi0 = (b + 3) >> 2, fi1 = e >> 2;
  const int fm = fi0 + max(fi1 - fi0, 0) / 2;
  const float tauf = key_threshold_float(tau);
  const float* srow = p.scores + (int64_t)row * p.ld;
  uint32_t* hk = p.cand_key + (int64_t)row * ROW_SLOTS + half * cap;
  int32_t* hi_ = p.cand_idx + (int64_t)row * ROW_SLOTS + half * cap;
  rt_stream<TIES>(reinterpret_cast<const float4*>(srow), half ? fm : fi0, half == parts - 1 ? fi1 : fm, tauf, tau, K,
                  hk, hi_, cap, &misc[12], &misc[15], reinterpret_cast<float4*>(smem + RT_OFF_STAGE) + warp * RT_U * 32,
                  reinterpret_cast<uint16_t*>(smem + RT_OFF_LIST) + warp * RT_U * 32 * 4);
  if (warp == 0 && ((lane == 0 && half == 0) || (lane == 1 && half == parts - 1))) {
    const int head_hi = min(e, 4 * fi0), tail_lo = max(4 * fi1, head_hi);
    const int lo = lane ? tail_lo : b, hi = lane ? e : head_hi;
    for (int s = lo; s < hi; ++s) {
      const float val = srow[s];
      const uint32_t key = ordered_key(val);
      if (val >= tauf && (!TIES || key != tau || atomicAdd(&misc[15], 1) < K)) {
        const int pos = atomicAdd(&misc[12], 1);
        if (pos < cap) {
          hk[pos] = key;
          hi_[pos] = s;
        }
      }
    }
  }
}

template <int KPL, int PARTS>
__global__ void __launch_bounds__(RT_THREADS, RT_CTAS) matrix_topk_kernel(const MatrixTopkParams p) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t smem[];
  int* whist = (int*)(smem + RT_OFF_WHIST);
  int* wpick = (int*)(smem + RT_OFF_WPICK);
  // [2..4] bin pick, [8] the next item's threshold, [10] the next item, [12]
  // candidates appended, [13] the row's ticket, [14] the other half's
  // count, [15] keys at the threshold met, [17] staged count, [21] theta,
  // [22] rr, [23..25] emission counters, [32..39] warp sums
  int* misc = (int*)(smem + RT_OFF_MISC);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.K, R = p.rs.R;
  constexpr int parts = PARTS, cap = ROW_SLOTS / PARTS;  // items per row (1 or 2), candidate slots per item
  const int items = parts * R;
  const int target = (int)(((int64_t)p.target16 * K) / 16);
  // items: part (item % parts) of row R - 1 - item / parts (prefill
  // chunks: the longest rows first); the CTA's own first, then from a
  // counter, each taken with its row's threshold by the threshold warp one
  // item ahead of the stream
  auto take = [&](int it) {
    uint32_t tau = 0u;
    if (it < items) {
      const int row = R - 1 - it / parts, b = p.rb[row], e = p.re[row];
      if (e - b > K) tau = rt_threshold<KPL>(p, row, b, e, target, whist, wpick);
      if (lane == 0 && it % parts == 0) p.tau[row] = tau;
    }
    if (lane == 0) {
      misc[10] = it;
      misc[8] = (int)tau;
    }
  };
  if (warp == RT_SW) take(blockIdx.x);
  __syncthreads();
  int ntriv = 0;
  while (true) {
    const int it = misc[10];
    if (it >= items) break;  // uniform
    const uint32_t tau = (uint32_t)misc[8];
    const int row = R - 1 - it / parts, half = it % parts;
    const int b = p.rb[row], e = p.re[row], L = e - b;
    uint32_t* ck = p.cand_key + (int64_t)row * ROW_SLOTS;
    int32_t* ci = p.cand_idx + (int64_t)row * ROW_SLOTS;
    if (tid == 0) misc[12] = misc[15] = 0;
    __syncthreads();  // the item is taken from the slot
    if (warp == RT_SW) {
      int itn = 0;
      if (lane == 0) itn = (int)gridDim.x + atomicAdd(&p.stats->cs_next, 1);
      take(__shfl_sync(0xffffffffu, itn, 0));
    } else if (L > K) {
      rt_item<false>(p, row, b, e, half, parts, tau, K, misc);
    } else if (half == 0) {  // every valid index, then -1
      int32_t* o = p.out + (int64_t)row * K;
      for (int i = tid; i < K; i += RT_NS) o[i] = i < L ? b + i : -1;
      ntriv += tid == 0;
    }
    __syncthreads();  // the item is streamed, the next item's threshold is in the slot
    if (L > K && misc[12] > cap) {
      // the list overflowed: once more with the keys at the threshold kept
      // up to K (a threshold on a heavily tied value), before the row goes
      // to the repair
      __syncthreads();
      if (tid == 0) misc[12] = misc[15] = 0;
      __syncthreads();
      if (warp < RT_SW) rt_item<true>(p, row, b, e, half, parts, tau, K, misc);
      __syncthreads();
    }
    if (L > K) {
      // half rows: the half's count, then the row's ticket (the CTA that
      // streamed the second of the two halves selects the row)
      if (parts == 2) {
        if (tid == 0) {
          p.half_count[2 * row + half] = misc[12];
          __threadfence();
          const int t = atomicAdd(&p.row_ticket[row], 1);
          misc[13] = t;
          if (t == 1) {
            __threadfence();
            misc[14] = __ldcg(&p.half_count[2 * row + (half ^ 1)]);
          }
        }
        __syncthreads();
      }
      if (parts == 1 || misc[13] == 1) {
        // certificate: at least K candidates, none lost (an item's slots
        // hold cap)
        const int na = parts == 1 ? misc[12] : half ? misc[14] : misc[12];
        const int nb = parts == 1 ? 0 : half ? misc[12] : misc[14];
        bool ok = na + nb >= K && na <= cap && nb <= cap;
        if (ok) {
          if (tid == 0) atomicAdd(&p.stats->cand_total, na + nb);
          ok = rt_select<PARTS == 2>(ck, ci, na, nb, tau, K, p.out + (int64_t)row * K, smem, misc);
        }
        if (!ok && tid == 0) {
          const int fr = atomicAdd(&p.stats->fail_count, 1);
          p.failed_rows[fr] = row;
          atomicAdd(na + nb < K ? &p.stats->underflow : &p.stats->overflow, 1);
        }
      }
    }
    __syncthreads();
  }
  if (tid == 0 && ntriv) atomicAdd(&p.stats->trivial, ntriv);
}

template <int PARTS>
static cudaError_t launch_matrix_topk_parts(const MatrixTopkParams& p, int sms, cudaStream_t s) {
  static DeviceFlags attr_short, attr_long;
  const int grid = max(1, min(PARTS * p.rs.R, RT_CTAS * sms));
  // the threshold's grid keys sit in the threshold warp's registers: the
  // build holding up to 672 (rows of up to ~134K keys) or MAX_SAMPLES
  const int64_t max_m = std::min<int64_t>(MAX_SAMPLES, (int64_t)p.rs.N / SAMPLE_STRIDE + 2);
  if (max_m <= 32 * TAU_KPL_SHORT) {
    auto k = matrix_topk_kernel<TAU_KPL_SHORT, PARTS>;
    cudaError_t e = set_smem_attr_once(k, RT_SMEM, attr_short);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(RT_THREADS), RT_SMEM, s, p);
  }
  auto k = matrix_topk_kernel<MAX_SAMPLES / 32, PARTS>;
  cudaError_t e = set_smem_attr_once(k, RT_SMEM, attr_long);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(RT_THREADS), RT_SMEM, s, p);
}

cudaError_t launch_matrix_topk(const MatrixTopkParams& p, int sms, cudaStream_t s) {
  return p.parts == 2 ? launch_matrix_topk_parts<2>(p, sms, s) : launch_matrix_topk_parts<1>(p, sms, s);
}


}  // namespace dsa
