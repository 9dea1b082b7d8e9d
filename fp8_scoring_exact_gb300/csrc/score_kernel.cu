// score_kernel.cu -- persistent, warp-specialised tcgen05 scorer.
//
// One CTA per SM walks a static share of the work units (query-row pair x
// chunk of 128-key tiles) of a plan built on the device.  Roles:
//   warp 0      TMA producer: q rows of the pair, key tiles (128 keys x 128 B,
//               128-byte swizzle) into a STAGES-deep ring, key scales into a
//               separate SC_STAGES ring;
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4
//               (M = 128 keys, N = 64 heads x rows, K = 32) per tile into one
//               of ACC_BUFS TMEM accumulators; owns the TMEM allocation;
//   warps 2-3   TopK warps (MODE_FILTER): exact selection of finished rows;
//   warps 4-11  two epilogue warpgroups; warpgroup r handles row r of the
//               pair, one thread per key (= TMEM lane), 64 heads per thread:
//               score = k_scale * sum_j (w_j q_scale) ReLU(D_j), then
//               MODE_STORE writes the fp32 score, MODE_FILTER appends
//               (key, index) when the key reaches the row's sampled threshold.
//
// The method (candidate filter against a sampled threshold, radix select, the
// certificate and ready/free double buffering) follows "Fusing Indexer Scoring
// and Exact Top-k for DeepSeek-V3.2", sections 3.2 and 4; the tile shapes,
// TMEM accumulators and global candidate buffers are this GB300 design.
#include "common.cuh"
#include "kernels.h"
#include "rows.cuh"

namespace dsa {

namespace {

constexpr int KEY_STAGE_BYTES = TILE * D;            // 16384
constexpr int Q_SLOT_BYTES = GROUP_ROWS * H * D;     // 16384
constexpr int Q_ROW_BYTES = H * D;                   // 8192
constexpr int SC_STAGE_BYTES = TILE * 4;             // 512

constexpr uint32_t OFF_KEYS = 0;
constexpr uint32_t OFF_Q = OFF_KEYS + STAGES * KEY_STAGE_BYTES;
constexpr uint32_t OFF_SC = OFF_Q + 2 * Q_SLOT_BYTES;
constexpr uint32_t OFF_TK = OFF_SC + SC_STAGES * SC_STAGE_BYTES;
constexpr uint32_t OFF_HIST = OFF_TK + CAND_CAP * 4;
constexpr uint32_t OFF_BAR = OFF_HIST + 256 * 4;
constexpr int N_BARS = 2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + 2 * TOPK_QUEUE + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr uint32_t MISC_BYTES = 256;
constexpr uint32_t SMEM_USED = OFF_MISC + MISC_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_KEYS % 1024 == 0, "swizzled tiles need 1024-byte alignment");

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int tq_group[TOPK_QUEUE];
  int sc_page[SC_STAGES][2];
  int sdig[2];
  int s_above;
  int s_eq;
  int tk_group;
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc block");

struct Unit {
  int g, t0, t1, nunits;
};

__device__ __forceinline__ int find_group(const int32_t* unit_start, int n_groups, int u) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&unit_start[mid]) <= u)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Unit decode_unit(const ScoreParams& p, int n_groups, int u, Group& G) {
  Unit un;
  un.g = find_group(p.unit_start, n_groups, u);
  const int c = u - __ldg(&p.unit_start[un.g]);
  un.nunits = __ldg(&p.unit_start[un.g + 1]) - __ldg(&p.unit_start[un.g]);
  G = p.groups[un.g];
  const int lo_t = G.lo / TILE;
  const int hi_t = ceil_div(G.hi, TILE);
  un.t0 = lo_t + c * p.chunk_tiles;
  un.t1 = min(un.t0 + p.chunk_tiles, hi_t);
  return un;
}

}  // namespace

__global__ void __launch_bounds__(SCORE_THREADS, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_ks, const ScoreParams p) {
  const int n_groups = p.repair ? p.stats->r_groups : p.stats->n_groups;
  const int total = p.repair ? p.stats->r_units : p.stats->total_units;
  if ((int)blockIdx.x >= total) return;  // uniform over the CTA: no work

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  Misc* misc = (Misc*)(smem + OFF_MISC);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto key_full = [&](int i) { return bar0 + 8u * i; };
  auto key_empty = [&](int i) { return bar0 + 8u * (STAGES + i); };
  auto sc_full = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto sc_empty = [&](int i) { return bar0 + 8u * (2 * STAGES + SC_STAGES + i); };
  auto q_full = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + i); };
  auto q_empty = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 2 + i); };
  auto acc_full = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + i); };
  auto acc_empty = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + ACC_BUFS + i); };
  auto tq_full = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + i); };
  auto tq_empty = [&](int i) {
    return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + TOPK_QUEUE + i);
  };
  const uint32_t unit_bar = bar0 + 8u * (N_BARS - 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &misc->abort_flag;
  int* status = &p.stats->status;
  const bool filter = (p.mode == MODE_FILTER);

  if (threadIdx.x == 0) {
    misc->abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(key_full(i), 1);
      mbar_init(key_empty(i), 1);
    }
    for (int i = 0; i < SC_STAGES; ++i) {
      mbar_init(sc_full(i), 1);
      mbar_init(sc_empty(i), EPI_THREADS / 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), 1);
    }
    for (int i = 0; i < ACC_BUFS; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(acc_empty(i), EPI_THREADS / 32);
    }
    for (int i = 0; i < TOPK_QUEUE; ++i) {
      mbar_init(tq_full(i), 1);
      mbar_init(tq_empty(i), 1);
    }
    mbar_init(unit_bar, EPI_THREADS / 32);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), ACC_BUFS * ACC_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_ks);
      uint32_t kit = 0, ui = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++ui) {
        Group G;
        const Unit un = decode_unit(p, n_groups, u, G);
        const int qs = ui & 1;
        if (!(ok = mbar_wait(q_empty(qs), ((ui >> 1) & 1) ^ 1, abort_flag, status))) break;
        mbar_arrive_expect_tx(q_full(qs), G.nrows * Q_ROW_BYTES);
        for (int r = 0; r < G.nrows; ++r)
          tma_load_2d(sbase + OFF_Q + qs * Q_SLOT_BYTES + r * Q_ROW_BYTES, &tm_q, 0, G.row[r] * H, q_full(qs));
        for (int t = un.t0; t < un.t1; ++t, ++kit) {
          const int st = kit % STAGES;
          const uint32_t ph = (kit / STAGES) & 1;
          if (!(ok = mbar_wait(key_empty(st), ph ^ 1, abort_flag, status))) break;
          int pg0 = 0, pg1 = -1;
          if (p.rs.paged) {
            const int32_t* bt = p.rs.block_table + (int64_t)G.seq * p.rs.max_pages;
            // a page id outside the cache is clamped to the first row past it:
            // TMA then reads zeros there instead of touching foreign memory
            pg0 = __ldg(&bt[2 * t]);
            if (pg0 < 0 || pg0 >= p.rs.num_pages) pg0 = p.rs.num_pages;
            if (t * TILE + PAGE < G.hi) {
              pg1 = __ldg(&bt[2 * t + 1]);
              if (pg1 < 0 || pg1 >= p.rs.num_pages) pg1 = p.rs.num_pages;
            }
          }
          const uint32_t kdst = sbase + OFF_KEYS + st * KEY_STAGE_BYTES;
          if (!p.rs.paged) {
            mbar_arrive_expect_tx(key_full(st), KEY_STAGE_BYTES);
            tma_load_2d(kdst, &tm_k, 0, t * TILE, key_full(st));
          } else {
            mbar_arrive_expect_tx(key_full(st), (pg1 >= 0 ? 2 : 1) * PAGE * D);
            tma_load_2d(kdst, &tm_k, 0, pg0 * PAGE, key_full(st));
            if (pg1 >= 0) tma_load_2d(kdst + PAGE * D, &tm_k, 0, pg1 * PAGE, key_full(st));
          }
          const int ss = kit % SC_STAGES;
          const uint32_t sph = (kit / SC_STAGES) & 1;
          if (!(ok = mbar_wait(sc_empty(ss), sph ^ 1, abort_flag, status))) break;
          misc->sc_page[ss][0] = pg0;
          misc->sc_page[ss][1] = pg1;
          const uint32_t sdst = sbase + OFF_SC + ss * SC_STAGE_BYTES;
          if (!p.rs.paged) {
            mbar_arrive_expect_tx(sc_full(ss), SC_STAGE_BYTES);
            tma_load_1d(sdst, &tm_ks, t * TILE, sc_full(ss));
          } else {
            mbar_arrive_expect_tx(sc_full(ss), (pg1 >= 0 ? 2 : 1) * PAGE * 4);
            tma_load_1d(sdst, &tm_ks, pg0 * PAGE, sc_full(ss));
            if (pg1 >= 0) tma_load_1d(sdst + PAGE * 4, &tm_ks, pg1 * PAGE, sc_full(ss));
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t kit = 0, ait = 0, ui = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++ui) {
        Group G;
        const Unit un = decode_unit(p, n_groups, u, G);
        const int qs = ui & 1;
        if (!(ok = mbar_wait(q_full(qs), (ui >> 1) & 1, abort_flag, status))) break;
        const uint32_t idesc = idesc_e4m3_f32(TILE, H * G.nrows);
        const uint32_t qaddr = sbase + OFF_Q + qs * Q_SLOT_BYTES;
        for (int t = un.t0; t < un.t1; ++t, ++kit, ++ait) {
          const int st = kit % STAGES;
          if (!(ok = mbar_wait(key_full(st), (kit / STAGES) & 1, abort_flag, status))) break;
          const int ab = ait % ACC_BUFS;
          if (!(ok = mbar_wait(acc_empty(ab), ((ait / ACC_BUFS) & 1) ^ 1, abort_flag, status))) break;
          tc_fence_after();
          const uint32_t kaddr = sbase + OFF_KEYS + st * KEY_STAGE_BYTES;
          const uint32_t d = tmem_base + ab * ACC_COLS;
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            mma_e4m3(d, sw128_kmajor_desc(kaddr + 32 * k), sw128_kmajor_desc(qaddr + 32 * k), idesc, k > 0);
          mma_commit(key_empty(st));
          mma_commit(acc_full(ab));
        }
        if (ok) mma_commit(q_empty(qs));
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- TopK warps --
    if (filter) {
      const int tid = threadIdx.x - 64;
      int* hist = (int*)(smem + OFF_HIST);
      uint32_t* skey = (uint32_t*)(smem + OFF_TK);
      const int K = p.K;
      for (uint32_t qi = 0;; ++qi) {
        const int slot = qi % TOPK_QUEUE;
        // one thread waits (bounded) and decides for the whole TopK group
        if (tid == 0) {
          int gg = -2;
          if (mbar_wait(tq_full(slot), (qi / TOPK_QUEUE) & 1, abort_flag, status))
            gg = ((volatile int*)misc->tq_group)[slot];
          misc->tk_group = gg;
        }
        named_bar_sync(2, TOPK_THREADS);
        const int g = ((volatile Misc*)misc)->tk_group;
        if (g < 0) break;
        __threadfence();
        const Group G = p.groups[g];
        for (int r = 0; r < G.nrows; ++r) {
          const int row = G.row[r];
          const int n = __ldcg(&p.cand_count[row]);
          if (n < K || n > CAND_CAP) {
            if (tid == 0) {
              const int f = atomicAdd(&p.stats->fail_count, 1);
              p.failed_rows[f] = row;
              atomicAdd(n < K ? &p.stats->underflow : &p.stats->overflow, 1);
            }
            continue;
          }
          const uint32_t* ck = p.cand_key + (int64_t)row * CAND_CAP;
          const int32_t* ci = p.cand_idx + (int64_t)row * CAND_CAP;
          for (int i = tid; i < n; i += TOPK_THREADS) skey[i] = __ldcg(&ck[i]);
          if (tid == 0) {
            misc->s_above = 0;
            misc->s_eq = 0;
            atomicAdd(&p.stats->cand_total, n);
          }
          named_bar_sync(2, TOPK_THREADS);
          uint32_t theta;
          int rr;
          group_radix_select([&](int i) { return skey[i]; }, n, K, hist, misc->sdig, tid, TOPK_THREADS, 2, theta,
                             rr);
          int32_t* o = p.out + (int64_t)row * K;
          for (int i = tid; i < n; i += TOPK_THREADS) {
            const uint32_t k = skey[i];
            if (k > theta) {
              const int pos = atomicAdd(&misc->s_above, 1);
              o[pos] = __ldcg(&ci[i]);
            } else if (k == theta) {
              const int e = atomicAdd(&misc->s_eq, 1);
              if (e < rr) o[K - rr + e] = __ldcg(&ci[i]);
            }
          }
          named_bar_sync(2, TOPK_THREADS);
        }
        named_bar_sync(2, TOPK_THREADS);
        if (tid == 0) mbar_arrive(tq_empty(slot));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - 4;             // 0..7
    const int r = ew >> 2;               // row slot of the pair
    const int quarter = warp & 3;        // TMEM lane quarter of this warp
    const int etid = threadIdx.x - 128;  // 0..255
    const float* sc_base = (const float*)(smem + OFF_SC);
    uint32_t ait = 0, kit = 0, qi = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++ui) {
      Group G;
      const Unit un = decode_unit(p, n_groups, u, G);
      const bool active = r < G.nrows;
      const int row = active ? G.row[r] : 0;
      float wq[H];
      int rb = 0, re = 0;
      uint32_t tau = 0;
      int32_t* cnt = nullptr;
      uint32_t* ck = nullptr;
      int32_t* ci = nullptr;
      float* srow = nullptr;
      int64_t store_lim = 0;
      if (active) {
        const float qsc = __ldg(&p.q_scale[row]);
#pragma unroll
        for (int j = 0; j < H; ++j) wq[j] = __ldg(&p.w[(int64_t)row * H + j]) * qsc;
        rb = __ldg(&p.rb[row]);
        re = __ldg(&p.re[row]);
        if (filter) {
          tau = __ldg(&p.tau[row]);
          cnt = p.cand_count + row;
          ck = p.cand_key + (int64_t)row * CAND_CAP;
          ci = p.cand_idx + (int64_t)row * CAND_CAP;
        } else {
          srow = p.scores + (int64_t)G.slot[r] * p.ld;
          store_lim = min((int64_t)p.rs.N, p.ld);
        }
      }
      for (int t = un.t0; t < un.t1; ++t, ++ait, ++kit) {
        const int ab = ait % ACC_BUFS;
        if (!(ok = mbar_wait_warp(acc_full(ab), (ait / ACC_BUFS) & 1, abort_flag, status))) break;
        const int ss = kit % SC_STAGES;
        if (!(ok = mbar_wait_warp(sc_full(ss), (kit / SC_STAGES) & 1, abort_flag, status))) break;
        tc_fence_after();
        const int kt = quarter * 32 + lane;  // key within the tile = TMEM lane
        uint32_t v[H];
        if (active) {
          const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * ACC_COLS + r * H;
          tmem_ld32(ta, v);
          tmem_ld32(ta + 32, v + 32);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(ab));
        const float ks = sc_base[ss * TILE + kt];
        int page = 0;
        if (p.rs.paged) page = misc->sc_page[ss][kt >> 6];
        __syncwarp();
        if (lane == 0) mbar_arrive(sc_empty(ss));
        if (!active) continue;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int j = 0; j < H; j += 2) {
          a0 = fmaf(wq[j], fmaxf(__uint_as_float(v[j]), 0.f), a0);
          a1 = fmaf(wq[j + 1], fmaxf(__uint_as_float(v[j + 1]), 0.f), a1);
        }
        const float score = (a0 + a1) * ks;
        const int s = t * TILE + kt;
        const bool valid = (s >= rb) && (s < re);
        if (filter) {
          const bool pred = valid && (ordered_key(score) >= tau);
          const uint32_t m = __ballot_sync(0xffffffffu, pred);
          if (m) {
            int base = 0;
            if (lane == 0) base = atomicAdd(cnt, __popc(m));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (pred) {
              const int pos = base + __popc(m & lanemask_lt());
              if (pos < CAND_CAP) {
                ck[pos] = ordered_key(score);
                ci[pos] = p.rs.paged ? page * PAGE + (s & (PAGE - 1)) : s;
              }
            }
          }
        } else if (s < store_lim) {
          srow[s] = valid ? score : -__int_as_float(0x7f800000);
        }
      }
      if (filter && ok) {
        // unit done: publish this CTA's candidates, then count the unit; the
        // CTA finishing a group's last unit hands the group to its TopK warps
        __threadfence();
        __syncwarp();
        if (lane == 0) mbar_arrive(unit_bar);
        if (etid == 0) {
          if (!(ok = mbar_wait(unit_bar, ui & 1, abort_flag, status))) break;
          const int done = atomicAdd(&p.group_done[un.g], 1) + 1;
          if (done == un.nunits) {
            const int slot = qi % TOPK_QUEUE;
            if (!(ok = mbar_wait(tq_empty(slot), ((qi / TOPK_QUEUE) & 1) ^ 1, abort_flag, status))) break;
            ((volatile int*)misc->tq_group)[slot] = un.g;
            mbar_arrive(tq_full(slot));
            ++qi;
          }
        }
      }
    }
    if (filter && etid == 0) {
      const int slot = qi % TOPK_QUEUE;
      if (mbar_wait(tq_empty(slot), ((qi / TOPK_QUEUE) & 1) ^ 1, abort_flag, status)) {
        ((volatile int*)misc->tq_group)[slot] = -1;
        mbar_arrive(tq_full(slot));
      }
    }
  }

  __syncthreads();
  if (misc->abort_flag) {
    // a wait gave up: let copies and MMAs already issued land before the
    // shared memory and TMEM are released
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ACC_BUFS * ACC_COLS);
  }
}

cudaError_t launch_score(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_ks,
                         const ScoreParams& p, int grid, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  score_kernel<<<grid, SCORE_THREADS, SMEM_BYTES, s>>>(tm_q, tm_k, tm_ks, p);
  return cudaGetLastError();
}

}  // namespace dsa
