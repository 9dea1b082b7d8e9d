// score_kernel.cu -- persistent, warp-specialised tcgen05 scorer.
//
// One CTA per SM walks a static share (u = blockIdx.x, + gridDim.x, ...) of
// the work units of a plan built on the device: a unit is a group of up to 4
// query rows (which stream the same keys) with a chunk of 128-key tiles.
// Roles:
//   warp 0       TMA producer: q rows of the group (64 heads x 128 B each),
//                key tiles (128 keys x 128 B, 128-byte swizzle) into a
//                STAGES-deep ring, key scales into a separate ring;
//   warp 1       MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 per
//                tile, M = 128 keys, N = 64 heads x rows (256 for 4 rows),
//                K = 32, fp32 accumulators in one of two 256-column TMEM
//                buffers; owns the TMEM allocation;
//   warps 2-3    TopK warps (MODE_FILTER): exact selection of groups
//                blockIdx.x, + (CTAs with work), ..., each once every unit
//                of the group has published its candidates;
//   warps 4-19   epilogue: warpgroup r handles row r of the group.  Each
//                thread reads two keys x 16 heads per TMEM load (16x256b
//                shape), keeps the 16 weights w * q_scale in registers,
//                applies ReLU and the weights with packed f32x2 FMAs, and a
//                three-shuffle reduce-scatter over 4 lanes leaves one key's
//                64-head sum per thread; then score = sum * k_scale.
//                MODE_STORE writes the fp32 score.  MODE_FILTER keeps the
//                scores that reach the row's sampled threshold: key
//                (order-preserving uint32) and index go to the unit's region
//                of the row's candidate buffers, slots counted in shared
//                memory; at the end of the unit the count is stored and the
//                group's completion counter is released.
//
// The method (candidate filter against a sampled threshold, radix select, the
// certificate, selection overlapped with scoring) follows "Fusing Indexer
// Scoring and Exact Top-k for DeepSeek-V3.2", sections 3.2 and 4.  The
// readiness of a group for selection is a release/acquire counter; the
// candidate regions are per row, so no buffer has to be handed back.
#include "common.cuh"
#include "kernels.h"
#include "rows.cuh"

namespace dsa {

namespace {

constexpr int KEY_STAGE_BYTES = TILE * D;            // 16384
constexpr int Q_ROW_BYTES = H * D;                   // 8192
constexpr int Q_SLOT_BYTES = GROUP_ROWS * Q_ROW_BYTES;  // 32768
constexpr int SC_STAGE_BYTES = TILE * 4;             // 512

constexpr uint32_t OFF_KEYS = 0;
constexpr uint32_t OFF_Q = OFF_KEYS + STAGES * KEY_STAGE_BYTES;
constexpr uint32_t OFF_SC = OFF_Q + 2 * Q_SLOT_BYTES;
constexpr uint32_t OFF_TKEY = OFF_SC + SC_STAGES * SC_STAGE_BYTES;  // TopK: gathered keys
constexpr uint32_t OFF_TIDX = OFF_TKEY + CAND_CAP * 4;              // TopK: gathered indices
constexpr uint32_t OFF_HIST = OFF_TIDX + CAND_CAP * 4;
constexpr uint32_t OFF_BAR = OFF_HIST + 256 * 4;
constexpr int N_BARS = 2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr uint32_t MISC_BYTES = 256;
constexpr uint32_t SMEM_USED = OFF_MISC + MISC_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_KEYS % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(ACC_BUFS * ACC_COLS <= 512, "TMEM columns");

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int sc_page[SC_STAGES][2];
  int sdig[4];
  int emit_cnt[2];
  int gather_n;
  int ucnt[EPI_WGS];
};
static_assert(sizeof(Misc) <= MISC_BYTES, "misc block");

struct Unit {
  int g, c, t0, t1, nunits;
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
  un.c = u - __ldg(&p.unit_start[un.g]);
  un.nunits = __ldg(&p.unit_start[un.g + 1]) - __ldg(&p.unit_start[un.g]);
  G = p.groups[un.g];
  const int lo_t = G.lo / TILE;
  const int hi_t = ceil_div(G.hi, TILE);
  un.t0 = lo_t + un.c * p.chunk_tiles;
  un.t1 = (int)min((int64_t)un.t0 + p.chunk_tiles, (int64_t)hi_t);
  return un;
}

// Partial sums of two keys over this thread's 16 heads from one 16x256b.x8
// TMEM load: ReLU on the FMA pipe (saturating multiply by 2^-25, exact since
// |x| < 2^25), weights pre-scaled by 2^25, packed f32x2 FMAs.
__device__ __forceinline__ void two_key_partials(const uint32_t* v, const uint64_t* w, float& pa, float& pb) {
  uint64_t a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const uint64_t xa = pack2(relu_scaled_fma_pipe(__uint_as_float(v[4 * m])),
                              relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 1])));
    const uint64_t xb = pack2(relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 2])),
                              relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 3])));
    if (m & 1) {
      ffma2(a1, xa, w[m]);
      ffma2(b1, xb, w[m]);
    } else {
      ffma2(a0, xa, w[m]);
      ffma2(b0, xb, w[m]);
    }
  }
  const float2 x0 = unpack2(a0), x1 = unpack2(a1), y0 = unpack2(b0), y1 = unpack2(b1);
  pa = (x0.x + x0.y) + (x1.x + x1.y);
  pb = (y0.x + y0.y) + (y1.x + y1.y);
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
  const uint32_t tk_bar = bar0 + 8u * (N_BARS - 1);  // TopK gathers

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
    mbar_init(tk_bar, 1);
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
        const uint64_t qdesc = sw128_kmajor_desc(sbase + OFF_Q + qs * Q_SLOT_BYTES);
        for (int t = un.t0; t < un.t1; ++t, ++kit, ++ait) {
          const int st = kit % STAGES;
          if (!(ok = mbar_wait(key_full(st), (kit / STAGES) & 1, abort_flag, status))) break;
          const int ab = ait % ACC_BUFS;
          if (!(ok = mbar_wait(acc_empty(ab), ((ait / ACC_BUFS) & 1) ^ 1, abort_flag, status))) break;
          tc_fence_after();
          const uint64_t kdesc = sw128_kmajor_desc(sbase + OFF_KEYS + st * KEY_STAGE_BYTES);
          const uint32_t d = tmem_base + ab * ACC_COLS;
          // advancing K by 32 bytes = 2 in the descriptor's 16-byte address units
#pragma unroll
          for (int k = 0; k < D / 32; ++k) mma_e4m3(d, kdesc + 2 * k, qdesc + 2 * k, idesc, k > 0);
          mma_commit(key_empty(st));
          mma_commit(acc_full(ab));
        }
        if (ok) mma_commit(q_empty(qs));
      }
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------- TopK warps --
    // Group g is selected by CTA g % (CTAs that have work), balanced whatever
    // the unit counts; groups come up in unit order, the order in which they
    // complete.
    if (filter) {
      const int running = min((int)gridDim.x, total);
      const int tid = threadIdx.x - 64;
      int* hist = (int*)(smem + OFF_HIST);
      uint32_t* gkey = (uint32_t*)(smem + OFF_TKEY);
      int32_t* gidx = (int32_t*)(smem + OFF_TIDX);
      const int K = p.K;
      bool ok = true;
      uint32_t tk_phase = 0;
      for (int g = blockIdx.x; g < n_groups && ok; g += running) {
        const int us = __ldg(&p.unit_start[g]), ue = __ldg(&p.unit_start[g + 1]);
        if (ue == us) continue;
        // wait (bounded, with back-off) until every warpgroup of every unit published
        if (tid == 0) {
          const int want = (ue - us) * EPI_WGS;
          const uint64_t t0 = globaltimer_ns();
          uint32_t ns = 64;
          while (ld_acquire(&p.group_done[g]) < want) {
            if (*abort_flag) {
              ok = false;
              break;
            }
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
              *abort_flag = 1;
              atomicOr(status, ST_TIMEOUT);
              ok = false;
              break;
            }
            __nanosleep(ns);
            ns = min(ns * 2, 4096u);
          }
          misc->gather_n = ok ? 1 : 0;
        }
        __syncwarp();
        named_bar_sync(2, TOPK_THREADS);
        ok = ((volatile Misc*)misc)->gather_n != 0;
        if (!ok) break;
        const Group G = p.groups[g];
        const int nu = ue - us;
        for (int r = 0; r < G.nrows; ++r) {
          const int row = G.row[r];
          const int32_t* cnt = p.unit_count + (int64_t)row * p.max_units;
          // certificate: every unit kept all its candidates, K <= n; the
          // regions are gathered at 16-byte aligned offsets (4 keys)
          int n = 0, npad = 0;
          bool lost = false;
          for (int c = 0; c < nu; ++c) {
            const int x = __ldcg(&cnt[c]);
            lost |= x > UCAP;
            n += min(x, UCAP);
            npad += (min(x, UCAP) + 3) & ~3;
          }
          if (n < K || lost || npad > CAND_CAP) {
            if (tid == 0) {
              const int f = atomicAdd(&p.stats->fail_count, 1);
              p.failed_rows[f] = row;
              atomicAdd(n < K ? &p.stats->underflow : &p.stats->overflow, 1);
            }
            __syncwarp();
            continue;
          }
          const uint32_t* ck = p.cand_key + (int64_t)row * p.cand_stride;
          const int32_t* ci = p.cand_idx + (int64_t)row * p.cand_stride;
          if (tid == 0) {
            // the regions were written by other CTAs (published with
            // release / acquire); the copy engine reads them after this fence
            fence_proxy_async_global();
            mbar_arrive_expect_tx(tk_bar, 2u * npad * 4u);
            int off = 0;
            for (int c = 0; c < nu; ++c) {
              const int x4 = (__ldcg(&cnt[c]) + 3) & ~3;
              if (x4) {
                bulk_g2s(smem_u32(gkey + off), ck + c * UCAP, x4 * 4, tk_bar);
                bulk_g2s(smem_u32(gidx + off), ci + c * UCAP, x4 * 4, tk_bar);
              }
              off += x4;
            }
            misc->gather_n = mbar_wait(tk_bar, tk_phase & 1, abort_flag, status) ? 1 : 0;
            misc->emit_cnt[0] = 0;
            misc->emit_cnt[1] = 0;
            atomicAdd(&p.stats->cand_total, n);
          }
          ++tk_phase;
          __syncwarp();
          named_bar_sync(2, TOPK_THREADS);
          if (!((volatile Misc*)misc)->gather_n) {
            ok = false;
            break;
          }
          // key 0 in the pad slots (they may hold stale entries of the regions)
          for (int cu = tid; cu < nu; cu += TOPK_THREADS) {
            int off = 0;
            for (int c = 0; c < cu; ++c) off += (__ldcg(&cnt[c]) + 3) & ~3;
            const int x = __ldcg(&cnt[cu]);
            for (int j = x; j < ((x + 3) & ~3); ++j) gkey[off + j] = 0u;
          }
          named_bar_sync(2, TOPK_THREADS);
          uint32_t theta;
          int rr;
          group_radix_select4(gkey, npad >> 2, K, hist, misc->sdig, tid, TOPK_THREADS, 2, theta, rr);
          group_emit4(gkey, gidx, npad >> 2, theta, rr, K, p.out + (int64_t)row * K, misc->emit_cnt, tid,
                      TOPK_THREADS);
          named_bar_sync(2, TOPK_THREADS);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int r = (warp - 4) >> 2;       // row of the group this warpgroup handles
    const int quarter = warp & 3;        // TMEM lane quarter of this warp
    const int ltid = threadIdx.x & 127;  // thread within the warpgroup
    const int bar_wg = 3 + r;            // named barrier of this warpgroup
    // after the reduce-scatter this thread owns key (lane / 4) + 8 (lane % 4)
    // of its warp's 32 TMEM lanes
    const int kt = quarter * 32 + (lane >> 2) + 8 * (lane & 3);
    const float* sc_base = (const float*)(smem + OFF_SC);
    uint32_t ait = 0, kit = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++ui) {
      Group G;
      const Unit un = decode_unit(p, n_groups, u, G);
      const bool active = r < G.nrows;
      const int row = active ? G.row[r] : 0;
      int rb = 0, re = 0;
      uint32_t tau = 0;
      float* srow = nullptr;
      int64_t store_lim = 0;
      uint32_t* ck = p.cand_key + (int64_t)row * p.cand_stride + un.c * UCAP;
      int32_t* ci = p.cand_idx + (int64_t)row * p.cand_stride + un.c * UCAP;
      // this thread's 16 weights: heads 8m + 2 (lane % 4) + {0, 1}, q scale
      // folded in, pre-scaled for the FMA-pipe ReLU
      uint64_t w2[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) w2[m] = 0;
      if (active) {
        const float qsc = __ldg(&p.q_scale[row]) * RELU_SAT_WEIGHT_SCALE;
        const float* wr = p.w + (int64_t)row * H + 2 * (lane & 3);
#pragma unroll
        for (int m = 0; m < 8; ++m) w2[m] = pack2(__ldg(&wr[8 * m]) * qsc, __ldg(&wr[8 * m + 1]) * qsc);
        rb = __ldg(&p.rb[row]);
        re = __ldg(&p.re[row]);
        if (filter) {
          tau = __ldg(&p.tau[row]);
        } else {
          srow = p.scores + (int64_t)G.slot[r] * p.ld;
          store_lim = min((int64_t)p.rs.N, p.ld);
        }
      }
      if (filter) {
        named_bar_sync(bar_wg, 128);  // the previous unit's count has been read
        if (ltid == 0) misc->ucnt[r] = 0;
        __syncwarp();
        named_bar_sync(bar_wg, 128);
      }
      for (int t = un.t0; t < un.t1 && ok; ++t, ++ait, ++kit) {
        const int ab = ait % ACC_BUFS;
        if (!(ok = mbar_wait_warp(acc_full(ab), (ait / ACC_BUFS) & 1, abort_flag, status))) break;
        const int ss = kit % SC_STAGES;
        if (!(ok = mbar_wait_warp(sc_full(ss), (kit / SC_STAGES) & 1, abort_flag, status))) break;
        tc_fence_after();
        float part[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
          const uint32_t col = tmem_base + ab * ACC_COLS + r * H;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[32];
            tmem_ld16x256b_x8(col + ((uint32_t)(quarter * 32 + 16 * hh) << 16), v);
            tmem_wait_ld();
            two_key_partials(v, w2, part[2 * hh], part[2 * hh + 1]);
          }
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
        // reduce-scatter over the 4 lanes sharing keys: part[j] covers key
        // (lane / 4) + 8 j; lane keeps key j = lane % 4
        const bool hi2 = lane & 2, hi1 = lane & 1;
        float k0 = hi2 ? part[2] : part[0], k1 = hi2 ? part[3] : part[1];
        k0 += __shfl_xor_sync(0xffffffffu, hi2 ? part[0] : part[2], 2);
        k1 += __shfl_xor_sync(0xffffffffu, hi2 ? part[1] : part[3], 2);
        float sum = hi1 ? k1 : k0;
        sum += __shfl_xor_sync(0xffffffffu, hi1 ? k0 : k1, 1);
        const float score = sum * ks;
        const int s = t * TILE + kt;
        const bool valid = (s >= rb) && (s < re);
        if (!filter) {
          if (s < store_lim) srow[s] = valid ? score : -__int_as_float(0x7f800000);
          continue;
        }
        const uint32_t key = ordered_key(score);
        const bool pred = valid && (key >= tau);
        const uint32_t m = __ballot_sync(0xffffffffu, pred);
        if (!m) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(&misc->ucnt[r], __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(m & lanemask_lt());
        if (pred && pos < UCAP) {
          ck[pos] = key;
          ci[pos] = p.rs.paged ? page * PAGE + (s & (PAGE - 1)) : s;
        }
      }
      if (filter) {
        // unit done: store the row's count, publish (release) to the TopK
        // warps; the barrier orders the warpgroup's candidate stores before
        // the releasing thread's fence.  It runs even after a failed wait, so
        // every warp of the warpgroup passes the same barriers.
        named_bar_sync(bar_wg, 128);
        if (ltid == 0 && ok) {
          if (active) p.unit_count[(int64_t)row * p.max_units + un.c] = min(misc->ucnt[r], UCAP + 1);
          __threadfence();
          red_release_add(&p.group_done[un.g], 1);
        }
        __syncwarp();
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
