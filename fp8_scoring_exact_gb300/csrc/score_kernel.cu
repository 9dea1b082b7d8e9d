// score_kernel.cu -- persistent, warp-specialised tcgen05 scorer.
//
// One CTA per SM takes work units of a plan built on the device from a
// counter the plan resets (a CTA that finishes a unit early takes the next
// one, so uneven unit sizes leave no tail of unequal static shares;
// measured 2-4% faster than a static round-robin share): a unit is a group
// of up to 4 query rows (which stream the same keys) with a chunk of 128-key
// tiles.
// Roles:
//   warp 0       TMA producer: q rows of the group (64 heads x 128 B each)
//                and, beside them, the unit's descriptor and its rows'
//                weights, q scales, ranges and thresholds (cp.async), so the
//                MMA and epilogue warps start a unit from shared memory
//                instead of a binary search and a chain of global loads;
//                key tiles (128 keys x 128 B, 128-byte swizzle) into a
//                STAGES-deep ring; paged keys: also each tile's 128 key
//                scales and two page ids into the same stage (the
//                block-table entry and the scale behind it are two dependent
//                reads that mostly miss L2), and the stage is then released
//                by the MMA and by every epilogue warp;
//   warp 1       MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 per
//                tile, M = 128 keys, N = 64 heads x rows (256 for 4 rows),
//                K = 32, fp32 accumulators in one of two 256-column TMEM
//                buffers; owns the TMEM allocation;
//   warps 2-17   epilogue: warps 2 + 4r .. 5 + 4r handle row r of the group,
//                warp w the TMEM lane quarter w % 4.  A paged group of at
//                most two rows splits them into two teams (rows 0-1 and rows
//                2-3 of the warps) that take alternate tiles, one
//                accumulator buffer each, so no warp idles (decode batches
//                have one or two rows per sequence; dense groups keep the
//                plain loop, whose issue slots the extra test would cost).  Each thread reads two
//                keys x 16 heads per TMEM load (16x256b shape), keeps the 16
//                weights w * q_scale in registers, applies ReLU and the
//                weights with packed f32x2 FMAs, and a three-shuffle
//                reduce-scatter over 4 lanes leaves one key's 64-head sum per
//                thread; then score = sum * k_scale, the key scale loaded from
//                global memory at the top of the tile's iteration (dense: the
//                scales are contiguous and stay in L2) or read from the key
//                stage (paged).
//                MODE_STORE writes the fp32 score.  MODE_FILTER keeps the
//                scores that reach the row's sampled threshold: key
//                (order-preserving uint32) and index go to the warp's region
//                of the row's candidate buffers, counted in a register; the
//                count is stored at the end of the unit.
//
// The method (candidate filter against a sampled threshold, then an exact
// selection with a certificate) follows "Fusing Indexer Scoring and Exact
// Top-k for DeepSeek-V3.2", sections 3.2 and 4.  The selection itself runs in
// the candidate selector after this kernel (select_kernels.cu): selecting
// inside this kernel, overlapped with scoring, was measured slower on GB300,
// where the epilogue's issue slots and its latency chain with the MMA are the
// bound and any extra warp work lengthens it.
#include "common.cuh"
#include "kernels.h"
#include "rows.cuh"

namespace dsa {

namespace {

constexpr int KEY_STAGE_BYTES = TILE * D;            // 16384
constexpr int Q_ROW_BYTES = H * D;                   // 8192
constexpr int Q_SLOT_BYTES = GROUP_ROWS * Q_ROW_BYTES;  // 32768

// Key scales in shared memory: paged keys, one block of the tile's 128
// scales (two pages of 64) per key stage, beside its two page ids; dense
// keys, a ring of SCALE_RING blocks indexed by the tile count.  A dense
// block needs no barrier of its own: it lands with the stage's keys (same
// barrier), and the producer runs at most STAGES + ACC_BUFS - 1 = 7 tiles
// ahead of the slowest epilogue warp, which reads the scales of a tile
// before it releases that tile's accumulator, so a block is not refilled
// while it can still be read.
constexpr int SCALE_STAGE_BYTES = TILE * 4;
constexpr int SCALE_RING = 16;
static_assert(SCALE_RING >= STAGES + ACC_BUFS, "dense scale ring depth");

constexpr uint32_t OFF_KEYS = 0;
constexpr uint32_t OFF_Q = OFF_KEYS + STAGES * KEY_STAGE_BYTES;
constexpr uint32_t OFF_SCALE = OFF_Q + 2 * Q_SLOT_BYTES;
constexpr uint32_t OFF_PAGE = OFF_SCALE + SCALE_RING * SCALE_STAGE_BYTES;  // paged: [STAGES][2] page ids
// per q slot: the unit those q rows belong to, as the MMA and epilogue
// warps need it (producer-written)
struct UnitSlot {
  int t0, t1, c, nunits, nrows, pad[3];
  int row[GROUP_ROWS], slot[GROUP_ROWS];
  float w[GROUP_ROWS][H];  // the rows' head weights (cp.async)
  float qsc[GROUP_ROWS];   // q scales (cp.async)
  int rb[GROUP_ROWS], re[GROUP_ROWS];
  uint32_t tau[GROUP_ROWS];  // threshold keys (filter mode)
};
static_assert(sizeof(UnitSlot) % 16 == 0 && offsetof(UnitSlot, w) % 16 == 0, "unit slot layout");
constexpr uint32_t OFF_UNIT = OFF_PAGE + 128;
constexpr uint32_t OFF_BAR = OFF_UNIT + 2 * sizeof(UnitSlot);
constexpr int N_BARS = 2 * STAGES + 4 + 2 * ACC_BUFS + 1;  // + the MMA's drain barrier (abort path)
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr uint32_t MISC_BYTES = 64;
constexpr uint32_t SMEM_USED = OFF_MISC + MISC_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_KEYS % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(OFF_SCALE % 128 == 0 && SCALE_STAGE_BYTES % 128 == 0, "TMA destinations 128-byte aligned");
static_assert(STAGES * 2 * 4 <= 128, "page-id block");
static_assert(ACC_BUFS * ACC_COLS <= 512, "TMEM columns");

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
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

// One 16x256b.x4 TMEM chunk (two keys x 8 of this thread's heads: column
// blocks m0 .. m0 + 3 of the row) into the packed accumulators of the two
// keys: ReLU on the FMA pipe (saturating multiply by 2^-25, exact since
// |x| < 2^25), weights pre-scaled by 2^25, one f32x2 FMA chain per key.  The
// arithmetic is volatile asm, so it stays between the TMEM loads and waits it
// is written between (measured: letting the compiler move it is slower).
template <bool FIRST>
__device__ __forceinline__ void chunk_partials(const uint32_t* v, const uint64_t* w, uint64_t& a, uint64_t& b) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint64_t xa = pack2(relu_scaled_fma_pipe(__uint_as_float(v[4 * m])),
                              relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 1])));
    const uint64_t xb = pack2(relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 2])),
                              relu_scaled_fma_pipe(__uint_as_float(v[4 * m + 3])));
    if (FIRST && m == 0) {
      a = fmul2(xa, w[0]);
      b = fmul2(xb, w[0]);
    } else {
      ffma2(a, xa, w[m]);
      ffma2(b, xb, w[m]);
    }
  }
}
__device__ __forceinline__ float hsum2(uint64_t v) {
  const float2 x = unpack2(v);
  return x.x + x.y;
}
}  // namespace

// Compiled once per (mode, key layout): the hot loops carry no mode tests.
template <int MODE, bool PAGED>
__global__ void __launch_bounds__(SCORE_THREADS, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const ScoreParams p) {
  pdl_enter();
  const int n_groups = p.plan == PLAN_REPAIR   ? p.stats->r_groups
                       : p.plan == PLAN_SAMPLE ? p.stats->s_groups
                                               : p.stats->n_groups;
  const int total = p.plan == PLAN_REPAIR   ? p.stats->r_units
                    : p.plan == PLAN_SAMPLE ? p.stats->s_units
                                            : p.stats->total_units;
  if ((int)blockIdx.x >= total) return;  // uniform over the CTA: no work

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  Misc* misc = (Misc*)(smem + OFF_MISC);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto key_full = [&](int i) { return bar0 + 8u * i; };
  auto key_empty = [&](int i) { return bar0 + 8u * (STAGES + i); };
  auto q_full = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto q_empty = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  auto acc_full = [&](int i) { return bar0 + 8u * (2 * STAGES + 4 + i); };
  auto acc_empty = [&](int i) { return bar0 + 8u * (2 * STAGES + 4 + ACC_BUFS + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4 + 2 * ACC_BUFS);
  const float* stage_scales = (const float*)(smem + OFF_SCALE);
  UnitSlot* unit_slots = (UnitSlot*)(smem + OFF_UNIT);
  int* stage_pages = (int*)(smem + OFF_PAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t lt_mask = lanemask_lt();
  volatile int* abort_flag = &misc->abort_flag;
  int* status = &p.stats->status;
  constexpr bool filter = (MODE == MODE_FILTER);
  constexpr bool paged = PAGED;

  if (threadIdx.x == 0) {
    misc->abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(key_full(i), 1);
      // paged: the epilogue warps read the stage's scales and page ids too
      mbar_init(key_empty(i), paged ? 1 + EPI_THREADS / 32 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      // released by the MMA (last tile of the unit) and by every epilogue
      // warp (once it holds the unit's slot data in registers)
      mbar_init(q_empty(i), 1 + EPI_THREADS / 32);
    }
    for (int i = 0; i < ACC_BUFS; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(acc_empty(i), EPI_THREADS / 32);
    }
    mbar_init(drain_bar, 1);
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
  // producer: key tiles issued and q slots armed (the abort path waits for
  // the last copy of each stage and slot)
  uint32_t kit = 0, q_armed = 0;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer --
    // The whole warp runs the loop (uniform control flow); lane 0 arms the
    // barriers and issues the TMA copies.  Paged keys: the block-table
    // entries come in batches of 16 tiles, one entry per lane, and the
    // tile's 128 key scales are one cp.async of 16 bytes per lane, so the
    // tile costs two TMA issues (one per page) and no global load in this
    // warp's chain (measured: each TMA issue takes this warp 100-200 cycles,
    // and four of them per tile bounded the paged pipeline).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
    }
    const int num_pages = p.rs.num_pages;
    uint32_t ui = 0;
    bool ok = true;
    int* next_unit = &p.stats->next_unit[p.plan];
    for (; ok; ++ui) {
      // units are taken from a counter the plan reset: a CTA that finishes
      // early takes more (no static share, so no tail of uneven shares)
      int u = 0;
      if (lane == 0) u = atomicAdd(next_unit, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      const int qs = ui & 1;
      if (!(ok = mbar_wait_warp_backoff(q_empty(qs), ((ui >> 1) & 1) ^ 1, abort_flag, p.stats))) break;
      ++q_armed;
      if (u >= total) {
        // no unit left: the slot says so to the MMA and epilogue warps
        if (lane == 0) {
          unit_slots[qs].nunits = -1;
          mbar_arrive(q_full(qs));
        }
        break;
      }
      // every unit writes only its own candidate regions and count, so the
      // order they are handed out in cannot change the result (a test
      // option hands them out last first)
      if (p.reverse_units) u = total - 1 - u;
      Group G;
      const Unit un = decode_unit(p, n_groups, u, G);
      {
        // the unit's slot: row data by cp.async (4-byte weight copies when
        // the weight array is not 16-byte aligned), which q_full tracks,
        // and the descriptor by plain stores, published by the arrive below
        UnitSlot* us = unit_slots + qs;
        int rowr[GROUP_ROWS];
#pragma unroll
        for (int r = 0; r < GROUP_ROWS; ++r) rowr[r] = r < G.nrows ? G.row[r] : 0;
        // row id of a lane-dependent row index, without indexing registers
        auto row_of = [&](int r) { return r == 0 ? rowr[0] : r == 1 ? rowr[1] : r == 2 ? rowr[2] : rowr[3]; };
        const bool w16 = (reinterpret_cast<uintptr_t>(p.w) & 15u) == 0;
        if (w16) {
#pragma unroll
          for (int k = lane; k < GROUP_ROWS * H / 4; k += 32) {
            const int r = k / (H / 4), ch = k % (H / 4);
            if (r < G.nrows) cp_async_16(smem_u32(&us->w[r][4 * ch]), p.w + (int64_t)row_of(r) * H + 4 * ch, 16);
          }
        } else {
#pragma unroll
          for (int k = lane; k < GROUP_ROWS * H; k += 32) {
            const int r = k / H, h = k % H;
            if (r < G.nrows) cp_async_4(smem_u32(&us->w[r][h]), p.w + (int64_t)row_of(r) * H + h);
          }
        }
        if (lane < 4 * GROUP_ROWS) {
          const int r = lane >> 2, f = lane & 3;
          if (r < G.nrows) {
            const int row = row_of(r);
            if (f == 0) cp_async_4(smem_u32(&us->qsc[r]), p.q_scale + row);
            if (f == 1) cp_async_4(smem_u32(&us->rb[r]), p.rb + row);
            if (f == 2) cp_async_4(smem_u32(&us->re[r]), p.re + row);
            if (f == 3 && p.tau) cp_async_4(smem_u32(&us->tau[r]), p.tau + row);
          }
        }
        cp_async_mbar_arrive(q_full(qs));
        if (lane == 0) {
          us->t0 = un.t0;
          us->t1 = un.t1;
          us->c = un.c;
          us->nunits = un.nunits;
          us->nrows = G.nrows;
#pragma unroll
          for (int r = 0; r < GROUP_ROWS; ++r) {
            us->row[r] = rowr[r];
            us->slot[r] = r < G.nrows ? G.slot[r] : 0;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(q_full(qs), G.nrows * Q_ROW_BYTES);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < GROUP_ROWS; ++r)
        if (lane == r && r < G.nrows)
          tma_load_2d(sbase + OFF_Q + qs * Q_SLOT_BYTES + r * Q_ROW_BYTES, &tm_q, 0, G.row[r] * H, q_full(qs));
      const int32_t* bt = paged ? p.rs.block_table + (int64_t)G.seq * p.rs.max_pages : nullptr;
      int btv = -1;  // paged: lane j holds entry 2 tb + j of the batch starting at tile tb
      for (int t = un.t0; t < un.t1; ++t, ++kit) {
        const int st = kit % STAGES;
        if (paged && ((t - un.t0) & 15) == 0) {
          // a page id outside the cache is clamped to the first row past
          // it (TMA then reads zeros there instead of foreign memory) and
          // reported (ST_RANGE); -1: the entry is past the sequence
          const int j = 2 * t + lane;
          btv = -1;
          bool bad = false;
          if ((int64_t)j * PAGE < G.hi) {
            btv = __ldg(&bt[j]);
            bad = btv < 0 || btv >= num_pages;
            if (bad) btv = num_pages;
          }
          if (__ballot_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, ST_RANGE);
        }
        if (!(ok = mbar_wait_warp_backoff(key_empty(st), ((kit / STAGES) & 1) ^ 1, abort_flag, p.stats)))
          break;
        const uint32_t kdst = sbase + OFF_KEYS + st * KEY_STAGE_BYTES;
        if (!paged) {
          // the tile's key scales, 16 bytes per lane into ring block
          // kit % SCALE_RING (zeros past N), tracked by the stage's barrier
          const int s0 = t * TILE + 4 * lane;
          const int nb = max(0, min(16, 4 * (p.rs.N - s0)));
          cp_async_16(sbase + OFF_SCALE + (kit % SCALE_RING) * SCALE_STAGE_BYTES + lane * 16,
                      p.k_scale + (nb ? s0 : 0), nb);
          cp_async_mbar_arrive(key_full(st));
          __syncwarp();
          if (lane == 0) {
            mbar_arrive_expect_tx(key_full(st), KEY_STAGE_BYTES);
            tma_load_2d(kdst, &tm_k, 0, t * TILE, key_full(st));
          }
        } else {
          // keys, page ids and key scales of the tile in one stage (a page
          // past the sequence reads as the page past the cache: scale 0);
          // the page ids are plain stores, published by the arrive
          const int i0 = 2 * ((t - un.t0) & 15);
          const int pg0 = __shfl_sync(0xffffffffu, btv, i0);
          const int pg1 = __shfl_sync(0xffffffffu, btv, i0 + 1);
          const int pg1s = pg1 >= 0 ? pg1 : num_pages;
          // lane l copies scales 4 (l % 16) .. +3 of page l < 16 ? pg0 : pg1
          // (zeros for the page past the cache); the barrier counts the
          // copies before the arrive below can complete its phase
          const int pl = lane < 16 ? pg0 : pg1s;
          cp_async_16(sbase + OFF_SCALE + st * SCALE_STAGE_BYTES + lane * 16,
                      p.k_scale + (int64_t)min(pl, num_pages - 1) * PAGE + 4 * (lane & 15), pl < num_pages ? 16 : 0);
          cp_async_mbar_arrive(key_full(st));
          __syncwarp();
          if (lane == 0) {
            stage_pages[2 * st] = pg0;
            stage_pages[2 * st + 1] = pg1s;
            mbar_arrive_expect_tx(key_full(st), (pg1 >= 0 ? 2 : 1) * PAGE * D);
            tma_load_2d(kdst, &tm_k, 0, pg0 * PAGE, key_full(st));
            if (pg1 >= 0) tma_load_2d(kdst + PAGE * D, &tm_k, 0, pg1 * PAGE, key_full(st));
          }
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t mit = 0, ait = 0, ui = 0;
      bool ok = true;
      for (; ok; ++ui) {
        const int qs = ui & 1;
        if (!(ok = mbar_wait(q_full(qs), (ui >> 1) & 1, abort_flag, p.stats))) break;
        const UnitSlot* us = unit_slots + qs;
        if (us->nunits < 0) break;  // no unit left
        const int t0 = us->t0, t1 = us->t1;
        const uint32_t idesc = idesc_e4m3_f32(TILE, H * us->nrows);
        const uint64_t qdesc = sw128_kmajor_desc(sbase + OFF_Q + qs * Q_SLOT_BYTES);
        for (int t = t0; t < t1; ++t, ++mit, ++ait) {
          const int st = mit % STAGES;
          if (!(ok = mbar_wait(key_full(st), (mit / STAGES) & 1, abort_flag, p.stats))) break;
          const int ab = ait % ACC_BUFS;
          if (!(ok = mbar_wait(acc_empty(ab), ((ait / ACC_BUFS) & 1) ^ 1, abort_flag, p.stats))) break;
          tc_fence_after();
          const uint64_t kdesc = sw128_kmajor_desc(sbase + OFF_KEYS + st * KEY_STAGE_BYTES);
          const uint32_t d = tmem_base + ab * ACC_COLS;
          // advancing K by 32 bytes = 2 in the descriptor's 16-byte address units
#pragma unroll
          for (int k = 0; k < D / 32; ++k) mma_e4m3(d, kdesc + 2 * k, qdesc + 2 * k, idesc, k > 0);
          mma_commit(key_empty(st));
          // (test option: the first accumulator is never signalled, so the
          // epilogue's bounded wait for it runs out)
          if (!(p.withhold_first_acc && ait == 0)) mma_commit(acc_full(ab));
        }
        if (ok) mma_commit(q_empty(qs));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int r4 = (warp - 2) >> 2;  // row slot of these four warps (0-3)
    const int quarter = warp & 3;    // TMEM lane quarter of this warp
    // after the reduce-scatter this thread owns key (lane / 4) + 8 (lane % 4)
    // of its warp's 32 TMEM lanes
    const int kt = quarter * 32 + (lane >> 2) + 8 * (lane & 3);
    uint32_t ait = 0, ui = 0;
    bool ok = true;
    float checksum = 0.f;  // MODE_CONTROL
    for (; ok; ++ui) {
      // the unit as the producer staged it beside its q rows; the slot is
      // released as soon as this warp holds what it needs in registers
      const int qs = ui & 1;
      if (!(ok = mbar_wait_warp(q_full(qs), (ui >> 1) & 1, abort_flag, p.stats))) break;
      const UnitSlot* us = unit_slots + qs;
      if (us->nunits < 0) break;  // no unit left
      const int t0 = us->t0, t1 = us->t1, nrows = us->nrows;
      // two teams for a paged group of at most two rows: team t handles the
      // tiles of accumulator buffer t, and its candidate regions are those
      // of the virtual unit 2 c + t; a warp's arrivals then count for its
      // idle twin of the other team as well
      const bool split = paged && nrows <= 2;
      const int team = split ? (r4 >> 1) : 0;
      const int r = split ? (r4 & 1) : r4;
      const int vunits = split ? 2 * us->nunits : us->nunits;
      const int vc = split ? 2 * us->c + team : us->c;
      const uint32_t arrivals = split ? 2u : 1u;
      const bool active = r < nrows;
      const int row = active ? us->row[r] : 0;
      int rb = 0, re = 0;
      float tauf = 0.f;
      float* srow = nullptr;
      int64_t store_lim = 0;
      // this warp's candidate region of the unit
      const int wcap = region_cap(vunits);
      const int64_t region = (int64_t)row * ROW_SLOTS + (int64_t)(vc * UNIT_REGIONS + quarter) * wcap;
      uint32_t* ck = p.cand_key + region;
      int32_t* ci = p.cand_idx + region;
      int wcnt = 0;
      // this thread's 16 weights: heads 8m + 2 (lane % 4) + {0, 1}, q scale
      // folded in, pre-scaled for the FMA-pipe ReLU
      uint64_t w2[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) w2[m] = 0;
      if (active) {
        const float qsc = us->qsc[r] * RELU_SAT_WEIGHT_SCALE;
        const float* wr = &us->w[r][2 * (lane & 3)];
#pragma unroll
        for (int m = 0; m < 8; ++m) w2[m] = pack2(wr[8 * m] * qsc, wr[8 * m + 1] * qsc);
        rb = us->rb[r];
        re = us->re[r];
        if (filter) {
          tauf = key_threshold_float(us->tau[r]);
        } else {
          srow = p.scores + (int64_t)us->slot[r] * p.ld;
          store_lim = min((int64_t)p.rs.N, p.ld);
        }
      }
      __syncwarp();
      mbar_arrive_warp(q_empty(qs));
      if constexpr (MODE == MODE_CONTROL) {
        // math-only control: wait for each accumulator, fold one of its
        // columns into the checksum, release it
        for (int t = t0; t < t1 && ok; ++t, ++ait) {
          const int ab = ait & (ACC_BUFS - 1);
          if (!(ok = mbar_wait_warp(acc_full(ab), (ait / ACC_BUFS) & 1, abort_flag, p.stats))) break;
          tc_fence_after();
          const uint32_t v = tmem_ld1(tmem_base + ab * ACC_COLS + r * H + ((uint32_t)(quarter * 32) << 16));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive_warp(acc_empty(ab));
          checksum += __uint_as_float(v);
        }
        continue;
      }
      for (int t = t0; t < t1 && ok; ++t, ++ait) {
        if (split && (int)(ait & 1) != team) continue;  // the other team's tile
        // this thread's key scale, used at the end of the iteration (paged:
        // and the page holding the key, from the tile's key stage, which
        // this warp then releases with the accumulator; the stage cannot be
        // refilled before that, so its full phase is still this tile's)
        const int kst = ait % STAGES;
        float ks = 0.f;
        int page = 0;
        if constexpr (paged) {
          if (!(ok = mbar_wait_warp(key_full(kst), (ait / STAGES) & 1, abort_flag, p.stats))) break;
          ks = stage_scales[kst * TILE + kt];
          page = stage_pages[2 * kst + (kt >> 6)];
        }
        const int ab = ait & (ACC_BUFS - 1);
        if (!(ok = mbar_wait_warp(acc_full(ab), (ait / ACC_BUFS) & 1, abort_flag, p.stats))) break;
        tc_fence_after();
        // dense: the scales landed with the tile's keys, before its MMA
        if constexpr (!paged) ks = stage_scales[(ait % SCALE_RING) * TILE + kt];
        float part[4] = {0.f, 0.f, 0.f, 0.f};
        if (active) {
          // four 16x256b.x4 chunks (lanes +0 / +16 x heads 0-31 / 32-63)
          // through two register buffers: each load is in flight while the
          // previous chunk is reduced; the buffer goes back to the MMA once
          // the last chunk is in registers
          const uint32_t col = tmem_base + ab * ACC_COLS + r * H + ((uint32_t)(quarter * 32) << 16);
          uint32_t va[16], vb[16];
          uint64_t aL, bL, aH, bH;
          tmem_ld16x256b_x4(col, va);
          tmem_ld16x256b_x4(col + 32, vb);
          tmem_wait_ld();
          chunk_partials<true>(va, w2, aL, bL);
          tmem_ld16x256b_x4(col + (16u << 16), va);
          chunk_partials<false>(vb, w2 + 4, aL, bL);
          tmem_wait_ld();
          tmem_ld16x256b_x4(col + (16u << 16) + 32, vb);
          chunk_partials<true>(va, w2, aH, bH);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive_warp_n(acc_empty(ab), arrivals);
          if (paged) mbar_arrive_warp_n(key_empty(kst), arrivals);
          chunk_partials<false>(vb, w2 + 4, aH, bH);
          part[0] = hsum2(aL);
          part[1] = hsum2(bL);
          part[2] = hsum2(aH);
          part[3] = hsum2(bH);
        } else {
          tc_fence_before();
          mbar_arrive_warp_n(acc_empty(ab), arrivals);
          if (paged) mbar_arrive_warp_n(key_empty(kst), arrivals);
        }
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
        // score >= the threshold's float  <=>  its key >= the threshold key
        const bool pred = valid && score >= tauf;
        const uint32_t m = __ballot_sync(0xffffffffu, pred);
        const int pos = wcnt + __popc(m & lt_mask);
        wcnt += __popc(m);
        if (pred && pos < wcap) {
          ck[pos] = ordered_key(score);
          ci[pos] = paged ? page * PAGE + (s & (PAGE - 1)) : s;
        }
      }
      // unit done: the warp's count (wcap + 1 = some were lost)
      if (filter && active && ok && lane == 0)
        p.unit_count[(int64_t)row * p.max_units * UNIT_REGIONS + vc * UNIT_REGIONS + quarter] = min(wcnt, wcap + 1);
    }
    if constexpr (MODE == MODE_CONTROL) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) checksum += __shfl_xor_sync(0xffffffffu, checksum, o);
      if (lane == 0) atomicAdd(p.scores, checksum);
    }
  }

  __syncthreads();
  if (misc->abort_flag) {
    // a wait gave up: before the shared memory and TMEM are released, the
    // copies and MMAs already issued land.  A stage or q slot has at most
    // one copy outstanding, the last one armed on it, so waiting for that
    // phase of its barrier covers it (the TMA bytes and the cp.async
    // arrivals of the same phase); a last commit tracks every MMA issued.
    if (warp == 0) {
      cp_async_wait_all();
      if (lane == 0) {
        for (uint32_t st = 0; st < (uint32_t)STAGES; ++st)
          if (kit > st) {
            const uint32_t last = st + STAGES * ((kit - 1 - st) / STAGES);
            mbar_drain(key_full(st), (last / STAGES) & 1);
          }
        for (uint32_t qs = 0; qs < 2; ++qs)
          if (q_armed > qs) {
            const uint32_t last = qs + 2 * ((q_armed - 1 - qs) / 2);
            mbar_drain(q_full(qs), (last >> 1) & 1);
          }
      }
    } else if (warp == 1 && lane == 0) {
      mma_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, ACC_BUFS * ACC_COLS);
  }
}

template <int MODE, bool PAGED>
static cudaError_t launch_variant(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const ScoreParams& p, int grid,
                                  cudaStream_t s) {
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_attr_once(score_kernel<MODE, PAGED>, SMEM_BYTES, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(score_kernel<MODE, PAGED>, dim3(grid), dim3(SCORE_THREADS), SMEM_BYTES, s, tm_q, tm_k, p);
}

cudaError_t launch_score(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const ScoreParams& p, int grid,
                         cudaStream_t s) {
  const bool paged = p.rs.paged != 0;
  if (p.mode == MODE_CONTROL) return paged ? cudaErrorInvalidValue : launch_variant<MODE_CONTROL, false>(tm_q, tm_k, p, grid, s);
  if (p.mode == MODE_FILTER)
    return paged ? launch_variant<MODE_FILTER, true>(tm_q, tm_k, p, grid, s)
                 : launch_variant<MODE_FILTER, false>(tm_q, tm_k, p, grid, s);
  return paged ? launch_variant<MODE_STORE, true>(tm_q, tm_k, p, grid, s)
               : launch_variant<MODE_STORE, false>(tm_q, tm_k, p, grid, s);
}

}  // namespace dsa
