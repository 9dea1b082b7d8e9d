// score_kernel.cu -- persistent, warp-specialised tcgen05 scorer.
//
// One CTA per SM walks a static share of the work units of a plan built on
// the device (a unit is a query-row pair with a range of 128-key tiles: the
// whole pair in MODE_FILTER_SLOTS, a chunk otherwise).  Roles:
//   warp 0       TMA producer: q rows of the pair, key tiles (128 keys x 128 B,
//                128-byte swizzle) into a STAGES-deep ring, key scales into a
//                separate SC_STAGES ring;
//   warp 1       MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4
//                (M = 128 keys, N = 64 heads x rows, K = 32) per tile into one
//                of ACC_BUFS TMEM accumulators; owns the TMEM allocation;
//   warps 2-3    TopK warps (MODE_FILTER_SLOTS): exact selection of the pair
//                the epilogue finished, from a shared-memory slot;
//   warps 4-19   four epilogue warpgroups; warpgroup e handles row (e & 1) of
//                the pair on tiles of parity (e >> 1), one thread per key
//                (= TMEM lane), 64 heads per thread:
//                score = k_scale * sum_j (w_j q_scale) ReLU(D_j).
//                MODE_STORE writes the fp32 score.  MODE_FILTER_SLOTS appends
//                the key (order-preserving uint32 of the score) to the row's
//                shared slot and its index to global memory when the key
//                reaches the row's sampled threshold; two slots alternate
//                between consecutive pairs (ready / free mbarriers), so the
//                TopK warps select pair i while the epilogue fills pair i + 1.
//                MODE_FILTER_GLOBAL stages (key, index) per warpgroup and
//                flushes them to the row's global buffer at the end of a
//                chunk.
//
// The method (candidate filter against a sampled threshold, radix select, the
// certificate, ready/free double buffering between scoring and selection)
// follows "Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2",
// sections 3.2 and 4; the tile shapes, TMEM accumulators, split FMA/ALU ReLU
// and the split-chunk mode are this GB300 design.
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
constexpr uint32_t OFF_WQ = OFF_SC + SC_STAGES * SC_STAGE_BYTES;
constexpr uint32_t OFF_HIST = OFF_WQ + EPI_WGS * H * 4;
constexpr uint32_t OFF_CMP = OFF_HIST + 256 * 4;
constexpr uint32_t OFF_CAND = OFF_CMP + TOPK_CMP_CAP * 4;
// candidate area: slots [2][GROUP_ROWS][SLOT_CAP] keys (MODE_FILTER_SLOTS) or
// staging keys [EPI_WGS][STG_CAP] + indices [EPI_WGS][STG_CAP] (MODE_FILTER_GLOBAL)
constexpr uint32_t SLOTS_BYTES = 2 * GROUP_ROWS * SLOT_CAP * 4;
constexpr uint32_t STAGING_BYTES = 2 * EPI_WGS * STG_CAP * 4;
constexpr uint32_t CAND_BYTES = SLOTS_BYTES > STAGING_BYTES ? SLOTS_BYTES : STAGING_BYTES;
constexpr uint32_t OFF_BAR = OFF_CAND + CAND_BYTES;
constexpr int N_BARS = 2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + 4;
constexpr uint32_t OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr uint32_t MISC_BYTES = 256;
constexpr uint32_t SMEM_USED = OFF_MISC + MISC_BYTES;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_KEYS % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(OFF_WQ % 16 == 0, "weights are read 16 bytes at a time");
static_assert(SLOT_CAP <= CAND_CAP, "slot positions index the global index buffer");

struct Misc {
  uint32_t tmem_base;
  int abort_flag;
  int sc_page[SC_STAGES][2];
  int sdig[4];
  int emit_cnt[2];
  int tk_ok;
  int slot_n[2][GROUP_ROWS];
  int stg_n[EPI_WGS];
  int stg_base[EPI_WGS];
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
  un.t1 = (int)min((int64_t)un.t0 + p.chunk_tiles, (int64_t)hi_t);
  return un;
}

// Heads whose ReLU runs on the ALU pipe (max) rather than the FMA pipe
// (saturating multiply): ALU8 of every 8 heads.
template <int ALU8>
__device__ __forceinline__ constexpr bool alu_head(int j) {
  return (j & 7) < ALU8;
}

// sum_j wq[j] * ReLU(x[j]) over 32 heads starting at head h0; wq in shared
// memory at wq_addr (weights of FMA-pipe heads pre-scaled by 2^25).
template <int ALU8>
__device__ __forceinline__ void head_block(const uint32_t* v, uint32_t wq_addr, int h0, uint64_t (&acc)[4]) {
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    uint64_t w01, w23;
    lds_2x64(wq_addr + (h0 + j) * 4, w01, w23);
    float x[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float d = __uint_as_float(v[j + c]);
      x[c] = alu_head<ALU8>(h0 + j + c) ? fmaxf(d, 0.f) : relu_scaled_fma_pipe(d);
    }
    ffma2(acc[(j >> 2) & 3], pack2(x[0], x[1]), w01);
    ffma2(acc[((j >> 2) + 2) & 3], pack2(x[2], x[3]), w23);
  }
}

}  // namespace

template <int ALU8>
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
  auto slot_ready = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + i); };
  auto slot_free = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 * SC_STAGES + 4 + 2 * ACC_BUFS + 2 + i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &misc->abort_flag;
  int* status = &p.stats->status;
  const bool slots_mode = (p.mode == MODE_FILTER_SLOTS);
  const bool global_mode = (p.mode == MODE_FILTER_GLOBAL);

  if (threadIdx.x == 0) {
    misc->abort_flag = 0;
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(key_full(i), 1);
      mbar_init(key_empty(i), 1);
    }
    for (int i = 0; i < SC_STAGES; ++i) {
      mbar_init(sc_full(i), 1);
      mbar_init(sc_empty(i), 8);  // the 8 warps of the two warpgroups reading a tile
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), 1);
      mbar_init(slot_ready(i), EPI_THREADS / 32);
      mbar_init(slot_free(i), 1);
      misc->slot_n[i][0] = 0;
      misc->slot_n[i][1] = 0;
    }
    for (int i = 0; i < ACC_BUFS; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(acc_empty(i), 8);
    }
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
    if (slots_mode) {
      const int tid = threadIdx.x - 64;
      int* hist = (int*)(smem + OFF_HIST);
      uint32_t* cmp = (uint32_t*)(smem + OFF_CMP);
      const int K = p.K;
      uint32_t ui = 0;
      for (int u = blockIdx.x; u < total; u += gridDim.x, ++ui) {
        const int slot = ui & 1;
        // one thread waits (bounded) for the epilogue to fill the slot
        if (tid == 0) misc->tk_ok = mbar_wait(slot_ready(slot), (ui >> 1) & 1, abort_flag, status) ? 1 : 0;
        __syncwarp();
        named_bar_sync(2, TOPK_THREADS);
        if (!((volatile Misc*)misc)->tk_ok) break;
        Group G;
        decode_unit(p, n_groups, u, G);
        for (int r = 0; r < G.nrows; ++r) {
          const int row = G.row[r];
          const int n = ((volatile Misc*)misc)->slot_n[slot][r];
          if (n < K || n > SLOT_CAP) {
            // certificate failed: fewer than K candidates, or some were lost
            if (tid == 0) {
              const int f = atomicAdd(&p.stats->fail_count, 1);
              p.failed_rows[f] = row;
              atomicAdd(n < K ? &p.stats->underflow : &p.stats->overflow, 1);
            }
            __syncwarp();
            continue;
          }
          const uint32_t* skey = (const uint32_t*)(smem + OFF_CAND) + (slot * GROUP_ROWS + r) * SLOT_CAP;
          const int32_t* ci = p.cand_idx + (int64_t)row * CAND_CAP;
          if (tid == 0) {
            misc->emit_cnt[0] = 0;
            misc->emit_cnt[1] = 0;
            atomicAdd(&p.stats->cand_total, n);
          }
          __syncwarp();
          named_bar_sync(2, TOPK_THREADS);
          uint32_t theta;
          int rr;
          group_radix_select([&](int i) { return skey[i]; }, n, K, hist, misc->sdig, tid, TOPK_THREADS, 2, theta,
                             rr, cmp, TOPK_CMP_CAP);
          group_emit([&](int i) { return skey[i]; }, [&](int i) { return __ldcg(&ci[i]); }, n, theta, rr, K,
                     p.out + (int64_t)row * K, misc->emit_cnt, tid, TOPK_THREADS);
          named_bar_sync(2, TOPK_THREADS);
        }
        // hand the slot back to the epilogue
        named_bar_sync(2, TOPK_THREADS);
        if (tid == 0) {
          misc->slot_n[slot][0] = 0;
          misc->slot_n[slot][1] = 0;
          mbar_arrive(slot_free(slot));
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int e = (warp - 4) >> 2;       // epilogue warpgroup 0..3
    const int r = e & 1;                 // row slot of the pair
    const uint32_t par = e >> 1;         // tile parity handled
    const int quarter = warp & 3;        // TMEM lane quarter of this warp
    const int ltid = threadIdx.x & 127;  // thread within the warpgroup
    const int bar_wg = 3 + e;            // named barrier of this warpgroup
    const float* sc_base = (const float*)(smem + OFF_SC);
    float* wq_s = (float*)(smem + OFF_WQ) + e * H;
    const uint32_t wq_addr = smem_u32(wq_s);
    uint32_t* stg_key = (uint32_t*)(smem + OFF_CAND) + e * STG_CAP;
    int32_t* stg_idx = (int32_t*)(smem + OFF_CAND) + (EPI_WGS + e) * STG_CAP;
    uint32_t ait = 0, kit = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++ui) {
      Group G;
      const Unit un = decode_unit(p, n_groups, u, G);
      const bool active = r < G.nrows;
      const int row = active ? G.row[r] : 0;
      const int slot = ui & 1;
      int rb = 0, re = 0;
      uint32_t tau = 0;
      float* srow = nullptr;
      int64_t store_lim = 0;
      uint32_t* skey = (uint32_t*)(smem + OFF_CAND) + (slot * GROUP_ROWS + r) * SLOT_CAP;
      int* scount = &misc->slot_n[slot][r];
      int32_t* gidx = p.cand_idx + (int64_t)row * CAND_CAP;
      // unit start: this warpgroup's weights (q scale folded in) and staging
      named_bar_sync(bar_wg, 128);
      if (active) {
        if (ltid < H) {
          const float wv = __ldg(&p.w[(int64_t)row * H + ltid]) * __ldg(&p.q_scale[row]);
          wq_s[ltid] = alu_head<ALU8>(ltid) ? wv : wv * RELU_SAT_WEIGHT_SCALE;
        }
        rb = __ldg(&p.rb[row]);
        re = __ldg(&p.re[row]);
        if (p.mode != MODE_STORE) {
          tau = __ldg(&p.tau[row]);
        } else {
          srow = p.scores + (int64_t)G.slot[r] * p.ld;
          store_lim = min((int64_t)p.rs.N, p.ld);
        }
      }
      if (ltid == 0) misc->stg_n[e] = 0;
      __syncwarp();
      named_bar_sync(bar_wg, 128);
      // the TopK warps must have released this unit's candidate slot
      if (slots_mode && ok) ok = mbar_wait_warp(slot_free(slot), ((ui >> 1) & 1) ^ 1, abort_flag, status);
      for (int t = un.t0; t < un.t1; ++t, ++ait, ++kit) {
        if ((ait & 1) != par || !ok) continue;  // the other parity's warpgroups take this tile
        const int ab = ait % ACC_BUFS;
        if (!(ok = mbar_wait_warp(acc_full(ab), (ait / ACC_BUFS) & 1, abort_flag, status))) continue;
        const int ss = kit % SC_STAGES;
        if (!(ok = mbar_wait_warp(sc_full(ss), (kit / SC_STAGES) & 1, abort_flag, status))) continue;
        tc_fence_after();
        const int kt = quarter * 32 + lane;  // key within the tile = TMEM lane
        uint64_t acc[4] = {0, 0, 0, 0};
        if (active) {
          const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32) << 16) + ab * ACC_COLS + r * H;
          uint32_t v[32];
          tmem_ld32(ta, v);
          tmem_wait_ld();
          head_block<ALU8>(v, wq_addr, 0, acc);
          tmem_ld32(ta + 32, v);
          tmem_wait_ld();
          head_block<ALU8>(v, wq_addr, 32, acc);
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
        const float2 a01 = unpack2(acc[0]), a23 = unpack2(acc[1]), a45 = unpack2(acc[2]), a67 = unpack2(acc[3]);
        const float score = (((a01.x + a01.y) + (a23.x + a23.y)) + ((a45.x + a45.y) + (a67.x + a67.y))) * ks;
        const int s = t * TILE + kt;
        const bool valid = (s >= rb) && (s < re);
        if (p.mode == MODE_STORE) {
          if (s < store_lim) srow[s] = valid ? score : -__int_as_float(0x7f800000);
          continue;
        }
        const uint32_t key = ordered_key(score);
        const bool pred = valid && (key >= tau);
        const uint32_t m = __ballot_sync(0xffffffffu, pred);
        if (!m) continue;
        const int32_t id = p.rs.paged ? page * PAGE + (s & (PAGE - 1)) : s;
        int base = 0;
        if (slots_mode) {
          // key to the shared slot, index straight to global memory
          if (lane == 0) base = atomicAdd(scount, __popc(m));
          base = __shfl_sync(0xffffffffu, base, 0);
          const int pos = base + __popc(m & lanemask_lt());
          if (pred && pos < SLOT_CAP) {
            skey[pos] = key;
            gidx[pos] = id;
          }
          continue;
        }
        // split mode: stage in shared memory, overflow straight to global
        if (lane == 0) base = atomicAdd(&misc->stg_n[e], __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(m & lanemask_lt());
        if (pred && pos < STG_CAP) {
          stg_key[pos] = key;
          stg_idx[pos] = id;
        }
        const uint32_t mo = __ballot_sync(0xffffffffu, pred && pos >= STG_CAP);
        if (mo) {
          int gb = 0;
          if (lane == 0) gb = atomicAdd(&p.cand_count[row], __popc(mo));
          gb = __shfl_sync(0xffffffffu, gb, 0);
          if (pred && pos >= STG_CAP) {
            const int gp = gb + __popc(mo & lanemask_lt());
            if (gp < CAND_CAP) {
              p.cand_key[(int64_t)row * CAND_CAP + gp] = key;
              p.cand_idx[(int64_t)row * CAND_CAP + gp] = id;
            }
          }
        }
      }
      if (slots_mode) {
        // pair done: the slot goes to the TopK warps (release at CTA scope
        // also covers the indices written to global memory)
        __syncwarp();
        if (lane == 0) mbar_arrive(slot_ready(slot));
      } else if (global_mode) {
        // chunk done: reserve room in the row's global buffer once, copy
        named_bar_sync(bar_wg, 128);
        if (active && ltid == 0) {
          const int n = min(misc->stg_n[e], STG_CAP);
          misc->stg_base[e] = n ? atomicAdd(&p.cand_count[row], n) : 0;
          misc->stg_n[e] = n;
        }
        __syncwarp();
        named_bar_sync(bar_wg, 128);
        if (active) {
          const int n = misc->stg_n[e], gb = misc->stg_base[e];
          uint32_t* ck = p.cand_key + (int64_t)row * CAND_CAP;
          int32_t* ci = p.cand_idx + (int64_t)row * CAND_CAP;
          for (int i = ltid; i < n && gb + i < CAND_CAP; i += 128) {
            ck[gb + i] = stg_key[i];
            ci[gb + i] = stg_idx[i];
          }
        }
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

template <int ALU8>
static cudaError_t launch_variant(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_ks,
                                  const ScoreParams& p, int grid, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(score_kernel<ALU8>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  score_kernel<ALU8><<<grid, SCORE_THREADS, SMEM_BYTES, s>>>(tm_q, tm_k, tm_ks, p);
  return cudaGetLastError();
}

cudaError_t launch_score(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_ks,
                         const ScoreParams& p, int grid, cudaStream_t s) {
  switch (p.relu_alu8) {
    case 0:
      return launch_variant<0>(tm_q, tm_k, tm_ks, p, grid, s);
    case 2:
      return launch_variant<2>(tm_q, tm_k, tm_ks, p, grid, s);
    case 4:
      return launch_variant<4>(tm_q, tm_k, tm_ks, p, grid, s);
    default:
      return launch_variant<8>(tm_q, tm_k, tm_ks, p, grid, s);
  }
}

}  // namespace dsa
