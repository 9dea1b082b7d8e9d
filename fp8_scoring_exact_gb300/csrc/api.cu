// api.cu -- C ABI of the indexer library (include/dsa_indexer.h): argument
// validation, per-(device, stream) scratch arena, tensor-map encoding and the
// launch sequences of the fused, paged, unfused and standalone operators.
//
// Launch sequence of the fused operator (all on the caller's stream, no host
// synchronisation; every kernel launched with programmatic dependent launch):
//   plan (ranges, 4-row groups, work units) -> sampled thresholds (dense: the
//   shared grid gathered once, scored by the scorer in store mode, one
//   threshold per row; paged and short rows: the per-pair sampling kernel)
//   -> persistent scorer in filter mode (candidates to per-row regions)
//   -> candidate selector (certificate, radix select, emission)
//   -> repair plan -> scorer in store mode over the failed rows
//   -> cluster radix select of those rows.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "dsa_indexer.h"
#include "common.cuh"
#include "kernels.h"

using namespace dsa;

namespace {

// ---------------------------------------------------------------- options --
std::mutex g_mu;
int64_t g_chunk_tiles = -1;  // -1: chosen per call (chunk_for)
int64_t g_tau_bias = 0;
int64_t g_profile = 0;
int64_t g_grid = 0;
int64_t g_target16 = 36;  // candidates aimed at, in K/16: 2.25 K (measured on GB300; the pages aim at 2 K)
int64_t g_host_chunk_rows = 0;  // 0: chosen per call (host_chunk_rows)
int64_t g_unit_order = 0;       // 1: scorer units handed out last first (test option)
int64_t g_wait_us = WAIT_LIMIT_NS / 1000;  // limit of every pipeline wait
int64_t g_withhold = 0;         // 1: the main scorer never signals its first accumulator (test option)
int64_t g_matrix_row_min = -1;  // standalone top-K: rows from which CTAs take whole rows (-1: one wave)
std::atomic<int64_t> g_launches{0};

// ----------------------------------------------------------------- arena ----
struct Layout {
  size_t stats, rb, re, tau, groups, unit_start, rgroups, runit_start, unit_count, failed;
  size_t cand_key, cand_idx, scores;
  size_t srb, sre, sgroups, sunit_start, skeys, sks, sscores;  // dense sampled thresholds
  size_t pair_cnt;                                             // split sampling tickets
  size_t total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static_assert(MAX_K == DSA_MAX_K, "kernel K cap matches the public header");
constexpr int64_t SAMPLE_LD = (MAX_SAMPLES + 2 + 3) / 4 * 4;  // sample-score row stride

// cand_stride: candidate slots per row (0: no candidate buffers); max_units:
// work units per group at most (per-row unit counts)
Layout make_layout(int64_t R, int64_t G, int64_t cand_stride, int64_t max_units, int64_t score_rows, int64_t ld) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.stats = take(sizeof(Stats));
  L.rb = take(R * 4);
  L.re = take(R * 4);
  L.tau = take(R * 4);
  L.groups = take(G * sizeof(Group));
  L.unit_start = take((G + 1) * 4);
  L.rgroups = take(R * sizeof(Group));
  L.runit_start = take((R + 1) * 4);
  L.unit_count = take((size_t)R * max_units * UNIT_REGIONS * 4);
  L.failed = take(R * 4);
  L.cand_key = take((size_t)R * cand_stride * 4);
  L.cand_idx = take((size_t)R * cand_stride * 4);
  L.scores = take((size_t)score_rows * ld * 4);
  if (cand_stride) {  // fused calls: the sample grid's key set and its scores
    L.srb = take(R * 4);
    L.sre = take(R * 4);
    L.sgroups = take(G * sizeof(Group));
    L.sunit_start = take((G + 1) * 4);
    L.skeys = take((size_t)(MAX_SAMPLES + 2) * D);
    L.sks = take((size_t)(MAX_SAMPLES + 2) * 4);
    L.sscores = take((size_t)R * SAMPLE_LD * 4);
    L.pair_cnt = take(R * 4);
  }
  L.total = off;
  return L;
}

struct Arena {
  uint8_t* base = nullptr;
  size_t cap = 0;
  Layout L{};
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  bool profiled = false;
  bool used = false;
};

std::map<std::pair<int, cudaStream_t>, Arena> g_arenas;

// Returns the arena of (current device, stream) with room for `need` bytes.
Arena* get_arena(cudaStream_t stream, const Layout& L, int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = DSA_ERR_CUDA;
    return nullptr;
  }
  Arena& a = g_arenas[{dev, stream}];
  if (a.cap < L.total) {
    if (a.base) {
      cudaDeviceSynchronize();
      cudaFree(a.base);
      a.base = nullptr;
      a.cap = 0;
    }
    const size_t want = align_up(L.total + L.total / 8, 1 << 20);
    if (cudaMalloc(&a.base, want) != cudaSuccess) {
      cudaGetLastError();
      *err = DSA_ERR_CUDA;
      return nullptr;
    }
    a.cap = want;
  }
  if (!a.ev0) {
    cudaEventCreate(&a.ev0);
    cudaEventCreate(&a.ev1);
  }
  a.L = L;
  a.used = true;
  return &a;
}

template <class T>
T* at(Arena* a, size_t off) {
  return reinterpret_cast<T*>(a->base + off);
}

// ------------------------------------------------------------ tensor maps --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// rows of 128 FP8 bytes, 128-byte swizzle, box = 128 bytes x box_rows
bool tmap_rows_u8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D};
  cuuint32_t box[2] = {(cuuint32_t)D, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

#define DSA_LAUNCH(expr)                        \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    g_launches.fetch_add(1);                    \
    if (e_ != cudaSuccess) return DSA_ERR_CUDA; \
  } while (0)

struct Opts {
  int chunk, grid, target16;
  int64_t bias;
  bool profile;
  int reverse_units;
  int withhold;
  uint64_t wait_ns;
  int64_t matrix_row_min;
};

// Tiles per work unit: the option when set, else 64 for dense rows and 32
// for paged ones (decode batches mix very short and very long sequences:
// smaller units balance the long tail), halved (down to 8) while the row
// groups would give fewer than 4 units per CTA (few rows with long
// histories: the key dimension supplies the parallelism).  Measured on
// GB300.  Never so small that a row's candidate regions (4 per unit, twice
// that for paged rows) exceed what the candidate selector reads: such rows
// would all fail their certificate and go to repair.
constexpr int REPAIR_CHUNK = 8;  // tiles per unit of the repair scorer
constexpr int SHARED_GRID_MIN_ROWS = 256;  // dense rows above this share one gathered sample grid
int min_chunk_for(const RowSpace& rs) {
  const int tiles = ceil_div(rs.N, TILE);
  const int per_unit = UNIT_REGIONS * (rs.paged ? 2 : 1);
  return ceil_div(tiles * per_unit, CAND_MAX_REGIONS);
}
int chunk_for(const Opts& o, const RowSpace& rs) {
  if (o.chunk > 0) return o.chunk;
  const int64_t tiles = (int64_t)n_groups(rs) * ceil_div(rs.N, TILE);
  int c = rs.paged ? 32 : 64;
  while (c > 8 && tiles / c < 4LL * o.grid) c >>= 1;
  return std::max(c, min_chunk_for(rs));
}

// Tiles per work unit of the selection over a stored score matrix: 256
// (fewer, longer units than the scorer's: measured 0.888 against 0.912 ms
// for the headline-size standalone top-K), halved (down to 16) while there
// would be fewer than 4 units per CTA of its filter; the option overrides
// it as above.
int matrix_chunk_for(const Opts& o, const RowSpace& rs) {
  if (o.chunk > 0) return o.chunk;
  const int64_t tiles = (int64_t)n_groups(rs) * ceil_div(rs.N, TILE);
  int c = 256;
  while (c > 16 && tiles / c < 8LL * o.grid) c >>= 1;
  return std::max(c, min_chunk_for(rs));
}

Opts read_opts() {
  std::lock_guard<std::mutex> lk(g_mu);
  Opts o;
  o.chunk = (int)g_chunk_tiles;
  o.bias = g_tau_bias;
  o.profile = g_profile != 0;
  o.target16 = (int)g_target16;
  o.reverse_units = g_unit_order != 0;
  o.withhold = g_withhold != 0;
  o.wait_ns = (uint64_t)g_wait_us * 1000ull;
  o.matrix_row_min = g_matrix_row_min;
  const int sms = sm_count();
  o.grid = g_grid > 0 ? (int)g_grid : (sms > 0 ? sms : 1);
  return o;
}

// ------------------------------------------------- shared launch sequence --
// Fused pipeline over a row space whose keys are described by tm_k.
int run_fused(const RowSpace& rs_in, int K, const CUtensorMap& tm_q, const CUtensorMap& tm_k, const uint8_t* k_raw,
              const float* ks_raw, const float* q_scale,
              const float* w, const int32_t* row_begin, const int32_t* row_end, int32_t* out, cudaStream_t stream) {
  const Opts o = read_opts();
  const int chunk = chunk_for(o, rs_in);
  const int G = n_groups(rs_in);
  const int64_t ld = align_up((size_t)rs_in.N, 4);
  // candidate-region units per row: paged, twice the work units (a group of
  // at most two rows runs two epilogue teams per unit)
  const int max_units = (rs_in.paged ? 2 : 1) * ceil_div(ceil_div(rs_in.N, TILE), chunk);
  const int64_t cand_stride = ROW_SLOTS;
  std::lock_guard<std::mutex> lk(g_mu);
  int err = DSA_OK;
  Arena* a = get_arena(stream, make_layout(rs_in.R, G, cand_stride, max_units, rs_in.R, ld), &err);
  if (!a) return err;
  const Layout& L = a->L;
  Stats* st = at<Stats>(a, L.stats);
  RowSpace rs = rs_in;
  if (rs.paged) rs.status = &st->status;

  PlanParams pp{};
  pp.rs = rs;
  pp.plan = PLAN_MAIN;
  pp.K = K;
  pp.trivial_len = K;
  pp.chunk_tiles = chunk;
  pp.row_begin_in = row_begin;
  pp.row_end_in = row_end;
  pp.rb = at<int32_t>(a, L.rb);
  pp.re = at<int32_t>(a, L.re);
  pp.groups = at<Group>(a, L.groups);
  pp.unit_start = at<int32_t>(a, L.unit_start);
  pp.failed_rows = at<int32_t>(a, L.failed);
  pp.stats = st;
  pp.wait_ns = o.wait_ns;
  pp.pair_cnt = at<int>(a, L.pair_cnt);
  pp.n_pairs = n_pairs(rs);
  DSA_LAUNCH(launch_plan(pp, stream));

  uint32_t* tau = at<uint32_t>(a, L.tau);
  const int S = sample_stride_for(rs.N);
  const int ns = rs.N > SAMPLE_OFFSET ? ceil_div(rs.N - SAMPLE_OFFSET, S) : 0;
  // dense grids of several tiles over many rows: the shared-grid chain
  // below; few rows take the per-pair kernel in split mode (two launches
  // instead of four)
  const bool shared_grid = !rs.paged && ns > TILE && rs.R > SHARED_GRID_MIN_ROWS;
  if (shared_grid) {
    // sampled thresholds: the grid keys gathered once, scored by the scorer
    // for every row, then one threshold per row (a grid of one tile or less
    // is cheaper in the per-pair sampling kernel below)
    SamplePrepParams sx{};
    sx.rs = rs;
    sx.K = K;
    sx.stride = S;
    sx.n_samples = ns;
    sx.k = k_raw;
    sx.k_scale = ks_raw;
    sx.sk = at<uint8_t>(a, L.skeys);
    sx.sks = at<float>(a, L.sks);
    sx.rb = pp.rb;
    sx.re = pp.re;
    sx.out = out;
    sx.stats = st;
    PlanParams spl = pp;
    spl.plan = PLAN_SAMPLE;
    spl.sample_stride = S;
    spl.chunk_tiles = WHOLE_PAIR_TILES;
    spl.row_begin_in = pp.rb;
    spl.row_end_in = pp.re;
    spl.rb = at<int32_t>(a, L.srb);
    spl.re = at<int32_t>(a, L.sre);
    spl.groups = at<Group>(a, L.sgroups);
    spl.unit_start = at<int32_t>(a, L.sunit_start);
    sx.plan = spl;
    DSA_LAUNCH(launch_sample_prep(sx, stream));
    {
      CUtensorMap tks;
      if (!tmap_rows_u8(&tks, sx.sk, (uint64_t)ns, TILE)) return DSA_ERR_CUDA;
      RowSpace srs = rs;
      srs.N = ns;
      ScoreParams scp{};
      scp.rs = srs;
      scp.mode = MODE_STORE;
      scp.chunk_tiles = WHOLE_PAIR_TILES;
      scp.plan = PLAN_SAMPLE;
      scp.reverse_units = o.reverse_units;
      scp.k_scale = sx.sks;
      scp.q_scale = q_scale;
      scp.w = w;
      scp.rb = spl.rb;
      scp.re = spl.re;
      scp.groups = spl.groups;
      scp.unit_start = spl.unit_start;
      scp.scores = at<float>(a, L.sscores);
      scp.ld = SAMPLE_LD;
      scp.stats = st;
      DSA_LAUNCH(launch_score(tm_q, tks, scp, o.grid, stream));
    }
    SampleTauParams tp{};
    tp.rs = rs;
    tp.K = K;
    tp.target16 = o.target16;
    tp.tau_bias = o.bias;
    tp.rb = pp.rb;
    tp.re = pp.re;
    tp.srb = spl.rb;
    tp.sre = spl.re;
    tp.sscores = at<float>(a, L.sscores);
    tp.sld = SAMPLE_LD;
    tp.tau = tau;
    tp.stats = st;
    DSA_LAUNCH(launch_sample_tau(tp, stream));
  } else {
    SampleParams sp{};
    sp.rs = rs;
    sp.K = K;
    sp.target16 = o.target16;
    sp.tau_bias = o.bias;
    sp.k = k_raw;
    sp.k_scale = ks_raw;
    sp.q_scale = q_scale;
    sp.w = w;
    sp.rb = pp.rb;
    sp.re = pp.re;
    sp.tau = tau;
    sp.out = out;
    sp.stats = st;
    // grids of several tiles (paged rows, and few dense rows over long key
    // ranges; up to 8 tiles): one CTA per (pair, tile), then one warp per
    // row selects its threshold
    sp.split = rs.paged || ns > TILE;
    sp.pair_cnt = pp.pair_cnt;
    sp.sscores = at<float>(a, L.sscores);
    sp.sld = SAMPLE_LD;
    sp.srb = at<int32_t>(a, L.srb);
    sp.sre = at<int32_t>(a, L.sre);
    DSA_LAUNCH(launch_sample(tm_q, sp, n_pairs(rs), stream));
  }

  ScoreParams cp{};
  cp.rs = rs;
  cp.mode = MODE_FILTER;
  cp.chunk_tiles = chunk;
  cp.plan = PLAN_MAIN;
  cp.reverse_units = o.reverse_units;
  cp.withhold_first_acc = o.withhold;
  cp.k_scale = ks_raw;
  cp.q_scale = q_scale;
  cp.w = w;
  cp.rb = pp.rb;
  cp.re = pp.re;
  cp.groups = pp.groups;
  cp.unit_start = pp.unit_start;
  cp.tau = tau;
  cp.cand_key = at<uint32_t>(a, L.cand_key);
  cp.cand_idx = at<int32_t>(a, L.cand_idx);
  cp.unit_count = at<int32_t>(a, L.unit_count);
  cp.max_units = max_units;
  cp.stats = st;
  a->profiled = o.profile;
  if (o.profile) cudaEventRecord(a->ev0, stream);
  DSA_LAUNCH(launch_score(tm_q, tm_k, cp, o.grid, stream));
  if (o.profile) cudaEventRecord(a->ev1, stream);

  CandParams cs{};
  cs.rs = rs;
  cs.K = K;
  cs.groups = pp.groups;
  cs.unit_start = pp.unit_start;
  cs.unit_count = cp.unit_count;
  cs.cand_key = cp.cand_key;
  cs.cand_idx = cp.cand_idx;
  cs.max_units = max_units;
  cs.failed_rows = at<int32_t>(a, L.failed);
  cs.tau = tau;
  cs.out = out;
  cs.stats = st;
  // exact repair of rows whose certificate failed: a store-mode scorer has
  // no candidate regions, so its units are short (REPAIR_CHUNK tiles) and
  // even a single failed long row is spread over many SMs; the selector's
  // last CTA writes this plan
  PlanParams rp = pp;
  rp.plan = PLAN_REPAIR;
  rp.chunk_tiles = REPAIR_CHUNK;
  rp.groups = at<Group>(a, L.rgroups);
  rp.unit_start = at<int32_t>(a, L.runit_start);
  cs.plan_repair = 1;
  cs.repair = rp;
  DSA_LAUNCH(launch_cand_select(cs, o.grid, stream));

  ScoreParams rcp = cp;
  rcp.withhold_first_acc = 0;
  rcp.chunk_tiles = REPAIR_CHUNK;
  rcp.mode = MODE_STORE;
  rcp.plan = PLAN_REPAIR;
  rcp.groups = rp.groups;
  rcp.unit_start = rp.unit_start;
  rcp.scores = at<float>(a, L.scores);
  rcp.ld = ld;
  DSA_LAUNCH(launch_score(tm_q, tm_k, rcp, o.grid, stream));

  // their exact top-K: one thread-block cluster per row
  WideParams wp{};
  wp.rs = rs;
  wp.K = K;
  wp.list = pp.failed_rows;
  wp.scores = rcp.scores;
  wp.ld = ld;
  wp.rb = pp.rb;
  wp.re = pp.re;
  wp.out = out;
  wp.stats = st;
  DSA_LAUNCH(launch_wide_select(wp, o.grid / 2 > 0 ? o.grid / 2 : 1, stream));  // 4 CTAs per SM
  return DSA_OK;
}

int check_dense(const uint8_t* q, const float* qs, const uint8_t* k, const float* ks, const float* w,
                const int32_t* rb, const int32_t* re, int Q, int N) {
  if (!q || !qs || !k || !ks || !w || !rb || !re) return DSA_ERR_ARG;
  if (Q <= 0 || N <= 0) return DSA_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(ks)) return DSA_ERR_ARG;
  if ((int64_t)Q * H >= (1ll << 31) || (int64_t)N >= (1ll << 31) - TILE) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// ------------------------------------------------- no-allocation variant --
// Scratch of dsa_indexer_topk_from_scores_noalloc: a fixed array in device
// memory that exists on every GPU that loads this library, for callers that
// must not allocate (see the declaration in the header).  The host-side name
// g_noalloc_scratch is only a stand-in for the symbol: the kernels get the
// device address that cudaGetSymbolAddress returns for the current device.
constexpr int NOALLOC_MAX_ROWS = 4096;
constexpr size_t NOALLOC_SCRATCH_BYTES = 512 * 1024;
__device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_addr;  // device -> address of g_noalloc_scratch there

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device does this lookup).
void* noalloc_scratch(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = DSA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  auto it = g_noalloc_addr.find(dev);
  if (it != g_noalloc_addr.end()) return it->second;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    *err = DSA_ERR_CUDA;
    return nullptr;
  }
  g_noalloc_addr[dev] = p;
  return p;
}

// ------------------------------------------------- sparse-attention scratch --
// Per (device, stream): the status word and the split partials of
// dsa_sparse_attention, grown on demand (growing synchronises the device).
struct AuxScratch {
  uint8_t* base = nullptr;
  size_t cap = 0;
};
std::map<std::pair<int, cudaStream_t>, AuxScratch> g_aux;  // guarded by g_mu

uint8_t* aux_scratch(cudaStream_t stream, size_t need, int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *err = DSA_ERR_CUDA;
    return nullptr;
  }
  AuxScratch& a = g_aux[{dev, stream}];
  if (a.cap < need) {
    if (a.base) {
      cudaDeviceSynchronize();
      cudaFree(a.base);
      a.base = nullptr;
      a.cap = 0;
    }
    const size_t want = align_up(need + need / 8, 1 << 20);
    if (cudaMalloc(&a.base, want) != cudaSuccess) {
      cudaGetLastError();
      *err = DSA_ERR_CUDA;
      return nullptr;
    }
    a.cap = want;
  }
  return a.base;
}

// ----------------------------------------------------- host-buffer entry --
// Device staging of dsa_indexer_topk_host per (device, stream): two row-chunk
// slots (q, q scales, weights, ranges, indices) and the keys with their
// scales.  While one chunk is scored on the caller's stream, a copy stream
// owned by the stage brings in the next chunk's rows and takes out the
// previous chunk's indices.
constexpr int HOST_MAX_CHUNKS = 64;

struct HostLayout {
  size_t q, qs, w, rb, re, out, slot;  // offsets inside a slot, slot size
  size_t k, ks, total;                 // keys and key scales after the two slots
};

HostLayout host_layout(int64_t N, int64_t C, int K) {
  HostLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.q = take((size_t)C * H * D);
  L.qs = take((size_t)C * 4);
  L.w = take((size_t)C * H * 4);
  L.rb = take((size_t)C * 4);
  L.re = take((size_t)C * 4);
  L.out = take((size_t)C * K * 4);
  L.slot = off;
  off = 2 * L.slot;
  L.k = take((size_t)N * D);
  L.ks = take((size_t)N * 4);
  L.total = off;
  return L;
}

struct HostStage {
  uint8_t* base = nullptr;
  size_t cap = 0;
  cudaStream_t copy = nullptr;
  cudaEvent_t entry = nullptr, copies_done = nullptr, in_ready[2] = {nullptr, nullptr}, done[2] = {nullptr, nullptr};
  Stats* stats_h = nullptr;  // pinned: the status block of each chunk
};

std::mutex g_host_mu;  // one host-buffer call at a time (it synchronises before returning)
std::map<std::pair<int, cudaStream_t>, HostStage> g_host;

// Rows per chunk: the option when set, else half of the rows but at least
// 2048 (every chunk pays the fused call's fixed launch sequence and its
// scorer's tail again; measured at Q = 4096 x N = 131072 from pinned host
// memory: 1 chunk 4.84 ms, 2 chunks 4.77, 4 chunks 4.88, 8 chunks 5.22);
// at most HOST_MAX_CHUNKS chunks; a multiple of the 4-row groups.
int host_chunk_rows(int Q) {
  int64_t c;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    c = g_host_chunk_rows;
  }
  if (c <= 0) c = std::max<int64_t>(2048, ((int64_t)Q + 1) / 2);
  c = std::max<int64_t>(c, ((int64_t)Q + HOST_MAX_CHUNKS - 1) / HOST_MAX_CHUNKS);
  c = (c + GROUP_ROWS - 1) / GROUP_ROWS * GROUP_ROWS;
  return (int)std::min<int64_t>(c, Q);
}

// Device address of the status block the last call on `stream` wrote.
Stats* arena_stats(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_arenas.find({dev, stream});
  if (it == g_arenas.end() || !it->second.base) return nullptr;
  return reinterpret_cast<Stats*>(it->second.base + it->second.L.stats);
}

int host_stage_init(HostStage& hs, const HostLayout& L, cudaStream_t stream) {
  if (!hs.copy) {
    // built in a local first: the stage takes it only once every part exists
    HostStage n;
    bool ok = cudaStreamCreateWithFlags(&n.copy, cudaStreamNonBlocking) == cudaSuccess;
    cudaEvent_t* evs[] = {&n.entry, &n.copies_done, &n.in_ready[0], &n.in_ready[1], &n.done[0], &n.done[1]};
    for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaMallocHost(&n.stats_h, HOST_MAX_CHUNKS * sizeof(Stats)) == cudaSuccess;
    if (!ok) {
      for (cudaEvent_t* e : evs)
        if (*e) cudaEventDestroy(*e);
      if (n.copy) cudaStreamDestroy(n.copy);
      if (n.stats_h) cudaFreeHost(n.stats_h);
      return DSA_ERR_CUDA;
    }
    n.base = hs.base;
    n.cap = hs.cap;
    hs = n;
  }
  if (hs.cap < L.total) {
    if (hs.base) {
      if (cudaStreamSynchronize(stream) != cudaSuccess || cudaStreamSynchronize(hs.copy) != cudaSuccess)
        return DSA_ERR_CUDA;
      cudaFree(hs.base);
      hs.base = nullptr;
      hs.cap = 0;
    }
    const size_t want = align_up(L.total + L.total / 8, 1 << 20);
    if (cudaMalloc(&hs.base, want) != cudaSuccess) return DSA_ERR_CUDA;
    hs.cap = want;
  }
  return DSA_OK;
}

}  // namespace

// =================================================================== C ABI ==
extern "C" {

int dsa_indexer_topk(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                     const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, int K,
                     int32_t* out_idx, dsa_stream_t stream_) {
  int rc = check_dense(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N);
  if (rc != DSA_OK) return rc;
  if (!out_idx || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  CUtensorMap tq, tk;
  if (!tmap_rows_u8(&tq, q_fp8, (uint64_t)Q * H, H) || !tmap_rows_u8(&tk, k_fp8, N, TILE)) return DSA_ERR_CUDA;
  RowSpace rs{};
  rs.R = Q;
  rs.N = N;
  return run_fused(rs, K, tq, tk, k_fp8, k_scale, q_scale, w, row_begin, row_end, out_idx, stream);
}

int dsa_indexer_topk_host(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                          const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, int K,
                          int32_t* out_idx, dsa_stream_t stream_) {
  if (!q_fp8 || !q_scale || !k_fp8 || !k_scale || !w || !row_begin || !row_end || !out_idx) return DSA_ERR_ARG;
  if (Q <= 0 || N <= 0 || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  if ((int64_t)Q * H >= (1ll << 31) || (int64_t)N >= (1ll << 31) - TILE) return DSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int C = host_chunk_rows(Q);
  const int nch = ceil_div(Q, C);
  const HostLayout L = host_layout(N, C, K);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> hl(g_host_mu);
  HostStage& hs = g_host[{dev, stream}];
  int rc = host_stage_init(hs, L, stream);
  if (rc != DSA_OK) {
    cudaGetLastError();
    return rc;
  }
  // on an error, the copies already enqueued may still write out_idx or read
  // the caller's buffers: they are waited for before returning
  auto fail = [&](int code) {
    cudaGetLastError();
    cudaStreamSynchronize(hs.copy);
    cudaStreamSynchronize(stream);
    cudaGetLastError();
    return code;
  };
#define DSA_HOST_CK(expr)                                 \
  do {                                                    \
    if ((expr) != cudaSuccess) return fail(DSA_ERR_CUDA); \
  } while (0)
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  auto slot = [&](int c) { return hs.base + (size_t)(c & 1) * L.slot; };
  // the copy stream starts behind the work already on the caller's stream
  // (an earlier call may still be reading the staging)
  DSA_HOST_CK(cudaEventRecord(hs.entry, stream));
  DSA_HOST_CK(cudaStreamWaitEvent(hs.copy, hs.entry, 0));
  DSA_HOST_CK(cudaMemcpyAsync(hs.base + L.k, k_fp8, (size_t)N * D, h2d, hs.copy));
  DSA_HOST_CK(cudaMemcpyAsync(hs.base + L.ks, k_scale, (size_t)N * 4, h2d, hs.copy));
  auto h2d_chunk = [&](int c) -> cudaError_t {
    const int64_t r0 = (int64_t)c * C;
    const size_t n = (size_t)std::min<int64_t>(C, Q - r0);
    uint8_t* s = slot(c);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(s + L.q, q_fp8 + r0 * H * D, n * H * D, h2d, hs.copy)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(s + L.qs, q_scale + r0, n * 4, h2d, hs.copy)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(s + L.w, w + r0 * H, n * H * 4, h2d, hs.copy)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(s + L.rb, row_begin + r0, n * 4, h2d, hs.copy)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(s + L.re, row_end + r0, n * 4, h2d, hs.copy)) != cudaSuccess) return e;
    return cudaEventRecord(hs.in_ready[c & 1], hs.copy);
  };
  DSA_HOST_CK(h2d_chunk(0));
  if (nch > 1) DSA_HOST_CK(h2d_chunk(1));
  CUtensorMap tk;
  if (!tmap_rows_u8(&tk, hs.base + L.k, N, TILE)) return fail(DSA_ERR_CUDA);
  for (int c = 0; c < nch; ++c) {
    const int64_t r0 = (int64_t)c * C;
    const int n = (int)std::min<int64_t>(C, Q - r0);
    uint8_t* s = slot(c);
    DSA_HOST_CK(cudaStreamWaitEvent(stream, hs.in_ready[c & 1], 0));
    CUtensorMap tq;
    if (!tmap_rows_u8(&tq, s + L.q, (uint64_t)n * H, H)) return fail(DSA_ERR_CUDA);
    RowSpace rs{};
    rs.R = n;
    rs.N = N;
    rc = run_fused(rs, K, tq, tk, hs.base + L.k, reinterpret_cast<const float*>(hs.base + L.ks),
                   reinterpret_cast<const float*>(s + L.qs), reinterpret_cast<const float*>(s + L.w),
                   reinterpret_cast<const int32_t*>(s + L.rb), reinterpret_cast<const int32_t*>(s + L.re),
                   reinterpret_cast<int32_t*>(s + L.out), stream);
    if (rc != DSA_OK) return fail(rc);
    // this chunk's status block, taken before the next chunk's plan resets it
    Stats* st = arena_stats(stream);
    if (!st) return fail(DSA_ERR_CUDA);
    DSA_HOST_CK(cudaMemcpyAsync(&hs.stats_h[c], st, sizeof(Stats), d2h, stream));
    DSA_HOST_CK(cudaEventRecord(hs.done[c & 1], stream));
    DSA_HOST_CK(cudaStreamWaitEvent(hs.copy, hs.done[c & 1], 0));
    DSA_HOST_CK(cudaMemcpyAsync(out_idx + r0 * K, s + L.out, (size_t)n * K * 4, d2h, hs.copy));
    if (c + 2 < nch) DSA_HOST_CK(h2d_chunk(c + 2));
  }
  DSA_HOST_CK(cudaEventRecord(hs.copies_done, hs.copy));
  DSA_HOST_CK(cudaStreamWaitEvent(stream, hs.copies_done, 0));
  DSA_HOST_CK(cudaStreamSynchronize(stream));
#undef DSA_HOST_CK
  int status = 0;
  for (int c = 0; c < nch; ++c) status |= hs.stats_h[c].status;
  if (status & ST_TIMEOUT) return DSA_ERR_TIMEOUT;
  if (status & ST_RANGE) return DSA_ERR_RANGE;
  return DSA_OK;
}

int dsa_indexer_topk_paged(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_cache,
                           const float* k_cache_scale, const float* w, const int32_t* block_table,
                           const int32_t* seq_lens, int B, int next_n, int max_pages, int num_pages, int K,
                           int32_t* out_idx, dsa_stream_t stream_) {
  if (!q_fp8 || !q_scale || !k_cache || !k_cache_scale || !w || !block_table || !seq_lens || !out_idx)
    return DSA_ERR_ARG;
  if (B <= 0 || next_n <= 0 || max_pages <= 0 || num_pages <= 0 || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  if (!aligned16(q_fp8) || !aligned16(k_cache) || !aligned16(k_cache_scale)) return DSA_ERR_ARG;
  const int64_t R = (int64_t)B * next_n;
  if (R * H >= (1ll << 31) || (int64_t)max_pages * PAGE >= (1ll << 31) - TILE ||
      (int64_t)num_pages * PAGE >= (1ll << 31))
    return DSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  CUtensorMap tq, tk;
  if (!tmap_rows_u8(&tq, q_fp8, (uint64_t)R * H, H) ||
      !tmap_rows_u8(&tk, k_cache, (uint64_t)num_pages * PAGE, PAGE))
    return DSA_ERR_CUDA;
  RowSpace rs{};
  rs.R = (int)R;
  rs.N = max_pages * PAGE;
  rs.paged = 1;
  rs.block_table = block_table;
  rs.seq_lens = seq_lens;
  rs.max_pages = max_pages;
  rs.next_n = next_n;
  rs.num_pages = num_pages;
  return run_fused(rs, K, tq, tk, k_cache, k_cache_scale, q_scale, w, nullptr, nullptr, out_idx, stream);
}

// The standalone top-K takes whole or half rows per CTA item (the ticket of
// each row in the plan's zeroed pair_cnt) from a third of a row per SM on;
// fewer rows are split over the SMs (measured on GB300, rows of 131072 keys,
// split path against the per-row kernel: 48 rows 0.048 / 0.046 ms, 128 rows
// 0.061 / 0.048 ms, 384 rows 0.107 / 0.075 ms, 4096 rows 0.655 / 0.438 ms;
// 8 rows 0.041 / 0.056 ms).
bool matrix_by_rows(const Opts& o, const RowSpace& rs) {
  const int64_t row_min = o.matrix_row_min >= 0 ? o.matrix_row_min : ((int64_t)o.grid + 2) / 3;
  return rs.R >= row_min;
}
// Items per row of the per-row kernel: half rows for fewer rows than SMs
// (twice the items: 128 x 131072 0.057 -> 0.048 ms) and for three waves of
// rows or more of at least 64K keys (4096 x 131072 0.453 -> 0.437 ms);
// whole rows in between, where halves were slower (1216 x 131072 0.155 ->
// 0.167 ms, 2048 x 16384 0.105 -> 0.124 ms).  Measured on GB300.
int matrix_parts(const Opts& o, const RowSpace& rs) {
  const bool many_long = rs.R >= 3LL * MATRIX_TOPK_CTAS_PER_SM * o.grid && rs.N >= 65536;
  return many_long || rs.R < o.grid ? 2 : 1;
}

// Exact top-K over a given fp32 score matrix [R, ld] (the standalone
// selector and the unfused pipeline's second stage), after a main plan `pp`
// (trivial_len = K) on the same arena: one threshold per row from its own
// sample grid in the matrix (rows with L <= K get every valid index there),
// the compare-and-append filter over the matrix into the rows' candidate
// regions, the candidate selector with its certificate, and exact repair of
// the rows that fail it straight from their matrix rows.
int enqueue_matrix_select(Arena* a, const RowSpace& rs, int K, const Opts& o, const float* scores, int64_t ld,
                          const PlanParams& pp, int max_units, int32_t* out, cudaStream_t stream) {
  const Layout& L = a->L;
  Stats* st = pp.stats;
  uint32_t* tau = at<uint32_t>(a, L.tau);
  const int sms = o.grid;
  if (matrix_by_rows(o, rs)) {
    // rows enough to fill the GPU: one CTA per row at a time (threshold,
    // one pass, selection), then the repair of the rows that failed
    MatrixTopkParams mt{};
    mt.rs = rs;
    mt.K = K;
    mt.target16 = o.target16;
    mt.tau_bias = o.bias;
    mt.scores = scores;
    mt.ld = ld;
    mt.rb = pp.rb;
    mt.re = pp.re;
    mt.tau = tau;
    mt.cand_key = at<uint32_t>(a, L.cand_key);
    mt.cand_idx = at<int32_t>(a, L.cand_idx);
    mt.failed_rows = at<int32_t>(a, L.failed);
    mt.out = out;
    mt.stats = st;
    mt.parts = matrix_parts(o, rs);
    mt.half_count = at<int32_t>(a, L.unit_count);
    mt.row_ticket = pp.pair_cnt;
    DSA_LAUNCH(launch_matrix_topk(mt, sms, stream));
    WideParams wp{};
    wp.rs = rs;
    wp.K = K;
    wp.list = mt.failed_rows;
    wp.scores = scores;
    wp.ld = ld;
    wp.by_row = 1;
    wp.rb = pp.rb;
    wp.re = pp.re;
    wp.out = out;
    wp.stats = st;
    DSA_LAUNCH(launch_wide_select(wp, o.grid / 2 > 0 ? o.grid / 2 : 1, stream));
    return DSA_OK;
  }
  SampleTauParams tp{};
  tp.rs = rs;
  tp.K = K;
  tp.target16 = o.target16;
  tp.tau_bias = o.bias;
  tp.rb = pp.rb;
  tp.re = pp.re;
  tp.sscores = scores;
  tp.sld = ld;
  tp.tau = tau;
  tp.stats = st;
  tp.from_matrix = 1;
  tp.out = out;
  DSA_LAUNCH(launch_sample_tau(tp, stream));
  MatrixFilterParams mf{};
  mf.rs = rs;
  mf.chunk_tiles = pp.chunk_tiles;
  mf.scores = scores;
  mf.ld = ld;
  mf.rb = pp.rb;
  mf.re = pp.re;
  mf.groups = pp.groups;
  mf.unit_start = pp.unit_start;
  mf.tau = tau;
  mf.cand_key = at<uint32_t>(a, L.cand_key);
  mf.cand_idx = at<int32_t>(a, L.cand_idx);
  mf.unit_count = at<int32_t>(a, L.unit_count);
  mf.max_units = max_units;
  mf.stats = st;
  DSA_LAUNCH(launch_matrix_filter(mf, 2 * o.grid, stream));  // one wave: 2 CTAs of 512 threads per SM
  CandParams cs{};
  cs.rs = rs;
  cs.K = K;
  cs.groups = pp.groups;
  cs.unit_start = pp.unit_start;
  cs.unit_count = mf.unit_count;
  cs.cand_key = mf.cand_key;
  cs.cand_idx = mf.cand_idx;
  cs.max_units = max_units;
  cs.failed_rows = at<int32_t>(a, L.failed);
  cs.tau = tau;
  cs.out = out;
  cs.stats = st;
  DSA_LAUNCH(launch_cand_select(cs, o.grid, stream));
  WideParams wp{};
  wp.rs = rs;
  wp.K = K;
  wp.list = cs.failed_rows;
  wp.scores = scores;
  wp.ld = ld;
  wp.by_row = 1;
  wp.rb = pp.rb;
  wp.re = pp.re;
  wp.out = out;
  wp.stats = st;
  DSA_LAUNCH(launch_wide_select(wp, o.grid / 2 > 0 ? o.grid / 2 : 1, stream));
  return DSA_OK;
}

static int scores_impl(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                       const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, int K,
                       float* scores, int64_t ld, int32_t* out_idx, cudaStream_t stream) {
  // out_idx == nullptr: scores only (every non-empty row is scored)
  const Opts o = read_opts();
  CUtensorMap tq, tk;
  if (!tmap_rows_u8(&tq, q_fp8, (uint64_t)Q * H, H) || !tmap_rows_u8(&tk, k_fp8, N, TILE)) return DSA_ERR_CUDA;
  RowSpace rs{};
  rs.R = Q;
  rs.N = N;
  const int G = n_groups(rs);
  const int64_t own_ld = align_up((size_t)N, 4);
  // the unfused pipeline's plan also serves its matrix selection
  const int chunk = out_idx ? matrix_chunk_for(o, rs) : chunk_for(o, rs);
  const int max_units = ceil_div(ceil_div(N, TILE), chunk);
  std::lock_guard<std::mutex> lk(g_mu);
  int err = DSA_OK;
  Arena* a = get_arena(stream,
                       make_layout(Q, G, out_idx ? ROW_SLOTS : 0, out_idx ? max_units : 0, scores ? 0 : Q, own_ld),
                       &err);
  if (!a) return err;
  const Layout& L = a->L;
  Stats* st = at<Stats>(a, L.stats);
  float* sbuf = scores ? scores : at<float>(a, L.scores);
  const int64_t sld = scores ? ld : own_ld;

  PlanParams pp{};
  pp.rs = rs;
  pp.K = K;
  pp.trivial_len = out_idx ? K : 0;
  pp.chunk_tiles = chunk;
  pp.row_begin_in = row_begin;
  pp.row_end_in = row_end;
  pp.rb = at<int32_t>(a, L.rb);
  pp.re = at<int32_t>(a, L.re);
  pp.groups = at<Group>(a, L.groups);
  pp.unit_start = at<int32_t>(a, L.unit_start);
  pp.failed_rows = at<int32_t>(a, L.failed);
  if (out_idx && matrix_by_rows(o, rs)) {  // the rows' tickets, zeroed by the plan
    pp.pair_cnt = at<int>(a, L.pair_cnt);
    pp.n_pairs = Q;
  }
  pp.stats = st;
  pp.wait_ns = o.wait_ns;
  DSA_LAUNCH(launch_plan(pp, stream));

  ScoreParams cp{};
  cp.rs = rs;
  cp.mode = MODE_STORE;
  cp.chunk_tiles = pp.chunk_tiles;
  cp.reverse_units = o.reverse_units;
  cp.k_scale = k_scale;
  cp.q_scale = q_scale;
  cp.w = w;
  cp.rb = pp.rb;
  cp.re = pp.re;
  cp.groups = pp.groups;
  cp.unit_start = pp.unit_start;
  cp.scores = sbuf;
  cp.ld = sld;
  cp.stats = st;
  a->profiled = o.profile;
  if (o.profile) cudaEventRecord(a->ev0, stream);
  DSA_LAUNCH(launch_score(tq, tk, cp, o.grid, stream));
  if (o.profile) cudaEventRecord(a->ev1, stream);
  if (!out_idx) return DSA_OK;
  return enqueue_matrix_select(a, rs, K, o, sbuf, sld, pp, max_units, out_idx, stream);
}

int dsa_indexer_topk_unfused(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                             const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, int K,
                             int32_t* out_idx, dsa_stream_t stream) {
  int rc = check_dense(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N);
  if (rc != DSA_OK) return rc;
  if (!out_idx || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  return scores_impl(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N, K, nullptr, 0, out_idx,
                     reinterpret_cast<cudaStream_t>(stream));
}

int dsa_indexer_scores(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                       const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, float* scores,
                       int64_t ld, dsa_stream_t stream) {
  int rc = check_dense(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N);
  if (rc != DSA_OK) return rc;
  if (!scores || ld < N || (ld & 3) || !aligned16(scores)) return DSA_ERR_ARG;
  return scores_impl(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N, 1, scores, ld, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

int dsa_indexer_topk_from_scores(const float* scores, int64_t ld, const int32_t* row_begin, const int32_t* row_end,
                                 int Q, int N, int K, int32_t* out_idx, dsa_stream_t stream_) {
  if (!scores || !row_begin || !row_end || !out_idx) return DSA_ERR_ARG;
  if (Q <= 0 || N <= 0 || ld < N || (ld & 3) || !aligned16(scores) || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const Opts o = read_opts();
  RowSpace rs{};
  rs.R = Q;
  rs.N = N;
  const int chunk = matrix_chunk_for(o, rs);
  const int max_units = ceil_div(ceil_div(N, TILE), chunk);
  std::lock_guard<std::mutex> lk(g_mu);
  int err = DSA_OK;
  Arena* a = get_arena(stream, make_layout(Q, n_groups(rs), ROW_SLOTS, max_units, 0, 0), &err);
  if (!a) return err;
  const Layout& L = a->L;
  PlanParams pp{};
  pp.rs = rs;
  pp.K = K;
  pp.trivial_len = K;
  pp.chunk_tiles = chunk;
  pp.row_begin_in = row_begin;
  pp.row_end_in = row_end;
  pp.rb = at<int32_t>(a, L.rb);
  pp.re = at<int32_t>(a, L.re);
  pp.groups = at<Group>(a, L.groups);
  pp.unit_start = at<int32_t>(a, L.unit_start);
  pp.failed_rows = at<int32_t>(a, L.failed);
  if (matrix_by_rows(o, rs)) {  // the rows' tickets, zeroed by the plan
    pp.pair_cnt = at<int>(a, L.pair_cnt);
    pp.n_pairs = Q;
  }
  pp.stats = at<Stats>(a, L.stats);
  pp.wait_ns = o.wait_ns;
  DSA_LAUNCH(launch_plan(pp, stream));
  a->profiled = false;
  return enqueue_matrix_select(a, rs, K, o, scores, ld, pp, max_units, out_idx, stream);
}

int dsa_indexer_topk_from_scores_noalloc(const float* scores, int64_t ld, const int32_t* row_begin,
                                         const int32_t* row_end, int Q, int N, int K, int32_t* out_idx,
                                         dsa_stream_t stream_) {
  if (!scores || !row_begin || !row_end || !out_idx) return DSA_ERR_ARG;
  if (Q <= 0 || N <= 0 || ld < N || (ld & 3) || !aligned16(scores) || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  if (Q > NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;
  RowSpace rs{};
  rs.R = Q;
  rs.N = N;
  const Layout L = make_layout(Q, n_groups(rs), 0, 0, 0, 0);
  if (L.total > NOALLOC_SCRATCH_BYTES) return DSA_ERR_UNSUPPORTED;
  int err = DSA_OK;
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch(&err));
  if (!base) return err;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const Opts o = read_opts();
  // the plan kernel rewrites every part of the scratch this call reads:
  // counters and status are zeroed, row ranges validated and stored
  PlanParams pp{};
  pp.rs = rs;
  pp.K = K;
  pp.trivial_len = 0x7fffffff;
  pp.chunk_tiles = 64;
  pp.row_begin_in = row_begin;
  pp.row_end_in = row_end;
  pp.rb = reinterpret_cast<int32_t*>(base + L.rb);
  pp.re = reinterpret_cast<int32_t*>(base + L.re);
  pp.groups = reinterpret_cast<Group*>(base + L.groups);
  pp.unit_start = reinterpret_cast<int32_t*>(base + L.unit_start);
  pp.failed_rows = reinterpret_cast<int32_t*>(base + L.failed);
  pp.stats = reinterpret_cast<Stats*>(base + L.stats);
  pp.wait_ns = o.wait_ns;
  DSA_LAUNCH(launch_plan(pp, stream));
  SelectParams sel{};
  sel.rs = rs;
  sel.K = K;
  sel.target16 = o.target16;
  sel.scores = scores;
  sel.ld = ld;
  sel.rb = pp.rb;
  sel.re = pp.re;
  sel.out = out_idx;
  sel.stats = pp.stats;
  DSA_LAUNCH(launch_select(sel, 2 * o.grid, stream));
  return DSA_OK;
}

int dsa_indexer_math_control(const uint8_t* q_fp8, const float* q_scale, const uint8_t* k_fp8, const float* k_scale,
                             const float* w, const int32_t* row_begin, const int32_t* row_end, int Q, int N, int K,
                             float* checksum, dsa_stream_t stream_) {
  int rc = check_dense(q_fp8, q_scale, k_fp8, k_scale, w, row_begin, row_end, Q, N);
  if (rc != DSA_OK) return rc;
  if (!checksum || K < 1 || K > DSA_MAX_K) return DSA_ERR_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  CUtensorMap tq, tk;
  if (!tmap_rows_u8(&tq, q_fp8, (uint64_t)Q * H, H) || !tmap_rows_u8(&tk, k_fp8, N, TILE)) return DSA_ERR_CUDA;
  const Opts o = read_opts();
  RowSpace rs{};
  rs.R = Q;
  rs.N = N;
  // the fused call's main plan: the same rows (L > K), groups and units
  const int chunk = chunk_for(o, rs);
  std::lock_guard<std::mutex> lk(g_mu);
  int err = DSA_OK;
  Arena* a = get_arena(stream, make_layout(Q, n_groups(rs), 0, 0, 0, 0), &err);
  if (!a) return err;
  const Layout& L = a->L;
  PlanParams pp{};
  pp.rs = rs;
  pp.plan = PLAN_MAIN;
  pp.K = K;
  pp.trivial_len = K;
  pp.chunk_tiles = chunk;
  pp.row_begin_in = row_begin;
  pp.row_end_in = row_end;
  pp.rb = at<int32_t>(a, L.rb);
  pp.re = at<int32_t>(a, L.re);
  pp.groups = at<Group>(a, L.groups);
  pp.unit_start = at<int32_t>(a, L.unit_start);
  pp.failed_rows = at<int32_t>(a, L.failed);
  pp.stats = at<Stats>(a, L.stats);
  pp.wait_ns = o.wait_ns;
  DSA_LAUNCH(launch_plan(pp, stream));
  ScoreParams cp{};
  cp.rs = rs;
  cp.mode = MODE_CONTROL;
  cp.chunk_tiles = chunk;
  cp.plan = PLAN_MAIN;
  cp.k_scale = k_scale;
  cp.q_scale = q_scale;
  cp.w = w;
  cp.rb = pp.rb;
  cp.re = pp.re;
  cp.groups = pp.groups;
  cp.unit_start = pp.unit_start;
  cp.scores = checksum;
  cp.stats = pp.stats;
  a->profiled = o.profile;
  if (o.profile) cudaEventRecord(a->ev0, stream);
  DSA_LAUNCH(launch_score(tq, tk, cp, o.grid, stream));
  if (o.profile) cudaEventRecord(a->ev1, stream);
  return DSA_OK;
}

int dsa_sparse_attention(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* ckv, const uint16_t* kpe,
                         const int32_t* indices, int T, int H, int K, int num_slots, float sm_scale, uint16_t* out,
                         float* lse, dsa_stream_t stream_) {
  if (!q_nope || !q_pe || !ckv || !kpe || !indices || !out || !lse) return DSA_ERR_ARG;
  if (T <= 0 || H <= 0 || (H % 16) || K < 1 || num_slots <= 0 || !(sm_scale > 0.f)) return DSA_ERR_ARG;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(ckv) || !aligned16(kpe) || !aligned16(out))
    return DSA_ERR_ARG;
  if ((int64_t)T * H >= (1ll << 31) / 512 || (int64_t)T * K >= (1ll << 31) || T > 65535) return DSA_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const Opts o = read_opts();
  // splits of each token's key list: about one wave of resident CTAs, at
  // least 64 keys per split
  const int ctas = T * (H / 16);
  int splits = std::max(1, std::min(sparse_attn_ctas_per_sm() * o.grid / std::max(ctas, 1), K / 64));
  // (a split's slots, at most SA_MAX_PER = 2048, are staged in shared memory)
  int per = std::min(ceil_div(ceil_div(K, splits), 32) * 32, 2048);
  splits = ceil_div(K, per);
  const int64_t rows = (int64_t)T * H;
  const size_t off_ml = 256, off_o = align_up(off_ml + (size_t)splits * rows * 8, 256);
  const size_t need = splits > 1 ? off_o + (size_t)splits * rows * 512 * 4 : 256;
  std::lock_guard<std::mutex> lk(g_mu);
  int err = DSA_OK;
  uint8_t* base = aux_scratch(stream, need, &err);
  if (!base) return err;
  SparseAttnParams p{};
  p.q_nope = reinterpret_cast<const __nv_bfloat16*>(q_nope);
  p.q_pe = reinterpret_cast<const __nv_bfloat16*>(q_pe);
  p.ckv = reinterpret_cast<const __nv_bfloat16*>(ckv);
  p.kpe = reinterpret_cast<const __nv_bfloat16*>(kpe);
  p.idx = indices;
  p.T = T;
  p.H = H;
  p.K = K;
  p.num_slots = num_slots;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.splits = splits;
  p.keys_per_split = per;
  p.part_ml = reinterpret_cast<float2*>(base + off_ml);
  p.part_o = reinterpret_cast<float*>(base + off_o);
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = reinterpret_cast<int*>(base);
  if (cudaMemsetAsync(p.status, 0, sizeof(int), stream) != cudaSuccess) return DSA_ERR_CUDA;
  DSA_LAUNCH(launch_sparse_attn(p, stream));
  return DSA_OK;
}

int dsa_sparse_attention_last_status(dsa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_aux.find({dev, stream});
  if (it == g_aux.end() || !it->second.base) return DSA_OK;
  int st = 0;
  if (cudaMemcpy(&st, it->second.base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DSA_ERR_CUDA;
  return (st & ST_RANGE) ? DSA_ERR_RANGE : DSA_OK;
}

int dsa_indexer_last_device_status(dsa_stream_t stream_, int32_t* failures_out) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_arenas.find({dev, stream});
  if (it == g_arenas.end() || !it->second.used) {
    if (failures_out) memset(failures_out, 0, 4 * sizeof(int32_t));
    return DSA_OK;
  }
  Stats st;
  if (cudaMemcpy(&st, it->second.base + it->second.L.stats, sizeof(Stats), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (failures_out) {
    failures_out[0] = st.underflow;
    failures_out[1] = st.overflow;
    failures_out[2] = st.trivial;
    failures_out[3] = st.cand_total;
  }
  if (st.status & ST_TIMEOUT) return DSA_ERR_TIMEOUT;
  if (st.status & ST_RANGE) return DSA_ERR_RANGE;
  return DSA_OK;
}

int dsa_indexer_last_repaired_rows(dsa_stream_t stream_, int32_t* rows_out, int cap) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cap < 0 || (cap > 0 && !rows_out)) return DSA_ERR_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_arenas.find({dev, stream});
  if (it == g_arenas.end() || !it->second.used) return 0;
  Stats st;
  const Arena& a = it->second;
  if (cudaMemcpy(&st, a.base + a.L.stats, sizeof(Stats), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  const int n = st.fail_count < cap ? st.fail_count : cap;
  if (n > 0 && cudaMemcpy(rows_out, a.base + a.L.failed, n * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  return st.fail_count;
}

int dsa_indexer_set_option(int option, int64_t value) {
  std::lock_guard<std::mutex> lk(g_mu);
  switch (option) {
    case DSA_OPT_CHUNK_TILES:
      if (value != -1 && (value < 1 || value > (1 << 20))) return DSA_ERR_ARG;
      g_chunk_tiles = value;
      return DSA_OK;
    case DSA_OPT_TAU_BIAS:
      g_tau_bias = value;
      return DSA_OK;
    case DSA_OPT_PROFILE:
      g_profile = value ? 1 : 0;
      return DSA_OK;
    case DSA_OPT_GRID_CTAS:
      if (value < 0 || value > 65535) return DSA_ERR_ARG;
      g_grid = value;
      return DSA_OK;
    case DSA_OPT_SAMPLE_TARGET:
      if (value < 1 || value > 256) return DSA_ERR_ARG;
      g_target16 = value;
      return DSA_OK;
    case DSA_OPT_HOST_CHUNK_ROWS:
      if (value < 0 || value > (1 << 30)) return DSA_ERR_ARG;
      g_host_chunk_rows = value;
      return DSA_OK;
    case DSA_OPT_UNIT_ORDER:
      if (value != 0 && value != 1) return DSA_ERR_ARG;
      g_unit_order = value;
      return DSA_OK;
    case DSA_OPT_WAIT_LIMIT_US:
      if (value < 1 || value > 60000000) return DSA_ERR_ARG;
      g_wait_us = value;
      return DSA_OK;
    case DSA_OPT_TEST_WITHHOLD:
      if (value != 0 && value != 1) return DSA_ERR_ARG;
      g_withhold = value;
      return DSA_OK;
    case DSA_OPT_MATRIX_ROW_MIN:
      if (value < -1) return DSA_ERR_ARG;
      g_matrix_row_min = value;
      return DSA_OK;

    default:
      return DSA_ERR_ARG;
  }
}

int64_t dsa_indexer_get_option(int option) {
  std::lock_guard<std::mutex> lk(g_mu);
  switch (option) {
    case DSA_OPT_CHUNK_TILES:
      return g_chunk_tiles;
    case DSA_OPT_TAU_BIAS:
      return g_tau_bias;
    case DSA_OPT_PROFILE:
      return g_profile;
    case DSA_OPT_GRID_CTAS:
      return g_grid;
    case DSA_OPT_SAMPLE_TARGET:
      return g_target16;
    case DSA_OPT_HOST_CHUNK_ROWS:
      return g_host_chunk_rows;
    case DSA_OPT_UNIT_ORDER:
      return g_unit_order;
    case DSA_OPT_WAIT_LIMIT_US:
      return g_wait_us;
    case DSA_OPT_TEST_WITHHOLD:
      return g_withhold;
    case DSA_OPT_MATRIX_ROW_MIN:
      return g_matrix_row_min;

    default:
      return DSA_ERR_ARG;
  }
}

float dsa_indexer_profiled_main_ms(dsa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1.f;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_arenas.find({dev, stream});
  if (it == g_arenas.end() || !it->second.profiled) return -1.f;
  if (cudaEventSynchronize(it->second.ev1) != cudaSuccess) return -1.f;
  float ms = -1.f;
  if (cudaEventElapsedTime(&ms, it->second.ev0, it->second.ev1) != cudaSuccess) return -1.f;
  return ms;
}

int64_t dsa_indexer_launch_count(void) { return g_launches.load(); }

const char* dsa_indexer_version(void) { return "dsa_indexer 0.1 (sm_103a, tcgen05 + TMA)"; }

int dsa_indexer_release(void) {
  // lock order of the library: g_host_mu before g_mu
  std::lock_guard<std::mutex> hl(g_host_mu);
  for (auto& kv : g_host) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(kv.first.first);
    HostStage& hs = kv.second;
    if (hs.copy) cudaStreamSynchronize(hs.copy);
    if (hs.base) cudaFree(hs.base);
    cudaEvent_t evs[] = {hs.entry, hs.copies_done, hs.in_ready[0], hs.in_ready[1], hs.done[0], hs.done[1]};
    for (cudaEvent_t e : evs)
      if (e) cudaEventDestroy(e);
    if (hs.copy) cudaStreamDestroy(hs.copy);
    if (hs.stats_h) cudaFreeHost(hs.stats_h);
    cudaSetDevice(cur);
  }
  g_host.clear();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_arenas.empty() || !g_aux.empty()) cudaDeviceSynchronize();
  for (auto& kv : g_arenas) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(kv.first.first);
    if (kv.second.base) cudaFree(kv.second.base);
    if (kv.second.ev0) cudaEventDestroy(kv.second.ev0);
    if (kv.second.ev1) cudaEventDestroy(kv.second.ev1);
    cudaSetDevice(cur);
  }
  g_arenas.clear();
  for (auto& kv : g_aux) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(kv.first.first);
    if (kv.second.base) cudaFree(kv.second.base);
    cudaSetDevice(cur);
  }
  g_aux.clear();
  return DSA_OK;
}

}  // extern "C"
