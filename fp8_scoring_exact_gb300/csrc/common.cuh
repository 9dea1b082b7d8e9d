// common.cuh -- shared constants, plan structures and inline-PTX wrappers for
// the sm_103a DSA indexer kernels (tcgen05 MMA with TMEM accumulators, TMA
// tensor copies, mbarriers with bounded waits).
//
// Written from the public PTX ISA description of these instructions; no
// library code is used.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

// ---------------------------------------------------------------- geometry --
constexpr int H = 64;              // indexer heads
constexpr int D = 128;             // head dimension (bytes per FP8 vector)
constexpr int TILE = 128;          // keys per MMA tile (MMA M, one TMEM lane per key)
constexpr int GROUP_ROWS = 4;      // query rows sharing one key stream (MMA N = 64 * rows <= 256)
constexpr int SAMPLE_ROWS = 2;     // query rows per CTA of the threshold-sampling kernel
constexpr int PAGE = 64;           // tokens per paged-cache page

// ------------------------------------------------------- persistent scorer --
constexpr int STAGES = 6;          // key-tile ring depth (TMA -> MMA)
constexpr int ACC_BUFS = 2;        // TMEM accumulators (MMA -> epilogue)
constexpr int ACC_COLS = 256;      // TMEM columns per accumulator (4 rows x 64 heads)
constexpr int EPI_WGS = GROUP_ROWS; // epilogue warpgroups: one per row of the group
constexpr int EPI_THREADS = EPI_WGS * 128;
constexpr int SCORE_THREADS = 64 + EPI_THREADS;  // warp 0: TMA, warp 1: MMA; then the epilogue
// Candidate slots of a row, shared evenly by its regions: every work unit of
// the row's group leaves candidates in UNIT_REGIONS regions (one per epilogue
// warp, i.e. TMEM lane quarter).  Splitting a fixed budget keeps each region
// about 4x its expected fill whatever the row length: ~2K candidates spread
// over the row's regions.
constexpr int ROW_SLOTS = 16384;
constexpr int UNIT_REGIONS = 4;
__host__ __device__ constexpr int region_cap(int nunits) {
  return (ROW_SLOTS / (nunits * UNIT_REGIONS)) & ~3;
}

// -------------------------------------------------------------- selection --
constexpr int MAX_K = 2048;        // largest K (the public header's DSA_MAX_K)
constexpr int CAND_MAX_REGIONS = 1024;  // regions (units x 4) one row may have
constexpr int SAMPLE_STRIDE = 200; // one sample per 200 keys: ~0.5% of the row
constexpr int SAMPLE_OFFSET = 100; // samples at keys 100 mod 200
constexpr int MAX_SAMPLES = 1024;  // per row; longer rows widen the stride
constexpr int SELECT_THREADS = 512;
constexpr int SELECT_CAP = 12288;  // candidates the standalone selector keeps in SMEM
constexpr int SEL_UNROLL = 4;      // float4 loads in flight per thread in its filter pass

// Which plan a kernel reads: every row, the rows queued for repair, or the
// rows' sample grids.
enum Plan : int { PLAN_MAIN = 0, PLAN_REPAIR = 1, PLAN_SAMPLE = 2 };

// MODE_STORE: fp32 scores to a matrix.  MODE_FILTER: scores at or above the
// row's threshold become candidates for the candidate selector.
// MODE_CONTROL: the math-only control (a measurement, never part of an
// operator): the same loads, MMAs and barriers, but the epilogue only reads
// one accumulator column per warp and tile into a checksum and releases the
// accumulator (no ReLU, head reduction or candidates).
enum Mode : int { MODE_STORE = 0, MODE_FILTER = 1, MODE_CONTROL = 2 };

// status word bits (per call)
constexpr int ST_TIMEOUT = 1;
constexpr int ST_RANGE = 2;

// device counters of one call, laid out at the start of the arena
struct Stats {
  int status;
  int underflow;     // rows whose candidate set had fewer than K entries
  int overflow;      // rows of which a candidate region lost candidates (more than it holds)
  int trivial;       // rows with L <= K (remapping path)
  int cand_total;    // candidates appended (all rows)
  int fail_count;    // rows queued for repair
  int n_groups;      // main plan
  int total_units;
  int r_groups;      // repair plan
  int r_units;
  int s_groups;      // sample plan
  int s_units;
  int next_unit[3];  // per plan (PLAN_*): the next work unit a scorer CTA takes
  int cs_done;       // candidate-selector CTAs finished (the last one plans the repair)
  int cs_next;       // candidate selector: items handed out past each CTA's first
  unsigned long long wait_ns;  // limit of the call's pipeline waits (read only by a wait that stalls)
};

// A work group: up to GROUP_ROWS (4) query rows that stream the same keys.  Key range is
// the union of the rows' valid ranges, in logical key coordinates.
struct Group {
  int nrows;
  int row[GROUP_ROWS];   // logical row ids (dense: t; paged: b * next_n + i)
  int slot[GROUP_ROWS];  // score-matrix row for MODE_STORE
  int lo, hi;            // union key range [lo, hi)
  int seq;               // paged: sequence b; dense: -1
};

// --------------------------------------------------------------- helpers ----
__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Order-preserving float -> uint32 map (-0 canonicalised to +0).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// The float T with (x >= T) == (ordered_key(x) >= key) for every non-NaN x:
// the filter compares scores against it instead of mapping each score.
__device__ __forceinline__ float key_threshold_float(uint32_t key) {
  if (key <= 0x007FFFFFu) return -__int_as_float(0x7f800000);  // at or below -inf's key: all pass
  if (key > 0xFF800000u) return __int_as_float(0x7fffffff);     // above +inf's key: none (NaN)
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Named barrier over `nthreads` threads.  The non-aligned form: threads of a
// warp may arrive at different times (e.g. after one lane waited alone).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- mbarriers ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Test (or briefly wait for) completion of the phase with `parity`.  An
// explicit suspend-time hint was measured and made the scorer slower, so the
// system default window is used.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Pipeline waits give up after the call's limit (Stats::wait_ns, by default
// WAIT_LIMIT_NS; the kernel then records ST_TIMEOUT, lets what it already
// issued land and returns instead of hanging the GPU).
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s
// Waits of the abort path, for copies and MMAs issued before the abort
// (they complete within microseconds; the bound only guarantees an end).
constexpr uint64_t DRAIN_LIMIT_NS = 2000000000ull;

// The call's wait limit, from its status block (the plan kernel stores it).
__device__ __forceinline__ uint64_t wait_limit(const Stats* st) {
  const uint64_t l = *(volatile const unsigned long long*)&st->wait_ns;
  return l ? l : WAIT_LIMIT_NS;
}

// Bounded wait: true when the phase with `parity` completed; false when the
// CTA-wide abort flag is set or the time limit passed (then it sets both the
// abort flag and the status bit).  The polling loop is out of line: the hot
// loops only pay for one test when the phase has already completed.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            Stats* st) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 7u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > wait_limit(st)) {
        *abort_flag = 1;
        atomicOr(&st->status, ST_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          Stats* st) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, st);
}

// Abort path: wait, bounded by DRAIN_LIMIT_NS and regardless of the abort
// flag, for the phase with `parity` of a barrier that copies or MMAs issued
// before the abort arrive on; false if the bound passed.
static __device__ __noinline__ bool mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > DRAIN_LIMIT_NS) return false;
  return true;
}

// Warp-uniform bounded wait: every lane polls (so every lane acquires the
// phase) and every lane returns the same value, so code after it that needs
// a converged warp (tcgen05.ld .sync.aligned, shuffles) never diverges.
static __device__ __noinline__ bool mbar_wait_warp_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 Stats* st) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    const bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    if ((it & 7u) == 7u) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*abort_flag) {
          give_up = 1;
        } else {
          const uint64_t now = globaltimer_ns();
          if (t0 == 0) {
            t0 = now;
          } else if (now - t0 > wait_limit(st)) {
            *abort_flag = 1;
            atomicOr(&st->status, ST_TIMEOUT);
            give_up = 1;
          }
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               Stats* st) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return mbar_wait_warp_slow(bar, parity, abort_flag, st);
}

// Warp-uniform bounded wait for a warp whose wake-up latency has slack (the
// TMA producer, which runs ahead of the MMA): between polls it sleeps, so it
// takes no issue slots from the epilogue warps that share its SM
// sub-partition (measured: 1% on the dense scorer).
static __device__ __noinline__ bool mbar_wait_warp_backoff_slow(uint32_t bar, uint32_t parity,
                                                         volatile int* abort_flag, Stats* st) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(128);
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int give_up = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*abort_flag) {
        give_up = 1;
      } else if (globaltimer_ns() - t0 > wait_limit(st)) {
        *abort_flag = 1;
        atomicOr(&st->status, ST_TIMEOUT);
        give_up = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
  }
}
__device__ __forceinline__ bool mbar_wait_warp_backoff(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                       Stats* st) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  return mbar_wait_warp_backoff_slow(bar, parity, abort_flag, st);
}

// n arrivals (a warp arriving for itself and n - 1 others), from the lane
// elect.sync picks (the warp must be converged).
__device__ __forceinline__ void mbar_arrive_warp_n(uint32_t bar, uint32_t n) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
      "r"(n)
      : "memory");
}

// One arrival per warp, from the lane elect.sync picks (the warp must be
// converged); no branch around it.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ------------------------------------------------------------------- TMA ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// generic-proxy writes to shared memory -> visible to the async proxy (MMA)
// Programmatic dependent launch: the library launches every kernel with
// programmatic stream serialisation.  A kernel first lets the next launch
// begin (it starts once every CTA of this grid has reached this point, and
// its CTAs take SM resources only as they free up), then waits until the
// previous grid of the stream has completed and its memory is visible: the
// launch latency between the call's kernels overlaps the previous kernel's
// tail.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 16 bytes global -> shared without registers (cp.async); n_src = 0 writes
// zeros and reads nothing.  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int n_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n_src) : "memory");
}
// 4 bytes global -> shared (cp.async; both addresses 4-byte aligned)
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Waits until every cp.async this thread issued has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// The mbarrier tracks this thread's earlier cp.async copies: its pending
// count rises by one now and falls by one when they have landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// --------------------------------------------------------------- tcgen05 ----
// Shared-memory matrix descriptor for a K-major operand stored in the 128-byte
// swizzled layout TMA writes (rows of 128 bytes, 8-row / 1024-byte swizzle
// atoms): start address >> 4, leading-byte offset 1 (unused for this layout),
// stride-byte offset 1024 >> 4 between 8-row groups, descriptor version 1,
// layout type 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, one 128 x N x 32 e4m3 step.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// mbarrier arrives once when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 1 column: thread i gets lane (base + i).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 lanes x 32 columns: thread t receives, for each block m (0..3) of 8
// columns, columns 8m + 2(t % 4) + {0, 1} of lanes base + t / 4 (r[4m],
// r[4m+1]) and base + 8 + t / 4 (r[4m+2], r[4m+3]).
__device__ __forceinline__ void tmem_ld16x256b_x4(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Read-only global loads issued where they are written (volatile): a load at
// the top of a loop iteration whose value is used at its end keeps its
// latency behind the iteration's work.
__device__ __forceinline__ float ldg_pinned_f32(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------- epilogue arithmetic --
// ReLU on the FMA pipe: x * 2^-25 saturated to [0, 1] equals ReLU(x) * 2^-25
// exactly, because every accumulator of a 128-long e4m3 dot satisfies
// |x| <= 128 * 448^2 < 2^25 and, when non-zero, |x| >= 2^-18 (so the scaled
// value is a normal number and the power-of-two scaling is exact).  The
// weight of such a head is stored pre-multiplied by 2^25.
__device__ __forceinline__ float relu_scaled_fma_pipe(float x) {
  float r;
  asm volatile("mul.rn.sat.f32 %0, %1, 0f33000000;" : "=f"(r) : "f"(x));
  return r;
}
constexpr float RELU_SAT_WEIGHT_SCALE = 33554432.0f;  // 2^25

__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// a * b on two fp32 lanes
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// acc += a * b on two fp32 lanes (sm_100+ packed FMA)
__device__ __forceinline__ void ffma2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm volatile("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// ------------------------------------------------- radix select (shared) ----
// Find the bucket of the K-th largest among `hist[256]` (counts of live keys
// by the current byte), scanning from bucket 255 down.  Executed by one full
// warp; writes the digit, the remaining rank (rank within that bucket) and
// the bucket's count to out[0], out[1], out[2].
__device__ __forceinline__ void radix_pick_digit(const int* hist, int rem, int* out) {
  const int lane = threadIdx.x & 31;
  // lane l owns buckets 255-8l .. 248-8l (descending)
  int c[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = hist[255 - 8 * lane - i];
    sum += c[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - sum;
  const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
  const int src = hit ? (__ffs(hit) - 1) : 31;
  if (lane == src) {
    int acc = excl;
    int digit = 255 - 8 * lane - 7;
    int r = rem - acc;
    int cnt = c[7];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (acc + c[i] >= rem) {
        digit = 255 - 8 * lane - i;
        r = rem - acc;
        cnt = c[i];
        break;
      }
      acc += c[i];
    }
    out[0] = digit;
    out[1] = r;
    out[2] = cnt;
  }
}

}  // namespace dsa
