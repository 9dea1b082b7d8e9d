// kernels.h -- parameter blocks and launchers of the indexer kernels
// (internal to the library; the public ABI is include/dsa_indexer.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace dsa {

// Row geometry shared by every kernel: dense rows are t = 0..R-1 with
// explicit ranges; paged rows are b * next_n + i over sequences b.
struct RowSpace {
  int R;          // logical rows
  int N;          // dense: keys; paged: max_pages * 64
  int paged;
  const int32_t* block_table;  // paged: [B, max_pages]
  const int32_t* seq_lens;     // paged: [B]
  int max_pages;
  int next_n;
  int num_pages;
  int* status;                 // paged: the call's status word (a used block-table entry outside [0, num_pages))
};

// chunk size that makes every work unit a whole row pair (tiles per row < 2^24)
constexpr int WHOLE_PAIR_TILES = 1 << 24;

struct PlanParams {
  RowSpace rs;
  int plan;                    // PLAN_MAIN: every row; PLAN_REPAIR: the queued rows; PLAN_SAMPLE: sample grids
  int sample_stride;           // PLAN_SAMPLE: grid keys are SAMPLE_OFFSET + j * sample_stride
  int K;
  int trivial_len;             // rows with L <= trivial_len are not scored
  int chunk_tiles;
  const int32_t* row_begin_in; // dense input ranges
  const int32_t* row_end_in;
  int32_t* rb;                 // [R] validated ranges (written in main mode; sample-grid ranges in sample mode)
  int32_t* re;
  Group* groups;               // [G]
  int32_t* unit_start;         // [G + 1]
  const int32_t* failed_rows;  // repair mode input
  Stats* stats;
  uint64_t wait_ns;            // main plan: the call's pipeline wait limit (stored in the status block)
  int* pair_cnt;               // main plan: sampling tickets per row pair, zeroed (null: none)
  int n_pairs;
};

struct SampleParams {
  RowSpace rs;
  int K;
  int target16;                // threshold aims at target16 * K / 16 candidates
  int64_t tau_bias;            // test knob added to every threshold key
  const uint8_t* k;            // dense keys [N, 128] or paged cache [P * 64, 128]
  const float* k_scale;        // dense [N] or paged [P * 64]
  const float* q_scale;
  const float* w;
  const int32_t* rb;
  const int32_t* re;
  uint32_t* tau;               // [R] threshold keys (written; not in split mode)
  int32_t* out;                // [R, K] (trivial rows written here)
  Stats* stats;
  // split mode: one CTA per (row pair, 128-key sample tile) writes the
  // sample scores; the pair's last tile CTA to finish (pair_cnt ticket,
  // zeroed by the main plan) selects the pair's thresholds
  int split;
  int* pair_cnt;               // [pairs]
  float* sscores;              // [R, sld]: row r's score of pair-grid sample j at r * sld + j
  int64_t sld;
  int32_t* srb;                // [R] first / end pair-grid sample inside the row's range
  int32_t* sre;
};

struct ScoreParams {
  RowSpace rs;
  int mode;                    // MODE_STORE or MODE_FILTER
  int chunk_tiles;
  int plan;                    // which plan to read (PLAN_*)
  int reverse_units;           // 1: the counter hands the plan's units out last first (a test of order independence)
  int withhold_first_acc;      // test option: the MMA never signals its first accumulator (a wait must run out)
  const float* k_scale;        // dense [N] or paged [P * 64]
  const float* q_scale;
  const float* w;
  const int32_t* rb;
  const int32_t* re;
  const Group* groups;
  const int32_t* unit_start;
  // MODE_FILTER: epilogue warp q of unit c leaves at most region_cap(units)
  // candidates of a row in region (4 c + q) of that row's ROW_SLOTS
  const uint32_t* tau;
  uint32_t* cand_key;          // [R, ROW_SLOTS]
  int32_t* cand_idx;           // [R, ROW_SLOTS]
  int32_t* unit_count;         // [R, max_units, 4]: candidates region (c, q) holds (cap + 1: lost some)
  int max_units;               // candidate-region units per row, at most (2 x work units)
  // MODE_STORE (MODE_CONTROL: the checksum word, added to)
  float* scores;               // [slots, ld]
  int64_t ld;
  Stats* stats;
};

// Candidate selector: exact top-K of each planned row from the candidate
// regions the filter left, with the certificate (K <= n, no region lost
// candidates); rows that fail it are queued for repair.
struct CandParams {
  RowSpace rs;
  int K;
  const Group* groups;
  const int32_t* unit_start;
  const int32_t* unit_count;
  const uint32_t* cand_key;     // [R, ROW_SLOTS]
  const int32_t* cand_idx;
  const uint32_t* tau;         // [R] threshold keys (every candidate is at or above its row's)
  int max_units;
  int32_t* failed_rows;        // [R] (appended, count in stats->fail_count)
  int32_t* out;                // [R, K]
  Stats* stats;
  int plan_repair;             // 1: the CTA that finishes last writes the repair plan below
  PlanParams repair;           // (plan PLAN_REPAIR)
};

struct SelectParams {
  RowSpace rs;
  int K;
  int target16;
  const float* scores;
  int64_t ld;
  const int32_t* rb;
  const int32_t* re;
  int32_t* out;
  Stats* stats;
};

// grid stride of the sampled thresholds for rows up to N keys: 200, widened
// so that no row has more than MAX_SAMPLES grid keys
__host__ __device__ inline int sample_stride_for(int N) {
  const int widen = (N + SAMPLE_STRIDE * MAX_SAMPLES - 1) / (SAMPLE_STRIDE * MAX_SAMPLES);
  return SAMPLE_STRIDE * (widen > 1 ? widen : 1);
}

// Exact top-K of the score rows of the repair list (few long rows): one
// thread-block cluster per row, four 8-bit radix passes over row slices,
// then emission by slices.
struct WideParams {
  RowSpace rs;
  int K;
  const int32_t* list;         // repair rows; count in stats->fail_count
  const float* scores;         // score row of list entry f at f * ld (by_row: at row * ld)
  int by_row;
  int64_t ld;
  const int32_t* rb;
  const int32_t* re;
  int32_t* out;                // [R, K]
  const Stats* stats;
};

// Sampled thresholds of dense rows from the scorer: sample_prep gathers the
// grid keys (SAMPLE_OFFSET + j * stride) into a contiguous key set and writes
// the trivial rows; the scorer (store mode, sample plan) scores every row's
// grid keys; sample_tau selects each row's threshold from its sample scores.
struct SamplePrepParams {
  RowSpace rs;                 // dense
  int K;
  int stride;
  int n_samples;               // grid keys below N
  const uint8_t* k;            // [N, 128]
  const float* k_scale;
  uint8_t* sk;                 // [n_samples, 128] (written)
  float* sks;                  // [n_samples] (written)
  const int32_t* rb;           // validated ranges
  const int32_t* re;
  int32_t* out;                // [R, K]: trivial rows written
  Stats* stats;
  PlanParams plan;             // the sample plan (PLAN_SAMPLE), built by the first CTA
};
struct SampleTauParams {
  RowSpace rs;
  int K;
  int target16;
  int64_t tau_bias;
  const int32_t* rb;           // key-space ranges
  const int32_t* re;
  const int32_t* srb;          // sample-grid ranges
  const int32_t* sre;
  const float* sscores;        // [R, sld] sample scores (row r at r * sld)
  int64_t sld;
  uint32_t* tau;               // [R] (written for rows with L > K)
  Stats* stats;
  // from_matrix: sscores is a full fp32 score matrix [R, sld]; a row's
  // samples are its own 1-in-200 grid inside [rb, re) (srb / sre unused),
  // and rows with L <= K get every valid index in out (trivial path)
  int from_matrix;
  int32_t* out;
};

// Candidate filter over a given fp32 score matrix (the standalone top-K):
// the work units of a main plan, each warp (row slot r, key quarter q) of a
// 512-thread CTA appending the scores of its row that reach the row's
// threshold to region (c, q) of the row, like the scorer's filter epilogue
// (the candidate selector then takes over unchanged).
struct MatrixFilterParams {
  RowSpace rs;
  int chunk_tiles;
  const float* scores;         // [R, ld]
  int64_t ld;
  const int32_t* rb;
  const int32_t* re;
  const Group* groups;
  const int32_t* unit_start;
  const uint32_t* tau;
  uint32_t* cand_key;          // [R, ROW_SLOTS]
  int32_t* cand_idx;
  int32_t* unit_count;         // [R, max_units, 4]
  int max_units;
  Stats* stats;
};

// Exact top-K over a given fp32 score matrix by whole or half rows (the
// standalone top-K when the rows fill the GPU): an item's scores at or
// above the row's threshold (from its own sample grid) go to its share of
// the row's ROW_SLOTS candidate slots, and the CTA that finishes a row
// selects it from its lists; rows that fail the certificate are queued for
// repair.
#ifndef DSA_RT_CTAS
#define DSA_RT_CTAS 4
#endif
constexpr int MATRIX_TOPK_CTAS_PER_SM = DSA_RT_CTAS;
struct MatrixTopkParams {
  RowSpace rs;
  int K;
  int target16;
  int64_t tau_bias;
  const float* scores;         // [R, ld]
  int64_t ld;
  const int32_t* rb;           // validated ranges
  const int32_t* re;
  uint32_t* tau;               // [R] threshold keys (written)
  uint32_t* cand_key;          // [R, ROW_SLOTS]
  int32_t* cand_idx;
  int32_t* failed_rows;        // [R] (appended, count in stats->fail_count)
  int32_t* out;                // [R, K]
  Stats* stats;
  int parts;                   // items per row: 1 (whole rows) or 2 (half rows)
  int* half_count;             // half rows: [R, 2] candidates of each half of a row
  int* row_ticket;             // half rows: [R] halves streamed (zeroed by the plan)
};

// A kernel launch with programmatic stream serialisation (the kernels open
// with pdl_enter()); returns the launch's error.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Sparse-attention decode over the indexer's slots (sparse_attn.cu): grid
// (H / 16, T, splits); each split of a token's key list leaves an
// unnormalised partial output and its (max, sum) for the merge kernel, or,
// with one split, the result.
struct SparseAttnParams {
  const __nv_bfloat16* q_nope;  // [T, H, 512]
  const __nv_bfloat16* q_pe;    // [T, H, 64]
  const __nv_bfloat16* ckv;     // [num_slots, 512]
  const __nv_bfloat16* kpe;     // [num_slots, 64]
  const int32_t* idx;           // [T, K] slots (-1: padding)
  int T, H, K, num_slots;
  float scale_log2;             // sm_scale * log2(e)
  int splits, keys_per_split;
  float* part_o;                // [splits, T, H, 512]
  float2* part_ml;              // [splits, T, H]: running max (base-2 units) and sum
  __nv_bfloat16* out;           // [T, H, 512]
  float* lse;                   // [T, H]
  int* status;                  // ST_RANGE: a slot >= num_slots was named (read as padding)
};

// One bit per device (0..63) for a per-device, once-only host action.
struct DeviceFlags {
  std::atomic<uint64_t> bits{0};
};

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device: the attribute belongs to the device's context, so a process
// that calls the library on several GPUs sets it on each (devices past 63
// set it on every launch).  Two threads setting it at once is harmless.
template <typename... KArgs>
inline cudaError_t set_smem_attr_once(void (*kernel)(KArgs...), int bytes, DeviceFlags& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.bits.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.bits.fetch_or(bit, std::memory_order_release);
  return e;
}

// host launchers (return cudaGetLastError() of the launch)
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);
cudaError_t launch_sample(const CUtensorMap& tm_q, const SampleParams& p, int n_pairs, cudaStream_t s);
cudaError_t launch_sample_prep(const SamplePrepParams& p, cudaStream_t s);
cudaError_t launch_sample_tau(const SampleTauParams& p, cudaStream_t s);
cudaError_t launch_score(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const ScoreParams& p, int grid,
                         cudaStream_t s);
cudaError_t launch_select(const SelectParams& p, int grid, cudaStream_t s);
cudaError_t launch_cand_select(const CandParams& p, int sms, cudaStream_t s);  // grid: a few CTAs per SM
cudaError_t launch_wide_select(const WideParams& p, int clusters, cudaStream_t s);
cudaError_t launch_matrix_filter(const MatrixFilterParams& p, int grid, cudaStream_t s);
cudaError_t launch_matrix_topk(const MatrixTopkParams& p, int sms, cudaStream_t s);  // grid: CTAs of one wave, at most R
cudaError_t launch_sparse_attn(const SparseAttnParams& p, cudaStream_t s);
int sparse_attn_ctas_per_sm();  // CTAs of the sparse-attention kernel resident per SM

// number of work groups of G query rows for a row space
template <int G>
__host__ __device__ inline int n_row_groups(const RowSpace& rs) {
  if (!rs.paged) return (rs.R + G - 1) / G;
  const int per = (rs.next_n + G - 1) / G;
  return (rs.R / rs.next_n) * per;
}
__host__ __device__ inline int n_groups(const RowSpace& rs) { return n_row_groups<GROUP_ROWS>(rs); }
__host__ __device__ inline int n_pairs(const RowSpace& rs) { return n_row_groups<SAMPLE_ROWS>(rs); }

}  // namespace dsa
