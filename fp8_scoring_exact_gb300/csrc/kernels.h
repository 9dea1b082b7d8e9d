// kernels.h -- parameter blocks and launchers of the indexer kernels
// (internal to the library; the public ABI is include/dsa_indexer.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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
};

// chunk size that makes every work unit a whole row pair (tiles per row < 2^24)
constexpr int WHOLE_PAIR_TILES = 1 << 24;

struct PlanParams {
  RowSpace rs;
  int repair;                  // 0: plan every row; 1: plan the rows queued for repair
  int K;
  int trivial_len;             // rows with L <= trivial_len are not scored
  int chunk_tiles;
  const int32_t* row_begin_in; // dense input ranges
  const int32_t* row_end_in;
  int32_t* rb;                 // [R] validated ranges (written in main mode)
  int32_t* re;
  Group* groups;               // [G]
  int32_t* unit_start;         // [G + 1]
  int32_t* group_done;         // [G]
  int32_t* cand_count;         // [R]
  const int32_t* failed_rows;  // repair mode input
  Stats* stats;
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
  uint32_t* tau;               // [R] threshold keys (written)
  int32_t* out;                // [R, K] (trivial rows written here)
  Stats* stats;
};

struct ScoreParams {
  RowSpace rs;
  int mode;                    // MODE_STORE or MODE_FILTER
  int K;
  int chunk_tiles;
  int repair;                  // which plan to read
  int relu_alu8;               // heads (of every 8) whose ReLU uses the ALU pipe
  const float* q_scale;
  const float* w;
  const int32_t* rb;
  const int32_t* re;
  const Group* groups;
  const int32_t* unit_start;
  // MODE_FILTER
  const uint32_t* tau;
  uint32_t* cand_key;          // [R, CAND_CAP]
  int32_t* cand_idx;           // [R, CAND_CAP]
  int32_t* cand_count;         // [R]
  int32_t* group_done;         // [G]
  int32_t* failed_rows;        // [R]
  int32_t* out;                // [R, K]
  // MODE_STORE
  float* scores;               // [slots, ld]
  int64_t ld;
  Stats* stats;
};

enum SelectSource : int { SELECT_FROM_SCORES = 0, SELECT_FROM_CANDIDATES = 1 };

struct SelectParams {
  RowSpace rs;
  int K;
  int target16;
  int source;                  // SelectSource
  int list_mode;               // 1: rows = failed_rows[0 .. stats->fail_count), score row f
  const int32_t* list;
  // SELECT_FROM_CANDIDATES
  const uint32_t* cand_key;    // [R, CAND_CAP]
  const int32_t* cand_idx;
  const int32_t* cand_count;
  int32_t* failed_rows;
  const float* scores;
  int64_t ld;
  const int32_t* rb;
  const int32_t* re;
  int32_t* out;
  Stats* stats;
};

// host launchers (return cudaGetLastError() of the launch)
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);
cudaError_t launch_sample(const CUtensorMap& tm_q, const SampleParams& p, int n_pairs, cudaStream_t s);
cudaError_t launch_score(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_ks,
                         const ScoreParams& p, int grid, cudaStream_t s);
cudaError_t launch_select(const SelectParams& p, int grid, cudaStream_t s);

// number of query-row pairs (work groups) for a row space
__host__ __device__ inline int n_pairs(const RowSpace& rs) {
  if (!rs.paged) return (rs.R + 1) / 2;
  const int per = (rs.next_n + 1) / 2;
  return (rs.R / rs.next_n) * per;
}

}  // namespace dsa
