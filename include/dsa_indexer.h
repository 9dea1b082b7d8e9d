/*
 * dsa_indexer.h -- C ABI of the GB300 (sm_103a) DeepSeek-V3.2 DSA indexer with
 * exact top-K selection.
 *
 * Operation ("Fusing Indexer Scoring and Exact Top-k for DeepSeek-V3.2",
 * section 1.1 equation and section 2.3 problem definition): for every query
 * row t and every valid key s in [row_begin[t], row_end[t])
 *
 *     I[t, s] = sum_{j=0..63} w[t, j] * ReLU( (q_scale[t] * q[t, j, :]) . (k_scale[s] * k[s, :]) )
 *
 * with q and k FP8 e4m3 codes (64 heads x 128 dims; keys shared by all heads),
 * and return the K valid key indices with the largest I[t, s].
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers of the current CUDA device, owned by
 *     the caller, C-contiguous, row-major, and must stay valid until the work
 *     enqueued on `stream` has finished.  The library keeps no pointer to them
 *     after the call returns.
 *   - FP8 arrays and float scale arrays must be 16-byte aligned (the library
 *     reads them with the Tensor Memory Accelerator); any cudaMalloc or torch
 *     allocation is.
 *   - Output rows are unordered (section 2.3).  A row with L = end - begin
 *     valid keys and L >= K gets exactly K distinct indices of valid keys whose
 *     scores are the K largest (ties resolve to any valid index).  A row with
 *     L < K gets its L valid indices in slots [0, L) and -1 in slots [L, K).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream); no entry point except dsa_indexer_last_device_status()
 *     synchronises the host.  Argument errors are returned synchronously
 *     before anything is enqueued.  Errors the device detects (a row range
 *     outside [0, N], a pipeline wait that timed out) are recorded in a
 *     per-stream status word read by dsa_indexer_last_device_status().
 *   - The library owns per-(device, stream) scratch memory (plan, thresholds,
 *     candidate buffers, repair scores), allocated on first use and grown on
 *     demand; growing synchronises the device once.  Calls on the same stream
 *     are serialised by the stream; calls on different streams use different
 *     scratch.  The scratch is released by dsa_indexer_release() or at exit.
 *   - Fixed geometry: 64 heads, head dimension 128 (section 2.3); 1 <= K <=
 *     DSA_MAX_K.
 *
 * Return values: DSA_OK (0) or a negative dsa_status.
 */
#ifndef DSA_INDEXER_H
#define DSA_INDEXER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

struct CUstream_st;
typedef struct CUstream_st* dsa_stream_t; /* identical to cudaStream_t */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_ARG = -1,          /* null pointer, non-positive size, misaligned pointer, K out of range */
  DSA_ERR_UNSUPPORTED = -2,  /* a size beyond what the kernels address (e.g. N >= 2^31 / 128) */
  DSA_ERR_CUDA = -3,         /* a CUDA runtime call failed (no device, launch failure, out of memory) */
  DSA_ERR_TIMEOUT = -4,      /* device status: a bounded pipeline wait gave up (kernel returned early) */
  DSA_ERR_RANGE = -5         /* device status: some row range was outside [0, N] (that row got all -1), or a
                                used block-table entry was outside [0, num_pages) (that sequence's rows are
                                undefined: the bad page reads as zeros, its slots as -1 or out of range) */
} dsa_status;

#define DSA_HEADS 64
#define DSA_HEAD_DIM 128
#define DSA_MAX_K 2048

/*
 * Fused operator (sections 3.2 and 4 of the indexer study): sampled
 * threshold per row, tcgen05 FP8 scoring with the ReLU / weight / head
 * reduction applied on chip, compare-and-append of candidates, four-pass radix
 * select of each row's candidates, certificate check, and exact repair of rows
 * whose candidate set underflowed or overflowed.  The [Q, N] score matrix is
 * never written (only the repaired rows' scores are, in library scratch).
 *
 *   q_fp8     [Q, 64, 128] e4m3 codes           q_scale [Q]  fp32 (> 0)
 *   k_fp8     [N, 128]     e4m3 codes           k_scale [N]  fp32 (> 0)
 *   w         [Q, 64]      fp32 head weights
 *   row_begin, row_end [Q] int32, 0 <= row_begin[t] <= row_end[t] <= N
 *   out_idx   [Q, K]       int32 (written)
 */
DSA_API int dsa_indexer_topk(const uint8_t* q_fp8, const float* q_scale,
                     const uint8_t* k_fp8, const float* k_scale,
                     const float* w,
                     const int32_t* row_begin, const int32_t* row_end,
                     int Q, int N, int K,
                     int32_t* out_idx, dsa_stream_t stream);

/*
 * The fused operator of dsa_indexer_topk on HOST buffers (every array
 * argument is host memory, same layouts and meaning): the library copies the
 * inputs to device staging it owns, runs the fused operator over chunks of
 * rows, and copies the indices back into out_idx.  Rows are independent, so
 * the chunks give the same result as one call; while one chunk is scored on
 * `stream`, an internal copy stream brings in the next chunk's rows and takes
 * out the previous chunk's indices.  Rows per chunk: DSA_OPT_HOST_CHUNK_ROWS,
 * by default half of Q but at least 2048 rows.
 *
 * Synchronous: returns when out_idx holds the result.  Return value: DSA_OK,
 * an argument error (nothing enqueued), DSA_ERR_CUDA, or the device status of
 * the call (DSA_ERR_RANGE or DSA_ERR_TIMEOUT, combined over all chunks).
 * Host buffers in page-locked memory (cudaHostAlloc / pinned) let the copies
 * overlap the scoring; pageable buffers work but serialise them.  The device
 * staging (keys, two row chunks) is allocated on the first call and grown on
 * demand, per (device, stream).  Host-buffer calls are serialised within a
 * process.  dsa_indexer_last_device_status and dsa_indexer_last_repaired_rows
 * describe the last chunk only (repaired row ids relative to that chunk).
 */
DSA_API int dsa_indexer_topk_host(const uint8_t* q_fp8, const float* q_scale,
                          const uint8_t* k_fp8, const float* k_scale,
                          const float* w,
                          const int32_t* row_begin, const int32_t* row_end,
                          int Q, int N, int K,
                          int32_t* out_idx, dsa_stream_t stream);

/*
 * Paged variant (contest write-up, "DSA TopK Indexer"): keys in a cache of
 * 64-token pages with one fp32 scale per token; logical token s of sequence b
 * lives in physical slot block_table[b][s / 64] * 64 + s % 64.  Query row i of
 * sequence b (next_n query tokens per sequence) sees logical keys
 * [0, seq_lens[b] - next_n + i + 1).  Returned indices are PHYSICAL slots.
 * Rows with at most K valid keys take the index-remapping path (no scoring).
 *
 *   q_fp8         [B, next_n, 64, 128] e4m3     q_scale [B, next_n] fp32
 *   k_cache       [P, 64, 128] e4m3             k_cache_scale [P, 64] fp32
 *   w             [B, next_n, 64] fp32
 *   block_table   [B, max_pages] int32 (entries past a sequence's pages unused)
 *   seq_lens      [B] int32, 0 <= seq_lens[b] <= max_pages * 64
 *   num_pages     P (bounds every block_table entry that is used)
 *   out_idx       [B, next_n, K] int32 (written)
 *
 * A used block_table entry (entry s / 64 of a key s the sequence's rows see)
 * outside [0, P) is never followed: the page reads as zeros and the call's
 * device status reports DSA_ERR_RANGE; that sequence's rows are undefined,
 * every other sequence is unaffected.
 */
DSA_API int dsa_indexer_topk_paged(const uint8_t* q_fp8, const float* q_scale,
                           const uint8_t* k_cache, const float* k_cache_scale,
                           const float* w,
                           const int32_t* block_table, const int32_t* seq_lens,
                           int B, int next_n, int max_pages, int num_pages, int K,
                           int32_t* out_idx, dsa_stream_t stream);

/*
 * Unfused attribution baseline (section 1.1, "the usual implementation"):
 * the same tcgen05 scorer writes the FP32 score matrix [Q, N] to device memory
 * (entries of a touched tile outside the row's range hold -inf; other entries
 * are not written), then the standalone exact top-K of section 3 reads it
 * back.  Same arguments and result contract as dsa_indexer_topk.
 */
DSA_API int dsa_indexer_topk_unfused(const uint8_t* q_fp8, const float* q_scale,
                             const uint8_t* k_fp8, const float* k_scale,
                             const float* w,
                             const int32_t* row_begin, const int32_t* row_end,
                             int Q, int N, int K,
                             int32_t* out_idx, dsa_stream_t stream);

/*
 * Scores only: scores[t, s] = I[t, s] in fp32 for s in [row_begin[t],
 * row_end[t]) of every row; other entries of the 128-key tiles the row touches
 * hold -inf; the rest of the row is left untouched.  scores is [Q, ld] fp32,
 * ld >= N, ld % 4 == 0.
 */
DSA_API int dsa_indexer_scores(const uint8_t* q_fp8, const float* q_scale,
                       const uint8_t* k_fp8, const float* k_scale,
                       const float* w,
                       const int32_t* row_begin, const int32_t* row_end,
                       int Q, int N, float* scores, int64_t ld, dsa_stream_t stream);

/*
 * Standalone exact top-K over a given fp32 score matrix (section 3: each
 * row's threshold from a sample of its own scores, compare-and-append of the
 * scores at or above it, exact selection of those candidates with a
 * certificate, and a full-row radix select for the rows that fail it).  From
 * a third of a row per SM on, CTAs take whole or half rows and select each
 * row as its last part is streamed, so the matrix is read once; fewer rows
 * are split over the SMs.  Row t considers
 * scores[t, s] for s in [row_begin[t], row_end[t]) and returns the indices s.
 * NaN scores are not supported.  scores is [Q, ld] fp32.
 */
DSA_API int dsa_indexer_topk_from_scores(const float* scores, int64_t ld,
                                 const int32_t* row_begin, const int32_t* row_end,
                                 int Q, int N, int K,
                                 int32_t* out_idx, dsa_stream_t stream);

/*
 * Same operation and result as dsa_indexer_topk_from_scores, but this entry
 * point allocates no memory at all, for callers that cannot call cudaMalloc:
 * an embedding runtime that owns every device allocation and forbids others
 * (a serving engine that reserves all free memory for its KV cache at start-up
 * and accounts for every byte), or a plugin host whose memory budget is fixed
 * before this library is loaded.
 * The paper has no counterpart; it is a deployment convenience.
 *
 * Its scratch is one fixed device array of 512 KiB compiled into this
 * library; every GPU that loads the library holds it until the process
 * exits.  Limits: Q <= 4096 rows (larger Q returns DSA_ERR_UNSUPPORTED and
 * enqueues nothing).  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before
 * any stream capture on that device.  Every call resets the parts of the
 * array it reads, but all calls share the one array: calls that may overlap
 * on the GPU (on different streams, or from different threads without
 * ordering) race and must be serialised by the caller.  Calls to this entry
 * point are not reported by dsa_indexer_last_device_status(): a row whose
 * range lies outside [0, N] (or has begin > end) comes back as K entries of
 * -1, exactly like an empty row, and nothing else signals it; callers that
 * cannot vouch for their ranges validate them before the call.
 */
DSA_API int dsa_indexer_topk_from_scores_noalloc(const float* scores, int64_t ld,
                                                 const int32_t* row_begin, const int32_t* row_end,
                                                 int Q, int N, int K,
                                                 int32_t* out_idx, dsa_stream_t stream);

/*
 * Sparse-attention decode over the indexer's result (contest write-up, "DSA
 * Sparse Attention"), the step that consumes the top-K slots: for every query
 * token t and head h, with u_j = sm_scale * log2(e) * (q_nope[t, h] .
 * ckv[i_j] + q_pe[t, h] . kpe[i_j]) over the slots i_j listed in
 * indices[t, :] (negative entries are padding),
 *
 *     out[t, h] = sum_j 2^(u_j) ckv[i_j] / sum_j 2^(u_j)       (base-2 softmax)
 *     lse[t, h] = log2(sum_j 2^(u_j))                       (-inf: no valid slot)
 *
 *   q_nope   [T, H, 512] bf16       q_pe [T, H, 64] bf16    (H a multiple of 16)
 *   ckv      [num_slots, 512] bf16  kpe  [num_slots, 64] bf16 (the compressed KV
 *            cache and its rope part, slot-major: for a paged cache of
 *            64-token pages, slot = page * 64 + offset, as the paged indexer
 *            returns it)
 *   indices  [T, K] int32           out [T, H, 512] bf16    lse [T, H] fp32
 *
 * bf16 arrays are passed as their 16-bit patterns; they must be 16-byte
 * aligned.  Arithmetic: bf16 products accumulated in fp32, weights rounded
 * to bf16 for the weighted sum, output rounded to bf16.  A slot >= num_slots
 * is read as padding and reported by dsa_sparse_attention_last_status
 * (DSA_ERR_RANGE).  Scratch (split partials) is owned by the library per
 * (device, stream), grown on demand.
 */
DSA_API int dsa_sparse_attention(const uint16_t* q_nope, const uint16_t* q_pe,
                                 const uint16_t* ckv, const uint16_t* kpe,
                                 const int32_t* indices, int T, int H, int K, int num_slots,
                                 float sm_scale, uint16_t* out, float* lse, dsa_stream_t stream);

/* Synchronises `stream`; DSA_OK, or DSA_ERR_RANGE if the most recent
 * dsa_sparse_attention call on it met a slot outside [0, num_slots). */
DSA_API int dsa_sparse_attention_last_status(dsa_stream_t stream);

/*
 * Math-only control (a measurement, not an operator; section 5.2 of the
 * indexer study, "Math-only control"): the fused operator's plan and its main
 * scorer with the same work units, tile loads, tcgen05 MMAs and barriers, but
 * an epilogue that only reads one accumulator column per warp and tile, adds
 * it to a checksum and releases the accumulator: no ReLU, head reduction,
 * threshold, candidates or selection, and no sampled threshold before it.
 * Timing it against dsa_indexer_topk on the same inputs shows how much of
 * the main kernel's time the score reduction and candidate filter still
 * add.  Same arguments as dsa_indexer_topk; instead of indices it adds the
 * checksum (meaningless as a value) to *checksum (one device float).  With
 * DSA_OPT_PROFILE set, dsa_indexer_profiled_main_ms reports its scorer.
 */
DSA_API int dsa_indexer_math_control(const uint8_t* q_fp8, const float* q_scale,
                                     const uint8_t* k_fp8, const float* k_scale,
                                     const float* w,
                                     const int32_t* row_begin, const int32_t* row_end,
                                     int Q, int N, int K,
                                     float* checksum, dsa_stream_t stream);

/*
 * Synchronises `stream`, then reports the device status of the most recent
 * call enqueued on it: DSA_OK, DSA_ERR_TIMEOUT or DSA_ERR_RANGE (or
 * DSA_ERR_CUDA if synchronising failed).  failures_out (may be NULL) receives
 * 4 counters of that call: rows repaired after candidate underflow, rows
 * repaired after candidate overflow, rows taken by the remapping path
 * (L <= K), and the total number of candidates appended.
 */
DSA_API int dsa_indexer_last_device_status(dsa_stream_t stream, int32_t* failures_out);

/*
 * Synchronises `stream` and copies the ids of the rows that the most recent
 * selecting call on it (fused, unfused or dsa_indexer_topk_from_scores) sent
 * to exact repair (certificate failed) into rows_out (at most `cap` of them,
 * in no particular order).  Returns their number (>= 0) or a negative
 * dsa_status.
 */
DSA_API int dsa_indexer_last_repaired_rows(dsa_stream_t stream, int32_t* rows_out, int cap);

/* Tuning and diagnostics (process-wide; take effect on the next call). */
typedef enum {
  DSA_OPT_CHUNK_TILES = 1,    /* 128-key tiles per work unit of the persistent scorer (default -1: chosen per
                                 call, 64 dense / 32 paged, halved down to 16 while there would be fewer than
                                 4 units per SM); a row's
                                 16384 candidate slots are split evenly over its units' regions, and a region
                                 that fills up fails the row's certificate (-> repair) */
  DSA_OPT_TAU_BIAS = 2,       /* added to every sampled threshold key: >0 forces underflow, <0 overflow (test knob; default 0) */
  DSA_OPT_PROFILE = 3,        /* 1: time the main kernel of each call with CUDA events (default 0) */
  DSA_OPT_GRID_CTAS = 4,      /* CTAs of the persistent kernels (default: SM count) */
  DSA_OPT_SAMPLE_TARGET = 5,  /* candidates the threshold aims at, in units of K/16 (default 36 = 2.25K) */
  DSA_OPT_HOST_CHUNK_ROWS = 6, /* rows per chunk of dsa_indexer_topk_host (default 0: chosen per call) */
  DSA_OPT_UNIT_ORDER = 7,      /* order the scorer's work units are handed out in: 0 plan order (default),
                                  1 last first; the result does not depend on it (test option) */
  DSA_OPT_WAIT_LIMIT_US = 8,   /* microseconds after which a pipeline wait inside a kernel gives up (default
                                  2000000, range 1..60000000): the kernel then lets the copies and MMAs it
                                  already issued land, returns early, and the call reports DSA_ERR_TIMEOUT */
  DSA_OPT_TEST_WITHHOLD = 9,   /* test option: 1 makes the fused operator's main scorer never signal its first
                                  accumulator, so that its epilogue's wait runs out after DSA_OPT_WAIT_LIMIT_US
                                  and the call reports DSA_ERR_TIMEOUT (its output is then undefined); default 0 */
  DSA_OPT_MATRIX_ROW_MIN = 10  /* dsa_indexer_topk_from_scores and the unfused operator's selection: rows from
                                  which CTAs take whole rows, or half rows when there are many long ones
                                  (threshold, one pass over the row, selection by the CTA that finishes the
                                  row), instead of splitting rows over the SMs (default -1: chosen per call,
                                  a third of a row per SM; 0: always; the result does not depend on it) */
} dsa_option;
DSA_API int dsa_indexer_set_option(int option, int64_t value);
DSA_API int64_t dsa_indexer_get_option(int option);

/* Milliseconds spent in the main kernel of the most recent profiled call on
 * `stream` (synchronises the stream); -1 if none was profiled. */
DSA_API float dsa_indexer_profiled_main_ms(dsa_stream_t stream);

/* Number of kernels this process has launched through the library. */
DSA_API int64_t dsa_indexer_launch_count(void);

/* Library version string and the compute capability it was built for. */
DSA_API const char* dsa_indexer_version(void);

/* Frees all scratch memory the library holds (synchronises the device). */
DSA_API int dsa_indexer_release(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_INDEXER_H */
