// sparse_attn.cu -- sparse-attention decode over the indexer's top-K slots.
//
// For each query token t and head h (contest write-up, "DSA Sparse
// Attention"): gather the KV entries the token's index list names, logits
// z_j = q_nope . ckv[i_j] + q_pe . kpe[i_j], a base-2 softmax of
// u_j = z_j * sm_scale * log2(e), out = sum_j p_j ckv[i_j] (512 dims) and
// lse = log2(sum_j 2^u_j).
//
// The step is bound by the gather (2048 rows x 1152 bytes per token, read
// once for all of the token's heads: ~30 FLOP per byte), so the contraction
// runs on warp-level bf16 tensor-core MMAs (m16n8k16, fp32 accumulation),
// which keep the arithmetic well below the gather time, with the token's 16
// heads as the MMA's M dimension.
//
// One CTA (8 warps) per (token, block of 16 heads, split of the key list):
//   - the 16 query rows (q_nope | q_pe, 576 dims) are loaded once; warp w
//     keeps the A fragments of dims [144 (w % 4), + 144) in registers;
//   - key tiles of 32 slots are gathered with cp.async (16 bytes per copy):
//     warp w copies rows 4w .. 4w + 3, its lanes consecutive 16-byte chunks
//     of each 1152-byte row (ckv, then kpe), a padding slot's row zero-filled,
//     into a ring of SA_STAGES shared tiles, SA_STAGES - 1 gathers in
//     flight while a tile is processed (measured: 32-key tiles in a 2-deep
//     ring, two CTAs per SM, beat 16-key tiles or deeper rings with one CTA
//     per SM; bulk copies of whole rows by one warp were slower);
//   - QK: warp w multiplies its 144 dims for its 16 keys (key half w / 4;
//     partial logits to shared memory), then all 256 threads sum the 4
//     partials, apply the running (online) max and sums of the base-2
//     softmax per head, and write the tile's weights as bf16;
//   - PV: warp w owns output dims [64 w, 64 w + 64): its accumulators are
//     rescaled by 2^(m_old - m_new) (skipped when no head's maximum moved)
//     and take the tile's weights times the tile's ckv rows
//     (ldmatrix.trans).
// (Measured: 8 warps per CTA in this split beat 4 warps with each warp
// covering all keys / 128 output dims; the 4-warp kernel had 8 warps per SM
// and stalled on its barriers and MMA chains.)
// Splits of one token's key list are merged by a second kernel (running max,
// rescaled sums); a single split writes the result directly.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace dsa {

namespace {

constexpr int SA_DC = 512;                 // compressed KV dims (output)
constexpr int SA_DP = 64;                  // rope dims
constexpr int SA_DQ = SA_DC + SA_DP;       // 576
constexpr int SA_HB = 16;                  // heads per CTA (MMA M)
constexpr int SA_TK = 32;                  // keys per tile
#ifndef DSA_SA_STAGES
#define DSA_SA_STAGES 2
#endif
constexpr int SA_STAGES = DSA_SA_STAGES;   // gathered tiles in the ring
constexpr int SA_CTAS_PER_SM = SA_STAGES <= 2 ? 2 : 1;
constexpr int SA_WARPS = 8;
constexpr int SA_THREADS = 32 * SA_WARPS;
constexpr int SA_PVN = SA_DC / SA_WARPS / 8;  // output n-blocks (8 dims) per warp
static_assert(SA_TK == 32 && SA_HB * SA_TK == 2 * SA_THREADS, "2 key halves x 4 dim groups; 2 keys per softmax thread");
constexpr int SA_ROW = SA_DQ + 8;          // shared row stride (bf16): 1168 bytes, ldmatrix without conflicts
constexpr int SA_CHUNKS = SA_DQ * 2 / 16;  // 16-byte copies per row: 72
constexpr int SA_SROW = SA_TK + 8;         // partial-logit row stride (floats): float2 stores without conflicts
constexpr int SA_PROW = SA_TK + 8;         // weight row stride (bf16): 80 bytes, ldmatrix without conflicts

constexpr uint32_t SA_OFF_Q = 0;
constexpr uint32_t SA_OFF_KV = SA_OFF_Q + SA_HB * SA_ROW * 2;               // 18688
constexpr uint32_t SA_KV_BYTES = SA_TK * SA_ROW * 2;                        // 37376
constexpr uint32_t SA_OFF_S = SA_OFF_KV + SA_STAGES * SA_KV_BYTES;
constexpr uint32_t SA_OFF_P = SA_OFF_S + 4 * SA_HB * SA_SROW * 4;
constexpr uint32_t SA_OFF_STAT = SA_OFF_P + SA_HB * SA_PROW * 2;
constexpr uint32_t SA_OFF_IDX = SA_OFF_STAT + 3 * SA_HB * 4;                // m, l, alpha per head
constexpr int SA_MAX_PER = 2048;           // slots of one split, loaded into shared memory at the start
constexpr uint32_t SA_SMEM = SA_OFF_IDX + SA_MAX_PER * 4;
static_assert((SA_ROW * 2) % 16 == 0 && SA_TK == 4 * SA_WARPS, "rows aligned; 4 rows per warp");
static_assert(SA_OFF_KV % 16 == 0 && SA_OFF_S % 16 == 0 && SA_OFF_P % 16 == 0, "sparse attention layout");
static_assert(SA_SMEM * SA_CTAS_PER_SM <= 226 * 1024, "shared memory per SM");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float exp2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
}  // namespace

__global__ void __launch_bounds__(SA_THREADS, SA_CTAS_PER_SM) sparse_attn_kernel(const SparseAttnParams p) {
  pdl_enter();
  extern __shared__ __align__(16) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  float* sS = reinterpret_cast<float*>(smem + SA_OFF_S);
  __nv_bfloat16* sP = reinterpret_cast<__nv_bfloat16*>(smem + SA_OFF_P);
  float* sM = reinterpret_cast<float*>(smem + SA_OFF_STAT);
  float* sL = sM + SA_HB;
  float* sA = sL + SA_HB;
  int* sSlot = reinterpret_cast<int*>(smem + SA_OFF_IDX);  // this split's slots, -1 past its end

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hb = blockIdx.x, t = blockIdx.y, split = blockIdx.z;
  const int H = p.H, K = p.K;
  const int j_begin = split * p.keys_per_split;
  const int j_end = min(K, j_begin + p.keys_per_split);
  const int n_tiles = j_end > j_begin ? ceil_div(j_end - j_begin, SA_TK) : 0;
  const int32_t* idx_row = p.idx + (int64_t)t * K;
  const int64_t qrow0 = (int64_t)t * H + hb * SA_HB;  // first (token, head) row of this CTA

  // query rows: 16 x (512 + 64) bf16
  for (int c = tid; c < SA_HB * SA_CHUNKS; c += SA_THREADS) {
    const int r = c / SA_CHUNKS, k = c % SA_CHUNKS;
    const void* src = k < SA_DC / 8 ? (const void*)(p.q_nope + (qrow0 + r) * SA_DC + 8 * k)
                                    : (const void*)(p.q_pe + (qrow0 + r) * SA_DP + 8 * (k - SA_DC / 8));
    cp_async_16(sbase + SA_OFF_Q + (r * SA_ROW + 8 * k) * 2, src, 16);
  }
  // this split's slots into shared memory once (-1: padding, past the list,
  // or a slot outside the cache, which is reported): the gathers then take
  // their rows' slots from there instead of waiting on global loads
  for (int i = tid; i < n_tiles * SA_TK; i += SA_THREADS) {
    const int j = j_begin + i;
    int sl = j < j_end ? __ldg(&idx_row[j]) : -1;
    if (sl >= p.num_slots) {
      atomicOr(p.status, ST_RANGE);
      sl = -1;
    }
    sSlot[i] = sl;
  }
  __syncthreads();
  // tile i into buffer b: warp w copies rows 4w .. 4w + 3 (a padding slot's
  // row zero-filled), its lanes consecutive 16-byte chunks of each row
  auto gather = [&](int i, int b) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int sr = sSlot[i * SA_TK + 4 * warp + rr];
      const int64_t slot = sr < 0 ? 0 : sr;
      const int n = sr < 0 ? 0 : 16;
      const uint32_t dst = sbase + SA_OFF_KV + b * SA_KV_BYTES + (4 * warp + rr) * SA_ROW * 2 + 16 * lane;
      const uint8_t* ck = reinterpret_cast<const uint8_t*>(p.ckv + slot * SA_DC) + 16 * lane;
      cp_async_16(dst, ck, n);
      cp_async_16(dst + 512, ck + 512, n);
      if (lane < 8) cp_async_16(dst + 1024, reinterpret_cast<const uint8_t*>(p.kpe + slot * SA_DP) + 16 * lane, n);
    }
  };
  if (tid < SA_HB) {
    sM[tid] = -__int_as_float(0x7f800000);
    sL[tid] = 0.f;
  }
  // prologue: the first SA_STAGES - 1 tiles (one commit group each, the
  // query rows in the first; empty groups past the end keep the count uniform)
#pragma unroll
  for (int i = 0; i < SA_STAGES - 1; ++i) {
    if (i < n_tiles) gather(i, i);
    cp_async_commit();
  }

  // warp w: logit dims [144 (w % 4), + 144) for keys [16 (w / 4), + 16) of
  // each tile; output dims [64 w, 64 w + 64) (8 n-blocks of 8)
  const int kd0 = (warp & 3) * 144;
  const int kh = warp >> 2;
  float acc[SA_PVN][4];
#pragma unroll
  for (int i = 0; i < SA_PVN; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  uint32_t qa[9][4];  // this warp's 9 k-steps of the query rows (A fragments)

  for (int it = 0; it < n_tiles; ++it) {
    const int b = it % SA_STAGES;
    cp_async_wait<SA_STAGES - 2>();
    __syncthreads();  // tile `it` landed for every thread; the previous tile's readers are done
    if (it == 0) {
#pragma unroll
      for (int ks = 0; ks < 9; ++ks) {
        const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int col = kd0 + 16 * ks + 8 * (lane >> 4);
        ldsm_x4(sbase + SA_OFF_Q + (row * SA_ROW + col) * 2, qa[ks]);
      }
    }
    // refill the buffer the previous tile used
    if (it + SA_STAGES - 1 < n_tiles) gather(it + SA_STAGES - 1, (it + SA_STAGES - 1) % SA_STAGES);
    cp_async_commit();

    // ---- partial logits over this warp's 144 dims: 16 heads x its 16 keys
    const uint32_t kv = sbase + SA_OFF_KV + b * SA_KV_BYTES;
    float s[2][4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
      const int krow = 16 * kh + 8 * nb + (lane & 7);
#pragma unroll
      for (int ks2 = 0; ks2 < 4; ++ks2) {  // k-steps 2 ks2, 2 ks2 + 1
        uint32_t bf[4];
        ldsm_x4(kv + (krow * SA_ROW + kd0 + 32 * ks2 + 8 * (lane >> 3)) * 2, bf);
        mma_bf16(s[nb], qa[2 * ks2], bf[0], bf[1]);
        mma_bf16(s[nb], qa[2 * ks2 + 1], bf[2], bf[3]);
      }
      uint32_t bf[2];
      ldsm_x2(kv + (krow * SA_ROW + kd0 + 128 + 8 * ((lane >> 3) & 1)) * 2, bf);
      mma_bf16(s[nb], qa[8], bf[0], bf[1]);
    }
    {
      float* sw = sS + (warp & 3) * SA_HB * SA_SROW + 16 * kh;
      const int r0 = lane >> 2, c0 = 2 * (lane & 3);
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        *reinterpret_cast<float2*>(&sw[r0 * SA_SROW + 8 * nb + c0]) = make_float2(s[nb][0], s[nb][1]);
        *reinterpret_cast<float2*>(&sw[(r0 + 8) * SA_SROW + 8 * nb + c0]) = make_float2(s[nb][2], s[nb][3]);
      }
    }
    __syncthreads();

    // ---- online base-2 softmax: thread (head h = tid / 16, keys 2 kq, 2 kq + 1)
    {
      const int h = tid >> 4, kq = tid & 15;
      float u[2];
      {
        float2 a = *reinterpret_cast<const float2*>(&sS[(0 * SA_HB + h) * SA_SROW + 2 * kq]);
#pragma unroll
        for (int w = 1; w < 4; ++w) {
          const float2 x = *reinterpret_cast<const float2*>(&sS[(w * SA_HB + h) * SA_SROW + 2 * kq]);
          a.x += x.x;
          a.y += x.y;
        }
        const int* si = sSlot + it * SA_TK + 2 * kq;
        u[0] = si[0] >= 0 ? a.x * p.scale_log2 : -__int_as_float(0x7f800000);
        u[1] = si[1] >= 0 ? a.y * p.scale_log2 : -__int_as_float(0x7f800000);
      }
      float tmax = fmaxf(u[0], u[1]);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_old = sM[h];
      const float m_new = fmaxf(m_old, tmax);
      const float m_use = m_new == -__int_as_float(0x7f800000) ? 0.f : m_new;
      // weights rounded to bf16 for the PV product; the sums use the
      // rounded values, so the normalisation matches what is accumulated
      const __nv_bfloat162 w2 = __floats2bfloat162_rn(exp2_approx(u[0] - m_use), exp2_approx(u[1] - m_use));
      const float2 f2 = __bfloat1622float2(w2);
      float psum = f2.x + f2.y;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      *reinterpret_cast<__nv_bfloat162*>(sP + h * SA_PROW + 2 * kq) = w2;
      __syncwarp();
      if (kq == 0) {
        const float alpha = exp2_approx(m_old - m_use);  // 0 when m_old is -inf
        sA[h] = alpha;
        sL[h] = sL[h] * alpha + psum;
        sM[h] = m_new;
      }
    }
    __syncthreads();

    // ---- PV: this warp's 64 output dims, SA_TK / 16 key k-steps
    {
      const float a_lo = sA[lane >> 2], a_hi = sA[(lane >> 2) + 8];
      // once the running maxima settle, most tiles leave them unchanged
      if (!__all_sync(0xffffffffu, a_lo == 1.f && a_hi == 1.f)) {
#pragma unroll
        for (int nb = 0; nb < SA_PVN; ++nb) {
          acc[nb][0] *= a_lo;
          acc[nb][1] *= a_lo;
          acc[nb][2] *= a_hi;
          acc[nb][3] *= a_hi;
        }
      }
      const int d0 = warp * (SA_DC / SA_WARPS);
#pragma unroll
      for (int ks = 0; ks < SA_TK / 16; ++ks) {
        uint32_t pa[4];
        const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4(sbase + SA_OFF_P + (row * SA_PROW + 16 * ks + 8 * (lane >> 4)) * 2, pa);
        const int krow = 16 * ks + row;
#pragma unroll
        for (int nb2 = 0; nb2 < SA_PVN / 2; ++nb2) {
          uint32_t bf[4];
          ldsm_x4_t(kv + (krow * SA_ROW + d0 + 16 * nb2 + 8 * (lane >> 4)) * 2, bf);
          mma_bf16(acc[2 * nb2], pa, bf[0], bf[1]);
          mma_bf16(acc[2 * nb2 + 1], pa, bf[2], bf[3]);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- this split's result: rows r0 = lane / 4 and r0 + 8, dims
  // 64 warp + 8 nb + 2 (lane % 4) + {0, 1}
  const int r0 = lane >> 2;
  const int64_t ro0 = qrow0 + r0, ro1 = ro0 + 8;
  const int dbase = warp * (SA_DC / SA_WARPS) + 2 * (lane & 3);
  if (p.splits == 1) {
    const float l0 = sL[r0], l1 = sL[r0 + 8];
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int nb = 0; nb < SA_PVN; ++nb) {
      *reinterpret_cast<__nv_bfloat162*>(p.out + ro0 * SA_DC + dbase + 8 * nb) =
          __floats2bfloat162_rn(acc[nb][0] * i0, acc[nb][1] * i0);
      *reinterpret_cast<__nv_bfloat162*>(p.out + ro1 * SA_DC + dbase + 8 * nb) =
          __floats2bfloat162_rn(acc[nb][2] * i1, acc[nb][3] * i1);
    }
    if (tid < SA_HB) {
      const float l = sL[tid];
      p.lse[qrow0 + tid] = l > 0.f ? sM[tid] + __log2f(l) : -__int_as_float(0x7f800000);
    }
    return;
  }
  float* po = p.part_o + ((int64_t)split * p.T * H) * SA_DC;
#pragma unroll
  for (int nb = 0; nb < SA_PVN; ++nb) {
    *reinterpret_cast<float2*>(po + ro0 * SA_DC + dbase + 8 * nb) = make_float2(acc[nb][0], acc[nb][1]);
    *reinterpret_cast<float2*>(po + ro1 * SA_DC + dbase + 8 * nb) = make_float2(acc[nb][2], acc[nb][3]);
  }
  if (tid < SA_HB) p.part_ml[(int64_t)split * p.T * H + qrow0 + tid] = make_float2(sM[tid], sL[tid]);
}

// Merge of the splits of one (token, head): one warp, 16 dims per lane.
constexpr int SM_THREADS = 256;
__global__ void __launch_bounds__(SM_THREADS) sparse_attn_merge_kernel(const SparseAttnParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (SM_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t rows = (int64_t)p.T * p.H;
  if (row >= rows) return;
  float M = -__int_as_float(0x7f800000);
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, p.part_ml[s * rows + row].x);
  const float m_use = M == -__int_as_float(0x7f800000) ? 0.f : M;
  float L = 0.f;
  float o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float2 ml = p.part_ml[s * rows + row];
    const float w = exp2_approx(ml.x - m_use);  // 0 for a split with no valid key
    L += w * ml.y;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + (s * rows + row) * SA_DC + 16 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 x = __ldcs(src + i);
      o[4 * i] += w * x.x;
      o[4 * i + 1] += w * x.y;
      o[4 * i + 2] += w * x.z;
      o[4 * i + 3] += w * x.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(p.out + row * SA_DC + 16 * lane);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = __floats2bfloat162_rn(o[2 * i] * inv, o[2 * i + 1] * inv);
  if (lane == 0) p.lse[row] = L > 0.f ? M + __log2f(L) : -__int_as_float(0x7f800000);
}

int sparse_attn_ctas_per_sm() { return SA_CTAS_PER_SM; }

cudaError_t launch_sparse_attn(const SparseAttnParams& p, cudaStream_t s) {
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_attr_once(sparse_attn_kernel, SA_SMEM, attr_set);
  if (e != cudaSuccess) return e;
  e = launch_pdl(sparse_attn_kernel, dim3(p.H / SA_HB, p.T, p.splits), dim3(SA_THREADS), SA_SMEM, s, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t rows = (int64_t)p.T * p.H;
  return launch_pdl(sparse_attn_merge_kernel, dim3((unsigned)ceil_div((int)rows, SM_THREADS / 32)),
                    dim3(SM_THREADS), 0, s, p);
}

}  // namespace dsa
