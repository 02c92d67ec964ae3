// Skinny GEMMs of the sketch path on the 5th-generation tensor cores:
//   (b) XP = bf16(X P)        M = tokens, N = r, K = k       (A, B K-major)
//   (c) C (+)= D^T XP (fp32)  M = d,      N = r, K = tokens  (A, B MN-major)
// ("Randomized Gradient Compression", "How it works": the layer saves X P and
// accumulates C += D.T (X P); "LoGRA: Scaling LLM Reinforcement Learning with
// Low-Rank Gradient Sketches", Key Contributions 1: in fp32.)
//
// Both are HBM-bound streams of one BF16 operand (X or D) against a small,
// L2-resident second operand.  Design per CTA (128 threads):
//   * 128 output rows; the K range is split across a thread-block cluster of S
//     CTAs (S in 1..8), so a few M tiles still fill the GPU;
//   * warp 0 lane 0 streams 64-wide K chunks into a ring of shared-memory stages
//     with TMA (128-byte swizzle), completion counted on mbarriers;
//   * warp 1 lane 0 issues tcgen05.mma (M=128, N=r rounded to 16, K=16) into a
//     TMEM accumulator and releases each stage with tcgen05.commit;
//   * the four warps move the accumulator TMEM -> shared memory, then each CTA
//     of the cluster sums a 128/S-row slice of all S partial tiles through
//     distributed shared memory in a fixed order (deterministic, no atomics and
//     no global scratch) and writes its rows.
// XP = X P uses P split into BF16 high and low parts (P = hi + lo to 2^-17),
// summed by two MMAs into the same accumulator, so XP is fp32-accurate before
// its final rounding.  Every wait is bounded (tc.cuh) and sets the device error
// word instead of hanging.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace rgs {
namespace {

constexpr int kThreads = 128;
constexpr int kChunk = 64;  // K elements per pipeline stage (one 128-byte swizzle row)
constexpr int kMaxStages = 8;
constexpr int kAccStripTiles = 1;  // 128-row tiles of C per persistent accumulation item

// A launch covers up to kMaxProblems independent problems that share r (and so
// N): one GEMM per layer.  Their M tiles are laid end to end along grid.y.
constexpr int kMaxProblems = 96;

struct SkinnyBatch {
  CUtensorMap tmA[kMaxProblems];   // X (K-major) or D (MN-major) of each problem
  CUtensorMap tmB[kMaxProblems];   // P^T split [hi rows; lo rows] or XP
  void* out[kMaxProblems];
  int64_t ld_out[kMaxProblems];    // row stride of out, in elements
  int M[kMaxProblems];             // output rows
  int kchunks[kMaxProblems];       // 64-wide K chunks
  int tile_begin[kMaxProblems + 1];
  int n;                           // problems in this launch
  int N;                           // output columns (r)
  int n_pad;                       // MMA N: r rounded up to 16
  int stages;                      // pipeline depth
  uint32_t a_bytes;                // A tile bytes per stage (16 KB)
  uint32_t b_bytes;                // bytes of one B tile per stage
  uint32_t stage_bytes;            // a_bytes + NB * b_bytes
  int red_stride;                  // floats per row of the fp32 reduction tile
  uint32_t tmem_cols;              // power of two >= max(32, n_pad)
  int out_mode;                    // 0: BF16 round-to-nearest store; 1: fp32 store; 2: fp32 add;
                                   // 3: BF16 split store, hi in columns [0, N), lo at [n_pad, n_pad + N)
  int b_col_off;                   // MN-major B: column offset of B operand nb is nb * b_col_off
  int k_parts;                     // persistent projection: partial accumulators per tile (K ranges)
  int acc_bufs;                    // persistent projection: TMEM buffers (tiles in flight)
  int* err;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <bool A_MN, bool B_MN, int NB>
__global__ void __launch_bounds__(kThreads, 1) skinny_gemm_kernel(const __grid_constant__ SkinnyBatch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int issued, consumed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t S = gridDim.x;
  const uint32_t rank = (S > 1) ? tc::cluster_ctarank() : 0u;
  int p = 0;
  while (p + 1 < a.n && a.tile_begin[p + 1] <= (int)blockIdx.y) ++p;
  const CUtensorMap* tmA = &a.tmA[p];
  const CUtensorMap* tmB = &a.tmB[p];
  const int M = a.M[p];
  const int kchunks = a.kchunks[p];
  const int m0 = ((int)blockIdx.y - a.tile_begin[p]) * 128;
  const int c_begin = (int)((int64_t)kchunks * rank / S);
  const int c_end = (int)((int64_t)kchunks * (rank + 1) / S);
  const int nmine = c_end - c_begin;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued = 0;
    consumed = 0;
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    tc::mbar_init(&acc_bar, 1);
    tc::fence_mbar_init();
    tc::prefetch_tmap(tmA);
    tc::prefetch_tmap(tmB);
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, a.tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA ring ----
    int s = 0;        // stage of chunk i: i % stages, kept without a division
    uint32_t ph = 0;  // (i / stages) & 1
    for (int i = 0; i < nmine; ++i) {
      if (i >= a.stages && !tc::mbar_wait(&empty_bar[s], ph ^ 1u, &abort_flag, a.err, tc::kErrTimeoutStage))
        break;
      uint8_t* st = smem + (size_t)s * a.stage_bytes;
      tc::mbar_arrive_expect_tx(&full_bar[s], a.stage_bytes);
      const int kc = (c_begin + i) * kChunk;
      if (A_MN) {  // D: [64 tokens][64 rows of C] per box, two boxes for 128 rows
        tc::tma_load_2d(st, tmA, &full_bar[s], m0, kc);
        tc::tma_load_2d(st + 8192, tmA, &full_bar[s], m0 + 64, kc);
      } else {  // X: [128 tokens][64 k]
        tc::tma_load_2d(st, tmA, &full_bar[s], kc, m0);
      }
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        uint8_t* bt = st + a.a_bytes + nb * a.b_bytes;
        if (B_MN) {  // XP: [64 tokens][64 rank columns] per box
          for (int j = 0; j * 64 < a.n_pad; ++j)
            tc::tma_load_2d(bt + j * 8192, tmB, &full_bar[s], nb * a.b_col_off + j * 64, kc);
        } else {  // P^T split: [n_pad rank rows][64 k]; high part in rows [0, n_pad), low in [n_pad, 2 n_pad)
          tc::tma_load_2d(bt, tmB, &full_bar[s], kc, nb * a.n_pad);
        }
      }
      issued = i + 1;
      if (++s == a.stages) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = tc::idesc_bf16(128, a.n_pad, A_MN, B_MN);
    int s = 0;        // as in the producer
    uint32_t ph = 0;
    for (int i = 0; i < nmine; ++i) {
      if (!tc::mbar_wait(&full_bar[s], ph, &abort_flag, a.err, tc::kErrTimeoutLoad)) break;
      tc::tc_fence_after();
      const uint32_t sa = tc::smem_u32(smem + (size_t)s * a.stage_bytes);
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk) {
        const uint64_t ad = A_MN ? tc::sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                 : tc::sdesc_sw128(sa + kk * 32, 16, 1024);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const uint32_t sb = sa + a.a_bytes + nb * a.b_bytes;
          const uint64_t bd = B_MN ? tc::sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                   : tc::sdesc_sw128(sb + kk * 32, 16, 1024);
          tc::mma_bf16(tmem, ad, bd, idesc, (i > 0 || kk > 0 || nb > 0) ? 1u : 0u);
        }
      }
      tc::mma_commit(&empty_bar[s]);
      consumed = i + 1;
      if (++s == a.stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (nmine > 0) tc::mma_commit(&acc_bar);
  }
  __syncwarp();

  // ---- accumulator -> shared memory (fp32, row stride red_stride) ----
  float* red = reinterpret_cast<float*>(smem);  // all stages are consumed once acc_bar fires
  const int q = warp * 32 + lane;               // accumulator row = TMEM lane
  const int ncols32 = (a.n_pad + 31) / 32;
  bool have = false;
  if (nmine > 0) have = tc::mbar_wait(&acc_bar, 0, &abort_flag, a.err, tc::kErrTimeoutMma);
  tc::tc_fence_after();
  if (have) {
    for (int cg = 0; cg < ncols32; ++cg) {
      uint32_t v[32];
      tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cg * 32), v);
      tc::tmem_wait_ld();
      float4* dst = reinterpret_cast<float4*>(red + (size_t)q * a.red_stride + cg * 32);
#pragma unroll
      for (int t = 0; t < 8; ++t)
        dst[t] = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                             __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
    }
  } else {
    float4* dst = reinterpret_cast<float4*>(red + (size_t)q * a.red_stride);
    for (int t = 0; t < ncols32 * 8; ++t) dst[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (S > 1) tc::cluster_sync();
  else __syncthreads();

  // ---- cluster reduction of this CTA's row slice, fixed order over ranks ----
  const int rows_per = 128 / (int)S;
  const int r0 = (int)rank * rows_per;
  const int ncol4 = (a.N + 3) / 4;
  const uint32_t red_base = tc::smem_u32(red);
  for (int e = threadIdx.x; e < rows_per * ncol4; e += kThreads) {
    const int row = r0 + e / ncol4, c = (e % ncol4) * 4;
    const uint32_t off = (uint32_t)((row * a.red_stride + c) * 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (uint32_t src = 0; src < S; ++src) {
      const float4 v = (S > 1) ? tc::ld_dsmem_f4(tc::mapa_shared(red_base + off, src))
                               : *reinterpret_cast<const float4*>(red + row * a.red_stride + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int64_t grow = (int64_t)m0 + row;
    if (grow >= M || abort_flag) continue;
    const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
    if (a.out_mode == 0) {
      uint16_t* o = static_cast<uint16_t*>(a.out[p]) + grow * a.ld_out[p] + c;
      for (int t = 0; t < 4 && c + t < a.N; ++t) o[t] = __bfloat16_as_ushort(__float2bfloat16_rn(vals[t]));
    } else if (a.out_mode == 3) {
      uint16_t* o = static_cast<uint16_t*>(a.out[p]) + grow * a.ld_out[p] + c;
      for (int t = 0; t < 4 && c + t < a.N; ++t) {
        const __nv_bfloat16 h = __float2bfloat16_rn(vals[t]);
        o[t] = __bfloat16_as_ushort(h);
        o[a.n_pad + t] = __bfloat16_as_ushort(__float2bfloat16_rn(vals[t] - __bfloat162float(h)));
      }
    } else {
      float* o = static_cast<float*>(a.out[p]) + grow * a.ld_out[p] + c;
      for (int t = 0; t < 4 && c + t < a.N; ++t) o[t] = (a.out_mode == 2) ? o[t] + vals[t] : vals[t];
    }
  }
  if (S > 1) tc::cluster_sync();  // no CTA leaves while its tile may still be read

  // ---- on a timeout, give copies still in flight a bounded chance to land ----
  if (threadIdx.x == 0 && abort_flag) {
    volatile int dummy = 0;
    for (int i = consumed; i < issued; ++i)
      tc::mbar_wait(&full_bar[i % a.stages], (i / a.stages) & 1, &dummy, nullptr, 0, 100000000ull);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, a.tmem_cols);
}

// ---- persistent sketch accumulation ------------------------------------------
// C (+)= D^T XP for many layers with one CTA per SM.  A work item is one layer's
// strip of MT 128-row tiles of C over all tokens; the CTAs take the items
// round robin (every item of a launch has the same token count, so the split
// is even).  Warp 0 (one lane) streams the strip's D columns and the XP rows
// of each 64-token chunk into a ring of stages with TMA; warp 1 (one lane)
// issues the MMAs of each chunk into the item's accumulators, which alternate
// between two TMEM buffers; warps 2..5 read a finished item's accumulators
// (one row of C per thread) and add them to C while the next item streams.
// Each row of C is written by one thread after a fixed-order accumulation over
// the tokens, so results do not depend on timing.
constexpr int kAccThreads = 192;

template <int MT, int NB>
__global__ void __launch_bounds__(kAccThreads, 1) acc_persistent_kernel(const __grid_constant__ SkinnyBatch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int issued, consumed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = a.tile_begin[a.n];
  const uint32_t acc_cols = (uint32_t)(MT * a.n_pad);  // one buffer: MT accumulators

  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued = 0;
    consumed = 0;
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull_bar[b], 1);
      tc::mbar_init(&tempty_bar[b], 4);  // the four epilogue warps
    }
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, a.tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  auto decode = [&](int item, int& p, int& m0) {
    p = 0;
    while (p + 1 < a.n && a.tile_begin[p + 1] <= item) ++p;
    m0 = (item - a.tile_begin[p]) * 128 * MT;
  };

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA ring over the items' chunks ----
    int it = 0;
    int s = 0;        // stage of chunk it: it % stages, kept without a division
    uint32_t ph = 0;  // (it / stages) & 1
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
      int p, m0;
      decode(item, p, m0);
      const CUtensorMap* tmA = &a.tmA[p];
      const CUtensorMap* tmB = &a.tmB[p];
      for (int c = 0; c < a.kchunks[p]; ++c, ++it) {
        if (it >= a.stages && !tc::mbar_wait(&empty_bar[s], ph ^ 1u, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* st = smem + (size_t)s * a.stage_bytes;
        tc::mbar_arrive_expect_tx(&full_bar[s], a.stage_bytes);
        const int kc = c * kChunk;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {  // D: [64 tokens][64 rows of C] per box, two per tile
          tc::tma_load_2d(st + mt * 16384, tmA, &full_bar[s], m0 + 128 * mt, kc);
          tc::tma_load_2d(st + mt * 16384 + 8192, tmA, &full_bar[s], m0 + 128 * mt + 64, kc);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {  // XP: [64 tokens][64 rank columns] per box
          uint8_t* bt = st + MT * 16384 + nb * a.b_bytes;
          for (int j = 0; j * 64 < a.n_pad; ++j)
            tc::tma_load_2d(bt + j * 8192, tmB, &full_bar[s], nb * a.b_col_off + j * 64, kc);
        }
        issued = it + 1;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    const uint32_t idesc = tc::idesc_bf16(128, a.n_pad, true, true);
    int it = 0, j = 0;
    int s = 0;        // stage of chunk it and its phase, as in the producer
    uint32_t ph = 0;
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x, ++j) {
      int p, m0;
      decode(item, p, m0);
      const int b = j & 1;
      if (j >= 2 && !tc::mbar_wait(&tempty_bar[b], ((j >> 1) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage))
        break;
      tc::tc_fence_after();
      const uint32_t acc0 = tmem + (uint32_t)b * acc_cols;
      for (int c = 0; c < a.kchunks[p]; ++c, ++it) {
        if (!tc::mbar_wait(&full_bar[s], ph, &abort_flag, a.err, tc::kErrTimeoutLoad)) {
          stop = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t sa = tc::smem_u32(smem + (size_t)s * a.stage_bytes);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk) {
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint64_t ad = tc::sdesc_sw128(sa + mt * 16384 + kk * 2048, 8192, 1024);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const uint64_t bd = tc::sdesc_sw128(sa + MT * 16384 + nb * a.b_bytes + kk * 2048, 8192, 1024);
              tc::mma_bf16(acc0 + (uint32_t)(mt * a.n_pad), ad, bd, idesc, (c > 0 || kk > 0 || nb > 0) ? 1u : 0u);
            }
          }
        }
        tc::mma_commit(&empty_bar[s]);
        consumed = it + 1;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!stop) tc::mma_commit(&tfull_bar[b]);
    }
  } else if (warp >= 2) {
    // ---- epilogue: accumulators -> C, one row per thread ----
    const int quarter = warp & 3;  // TMEM lanes 32 (warp % 4) .. +31
    const int q = quarter * 32 + lane;
    const int ncols32 = (a.n_pad + 31) / 32;
    const bool vec = (a.N & 3) == 0;
    int j = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
      int p, m0;
      decode(item, p, m0);
      const int b = j & 1;
      const bool live = tc::mbar_wait(&tfull_bar[b], (j >> 1) & 1, &abort_flag, a.err, tc::kErrTimeoutMma);
      if (!__all_sync(0xFFFFFFFFu, live)) break;
      tc::tc_fence_after();
      const int M = a.M[p];
      float* Cp = static_cast<float*>(a.out[p]);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int64_t grow = (int64_t)m0 + 128 * mt + q;
        for (int cg = 0; cg < ncols32; ++cg) {
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)b * acc_cols +
                                     (uint32_t)(mt * a.n_pad + cg * 32), v);
          tc::tmem_wait_ld();
          if (grow >= M) continue;
          float* row = Cp + grow * a.ld_out[p] + cg * 32;
          const int ncol = a.N - cg * 32 < 32 ? a.N - cg * 32 : 32;
          if (vec) {
            float4* r4 = reinterpret_cast<float4*>(row);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (4 * t >= ncol) break;
              float4 o = make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                     __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]));
              if (a.out_mode == 2) {
                const float4 c0 = r4[t];
                o.x += c0.x;
                o.y += c0.y;
                o.z += c0.z;
                o.w += c0.w;
              }
              r4[t] = o;
            }
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t < ncol) row[t] = (a.out_mode == 2) ? row[t] + __uint_as_float(v[t]) : __uint_as_float(v[t]);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty_bar[b]);
    }
  }
  __syncwarp();
  // ---- on a timeout, give copies still in flight a bounded chance to land ----
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) {
    volatile int dummy = 0;
    for (int i = consumed; i < issued; ++i)
      tc::mbar_wait(&full_bar[i % a.stages], (i / a.stages) & 1, &dummy, nullptr, 0, 100000000ull);
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, a.tmem_cols);
}

// ---- persistent input projection ---------------------------------------------
// XP = bf16(X (P_hi + P_lo)) for many layers with one CTA per SM.  A work item
// is one problem's tile of 128 token rows over all of K; the CTAs take the
// items round robin.  Warp 0 (one lane) streams each 64-wide K chunk of the
// tile's X rows and of both parts of P^T into a ring of stages with TMA; warp 1
// (one lane) issues the chunk's MMAs (both parts into the same accumulator)
// into one of two TMEM buffers; warps 2..5 round a finished item's
// accumulators to BF16 and store them (one token row per thread) while the
// next item streams.  The tensor cores' fp32 accumulation loses a little with
// every addition, so a tile's K chunks go to k_parts accumulators of
// contiguous K ranges (as many as TMEM holds: up to 4), added in a fixed order
// by the epilogue; a long single chain (192 chunks for k = 12288) would leave
// XP measurably less accurate than the split over a cluster does.
template <int NB, int CB, bool STACK>
__global__ void __launch_bounds__(kAccThreads, 1) proj_persistent_kernel(const __grid_constant__ SkinnyBatch a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ volatile int issued, consumed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = a.tile_begin[a.n];

  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued = 0;
    consumed = 0;
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull_bar[b], 1);
      tc::mbar_init(&tempty_bar[b], 4);  // the four epilogue warps
    }
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, a.tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  auto decode = [&](int item, int& p, int& m0) {
    p = 0;
    while (p + 1 < a.n && a.tile_begin[p + 1] <= item) ++p;
    m0 = (item - a.tile_begin[p]) * 128;
  };

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA ring over the items' chunks ----
    int it = 0;
    int s = 0;        // stage of chunk it: it % stages, kept without a division
    uint32_t ph = 0;  // (it / stages) & 1
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
      int p, m0;
      decode(item, p, m0);
      const CUtensorMap* tmA = &a.tmA[p];
      const CUtensorMap* tmB = &a.tmB[p];
      const int nst = (a.kchunks[p] + CB - 1) / CB;  // stages of CB chunks
      for (int c = 0; c < nst; ++c, ++it) {
        if (it >= a.stages && !tc::mbar_wait(&empty_bar[s], ph ^ 1u, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* st = smem + (size_t)s * a.stage_bytes;
        tc::mbar_arrive_expect_tx(&full_bar[s], a.stage_bytes);
        // X: CB boxes of [128 tokens][64 k] (past M or K: zeros), then per
        // box the parts of the P^T split, [n_pad rank rows][64 k] each, side by
        // side (so that STACK reads both parts as one operand of 2 n_pad rows)
#pragma unroll
        for (int bx = 0; bx < CB; ++bx) {
          const int kc = (c * CB + bx) * kChunk;
          tc::tma_load_2d(st + bx * a.a_bytes, tmA, &full_bar[s], kc, m0);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            tc::tma_load_2d(st + CB * a.a_bytes + (bx * NB + nb) * a.b_bytes, tmB, &full_bar[s], kc, nb * a.n_pad);
        }
        issued = it + 1;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    // This one thread paces the kernel: per chunk it only waits, forms two
    // descriptors and issues the MMAs (no divisions; the partial accumulator
    // of each chunk follows from running boundaries)
    // STACK: one MMA per K step against both parts at once (N = 2 n_pad),
    // the parts' products in adjacent accumulator columns; else one MMA per
    // part into the same accumulator
    const int acc_n = STACK ? NB * a.n_pad : a.n_pad;
    const uint32_t idesc = tc::idesc_bf16(128, acc_n, false, false);
    const int nbuf = a.acc_bufs, kp = a.k_parts;
    int it = 0, j = 0;
    int s = 0;        // stage of chunk it and its phase, as in the producer
    uint32_t ph = 0;
    bool stop = false;
    for (int item = blockIdx.x; item < n_items && !stop; item += gridDim.x, ++j) {
      int p, m0;
      decode(item, p, m0);
      const int b = j % nbuf, use = j / nbuf;
      if (use >= 1 && !tc::mbar_wait(&tempty_bar[b], (use - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage))
        break;
      tc::tc_fence_after();
      const int kc = (a.kchunks[p] + CB - 1) / CB;  // stages of the item
      // partial accumulators: contiguous K ranges over min(k_parts, stages)
      // partials, part q starting at stage ceil(q kc / kpe)
      const int kpe = kc < kp ? kc : kp;
      int part = 0, next = (kc + kpe - 1) / kpe;
      bool first = true;
      for (int c = 0; c < kc; ++c, ++it) {
        if (c == next) {
          ++part;
          next = ((part + 1) * kc + kpe - 1) / kpe;
          first = true;
        }
        if (!tc::mbar_wait(&full_bar[s], ph, &abort_flag, a.err, tc::kErrTimeoutLoad)) {
          stop = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t sa = tc::smem_u32(smem + (size_t)s * a.stage_bytes);
        const uint32_t acc0 = tmem + (uint32_t)((b * kp + part) * acc_n);
        // descriptors of the stage's operands; each 16-wide K step adds 32
        // bytes (2 in the descriptor's address field), each box its size
        const uint64_t ad0 = tc::sdesc_sw128(sa, 16, 1024);
        uint64_t bd0[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) bd0[nb] = tc::sdesc_sw128(sa + CB * a.a_bytes + nb * a.b_bytes, 16, 1024);
        const uint32_t a_step = a.a_bytes >> 4, b_step = (NB * a.b_bytes) >> 4;
#pragma unroll
        for (int bx = 0; bx < CB; ++bx) {
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk) {
            if (STACK) {
              tc::mma_bf16(acc0, ad0 + bx * a_step + 2u * kk, bd0[0] + bx * b_step + 2u * kk, idesc,
                           (!first || bx > 0 || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int nb = 0; nb < NB; ++nb)
                tc::mma_bf16(acc0, ad0 + bx * a_step + 2u * kk, bd0[nb] + bx * b_step + 2u * kk, idesc,
                             (!first || bx > 0 || kk > 0 || nb > 0) ? 1u : 0u);
            }
          }
        }
        tc::mma_commit(&empty_bar[s]);
        consumed = it + 1;
        first = false;
        if (++s == a.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!stop) tc::mma_commit(&tfull_bar[b]);
    }
  } else if (warp >= 2) {
    // ---- epilogue: accumulators -> XP, one token row per thread ----
    const int quarter = warp & 3;  // TMEM lanes 32 (warp % 4) .. +31
    const int q = quarter * 32 + lane;
    const int ncols32 = (a.n_pad + 31) / 32;
    const int nbuf = a.acc_bufs, kp = a.k_parts;
    int j = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
      int p, m0;
      decode(item, p, m0);
      const int b = j % nbuf;
      const bool live = tc::mbar_wait(&tfull_bar[b], (j / nbuf) & 1, &abort_flag, a.err, tc::kErrTimeoutMma);
      if (!__all_sync(0xFFFFFFFFu, live)) break;
      tc::tc_fence_after();
      const int64_t grow = (int64_t)m0 + q;
      uint16_t* row = static_cast<uint16_t*>(a.out[p]) + grow * a.ld_out[p];
      const int nst = (a.kchunks[p] + CB - 1) / CB;
      const int nparts = nst < kp ? nst : kp;  // partials that received stages
      const int acc_n = STACK ? NB * a.n_pad : a.n_pad;
      for (int cg = 0; cg < ncols32; ++cg) {
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cg * 32);
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(b * kp * acc_n), v);
        tc::tmem_wait_ld();
        // the partials in K order; with STACK each partial's part products
        // (columns c and n_pad + c) in part order
        for (int pt = 0; pt < nparts; ++pt) {
          for (int nb = (pt == 0 ? 1 : 0); nb < (STACK ? NB : 1); ++nb) {
            uint32_t w[32];
            tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)((b * kp + pt) * acc_n + nb * a.n_pad), w);
            tc::tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(w[t]));
          }
        }
        if (grow >= a.M[p]) continue;
        const int c0 = cg * 32;
        const int ncol = a.N - c0 < 32 ? a.N - c0 : 32;
        if (ncol <= 0) continue;
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float f0 = __uint_as_float(v[2 * t]), f1 = __uint_as_float(v[2 * t + 1]);
          const __nv_bfloat16 h0 = __float2bfloat16_rn(f0), h1 = __float2bfloat16_rn(f1);
          hi[t] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
          if (a.out_mode == 3)
            lo[t] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f0 - __bfloat162float(h0))) |
                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f1 - __bfloat162float(h1))) << 16);
        }
        // the row stride is a multiple of 8 elements: 16-byte stores for
        // whole 8-column groups, single elements for a ragged end
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          const int cc = c0 + 8 * g8;
          if (cc + 8 <= a.N) {
            *reinterpret_cast<uint4*>(row + cc) = make_uint4(hi[4 * g8], hi[4 * g8 + 1], hi[4 * g8 + 2], hi[4 * g8 + 3]);
            if (a.out_mode == 3)
              *reinterpret_cast<uint4*>(row + a.n_pad + cc) =
                  make_uint4(lo[4 * g8], lo[4 * g8 + 1], lo[4 * g8 + 2], lo[4 * g8 + 3]);
          } else if (cc < a.N) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (cc + t < a.N) {
                row[cc + t] = (uint16_t)(hi[4 * g8 + (t >> 1)] >> (16 * (t & 1)));
                if (a.out_mode == 3) row[a.n_pad + cc + t] = (uint16_t)(lo[4 * g8 + (t >> 1)] >> (16 * (t & 1)));
              }
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty_bar[b]);
    }
  }
  __syncwarp();
  // ---- on a timeout, give copies still in flight a bounded chance to land ----
  tc::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && abort_flag) {
    volatile int dummy = 0;
    for (int i = consumed; i < issued; ++i)
      tc::mbar_wait(&full_bar[i % a.stages], (i / a.stages) & 1, &dummy, nullptr, 0, 100000000ull);
  }
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, a.tmem_cols);
}

// P (k x r fp32) -> P^T split into BF16 high and low parts: rows [0, n_pad)
// hold the high part, rows [n_pad, 2 n_pad) the low part, each k wide; rank
// rows r..n_pad-1 are zero.  64 x 32 tiles transposed through shared memory;
// grid.z indexes the problem.  Problem i writes rows [row_off, row_off + rows)
// of the high half and the same rows of the low half (which starts n_pad_out
// rows down); rows past r are zero.  A plain split has row_off 0 and rows =
// n_pad = n_pad_out; the members of a group write their r rows one after
// another and the last one also the padding.
struct SplitT {
  const float* P[kMaxProblems];
  uint16_t* out[kMaxProblems];
  int64_t k[kMaxProblems];
  int row_off[kMaxProblems];
  int rows[kMaxProblems];
  int n_pad_out[kMaxProblems];
  int r;
};

__global__ void __launch_bounds__(256) split_transpose_kernel(const __grid_constant__ SplitT a) {
  __shared__ float t[64][33];
  const int pr = blockIdx.z;
  const int64_t k = a.k[pr];
  const int64_t j0 = (int64_t)blockIdx.x * 64;
  if (j0 >= k) return;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int l0 = blockIdx.y * 32;
  const int r = a.r, rows = a.rows[pr];
  if (l0 >= rows) return;
  const float* P = a.P[pr];
  for (int dy = ty; dy < 64; dy += 8) {
    const int64_t j = j0 + dy;
    const int l = l0 + tx;
    t[dy][tx] = (j < k && l < r) ? P[j * r + l] : 0.f;
  }
  __syncthreads();
  // a pair of columns j, j + 1 per thread (k is a multiple of 8 and the
  // output 16-byte aligned, so the pair is one aligned 4-byte store per part)
  uint16_t* hi = a.out[pr] + (int64_t)a.row_off[pr] * k;
  uint16_t* lo = hi + (int64_t)a.n_pad_out[pr] * k;
  for (int dy = ty; dy < 32; dy += 8) {
    const int l = l0 + dy;
    const int64_t j = j0 + 2 * tx;
    if (l < rows && j < k) {
      uint32_t hp = 0, lp = 0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = t[2 * tx + e][dy];
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        const __nv_bfloat16 w = __float2bfloat16_rn(v - __bfloat162float(h));
        hp |= (uint32_t)__bfloat16_as_ushort(h) << (16 * e);
        lp |= (uint32_t)__bfloat16_as_ushort(w) << (16 * e);
      }
      *reinterpret_cast<uint32_t*>(hi + (int64_t)l * k + j) = hp;
      *reinterpret_cast<uint32_t*>(lo + (int64_t)l * k + j) = lp;
    }
  }
}

int round16(int r) { return (r + 15) / 16 * 16; }

uint32_t tmem_cols_for(int n_pad) {
  uint32_t c = 32;
  while ((int)c < n_pad) c <<= 1;
  return c;
}

// Cluster split: enough CTAs for two per SM, at most 8 per cluster and at
// least one K chunk per CTA.
int choose_split(int m_tiles, int kchunks) {
  const int target = 2 * num_sms();
  int s = 1;
  while (s < 8 && m_tiles * s < target && 2 * s <= kchunks) s *= 2;
  return s;
}

// Launch geometry of a batch: cluster split, stages, shared memory.
template <bool A_MN, bool B_MN, int NB>
cudaError_t launch_skinny(SkinnyBatch& a, cudaStream_t stream) {
  const int tiles = a.tile_begin[a.n];
  int min_chunks = a.kchunks[0];
  for (int i = 1; i < a.n; ++i) min_chunks = a.kchunks[i] < min_chunks ? a.kchunks[i] : min_chunks;
  const int split = choose_split(tiles, min_chunks);
  a.stage_bytes = a.a_bytes + NB * a.b_bytes;
  // two CTAs per SM when the stages fit in half of shared memory; stages wider
  // than 48 KB (a B of 192+ rank columns, as grouped projections have) get
  // the whole SM, since two of them per CTA would leave too few K chunks in
  // flight to cover the loads
  const uint32_t budget = a.stage_bytes > 48u * 1024u ? 208u * 1024u : 96u * 1024u;
  int stages = (int)(budget / a.stage_bytes);
  if (stages < 2) stages = 2;
  if (stages > kMaxStages) stages = kMaxStages;
  a.stages = stages;
  a.red_stride = (a.n_pad + 31) / 32 * 32 + 4;
  a.tmem_cols = tmem_cols_for(a.n_pad);
  size_t smem = (size_t)stages * a.stage_bytes;
  const size_t red_bytes = (size_t)128 * a.red_stride * sizeof(float);
  if (red_bytes > smem) smem = red_bytes;
  // at most two CTAs per SM, so their TMEM (<= 2 x 256 columns) always fits
  if (smem < 80 * 1024) smem = 80 * 1024;
  smem += 1024;  // alignment slack
  auto kernel = skinny_gemm_kernel<A_MN, B_MN, NB>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)split, (unsigned)tiles, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Tiles of C per persistent work item: wider strips read longer runs of each
// token row of D, up to what two TMEM buffers of accumulators hold.
int acc_strip_tiles(int n_pad) {
  const int mt = kAccStripTiles;
  return (2 * mt * n_pad <= 512) ? mt : 1;
}

template <int MT, int NB>
cudaError_t launch_acc_persistent(SkinnyBatch& a, cudaStream_t stream) {
  a.stage_bytes = MT * 16384u + NB * a.b_bytes;
  int stages = (int)((200u * 1024u) / a.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  a.tmem_cols = tmem_cols_for(2 * MT * a.n_pad);
  const size_t smem = (size_t)stages * a.stage_bytes + 1024;
  auto kernel = acc_persistent_kernel<MT, NB>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int items = a.tile_begin[a.n];
  const int grid = items < num_sms() ? items : num_sms();
  count_launch();
  kernel<<<grid, kAccThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_proj_persistent(SkinnyBatch& a, cudaStream_t stream) {
  // two 64-wide K chunks per stage (longer runs of each token row of X, half
  // the per-stage work of the issuing threads) where three such stages fit
  const uint32_t one = a.a_bytes + 2 * a.b_bytes;
  const int cb = (3 * 2 * one <= 200u * 1024u) ? 2 : 1;
  // both parts of the split in one MMA (N = 2 n_pad): half the MMA
  // instructions.  Up to rank 64 this keeps two tiles of accumulators in
  // TMEM; above, the wider accumulators would leave room for one tile only,
  // which measured slower than twice the MMAs (rank 128: 0.66 against 0.67 of HBM)
  const bool stack = a.n_pad <= 64;
  const int acc_n = stack ? 2 * a.n_pad : a.n_pad;
  a.stage_bytes = cb * one;
  int stages = (int)((200u * 1024u) / a.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  // partial accumulators: up to 4 per tile, two tiles in flight where TMEM
  // holds them, else one tile of two
  a.acc_bufs = 2;
  a.k_parts = 4;
  while (a.k_parts > 1 && a.acc_bufs * a.k_parts * acc_n > 512) a.k_parts >>= 1;
  if (a.k_parts == 1) {
    a.acc_bufs = 1;
    a.k_parts = 2;
  }
  a.tmem_cols = tmem_cols_for(a.acc_bufs * a.k_parts * acc_n);
  const size_t smem = (size_t)stages * a.stage_bytes + 1024;
  auto kernel = stack ? (cb == 2 ? proj_persistent_kernel<2, 2, true> : proj_persistent_kernel<2, 1, true>)
                      : (cb == 2 ? proj_persistent_kernel<2, 2, false> : proj_persistent_kernel<2, 1, false>);
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int items = a.tile_begin[a.n];
  const int grid = items < num_sms() ? items : num_sms();
  count_launch();
  kernel<<<grid, kAccThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t project_workspace_bytes(int64_t, int64_t k, int64_t r) {
  WsCursor cur;
  cur.take<uint16_t>((size_t)2 * round16((int)r) * k);
  cur.take<char>(0);  // a multiple of 256, so regions of a batch stay aligned
  return cur.offset;
}

cudaError_t launch_split_projection(int n, const float* const* P, const int64_t* k, uint16_t* const* out, int r,
                                    cudaStream_t stream) {
  static thread_local SplitT sp;
  const int n_pad = round16(r);
  for (int base = 0; base < n; base += kMaxProblems) {
    const int m = (n - base) < kMaxProblems ? (n - base) : kMaxProblems;
    int64_t max_k = 0;
    for (int i = 0; i < m; ++i) {
      sp.P[i] = P[base + i];
      sp.out[i] = out[base + i];
      sp.k[i] = k[base + i];
      sp.row_off[i] = 0;
      sp.rows[i] = n_pad;
      sp.n_pad_out[i] = n_pad;
      max_k = k[base + i] > max_k ? k[base + i] : max_k;
    }
    sp.r = r;
    count_launch();
    split_transpose_kernel<<<dim3((unsigned)ceil_div(max_k, 64), (unsigned)ceil_div(n_pad, 32), (unsigned)m), 256, 0,
                             stream>>>(sp);
  }
  return cudaGetLastError();
}

cudaError_t launch_split_projection_grouped(int n, const SplitGroup* groups, int r, cudaStream_t stream) {
  static thread_local SplitT sp;
  int i = 0, max_rows = 0;
  int64_t max_k = 0;
  auto flush = [&]() -> cudaError_t {
    if (i == 0) return cudaSuccess;
    sp.r = r;
    count_launch();
    split_transpose_kernel<<<dim3((unsigned)ceil_div(max_k, 64), (unsigned)ceil_div(max_rows, 32), (unsigned)i), 256,
                             0, stream>>>(sp);
    i = 0;
    max_rows = 0;
    max_k = 0;
    return cudaGetLastError();
  };
  for (int g = 0; g < n; ++g) {
    const SplitGroup& gr = groups[g];
    const int n_pad_out = round16(gr.m * r);
    for (int q = 0; q < gr.m; ++q) {
      if (i == kMaxProblems) {
        const cudaError_t err = flush();
        if (err != cudaSuccess) return err;
      }
      sp.P[i] = gr.P[q];
      sp.out[i] = gr.out;
      sp.k[i] = gr.k;
      sp.row_off[i] = q * r;
      sp.rows[i] = (q + 1 == gr.m) ? n_pad_out - q * r : r;
      sp.n_pad_out[i] = n_pad_out;
      max_rows = sp.rows[i] > max_rows ? sp.rows[i] : max_rows;
      max_k = gr.k > max_k ? gr.k : max_k;
      ++i;
    }
  }
  return flush();
}

cudaError_t launch_project_inputs(int n, const ProjectProblem* probs, int r, void* ws, cudaStream_t stream,
                                  bool xp_split) {
  const int n_pad = round16(r);
  int* errw = nullptr;
  cudaError_t err = device_error_word(&errw);
  if (err != cudaSuccess) return err;
  WsCursor cur;
  cur.base = static_cast<char*>(ws);
  static thread_local SkinnyBatch a;
  for (int base = 0; base < n; base += kMaxProblems) {
    const int m = (n - base) < kMaxProblems ? (n - base) : kMaxProblems;
    // problems without a ready split get one in their workspace region
    const float* sp_P[kMaxProblems];
    int64_t sp_k[kMaxProblems];
    uint16_t* sp_out[kMaxProblems];
    int nsplit = 0;
    a.tile_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const ProjectProblem& pr = probs[base + i];
      uint16_t* region = cur.take<uint16_t>((size_t)2 * n_pad * pr.k);
      cur.take<char>(0);
      const uint16_t* pt = pr.P_split;
      if (pt == nullptr) {
        sp_P[nsplit] = pr.P;
        sp_k[nsplit] = pr.k;
        sp_out[nsplit] = region;
        ++nsplit;
        pt = region;
      }
      err = make_tmap_bf16_2d(&a.tmA[i], pr.X, (uint64_t)pr.k, (uint64_t)pr.T, (uint64_t)pr.ld_x * 2, 64, 128);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tmB[i], pt, (uint64_t)pr.k, (uint64_t)2 * n_pad, (uint64_t)pr.k * 2, 64,
                                (uint32_t)n_pad);
      if (err != cudaSuccess) return err;
      a.out[i] = pr.XP;
      a.ld_out[i] = pr.ld_xp;
      a.M[i] = (int)pr.T;
      a.kchunks[i] = (int)ceil_div(pr.k, kChunk);
      a.tile_begin[i + 1] = a.tile_begin[i] + (int)ceil_div(pr.T, 128);
    }
    if (nsplit > 0) {
      err = launch_split_projection(nsplit, sp_P, sp_k, sp_out, r, stream);
      if (err != cudaSuccess) return err;
    }
    a.n = m;
    a.N = r;
    a.n_pad = n_pad;
    a.a_bytes = 128 * kChunk * 2;
    a.b_bytes = (uint32_t)n_pad * kChunk * 2;
    a.out_mode = xp_split ? 3 : 0;
    a.b_col_off = 0;
    a.err = errw;
    // enough token tiles to keep every SM busy: persistent CTAs, each tile
    // over all of K, the next tile's loads overlapping this one's epilogue
    // (measured against two split-K CTAs per SM on 36 layers of 4096 tokens:
    // 0.79 against 0.72 of HBM at rank 64, k = 4096; 0.66 against 0.57 at
    // rank 128); fewer tiles: split-K CTAs over a cluster
    err = (a.tile_begin[m] >= 2 * num_sms()) ? launch_proj_persistent(a, stream)
                                              : launch_skinny<false, false, 2>(a, stream);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

size_t accumulate_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_accumulate(int n, const AccumulateProblem* probs, int r, int overwrite, cudaStream_t stream,
                              bool xp_split) {
  const int n_pad = round16(r);
  int* errw = nullptr;
  cudaError_t err = device_error_word(&errw);
  if (err != cudaSuccess) return err;
  static thread_local SkinnyBatch a;
  for (int base = 0; base < n; base += kMaxProblems) {
    const int m = (n - base) < kMaxProblems ? (n - base) : kMaxProblems;
    a.tile_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const AccumulateProblem& pr = probs[base + i];
      err = make_tmap_bf16_2d(&a.tmA[i], pr.D, (uint64_t)pr.d, (uint64_t)pr.T, (uint64_t)pr.ld_d * 2, 64, 64);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tmB[i], pr.XP, (uint64_t)(xp_split ? 2 * n_pad : r), (uint64_t)pr.T,
                                (uint64_t)pr.ld_xp * 2, 64, 64);
      if (err != cudaSuccess) return err;
      a.out[i] = pr.C;
      a.ld_out[i] = r;
      a.M[i] = (int)pr.d;
      a.kchunks[i] = (int)ceil_div(pr.T, kChunk);
      a.tile_begin[i + 1] = a.tile_begin[i] + (int)ceil_div(pr.d, 128);
    }
    a.n = m;
    a.N = r;
    a.n_pad = n_pad;
    a.a_bytes = 128 * kChunk * 2;
    a.b_bytes = (uint32_t)((n_pad + 63) / 64) * 64 * kChunk * 2;
    a.out_mode = overwrite ? 1 : 2;
    a.err = errw;
    a.b_col_off = xp_split ? n_pad : 0;  // D^T XP_hi + D^T XP_lo, both into the same accumulator
    if (a.tile_begin[m] >= 2 * num_sms()) {
      // enough tiles to keep every SM busy: persistent CTAs over strips of
      // C, each over all tokens (no split over tokens)
      const int mt = acc_strip_tiles(n_pad);
      a.tile_begin[0] = 0;
      for (int i = 0; i < m; ++i) a.tile_begin[i + 1] = a.tile_begin[i] + (int)ceil_div(a.M[i], 128 * mt);
      if (mt == 1)
        err = xp_split ? launch_acc_persistent<1, 2>(a, stream) : launch_acc_persistent<1, 1>(a, stream);
      else if (mt == 2)
        err = xp_split ? launch_acc_persistent<2, 2>(a, stream) : launch_acc_persistent<2, 1>(a, stream);
      else
        err = xp_split ? launch_acc_persistent<4, 2>(a, stream) : launch_acc_persistent<4, 1>(a, stream);
    } else if (xp_split) {
      err = launch_skinny<true, true, 2>(a, stream);
    } else {
      err = launch_skinny<true, true, 1>(a, stream);
    }
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace rgs
