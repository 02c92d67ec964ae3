// Gram matrices G = A^T A of tall-skinny fp32 matrices (rows x r, r <= 256).
// Used by the CholeskyQR2 projection and by the normalized-SGD step, where
// ||C P^T||_F^2 = <P^T P, C^T C>.
//
// Two deterministic passes over a batch of matrices: partial Grams of fixed
// row chunks on the tensor cores (gram_tc_kernel), then a fixed-order sum over
// the chunks (gram_reduce_kernel).  Neither pass uses atomics, so the result
// does not depend on scheduling.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace rgs {
namespace {

// (hi, lo) += x with TwoSum (Knuth): exact error of the addition kept in lo.
__device__ __forceinline__ void acc2(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  hi = s;
  lo = __fadd_rn(lo, e);
}

// ---- tensor-core partial Gram ------------------------------------------------
// Chunks of gram_chunks_tc rows, one block per chunk that exists (the grid
// lists them matrix by matrix), the products on the tensor cores: a bound on
// the chunk's largest magnitude (given by the caller, recorded by A's
// producer, the largest of the rows' norms, or found by a pass over the chunk)
// gives a power of two 2^e that brings it into [2^14, 2^15) or a little
// below; each element x 2^e is split into
// FP16 high and low parts (hi + lo within ~2^-22 of it) written, 64 rows at a
// time, into shared-memory tiles laid out as the MMA's K-major operand (column m
// of A is row m of the tile, 128-byte swizzle), two sets of tiles so that one
// step's conversion overlaps the previous step's MMAs; tcgen05.mma (kind::f16,
// M = 128, N = r rounded to 16, K = 16) accumulates hi hi + hi lo + lo hi of
// A^T A into TMEM (two M halves when r > 128), the steps going to the
// gram_tc_accs accumulators in turn; warps 0..3, one per TMEM lane quarter, add
// the accumulators and scale the sums by 2^-2e into the chunk's partial (written with a
// zero low word), which gram_reduce_kernel adds up in chunk order.
constexpr int kGtcThreads = 256;
constexpr int kGtcStep = 64;  // rows per step: one 128-byte swizzled row of FP16 per column of A
__host__ __device__ inline int gtc_mpad(int r) { return r <= 128 ? 128 : 256; }
__host__ __device__ inline int gtc_npad(int r) { return (r + 15) / 16 * 16; }
// TMEM columns: the accumulators (nacc x M halves x npad), and at least the
// span the epilogue's 32-column reads cover
__host__ __device__ inline uint32_t gtc_tmem_cols(int r) {
  const int npad = gtc_npad(r), nmh = gtc_mpad(r) / 128, nacc = gram_tc_accs(r);
  const int reads = (nacc * nmh - 1) * npad + (npad + 31) / 32 * 32;
  const int cols = nacc * nmh * npad > reads ? nacc * nmh * npad : reads;
  uint32_t c = 32;
  while ((int)c < cols) c <<= 1;
  return c;
}
__device__ __forceinline__ uint8_t* gtc_align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}
// Largest magnitude of n floats from p (NaN if any is NaN): float4 loads, four
// in flight per thread, once p is 16-byte aligned.
__device__ __forceinline__ float gtc_chunk_max(const float* __restrict__ p, int64_t n) {
  float m = 0.f;
  auto take = [&](float x) { m = (m != m || x != x) ? __int_as_float(0x7FC00000) : fmaxf(m, fabsf(x)); };
  const int64_t head = (int64_t)(((16 - (reinterpret_cast<uintptr_t>(p) & 15)) & 15) / 4) < n
                           ? (int64_t)(((16 - (reinterpret_cast<uintptr_t>(p) & 15)) & 15) / 4) : n;
  if (threadIdx.x < head) take(p[threadIdx.x]);
  const float4* q = reinterpret_cast<const float4*>(p + head);
  const int64_t n4 = (n - head) / 4;
  int64_t i = threadIdx.x;
  for (; i + 3 * kGtcThreads < n4; i += 4 * kGtcThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = q[i + u * kGtcThreads];
#pragma unroll
    for (int u = 0; u < 4; ++u) { take(v[u].x); take(v[u].y); take(v[u].z); take(v[u].w); }
  }
  for (; i < n4; i += kGtcThreads) {
    const float4 v = q[i];
    take(v.x); take(v.y); take(v.z); take(v.w);
  }
  for (int64_t e = head + 4 * n4 + threadIdx.x; e < n; e += kGtcThreads) take(p[e]);
  return m;
}

// IPT: conversion items per thread per 64-row step (r * 8 items: 1 up to
// rank 32, 2 up to 64, 4 up to 128, 8 up to 256); each item is 8 rows of one
// column.  A step's rows are contiguous in A.  BULK (shared memory leaves room
// for a ring of at least two copies, batch.raw_stages, and every A starts on
// 16 bytes with rows * r a multiple of 4): thread 0 copies each step's rows
// into the ring with a bulk copy, raw_stages steps ahead, and the threads
// convert from there.  Otherwise each thread loads the next step's items into
// registers while this step's are converted.
constexpr int kGtcMaxRaw = 4;
template <int IPT, bool BULK>
__global__ void __launch_bounds__(kGtcThreads) gram_tc_kernel(const GramBatch batch) {
  extern __shared__ uint8_t gtc_raw[];
  __shared__ __align__(8) uint64_t mma_bar[2];
  __shared__ __align__(8) uint64_t raw_bar[kGtcMaxRaw];
  __shared__ uint32_t tmem_slot;
  __shared__ float wmax[kGtcThreads / 32];
  __shared__ volatile int abort_flag;
  // this block's matrix y and chunk c (the grid lists the chunks that exist)
  int y = 0;
  {
    int hi = batch.n - 1;
    while (y < hi) {
      const int mid = (y + hi + 1) >> 1;
      if (batch.chunk_begin[mid] <= (int)blockIdx.x) y = mid; else hi = mid - 1;
    }
  }
  const int chunk = (int)blockIdx.x - batch.chunk_begin[y];
  const GramEntry& en = batch.e[y];
  const int r = batch.r;
  const GramChunks g = gram_chunks_tc(en.rows, r);
  const int mpad = gtc_mpad(r), npad = gtc_npad(r), nmh = mpad / 128, nacc = gram_tc_accs(r);
  const uint32_t cols = gtc_tmem_cols(r);
  const uint32_t tile_bytes = (uint32_t)mpad * 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // buffer b: hi tile at base + 2 b tile_bytes, lo tile right after it
  const uint32_t base = tc::smem_u32(gtc_align1024(gtc_raw));
  const int64_t row_begin = (int64_t)chunk * g.chunk_rows;
  const int64_t row_end = row_begin + g.chunk_rows < en.rows ? row_begin + g.chunk_rows : en.rows;
  const float* __restrict__ A = en.A;
  const int nstages = batch.raw_stages;
  constexpr bool bulk = BULK;
  const uint32_t raw_base = base + 4 * tile_bytes, raw_bytes = (uint32_t)kGtcStep * r * 4;
  if (tid == 0) {
    abort_flag = 0;
    tc::mbar_init(&mma_bar[0], 1);
    tc::mbar_init(&mma_bar[1], 1);
    for (int q = 0; q < kGtcMaxRaw; ++q) tc::mbar_init(&raw_bar[q], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, cols);
  // every tile zero: rows m >= r (padding to the MMA's M and N) stay so
  for (uint32_t e = tid; e < 4 * tile_bytes / 16; e += kGtcThreads) tc::sts128(base + 16u * e, make_uint4(0, 0, 0, 0));
  // the largest magnitude: given by the producer of A (a bound, or the maximum
  // it recorded), else the chunk's own (NaN if any element is NaN)
  const bool given = en.amax != nullptr || en.bound > 0.f;
  float m = 0.f;
  if (!given && en.row_norms != nullptr) {
    // the largest row norm of the chunk (integer maximum of the bits: a NaN
    // norm wins), a bound within a factor sqrt(r) of the largest magnitude
    uint32_t nb = 0u;
    for (int64_t i = row_begin + tid; i < row_end; i += kGtcThreads) nb = max(nb, __float_as_uint(en.row_norms[i]));
    m = __uint_as_float(nb);
  } else if (!given) {
    m = gtc_chunk_max(A + row_begin * r, (row_end - row_begin) * r);
  }
  if (!given) {
    for (int o = 16; o > 0; o >>= 1) {
      const float om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      m = (m != m || om != om) ? __int_as_float(0x7FC00000) : fmaxf(m, om);
    }
    if (lane == 0) wmax[warp] = m;
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  float bm = 0.f;
  if (given) {
    bm = en.amax != nullptr ? __uint_as_float(*en.amax) : en.bound;
  } else {
    for (int w = 0; w < kGtcThreads / 32; ++w)
      bm = (bm != bm || wmax[w] != wmax[w]) ? __int_as_float(0x7FC00000) : fmaxf(bm, wmax[w]);
  }
  // 2^e brings the largest magnitude into [2^14, 2^15); a non-finite one keeps
  // e = 0, so that the products carry it into the Gram
  int e = 0;
  if (bm > 0.f && bm <= 3.4028234e38f) {
    int E;
    frexpf(bm, &E);
    e = 15 - E;
    e = e < -100 ? -100 : (e > 100 ? 100 : e);
  }
  const float scale = ldexpf(1.f, e), unscale = ldexpf(1.f, -e);
  const uint32_t idesc = tc::idesc_f16(128, npad, false, false);
  const int nsteps = (int)((row_end - row_begin + kGtcStep - 1) / kGtcStep);
  // item q of this thread: it = tid + q kGtcThreads, column it % r, rows 8 (it / r) ..
  const int nitems = r * 8;
  int mcq[IPT], k8q[IPT];
#pragma unroll
  for (int q = 0; q < IPT; ++q) {
    mcq[q] = (tid + q * kGtcThreads) % r;
    k8q[q] = (tid + q * kGtcThreads) / r;
  }
  float xn[IPT][8];
  auto load_step = [&](int st) {
    const int64_t row0 = row_begin + (int64_t)st * kGtcStep;
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
      const bool on = tid + q * kGtcThreads < nitems;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int64_t ra = row0 + 8 * k8q[q] + t;
        xn[q][t] = (on && ra < row_end) ? A[ra * r + mcq[q]] : 0.f;
      }
    }
  };
  // bulk path: step s goes to ring stage s % nstages (stage and phase kept
  // incrementally); thread 0 issues the first nstages steps here
  auto issue = [&](int sidx, uint32_t stage) {
    const int64_t r0 = row_begin + (int64_t)sidx * kGtcStep;
    const int64_t nr = row_end - r0 < kGtcStep ? row_end - r0 : kGtcStep;
    const uint32_t bytes = (uint32_t)(nr * r * 4);  // a multiple of 16: 64 r, or the chunk's remainder
    tc::mbar_arrive_expect_tx(&raw_bar[stage], bytes);
    tc::bulk_load_1d(raw_base + stage * raw_bytes, A + r0 * r, bytes, &raw_bar[stage]);
  };
  int issued = 0, consumed = 0;  // steps copied / converted (the same in every thread)
  uint32_t rstage = 0, rphase = 0;
  if (bulk) {
    issued = nsteps < nstages ? nsteps : nstages;
    if (tid == 0)
      for (int q = 0; q < issued; ++q) issue(q, (uint32_t)q);
  } else if (nsteps > 0) {
    load_step(0);
  }
  bool live = true;
  for (int st = 0; st < nsteps; ++st) {
    const int b = st & 1;
    const uint32_t hi_s = base + 2u * b * tile_bytes, lo_s = hi_s + tile_bytes;
    float xc[IPT][8];
    if constexpr (BULK) {
      // this step's rows (row m of the step at rs + 4 m r), zeros past the chunk
      live = tc::mbar_wait(&raw_bar[rstage], rphase, &abort_flag, nullptr, 0) && live;
      const uint32_t rs = raw_base + rstage * raw_bytes;
      const int64_t row0 = row_begin + (int64_t)st * kGtcStep;
      const int nr = (int)(row_end - row0 < kGtcStep ? row_end - row0 : kGtcStep);
#pragma unroll
      for (int q = 0; q < IPT; ++q) {
        const bool on = tid + q * kGtcThreads < nitems;
        const uint32_t a0 = rs + (uint32_t)(8 * k8q[q] * r + mcq[q]) * 4u;
        if (nr == kGtcStep) {  // a full step: every row is there
#pragma unroll
          for (int t = 0; t < 8; ++t) xc[q][t] = on ? tc::lds_f32(a0 + (uint32_t)(t * r) * 4u) : 0.f;
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            xc[q][t] = (on && 8 * k8q[q] + t < nr) ? tc::lds_f32(a0 + (uint32_t)(t * r) * 4u) : 0.f;
        }
      }
    } else {
#pragma unroll
      for (int q = 0; q < IPT; ++q)
#pragma unroll
        for (int t = 0; t < 8; ++t) xc[q][t] = xn[q][t];
      if (st + 1 < nsteps) load_step(st + 1);
    }
    if (st >= 2) {  // the MMAs of step st - 2 have read this buffer
      live = tc::mbar_wait(&mma_bar[b], (uint32_t)((st >> 1) - 1) & 1u, &abort_flag, nullptr, 0) && live;
      live = __syncthreads_and(live);
      if (!live) break;
    }
    // rows [row0, row0 + 64) into buffer b: item (column m of A, 8-row group
    // k8) is one 16-byte chunk of tile row m; consecutive threads take
    // consecutive columns, so that each row's loads are coalesced
#pragma unroll
    for (int q = 0; q < IPT; ++q) {
      const int it = tid + q * kGtcThreads;
      if (it < nitems) {
        const int mc = mcq[q], k8 = k8q[q];
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) hv[t] = tc::split_f16x2(xc[q][2 * t], xc[q][2 * t + 1], scale, lv[t]);
        const uint32_t off = (uint32_t)((mc >> 3) * 1024 + (mc & 7) * 128 + ((k8 ^ (mc & 7)) << 4));
        tc::sts128(hi_s + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
        tc::sts128(lo_s + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
      }
    }
    tc::fence_proxy_async_smem();  // also orders this step's reads of the ring before its refill
    live = __syncthreads_and(live);
    if (!live) break;
    consumed = st + 1;
    // the stage this step read takes step st + nstages
    const bool refill = bulk && st + nstages < nsteps;
    if (tid == 0) {
      if (refill) issue(st + nstages, rstage);
      tc::tc_fence_after();
      const int acc = st % nacc;  // this step's accumulator
      for (int mh = 0; mh < nmh; ++mh) {
        const uint32_t d = tmem + (uint32_t)((acc * nmh + mh) * npad);
        const uint32_t arow = (uint32_t)mh * 128 * 128;
#pragma unroll
        for (int kk = 0; kk < kGtcStep / 16; ++kk) {
          const uint64_t ah = tc::sdesc_sw128(hi_s + arow + kk * 32, 16, 1024);
          const uint64_t al = tc::sdesc_sw128(lo_s + arow + kk * 32, 16, 1024);
          const uint64_t bh = tc::sdesc_sw128(hi_s + kk * 32, 16, 1024);
          const uint64_t bl = tc::sdesc_sw128(lo_s + kk * 32, 16, 1024);
          tc::mma_bf16(d, ah, bh, idesc, (st >= nacc || kk > 0) ? 1u : 0u);
          tc::mma_bf16(d, ah, bl, idesc, 1u);
          tc::mma_bf16(d, al, bh, idesc, 1u);
        }
      }
      tc::mma_commit(&mma_bar[b]);  // also covers every earlier MMA of this thread
    }
    if (refill) ++issued;
    if (bulk && ++rstage == (uint32_t)nstages) {
      rstage = 0;
      rphase ^= 1u;
    }
  }
  // a loop that gave up leaves copies in flight: thread 0 waits (bounded, the
  // abort flag aside) until each has landed before the block's memory is released
  if (tid == 0 && bulk) {
    volatile int no_abort = 0;
    for (int q = consumed; q < issued; ++q)
      tc::mbar_wait(&raw_bar[q % nstages], (uint32_t)(q / nstages) & 1u, &no_abort, nullptr, 0);
  }
  if (live)
    live = tc::mbar_wait(&mma_bar[(nsteps - 1) & 1], (uint32_t)((nsteps - 1) >> 1) & 1u, &abort_flag, nullptr, 0);
  live = __syncthreads_and(live);
  tc::tc_fence_after();
  // warps 0..3: the sums of TMEM lane m (row m of A^T A) scaled back by
  // 2^-2e; a wait that gave up leaves the partial NaN
  if (warp < 4) {
    float2* out = en.partials + (size_t)chunk * r * r;
    for (int mh = 0; mh < nmh; ++mh) {
      const int mrow = mh * 128 + warp * 32 + lane;
      for (int cg = 0; cg * 32 < npad; ++cg) {
        uint32_t v[32];
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cg * 32);
        tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)(mh * npad), v);
        tc::tmem_wait_ld();
        // the accumulators that received steps, added in order
        for (int a = 1; a < nacc && a < nsteps; ++a) {
          uint32_t w[32];
          tc::tmem_ld_32x32b_x32(lane_base + (uint32_t)((a * nmh + mh) * npad), w);
          tc::tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(w[t]));
        }
        if (mrow < r) {
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int n = cg * 32 + t;
            if (n < r)
              out[(size_t)mrow * r + n] =
                  make_float2(live ? __uint_as_float(v[t]) * unscale * unscale : __int_as_float(0x7FC00000), 0.f);
          }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, cols);
}

// out[a][b] = sum over chunks c, in order, of partials[c][a][b] (TwoSum on the
// pairs), for the 4 x 4 blocks the partial kernel wrote (block row <= block
// column); the other entries are the mirror image.  grid (.., batch).
__global__ void gram_reduce_kernel(const GramBatch batch) {
  const GramEntry& en = batch.e[blockIdx.y];
  const int r = batch.r, rr = r * r;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= rr) return;
  int a = e / r, b = e % r;
  if (a / 4 > b / 4) {  // below the computed blocks: read the mirror
    const int t = a;
    a = b;
    b = t;
  }
  const int src = a * r + b;
  const int nchunks = gram_chunks_tc(en.rows, r).nchunks;
  float hi = 0.f, lo = 0.f;
#pragma unroll 8
  for (int c = 0; c < nchunks; ++c) {
    const float2 v = en.partials[(size_t)c * rr + src];
    acc2(hi, lo, v.x);
    lo = __fadd_rn(lo, v.y);
  }
  en.out[e] = (double)hi + (double)lo;
}

}  // namespace

cudaError_t launch_gram(const GramBatch& batch_in, cudaStream_t stream) {
  if (batch_in.n <= 0) return cudaSuccess;
  static thread_local GramBatch batch;
  batch = batch_in;
  const int r = batch.r;
  batch.chunk_begin[0] = 0;
  for (int i = 0; i < batch.n; ++i)
    batch.chunk_begin[i + 1] = batch.chunk_begin[i] + gram_chunks_tc(batch.e[i].rows, r).nchunks;
  // shared memory: two buffers of two tiles, or more, so that the blocks
  // resident on an SM never ask for more than its 512 TMEM columns
  const size_t tiles = (size_t)4 * gtc_mpad(r) * 128 + 1024;
  const int max_blocks = 512 / (int)gtc_tmem_cols(r);
  const size_t tmem_bound = (size_t)233472 / (size_t)(max_blocks + 1) - 1024 + 16;
  size_t smem = tiles > tmem_bound ? tiles : tmem_bound;
  // the ring of fp32 row copies in what the blocks an SM's TMEM admits leave
  // (each block also holds 1 KB reserved by the system and the kernel's
  // static shared memory)
  // (the static size is a property of the compiled kernel: asked once)
  static const size_t static_smem = [] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, gram_tc_kernel<2, true>) == cudaSuccess ? fa.sharedSizeBytes : (size_t)1024;
  }();
  cudaError_t err = cudaSuccess;
  const size_t per_block = (size_t)233472 / (size_t)max_blocks - 1024 - static_smem;
  const size_t raw_bytes = (size_t)kGtcStep * r * 4;
  int stages = per_block > tiles ? (int)((per_block - tiles) / raw_bytes) : 0;
  if (stages > kGtcMaxRaw) stages = kGtcMaxRaw;
  if (stages < 2 || r > 128) stages = 0;
  // the bulk copies need every A on 16 bytes and a whole number of 16-byte
  // pieces per chunk (chunks start on multiples of 64 rows)
  for (int i = 0; i < batch.n && stages > 0; ++i)
    if ((reinterpret_cast<uintptr_t>(batch.e[i].A) & 15) != 0 || (batch.e[i].rows * r) % 4 != 0) stages = 0;
  batch.raw_stages = stages;
  const int ipt = r <= 32 ? 1 : r <= 64 ? 2 : r <= 128 ? 4 : 8;
  auto kern = ipt == 1   ? gram_tc_kernel<1, false>
              : ipt == 2 ? (stages ? gram_tc_kernel<2, true> : gram_tc_kernel<2, false>)
              : ipt == 4 ? (stages ? gram_tc_kernel<4, true> : gram_tc_kernel<4, false>)
                         : gram_tc_kernel<8, false>;
  if (stages > 0 && tiles + stages * raw_bytes > smem) smem = tiles + stages * raw_bytes;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  count_launch();
  kern<<<(unsigned)batch.chunk_begin[batch.n], kGtcThreads, smem, stream>>>(batch);
  const int rr = r * r;
  count_launch();
  gram_reduce_kernel<<<dim3((unsigned)ceil_div(rr, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace rgs
