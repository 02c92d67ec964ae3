// Gram matrices G = A^T A of tall-skinny fp32 matrices (rows x r, r <= 256).
// Used by the CholeskyQR2 projection and by the normalized-SGD step, where
// ||C P^T||_F^2 = <P^T P, C^T C>.
//
// Two deterministic passes over a batch of matrices: partial Grams over at
// most 64 fixed row chunks, then a fixed-order sum over the chunks.  Within a
// chunk, products are summed in fp32 over 32-row steps and the step sums are
// added with TwoSum into a (hi, lo) pair; the chunk sum carries the pairs the
// same way.  Only the 32-term tile sums round, so an entry is good to about 1e-7 of
// the sum of its |terms| however many rows there are, without FP64 arithmetic
// (far slower than fp32 on this GPU).  Neither pass uses atomics, so the
// result does not depend on scheduling.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace rgs {
namespace {

constexpr int kTile = 64;   // output tile edge
constexpr int kRows = 32;   // rows staged per step

// (hi, lo) += x with TwoSum (Knuth): exact error of the addition kept in lo.
__device__ __forceinline__ void acc2(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bb = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
  hi = s;
  lo = __fadd_rn(lo, e);
}

constexpr int kStages = 3;  // row steps in flight

// Asynchronous copy of rows [row, row + 32) x columns [c0, c0 + 64) of A into
// a 32 x 64 shared tile (elements e = threadIdx.x + 256h, h < 2: row e / 16,
// columns 4 (e % 16) .. + 3), zero outside the matrix.  16-byte copies when r is
// a multiple of 4, else 4-byte ones.
__device__ __forceinline__ void stage_rows(float* tile, const float* __restrict__ A, int r, int64_t row,
                                           int64_t row_end, int c0) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = threadIdx.x + 256 * h;
    const int64_t rw = row + (e >> 4);
    const int c = c0 + 4 * (e & 15);
    const uint32_t dst = (uint32_t)__cvta_generic_to_shared(tile + (e >> 4) * kTile + 4 * (e & 15));
    const bool row_in = rw < row_end;
    if ((r & 3) == 0) {
      const bool in = row_in && c < r;
      const float* src = in ? A + rw * r + c : A;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16 : 0)
                   : "memory");
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool in = row_in && c + q < r;
        const float* src = in ? A + rw * r + c + q : A;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst + 4 * q), "l"(src), "r"(in ? 4 : 0)
                     : "memory");
      }
    }
  }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Dynamic shared memory of the partial kernel: the staged rows (one 32 x 64
// tile per stage for a diagonal pair, two otherwise) and every thread's 16
// (hi, lo) pairs.
__host__ __device__ inline size_t gram_smem_bytes(bool two_tiles) {
  return sizeof(float) * ((size_t)kStages * (two_tiles ? 2 : 1) * kRows * kTile + 256 * 32);
}

// grid (64 chunks, tile pairs ta <= tb, batch); block 256.  A tile pair is
// 16 x 16 blocks of 4 x 4 outputs a = a0 + 4bi + i, b = b0 + 4bj + j.  An
// off-diagonal pair gives thread t the block (t / 16, t % 16); a diagonal one
// needs only its 136 blocks bi <= bj (the rest is the mirror image), so
// threads 0..135 take those in row order and the other warps only stage rows.
// Rows arrive by asynchronous copies kStages - 1 steps ahead; each thread's
// (hi, lo) pairs live in shared memory (touched once per 32 rows), which keeps
// its registers for the products.
__global__ void __launch_bounds__(256, 4) gram_partial_kernel(const GramBatch batch) {
  extern __shared__ __align__(16) float gsm[];
  const GramEntry& en = batch.e[blockIdx.z];
  const int r = batch.r;
  const GramChunks g = gram_chunks(en.rows);
  if ((int)blockIdx.x >= g.nchunks) return;
  const int tiles = (int)ceil_div(r, kTile);
  // blockIdx.y enumerates the pairs ta <= tb row by row
  int ta = 0, rem = (int)blockIdx.y;
  while (rem >= tiles - ta) {
    rem -= tiles - ta;
    ++ta;
  }
  const int tb = ta + rem;
  const bool diag = ta == tb;
  const int a0 = ta * kTile, b0 = tb * kTile;
  int bi, bj;
  bool active = true;
  if (diag) {
    int t = threadIdx.x;
    bi = 0;
    while (bi < 16 && t >= 16 - bi) {
      t -= 16 - bi;
      ++bi;
    }
    bj = bi + t;
    active = threadIdx.x < 136;
  } else {
    bi = threadIdx.x >> 4;
    bj = threadIdx.x & 15;
  }
  const int64_t row_begin = (int64_t)blockIdx.x * g.chunk_rows;
  int64_t row_end = row_begin + g.chunk_rows;
  if (row_end > en.rows) row_end = en.rows;
  const int nsteps = (int)ceil_div(row_end - row_begin, kRows);
  const float* __restrict__ A = en.A;
  const int tile_floats = kRows * kTile;
  float* sa = gsm;                                       // kStages x (32 x 64)
  float* sb = diag ? sa : gsm + kStages * tile_floats;   // kStages x (32 x 64)
  float4* hl = reinterpret_cast<float4*>(gsm + kStages * tile_floats * (diag ? 1 : 2));  // [8][256]
#pragma unroll
  for (int q = 0; q < 8; ++q) hl[q * 256 + threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < nsteps) {
      stage_rows(sa + st * tile_floats, A, r, row_begin + (int64_t)st * kRows, row_end, a0);
      if (!diag) stage_rows(sb + st * tile_floats, A, r, row_begin + (int64_t)st * kRows, row_end, b0);
    }
    cp_async_commit();
  }
  for (int step = 0; step < nsteps; ++step) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // this step's rows are in; the slot refilled below is free
    {
      const int nx = step + kStages - 1;
      if (nx < nsteps) {
        const int slot = nx % kStages;
        stage_rows(sa + slot * tile_floats, A, r, row_begin + (int64_t)nx * kRows, row_end, a0);
        if (!diag) stage_rows(sb + slot * tile_floats, A, r, row_begin + (int64_t)nx * kRows, row_end, b0);
      }
      cp_async_commit();
    }
    if (active) {
      const float* ta_s = sa + (step % kStages) * tile_floats;
      const float* tb_s = sb + (step % kStages) * tile_floats;
      float t[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) t[e] = 0.f;
#pragma unroll 4
      for (int i = 0; i < kRows; ++i) {
        const float4 av = *reinterpret_cast<const float4*>(ta_s + i * kTile + 4 * bi);
        const float4 bv = *reinterpret_cast<const float4*>(tb_s + i * kTile + 4 * bj);
        const float aa[4] = {av.x, av.y, av.z, av.w}, bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) t[4 * p + q] = fmaf(aa[p], bb[q], t[4 * p + q]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 h = hl[q * 256 + threadIdx.x], l = hl[(4 + q) * 256 + threadIdx.x];
        acc2(h.x, l.x, t[4 * q + 0]);
        acc2(h.y, l.y, t[4 * q + 1]);
        acc2(h.z, l.z, t[4 * q + 2]);
        acc2(h.w, l.w, t[4 * q + 3]);
        hl[q * 256 + threadIdx.x] = h;
        hl[(4 + q) * 256 + threadIdx.x] = l;
      }
    }
  }
  cp_async_wait<0>();
  if (!active) return;
  float2* out = en.partials + (size_t)blockIdx.x * r * r;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float4 h = hl[p * 256 + threadIdx.x], l = hl[(4 + p) * 256 + threadIdx.x];
    const float hv[4] = {h.x, h.y, h.z, h.w}, lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + 4 * bi + p, b = b0 + 4 * bj + q;
      if (a < r && b < r) out[(size_t)a * r + b] = make_float2(hv[q], lv[q]);
    }
  }
}

// ---- tensor-core partial Gram ------------------------------------------------
// Chunks of gram_chunks_tc rows, one block per (chunk, matrix), the products
// on the tensor cores: the chunk's largest magnitude gives a power
// of two 2^e that brings it into [2^14, 2^15); each element x 2^e is split into
// FP16 high and low parts (hi + lo within ~2^-22 of it) written, 64 rows at a
// time, into shared-memory tiles laid out as the MMA's K-major operand (column m
// of A is row m of the tile, 128-byte swizzle), two sets of tiles so that one
// step's conversion overlaps the previous step's MMAs; tcgen05.mma (kind::f16,
// M = 128, N = r rounded to 16, K = 16) accumulates hi hi + hi lo + lo hi of
// A^T A into TMEM (two M halves when r > 128), the steps going to the
// gram_tc_accs accumulators in turn; warps 0..3, one per TMEM lane quarter, add
// the accumulators and scale the sums by 2^-2e into the chunk's partial (written with a
// zero low word), which gram_reduce_kernel adds up as for the SIMT kernel.
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
__device__ __forceinline__ uint32_t gtc_pack(float y0, float y1, uint32_t& lo) {
  const __half h0 = __float2half_rn(y0), h1 = __float2half_rn(y1);
  const __half l0 = __float2half_rn(y0 - __half2float(h0)), l1 = __float2half_rn(y1 - __half2float(h1));
  lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
  return (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
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
// column.  The next step's items are loaded into registers while this step's
// are converted.
template <int IPT>
__global__ void __launch_bounds__(kGtcThreads) gram_tc_kernel(const GramBatch batch) {
  extern __shared__ uint8_t gtc_raw[];
  __shared__ __align__(8) uint64_t mma_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float wmax[kGtcThreads / 32];
  __shared__ volatile int abort_flag;
  const GramEntry& en = batch.e[blockIdx.y];
  const int r = batch.r;
  const GramChunks g = gram_chunks_tc(en.rows, r);
  if ((int)blockIdx.x >= g.nchunks) return;  // the same for the whole block
  const int mpad = gtc_mpad(r), npad = gtc_npad(r), nmh = mpad / 128, nacc = gram_tc_accs(r);
  const uint32_t cols = gtc_tmem_cols(r);
  const uint32_t tile_bytes = (uint32_t)mpad * 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // buffer b: hi tile at base + 2 b tile_bytes, lo tile right after it
  const uint32_t base = tc::smem_u32(gtc_align1024(gtc_raw));
  const int64_t row_begin = (int64_t)blockIdx.x * g.chunk_rows;
  const int64_t row_end = row_begin + g.chunk_rows < en.rows ? row_begin + g.chunk_rows : en.rows;
  const float* __restrict__ A = en.A;
  if (tid == 0) {
    abort_flag = 0;
    tc::mbar_init(&mma_bar[0], 1);
    tc::mbar_init(&mma_bar[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, cols);
  // every tile zero: rows m >= r (padding to the MMA's M and N) stay so
  for (uint32_t e = tid; e < 4 * tile_bytes / 16; e += kGtcThreads) tc::sts128(base + 16u * e, make_uint4(0, 0, 0, 0));
  // the largest magnitude: given by the producer of A (a bound, or the maximum
  // it recorded), else the chunk's own (NaN if any element is NaN)
  const bool given = en.amax != nullptr || en.bound > 0.f;
  float m = 0.f;
  if (!given) {
    m = gtc_chunk_max(A + row_begin * r, (row_end - row_begin) * r);
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
  if (nsteps > 0) load_step(0);
  bool live = true;
  for (int st = 0; st < nsteps; ++st) {
    const int b = st & 1;
    const uint32_t hi_s = base + 2u * b * tile_bytes, lo_s = hi_s + tile_bytes;
    float xc[IPT][8];
#pragma unroll
    for (int q = 0; q < IPT; ++q)
#pragma unroll
      for (int t = 0; t < 8; ++t) xc[q][t] = xn[q][t];
    if (st + 1 < nsteps) load_step(st + 1);
    if (st >= 2) {  // the MMAs of step st - 2 have read this buffer
      live = tc::mbar_wait(&mma_bar[b], (uint32_t)((st >> 1) - 1) & 1u, &abort_flag, nullptr, 0);
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
        for (int t = 0; t < 4; ++t) hv[t] = gtc_pack(xc[q][2 * t] * scale, xc[q][2 * t + 1] * scale, lv[t]);
        const uint32_t off = (uint32_t)((mc >> 3) * 1024 + (mc & 7) * 128 + ((k8 ^ (mc & 7)) << 4));
        tc::sts128(hi_s + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
        tc::sts128(lo_s + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
      }
    }
  tc::fence_proxy_async_smem();
    live = __syncthreads_and(live);
    if (!live) break;
    if (tid == 0) {
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
  }
  if (live)
    live = tc::mbar_wait(&mma_bar[(nsteps - 1) & 1], (uint32_t)((nsteps - 1) >> 1) & 1u, &abort_flag, nullptr, 0);
  live = __syncthreads_and(live);
  tc::tc_fence_after();
  // warps 0..3: the sums of TMEM lane m (row m of A^T A) scaled back by
  // 2^-2e; a wait that gave up leaves the partial NaN
  if (warp < 4) {
    float2* out = en.partials + (size_t)blockIdx.x * r * r;
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
  const int nchunks = batch.tc ? gram_chunks_tc(en.rows, r).nchunks : gram_chunks(en.rows).nchunks;
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

cudaError_t launch_gram(const GramBatch& batch_in, cudaStream_t stream, bool tensor_cores) {
  if (batch_in.n <= 0) return cudaSuccess;
  static thread_local GramBatch batch;
  batch = batch_in;
  batch.tc = tensor_cores ? 1 : 0;
  cudaError_t err = cudaSuccess;
  if (tensor_cores) {
    // shared memory: two buffers of two tiles, or more, so that the blocks
    // resident on an SM never ask for more than its 512 TMEM columns
    const int r = batch.r;
    const size_t tiles = (size_t)4 * gtc_mpad(r) * 128 + 1024;
    const int max_blocks = 512 / (int)gtc_tmem_cols(r);
    const size_t tmem_bound = (size_t)233472 / (size_t)(max_blocks + 1) - 1024 + 16;
    const size_t smem = tiles > tmem_bound ? tiles : tmem_bound;
    const int ipt = r <= 32 ? 1 : r <= 64 ? 2 : r <= 128 ? 4 : 8;
    auto kern = ipt == 1 ? gram_tc_kernel<1> : ipt == 2 ? gram_tc_kernel<2> : ipt == 4 ? gram_tc_kernel<4> : gram_tc_kernel<8>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    count_launch();
    kern<<<dim3(64, batch.n), kGtcThreads, smem, stream>>>(batch);
  } else {
    const int tiles = (int)ceil_div(batch.r, kTile);
    const size_t smem = gram_smem_bytes(tiles > 1);
    err = cudaFuncSetAttribute(gram_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    count_launch();
    gram_partial_kernel<<<dim3(64, tiles * (tiles + 1) / 2, batch.n), 256, smem, stream>>>(batch);
  }
  const int rr = batch.r * batch.r;
  count_launch();
  gram_reduce_kernel<<<dim3((unsigned)ceil_div(rr, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace rgs
