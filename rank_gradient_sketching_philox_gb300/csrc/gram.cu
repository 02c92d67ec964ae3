// Gram matrices G = A^T A of tall-skinny fp32 matrices (rows x r, r <= 256).
// Used by the CholeskyQR2 projection and by the normalized-SGD step, where
// ||C P^T||_F^2 = <P^T P, C^T C>.
//
// Two deterministic passes over a batch of matrices: partial Grams over at
// most 64 fixed row chunks, then a fixed-order sum over the chunks.  Within a
// chunk, products are summed in fp32 over 32-row tiles and the tiles are added
// with TwoSum into a (hi, lo) pair; the chunk sum carries the pairs the same
// way.  Only the 32-term tile sums round, so an entry is good to about 1e-7 of
// the sum of its |terms| however many rows there are, without FP64 arithmetic
// (far slower than fp32 on this GPU).  Neither pass uses atomics, so the
// result does not depend on scheduling.
#include "common.cuh"
#include "internal.h"

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

// Rows [row, row + 32) x columns [c0, c0 + 64) of A into registers: element
// (e / 16, 4 (e % 16) .. + 3) for e = threadIdx.x and threadIdx.x + 256; zero
// outside the matrix.  Vector loads when r is a multiple of 4.
__device__ __forceinline__ void load_rows(const float* __restrict__ A, int r, int64_t row, int64_t row_end, int c0,
                                          float4 (&v)[2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = threadIdx.x + 256 * h;
    const int64_t rw = row + (e >> 4);
    const int c = c0 + 4 * (e & 15);
    v[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (rw >= row_end) continue;
    const float* src = A + rw * r + c;
    if ((r & 3) == 0 && c + 3 < r) {
      v[h] = *reinterpret_cast<const float4*>(src);
    } else {
      if (c < r) v[h].x = src[0];
      if (c + 1 < r) v[h].y = src[1];
      if (c + 2 < r) v[h].z = src[2];
      if (c + 3 < r) v[h].w = src[3];
    }
  }
}

// grid (64 chunks, tile pairs ta <= tb, batch); block 256 = 16 x 16 threads.
// Thread (tx, ty) owns the 4 x 4 outputs a = a0 + 4ty + i, b = b0 + 4tx + j.
// The next 32 rows are loaded into registers while the current ones are used.
__global__ void __launch_bounds__(256) gram_partial_kernel(const GramBatch batch) {
  __shared__ __align__(16) float sa[kRows][kTile];
  __shared__ __align__(16) float sb[kRows][kTile];
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
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t row_begin = (int64_t)blockIdx.x * g.chunk_rows;
  int64_t row_end = row_begin + g.chunk_rows;
  if (row_end > en.rows) row_end = en.rows;
  const float* __restrict__ A = en.A;
  const float(*sbb)[kTile] = diag ? sa : sb;
  float hi[16], lo[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) hi[e] = lo[e] = 0.f;
  float4 va[2], vb[2];
  load_rows(A, r, row_begin, row_end, a0, va);
  if (!diag) load_rows(A, r, row_begin, row_end, b0, vb);
  for (int64_t base = row_begin; base < row_end; base += kRows) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = threadIdx.x + 256 * h;
      *reinterpret_cast<float4*>(&sa[e >> 4][4 * (e & 15)]) = va[h];
      if (!diag) *reinterpret_cast<float4*>(&sb[e >> 4][4 * (e & 15)]) = vb[h];
    }
    __syncthreads();
    if (base + kRows < row_end) {
      load_rows(A, r, base + kRows, row_end, a0, va);
      if (!diag) load_rows(A, r, base + kRows, row_end, b0, vb);
    }
    float t[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) t[e] = 0.f;
#pragma unroll 4
    for (int i = 0; i < kRows; ++i) {
      const float4 av = *reinterpret_cast<const float4*>(&sa[i][4 * ty]);
      const float4 bv = *reinterpret_cast<const float4*>(&sbb[i][4 * tx]);
      const float aa[4] = {av.x, av.y, av.z, av.w}, bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) t[4 * p + q] = fmaf(aa[p], bb[q], t[4 * p + q]);
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) acc2(hi[e], lo[e], t[e]);
    __syncthreads();
  }
  float2* out = en.partials + (size_t)blockIdx.x * r * r;
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int a = a0 + 4 * ty + p, b = b0 + 4 * tx + q;
      if (a < r && b < r) out[(size_t)a * r + b] = make_float2(hi[4 * p + q], lo[4 * p + q]);
    }
}

// out[a][b] = sum over chunks c, in order, of partials[c][a][b] (TwoSum on the
// pairs), for the tiles ta <= tb the partial kernel wrote; the other half is
// the mirror image.  grid (.., batch).
__global__ void gram_reduce_kernel(const GramBatch batch) {
  const GramEntry& en = batch.e[blockIdx.y];
  const int r = batch.r, rr = r * r;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= rr) return;
  int a = e / r, b = e % r;
  if (a / kTile > b / kTile) {  // below the computed tiles: read the mirror
    const int t = a;
    a = b;
    b = t;
  }
  const int src = a * r + b;
  const int nchunks = gram_chunks(en.rows).nchunks;
  float hi = 0.f, lo = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const float2 v = en.partials[(size_t)c * rr + src];
    acc2(hi, lo, v.x);
    lo = __fadd_rn(lo, v.y);
  }
  en.out[e] = (double)hi + (double)lo;
}

}  // namespace

cudaError_t launch_gram(const GramBatch& batch, cudaStream_t stream) {
  if (batch.n <= 0) return cudaSuccess;
  const int tiles = (int)ceil_div(batch.r, kTile);
  count_launch();
  gram_partial_kernel<<<dim3(64, tiles * (tiles + 1) / 2, batch.n), 256, 0, stream>>>(batch);
  const int rr = batch.r * batch.r;
  count_launch();
  gram_reduce_kernel<<<dim3((unsigned)ceil_div(rr, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace rgs
