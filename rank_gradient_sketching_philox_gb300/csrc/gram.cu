// Gram matrices G = A^T A of tall-skinny fp32 matrices (rows x r, r <= 256).
// Used by the CholeskyQR2 projection and by the normalized-SGD step, where
// ||C P^T||_F^2 = <P^T P, C^T C>.
//
// Two deterministic passes over a batch of matrices: partial Grams over at
// most 64 fixed row chunks, then a fixed-order sum over the chunks.  Products
// are summed in fp32 over 32-row tiles and the tiles in double, so an entry is
// good to about 1e-8 relative.  Neither pass uses atomics, so the result does
// not depend on scheduling.
#include "common.cuh"
#include "internal.h"

namespace rgs {
namespace {

constexpr int kTile = 32;

// grid (64 chunks, tiles*tiles, batch); block 256 = 32 x 8 threads.
// Thread (tx, ty) owns outputs (a = a0 + ty + 8m, b = b0 + tx), m = 0..3.
__global__ void __launch_bounds__(256) gram_partial_kernel(const GramBatch batch) {
  __shared__ float sa[kTile][kTile + 1];
  __shared__ float sb[kTile][kTile + 1];
  const GramEntry& en = batch.e[blockIdx.z];
  const int r = batch.r;
  const GramChunks g = gram_chunks(en.rows);
  if ((int)blockIdx.x >= g.nchunks) return;
  const int tiles = (int)ceil_div(r, kTile);
  const int a0 = (blockIdx.y / tiles) * kTile, b0 = (blockIdx.y % tiles) * kTile;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t row_begin = (int64_t)blockIdx.x * g.chunk_rows;
  int64_t row_end = row_begin + g.chunk_rows;
  if (row_end > en.rows) row_end = en.rows;
  const float* __restrict__ A = en.A;
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  for (int64_t base = row_begin; base < row_end; base += kTile) {
    for (int i = ty; i < kTile; i += 8) {
      const int64_t row = base + i;
      const bool ok = row < row_end;
      sa[i][tx] = (ok && a0 + tx < r) ? A[row * r + a0 + tx] : 0.f;
      sb[i][tx] = (ok && b0 + tx < r) ? A[row * r + b0 + tx] : 0.f;
    }
    __syncthreads();
    float tile[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < kTile; ++i) {
      const float bv = sb[i][tx];
#pragma unroll
      for (int m = 0; m < 4; ++m) tile[m] = fmaf(sa[i][ty + 8 * m], bv, tile[m]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[m] += (double)tile[m];
    __syncthreads();
  }
  double* out = en.partials + (size_t)blockIdx.x * r * r;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int a = a0 + ty + 8 * m, b = b0 + tx;
    if (a < r && b < r) out[(size_t)a * r + b] = acc[m];
  }
}

// out[e] = sum over chunks c, in order, of partials[c][e].  grid (.., batch).
__global__ void gram_reduce_kernel(const GramBatch batch) {
  const GramEntry& en = batch.e[blockIdx.y];
  const int rr = batch.r * batch.r;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= rr) return;
  const int nchunks = gram_chunks(en.rows).nchunks;
  double s = 0.0;
  for (int c = 0; c < nchunks; ++c) s += en.partials[(size_t)c * rr + e];
  en.out[e] = s;
}

}  // namespace

cudaError_t launch_gram(const GramBatch& batch, cudaStream_t stream) {
  if (batch.n <= 0) return cudaSuccess;
  const int tiles = (int)ceil_div(batch.r, kTile);
  count_launch();
  gram_partial_kernel<<<dim3(64, tiles * tiles, batch.n), 256, 0, stream>>>(batch);
  const int rr = batch.r * batch.r;
  count_launch();
  gram_reduce_kernel<<<dim3((unsigned)ceil_div(rr, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace rgs
