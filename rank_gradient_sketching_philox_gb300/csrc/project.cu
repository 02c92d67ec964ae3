// (b) XP = X P, the projected input saved for backpropagation instead of X
// ("Randomized Gradient Compression", "How it works").  fp32 accumulation,
// one round-to-nearest-even to BF16 at the end.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace rgs {
namespace {

// SIMT tile: 64 tokens x 64 rank columns per block, k consumed 32 at a time.
// Thread (ty, tx) = (tid / 16, tid % 16) owns tokens ty*4+i, columns tx*4+j.
__global__ void __launch_bounds__(256) project_simt_kernel(const uint16_t* __restrict__ X, int64_t T,
                                                          int64_t k, int64_t ld_x,
                                                          const float* __restrict__ P, int r,
                                                          uint16_t* __restrict__ XP, int64_t ld_xp) {
  __shared__ float xs[32][64 + 4];  // [k within chunk][token]
  __shared__ float ps[32][64 + 4];  // [k within chunk][column]
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t t0 = (int64_t)blockIdx.x * 64;
  const int c0 = blockIdx.y * 64;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < k; k0 += 32) {
    {  // X chunk: 64 tokens x 32 k, one 8-element vector per thread
      const int tok = tid >> 2, kq = (tid & 3) * 8;
      const int64_t t = t0 + tok, j = k0 + kq;
      float v[8];
      if (t < T && j < k) {
        const uint4 raw = *reinterpret_cast<const uint4*>(X + t * ld_x + j);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[2 * q] = bf16_bits_to_float(w[q] & 0xFFFFu);
          v[2 * q + 1] = bf16_bits_to_float(w[q] >> 16);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[kq + q][tok] = v[q];
    }
    for (int e = tid; e < 32 * 64; e += 256) {  // P chunk: 32 k x 64 columns
      const int kk = e >> 6, c = e & 63;
      const int64_t j = k0 + kk;
      ps[kk][c] = (j < k && c0 + c < r) ? P[j * r + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ps[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < r) XP[t * ld_xp + c] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][j]));
    }
  }
}

}  // namespace

size_t project_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_project_inputs(const uint16_t* X, int64_t T, int64_t k, int64_t ld_x,
                                  const float* P, int r, uint16_t* XP, int64_t ld_xp, void*,
                                  cudaStream_t stream) {
  dim3 grid((unsigned)ceil_div(T, 64), (unsigned)ceil_div(r, 64));
  project_simt_kernel<<<grid, 256, 0, stream>>>(X, T, k, ld_x, P, r, XP, ld_xp);
  return cudaGetLastError();
}

}  // namespace rgs
