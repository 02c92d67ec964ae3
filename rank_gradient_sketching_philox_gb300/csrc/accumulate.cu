// (c) C = (overwrite ? 0 : C) + D^T XP in fp32 for one microbatch
// ("Randomized Gradient Compression", "How it works": C += D.T (X P);
// "LoGRA: Scaling LLM Reinforcement Learning with Low-Rank Gradient Sketches",
// Key Contributions 1: the sketch is accumulated in fp32 and the d x k
// gradient is never formed).
#include "common.cuh"
#include "internal.h"

namespace rgs {
namespace {

// SIMT tile: 64 rows of C (columns of D) x 64 rank columns, tokens consumed 32
// at a time.  Thread (ty, tx) = (tid / 16, tid % 16) owns rows ty*4+i, columns
// tx*4+j.
__global__ void __launch_bounds__(256) accumulate_simt_kernel(const uint16_t* __restrict__ D,
                                                             int64_t T, int64_t d, int64_t ld_d,
                                                             const uint16_t* __restrict__ XP,
                                                             int64_t ld_xp, int r,
                                                             float* __restrict__ C, int overwrite) {
  __shared__ float ds[32][64 + 4];  // [token][row of C]
  __shared__ float xs[32][64 + 4];  // [token][rank column]
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int64_t i0 = (int64_t)blockIdx.x * 64;
  const int c0 = blockIdx.y * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t row = i0 + ty * 4 + i;
      const int c = c0 + tx * 4 + j;
      acc[i][j] = (!overwrite && row < d && c < r) ? C[row * r + c] : 0.f;
    }
  for (int64_t t0 = 0; t0 < T; t0 += 32) {
    {  // D chunk: 32 tokens x 64 rows, one 8-element vector per thread
      const int tt = tid >> 3, iv = (tid & 7) * 8;
      const int64_t t = t0 + tt, row = i0 + iv;
      float v[8];
      if (t < T && row + 8 <= d) {
        const uint4 raw = *reinterpret_cast<const uint4*>(D + t * ld_d + row);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[2 * q] = bf16_bits_to_float(w[q] & 0xFFFFu);
          v[2 * q + 1] = bf16_bits_to_float(w[q] >> 16);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = (t < T && row + q < d) ? bf16_bits_to_float(D[t * ld_d + row + q]) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) ds[tt][iv + q] = v[q];
    }
    for (int e = tid; e < 32 * 64; e += 256) {  // XP chunk: 32 tokens x 64 columns
      const int tt = e >> 6, c = e & 63;
      const int64_t t = t0 + tt;
      xs[tt][c] = (t < T && c0 + c < r) ? bf16_bits_to_float(XP[t * ld_xp + c0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int tt = 0; tt < 32; ++tt) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = ds[tt][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = xs[tt][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t row = i0 + ty * 4 + i;
    if (row >= d) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < r) C[row * r + c] = acc[i][j];
    }
  }
}

}  // namespace

size_t accumulate_workspace_bytes(int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_accumulate(const uint16_t* D, int64_t T, int64_t d, int64_t ld_d,
                              const uint16_t* XP, int64_t ld_xp, int r, float* C, int overwrite,
                              void*, cudaStream_t stream) {
  dim3 grid((unsigned)ceil_div(d, 64), (unsigned)ceil_div(r, 64));
  accumulate_simt_kernel<<<grid, 256, 0, stream>>>(D, T, d, ld_d, XP, ld_xp, r, C, overwrite);
  return cudaGetLastError();
}

}  // namespace rgs
