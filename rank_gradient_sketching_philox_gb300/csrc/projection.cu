// (a) Projection P (k x r fp32): Rademacher signs or a Gaussian-QR frame.
//
// Rademacher: entries +-1/sqrt(r) ("LoGRA: Low-Rank Gradient Sketches", "Why
// the Sketch Can Be Accumulated Without a Full Gradient").  Element e = j*r + l
// takes bit e % 128 of Philox block e / 128 of the sign stream.
//
// Gaussian QR: P = sqrt(k/r) Q with Q the orthonormal factor of a Gaussian
// k x r matrix and diag(R) > 0 ("Randomized Gradient Compression",
// footnote 1).  The frame is computed by CholeskyQR2 in fp32: twice
// (Gram A = G^T G, Cholesky A = R^T R, G <- G R^-1).  Cholesky factors have a
// positive diagonal, so the result is the sign-corrected QR factor without an
// explicit sign fix.  For 4r <= k the Gaussian matrix is well conditioned and
// the second pass leaves P^T P = (k/r) I to about 1e-6.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace rgs {
namespace {

// One thread per 32 consecutive elements (one 32-bit word of a Philox block).
__global__ void __launch_bounds__(256) rademacher_kernel(const ProjBatch batch) {
  const ProjProblem& pb = batch.p[blockIdx.y];
  const int64_t n = pb.k * batch.r;
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t e0 = w * 32;
  if (e0 >= n) return;
  const Philox4 blk = stream_block(batch.seed, pb.layer, batch.step, kTagRademacher, (uint32_t)(w >> 2));
  const uint32_t word = (w & 3) == 0 ? blk.w0 : (w & 3) == 1 ? blk.w1 : (w & 3) == 2 ? blk.w2 : blk.w3;
  const float pos = pb.scale, neg = -pb.scale;
  float4* out = reinterpret_cast<float4*>(pb.P + e0);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    if (e0 + 4 * q >= n) break;  // n is a multiple of 8
    const uint32_t bits = word >> (4 * q);
    float4 v;
    v.x = (bits & 1u) ? neg : pos;
    v.y = (bits & 2u) ? neg : pos;
    v.z = (bits & 4u) ? neg : pos;
    v.w = (bits & 8u) ? neg : pos;
    out[q] = v;
  }
}

// Box-Muller on one Philox block: 4 standard normal draws for elements
// 4b .. 4b+3; lanes 0,1 use words (0,1) and lanes 2,3 use words (2,3); even
// lanes take the cosine branch, odd lanes the sine branch.  u = (w + 1/2) 2^-32.
// The hardware approximations serve: the draws only seed the QR frame, which is
// checked against the exact frame to 1e-5, and their errors (a few 2^-22
// absolute) are far below that.  cos and sin of 2 pi u are taken as -cos and
// -sin of 2 pi (u - 1/2), an argument in [-pi, pi) where the approximations hold
// their bound.
__device__ __forceinline__ float4 gaussian4(const Philox4& blk) {
  const float u0 = fmaf((float)blk.w0, 0x1p-32f, 0x1p-33f);
  const float u1 = fmaf((float)blk.w1, 0x1p-32f, 0x1p-33f);
  const float u2 = fmaf((float)blk.w2, 0x1p-32f, 0x1p-33f);
  const float u3 = fmaf((float)blk.w3, 0x1p-32f, 0x1p-33f);
  constexpr float kTwoPi = 6.28318530717958647692f;
  const float ra = sqrtf(-2.0f * __logf(u0));
  const float rb = sqrtf(-2.0f * __logf(u2));
  float sa, ca, sb, cb;
  __sincosf(kTwoPi * (u1 - 0.5f), &sa, &ca);
  __sincosf(kTwoPi * (u3 - 0.5f), &sb, &cb);
  return make_float4(-ra * ca, -ra * sa, -rb * cb, -rb * sb);
}

__global__ void __launch_bounds__(256) gaussian_kernel(const ProjBatch batch) {
  const ProjProblem& pb = batch.p[blockIdx.y];
  const int64_t n = pb.k * batch.r;
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (4 * b >= n) return;
  const Philox4 blk = stream_block(batch.seed, pb.layer, batch.step, kTagGaussian, (uint32_t)b);
  reinterpret_cast<float4*>(pb.P)[b] = gaussian4(blk);
}

__device__ __forceinline__ int packed_upper(int i, int j, int r) {
  return i * r - (i * (i - 1)) / 2 + (j - i);
}

// One block per problem: R with Gram = R^T R (Cholesky, upper triangular) and
// its inverse X = R^-1, written in full (zeros below the diagonal) to pb.rinv.
// Blocked in 32 x 32 tiles so that the block synchronises a few times per tile
// row rather than a few times per matrix row: the upper tiles live in shared
// memory (row stride 33, so that columns of a tile fall in distinct banks), the
// matrix padded to a multiple of 32 with the identity.
//   Cholesky, right-looking, per tile column k: one warp factors the diagonal
//   tile; each thread solves one column of the tile row (R_kj = R_kk^-T A_kj);
//   every warp updates four rows of the trailing tiles (A_ij -= R_ki^T R_kj).
//   Inverse: each warp inverts one diagonal tile (X_kk = R_kk^-1, one column per
//   lane); then tile rows from the bottom: X_ij = -X_ii (sum over i < m <= j of
//   R_im X_mj), the sums first (into scratch), then the products, which replace
//   row i of R, no longer needed.
constexpr int kCT = 32, kCTs = 33;  // tile size and row stride (floats)
__host__ __device__ inline int chol_tiles(int r) { return (r + kCT - 1) / kCT; }
__host__ __device__ inline size_t chol_smem_floats(int r) {
  const int nb = chol_tiles(r);
  return ((size_t)nb * (nb + 1) / 2 + nb) * kCT * kCTs;  // upper tiles, then a tile row of scratch
}
__device__ __forceinline__ float* chol_tile(float* S, int nb, int bi, int bj) {
  return S + (size_t)(bi * nb - bi * (bi - 1) / 2 + (bj - bi)) * (kCT * kCTs);
}
__global__ void __launch_bounds__(256) chol_inv_kernel(const ProjBatch batch) {
  extern __shared__ float S[];
  __shared__ int broken;
  const ProjProblem& pb = batch.p[blockIdx.x];
  const int r = batch.r, nb = chol_tiles(r);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = 8;
  float* T = S + (size_t)nb * (nb + 1) / 2 * (kCT * kCTs);  // scratch: nb tiles
  if (tid == 0) broken = 0;
  for (int bi = 0; bi < nb; ++bi)
    for (int bj = bi; bj < nb; ++bj) {
      float* B = chol_tile(S, nb, bi, bj);
      for (int e = tid; e < kCT * kCT; e += 256) {
        const int a = e >> 5, c = e & 31, i = bi * kCT + a, j = bj * kCT + c;
        B[a * kCTs + c] = (i < r && j < r) ? (float)pb.gram[(size_t)i * r + j] : (i == j ? 1.0f : 0.0f);
      }
    }
  __syncthreads();

  // ---- Cholesky ----
  for (int k = 0; k < nb; ++k) {
    float* D = chol_tile(S, nb, k, k);
    if (warp == 0) {  // the diagonal tile, in place
      for (int p = 0; p < kCT; ++p) {
        const float d = D[p * kCTs + p];
        if (!(d > 0.0f) || !isfinite(d)) {  // the same in every lane
          if (lane == 0) broken = 1;
          break;
        }
        const float rp = sqrtf(d), inv = 1.0f / rp;
        __syncwarp();
        const float rpl = lane > p ? D[p * kCTs + lane] * inv : 0.0f;
        if (lane > p) D[p * kCTs + lane] = rpl;
        if (lane == p) D[p * kCTs + p] = rp;
        __syncwarp();
        if (lane > p)
          for (int i = p + 1; i <= lane; ++i) D[i * kCTs + lane] = fmaf(-D[p * kCTs + i], rpl, D[i * kCTs + lane]);
        __syncwarp();
      }
    }
    __syncthreads();
    if (broken) break;
    // tile row k: R_kj = R_kk^-T A_kj, one column per thread (forward substitution)
    for (int cidx = tid; cidx < (nb - 1 - k) * kCT; cidx += 256) {
      float* B = chol_tile(S, nb, k, k + 1 + (cidx >> 5));
      const int c = cidx & 31;
      for (int p = 0; p < kCT; ++p) {
        float v = B[p * kCTs + c];
        for (int m = 0; m < p; ++m) v = fmaf(-D[m * kCTs + p], B[m * kCTs + c], v);
        B[p * kCTs + c] = v / D[p * kCTs + p];
      }
    }
    __syncthreads();
    // trailing tiles k < bi <= bj: A_ij -= R_ki^T R_kj, four rows per warp step
    const int nt = nb - 1 - k, npairs = nt * (nt + 1) / 2;
    for (int u = warp; u < npairs * 8; u += kWarps) {
      int pr = u >> 3, bi = k + 1;
      for (int len = nt; pr >= len; pr -= len, --len) ++bi;
      const int bj = bi + pr, a0 = (u & 7) * 4;
      const float* Ri = chol_tile(S, nb, k, bi);
      const float* Rj = chol_tile(S, nb, k, bj);
      float* A = chol_tile(S, nb, bi, bj);
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int p = 0; p < kCT; ++p) {
        const float rj = Rj[p * kCTs + lane];
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t] = fmaf(Ri[p * kCTs + a0 + t], rj, acc[t]);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) A[(a0 + t) * kCTs + lane] -= acc[t];
    }
    __syncthreads();
  }
  if (broken) {
    for (int e = tid; e < r * r; e += 256) pb.rinv[e] = 0.0f;
    if (tid == 0) atomicOr(batch.status, SKETCH_DEV_QR_BREAKDOWN);
    return;
  }

  // ---- inverse: diagonal tiles, one warp each, one column per lane ----
  for (int k = warp; k < nb; k += kWarps) {
    const float* D = chol_tile(S, nb, k, k);
    float* X = T + (size_t)k * (kCT * kCTs);
    const int j = lane;
    X[j * kCTs + j] = 1.0f / D[j * kCTs + j];
    for (int i = j - 1; i >= 0; --i) {
      float s = 0.0f;
      for (int m = i + 1; m <= j; ++m) s = fmaf(D[i * kCTs + m], X[m * kCTs + j], s);
      X[i * kCTs + j] = -s / D[i * kCTs + i];
    }
    for (int i = j + 1; i < kCT; ++i) X[i * kCTs + j] = 0.0f;
    __syncwarp();
    float* Dw = chol_tile(S, nb, k, k);
    for (int i = 0; i < kCT; ++i) Dw[i * kCTs + lane] = X[i * kCTs + lane];
  }
  __syncthreads();
  // ---- inverse: off-diagonal tiles, tile rows from the bottom ----
  for (int bi = nb - 2; bi >= 0; --bi) {
    const int nt = nb - 1 - bi;
    // sums: T_j = sum_{bi < m <= bj} R_{bi,m} X_{m,bj}, into scratch tile j - bi - 1
    for (int u = warp; u < nt * 8; u += kWarps) {
      const int bj = bi + 1 + (u >> 3), a0 = (u & 7) * 4;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int m = bi + 1; m <= bj; ++m) {
        const float* Rm = chol_tile(S, nb, bi, m);
        const float* Xm = chol_tile(S, nb, m, bj);
        for (int p = 0; p < kCT; ++p) {
          const float x = Xm[p * kCTs + lane];
#pragma unroll
          for (int t = 0; t < 4; ++t) acc[t] = fmaf(Rm[(a0 + t) * kCTs + p], x, acc[t]);
        }
      }
      float* Tj = T + (size_t)(bj - bi - 1) * (kCT * kCTs);
#pragma unroll
      for (int t = 0; t < 4; ++t) Tj[(a0 + t) * kCTs + lane] = acc[t];
    }
    __syncthreads();
    // products: X_{bi,bj} = -X_{bi,bi} T_j, over row bi of R (no longer needed)
    const float* Xd = chol_tile(S, nb, bi, bi);
    for (int u = warp; u < nt * 8; u += kWarps) {
      const int bj = bi + 1 + (u >> 3), a0 = (u & 7) * 4;
      const float* Tj = T + (size_t)(bj - bi - 1) * (kCT * kCTs);
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int p = 0; p < kCT; ++p) {
        const float tv = Tj[p * kCTs + lane];
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t] = fmaf(Xd[(a0 + t) * kCTs + p], tv, acc[t]);
      }
      float* O = chol_tile(S, nb, bi, bj);
#pragma unroll
      for (int t = 0; t < 4; ++t) O[(a0 + t) * kCTs + lane] = -acc[t];
    }
    __syncthreads();
  }
  // ---- out: X in full, zeros below the diagonal ----
  for (int e = tid; e < r * r; e += 256) {
    const int i = e / r, j = e % r;
    pb.rinv[e] = (j < i) ? 0.0f : chol_tile(S, nb, i >> 5, j >> 5)[(i & 31) * kCTs + (j & 31)];
  }
}

// P rows [32*blockIdx.x, +32) <- scale * P_rows * Rinv (Rinv upper triangular).
// P rows <- (P rows) X, X = R^-1 upper triangular, in place; on the final pass
// also times the scale sqrt(k/r).  With r8 = r rounded up to 8 and co = r8/8
// column octets, a block of 256 threads takes RB = 8 * floor(256 / co) rows and
// all columns: thread t < RB/8 * co owns the 8 x 8 outputs of column octet
// t % co and row octet t / co (the rest only help to stage).  The block's
// rows are staged (transposed) in shared memory first, so the in-place writes
// cannot race its reads; X follows 32 rows at a time.  Per row m of X a thread
// reads 8 staged values and 8 X values (four 16-byte shared loads) for 64 FMAs.
constexpr int kXRows = 32;
__host__ __device__ inline int tri_rows(int r) { return 8 * (256 / ((r + 7) / 8)); }
__host__ __device__ inline size_t tri_smem_floats(int r) {
  const int r8 = (r + 7) / 8 * 8, rb = tri_rows(r);
  return (size_t)r * (rb + 4) + 4 + (size_t)kXRows * r8;
}
__global__ void __launch_bounds__(256) tri_apply_kernel(const ProjBatch batch, int final_pass) {
  extern __shared__ __align__(16) float smem[];
  const ProjProblem& pb = batch.p[blockIdx.y];
  const int r = batch.r, r8 = (r + 7) / 8 * 8, co_n = r8 / 8, RB = tri_rows(r), ldt = RB + 4;
  float* St = smem;                                   // r x (RB + 4): St[m][row]
  float* Xs = smem + (((size_t)r * ldt + 3) & ~size_t(3));  // kXRows x r8
  const int64_t row0 = (int64_t)blockIdx.x * RB;
  if (row0 >= pb.k) return;
  const int rows = (int)((pb.k - row0) < RB ? (pb.k - row0) : RB);
  float* P = pb.P + row0 * r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Staging: thread t takes rows t, t + 256, ... and reads each in pieces of up
  // to 64 values, all loads of a piece issued before its transposed stores
  // (consecutive threads write consecutive rows: no bank conflicts).
  if ((r & 3) == 0) {
    const int nv = r >> 2;  // float4 per row
    for (int row = threadIdx.x; row < rows; row += 256) {
      const float4* src = reinterpret_cast<const float4*>(P + (size_t)row * r);
      for (int c0 = 0; c0 < nv; c0 += 16) {
        float4 v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = (c0 + m < nv) ? src[c0 + m] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          if (c0 + m >= nv) break;
          float* dst = St + (size_t)(4 * (c0 + m)) * ldt + row;
          dst[0] = v[m].x;
          dst[ldt] = v[m].y;
          dst[2 * ldt] = v[m].z;
          dst[3 * ldt] = v[m].w;
        }
      }
    }
  } else {
    for (int row = threadIdx.x; row < rows; row += 256) {
      const float* src = P + (size_t)row * r;
      for (int c0 = 0; c0 < r; c0 += 16) {
        float v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = (c0 + m < r) ? src[c0 + m] : 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (c0 + m < r) St[(size_t)(c0 + m) * ldt + row] = v[m];
      }
    }
  }
  const int co = threadIdx.x % co_n, ro = threadIdx.x / co_n;
  const bool active = ro < RB / 8;
  const int c0 = 8 * co, q0 = 8 * ro;
  const float* __restrict__ X = pb.rinv;
  float acc[8][8];
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[p][q] = 0.f;
  for (int m0 = 0; m0 < r; m0 += kXRows) {
    const int mrows = (r - m0) < kXRows ? (r - m0) : kXRows;
    __syncthreads();  // St staged (first chunk) / the previous X chunk used
    for (int mm = warp; mm < mrows; mm += 8)
      for (int c = lane; c < r8; c += 32) Xs[mm * r8 + c] = c < r ? X[(size_t)(m0 + mm) * r + c] : 0.f;
    __syncthreads();
    if (!active) continue;
    // X is upper triangular: rows m > c0 + 7 add nothing to these columns
    int mend = c0 + 8 - m0;
    if (mend > mrows) mend = mrows;
#pragma unroll 2
    for (int mm = 0; mm < mend; ++mm) {
      const float4 sa = *reinterpret_cast<const float4*>(St + (size_t)(m0 + mm) * ldt + q0);
      const float4 sb = *reinterpret_cast<const float4*>(St + (size_t)(m0 + mm) * ldt + q0 + 4);
      const float4 xa = *reinterpret_cast<const float4*>(Xs + mm * r8 + c0);
      const float4 xb = *reinterpret_cast<const float4*>(Xs + mm * r8 + c0 + 4);
      const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(sv[p], xv[q], acc[p][q]);
    }
  }
  if (!active) return;
  const float scale = final_pass ? pb.scale : 1.0f;
  const bool vec = (r & 3) == 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (q0 + p >= rows) break;
    float* out = P + (size_t)(q0 + p) * r + c0;
    if (vec && c0 + 8 <= r) {
      *reinterpret_cast<float4*>(out) =
          make_float4(acc[p][0] * scale, acc[p][1] * scale, acc[p][2] * scale, acc[p][3] * scale);
      *reinterpret_cast<float4*>(out + 4) =
          make_float4(acc[p][4] * scale, acc[p][5] * scale, acc[p][6] * scale, acc[p][7] * scale);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + q < r) out[q] = acc[p][q] * scale;
    }
  }
}

// The same product for r <= 64 (at most eight column octets), arranged so that
// every lane of a warp has the same triangular extent: warp w takes column
// octet co = w % co_n of the 256-row group w / co_n, lane l the row octet l of
// that group (8 x 8 outputs each).  A block covers RB = 256 * (8 / co_n) rows,
// staged (transposed) with all of X before any output is written.  Warps of
// low octets finish early and leave the SM to other blocks; no lane idles
// inside a warp.
__host__ __device__ inline int tri_rows_small(int r) { return 256 * (8 / ((r + 7) / 8)); }
__host__ __device__ inline size_t tri_small_smem_floats(int r) {
  const int r8 = (r + 7) / 8 * 8;
  return (((size_t)r * (tri_rows_small(r) + 4) + 3) & ~size_t(3)) + (size_t)r * r8;
}
__global__ void __launch_bounds__(256, 2) tri_apply_small_kernel(const ProjBatch batch, int final_pass) {
  extern __shared__ __align__(16) float smem[];
  const ProjProblem& pb = batch.p[blockIdx.y];
  const int r = batch.r, r8 = (r + 7) / 8 * 8, co_n = r8 / 8, ng = 8 / co_n, RB = 256 * ng, ldt = RB + 4;
  float* St = smem;                                          // r x (RB + 4): St[m][row]
  float* Xs = smem + (((size_t)r * ldt + 3) & ~size_t(3));  // r x r8
  const int64_t row0 = (int64_t)blockIdx.x * RB;
  if (row0 >= pb.k) return;
  const int rows = (int)((pb.k - row0) < RB ? (pb.k - row0) : RB);
  float* P = pb.P + row0 * r;
  if ((r & 3) == 0) {
    const int nv = r >> 2;
    for (int row = threadIdx.x; row < rows; row += 256) {
      const float4* src = reinterpret_cast<const float4*>(P + (size_t)row * r);
      float4 v[16];
#pragma unroll
      for (int m = 0; m < 16; ++m) v[m] = (m < nv) ? src[m] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        if (m >= nv) break;
        float* dst = St + (size_t)(4 * m) * ldt + row;
        dst[0] = v[m].x;
        dst[ldt] = v[m].y;
        dst[2 * ldt] = v[m].z;
        dst[3 * ldt] = v[m].w;
      }
    }
  } else {
    for (int row = threadIdx.x; row < rows; row += 256) {
      const float* src = P + (size_t)row * r;
      for (int c0 = 0; c0 < r; c0 += 16) {
        float v[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = (c0 + m < r) ? src[c0 + m] : 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (c0 + m < r) St[(size_t)(c0 + m) * ldt + row] = v[m];
      }
    }
  }
  const float* __restrict__ X = pb.rinv;
  for (int e = threadIdx.x; e < r * r8; e += 256) {
    const int m = e / r8, c = e % r8;
    Xs[e] = c < r ? X[(size_t)m * r + c] : 0.f;
  }
  __syncthreads();  // no block-wide barrier after this point
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int co = warp % co_n, grp = warp / co_n;
  if (grp >= ng) return;
  const int c0 = 8 * co, q0 = grp * 256 + 8 * lane;
  if (q0 >= rows) return;
  float acc[8][8];
#pragma unroll
  for (int p = 0; p < 8; ++p)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[p][q] = 0.f;
  // X is upper triangular: rows m > c0 + 7 add nothing to these columns
  const int mend = (c0 + 8) < r ? (c0 + 8) : r;
#pragma unroll 2
  for (int m = 0; m < mend; ++m) {
    const float4 sa = *reinterpret_cast<const float4*>(St + (size_t)m * ldt + q0);
    const float4 sb = *reinterpret_cast<const float4*>(St + (size_t)m * ldt + q0 + 4);
    const float4 xa = *reinterpret_cast<const float4*>(Xs + m * r8 + c0);
    const float4 xb = *reinterpret_cast<const float4*>(Xs + m * r8 + c0 + 4);
    const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
    for (int p = 0; p < 8; ++p)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(sv[p], xv[q], acc[p][q]);
  }
  const float scale = final_pass ? pb.scale : 1.0f;
  const bool vec = (r & 3) == 0;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    if (q0 + p >= rows) break;
    float* out = P + (size_t)(q0 + p) * r + c0;
    if (vec && c0 + 8 <= r) {
      *reinterpret_cast<float4*>(out) =
          make_float4(acc[p][0] * scale, acc[p][1] * scale, acc[p][2] * scale, acc[p][3] * scale);
      *reinterpret_cast<float4*>(out + 4) =
          make_float4(acc[p][4] * scale, acc[p][5] * scale, acc[p][6] * scale, acc[p][7] * scale);
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + q < r) out[q] = acc[p][q] * scale;
    }
  }
}

// The same product for 32 <= r <= 64 with r a multiple of 4, pipelined: a block
// takes up to kTriBlocks consecutive 256-row groups of one problem (the grid
// lists exactly the groups that exist) and copies the next group into shared
// memory (asynchronous 16-byte copies, row-major with the 16-byte chunks of
// row R XOR-swizzled by (R / 8) % 8) while it computes the current one.  Its 16
// warps each take one column quad co4 (8 x 4 outputs per lane, lane l the row
// octet l); the quads are dealt so that every scheduler's four warps carry the
// same triangular work (1 + 8 + 9 + 16 = 2 + 7 + 10 + 15 = ... rows of X).  Per
// four rows m of X a thread reads its 8 x 4 staged values and 4 x 4 X values
// (twelve 16-byte shared loads, conflict-free) for 128 FMAs.
constexpr int kTriBlocks = 4;
constexpr int kTriThreads = 512;
__host__ __device__ inline int tri_pipe_chunks(int r) { return r > 32 ? 16 : 8; }  // 16-byte chunks per staged row
__host__ __device__ inline bool tri_pipe_ok(int r) { return r >= 32 && r <= 64 && (r & 3) == 0; }
__host__ __device__ inline size_t tri_pipe_smem_bytes(int r) {
  return 2 * (size_t)256 * tri_pipe_chunks(r) * 16 + (size_t)r * ((r + 7) / 8 * 8) * 4;
}
struct TriGrid {
  int blk_begin[kMaxBatch + 1];  // blocks of problem i: [blk_begin[i], blk_begin[i + 1])
};
__global__ void __launch_bounds__(kTriThreads, 1) tri_apply_pipe_kernel(const __grid_constant__ ProjBatch batch,
                                                                        const __grid_constant__ TriGrid grid,
                                                                        int final_pass) {
  extern __shared__ __align__(16) float smem[];
  int y = 0;  // this block's problem
  {
    int lo = 0, hi = batch.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (grid.blk_begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    y = lo;
  }
  const ProjProblem& pb = batch.p[y];
  const int r = batch.r, r8 = (r + 7) / 8 * 8, ldc = tri_pipe_chunks(r), nc = r >> 2;
  float* Sbuf = smem;                    // 2 x 256 rows x ldc chunks
  float* Xs = smem + 2 * 256 * ldc * 4;  // r x r8
  const int64_t first = (int64_t)((int)blockIdx.x - grid.blk_begin[y]) * kTriBlocks * 256;
  const int64_t left = (pb.k - first + 255) / 256;
  const int nblk = left < kTriBlocks ? (int)left : kTriBlocks;
  float* P = pb.P;
  auto stage = [&](int blk, int buf) {  // rows [row0, row0 + 256) into buffer buf, zero past k
    const int64_t row0 = first + (int64_t)blk * 256;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(Sbuf + (size_t)buf * 256 * ldc * 4);
    for (int e = threadIdx.x; e < 256 * nc; e += kTriThreads) {
      const int R = e / nc, c = e % nc;
      const bool in = row0 + R < pb.k;
      const float* src = in ? P + (row0 + R) * r + 4 * c : P;
      const uint32_t dst = base + (uint32_t)(R * ldc + (c ^ ((R >> 3) & 7))) * 16u;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16 : 0)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  stage(0, 0);
  const float* __restrict__ X = pb.rinv;
  for (int e = threadIdx.x; e < r * r8; e += kTriThreads) {
    const int m = e / r8, c = e % r8;
    Xs[e] = c < r ? X[(size_t)m * r + c] : 0.f;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // scheduler warp % 4 holds the quads {s, 7 - s, 8 + s, 15 - s}
  const int sch = warp & 3, slot = warp >> 2;
  const int co4 = slot == 0 ? sch : slot == 1 ? 7 - sch : slot == 2 ? 8 + sch : 15 - sch;
  const int c0 = 4 * co4, q0 = 8 * lane;
  const bool busy = c0 < r;
  const int mend = (c0 + 4) < r ? (c0 + 4) : r;  // X is upper triangular; a multiple of 4
  const float scale = final_pass ? pb.scale : 1.0f;
  for (int blk = 0; blk < nblk; ++blk) {
    if (blk + 1 < nblk) {
      stage(blk + 1, (blk + 1) & 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // this group's rows (and X) are in shared memory
    const int64_t row0 = first + (int64_t)blk * 256;
    if (busy && row0 + q0 < pb.k) {
      const float4* S4 = reinterpret_cast<const float4*>(Sbuf + (size_t)(blk & 1) * 256 * ldc * 4);
      float acc[8][4];
#pragma unroll
      for (int p = 0; p < 8; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
      for (int m0 = 0; m0 < mend; m0 += 4) {
        const int ch = (m0 >> 2) ^ (lane & 7);
        float4 sv[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) sv[p] = S4[(q0 + p) * ldc + ch];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          const float4 xa = *reinterpret_cast<const float4*>(Xs + (m0 + mm) * r8 + c0);
          const float xv[4] = {xa.x, xa.y, xa.z, xa.w};
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float sp = mm == 0 ? sv[p].x : mm == 1 ? sv[p].y : mm == 2 ? sv[p].z : sv[p].w;
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(sp, xv[q], acc[p][q]);
          }
        }
      }
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (row0 + q0 + p >= pb.k) break;
        float* out = P + (row0 + q0 + p) * r + c0;
        *reinterpret_cast<float4*>(out) =
            make_float4(acc[p][0] * scale, acc[p][1] * scale, acc[p][2] * scale, acc[p][3] * scale);
      }
    }
    __syncthreads();  // the buffer is refilled two groups on
  }
}

// P rows <- (P rows) X on the tensor cores, for r <= 128: a block takes up to
// kTtcRows consecutive rows of one problem (the grid lists the row groups that
// exist), 128 at a time.  X (scaled by a power of two 2^g from its largest
// magnitude) is split once per block into FP16 high and low parts and written
// transposed into swizzled K-major tiles (row n of the tile is column n of X);
// each 128-row tile of P likewise, each row m scaled by its own 2^e_m (row m of
// P is row m of the tile, K = r in 64-wide chunks; a row's scale factors out
// of its products).  tcgen05.mma (kind::f16,
// M = 128, N = r rounded to 16) accumulates hi hi + hi lo + lo hi into TMEM,
// and warps 0..3 (one per TMEM lane quarter) write each row's products times
// 2^-(e_m+g) (and the final pass's scale) over the row, which only this block
// reads.  Zero padding past r in both operands keeps the padded sums exact.
constexpr int kTtcRows = 1024;
constexpr int kTtcThreads = 256;
__host__ __device__ inline int ttc_npad(int r) { return (r + 15) / 16 * 16; }
__host__ __device__ inline int ttc_kc(int r) { return (ttc_npad(r) + 63) / 64; }
__host__ __device__ inline bool ttc_ok(int r) { return r <= 128; }
__host__ __device__ inline size_t ttc_smem_bytes(int r) {
  return (size_t)ttc_kc(r) * 2 * 16384 + (size_t)ttc_kc(r) * 2 * ttc_npad(r) * 128 + 1024;
}
__host__ __device__ inline uint32_t ttc_tmem_cols(int r) {
  uint32_t c = 32;
  while ((int)c < ttc_npad(r)) c <<= 1;
  return c;
}
__device__ __forceinline__ uint32_t ttc_split2(float y0, float y1, uint32_t& lo) {
  const __half h0 = __float2half_rn(y0), h1 = __float2half_rn(y1);
  const __half l0 = __float2half_rn(y0 - __half2float(h0)), l1 = __float2half_rn(y1 - __half2float(h1));
  lo = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
  return (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
}
// 2^e that brings a largest magnitude m into [2^14, 2^15) (0 for m = 0 or not finite)
__device__ __forceinline__ int ttc_exponent(float m) {
  if (!(m > 0.f) || !(m <= 3.4028234e38f)) return 0;
  int E;
  frexpf(m, &E);
  const int e = 15 - E;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}
// largest magnitude over the block (NaN if any is NaN)
__device__ __forceinline__ float ttc_block_max(float m, float* wmax) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    m = (m != m || om != om) ? __int_as_float(0x7FC00000) : fmaxf(m, om);
  }
  __syncthreads();  // wmax is free
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  float bm = 0.f;
  for (int w = 0; w < kTtcThreads / 32; ++w)
    bm = (bm != bm || wmax[w] != wmax[w]) ? __int_as_float(0x7FC00000) : fmaxf(bm, wmax[w]);
  return bm;
}
__global__ void __launch_bounds__(kTtcThreads) tri_apply_tc_kernel(const __grid_constant__ ProjBatch batch,
                                                                   const __grid_constant__ TriGrid grid,
                                                                   int final_pass) {
  extern __shared__ uint8_t ttc_raw[];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ float wmax[kTtcThreads / 32];
  __shared__ int row_e[128];  // each row's scale exponent
  __shared__ volatile int abort_flag;
  int y = 0;  // this block's problem
  {
    int lo = 0, hi = batch.n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (grid.blk_begin[mid] <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    y = lo;
  }
  const ProjProblem& pb = batch.p[y];
  const int r = batch.r, npad = ttc_npad(r), kc = ttc_kc(r);
  const uint32_t cols = ttc_tmem_cols(r);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t first = (int64_t)((int)blockIdx.x - grid.blk_begin[y]) * kTtcRows;
  const int64_t last = first + kTtcRows < pb.k ? first + kTtcRows : pb.k;
  float* __restrict__ P = pb.P;
  const float* __restrict__ X = pb.rinv;
  const uint32_t base = tc::smem_u32(reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(ttc_raw) + 1023) & ~uintptr_t(1023)));
  // A chunk c: hi at a_s + 2c 16384, lo 16384 further; B chunk c likewise with npad 128-byte rows
  const uint32_t a_s = base, b_s = base + (uint32_t)kc * 2 * 16384, b_part = (uint32_t)npad * 128;
  if (tid == 0) {
    abort_flag = 0;
    tc::mbar_init(&mma_bar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&tmem_slot, cols);
  for (uint32_t e = tid; e < (uint32_t)((kc * 2 * 16384 + kc * 2 * npad * 128) / 16); e += kTtcThreads)
    tc::sts128(base + 16u * e, make_uint4(0, 0, 0, 0));
  float m = 0.f;
  for (int e = tid; e < r * r; e += kTtcThreads) {
    const float x = X[e];
    m = (m != m || x != x) ? __int_as_float(0x7FC00000) : fmaxf(m, fabsf(x));
  }
  tc::tc_fence_before();
  const int g = ttc_exponent(ttc_block_max(m, wmax));  // (its barriers also publish the zeroed tiles)
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // B = X^T split: item (column n of X, chunk c, 8-row group k8) is one
  // 16-byte chunk of tile row n; consecutive threads take consecutive n
  {
    const float sx = ldexpf(1.f, g);
    for (int it = tid; it < r * kc * 8; it += kTtcThreads) {
      const int n = it % r, rest = it / r, k8 = rest & 7, c = rest >> 3;
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int k0 = c * 64 + k8 * 8 + 2 * t;
        const float x0 = k0 < r ? X[k0 * r + n] : 0.f, x1 = k0 + 1 < r ? X[(k0 + 1) * r + n] : 0.f;
        hv[t] = ttc_split2(x0 * sx, x1 * sx, lv[t]);
      }
      const uint32_t off = (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((k8 ^ (n & 7)) << 4));
      const uint32_t bc = b_s + (uint32_t)c * 2 * b_part;
      tc::sts128(bc + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
      tc::sts128(bc + b_part + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
    }
  }
  const uint32_t idesc = tc::idesc_f16(128, npad, false, false);
  const float out_scale = final_pass ? pb.scale : 1.0f;
  const bool vec = (r & 3) == 0;
  const int per_row = 8 * kc;  // conversion items of one row: consecutive threads (8 or 16)
  uint32_t phase = 0;
  bool live = true;
  for (int64_t row0 = first; row0 < last && live; row0 += 128) {
    const int rows = (int)(last - row0 < 128 ? last - row0 : 128);
    // A = this tile of P, each row scaled by its own power of two 2^e_m: item
    // (row m, chunk c, 8-column group k8), the items of a row on consecutive
    // threads, which find the row's largest magnitude together
    for (int it = tid; it < 128 * per_row; it += kTtcThreads) {
      const int k8 = it & 7, c = (it >> 3) % kc, mr = it / per_row;
      const int k0 = c * 64 + k8 * 8;
      const float* src = P + (row0 + mr) * r + k0;
      float x[8];
      if (vec && mr < rows && k0 + 8 <= r) {  // two 16-byte loads (rows start on 16 bytes when 4 | r)
        const float4 u0 = reinterpret_cast<const float4*>(src)[0], u1 = reinterpret_cast<const float4*>(src)[1];
        x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
        x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = (mr < rows && k0 + t < r) ? src[t] : 0.f;
      }
      float mx = 0.f;
#pragma unroll
      for (int t = 0; t < 8; ++t) mx = (mx != mx || x[t] != x[t]) ? __int_as_float(0x7FC00000) : fmaxf(mx, fabsf(x[t]));
      for (int o = 1; o < per_row; o <<= 1) {
        const float om = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
        mx = (mx != mx || om != om) ? __int_as_float(0x7FC00000) : fmaxf(mx, om);
      }
      const int em = ttc_exponent(mx);
      if ((it & (per_row - 1)) == 0) row_e[mr] = em;
      const float sp = ldexpf(1.f, em);
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) hv[t] = ttc_split2(x[2 * t] * sp, x[2 * t + 1] * sp, lv[t]);
      const uint32_t off = (uint32_t)((mr >> 3) * 1024 + (mr & 7) * 128 + ((k8 ^ (mr & 7)) << 4));
      const uint32_t ac = a_s + (uint32_t)c * 2 * 16384;
      tc::sts128(ac + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
      tc::sts128(ac + 16384 + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
    }
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc::tc_fence_after();
      for (int c = 0; c < kc; ++c) {
        const uint32_t ac = a_s + (uint32_t)c * 2 * 16384, bc = b_s + (uint32_t)c * 2 * b_part;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ah = tc::sdesc_sw128(ac + kk * 32, 16, 1024), al = tc::sdesc_sw128(ac + 16384 + kk * 32, 16, 1024);
          const uint64_t bh = tc::sdesc_sw128(bc + kk * 32, 16, 1024), bl = tc::sdesc_sw128(bc + b_part + kk * 32, 16, 1024);
          tc::mma_bf16(tmem, ah, bh, idesc, (c > 0 || kk > 0) ? 1u : 0u);
          tc::mma_bf16(tmem, ah, bl, idesc, 1u);
          tc::mma_bf16(tmem, al, bh, idesc, 1u);
        }
      }
      tc::mma_commit(&mma_bar);
    }
    live = tc::mbar_wait(&mma_bar, phase, &abort_flag, nullptr, 0);
    phase ^= 1u;
    live = __syncthreads_and(live);
    tc::tc_fence_after();
    if (!live) break;
    // warps 0..3: row m = TMEM lane 32 w + lane, scaled back and written over P
    if (warp < 4) {
      const int mr = warp * 32 + lane;
      const float us = ldexpf(1.f, -(row_e[mr] + g)) * out_scale;
      for (int cg = 0; cg * 32 < npad; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cg * 32), v);
        tc::tmem_wait_ld();
        if (mr < rows) {
          float* dst = P + (row0 + mr) * r + cg * 32;
          if (vec && cg * 32 + 32 <= r) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              reinterpret_cast<float4*>(dst)[t] =
                  make_float4(__uint_as_float(v[4 * t]) * us, __uint_as_float(v[4 * t + 1]) * us,
                              __uint_as_float(v[4 * t + 2]) * us, __uint_as_float(v[4 * t + 3]) * us);
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (cg * 32 + t < r) dst[t] = __uint_as_float(v[t]) * us;
          }
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();  // the TMEM reads and row_e are done before the next tile
    tc::tc_fence_after();
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, cols);
}

}  // namespace

void carve_qr_workspace(WsCursor& cur, int64_t k, int r, ProjProblem* p) {
  const GramChunks g = gram_chunks(k);
  float2* partials = cur.take<float2>((size_t)g.nchunks * r * r);
  double* gram = cur.take<double>((size_t)r * r);
  float* rinv = cur.take<float>((size_t)r * r);
  if (p) {
    p->partials = partials;
    p->gram = gram;
    p->rinv = rinv;
  }
}

cudaError_t launch_rademacher(const ProjBatch& batch, int64_t max_k, cudaStream_t stream) {
  const int64_t words = ceil_div(max_k * batch.r, 32);
  count_launch();
  rademacher_kernel<<<dim3((unsigned)ceil_div(words, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

cudaError_t launch_gaussian_qr(const ProjBatch& batch, int64_t max_k, cudaStream_t stream) {
  const int r = batch.r;
  const int64_t blocks4 = ceil_div(max_k * r, 4);
  count_launch();
  gaussian_kernel<<<dim3((unsigned)ceil_div(blocks4, 256), batch.n), 256, 0, stream>>>(batch);
  GramBatch gb;
  gb.n = batch.n;
  gb.r = r;
  for (int i = 0; i < batch.n; ++i) {
    gb.e[i].A = batch.p[i].P;
    gb.e[i].rows = batch.p[i].k;
    gb.e[i].partials = batch.p[i].partials;
    gb.e[i].out = batch.p[i].gram;
  }
  const size_t chol_smem = sizeof(float) * chol_smem_floats(r);
  const int apply_rows = tri_rows(r);
  const size_t apply_smem = sizeof(float) * tri_smem_floats(r);
  cudaError_t err = cudaFuncSetAttribute(chol_inv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)chol_smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(tri_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)apply_smem);
  if (err != cudaSuccess) return err;
  // the triangular products: on the tensor cores up to rank 128, else SIMT
  const bool tcore = ttc_ok(r);
  const size_t tc_smem = tcore ? ttc_smem_bytes(r) : 0;
  if (tcore) {
    err = cudaFuncSetAttribute(tri_apply_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem);
    if (err != cudaSuccess) return err;
  }
  const bool pipe = !tcore && tri_pipe_ok(r);
  const size_t pipe_smem = pipe ? tri_pipe_smem_bytes(r) : 0;
  if (pipe) {
    err = cudaFuncSetAttribute(tri_apply_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)pipe_smem);
    if (err != cudaSuccess) return err;
  }
  static thread_local TriGrid tg;
  if (tcore || pipe) {
    const int64_t rows = tcore ? kTtcRows : (int64_t)256 * kTriBlocks;
    tg.blk_begin[0] = 0;
    for (int i = 0; i < batch.n; ++i) tg.blk_begin[i + 1] = tg.blk_begin[i] + (int)ceil_div(batch.p[i].k, rows);
  }
  const bool small = !tcore && !pipe && r <= 64;
  const int small_rows = small ? tri_rows_small(r) : 0;
  const size_t small_smem = small ? sizeof(float) * tri_small_smem_floats(r) : 0;
  if (small) {
    err = cudaFuncSetAttribute(tri_apply_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)small_smem);
    if (err != cudaSuccess) return err;
  }
  for (int pass = 0; pass < 2; ++pass) {
    err = launch_gram(gb, stream, true);
    if (err != cudaSuccess) return err;
    count_launch();
    chol_inv_kernel<<<batch.n, 256, chol_smem, stream>>>(batch);
    count_launch();
    if (tcore)
      tri_apply_tc_kernel<<<(unsigned)tg.blk_begin[batch.n], kTtcThreads, tc_smem, stream>>>(batch, tg, pass == 1);
    else if (pipe)
      tri_apply_pipe_kernel<<<(unsigned)tg.blk_begin[batch.n], kTriThreads, pipe_smem, stream>>>(batch, tg,
                                                                                                  pass == 1);
    else if (small)
      tri_apply_small_kernel<<<dim3((unsigned)ceil_div(max_k, small_rows), batch.n), 256, small_smem, stream>>>(
          batch, pass == 1);
    else
      tri_apply_kernel<<<dim3((unsigned)ceil_div(max_k, apply_rows), batch.n), 256, apply_smem, stream>>>(
          batch, pass == 1);
  }
  return cudaGetLastError();
}

}  // namespace rgs
