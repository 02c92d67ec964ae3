// (a) Projection P (k x r fp32): Rademacher signs or a Gaussian-QR frame.
//
// Rademacher: entries +-1/sqrt(r) ("LoGRA: Low-Rank Gradient Sketches", "Why
// the Sketch Can Be Accumulated Without a Full Gradient").  Element e = j*r + l
// takes bit e % 128 of Philox block e / 128 of the sign stream.
//
// Gaussian QR: P = sqrt(k/r) Q with Q the orthonormal factor of a Gaussian
// k x r matrix and diag(R) > 0 ("Randomized Gradient Compression",
// footnote 1).  For 4r <= k the frame is computed by CholeskyQR2 in fp32:
// twice (Gram A = G^T G, Cholesky A = R^T R, G <- G R^-1).  Cholesky factors
// have a positive diagonal, so the result is the sign-corrected QR factor
// without an explicit sign fix.  There the Gaussian matrix is well conditioned
// and the second pass leaves P^T P = (k/r) I to about 1e-6.
// For r <= k < 4r (at most 1023 x 256, up to square) the Gaussian matrix can be
// as ill conditioned as a square one, whose condition number grows like k, so
// the frame is drawn and factored in fp64 by Householder QR, one block per
// problem (wide_qr_kernel), and the signs of R's diagonal applied explicitly.
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
  const Philox4 blk = philox4x32_10_rk((uint32_t)(w >> 2), batch.step, pb.layer, kTagRademacher, batch.rk0, batch.rk1);
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

// |draw| <= sqrt(-2 ln 2^-33) ~ 6.77 (u >= 2^-33, |cos|, |sin| <= 1), so 8
// bounds every value gaussian4 returns.
constexpr float kGaussianBound = 8.0f;

__global__ void __launch_bounds__(256) gaussian_kernel(const ProjBatch batch) {
  const ProjProblem& pb = batch.p[blockIdx.y];
  const int64_t n = pb.k * batch.r;
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (4 * b >= n) return;
  const Philox4 blk = philox4x32_10_rk((uint32_t)b, batch.step, pb.layer, kTagGaussian, batch.rk0, batch.rk1);
  reinterpret_cast<float4*>(pb.P)[b] = gaussian4(blk);
}


// One block per problem: R with Gram = R^T R (Cholesky, upper triangular) and
// its inverse X = R^-1, written in full (zeros below the diagonal) to pb.rinv.
// Blocked in 32 x 32 tiles so that the block synchronises a few times per tile
// row rather than a few times per matrix row: the upper tiles live in shared
// memory (row stride 33, so that columns of a tile fall in distinct banks), the
// matrix padded to a multiple of 32 with the identity.
//   Cholesky, right-looking, per tile column k: the block factors the diagonal
//   tile pivot by pivot (one warp scales the pivot row, every thread updates
//   one trailing element); each thread solves one column of the tile row
//   (R_kj = R_kk^-T A_kj, the column in registers);
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
// reset_amax: clear the problem's max |P| word, which the triangular product
// that follows records for the next Gram.
__global__ void __launch_bounds__(256) chol_inv_kernel(const ProjBatch batch, int reset_amax) {
  extern __shared__ float S[];
  __shared__ int broken;
  const ProjProblem& pb = batch.p[blockIdx.x];
  const int r = batch.r, nb = chol_tiles(r);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (reset_amax && tid == 0) *pb.amax = 0u;
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
    // the diagonal tile, in place, pivot by pivot with the whole block: the
    // pivot row scaled by 1/sqrt(pivot) (warp 0), then the trailing triangle
    // A_ic -= R_pi R_pc (p < i <= c) one element per thread
    for (int p = 0; p < kCT; ++p) {
      if (warp == 0) {
        const float d = D[p * kCTs + p];
        if (!(d > 0.0f) || !isfinite(d)) {  // the same in every lane
          if (lane == 0) broken = 1;
        } else {
          const float rp = sqrtf(d), inv = 1.0f / rp;
          if (lane > p) D[p * kCTs + lane] = D[p * kCTs + lane] * inv;
          if (lane == p) D[p * kCTs + p] = rp;
        }
      }
      __syncthreads();
      if (broken) break;
      const int n = kCT - 1 - p;
      for (int e = tid; e < n * n; e += 256) {
        const int i = p + 1 + e / n, c = p + 1 + e % n;
        if (i <= c) D[i * kCTs + c] = fmaf(-D[p * kCTs + i], D[p * kCTs + c], D[i * kCTs + c]);
      }
      __syncthreads();
    }
    __syncthreads();
    if (broken) break;
    // tile row k: R_kj = R_kk^-T A_kj, one column per thread (forward
    // substitution; the column in registers, R_kk read by every lane at once)
    for (int cidx = tid; cidx < (nb - 1 - k) * kCT; cidx += 256) {
      float* B = chol_tile(S, nb, k, k + 1 + (cidx >> 5));
      const int c = cidx & 31;
      float bc[kCT];
#pragma unroll
      for (int p = 0; p < kCT; ++p) bc[p] = B[p * kCTs + c];
#pragma unroll
      for (int p = 0; p < kCT; ++p) {
        float v = bc[p];
#pragma unroll
        for (int m = 0; m < p; ++m) v = fmaf(-D[m * kCTs + p], bc[m], v);
        bc[p] = v / D[p * kCTs + p];
        B[p * kCTs + c] = bc[p];
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

// Rows of a problem per block of the triangular product, listed per problem.
struct TriGrid {
  int blk_begin[kMaxBatch + 1];  // blocks of problem i: [blk_begin[i], blk_begin[i + 1])
};

// P rows <- (P rows) X on the tensor cores: a block takes up to
// kTtcRows consecutive rows of one problem (the grid lists the row groups that
// exist), 128 at a time.  X (scaled by a power of two 2^g from its largest
// magnitude) is split into FP16 high and low parts and written transposed into
// swizzled K-major tiles (row n of the tile is column n of X): all of it once
// per block up to rank 128, above one 64-row chunk of X at a time per tile;
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
// chunks of X^T held at once: all of them up to rank 128, else one at a time
__host__ __device__ inline int ttc_bchunks(int r) { return ttc_kc(r) <= 2 ? ttc_kc(r) : 1; }
__host__ __device__ inline size_t ttc_smem_bytes(int r) {
  return (size_t)ttc_kc(r) * 2 * 16384 + (size_t)ttc_bchunks(r) * 2 * ttc_npad(r) * 128 + 1024;
}
__host__ __device__ inline uint32_t ttc_tmem_cols(int r) {
  uint32_t c = 32;
  while ((int)c < ttc_npad(r)) c <<= 1;
  return c;
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
  const int r = batch.r, npad = ttc_npad(r), kc = ttc_kc(r), nbc = ttc_bchunks(r);
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
  for (uint32_t e = tid; e < (uint32_t)((kc * 2 * 16384 + nbc * 2 * npad * 128) / 16); e += kTtcThreads)
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
  // B = X^T split, chunk c into the buffer at bc: item (column n of X,
  // 8-row group k8) is one 16-byte chunk of tile row n; consecutive threads
  // take consecutive n, so that each row of X is read coalesced
  const float sx = ldexpf(1.f, g);
  auto convert_b = [&](int c, uint32_t bc) {
    for (int it = tid; it < r * 8; it += kTtcThreads) {
      const int n = it % r, k8 = it / r;
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int k0 = c * 64 + k8 * 8 + 2 * t;
        const float x0 = k0 < r ? X[k0 * r + n] : 0.f, x1 = k0 + 1 < r ? X[(k0 + 1) * r + n] : 0.f;
        hv[t] = tc::split_f16x2(x0, x1, sx, lv[t]);
      }
      const uint32_t off = (uint32_t)((n >> 3) * 1024 + (n & 7) * 128 + ((k8 ^ (n & 7)) << 4));
      tc::sts128(bc + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
      tc::sts128(bc + b_part + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
    }
  };
  if (nbc == kc)  // all of X^T, once per block
    for (int c = 0; c < kc; ++c) convert_b(c, b_s + (uint32_t)c * 2 * b_part);
  const uint32_t idesc = tc::idesc_f16(128, npad, false, false);
  const float out_scale = final_pass ? pb.scale : 1.0f;
  const bool vec = (r & 3) == 0;
  // conversion items of one row: 8 per 64-wide chunk, padded to a power of two
  // (8, 16 or 32 consecutive threads, which reduce the row's maximum by shuffles)
  const int kcp = kc == 3 ? 4 : kc;
  const int per_row = 8 * kcp;
  uint32_t phase = 0;
  bool live = true;
  for (int64_t row0 = first; row0 < last && live; row0 += 128) {
    const int rows = (int)(last - row0 < 128 ? last - row0 : 128);
    // A = this tile of P, each row scaled by its own power of two 2^e_m: item
    // (row m, chunk c, 8-column group k8), the items of a row on consecutive
    // threads, which find the row's largest magnitude together
    // 128 per_row items are a multiple of 4 kTtcThreads: each thread loads four
    // items before it converts any, so that their loads are in flight together
    for (int it0 = tid; it0 < 128 * per_row; it0 += 4 * kTtcThreads) {
      float xb[4][8];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int it = it0 + b * kTtcThreads;
        const int k8 = it & 7, c = (it >> 3) & (kcp - 1), mr = it / per_row;
        const int k0 = c * 64 + k8 * 8;  // c >= kc: padding items (zeros, not stored)
        const float* src = P + (row0 + mr) * r + k0;
        float* x = xb[b];
        if (vec && mr < rows && c < kc && k0 + 8 <= r) {  // two 16-byte loads (rows start on 16 bytes when 4 | r)
          const float4 u0 = reinterpret_cast<const float4*>(src)[0], u1 = reinterpret_cast<const float4*>(src)[1];
          x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
          x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) x[t] = (mr < rows && c < kc && k0 + t < r) ? src[t] : 0.f;
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int it = it0 + b * kTtcThreads;
        const int k8 = it & 7, c = (it >> 3) & (kcp - 1), mr = it / per_row;
        const float* x = xb[b];
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
        for (int t = 0; t < 4; ++t) hv[t] = tc::split_f16x2(x[2 * t], x[2 * t + 1], sp, lv[t]);
        if (c < kc) {
          const uint32_t off = (uint32_t)((mr >> 3) * 1024 + (mr & 7) * 128 + ((k8 ^ (mr & 7)) << 4));
          const uint32_t ac = a_s + (uint32_t)c * 2 * 16384;
          tc::sts128(ac + off, make_uint4(hv[0], hv[1], hv[2], hv[3]));
          tc::sts128(ac + 16384 + off, make_uint4(lv[0], lv[1], lv[2], lv[3]));
        }
      }
    }
    // the K chunks' MMAs: with X^T resident one batch; else per chunk, each
    // chunk of X^T converted once the previous chunk's MMAs have read the buffer
    const int nb = nbc == kc ? 1 : kc;
    for (int bi = 0; bi < nb && live; ++bi) {
      if (nbc != kc) {
        if (bi > 0) {
          live = tc::mbar_wait(&mma_bar, phase, &abort_flag, nullptr, 0);
          phase ^= 1u;
          live = __syncthreads_and(live);
          if (!live) break;
        }
        convert_b(bi, b_s);
      }
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc::tc_fence_after();
        const int c0 = nbc == kc ? 0 : bi, c1 = nbc == kc ? kc : bi + 1;
        for (int c = c0; c < c1; ++c) {
          const uint32_t ac = a_s + (uint32_t)c * 2 * 16384, bc = b_s + (uint32_t)(nbc == kc ? c : 0) * 2 * b_part;
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
    }
    if (live) live = tc::mbar_wait(&mma_bar, phase, &abort_flag, nullptr, 0);
    phase ^= 1u;
    live = __syncthreads_and(live);
    tc::tc_fence_after();
    if (!live) break;
    // warps 0..3: row m = TMEM lane 32 w + lane, scaled back and written over
    // P; the first pass also records max |P| (as bits, so that a NaN, whose
    // bits exceed those of +inf, wins) for the next Gram
    if (warp < 4) {
      const int mr = warp * 32 + lane;
      const float us = ldexpf(1.f, -(row_e[mr] + g)) * out_scale;
      uint32_t mbits = 0u;
      for (int cg = 0; cg * 32 < npad; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cg * 32), v);
        tc::tmem_wait_ld();
        if (mr < rows) {
          float* dst = P + (row0 + mr) * r + cg * 32;
          if (vec && cg * 32 + 32 <= r) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float4 o = make_float4(__uint_as_float(v[4 * t]) * us, __uint_as_float(v[4 * t + 1]) * us,
                                           __uint_as_float(v[4 * t + 2]) * us, __uint_as_float(v[4 * t + 3]) * us);
              reinterpret_cast<float4*>(dst)[t] = o;
              if (!final_pass)
                mbits = max(max(max(mbits, __float_as_uint(fabsf(o.x))), __float_as_uint(fabsf(o.y))),
                            max(__float_as_uint(fabsf(o.z)), __float_as_uint(fabsf(o.w))));
            }
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (cg * 32 + t < r) {
                const float o = __uint_as_float(v[t]) * us;
                dst[t] = o;
                mbits = max(mbits, __float_as_uint(fabsf(o)));
              }
          }
        }
      }
      if (!final_pass) {
        mbits = __reduce_max_sync(0xFFFFFFFFu, mbits);
        if (lane == 0) atomicMax(pb.amax, mbits);
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


// ---- fp64 Householder QR for r <= k < 4r ------------------------------------
// One block per problem.  The block draws the Gaussian matrix G (k x r) in fp64
// from the same Philox stream as gaussian_kernel (Box-Muller in double, as the
// exact definition reads), factors it by Householder reflections
// H_j = I - tau_j v_j v_j^T, forms Q = H_0 ... H_{r-1} [I; 0], flips the columns
// whose R_jj is negative and writes P = sqrt(k/r) Q rounded to fp32.
// Workspace: two column-major k x r fp64 arrays (column l of G, then of Q, is
// k contiguous doubles): `a` holds G, then R above the diagonal and v_j from
// the diagonal down; `q` holds Q.  A k x r problem touches about 4 k r^2
// doubles in L1/L2, a few ms at the largest size (1016 x 256).
constexpr int kWqThreads = 512, kWqWarps = kWqThreads / 32, kWqMaxK = 1024;

__device__ __forceinline__ double wq_warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kWqThreads) wide_qr_kernel(const ProjBatch batch) {
  __shared__ double vsh[kWqMaxK];           // the current reflector, rows j .. k-1
  __shared__ double tau[kMaxRank], diag[kMaxRank];
  __shared__ double red[kWqWarps];
  __shared__ double norm2;                  // ||a[j:, j]||^2 of the next column
  const ProjProblem& pb = batch.p[blockIdx.x];
  const int k = (int)pb.k, r = batch.r;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  double* a = pb.wide;
  double* q = pb.wide + (size_t)k * r;

  // G: element e = i*r + l from Philox block e/4, lane e%4 (as gaussian4)
  for (int b = tid; b < k * r / 4; b += kWqThreads) {
    const Philox4 blk = stream_block(batch.seed, pb.layer, batch.step, kTagGaussian, (uint32_t)b);
    const uint32_t w[4] = {blk.w0, blk.w1, blk.w2, blk.w3};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const double ua = ((double)w[2 * t] + 0.5) * 0x1p-32;
      const double ub = ((double)w[2 * t + 1] + 0.5) * 0x1p-32;
      const double radius = sqrt(-2.0 * log(ua));
      double sn, cs;
      sincospi(2.0 * ub, &sn, &cs);
      const int e0 = 4 * b + 2 * t;
      a[(size_t)(e0 % r) * k + e0 / r] = radius * cs;
      a[(size_t)((e0 + 1) % r) * k + (e0 + 1) / r] = radius * sn;
    }
  }
  __syncthreads();
  {  // ||a[:, 0]||^2
    double s = 0.0;
    for (int i = tid; i < k; i += kWqThreads) s += a[i] * a[i];
    s = wq_warp_sum(s);
    if (lane == 0) red[warp] = s;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < kWqWarps; ++w) t += red[w];
      norm2 = t;
    }
    __syncthreads();
  }

  // factorization, one column at a time
  for (int j = 0; j < r; ++j) {
    double* aj = a + (size_t)j * k;
    const double x0 = aj[j], nrm2 = norm2;
    const double alpha = x0 >= 0.0 ? -sqrt(nrm2) : sqrt(nrm2);
    const double v0 = x0 - alpha;
    const double vnorm2 = (nrm2 - x0 * x0) + v0 * v0;
    const bool skip = !(vnorm2 > 0.0);  // a zero column: H_j = I, R_jj = x0
    const double tj = skip ? 0.0 : 2.0 / vnorm2;
    for (int i = j + tid; i < k; i += kWqThreads) vsh[i] = (i == j) ? v0 : aj[i];
    __syncthreads();  // every thread has read x0 and norm2; vsh is complete
    if (tid == 0) {
      tau[j] = tj;
      diag[j] = skip ? x0 : alpha;
      aj[j] = v0;
    }
    if (!skip) {
      for (int c = j + 1 + warp; c < r; c += kWqWarps) {
        double* ac = a + (size_t)c * k;
        double dot = 0.0;
        for (int i = j + lane; i < k; i += 32) dot += vsh[i] * ac[i];
        const double f = tj * wq_warp_sum(dot);
        double s = 0.0;
        for (int i = j + lane; i < k; i += 32) {
          const double x = fma(-f, vsh[i], ac[i]);
          ac[i] = x;
          if (i > j) s += x * x;
        }
        if (c == j + 1) {
          s = wq_warp_sum(s);
          if (lane == 0) norm2 = s;
        }
      }
    } else if (j + 1 < r && warp == 0) {
      const double* ac = a + (size_t)(j + 1) * k;
      double s = 0.0;
      for (int i = j + 1 + lane; i < k; i += 32) s += ac[i] * ac[i];
      s = wq_warp_sum(s);
      if (lane == 0) norm2 = s;
    }
    __syncthreads();
  }

  // Q = H_0 ... H_{r-1} [I; 0], right to left; H_j touches rows j.. of columns j..
  for (int e = tid; e < k * r; e += kWqThreads) q[e] = (e % k == e / k) ? 1.0 : 0.0;
  __syncthreads();
  for (int j = r - 1; j >= 0; --j) {
    const double tj = tau[j];
    if (tj == 0.0) continue;  // uniform over the block
    const double* aj = a + (size_t)j * k;
    for (int i = j + tid; i < k; i += kWqThreads) vsh[i] = aj[i];
    __syncthreads();
    for (int c = j + warp; c < r; c += kWqWarps) {
      double* qc = q + (size_t)c * k;
      double dot = 0.0;
      for (int i = j + lane; i < k; i += 32) dot += vsh[i] * qc[i];
      const double f = tj * wq_warp_sum(dot);
      for (int i = j + lane; i < k; i += 32) qc[i] = fma(-f, vsh[i], qc[i]);
    }
    __syncthreads();
  }

  // P = sqrt(k/r) sign(R_ll) Q, row-major fp32
  const double scale = sqrt((double)k / (double)r);
  for (int e = tid; e < k * r; e += kWqThreads) {
    const int i = e / r, l = e % r;
    const double sg = diag[l] < 0.0 ? -scale : scale;
    pb.P[e] = (float)(sg * q[(size_t)l * k + i]);
  }
}

}  // namespace

void carve_qr_workspace(WsCursor& cur, int64_t k, int r, ProjProblem* p) {
  if (qr_is_wide(k, r)) {
    double* a = cur.take<double>((size_t)2 * k * r);
    if (p) {
      p->partials = nullptr;
      p->gram = nullptr;
      p->rinv = nullptr;
      p->wide = a;
      p->amax = nullptr;
    }
    return;
  }
  const GramChunks g = gram_chunks_tc(k, r);
  float2* partials = cur.take<float2>((size_t)g.nchunks * r * r);
  double* gram = cur.take<double>((size_t)r * r);
  float* rinv = cur.take<float>((size_t)r * r);
  uint32_t* amax = cur.take<uint32_t>(1);
  if (p) {
    p->partials = partials;
    p->gram = gram;
    p->rinv = rinv;
    p->wide = nullptr;
    p->amax = amax;
  }
}

cudaError_t launch_rademacher(const ProjBatch& batch, int64_t max_k, cudaStream_t stream) {
  const int64_t words = ceil_div(max_k * batch.r, 32);
  count_launch();
  rademacher_kernel<<<dim3((unsigned)ceil_div(words, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

cudaError_t launch_wide_qr(const ProjBatch& batch, cudaStream_t stream) {
  count_launch();
  wide_qr_kernel<<<batch.n, kWqThreads, 0, stream>>>(batch);
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
  cudaError_t err = cudaFuncSetAttribute(chol_inv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)chol_smem);
  if (err != cudaSuccess) return err;
  // the triangular products on the tensor cores, kTtcRows rows of one problem per block
  const size_t tc_smem = ttc_smem_bytes(r);
  err = cudaFuncSetAttribute(tri_apply_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem);
  if (err != cudaSuccess) return err;
  static thread_local TriGrid tg;
  tg.blk_begin[0] = 0;
  for (int i = 0; i < batch.n; ++i) tg.blk_begin[i + 1] = tg.blk_begin[i] + (int)ceil_div(batch.p[i].k, (int64_t)kTtcRows);
  for (int pass = 0; pass < 2; ++pass) {
    // the Gram's scale: the first pass's from a bound on the draws, the
    // second's from the maximum the first triangular product recorded
    for (int i = 0; i < batch.n; ++i) {
      gb.e[i].bound = pass == 0 ? kGaussianBound : 0.f;
      gb.e[i].amax = pass == 0 ? nullptr : batch.p[i].amax;
    }
    err = launch_gram(gb, stream);
    if (err != cudaSuccess) return err;
    count_launch();
    chol_inv_kernel<<<batch.n, 256, chol_smem, stream>>>(batch, pass == 0);
    count_launch();
    tri_apply_tc_kernel<<<(unsigned)tg.blk_begin[batch.n], kTtcThreads, tc_smem, stream>>>(batch, tg, pass == 1);
  }
  return cudaGetLastError();
}

}  // namespace rgs
