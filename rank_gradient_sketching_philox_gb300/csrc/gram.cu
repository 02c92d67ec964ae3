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
  const int nchunks = gram_chunks(en.rows).nchunks;
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

cudaError_t launch_gram(const GramBatch& batch, cudaStream_t stream) {
  if (batch.n <= 0) return cudaSuccess;
  const int tiles = (int)ceil_div(batch.r, kTile);
  const size_t smem = gram_smem_bytes(tiles > 1);
  cudaError_t err = cudaFuncSetAttribute(gram_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  count_launch();
  gram_partial_kernel<<<dim3(64, tiles * (tiles + 1) / 2, batch.n), 256, smem, stream>>>(batch);
  const int rr = batch.r * batch.r;
  count_launch();
  gram_reduce_kernel<<<dim3((unsigned)ceil_div(rr, 256), batch.n), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace rgs
