// (d) Rebuild H = C P^T fused with the weight update and BF16 stochastic
// rounding.
//
// Normalized SGD: W <- W - tau ||W|| H / ||H|| ("Randomized Gradient
// Compression", "How it works").  The scale s = fl32(tau ||W|| / ||H||) is
// formed on the device from ||W||^2 (one read of W, or the value carried from
// the previous update) and ||H||^2 = <P^T P, C^T C> (two r x r Grams), so H is
// never stored.  LoGRA SGD: W <- W - alpha*eta C P^T ("LoGRA: Low-Rank
// Gradient Sketches", "Why the Update Is Low-Rank but Not an Exact Recovery").
//
// Each weight: v = fmaf(-s, H_ij, W_ij), then stochastic rounding to BF16 with
// 16 bits of Philox block (i*k + j) / 8 of the rounding stream (lane
// (i*k + j) % 8 is the low or high half of word lane / 2).
#include "common.cuh"
#include "internal.h"

namespace rgs {
namespace {

__device__ __forceinline__ double block_sum_double(double v, double* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xFFFFFFFFu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double total = 0.0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += red[w];
  }
  __syncthreads();
  return total;  // valid in thread 0
}

// Partial sums of W^2 over a fixed assignment of 8-element vectors to threads
// (Kahan-compensated fp32 per thread, double across threads).
__global__ void __launch_bounds__(256) wnorm_partial_kernel(const uint16_t* __restrict__ W,
                                                           int64_t d, int64_t k, int64_t ld_w,
                                                           double* __restrict__ partials) {
  __shared__ double red[8];
  const int64_t vec_per_row = k / 8;
  const int64_t nvec = d * vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float sum = 0.f, comp = 0.f;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const int64_t i = v / vec_per_row, j = (v % vec_per_row) * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(W + i * ld_w + j);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = bf16_bits_to_float(w[q] & 0xFFFFu), b = bf16_bits_to_float(w[q] >> 16);
      part = fmaf(a, a, part);
      part = fmaf(b, b, part);
    }
    const float y = part - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  }
  const double total = block_sum_double((double)sum - (double)comp, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = total;
}

// One block: ||W||^2, ||H||^2 = <Gp, Gc>, the status and the scale s.
__global__ void __launch_bounds__(256) normsgd_finalize_kernel(
    const double* __restrict__ wnorm_partials, int nwp, const double* __restrict__ wnorm2_in,
    const float* __restrict__ gram_p, const float* __restrict__ gram_c, int rr, float tau,
    float* __restrict__ scale, int32_t* __restrict__ status, uint32_t* __restrict__ ticket,
    double* __restrict__ wnorm2_out) {
  __shared__ double red[8];
  double hpart = 0.0;
  for (int e = threadIdx.x; e < rr; e += blockDim.x) hpart += (double)gram_p[e] * (double)gram_c[e];
  const double nh2 = block_sum_double(hpart, red);
  double wpart = 0.0;
  if (wnorm2_in == nullptr) {
    for (int e = threadIdx.x; e < nwp; e += blockDim.x) wpart += wnorm_partials[e];
  }
  const double nw2_sum = block_sum_double(wpart, red);
  if (threadIdx.x == 0) {
    const double nw2 = wnorm2_in ? *wnorm2_in : nw2_sum;
    int32_t st = 0;
    if (!isfinite(nw2)) st |= SKETCH_DEV_W_NONFINITE;
    if (!isfinite(nh2)) st |= SKETCH_DEV_H_NONFINITE;
    else if (nh2 <= 0.0) st |= SKETCH_DEV_H_ZERO;
    const double s = st ? 0.0 : (double)tau * sqrt(nw2) / sqrt(nh2);
    *scale = (float)s;
    *status = st;
    *ticket = 0u;
    if (st && wnorm2_out) *wnorm2_out = nw2;  // W stays unchanged
  }
}

// 64 x 64 weights per block; thread (tr, tc) = (tid / 8, tid % 8) owns rows
// 2tr, 2tr+1 and columns 8tc .. 8tc+7 of the tile.  C rows and P rows of the
// tile are staged in shared memory; H is accumulated in fp32 registers.
__global__ void __launch_bounds__(256) update_simt_kernel(
    uint16_t* __restrict__ W, int64_t d, int64_t k, int64_t ld_w, const float* __restrict__ C,
    const float* __restrict__ P, int r, const float* __restrict__ scale_dev, float scale_val,
    const int32_t* __restrict__ status_in, int32_t* __restrict__ status_out, uint64_t seed,
    uint32_t layer, uint32_t step, double* __restrict__ wnew_partials,
    uint32_t* __restrict__ ticket, double* __restrict__ wnorm2_out) {
  extern __shared__ float smem[];
  __shared__ double red[8];
  __shared__ bool is_last;
  if (status_in != nullptr && *status_in != 0) return;  // degenerate norms: W untouched
  if (status_out != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    *status_out = 0;
  const float s = scale_dev ? *scale_dev : scale_val;
  const int rs = r + 1;  // padded row stride in shared memory
  float* cs = smem;           // 64 x rs
  float* ps = smem + 64 * rs; // 64 x rs
  const int64_t i0 = (int64_t)blockIdx.y * 64, j0 = (int64_t)blockIdx.x * 64;
  for (int e = threadIdx.x; e < 64 * r; e += blockDim.x) {
    const int row = e / r, l = e % r;
    cs[row * rs + l] = (i0 + row < d) ? C[(i0 + row) * r + l] : 0.f;
    ps[row * rs + l] = (j0 + row < k) ? P[(j0 + row) * r + l] : 0.f;
  }
  __syncthreads();
  const int tr = threadIdx.x >> 3, tc = threadIdx.x & 7;
  float h[2][8] = {};
  for (int l = 0; l < r; ++l) {
    const float c0v = cs[(2 * tr) * rs + l], c1v = cs[(2 * tr + 1) * rs + l];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const float pv = ps[(8 * tc + b) * rs + l];
      h[0][b] = fmaf(c0v, pv, h[0][b]);
      h[1][b] = fmaf(c1v, pv, h[1][b]);
    }
  }
  float sq = 0.f;
  const int64_t j = j0 + 8 * tc;
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int64_t i = i0 + 2 * tr + a;
    if (i >= d || j >= k) continue;
    uint16_t* wp = W + i * ld_w + j;
    const uint4 raw = *reinterpret_cast<const uint4*>(wp);
    const uint32_t win[4] = {raw.x, raw.y, raw.z, raw.w};
    const uint64_t e = (uint64_t)i * (uint64_t)k + (uint64_t)j;  // multiple of 8
    const Philox4 rnd = stream_block(seed, layer, step, kTagSR, (uint32_t)(e >> 3));
    const uint32_t rw[4] = {rnd.w0, rnd.w1, rnd.w2, rnd.w3};
    uint32_t wout[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float w_lo = bf16_bits_to_float(win[q] & 0xFFFFu);
      const float w_hi = bf16_bits_to_float(win[q] >> 16);
      const float v_lo = fmaf(-s, h[a][2 * q], w_lo);
      const float v_hi = fmaf(-s, h[a][2 * q + 1], w_hi);
      const uint32_t o_lo = sr_bf16_bits(v_lo, rw[q] & 0xFFFFu);
      const uint32_t o_hi = sr_bf16_bits(v_hi, rw[q] >> 16);
      wout[q] = o_lo | (o_hi << 16);
      const float n_lo = bf16_bits_to_float(o_lo), n_hi = bf16_bits_to_float(o_hi);
      sq = fmaf(n_lo, n_lo, sq);
      sq = fmaf(n_hi, n_hi, sq);
    }
    *reinterpret_cast<uint4*>(wp) = make_uint4(wout[0], wout[1], wout[2], wout[3]);
  }
  if (wnorm2_out == nullptr) return;
  // ||W_new||^2: block partial, then the last block sums all partials in order.
  const double total = block_sum_double((double)sq, red);
  const unsigned nblocks = gridDim.x * gridDim.y;
  const unsigned bid = blockIdx.y * gridDim.x + blockIdx.x;
  if (threadIdx.x == 0) {
    wnew_partials[bid] = total;
    __threadfence();
    is_last = (atomicAdd(ticket, 1u) == nblocks - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  double part = 0.0;
  for (unsigned b = threadIdx.x; b < nblocks; b += blockDim.x)
    part += *((volatile double*)&wnew_partials[b]);
  const double all = block_sum_double(part, red);
  if (threadIdx.x == 0) {
    *wnorm2_out = all;
    *ticket = 0u;
  }
}

}  // namespace

void carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd,
                            UpdateWorkspace* ws) {
  UpdateWorkspace w{};
  if (normsgd) {
    w.gram_partials_p = cur.take<float>((size_t)gram_chunks(k).nchunks * r * r);
    w.gram_partials_c = cur.take<float>((size_t)gram_chunks(d).nchunks * r * r);
    w.gram_p = cur.take<float>((size_t)r * r);
    w.gram_c = cur.take<float>((size_t)r * r);
    w.wnorm_partials = cur.take<double>(kWnormBlocks);
    w.wnew_partials = cur.take<double>((size_t)ceil_div(d, 64) * ceil_div(k, 64));
    w.scale = cur.take<float>(1);
    w.status = cur.take<int32_t>(1);
    w.ticket = cur.take<uint32_t>(1);
  }
  if (ws) *ws = w;
}

static size_t update_smem_bytes(int r) { return sizeof(float) * 2 * 64 * (size_t)(r + 1); }

cudaError_t launch_update_normsgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                                  const float* P, int r, float tau, uint64_t seed, uint32_t layer,
                                  uint32_t step, const double* wnorm2_in, double* wnorm2_out,
                                  int32_t* dev_status, const UpdateWorkspace& ws,
                                  cudaStream_t stream) {
  int32_t* status = dev_status ? dev_status : ws.status;
  if (wnorm2_in == nullptr)
    wnorm_partial_kernel<<<kWnormBlocks, 256, 0, stream>>>(W, d, k, ld_w, ws.wnorm_partials);
  GramBatch gb;
  gb.n = 2;
  gb.r = r;
  gb.e[0] = GramEntry{P, k, ws.gram_partials_p, ws.gram_p};
  gb.e[1] = GramEntry{C, d, ws.gram_partials_c, ws.gram_c};
  cudaError_t err = launch_gram(gb, stream);
  if (err != cudaSuccess) return err;
  normsgd_finalize_kernel<<<1, 256, 0, stream>>>(ws.wnorm_partials, kWnormBlocks, wnorm2_in,
                                                 ws.gram_p, ws.gram_c, r * r, tau, ws.scale,
                                                 status, ws.ticket, wnorm2_out);
  const size_t smem = update_smem_bytes(r);
  err = cudaFuncSetAttribute(update_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)ceil_div(k, 64), (unsigned)ceil_div(d, 64));
  update_simt_kernel<<<grid, 256, smem, stream>>>(W, d, k, ld_w, C, P, r, ws.scale, 0.f, status,
                                                  nullptr, seed, layer, step, ws.wnew_partials,
                                                  ws.ticket, wnorm2_out);
  return cudaGetLastError();
}

cudaError_t launch_update_sgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                              const float* P, int r, float alpha_eta, uint64_t seed,
                              uint32_t layer, uint32_t step, int32_t* dev_status,
                              cudaStream_t stream) {
  const size_t smem = update_smem_bytes(r);
  cudaError_t err = cudaFuncSetAttribute(update_simt_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((unsigned)ceil_div(k, 64), (unsigned)ceil_div(d, 64));
  update_simt_kernel<<<grid, 256, smem, stream>>>(W, d, k, ld_w, C, P, r, nullptr, alpha_eta,
                                                  nullptr, dev_status, seed, layer, step, nullptr,
                                                  nullptr, nullptr);
  return cudaGetLastError();
}

}  // namespace rgs
