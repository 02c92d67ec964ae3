// (d) Rebuild H = C P^T fused with the weight update and BF16 stochastic
// rounding, for a batch of layers.
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
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace rgs {
namespace {

constexpr int kMaxUpd = 56;     // layers per rebuild+update launch (kernel parameter table, < 32 KB)
constexpr int kMaxCtas = 256;   // persistent CTAs per launch (one per SM)
constexpr int kMaxAux = 128;    // layers per norm / split launch

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

// ---- ||W||^2 partials ---------------------------------------------------------
struct WnormBatch {
  const uint16_t* W[kMaxAux];
  int64_t d[kMaxAux], k[kMaxAux], ld[kMaxAux];
  double* partials[kMaxAux];  // kWnormBlocks each
};

// Partial sums of W^2 over a fixed assignment of 8-element vectors to threads
// (Kahan-compensated fp32 per thread, double across threads).  grid (1024, n).
__global__ void __launch_bounds__(256) wnorm_partial_kernel(const __grid_constant__ WnormBatch b) {
  __shared__ double red[8];
  const int pr = blockIdx.y;
  const uint16_t* __restrict__ W = b.W[pr];
  const int64_t vec_per_row = b.k[pr] / 8, ld = b.ld[pr];
  const int64_t nvec = b.d[pr] * vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float sum = 0.f, comp = 0.f;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const int64_t i = v / vec_per_row, j = (v % vec_per_row) * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(W + i * ld + j);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float x = bf16_bits_to_float(w[q] & 0xFFFFu), y = bf16_bits_to_float(w[q] >> 16);
      part = fmaf(x, x, part);
      part = fmaf(y, y, part);
    }
    const float y = part - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
  }
  const double total = block_sum_double((double)sum - (double)comp, red);
  if (threadIdx.x == 0) b.partials[pr][blockIdx.x] = total;
}

// ---- scale, status ------------------------------------------------------------
struct FinalizeBatch {
  const double* wnorm_partials[kMaxAux];
  const double* wnorm2_in[kMaxAux];
  const double* gram_p[kMaxAux];
  const double* gram_c[kMaxAux];
  float* scale[kMaxAux];
  int32_t* status[kMaxAux];
  uint32_t* ticket[kMaxAux];
  double* wnorm2_out[kMaxAux];
  int rr;
  float tau;
};

// One block per layer: ||W||^2, ||H||^2 = <Gp, Gc>, the status and s.
__global__ void __launch_bounds__(256) normsgd_finalize_kernel(const __grid_constant__ FinalizeBatch b) {
  __shared__ double red[8];
  const int pr = blockIdx.x;
  const double* gp = b.gram_p[pr];
  const double* gc = b.gram_c[pr];
  double hpart = 0.0;
  for (int e = threadIdx.x; e < b.rr; e += blockDim.x) hpart += gp[e] * gc[e];
  const double nh2 = block_sum_double(hpart, red);
  const double* w_in = b.wnorm2_in[pr];
  double wpart = 0.0;
  if (w_in == nullptr) {
    for (int e = threadIdx.x; e < kWnormBlocks; e += blockDim.x) wpart += b.wnorm_partials[pr][e];
  }
  const double nw2_sum = block_sum_double(wpart, red);
  if (threadIdx.x == 0) {
    const double nw2 = w_in ? *w_in : nw2_sum;
    int32_t st = 0;
    if (!isfinite(nw2)) st |= SKETCH_DEV_W_NONFINITE;
    if (!isfinite(nh2)) st |= SKETCH_DEV_H_NONFINITE;
    else if (nh2 <= 0.0) st |= SKETCH_DEV_H_ZERO;
    const double s = st ? 0.0 : (double)b.tau * sqrt(nw2) / sqrt(nh2);
    *b.scale[pr] = (float)s;
    *b.status[pr] = st;
    *b.ticket[pr] = 0u;
    if (st && b.wnorm2_out[pr]) *b.wnorm2_out[pr] = nw2;  // W stays unchanged
  }
}

// ---- BF16 high/low split of C and P, and their row norms ---------------------
struct SplitBatch {
  const float* src[2 * kMaxAux];
  int64_t row_begin[2 * kMaxAux + 1];  // prefix of the entries' row counts
  uint16_t* dst[2 * kMaxAux];   // rows x (2 r_pad): [hi | lo]
  float* norm[2 * kMaxAux];     // rows: Euclidean norm of each source row
  int n;
  int r;
  int r_pad;
};

// Rows of all entries, grid-stride: x = hi + lo to 2^-17 relative (columns
// r..r_pad-1 zero) and ||row||_2.  A row takes lpr lanes (r_pad / 4 rounded up
// to a power of two, at most 32), lane c its columns 4c..4c+3 of each 4 lpr
// step; a warp holds 32 / lpr rows at a time and four such steps, their loads
// issued before any is used, so one round trip serves up to 4 * 32 / lpr rows.
__global__ void __launch_bounds__(256) split_rows_kernel(const __grid_constant__ SplitBatch b) {
  constexpr int kU = 4;
  const int lane = threadIdx.x & 31;
  const int64_t total = b.row_begin[b.n];
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const bool vec = (b.r & 3) == 0;
  int lpr = 1;
  while (lpr < 32 && 4 * lpr < b.r_pad) lpr <<= 1;
  const int rps = 32 / lpr, sub = lane / lpr, cl = lane % lpr;
  int en[kU];  // entry of each step's row (rows of a lane only move forward)
#pragma unroll
  for (int u = 0; u < kU; ++u) en[u] = 0;
  for (int64_t g0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kU * rps; g0 < total;
       g0 += warps * kU * rps) {
    float v[kU][4];
    int64_t row[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t gr = g0 + (int64_t)u * rps + sub;
      row[u] = -1;
#pragma unroll
      for (int t = 0; t < 4; ++t) v[u][t] = 0.f;
      if (gr >= total) continue;
      while (en[u] + 1 < b.n && b.row_begin[en[u] + 1] <= gr) ++en[u];
      row[u] = gr - b.row_begin[en[u]];
      const float* src = b.src[en[u]] + row[u] * b.r;
      const int c0 = 4 * cl;
      if (c0 >= b.r) continue;
      if (vec) {
        const float4 f = *reinterpret_cast<const float4*>(src + c0);
        v[u][0] = f.x;
        v[u][1] = f.y;
        v[u][2] = f.z;
        v[u][3] = f.w;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) v[u][t] = (c0 + t < b.r) ? src[c0 + t] : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float sq = 0.f;
      if (row[u] >= 0) {
        uint16_t* dst = b.dst[en[u]] + row[u] * 2 * b.r_pad;
        for (int c0 = 4 * cl; c0 < b.r_pad; c0 += 4 * lpr) {
          float w[4];
          if (c0 == 4 * cl) {
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = v[u][t];
          } else {  // rows wider than 4 lpr columns (r_pad > 128): the rest here
            const float* src = b.src[en[u]] + row[u] * b.r;
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = (c0 + t < b.r) ? src[c0 + t] : 0.f;
          }
          uint16_t hi[4], lo[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            sq = fmaf(w[t], w[t], sq);
            const __nv_bfloat16 h = __float2bfloat16_rn(w[t]);
            hi[t] = __bfloat16_as_ushort(h);
            lo[t] = __bfloat16_as_ushort(__float2bfloat16_rn(w[t] - __bfloat162float(h)));
          }
          // r_pad is a multiple of 16: the 4 columns are inside the row, 8-byte aligned
          *reinterpret_cast<uint2*>(dst + c0) =
              make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
          *reinterpret_cast<uint2*>(dst + b.r_pad + c0) =
              make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
        }
      }
      // the row's lanes sum their squares (groups of lpr lanes)
      for (int o = lpr >> 1; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
      if (row[u] >= 0 && cl == 0) b.norm[en[u]][row[u]] = sqrtf(sq);
    }
  }
}

// ---- the rebuild + update kernel -------------------------------------------------
// Work of a launch: up to kMaxUpd layers.  Layer p is cut into units of
// (128-row block, run of up to unit_tiles column tiles of NCOLS); units of all
// layers are numbered end to end and each persistent CTA takes a contiguous
// range of them, so consecutive units usually share the row block of C.
struct UpdBatch {
  CUtensorMap tm_c[kMaxUpd];   // C split, d x (2 r_pad) BF16: [hi | lo]
  CUtensorMap tm_p[kMaxUpd];   // P split, k x (2 r_pad) BF16: [hi | lo]
  CUtensorMap tm_w[kMaxUpd];   // W, d x k BF16 (tile loads)
  uint16_t* W[kMaxUpd];        // W for the results, stored from registers
  int64_t ld_w[kMaxUpd];
  const float* C[kMaxUpd];     // fp32 C and P for the exact recomputation
  const float* P[kMaxUpd];
  const float* c_norm[kMaxUpd];
  const float* p_norm[kMaxUpd];
  int64_t d[kMaxUpd], k[kMaxUpd];
  int n_ct[kMaxUpd];           // column tiles of the layer
  int n_cu[kMaxUpd];           // units per row block
  int unit_begin[kMaxUpd + 1];
  uint32_t layer[kMaxUpd];
  const float* scale_dev[kMaxUpd];     // normalized SGD: s on the device; NULL: scale_val
  const int32_t* status_in[kMaxUpd];   // skip the layer when nonzero
  int32_t* status_out[kMaxUpd];        // SGD: set to 0
  double* unit_partials[kMaxUpd];      // ||W_new||^2 of each unit
  uint32_t* ticket[kMaxUpd];
  double* wnorm2_out[kMaxUpd];
  int cta_unit_begin[kMaxCtas + 1];  // units of CTA b: [cta_unit_begin[b], cta_unit_begin[b + 1])
  int n;
  int unit_tiles;
  int p_stages;       // P ring depth
  int w_stages;       // W ring depth
  float scale_val;
  uint64_t seed;
  uint32_t rk0[10], rk1[10];  // Philox round keys of the seed
  uint32_t step;
  int r;
  int r_pad;          // r rounded up to 16 (MMA K extent)
  int kchunks;        // 64-wide chunks of r_pad
  uint32_t a_bytes;   // bytes of the C_hi (or C_lo) tile: kchunks x 16 KB
  uint32_t b_bytes;   // bytes of the P_hi (or P_lo) tile: kchunks x NCOLS x 128
  uint32_t w_bytes;   // bytes of the W tile: NCOLS/64 x 16 KB
  int list_cap;       // entries of the careful-word list that fit the dynamic shared memory
  int* err;
  // careful-group flags, one bit per 8-weight group: per tile (rb, ct), word
  // ew * (NCOLS/32) + g holds bit `lane` for row rb*128 + (ew&3)*32 + lane,
  // columns ct*NCOLS + (ew>>2)*(NCOLS/4) + 8g..+7 (ew = epilogue warp)
  uint32_t* flags[kMaxUpd];
};

// kernel parameters are limited to 32764 bytes
static_assert(sizeof(UpdBatch) <= 32764, "UpdBatch exceeds the kernel parameter limit");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int kEpiWarps = 16;                     // warps 4..19: four per TMEM lane quarter
constexpr int kUpdThreads = (4 + kEpiWarps) * 32;
constexpr int kMaxStagesUpd = 8;

struct Unit {
  int p, rb, ct0, ct1;
};

// Error-free transformations (Ogita, Rump and Oishi, "Accurate Sum and Dot
// Product", 2005): a + b = s + e and a * b = p + e exactly in fp32.  The
// explicit _rn intrinsics keep the compiler from fusing or reordering them.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ Unit decode_unit(const UpdBatch& a, int u) {
  Unit x;
  int p = 0;
  while (p + 1 < a.n && a.unit_begin[p + 1] <= u) ++p;
  const int lu = u - a.unit_begin[p];
  x.p = p;
  x.rb = lu / a.n_cu[p];
  const int cu = lu % a.n_cu[p];
  x.ct0 = cu * a.unit_tiles;
  x.ct1 = min(a.n_ct[p], x.ct0 + a.unit_tiles);
  return x;
}

// One careful group, warp-wide: W_new of the 8 elements (i, j..j+7) of
// problem p from their original W, with H_i,j+t computed by the compensated
// dot product (Dot2 of the same paper; lanes 4t..4t+3 take column t, every
// fourth term each, merged by TwoSum), v = fmaf(-s, fl32(H), w) and the
// group's Philox block.  The dot product is as accurate as one carried in
// twice fp32 precision and then rounded, so it is fl32 of the exact H except
// when H lies within ~2^-40 of its size of an fp32 rounding boundary.  All
// fp32: this GPU's FP64 rate is far too low for the purpose.
__device__ __forceinline__ void careful_group_warp(const UpdBatch& a, int p, int i, int j) {
  const int lane = threadIdx.x & 31, t = lane >> 2, q = lane & 3;
  const int r = a.r;
  const float* crow = a.C[p] + (int64_t)i * r;
  const float* prow = a.P[p] + (int64_t)(j + t) * r;
  uint16_t* wp = a.W[p] + (int64_t)i * a.ld_w[p] + j + t;
  const uint32_t w16 = *wp;  // the original: the update kernel left the group alone
  float hi = 0.f, lo = 0.f;
  auto term = [&](float c, float pv) {
    const float m = __fmul_rn(c, pv);
    float sum, err;
    two_sum(hi, m, sum, err);
    hi = sum;
    lo = __fadd_rn(lo, __fadd_rn(err, __fmaf_rn(c, pv, -m)));
  };
  // the terms l = q, q+4, ... of this lane, sixteen loads of C and P at a
  // time issued together (one round trip per 64 terms of the row)
  int l = q;
  for (; l + 60 < r; l += 64) {
    float cv[16], pv[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      cv[m] = crow[l + 4 * m];
      pv[m] = prow[l + 4 * m];
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) term(cv[m], pv[m]);
  }
  if (l < r) {
    float cv[16], pv[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const bool in = l + 4 * m < r;
      cv[m] = in ? crow[l + 4 * m] : 0.f;
      pv[m] = in ? prow[l + 4 * m] : 0.f;
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) term(cv[m], pv[m]);  // zero terms change nothing
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const float ohi = __shfl_xor_sync(0xFFFFFFFFu, hi, o), olo = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
    float sum, err;
    two_sum(hi, ohi, sum, err);
    hi = sum;
    lo = __fadd_rn(lo, __fadd_rn(olo, err));
  }
  const float h = __fadd_rn(hi, lo);
  const float s = a.scale_dev[p] ? *a.scale_dev[p] : a.scale_val;
  const uint32_t blk = (uint32_t)i * ((uint32_t)a.k[p] >> 3) + ((uint32_t)j >> 3);  // element index / 8
  const Philox4 rnd = philox4x32_10_rk(blk, a.step, a.layer[p], kTagSR, a.rk0, a.rk1);
  const uint32_t word = (t >> 1) == 0 ? rnd.w0 : (t >> 1) == 1 ? rnd.w1 : (t >> 1) == 2 ? rnd.w2 : rnd.w3;
  const float v = fmaf(-s, h, __uint_as_float(w16 << 16));
  const uint32_t o = sr_bf16_bits(v, (t & 1) ? (word >> 16) : (word & 0xFFFFu));
  __syncwarp();
  if (q == 0) *wp = (uint16_t)o;
}

// Persistent rebuild + update, one CTA per SM, each CTA a contiguous range of
// units (a unit: one 128-row block of one layer and up to unit_tiles column
// tiles of NCOLS).  Warp 0 (one lane) streams with TMA the split C row block of
// each unit (C_hi, C_lo), the P_hi/P_lo rows of each column tile into a P ring
// and the W tile into a deeper W ring.  Warp 1 (one lane) issues
// H = C_hi P_hi^T + C_hi P_lo^T + C_lo P_hi^T (tcgen05.mma, M=128, N=NCOLS)
// into one of two TMEM buffers and frees the P stage with tcgen05.commit.
// The 16 epilogue warps (warps 4..19, four per TMEM lane quarter, one column
// quarter each) read H from TMEM, form v = fmaf(-s, H, w) with w from the W
// stage, round it stochastically with 16 Philox bits per weight and write the
// BF16 results back into the stage; warp 2 (one lane) writes each finished
// tile to W with a TMA tensor store and frees the stage.  After the main loop
// all 20 warps redo the flagged groups (the careful groups, below).
//
// Exactness where it matters: |H_tc - H| <= ~2^-14.2 ||c_i|| ||p_j|| (the
// dropped lo*lo and residual terms, ~3 * 2^-16 of sum |c_l p_l|, plus the fp32
// accumulation), which moves v across at most one BF16 step unless
// |v| < s ||c_i|| ||p_j|| 2^-6.  A group of 8 weights holding a |v| below
// s ||c_i|| max_j ||p_j|| 2^-5 (the maximum over the warp's 32 columns of the
// tile: twice that margin) or a NaN keeps its original W in the stage and is
// flagged; the careful pass recomputes its elements with fl32(H_ij) from a
// compensated dot product, which is the value the definition rounds.
template <int NCOLS>
__global__ void __launch_bounds__(kUpdThreads, 1) update_persistent_kernel(const __grid_constant__ UpdBatch a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t pfull_bar[kMaxStagesUpd], pempty_bar[kMaxStagesUpd];
  __shared__ __align__(8) uint64_t wfull_bar[kMaxStagesUpd], wempty_bar[kMaxStagesUpd], sfull_bar[kMaxStagesUpd];
  __shared__ __align__(8) uint64_t cfull_bar, cempty_bar, tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ int clist_n;  // entries of the careful-word list
  __shared__ uint32_t skip_mask[(kMaxUpd + 31) / 32];  // layers whose status_in is nonzero
  __shared__ double warp_sq[kEpiWarps];

  uint8_t* smem = align1024(smem_raw);
  uint8_t* s_chi = smem;
  uint8_t* s_clo = s_chi + a.a_bytes;
  uint8_t* s_p0 = s_clo + a.a_bytes;                        // P ring: NSP x (hi, lo)
  uint8_t* s_w0 = s_p0 + (size_t)a.p_stages * 2 * a.b_bytes;  // W ring: NSW x W tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NSP = a.p_stages, NSW = a.w_stages;
  const int u_begin = a.cta_unit_begin[blockIdx.x];
  const int u_end = a.cta_unit_begin[blockIdx.x + 1];
  constexpr uint32_t kTmemCols = 2 * NCOLS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NSP; ++s) {
      tc::mbar_init(&pfull_bar[s], 1);
      tc::mbar_init(&pempty_bar[s], 1);           // MMA commit
    }
    for (int s = 0; s < NSW; ++s) {
      tc::mbar_init(&wfull_bar[s], 1);
      tc::mbar_init(&sfull_bar[s], kEpiWarps);    // every epilogue warp: results in the stage
      tc::mbar_init(&wempty_bar[s], 1);           // store warp: the stage's TMA store has read it
    }
    tc::mbar_init(&cfull_bar, 1);
    tc::mbar_init(&cempty_bar, 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull_bar[b], 1);
      tc::mbar_init(&tempty_bar[b], kEpiWarps);
    }
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, kTmemCols);
  if (warp == 3) {
    // the skipped layers, read once here instead of at every unit
#pragma unroll
    for (int h = 0; h < (kMaxUpd + 31) / 32; ++h) {
      const int pp = 32 * h + lane;
      const bool sk = pp < a.n && a.status_in[pp] != nullptr && *a.status_in[pp] != 0;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, sk);
      if (lane == 0) skip_mask[h] = m;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  auto layer_skipped = [&](int pp) { return (skip_mask[pp >> 5] >> (pp & 31)) & 1u; };

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    int it = 0, cl = 0, prev_p = -1, prev_rb = -1;
    bool stop = false;
    for (int u = u_begin; u < u_end && !stop; ++u) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      const int i0 = x.rb * 128;
      if (x.p != prev_p || x.rb != prev_rb) {
        if (cl > 0 && !tc::mbar_wait(&cempty_bar, (cl - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) break;
        tc::mbar_arrive_expect_tx(&cfull_bar, 2 * a.a_bytes);
        for (int c = 0; c < a.kchunks; ++c) {
          tc::tma_load_2d(s_chi + c * 16384, &a.tm_c[x.p], &cfull_bar, c * 64, i0);
          tc::tma_load_2d(s_clo + c * 16384, &a.tm_c[x.p], &cfull_bar, a.r_pad + c * 64, i0);
        }
        ++cl;
        prev_p = x.p;
        prev_rb = x.rb;
      }
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int j0 = ct * NCOLS;
        // W tile first: it comes from HBM and is waited on longest
        const int sw = it % NSW;
        if (it >= NSW && !tc::mbar_wait(&wempty_bar[sw], ((it / NSW) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* wst = s_w0 + (size_t)sw * a.w_bytes;
        tc::mbar_arrive_expect_tx(&wfull_bar[sw], a.w_bytes);
#pragma unroll
        for (int bx = 0; bx < NCOLS / 64; ++bx)
          tc::tma_load_2d(wst + bx * 16384, &a.tm_w[x.p], &wfull_bar[sw], j0 + 64 * bx, i0);
        const int sp = it % NSP;
        if (it >= NSP && !tc::mbar_wait(&pempty_bar[sp], ((it / NSP) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* pst = s_p0 + (size_t)sp * 2 * a.b_bytes;
        tc::mbar_arrive_expect_tx(&pfull_bar[sp], 2 * a.b_bytes);
        for (int c = 0; c < a.kchunks; ++c) {
          tc::tma_load_2d(pst + c * NCOLS * 128, &a.tm_p[x.p], &pfull_bar[sp], c * 64, j0);
          tc::tma_load_2d(pst + a.b_bytes + c * NCOLS * 128, &a.tm_p[x.p], &pfull_bar[sp], a.r_pad + c * 64, j0);
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = tc::idesc_bf16(128, NCOLS, false, false);
    int it = 0, cl = 0, prev_p = -1, prev_rb = -1;
    bool stop = false;
    for (int u = u_begin; u < u_end && !stop; ++u) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      if (x.p != prev_p || x.rb != prev_rb) {
        if (!tc::mbar_wait(&cfull_bar, cl & 1, &abort_flag, a.err, tc::kErrTimeoutLoad)) break;
        ++cl;
        prev_p = x.p;
        prev_rb = x.rb;
      }
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int sp = it % NSP, b = it & 1;
        if (!tc::mbar_wait(&pfull_bar[sp], (it / NSP) & 1, &abort_flag, a.err, tc::kErrTimeoutLoad) ||
            (it >= 2 && !tc::mbar_wait(&tempty_bar[b], ((it >> 1) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage))) {
          stop = true;
          break;
        }
        tc::tc_fence_after();
        const uint32_t pst = tc::smem_u32(s_p0 + (size_t)sp * 2 * a.b_bytes);
        const uint32_t d_tmem = tmem + (uint32_t)(b * NCOLS);
        uint32_t acc = 0;
        for (int c = 0; c < a.kchunks; ++c) {
          for (int kk = 0; kk < 4 && c * 64 + kk * 16 < a.r_pad; ++kk) {
            const uint32_t off_a = c * 16384 + kk * 32, off_b = c * NCOLS * 128 + kk * 32;
            const uint64_t ahi = tc::sdesc_sw128(tc::smem_u32(s_chi) + off_a, 16, 1024);
            const uint64_t alo = tc::sdesc_sw128(tc::smem_u32(s_clo) + off_a, 16, 1024);
            const uint64_t bhi = tc::sdesc_sw128(pst + off_b, 16, 1024);
            const uint64_t blo = tc::sdesc_sw128(pst + a.b_bytes + off_b, 16, 1024);
            tc::mma_bf16(d_tmem, ahi, bhi, idesc, acc);
            tc::mma_bf16(d_tmem, ahi, blo, idesc, 1u);
            tc::mma_bf16(d_tmem, alo, bhi, idesc, 1u);
            acc = 1u;
          }
        }
        tc::mma_commit(&pempty_bar[sp]);
        tc::mma_commit(&tfull_bar[b]);
      }
      // release the C row block once its last unit is issued
      bool last_of_c = (u + 1 == u_end);
      if (!last_of_c) {
        const Unit y = decode_unit(a, u + 1);
        last_of_c = (y.p != x.p || y.rb != x.rb);
      }
      if (last_of_c && !stop) tc::mma_commit(&cempty_bar);
    }
  } else if (warp == 2 && lane == 0) {
    // ---------------- store warp ----------------
    // Writes each finished tile from its W stage to W with TMA, then frees
    // the stage once the copy has read it.
    int it = 0;
    bool stop = false;
    for (int u = u_begin; u < u_end && !stop; ++u) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int sw = it % NSW;
        if (!tc::mbar_wait(&sfull_bar[sw], (it / NSW) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* wst = s_w0 + (size_t)sw * a.w_bytes;
        if (!abort_flag) {  // after a timed-out wait the stage may hold anything
#pragma unroll
          for (int bx = 0; bx < NCOLS / 64; ++bx)
            tc::tma_store_2d(&a.tm_w[x.p], wst + bx * 16384, ct * NCOLS + 64 * bx, x.rb * 128);
          tc::bulk_commit();
          tc::bulk_wait_read<0>();
        }
        tc::mbar_arrive(&wempty_bar[sw]);
      }
    }
    tc::bulk_wait_all();  // the writes are done before the CTA exits
    // ... and visible to the generic loads of the careful-group pass below
    asm volatile("fence.proxy.async.global;" ::: "memory");
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int ew = warp - 4;
    const int quarter = warp & 3;
    constexpr int kCols = NCOLS / 4;           // columns per thread per tile
    constexpr int kPass = kCols < 32 ? kCols : 32;  // columns per pass
    constexpr int kGroups = kPass / 8;              // 8-column groups (Philox blocks) per pass
    constexpr int kGroupsPerWarp = kCols / 8;       // flag words of a warp per tile
    // byte offset in a W stage (two 64-column, 128-byte-swizzled boxes) of this
    // thread's 8-column groups: row q, column col_base + 8g
    uint32_t stage_off[kGroupsPerWarp];
#pragma unroll
    for (int g = 0; g < kGroupsPerWarp; ++g) {
      const int col = (ew >> 2) * kCols + 8 * g;
      const int qq = (warp & 3) * 32 + lane;
      stage_off[g] = (uint32_t)((col >> 6) * 16384 + qq * 128 + ((((col & 63) >> 3) ^ (qq & 7)) << 4));
    }
    const int col_base = (ew >> 2) * kCols;    // column quarter of the tile
    const int q = quarter * 32 + lane;         // tile row = TMEM lane
    const bool storer = (ew == 0 && lane == 0);
    int it = 0;
    // Every epilogue warp runs the same loop and reaches every named barrier;
    // after a timed-out wait (abort) the work is skipped but the barriers are not.
    for (int u = u_begin; u < u_end; ++u) {
      const Unit x = decode_unit(a, u);
      const int p = x.p;
      if (layer_skipped(p)) continue;
      // d, k < 2^31 and d*k/8 < 2^32 (checked on the host): 32-bit indices
      const int d = (int)a.d[p], k = (int)a.k[p];
      const int i = x.rb * 128 + q;
      const uint32_t k8 = (uint32_t)k >> 3;
      const bool row_ok = i < d;
      const float s = a.scale_dev[p] ? *a.scale_dev[p] : a.scale_val;
      const float thr_row = row_ok ? fabsf(s) * a.c_norm[p][i] * 0x1p-5f : 0.f;
      const uint32_t layer = a.layer[p];
      const bool need_norm = a.wnorm2_out[p] != nullptr;
      float sq = 0.f, sq_comp = 0.f;  // Kahan-compensated sum of squares

      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int sw = it % NSW, b = it & 1;
        const int j0 = ct * NCOLS;
        // largest norm of the P rows of this thread's columns (for the exactness
        // test), loaded before the waits so that its latency hides behind them
        float pmax = 0.f;
        {
          const float* pnorm = a.p_norm[p];
          const int jc = j0 + col_base + 2 * (lane % (kCols / 2));
          if (jc + 1 < k) {
            const float2 pn = *reinterpret_cast<const float2*>(pnorm + jc);
            pmax = fmaxf(pn.x, pn.y);
          } else if (jc < k) {
            pmax = pnorm[jc];
          }
        }
        // W tile and H of this tile
        bool live = tc::mbar_wait(&wfull_bar[sw], (it / NSW) & 1, &abort_flag, a.err, tc::kErrTimeoutLoad) &&
                    tc::mbar_wait(&tfull_bar[b], (it >> 1) & 1, &abort_flag, a.err, tc::kErrTimeoutMma);
        live = __all_sync(0xFFFFFFFFu, live);
        tc::tc_fence_after();
        const uint32_t s_w32 = tc::smem_u32(s_w0) + (uint32_t)sw * a.w_bytes;
        for (int o = 16; o > 0; o >>= 1) pmax = fmaxf(pmax, __shfl_xor_sync(0xFFFFFFFFu, pmax, o));
        const float thr = thr_row * pmax;
        // live is the same in the whole warp: one branch per tile
        if (live) {
#pragma unroll 1
          for (int half = 0; half < kCols / kPass; ++half) {
            const int col32 = col_base + half * kPass;
            // H of the pass from TMEM, 16 columns at a time; the first load
            // completes while the Philox blocks of the pass (independent chains)
            // are computed
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * NCOLS + col32);
            uint32_t h[16];
            tc::tmem_ld_32x32b<16>(taddr, h);
            // Philox block of element index e = i*k + j (j a multiple of 8): e / 8
            uint32_t blks[kGroups];
#pragma unroll
            for (int g = 0; g < kGroups; ++g) blks[g] = (uint32_t)i * k8 + ((uint32_t)(j0 + col32 + 8 * g) >> 3);
            uint32_t rw[kGroups][4];
            philox4x32_10_rk_multi<kGroups>(blks, a.step, layer, kTagSR, a.rk0, a.rk1, rw);
            tc::tmem_wait_ld_regs<16>(h);
            // Per 8-column group: v = fmaf(-s, H, w) and stochastic rounding (add
            // 16 random bits below the BF16 mantissa, keep the upper halves: one
            // PRMT per pair); the results go back into the W stage in place (the
            // store warp writes the tile out with TMA, clipping rows and columns
            // outside W).  A group that holds a NaN or a value small enough for
            // the exactness test is flagged for the careful path.
            uint32_t fwords[kGroups];
            float gs = 0.f;  // sum of squares of this pass's results (normalized SGD)
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              if (g == 2) {  // next 16 columns of H
                tc::tmem_ld_32x32b<16>(taddr + 16, h);
                tc::tmem_wait_ld_regs<16>(h);
              }
              const int col = col32 + 8 * g;
              const uint32_t sp = s_w32 + stage_off[half * kGroups + g];
              const uint4 raw = tc::lds128(sp);
              const uint32_t win[4] = {raw.x, raw.y, raw.z, raw.w};
              const uint32_t* rwg = rw[g];
              uint32_t wout[4];
              float av[8];
#pragma unroll
              for (int t2 = 0; t2 < 4; ++t2) {
                // BF16 -> fp32 by shifting into the high half; the integer steps
                // use multiply-adds so that they share the multiplier pipe with
                // Philox instead of crowding the ALU pipe: r_hi = r >> 16,
                // r_lo = r - r_hi * 2^16 = r & 0xFFFF
                const uint32_t wword = win[t2], rword = rwg[t2];
                const float v0 = fmaf(-s, __uint_as_float(h[8 * (g & 1) + 2 * t2]),
                                      __uint_as_float(mad_lo(wword, 0x10000u, 0u)));
                const float v1 = fmaf(-s, __uint_as_float(h[8 * (g & 1) + 2 * t2 + 1]),
                                      __uint_as_float(wword & 0xFFFF0000u));
                const uint32_t r_hi = mad_hi(rword, 0x10000u, 0u);
                const uint32_t r_lo = mad_lo(r_hi, 0xFFFF0000u, rword);
                const uint32_t s0 = mad_lo(r_lo, 1u, __float_as_uint(v0));
                const uint32_t s1 = mad_hi(rword, 0x10000u, __float_as_uint(v1));
                wout[t2] = __byte_perm(s0, s1, 0x7632);
                av[2 * t2] = fabsf(v0);  // folded into the min as an operand modifier
                av[2 * t2 + 1] = fabsf(v1);
              }
              // smallest |v| of the group; NaN if any v is NaN
              const float gmin = fmin3_nan(fmin3_nan(av[0], av[1], av[2]), fmin3_nan(av[3], av[4], av[5]),
                                           fmin_nan(av[6], av[7]));
              const bool ok = row_ok && j0 + col < k;
              const bool flag = ok && !(gmin >= thr);  // small value or NaN
              // Careful path: a flagged group keeps its original W here and is
              // marked in the flag bitmap (the word of the whole warp, written on
              // every call); the careful-group pass at the end of this kernel
              // redoes its 8 elements exactly from the original W, once the
              // tiles are stored.  The norm sum keeps the tensor-core values of
              // the group (they differ from the exact ones by at most one BF16
              // step, or are below the threshold), except that a NaN makes it
              // NaN.  The rare writes are predicated, not branched around.
              fwords[g] = __ballot_sync(0xFFFFFFFFu, flag);
              tc::sts128(sp, make_uint4(wout[0], wout[1], wout[2], wout[3]));
              tc::sts128_if(sp, raw, flag);  // rare: the careful pass needs the original
              if (need_norm) {
                float t = gs;
#pragma unroll
                for (int t2 = 0; t2 < 4; ++t2) t = sq_acc_bf16x2(wout[t2], t);
                gs = ok ? t : gs;
                sq = (ok && gmin != gmin) ? __int_as_float(0x7FC00000) : sq;
              }
            }
            if (need_norm) {  // the pass's squares into the compensated sum
              const float y = gs - sq_comp;
              const float tsum = sq + y;
              sq_comp = (tsum - sq) - y;
              sq = tsum;
            }
            if (lane == 0) {  // every word of the layer is written on every call
              uint32_t* fw = a.flags[p] + ((size_t)x.rb * a.n_ct[p] + ct) * (16 * kGroupsPerWarp) +
                             ew * kGroupsPerWarp + half * kGroups;
              if constexpr (kGroups == 4)
                *reinterpret_cast<uint4*>(fw) = make_uint4(fwords[0], fwords[1], fwords[2], fwords[3]);
              else
                *reinterpret_cast<uint2*>(fw) = make_uint2(fwords[0], fwords[1]);
            }
          }
        }
        // this warp is done with the TMEM buffer
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty_bar[b]);
        // this warp's results are in the stage: make them visible to the TMA
        // engine and tell the store warp
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sfull_bar[sw]);
      }
      if (need_norm) {
        // ||W_new||^2 of this unit, then the layer's last unit sums all units in order
        double dsq = (double)sq - (double)sq_comp;
        for (int o = 16; o > 0; o >>= 1) dsq += __shfl_xor_sync(0xFFFFFFFFu, dsq, o);
        if (lane == 0) warp_sq[ew] = dsq;
        tc::named_barrier(1, kEpiWarps * 32);
        if (storer) {
          double tot = 0.0;
          for (int w = 0; w < kEpiWarps; ++w) tot += warp_sq[w];
          const int lu = u - a.unit_begin[p];
          a.unit_partials[p][lu] = tot;
          __threadfence();
          const unsigned nunits = (unsigned)(a.unit_begin[p + 1] - a.unit_begin[p]);
          if (atomicAdd(a.ticket[p], 1u) == nunits - 1) {
            __threadfence();
            double all = 0.0;
            for (unsigned b2 = 0; b2 < nunits; ++b2) all += *((volatile double*)&a.unit_partials[p][b2]);
            *a.wnorm2_out[p] = all;
            *a.ticket[p] = 0u;
          }
        }
        tc::named_barrier(1, kEpiWarps * 32);  // warp_sq reusable
      }
    }
  }
  // SGD: every layer's status word reads 0 (written by the first CTA)
  if (blockIdx.x == 0) {
    for (int p = threadIdx.x; p < a.n; p += blockDim.x)
      if (a.status_out[p] != nullptr) *a.status_out[p] = 0;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
  if (abort_flag) return;

  // Careful groups of this CTA's tiles.  Each flagged group still holds its
  // original W (the stage kept it and the TMA stores above have completed), so
  // it is redone exactly here.  Pass 1: the warps read the flag words of the
  // CTA's units (units in turn) and append the nonzero ones to a list in the
  // now idle dynamic shared memory.
  // Pass 2: the warps take the list's words in turn, so each warp redoes about
  // the same number of groups; the operands of a warp's next word are
  // prefetched into L2 while it works on the current one.  A word that finds
  // the list full is redone at once by the warp that read it.
  constexpr int kWarps = kUpdThreads / 32;
  constexpr int kGroupsPerWarpT = NCOLS / 32, kWordsPerTile = 16 * kGroupsPerWarpT;
  constexpr int kBatch = 8;  // flag words per lane per load batch
  uint4* clist = reinterpret_cast<uint4*>(smem);
  if (threadIdx.x == 0) clist_n = 0;
  __syncthreads();
  // the careful groups of word `bits` at word index widx of layer p
  auto redo_word = [&](int p, uint32_t widx, uint32_t bits) {
    const uint32_t tile = widx / kWordsPerTile, wt = widx % kWordsPerTile;
    const int n_ct = a.n_ct[p];
    const int rb = (int)(tile / (uint32_t)n_ct), ct = (int)(tile % (uint32_t)n_ct);
    const int ew = (int)wt / kGroupsPerWarpT, gw = (int)wt % kGroupsPerWarpT;
    const int j = ct * NCOLS + (ew >> 2) * (NCOLS / 4) + 8 * gw;
    while (bits) {
      const int row = __ffs(bits) - 1;
      bits &= bits - 1;
      careful_group_warp(a, p, rb * 128 + (ew & 3) * 32 + row, j);
    }
  };
  // pass 1: warp w reads the flag words of units w, w + kWarps, ... (a unit's
  // words are contiguous), kBatch words per lane at a time
  for (int u = u_begin + warp; u < u_end; u += kWarps) {
    const Unit x = decode_unit(a, u);
    if (layer_skipped(x.p)) continue;
    const uint32_t wbeg = (uint32_t)(x.rb * a.n_ct[x.p] + x.ct0) * (uint32_t)kWordsPerTile;
    const uint32_t nwords = (uint32_t)(x.ct1 - x.ct0) * (uint32_t)kWordsPerTile;
    const uint32_t* fw = a.flags[x.p] + wbeg;
    for (uint32_t w0 = 0; w0 < nwords; w0 += 32 * kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const uint32_t idx = w0 + 32 * b + lane;
        v[b] = idx < nwords ? fw[idx] : 0u;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const uint32_t nz = __ballot_sync(0xFFFFFFFFu, v[b] != 0u);
        if (nz == 0u) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(&clist_n, __popc(nz));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        const int slot = base + __popc(nz & ((1u << lane) - 1u));
        const uint32_t widx = wbeg + w0 + 32 * b + lane;
        const bool mine = v[b] != 0u;
        if (mine && slot < a.list_cap) clist[slot] = make_uint4((uint32_t)x.p, widx, v[b], 0u);
        uint32_t over = __ballot_sync(0xFFFFFFFFu, mine && slot >= a.list_cap);
        while (over) {  // the list is full: redo these words here
          const int src = __ffs(over) - 1;
          over &= over - 1;
          redo_word(x.p, __shfl_sync(0xFFFFFFFFu, widx, src), __shfl_sync(0xFFFFFFFFu, v[b], src));
        }
      }
    }
  }
  __syncthreads();
  const int n_list = clist_n < a.list_cap ? clist_n : a.list_cap;
  // pass 2: entries warp, warp + kWarps, ...; the operands of the warp's next
  // entry are prefetched into L2 while it works on the current one
  for (int e = warp; e < n_list; e += kWarps) {
    const uint4 en = clist[e];
    if (e + kWarps < n_list) {
      const uint4 nx = clist[e + kWarps];
      const int p2 = (int)nx.x;
      const uint32_t tile = nx.y / kWordsPerTile, wt = nx.y % kWordsPerTile;
      const int n_ct = a.n_ct[p2];
      const int rb = (int)(tile / (uint32_t)n_ct), ct = (int)(tile % (uint32_t)n_ct);
      const int ew = (int)wt / kGroupsPerWarpT, gw = (int)wt % kGroupsPerWarpT;
      const int j = ct * NCOLS + (ew >> 2) * (NCOLS / 4) + 8 * gw;
      const int i = rb * 128 + (ew & 3) * 32 + __ffs(nx.z) - 1;
      const int r = a.r, kk = (int)a.k[p2];
      const int jn = (kk - j) < 8 ? (kk - j) : 8;
      // P rows j..j+jn-1 (contiguous), the C row and the W group: one address
      // per 128-byte line, every address inside its buffer
      const char* pbase = reinterpret_cast<const char*>(a.P[p2] + (int64_t)j * r);
      const int pbytes = jn * r * 4, plines = pbytes / 128 + 2;
      const char* cbase = reinterpret_cast<const char*>(a.C[p2] + (int64_t)i * r);
      const int cbytes = r * 4, clines = cbytes / 128 + 2;
      for (int l = lane; l < plines + clines + 1; l += 32) {
        const char* ad = l < plines ? pbase + min(128 * l, pbytes - 1)
                         : l < plines + clines ? cbase + min(128 * (l - plines), cbytes - 1)
                                               : reinterpret_cast<const char*>(a.W[p2] + (int64_t)i * a.ld_w[p2] + j);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(ad));
      }
    }
    redo_word((int)en.x, en.y, en.z);
  }
}

int round16(int r) { return (r + 15) / 16 * 16; }

// Columns per tile: the C row block plus two or more stages of (P tile, W tile)
// must fit in shared memory.
int update_ncols(int r) { return round16(r) <= 64 ? 128 : 64; }

template <int NCOLS>
cudaError_t launch_update_tc(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, bool normsgd,
                             float scale_val, uint64_t seed, uint32_t step, cudaStream_t stream) {
  const int r_pad = round16(r);
  int* errw = nullptr;
  cudaError_t err = device_error_word(&errw);
  if (err != cudaSuccess) return err;
  static thread_local UpdBatch a;
  a.scale_val = scale_val;
  a.seed = seed;
  philox_round_keys(seed, a.rk0, a.rk1);
  a.step = step;
  a.r = r;
  a.r_pad = r_pad;
  a.kchunks = (r_pad + 63) / 64;
  a.a_bytes = (uint32_t)a.kchunks * 16384u;
  a.b_bytes = (uint32_t)a.kchunks * NCOLS * 128u;
  a.w_bytes = (uint32_t)(NCOLS / 64) * 16384u;
  a.err = errw;
  // dynamic shared memory: what the opt-in limit leaves next to the static arrays
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, update_persistent_kernel<NCOLS>);
  if (err != cudaSuccess) return err;
  const size_t max_smem = 227 * 1024 - fa.sharedSizeBytes;
  const size_t fixed = 2 * (size_t)a.a_bytes + 1024;
  const size_t p_stage = 2 * (size_t)a.b_bytes;
  // two P stages when they fit next to at least two W stages, else one
  int p_stages = (fixed + 2 * p_stage + 2 * a.w_bytes <= max_smem) ? 2 : 1;
  int w_stages = (int)((max_smem - fixed - p_stages * p_stage) / a.w_bytes);
  if (w_stages > kMaxStagesUpd) w_stages = kMaxStagesUpd;
  if (w_stages < 1) return cudaErrorInvalidConfiguration;
  a.p_stages = p_stages;
  a.w_stages = w_stages;
  const size_t smem = fixed + p_stages * p_stage + (size_t)w_stages * a.w_bytes;
  a.list_cap = (int)((smem - 1024) / 16);  // after the 1024-byte alignment
  err = cudaFuncSetAttribute(update_persistent_kernel<NCOLS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
  if (err != cudaSuccess) return err;
  const int nsm = num_sms();
  for (int base = 0; base < n; base += kMaxUpd) {
    const int m = (n - base) < kMaxUpd ? (n - base) : kMaxUpd;
    a.n = m;
    int64_t total_tiles = 0;
    for (int i = 0; i < m; ++i)
      total_tiles += ceil_div(probs[base + i].d, 128) * ceil_div(probs[base + i].k, NCOLS);
    // about twelve units per CTA, at least four tiles per unit so the C row
    // block is reused; CTAs then get contiguous unit ranges of equal tile count
    int64_t ut = total_tiles / (12 * (int64_t)nsm);
    if (ut < 4) ut = 4;
    if (ut > 64) ut = 64;
    a.unit_tiles = (int)ut;
    a.unit_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      const UpdateWorkspace& w = ws[base + i];
      err = make_tmap_bf16_2d(&a.tm_c[i], w.c_split, (uint64_t)2 * r_pad, (uint64_t)pr.d, (uint64_t)r_pad * 4, 64, 128);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tm_p[i], w.p_split, (uint64_t)2 * r_pad, (uint64_t)pr.k, (uint64_t)r_pad * 4, 64, NCOLS);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tm_w[i], pr.W, (uint64_t)pr.k, (uint64_t)pr.d, (uint64_t)pr.ld_w * 2, 64, 128);
      if (err != cudaSuccess) return err;
      a.W[i] = pr.W;
      a.ld_w[i] = pr.ld_w;
      a.C[i] = pr.C;
      a.P[i] = pr.P;
      a.c_norm[i] = w.c_norm;
      a.p_norm[i] = w.p_norm;
      a.d[i] = pr.d;
      a.k[i] = pr.k;
      a.n_ct[i] = (int)ceil_div(pr.k, NCOLS);
      a.n_cu[i] = (int)ceil_div(a.n_ct[i], a.unit_tiles);
      a.unit_begin[i + 1] = a.unit_begin[i] + a.n_cu[i] * (int)ceil_div(pr.d, 128);
      a.layer[i] = pr.layer;
      a.scale_dev[i] = normsgd ? w.scale : nullptr;
      a.status_in[i] = normsgd ? (pr.dev_status ? pr.dev_status : w.status) : nullptr;
      a.status_out[i] = normsgd ? nullptr : pr.dev_status;
      a.unit_partials[i] = w.wnew_partials;
      a.flags[i] = w.flags;
      a.ticket[i] = w.ticket;
      a.wnorm2_out[i] = normsgd ? pr.wnorm2_out : nullptr;
    }
    const int units = a.unit_begin[m];
    int grid = units < nsm ? units : nsm;
    if (grid > kMaxCtas) grid = kMaxCtas;
    {
      // split the units into `grid` contiguous ranges of about equal tile count
      int64_t tile_total = 0;
      for (int i = 0; i < m; ++i) tile_total += (int64_t)a.n_ct[i] * ceil_div(probs[base + i].d, 128);
      int cta = 0;
      int64_t acc = 0;
      a.cta_unit_begin[0] = 0;
      int u = 0;
      for (int i = 0; i < m; ++i) {
        const int nrb = (int)ceil_div(probs[base + i].d, 128);
        for (int rb = 0; rb < nrb; ++rb) {
          for (int cu = 0; cu < a.n_cu[i]; ++cu, ++u) {
            const int t0 = cu * a.unit_tiles;
            const int t1 = (t0 + a.unit_tiles < a.n_ct[i]) ? t0 + a.unit_tiles : a.n_ct[i];
            acc += t1 - t0;
            // close CTA ranges whose share of tiles is reached
            while (cta + 1 < grid && acc * grid >= tile_total * (cta + 1)) a.cta_unit_begin[++cta] = u + 1;
          }
        }
      }
      while (cta + 1 <= grid) a.cta_unit_begin[++cta] = units;
    }
    count_launch();
    update_persistent_kernel<NCOLS><<<grid, kUpdThreads, smem, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_split(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, cudaStream_t stream) {
  static thread_local SplitBatch sb;
  const int r_pad = round16(r);
  sb.r = r;
  sb.r_pad = r_pad;
  for (int base = 0; base < n; base += kMaxAux) {
    const int m = (n - base) < kMaxAux ? (n - base) : kMaxAux;
    sb.n = 2 * m;
    sb.row_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      sb.src[2 * i] = pr.C;
      sb.dst[2 * i] = ws[base + i].c_split;
      sb.norm[2 * i] = ws[base + i].c_norm;
      sb.row_begin[2 * i + 1] = sb.row_begin[2 * i] + pr.d;
      sb.src[2 * i + 1] = pr.P;
      sb.dst[2 * i + 1] = ws[base + i].p_split;
      sb.norm[2 * i + 1] = ws[base + i].p_norm;
      sb.row_begin[2 * i + 2] = sb.row_begin[2 * i + 1] + pr.k;
    }
    const int64_t blocks = ceil_div(sb.row_begin[2 * m], 8);
    const int grid = (int)(blocks < 8 * (int64_t)num_sms() ? blocks : 8 * (int64_t)num_sms());
    count_launch();
    split_rows_kernel<<<grid, 256, 0, stream>>>(sb);
  }
  return cudaGetLastError();
}

cudaError_t launch_update(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, bool normsgd,
                          float scale_val, uint64_t seed, uint32_t step, cudaStream_t stream) {
  cudaError_t err = launch_split(n, probs, ws, r, stream);
  if (err != cudaSuccess) return err;
  if (update_ncols(r) == 128)
    return launch_update_tc<128>(n, probs, ws, r, normsgd, scale_val, seed, step, stream);
  return launch_update_tc<64>(n, probs, ws, r, normsgd, scale_val, seed, step, stream);
}

}  // namespace

int64_t flag_words(int64_t d, int64_t k, int r) {
  const int ncols = update_ncols(r);
  return ceil_div(d, 128) * ceil_div(k, ncols) * (16 * ncols / 32);
}

size_t carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd, UpdateWorkspace* ws) {
  const size_t start = cur.offset;
  UpdateWorkspace w{};
  const int r_pad = round16(r);
  if (normsgd) {
    w.gram_partials_p = cur.take<float2>((size_t)gram_chunks(k).nchunks * r * r);
    w.gram_partials_c = cur.take<float2>((size_t)gram_chunks(d).nchunks * r * r);
    w.gram_p = cur.take<double>((size_t)r * r);
    w.gram_c = cur.take<double>((size_t)r * r);
    w.wnorm_partials = cur.take<double>(kWnormBlocks);
    w.scale = cur.take<float>(1);
    w.status = cur.take<int32_t>(1);
    w.ticket = cur.take<uint32_t>(1);
    w.wnew_partials = cur.take<double>((size_t)ceil_div(d, 128) * ceil_div(k, 64));
  }
  w.c_norm = cur.take<float>((size_t)d);
  w.p_norm = cur.take<float>((size_t)k);
  w.c_split = cur.take<uint16_t>((size_t)d * 2 * r_pad);
  w.p_split = cur.take<uint16_t>((size_t)k * 2 * r_pad);
  w.flags = cur.take<uint32_t>((size_t)flag_words(d, k, r));
  cur.take<char>(0);  // end on a 256-byte boundary
  if (ws) *ws = w;
  return cur.offset - start;
}

cudaError_t launch_update_normsgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float tau,
                                  uint64_t seed, uint32_t step, cudaStream_t stream) {
  static thread_local WnormBatch wb;
  static thread_local GramBatch gb;
  static thread_local FinalizeBatch fb;
  cudaError_t err = cudaSuccess;
  for (int base = 0; base < n; base += kMaxAux) {
    const int m = (n - base) < kMaxAux ? (n - base) : kMaxAux;
    int nw = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      if (pr.wnorm2_in != nullptr) continue;
      wb.W[nw] = pr.W;
      wb.d[nw] = pr.d;
      wb.k[nw] = pr.k;
      wb.ld[nw] = pr.ld_w;
      wb.partials[nw] = ws[base + i].wnorm_partials;
      ++nw;
    }
    if (nw > 0) {
      count_launch();
      wnorm_partial_kernel<<<dim3(kWnormBlocks, nw), 256, 0, stream>>>(wb);
    }
    gb.n = 2 * m;
    gb.r = r;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      const UpdateWorkspace& w = ws[base + i];
      gb.e[2 * i] = GramEntry{pr.P, pr.k, w.gram_partials_p, w.gram_p};
      gb.e[2 * i + 1] = GramEntry{pr.C, pr.d, w.gram_partials_c, w.gram_c};
      fb.wnorm_partials[i] = w.wnorm_partials;
      fb.wnorm2_in[i] = pr.wnorm2_in;
      fb.gram_p[i] = w.gram_p;
      fb.gram_c[i] = w.gram_c;
      fb.scale[i] = w.scale;
      fb.status[i] = pr.dev_status ? pr.dev_status : w.status;
      fb.ticket[i] = w.ticket;
      fb.wnorm2_out[i] = pr.wnorm2_out;
    }
    err = launch_gram(gb, stream);
    if (err != cudaSuccess) return err;
    fb.rr = r * r;
    fb.tau = tau;
    count_launch();
    normsgd_finalize_kernel<<<m, 256, 0, stream>>>(fb);
  }
  return launch_update(n, probs, ws, r, true, 0.f, seed, step, stream);
}

cudaError_t launch_update_sgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float alpha_eta,
                              uint64_t seed, uint32_t step, cudaStream_t stream) {
  return launch_update(n, probs, ws, r, false, alpha_eta, seed, step, stream);
}

}  // namespace rgs
