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

// ---- FP16 high/low split of C and P, and their row norms --------------------
// The tensor cores take C and P as two FP16 parts each, scaled by powers of two
// so that every part is a normal FP16 number: each row of C by its own 2^e
// (largest |c| in [2^14, 2^15)), P by one 2^f per block of 128 rows (the
// columns of W one update tile covers).  Then x = hi + lo to about 2^-22
// relative and the products the MMAs drop (lo lo) are below 2^-22 of the terms.
// The epilogue undoes the scale exactly: H = acc 2^-e 2^-f.
constexpr int kSplitRows = 128;  // rows per split block (P: one scale per block)

struct SplitBatch {
  const float* src[2 * kMaxAux];          // entry 2i: C of layer i; 2i + 1: its P
  int64_t rows[2 * kMaxAux];
  int64_t block_begin[2 * kMaxAux + 1];   // prefix of the entries' 128-row block counts
  uint16_t* dst[2 * kMaxAux];     // rows x 2 r_pad FP16 bits: [hi | lo] of the scaled row
  float* norm[2 * kMaxAux];       // rows: Euclidean norm of each source row
  float* unscale[2 * kMaxAux];    // C: 2^-e per row; P: 2^-f per 128-row block; NaN: no usable scale
  int n;
  int r;
  int r_pad;
  // each layer's exact-path counters, reset here before the update
  uint32_t* fix_ticket[kMaxAux];
  unsigned long long* fix_acc[kMaxAux];
};

// Exponent e that brings a largest magnitude m into [2^14, 2^15) (0 for m = 0);
// false when m is not finite or e falls outside [-100, 100], where the scaled
// parts or the unscaled products could leave the normal fp32 range.
__device__ __forceinline__ bool split_exponent(float m, int& e) {
  if (m == 0.f) {
    e = 0;
    return true;
  }
  if (!(m <= 3.4028234e38f)) {  // inf or NaN
    e = 0;
    return false;
  }
  int E;
  frexpf(m, &E);  // m = f 2^E, f in [0.5, 1)
  e = 15 - E;
  if (e < -100 || e > 100) {
    e = e < -100 ? -100 : 100;
    return false;
  }
  return true;
}

// One block of 256 threads per 128 rows of an entry (grid over all entries'
// blocks).  A row takes lpr lanes (r_pad / 16 rounded up to a power of two, at
// least 2 and at most 32), lane c its columns 4c..4c+3 of each of up to four 4 lpr-column
// steps, so that a lane converts up to 16 values per row and the row's lanes
// combine their sums and maxima in few shuffles; warp w takes rows
// 16w..16w+15.  Largest magnitudes are taken as integer maxima of the
// magnitude bits (a NaN's exceed +inf's, so a NaN wins).  For P the block's
// largest |p| is found first (the rows are read twice; the second read comes
// from L2).
__global__ void __launch_bounds__(256) split_fp16_kernel(const __grid_constant__ SplitBatch b) {
  __shared__ float wmax[8];
  __shared__ int blk_e;
  __shared__ bool blk_ok;
  if (blockIdx.x == 0) {
    for (int t = threadIdx.x; t < b.n / 2; t += blockDim.x) {
      *b.fix_ticket[t] = 0u;
      *b.fix_acc[t] = 0ull;
    }
  }
  // the entry of this block, by bisection of the block prefix
  int en = 0;
  {
    int hi = b.n - 1;
    while (en < hi) {
      const int mid = (en + hi + 1) >> 1;
      if (b.block_begin[mid] <= (int64_t)blockIdx.x) en = mid;
      else hi = mid - 1;
    }
  }
  const bool is_p = en & 1;
  const int64_t rows = b.rows[en];
  const int64_t row0 = ((int64_t)blockIdx.x - b.block_begin[en]) * kSplitRows;
  const float* __restrict__ src = b.src[en];
  const int r = b.r, r_pad = b.r_pad;
  const bool vec = (r & 3) == 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int lpr = 2;  // at least two, so that a warp step covers at most its 16 rows
  while (lpr < 32 && 16 * lpr < r_pad) lpr <<= 1;
  const int rps = 32 / lpr, sub = lane / lpr, cl = lane % lpr;
  const int nq = (r_pad + 4 * lpr - 1) / (4 * lpr);  // column steps: up to 4 (r_pad <= 512)
  auto load4 = [&](int64_t row, int c0, float (&v)[4]) {
    const float* s4 = src + row * r + c0;
    if (vec && c0 < r) {
      const float4 f = *reinterpret_cast<const float4*>(s4);
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    } else {
#pragma unroll
      for (int t = 0; t < 4; ++t) v[t] = (c0 + t < r) ? s4[t] : 0.f;
    }
  };
  if (is_p) {
    uint32_t mb = 0u;
    for (int st = 0; st < 16 / rps; ++st) {
      const int64_t row = row0 + warp * 16 + st * rps + sub;
      if (row >= rows) continue;
      for (int q = 0; q < nq; ++q) {
        float v[4];
        load4(row, 4 * cl + 4 * lpr * q, v);
#pragma unroll
        for (int t = 0; t < 4; ++t) mb = max(mb, __float_as_uint(v[t]) & 0x7FFFFFFFu);
      }
    }
    mb = __reduce_max_sync(0xFFFFFFFFu, mb);
    if (lane == 0) wmax[warp] = __uint_as_float(mb);
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t bb = 0u;
      for (int w = 0; w < 8; ++w) bb = max(bb, __float_as_uint(wmax[w]));
      const float bm = __uint_as_float(bb);
      int e;
      blk_ok = split_exponent(bm, e);
      blk_e = e;
      b.unscale[en][row0 / kSplitRows] = blk_ok ? ldexpf(1.f, -e) : __int_as_float(0x7FC00000);
    }
    __syncthreads();
  }
  for (int st = 0; st < 16 / rps; ++st) {
    const int64_t row = row0 + warp * 16 + st * rps + sub;
    const bool in = row < rows;
    float v[4][4];
    float sq = 0.f;
    uint32_t mb = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int t = 0; t < 4; ++t) v[q][t] = 0.f;
      if (in && q < nq) load4(row, 4 * cl + 4 * lpr * q, v[q]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        sq = fmaf(v[q][t], v[q][t], sq);
        mb = max(mb, __float_as_uint(v[q][t]) & 0x7FFFFFFFu);
      }
    // the row's lanes combine their squares and maxima (groups of lpr lanes)
    for (int o = lpr >> 1; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
      mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
    }
    const float m = __uint_as_float(mb);
    int e;
    bool ok;
    if (is_p) {
      e = blk_e;
      ok = blk_ok;
    } else {
      ok = split_exponent(m, e);
    }
    if (!in) continue;
    if (cl == 0) {
      b.norm[en][row] = sqrtf(sq);
      if (!is_p) b.unscale[en][row] = ok ? ldexpf(1.f, -e) : __int_as_float(0x7FC00000);
    }
    const float sc = ldexpf(1.f, e);
    uint16_t* dst = b.dst[en] + row * 2 * r_pad;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q >= nq) break;
      const int c0 = 4 * cl + 4 * lpr * q;
      if (c0 >= r_pad) continue;  // lanes past the padded row (r_pad not a multiple of 4 lpr)
      uint32_t hi2[2], lo2[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) hi2[t] = tc::split_f16x2(v[q][2 * t], v[q][2 * t + 1], sc, lo2[t]);
      // r_pad is a multiple of 16: the 4 columns are inside the row, 8-byte aligned
      *reinterpret_cast<uint2*>(dst + c0) = make_uint2(hi2[0], hi2[1]);
      *reinterpret_cast<uint2*>(dst + r_pad + c0) = make_uint2(lo2[0], lo2[1]);
    }
  }
}

// ---- the rebuild + update kernel -------------------------------------------------
// Work of a launch: up to kMaxUpd layers.  Layer p is cut into units of
// (128-row block, run of up to ut[p] column tiles of NCOLS); units of all
// layers are numbered end to end.  Each persistent CTA takes either a
// contiguous range of them, of about equal tile count, or (interleave) every
// G-th one: then the units in flight at once are neighbouring row blocks of
// the same layers, whose P tiles come from L2 rather than HBM.
struct UpdBatch {
  CUtensorMap tm_c[kMaxUpd];   // C split, d x (2 r_pad) FP16: [hi | lo] of each row scaled by 2^e
  CUtensorMap tm_p[kMaxUpd];   // P split, k x (2 r_pad) FP16, 2^f per 128 rows
  CUtensorMap tm_w[kMaxUpd];   // W, d x k BF16 (tile loads and stores)
  const float* C[kMaxUpd];     // fp32 C and P for the exact recomputation
  const float* P[kMaxUpd];
  const float* c_norm[kMaxUpd];
  const float* p_norm[kMaxUpd];
  const float* c_unscale[kMaxUpd];   // 2^-e of each row of the C split
  const float* p_unscale[kMaxUpd];   // 2^-f of each 128-row block of the P split
  int64_t d[kMaxUpd], k[kMaxUpd];
  int n_ct[kMaxUpd];           // column tiles of the layer
  int n_cu[kMaxUpd];           // units per row block
  int ut[kMaxUpd];             // column tiles per unit
  int unit_begin[kMaxUpd + 1];
  uint32_t layer[kMaxUpd];
  const float* scale_dev[kMaxUpd];     // normalized SGD: s on the device; NULL: scale_val
  const int32_t* status_in[kMaxUpd];   // skip the layer when nonzero
  int32_t* status_out[kMaxUpd];        // SGD: set to 0
  double* unit_partials[kMaxUpd];      // ||W_new||^2 of each unit
  uint32_t* ticket[kMaxUpd];
  double* wnorm2_out[kMaxUpd];
  int n;
  int interleave;     // 1: CTA b takes units b, b + G, ... below the last; 0: a range
  int u_step;         // G when interleaved, else 1
  int cta_first[kMaxCtas], cta_end[kMaxCtas];  // CTA b's units: cta_first[b], + u_step, ... < cta_end[b]
  int p_stages;       // P ring depth
  int w_stages;       // W ring depth
  float scale_val;
  float err_coef;     // 2^25 (beta + 2^-24): the margin bound is err_coef |s| ||c_i|| max_j ||p_j||
  uint32_t rk0[10], rk1[10];  // Philox round keys of the seed
  uint32_t step;
  int r;
  int r_pad;          // r rounded up to 16 (MMA K extent)
  int parts;          // FP16 parts of C and P: 2 (three products)
  int kchunks;        // 64-wide chunks of r_pad
  uint32_t a_bytes;   // bytes of one part of the C row block: kchunks x 16 KB
  uint32_t b_bytes;   // bytes of one part of one 64-wide chunk of a P tile: NCOLS x 128
  uint32_t w_bytes;   // bytes of the W tile: NCOLS/64 x 16 KB
  int* err;
  unsigned long long* exact_count;  // elements recomputed exactly (instrumentation)
  uint16_t* fix_tags[kMaxUpd];      // exact-path tags of each layer: kFixCap per (tile, warp)
  uint8_t* fix_counts[kMaxUpd];     // tags written per (tile, warp)
};

// kernel parameters are limited to 32764 bytes
static_assert(sizeof(UpdBatch) <= 32764, "UpdBatch exceeds the kernel parameter limit");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int kStoreWarps = 2;                    // tiles alternate between them: two stores drain at once
constexpr int kCtlWarps = 2 + kStoreWarps;        // producer, MMA issuer, store warps
constexpr int kEpiWarps = 16;                     // warps 4..19: four per TMEM lane quarter
constexpr int kUpdThreads = (kCtlWarps + kEpiWarps) * 32;
constexpr int kMaxStagesUpd = 8;
constexpr int kTmemBufs = 4;                      // accumulator tiles in flight
constexpr int kNormSlots = 8;                     // units whose ||W_new||^2 partials may be open at once

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
  x.ct0 = cu * a.ut[p];
  x.ct1 = min(a.n_ct[p], x.ct0 + a.ut[p]);
  return x;
}

// Packed pair of fp32 fused multiply-adds (one instruction for two lanes of
// work; each half rounds exactly like fmaf).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Rounding margin of one element, in units of the error bound.  S = bits(v) +
// rand16 is the stochastic-rounding sum (the result is S >> 16); L = S mod
// 2^16 lies min(L, 2^16 - L) fp32 steps of v from the nearest sum that would
// round the other way.  A value v' within D of v is at most 2D / ulp(v) + 2
// fp32 steps from v (the step halves below a power of two; both values are
// rounded once), and ulp(v) > |v| 2^-24, so v' rounds like v whenever
// (min(L, 2^16 - L) - 3) |v| >= 2^25 D.  Returns the left side (less a
// little more, for the rounding of this product): negative when the margin
// is three steps or less, NaN when v is NaN or infinite.
__device__ __forceinline__ float rounding_margin(uint32_t S, float v) {
  const float mg = __uint_as_float(__byte_perm(S, 0x4B000000u, 0x7610));  // 2^23 + (S mod 2^16)
  const float x = mg - 8421376.0f;                                        // (S mod 2^16) - 2^15, exact
  const float av = fabsf(v);
  return fmaf(-fabsf(x), av, 32764.0f * av);  // (min(L, 2^16 - L) - 4) |v|, rounded
}

template <int N>
__device__ __forceinline__ uint32_t pick(const uint32_t (&v)[N], int i) {
  uint32_t r = v[0];
#pragma unroll
  for (int t = 1; t < N; ++t) r = (i == t) ? v[t] : r;
  return r;
}

// Exact-path tags: an element whose rounding margin the error bound might
// cross keeps its original weight in W, and its lane's 8-column group gets a
// 16-bit tag: the flagged elements as bits 0..7 (bit t: column 8g + t of the
// warp's columns), the lane at bits 8..12, the group g at bits 13..15.  Each
// (tile, epilogue warp) owns room for a tag per group of the tile and a count
// byte; every other element of W holds the tensor-core result.
constexpr int kFixCap = 128;  // 32 lanes x up to 4 groups

// Byte offset in a W stage (NCOLS/64 boxes of 64 columns, 128-byte swizzled)
// of the 8-column group of tile row q that starts at column col.
__device__ __forceinline__ uint32_t w_stage_offset(int col, int q) {
  return (uint32_t)((col >> 6) * 16384 + q * 128 + ((((col & 63) >> 3) ^ (q & 7)) << 4));
}

// Persistent rebuild + update, one CTA per SM, each CTA a contiguous range of
// units (a unit: one 128-row block of one layer and up to unit_tiles column
// tiles of NCOLS).  Warp 0 (one lane) streams with TMA the FP16 parts of the C
// row block of each unit, the same parts of the P rows of each column tile
// into a P ring, and the W tile into a deeper W ring.  Warp 1 (one lane)
// issues the scaled H = sum of the part products hi hi + hi lo + lo hi
// (tcgen05.mma kind::f16, M=128, N=NCOLS) into one of four TMEM buffers and
// frees the P stage with tcgen05.commit.  The 16 epilogue warps
// (warps 4..19, four per TMEM lane quarter, one column quarter each) read H
// from TMEM, form v = fmaf(-s, H, w) with w from the W stage (the split's
// scales folded into s), round it
// stochastically with 16 Philox bits per weight and write the BF16 results
// back into the stage; warps 2 and 3 (one lane each, alternate tiles) write
// each finished tile to W with a TMA tensor store and free the stage.
//
// Exactness.  The definition rounds v = fmaf(-s, fl32(H), w) with fl32(H) the
// fp32 rounding of the exact product.  The tensor-core H differs from it by at
// most D = |s| (beta ||c_i|| ||p_j|| + 2^-24 |H|) with beta the split and
// accumulation error of the part products.  Each element's rounding margin
// (rounding_margin) is compared with that bound.  An element whose margin
// might be crossed keeps its original weight in W and its group is tagged
// for the fix kernel; exact_fix_kernel then recomputes those elements, H_ij from a
// compensated dot product of the fp32 row of C and the fp32 row of P (Dot2 of
// the paper above: as accurate as twice fp32 precision), and writes their
// results.  Every other element's result is the one the definition gives.
// The kernel itself holds no exact-path arithmetic, which keeps its register
// allocation to the streaming loop.
template <int NCOLS>
__global__ void __launch_bounds__(kUpdThreads, 1) update_persistent_kernel(const __grid_constant__ UpdBatch a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t pfull_bar[kMaxStagesUpd], pempty_bar[kMaxStagesUpd];
  __shared__ __align__(8) uint64_t wfull_bar[kMaxStagesUpd], wempty_bar[kMaxStagesUpd], sfull_bar[kMaxStagesUpd];
  __shared__ __align__(8) uint64_t cfull_bar, cempty_bar, tfull_bar[kTmemBufs], tempty_bar[kTmemBufs];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ uint32_t skip_mask[(kMaxUpd + 31) / 32];  // layers whose status_in is nonzero
  __shared__ double norm_slot[kNormSlots][kEpiWarps];  // ||W_new||^2 of each epilogue warp per open unit
  __shared__ int norm_count[kNormSlots];

  uint8_t* smem = align1024(smem_raw);
  uint8_t* s_c = smem;                                             // C row block: parts x a_bytes
  uint8_t* s_p0 = s_c + (size_t)a.parts * a.a_bytes;               // P ring: NSP x parts x b_bytes
  uint8_t* s_w0 = s_p0 + (size_t)a.p_stages * a.parts * a.b_bytes;  // W ring: NSW x W tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NSP = a.p_stages, NSW = a.w_stages;
  // this CTA's units: u_first, u_first + u_step, ... below u_total
  const int u_first = a.cta_first[blockIdx.x], u_step = a.u_step, u_total = a.cta_end[blockIdx.x];
  constexpr uint32_t kTmemCols = kTmemBufs * NCOLS;

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
    for (int b = 0; b < kTmemBufs; ++b) {
      tc::mbar_init(&tfull_bar[b], 1);
      tc::mbar_init(&tempty_bar[b], kEpiWarps);
    }
    for (int s = 0; s < kNormSlots; ++s) norm_count[s] = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, kTmemCols);
  if (warp == 2) {
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
    int sw = 0, sp = 0, ip = 0;     // W stage of tile it, P stage of chunk ip (kept without divisions)
    uint32_t wph = 0, pph = 0;      // their phases
    bool stop = false;
    for (int u = u_first; u < u_total && !stop; u += u_step) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      const int i0 = x.rb * 128;
      if (x.p != prev_p || x.rb != prev_rb) {
        if (cl > 0 && !tc::mbar_wait(&cempty_bar, (cl - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) break;
        tc::mbar_arrive_expect_tx(&cfull_bar, a.parts * a.a_bytes);
        for (int q2 = 0; q2 < a.parts; ++q2)
          for (int c = 0; c < a.kchunks; ++c)
            tc::tma_load_2d(s_c + q2 * a.a_bytes + c * 16384, &a.tm_c[x.p], &cfull_bar, q2 * a.r_pad + c * 64, i0);
        ++cl;
        prev_p = x.p;
        prev_rb = x.rb;
      }
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int j0 = ct * NCOLS;
        // W tile first: it comes from HBM and is waited on longest
        if (it >= NSW && !tc::mbar_wait(&wempty_bar[sw], wph ^ 1u, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        uint8_t* wst = s_w0 + (size_t)sw * a.w_bytes;
        tc::mbar_arrive_expect_tx(&wfull_bar[sw], a.w_bytes);
#pragma unroll
        for (int bx = 0; bx < NCOLS / 64; ++bx)
          tc::tma_load_2d(wst + bx * 16384, &a.tm_w[x.p], &wfull_bar[sw], j0 + 64 * bx, i0);
        // P: one stage per 64-wide chunk of r (both parts), so that wide
        // ranks keep two or more chunks in flight
        for (int c = 0; c < a.kchunks && !stop; ++c, ++ip) {
          if (ip >= NSP && !tc::mbar_wait(&pempty_bar[sp], pph ^ 1u, &abort_flag, a.err, tc::kErrTimeoutStage)) {
            stop = true;
            break;
          }
          uint8_t* pst = s_p0 + (size_t)sp * a.parts * a.b_bytes;
          tc::mbar_arrive_expect_tx(&pfull_bar[sp], a.parts * a.b_bytes);
          for (int q2 = 0; q2 < a.parts; ++q2)
            tc::tma_load_2d(pst + q2 * a.b_bytes, &a.tm_p[x.p], &pfull_bar[sp], q2 * a.r_pad + c * 64, j0);
          if (++sp == NSP) {
            sp = 0;
            pph ^= 1u;
          }
        }
        if (stop) break;
        if (++sw == NSW) {
          sw = 0;
          wph ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = tc::idesc_f16(128, NCOLS, false, false);
    int it = 0, cl = 0, prev_p = -1, prev_rb = -1;
    int sp = 0;        // P stage of the next chunk and its phase, as in the producer
    uint32_t pph = 0;
    bool stop = false;
    for (int u = u_first; u < u_total && !stop; u += u_step) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      if (x.p != prev_p || x.rb != prev_rb) {
        if (!tc::mbar_wait(&cfull_bar, cl & 1, &abort_flag, a.err, tc::kErrTimeoutLoad)) break;
        ++cl;
        prev_p = x.p;
        prev_rb = x.rb;
      }
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int b = it % kTmemBufs;
        if (it >= kTmemBufs &&
            !tc::mbar_wait(&tempty_bar[b], ((it / kTmemBufs) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage)) {
          stop = true;
          break;
        }
        const uint32_t sc = tc::smem_u32(s_c);
        const uint32_t d_tmem = tmem + (uint32_t)(b * NCOLS);
        // the products of the parts above ~2^-22 of the terms: hi*hi, hi*lo,
        // lo*hi (lo*lo is dropped)
        constexpr int kPairA[3] = {0, 0, 1}, kPairB[3] = {0, 1, 0};
        uint32_t acc = 0;
        for (int c = 0; c < a.kchunks; ++c) {
          if (!tc::mbar_wait(&pfull_bar[sp], pph, &abort_flag, a.err, tc::kErrTimeoutLoad)) {
            stop = true;
            break;
          }
          tc::tc_fence_after();
          const uint32_t pst = tc::smem_u32(s_p0 + (size_t)sp * a.parts * a.b_bytes);
          for (int kk = 0; kk < 4 && c * 64 + kk * 16 < a.r_pad; ++kk) {
            const uint32_t off_a = c * 16384 + kk * 32, off_b = kk * 32;
#pragma unroll
            for (int pr = 0; pr < 3; ++pr) {
              const uint64_t ad = tc::sdesc_sw128(sc + kPairA[pr] * a.a_bytes + off_a, 16, 1024);
              const uint64_t bd = tc::sdesc_sw128(pst + kPairB[pr] * a.b_bytes + off_b, 16, 1024);
              tc::mma_bf16(d_tmem, ad, bd, idesc, acc);
              acc = 1u;
            }
          }
          tc::mma_commit(&pempty_bar[sp]);
          if (++sp == NSP) {
            sp = 0;
            pph ^= 1u;
          }
        }
        if (stop) break;
        tc::mma_commit(&tfull_bar[b]);
      }
      // release the C row block once its last unit is issued
      bool last_of_c = (u + u_step >= u_total);
      if (!last_of_c) {
        const Unit y = decode_unit(a, u + u_step);
        last_of_c = (y.p != x.p || y.rb != x.rb);
      }
      if (last_of_c && !stop) tc::mma_commit(&cempty_bar);
    }
  } else if (warp >= 2 && warp < kCtlWarps && lane == 0) {
    // ---------------- store warps ----------------
    // Store warp w writes tiles w - 2, w - 2 + kStoreWarps, ... from their W
    // stages to W with TMA, and frees each stage once the copy has read it;
    // the store warps' copies drain side by side.
    int it = 0;
    bool stop = false;
    const int mine = warp - 2;
    for (int u = u_first; u < u_total && !stop; u += u_step) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(x.p)) continue;
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        if (it % kStoreWarps != mine) continue;
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
  } else if (warp >= kCtlWarps) {
    // ---------------- epilogue ----------------
    // warp w may read TMEM lanes 32 (w % 4) .. +31 only: the sixteen warps
    // cover each lane quarter four times, one column quarter each
    const int ew = warp - kCtlWarps;
    const int quarter = warp & 3;
    constexpr int kCols = NCOLS / 4;           // columns per thread per tile (one pass)
    constexpr int kGroups = kCols / 8;         // 8-column groups (Philox blocks) per tile
    static_assert(kCols == 16 || kCols == 32, "16 or 32 columns per thread");
    const int col_base = (ew >> 2) * kCols;    // column quarter of the tile
    const int q = quarter * 32 + lane;         // tile row = TMEM lane
    // byte offset in a W stage (NCOLS/64 boxes of 64 columns, 128-byte
    // swizzled) of this thread's 8-column groups: row q, column col_base + 8g
    uint32_t stage_off[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      stage_off[g] = w_stage_offset(col_base + 8 * g, q);
    }
    int it = 0;
    int sw = 0;        // W stage of tile it: it % NSW, kept without a division
    uint32_t wph = 0;  // its phase, (it / NSW) & 1
    int un = 0;  // this CTA's units so far (the norm slot)
    for (int u = u_first; u < u_total; u += u_step, ++un) {
      const Unit x = decode_unit(a, u);
      const int p = x.p;
      if (layer_skipped(p)) continue;
      // d, k < 2^31 and d*k/8 < 2^32 (checked on the host): 32-bit indices
      const int d = (int)a.d[p], k = (int)a.k[p];
      const int i = x.rb * 128 + q;
      const uint32_t k8 = (uint32_t)k >> 3;
      const bool row_ok = i < d;
      const float s = a.scale_dev[p] ? *a.scale_dev[p] : a.scale_val;
      const float bound_row = row_ok ? a.err_coef * fabsf(s) * a.c_norm[p][i] : 0.f;
      // the tensor cores return H scaled by this row's 2^e and the tile's 2^f
      const float s_row = row_ok ? s * a.c_unscale[p][i] : 0.f;
      const uint32_t layer = a.layer[p];
      const bool need_norm = a.wnorm2_out[p] != nullptr;
      float sq = 0.f, sq_comp = 0.f;  // Kahan-compensated sum of squares

      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int b = it % kTmemBufs;
        const int j0 = ct * NCOLS;
        // largest norm of the P rows of this warp's columns (for the margin
        // bound), loaded before the waits so that its latency hides behind them
        float pmax = 0.f;
        {
          const int jc = j0 + col_base + (lane % kCols);
          if (jc < k) pmax = a.p_norm[p][jc];
        }
        const float p_un = a.p_unscale[p][j0 / kSplitRows];
        // the Philox words of this warp's groups: element index e = i*k + j
        // (j a multiple of 8) gives block e / 8.  They need no tile data, so
        // they are formed before the waits, the groups' chains interleaved.
        uint32_t rw[kGroups][4];
        {
          uint32_t blks[kGroups];
#pragma unroll
          for (int g = 0; g < kGroups; ++g) blks[g] = (uint32_t)i * k8 + ((uint32_t)(j0 + col_base + 8 * g) >> 3);
          philox4x32_10_rk_multi<kGroups>(blks, a.step, layer, kTagSR, a.rk0, a.rk1, rw);
        }
        bool live = tc::mbar_wait(&wfull_bar[sw], wph, &abort_flag, a.err, tc::kErrTimeoutLoad) &&
                    tc::mbar_wait(&tfull_bar[b], (it / kTmemBufs) & 1, &abort_flag, a.err, tc::kErrTimeoutMma);
        live = __all_sync(0xFFFFFFFFu, live);
        tc::tc_fence_after();
        const uint32_t s_w32 = tc::smem_u32(s_w0) + (uint32_t)sw * a.w_bytes;
        for (int o = 16; o > 0; o >>= 1) pmax = fmaxf(pmax, __shfl_xor_sync(0xFFFFFFFFu, pmax, o));
        // v = fmaf(-s, H, w) as fmaf(-s_t, acc, w) with s_t = s 2^-e 2^-f, the
        // same number when s_t is a normal float (s = 0 gives v = w either
        // way); otherwise, or when a scale is missing (NaN), the bound is NaN
        // and every element of the tile takes the exact path
        const float s_t = s_row * p_un;
        const bool scaled_ok = s == 0.f || (fabsf(s_t) >= 0x1p-126f && fabsf(s_t) <= 3.4028234e38f);
        const float bound = scaled_ok ? bound_row * pmax : __int_as_float(0x7FC00000);  // 2^25 D
        const float2 ns2 = make_float2(-s_t, -s_t);
        // live is the same in the whole warp: one branch per tile
        // this warp's entry of the layer's exact-path map for this tile
        const size_t set = ((size_t)x.rb * (size_t)a.n_ct[p] + (size_t)ct) * kEpiWarps + ew;
        uint32_t fmap = 0;   // this lane's flagged elements, a byte per group
        uint32_t nflag = 0;  // the warp's flagged groups (warp-uniform)
        if (live) {
          const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * NCOLS + col_base);
          float gs = 0.f;  // sum of squares of this tile's results (normalized SGD)
          // 16 columns (two 8-column groups) at a time: their H from TMEM
#pragma unroll
          for (int hf = 0; hf < kGroups / 2; ++hf) {
            uint32_t h[16];
            tc::tmem_ld_32x32b<16>(taddr + 16 * hf, h);
            tc::tmem_wait_ld_regs<16>(h);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
              const int g = 2 * hf + gg;
              const int col = col_base + 8 * g;
              const uint32_t sp = s_w32 + stage_off[g];
              const uint4 raw = tc::lds128(sp);
              const uint32_t win[4] = {raw.x, raw.y, raw.z, raw.w};
              uint32_t wout[4];
              float ym[8];
              // Per pair: v = fmaf(-s, H, w) (one packed FMA) and stochastic
              // rounding (add 16 random bits below the BF16 mantissa, keep the
              // upper halves: one PRMT per pair); the results go back into the
              // W stage in place (the store warp writes the tile out with TMA,
              // clipping rows and columns outside W).  The integer steps use
              // multiply-adds so that they share the multiplier pipe with
              // Philox instead of crowding the ALU pipe: r_hi = r >> 16,
              // r_lo = r - r_hi * 2^16 = r & 0xFFFF.
#pragma unroll
              for (int t2 = 0; t2 < 4; ++t2) {
                const uint32_t wword = win[t2], rword = rw[g][t2];
                const float2 v = ffma2(ns2,
                                       make_float2(__uint_as_float(h[8 * gg + 2 * t2]),
                                                   __uint_as_float(h[8 * gg + 2 * t2 + 1])),
                                       make_float2(__uint_as_float(mad_lo(wword, 0x10000u, 0u)),
                                                   __uint_as_float(wword & 0xFFFF0000u)));
                const uint32_t r_hi = mad_hi(rword, 0x10000u, 0u);
                const uint32_t r_lo = mad_lo(r_hi, 0xFFFF0000u, rword);
                const uint32_t s0 = mad_lo(r_lo, 1u, __float_as_uint(v.x));
                const uint32_t s1 = mad_hi(rword, 0x10000u, __float_as_uint(v.y));
                wout[t2] = __byte_perm(s0, s1, 0x7632);
                ym[2 * t2] = rounding_margin(s0, v.x);
                ym[2 * t2 + 1] = rounding_margin(s1, v.y);
              }
              // smallest margin of the group; NaN if any is NaN
              const float gm = fmin3_nan(fmin3_nan(ym[0], ym[1], ym[2]), fmin3_nan(ym[3], ym[4], ym[5]),
                                         fmin_nan(ym[6], ym[7]));
              // rows past d hold v = 0 against a bound of 0 and pass; columns
              // past k (the last tile of a row) may flag, and are masked below
              const bool flag = !(gm >= bound);
              tc::sts128(sp, make_uint4(wout[0], wout[1], wout[2], wout[3]));
              float t = gs;
              if (need_norm) {
#pragma unroll
                for (int t2 = 0; t2 < 4; ++t2) t = sq_acc_bf16x2(wout[t2], t);
              }
              // Rare: a group with an element whose margin the bound might
              // cross.  The flagged elements inside W keep their original
              // weights in the stage (the fix kernel recomputes them from W)
              // and go into the lane's map word.
              if (__any_sync(0xFFFFFFFFu, flag)) {
                uint32_t emask = 0;
                if (flag && row_ok && j0 + col < k) {
#pragma unroll
                  for (int e = 0; e < 8; ++e) emask |= (ym[e] >= bound) ? 0u : (1u << e);
                  if (j0 + col + 8 > k) emask &= (1u << (k - j0 - col)) - 1u;  // columns inside W
                }
                if (emask != 0) {
                  uint32_t sel[4];
                  t = gs;
#pragma unroll
                  for (int t2 = 0; t2 < 4; ++t2) {
                    const uint32_t m = (((emask >> (2 * t2)) & 1u) ? 0x0000FFFFu : 0u) |
                                       (((emask >> (2 * t2 + 1)) & 1u) ? 0xFFFF0000u : 0u);
                    sel[t2] = (wout[t2] & ~m) | (win[t2] & m);
                    if (need_norm) t = sq_acc_bf16x2(sel[t2], t);
                  }
                  tc::sts128(sp, make_uint4(sel[0], sel[1], sel[2], sel[3]));
                  fmap |= emask << (8 * g);
                }
              }
              if (j0 + col < k) gs = t;
            }
          }
          // the tile's flagged groups into the warp's tag list, groups in order
          // and lanes in order within a group
          if (__any_sync(0xFFFFFFFFu, fmap != 0)) {
            uint16_t* const tags = a.fix_tags[p] + set * kFixCap;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) {
              const uint32_t em = (fmap >> (8 * g)) & 0xFFu;
              const uint32_t bal = __ballot_sync(0xFFFFFFFFu, em != 0);
              if (em != 0) tags[nflag + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)(em | ((uint32_t)lane << 8) | ((uint32_t)g << 13));
              nflag += __popc(bal);
            }
          }
          if (need_norm && row_ok) {  // the tile's squares into the compensated sum
            const float y = gs - sq_comp;
            const float tsum = sq + y;
            sq_comp = (tsum - sq) - y;
            sq = tsum;
          }
        }
        // the number of tags (written on every call)
        if (lane == 0) a.fix_counts[p][set] = (uint8_t)nflag;
        // this warp is done with the TMEM buffer
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty_bar[b]);
        // this warp's results are in the stage: make them visible to the TMA
        // engine and tell the store warp
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sfull_bar[sw]);
        if (++sw == NSW) {
          sw = 0;
          wph ^= 1u;
        }
      }
      if (need_norm) {
        // ||W_new||^2 of this unit: each warp leaves its share in a shared
        // slot of the unit; the unit's last warp adds the 16 shares in warp
        // order, and the layer's last unit (ticket) adds all units in order
        double dsq = (double)sq - (double)sq_comp;
        for (int o = 16; o > 0; o >>= 1) dsq += __shfl_xor_sync(0xFFFFFFFFu, dsq, o);
        if (lane == 0) {
          const int slot = un & (kNormSlots - 1);
          norm_slot[slot][ew] = dsq;
          __threadfence_block();
          if (atomicAdd(&norm_count[slot], 1) == kEpiWarps - 1) {
            __threadfence_block();
            double tot = 0.0;
            for (int w = 0; w < kEpiWarps; ++w) tot += *((volatile double*)&norm_slot[slot][w]);
            norm_count[slot] = 0;
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
        }
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
}

int round16(int r) { return (r + 15) / 16 * 16; }

// Columns per tile: the C row block (both parts, all of r) plus two P chunk
// stages and three or more W stages must fit in shared memory.
int update_ncols(int r) { return round16(r) <= 128 ? 128 : 64; }

// FP16 parts of C and P: two, so H takes three products (hi hi, hi lo, lo hi).
int update_parts(int) { return 2; }

// Error of the three-product tensor-core H relative to ||c_i|| ||p_j||: twice
// the largest error measured over millions of elements for each rank class
// (Gaussian C at two scales; Gaussian-QR and Rademacher P), whose largest were
// 2^-22.9 for r = 4, 2^-21.3 for r = 16, 2^-21.3 for r = 64, 2^-21.6 for
// r = 128 and 2^-21.1 for r = 256.  The margin test treats any H within this
// of the exact product as possible.
float tc_err_beta(int) { return 0x1p-20f; }

template <int NCOLS>
cudaError_t launch_update_tc(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, bool normsgd,
                             float scale_val, uint64_t seed, uint32_t step, cudaStream_t stream) {
  const int r_pad = round16(r);
  int* errw = nullptr;
  cudaError_t err = device_error_word(&errw);
  if (err != cudaSuccess) return err;
  unsigned long long* exact = nullptr;
  err = device_exact_counter(&exact);
  if (err != cudaSuccess) return err;
  static thread_local UpdBatch a;
  const int parts = update_parts(r);
  a.scale_val = scale_val;
  a.parts = parts;
  a.err_coef = 0x1p25f * (tc_err_beta(r) + 0x1p-24f);
  philox_round_keys(seed, a.rk0, a.rk1);
  a.step = step;
  a.r = r;
  a.r_pad = r_pad;
  a.kchunks = (r_pad + 63) / 64;
  a.a_bytes = (uint32_t)a.kchunks * 16384u;
  a.b_bytes = (uint32_t)NCOLS * 128u;
  a.w_bytes = (uint32_t)(NCOLS / 64) * 16384u;
  a.err = errw;
  a.exact_count = exact;
  // dynamic shared memory: what the opt-in limit leaves next to the static arrays
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, update_persistent_kernel<NCOLS>);
  if (err != cudaSuccess) return err;
  const size_t max_smem = 227 * 1024 - fa.sharedSizeBytes;
  const size_t fixed = (size_t)parts * a.a_bytes + 1024;
  const size_t p_stage = (size_t)parts * a.b_bytes;
  // P stages (each one 64-wide chunk of r): up to rank 128 two, when they
  // still leave three W stages (W comes from HBM and needs the deeper ring),
  // else one; above, as many as leave two W stages (rank 256: a tile's four
  // chunks, 4% faster than two).  The rest of shared memory goes to the W ring.
  int p_stages = (fixed + 2 * p_stage + 3 * (size_t)a.w_bytes <= max_smem) ? 2 : 1;
  if (a.kchunks > 2) {
    p_stages = 2 * a.kchunks;
    while (p_stages > 1 && fixed + p_stages * p_stage + 2 * (size_t)a.w_bytes > max_smem) --p_stages;
  }
  int w_stages = (int)((max_smem - fixed - p_stages * p_stage) / a.w_bytes);
  if (w_stages > kMaxStagesUpd) w_stages = kMaxStagesUpd;
  if (w_stages < 1) return cudaErrorInvalidConfiguration;
  a.p_stages = p_stages;
  a.w_stages = w_stages;
  const size_t smem = fixed + p_stages * p_stage + (size_t)w_stages * a.w_bytes;
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
    // Layers of under 2^24 weights on average take their units in turn
    // (measured on the Qwen3-1.7B stack: the update phase 11% faster at rank
    // 64, 6% at 128), larger ones contiguous ranges (the Qwen3-8B stack's 3%
    // faster that way).  In turn: units of the smallest layer's column tiles, so that
    // nearly every unit is equally long, doubled while CTAs would get more than
    // 64 units.  Ranges: about twelve units per CTA, at least four tiles each
    // so that the C row block is reused.  4 to 64 tiles either way.
    int64_t weights = 0;
    for (int i = 0; i < m; ++i) weights += probs[base + i].d * probs[base + i].k;
    a.interleave = weights < ((int64_t)m << 24) ? 1 : 0;
    int64_t ut;
    if (a.interleave) {
      int64_t min_ct = 64;
      for (int i = 0; i < m; ++i) min_ct = std::min(min_ct, ceil_div(probs[base + i].k, NCOLS));
      ut = min_ct < 4 ? 4 : min_ct;
      while (ut < 64 && total_tiles > 64 * ut * (int64_t)nsm) ut *= 2;
    } else {
      ut = total_tiles / (12 * (int64_t)nsm);
    }
    if (ut < 4) ut = 4;
    if (ut > 64) ut = 64;
    for (int i = 0; i < m; ++i) a.ut[i] = (int)ut;
    a.unit_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      const UpdateWorkspace& w = ws[base + i];
      err = make_tmap_bf16_2d(&a.tm_c[i], w.c_split, (uint64_t)parts * r_pad, (uint64_t)pr.d,
                              (uint64_t)parts * r_pad * 2, 64, 128);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tm_p[i], w.p_split, (uint64_t)parts * r_pad, (uint64_t)pr.k,
                                (uint64_t)parts * r_pad * 2, 64, NCOLS);
      if (err == cudaSuccess)
        err = make_tmap_bf16_2d(&a.tm_w[i], pr.W, (uint64_t)pr.k, (uint64_t)pr.d, (uint64_t)pr.ld_w * 2, 64, 128);
      if (err != cudaSuccess) return err;
      a.C[i] = pr.C;
      a.P[i] = pr.P;
      a.c_norm[i] = w.c_norm;
      a.p_norm[i] = w.p_norm;
      a.c_unscale[i] = w.c_unscale;
      a.p_unscale[i] = w.p_unscale;
      a.d[i] = pr.d;
      a.k[i] = pr.k;
      a.n_ct[i] = (int)ceil_div(pr.k, NCOLS);
      a.n_cu[i] = (int)ceil_div(a.n_ct[i], a.ut[i]);
      a.unit_begin[i + 1] = a.unit_begin[i] + a.n_cu[i] * (int)ceil_div(pr.d, 128);
      a.layer[i] = pr.layer;
      a.scale_dev[i] = normsgd ? w.scale : nullptr;
      a.status_in[i] = normsgd ? (pr.dev_status ? pr.dev_status : w.status) : nullptr;
      a.status_out[i] = normsgd ? nullptr : pr.dev_status;
      a.unit_partials[i] = w.wnew_partials;
      a.ticket[i] = w.ticket;
      a.wnorm2_out[i] = normsgd ? pr.wnorm2_out : nullptr;
      a.fix_tags[i] = w.fix_tags;
      a.fix_counts[i] = w.fix_counts;
    }
    const int units = a.unit_begin[m];
    int grid = units < nsm ? units : nsm;
    if (grid > kMaxCtas) grid = kMaxCtas;
    if (a.interleave) {
      a.u_step = grid;
      for (int b = 0; b < grid; ++b) {
        a.cta_first[b] = b;
        a.cta_end[b] = units;
      }
    } else {
      // split the units into `grid` contiguous ranges of about equal tile count
      a.u_step = 1;
      int64_t tile_total = 0;
      for (int i = 0; i < m; ++i) tile_total += (int64_t)a.n_ct[i] * ceil_div(probs[base + i].d, 128);
      int cta = 0;
      int64_t acc = 0;
      a.cta_first[0] = 0;
      int u = 0;
      for (int i = 0; i < m; ++i) {
        const int nrb = (int)ceil_div(probs[base + i].d, 128);
        for (int rb = 0; rb < nrb; ++rb) {
          for (int cu = 0; cu < a.n_cu[i]; ++cu, ++u) {
            const int t0 = cu * a.ut[i];
            const int t1 = (t0 + a.ut[i] < a.n_ct[i]) ? t0 + a.ut[i] : a.n_ct[i];
            acc += t1 - t0;
            // close CTA ranges whose share of tiles is reached
            while (cta + 1 < grid && acc * grid >= tile_total * (cta + 1)) {
              a.cta_end[cta] = u + 1;
              a.cta_first[++cta] = u + 1;
            }
          }
        }
      }
      while (cta + 1 < grid) {
        a.cta_end[cta] = units;
        a.cta_first[++cta] = units;
      }
      a.cta_end[cta] = units;
    }
    count_launch();
    update_persistent_kernel<NCOLS><<<grid, kUpdThreads, smem, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// ---- the exact path's queue ---------------------------------------------------
// The update kernel queues each 8-column group holding an element whose
// rounding margin its tensor-core H might cross (the group's original weights,
// the flagged elements and their position) and stores the tensor-core results.
// Once every tile is stored, exact_fix_kernel redoes each flagged element the
// way the definition does: H_ij as a compensated dot product (Dot2) of the fp32
// row i of C and row j of P, v = fmaf(-s, fl32(H_ij), w), the same stochastic
// rounding, and writes the weight.  For normalized SGD it also carries the
// change of ||W_new||^2: each element's change (new^2 - old^2, exact in
// double) in fixed point relative to its layer's norm, summed as integers so
// that the total does not depend on the order in which elements are fixed;
// exact_fix_finalize_kernel adds each layer's total to its norm.
struct FixBatch {
  const uint16_t* tags[kMaxUpd];
  const uint8_t* counts[kMaxUpd];
  uint32_t* ticket[kMaxUpd];           // bit 31: a non-finite change
  unsigned long long* acc[kMaxUpd];
  const float* C[kMaxUpd];
  const float* P[kMaxUpd];
  uint16_t* W[kMaxUpd];
  int64_t ld_w[kMaxUpd];
  int64_t d[kMaxUpd], k[kMaxUpd];
  int n_ct[kMaxUpd];                   // column tiles of the layer
  int tiles[kMaxUpd];
  const float* scale_dev[kMaxUpd];     // normalized SGD: s on the device; NULL: scale_val
  const int32_t* status_in[kMaxUpd];   // layer skipped when nonzero
  double* wnorm2_out[kMaxUpd];
  uint32_t layer[kMaxUpd];
  int n;
  int r;
  int ncols;                           // NCOLS of the update launch
  float scale_val;
  uint32_t rk0[10], rk1[10];           // Philox round keys of the seed
  uint32_t step;
  unsigned long long* exact_count;
};
constexpr int kFixFracBits = 40;  // fixed point: 2^-40 of the layer's norm
constexpr int kFixThreads = 256;
constexpr int kFixSetsPerLane = 4;  // (tile, warp) flag bytes each lane of the fix kernel reads

// Fixed-point scale of a layer's changes: ref (the tensor-core ||W_new||^2)
// is at least every tensor-core square and an exact result is within a step
// or two of its tensor-core one, so a change is at most ~1.1 ref, ~2^42 in
// fixed point.  A zero norm (every tensor-core result zero) takes a plain
// double sum instead.
__device__ __forceinline__ double fix_to_fixed(double ref) {
  return ref > 0.0 ? ldexp(1.0, kFixFracBits - ilogb(ref)) : 1.0;
}

// H_ij as a compensated dot product of c and p (r terms) by one thread: the
// operands come in 32-term chunks, every load of a chunk issued before its
// terms are summed (a TwoSum running pair), so an element waits on memory
// r / 32 times rather than once per term.  fl32 of the exact sum except
// within about 2^-40 of a rounding boundary.
__device__ __forceinline__ float thread_dot2(const float* c, const float* p, int r) {
  float hs = 0.f, he = 0.f;
  auto term = [&](float cv, float pv) {
    const float m = __fmul_rn(cv, pv);
    float sum, err;
    two_sum(hs, m, sum, err);
    hs = sum;
    he = __fadd_rn(he, __fadd_rn(err, __fmaf_rn(cv, pv, -m)));
  };
  if ((r & 3) == 0) {
    for (int l0 = 0; l0 < r; l0 += 16) {
      float4 cv[4], pv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool in = l0 + 4 * q < r;
        cv[q] = in ? __ldg(reinterpret_cast<const float4*>(c + l0) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        pv[q] = in ? __ldg(reinterpret_cast<const float4*>(p + l0) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (l0 + 4 * q >= r) break;
        term(cv[q].x, pv[q].x);
        term(cv[q].y, pv[q].y);
        term(cv[q].z, pv[q].z);
        term(cv[q].w, pv[q].w);
      }
    }
  } else {
    for (int l = 0; l < r; ++l) term(__ldg(c + l), __ldg(p + l));
  }
  return __fadd_rn(hs, he);
}

// One flagged element: H_ij by thread_dot2, then the same v and stochastic
// rounding as the tensor-core path from the original weight w16 (still in W),
// the result written over it.  Returns whether the weight changed; the change
// of ||W_new||^2 goes, in fixed point relative to the layer's norm, into an
// integer sum whose total does not depend on the order of the elements.
__device__ __forceinline__ void fix_element(const FixBatch& b, int p, uint16_t* wrow, const float* crow, int j,
                                            uint32_t w16, uint32_t r16, float s, double* wn) {
  const int r = b.r;
  const float hx = thread_dot2(crow, b.P[p] + (int64_t)j * r, r);
  const float v = fmaf(-s, hx, __uint_as_float(w16 << 16));
  const uint32_t out = sr_bf16_bits(v, r16);
  if (out == w16) return;
  wrow[j] = (uint16_t)out;
  if (wn == nullptr) return;
  const double ref = *wn;
  if (!isfinite(ref)) return;
  const double fo = (double)__uint_as_float(w16 << 16), fn = (double)__uint_as_float(out << 16);
  const double delta = fn * fn - fo * fo;  // exact: both squares have 16-bit mantissas
  if (!isfinite(delta)) atomicOr(b.ticket[p], 0x80000000u);
  else if (ref > 0.0) atomicAdd(b.acc[p], (unsigned long long)llrint(delta * fix_to_fixed(ref)));
  else atomicAdd(reinterpret_cast<double*>(b.acc[p]), delta);
}

// Each thread reads the tag counts of kFixSetsPerLane (tile, epilogue warp)
// sets of a layer (blockIdx.y); the warp keeps the running total of its sets'
// counts in shared memory and deals the tags out one per lane (a lane finds
// the set of its tag by binary search), so that no lane works through a full
// set while the others wait.  For a tag: the group's Philox block and weights
// (original ones where flagged) from W, then fix_element for each flagged
// element.
__global__ void __launch_bounds__(kFixThreads, 4) exact_fix_kernel(const __grid_constant__ FixBatch b) {
  constexpr int kSets = 32 * kFixSetsPerLane;
  __shared__ uint32_t pre[kFixThreads / 32][kSets];  // tags of the warp's sets before each set
  __shared__ uint32_t wtot[kFixThreads / 32];         // tags of each warp's sets
  __shared__ unsigned block_done;
  const int p = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) block_done = 0;
  __syncthreads();
  const bool skipped = b.status_in[p] != nullptr && *b.status_in[p] != 0;
  const int64_t sets = (int64_t)b.tiles[p] * kEpiWarps;
  // this warp's sets: base + 32 q + lane for q < kFixSetsPerLane (each load a
  // coalesced run of 32 counts, all issued before any is used)
  const int64_t base = ((int64_t)blockIdx.x * (kFixThreads / 32) + warp) * kSets;
  uint32_t cnt[kFixSetsPerLane];
#pragma unroll
  for (int q = 0; q < kFixSetsPerLane; ++q) {
    const int64_t set = base + 32 * q + lane;
    cnt[q] = (!skipped && set < sets) ? b.counts[p][set] : 0u;
  }
  uint32_t total = 0;
#pragma unroll
  for (int q = 0; q < kFixSetsPerLane; ++q) {
    uint32_t incl = cnt[q];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    pre[warp][32 * q + lane] = total + incl - cnt[q];
    total += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) wtot[warp] = total;
  __syncthreads();
  // the block's tags are dealt over all its threads: warp w's tags follow
  // those of warps 0 .. w-1
  uint32_t woff[kFixThreads / 32], btotal = 0;
#pragma unroll
  for (int w = 0; w < kFixThreads / 32; ++w) {
    woff[w] = btotal;
    btotal += wtot[w];
  }
  const int64_t bbase = (int64_t)blockIdx.x * (kFixThreads / 32) * kSets;
  unsigned done = 0;
  if (btotal != 0) {
    const int kcols = b.ncols / 4;
    const float s = b.scale_dev[p] ? *b.scale_dev[p] : b.scale_val;
    const uint32_t k8 = (uint32_t)b.k[p] >> 3;
    double* wn = b.wnorm2_out[p];
    for (uint32_t idx = threadIdx.x; idx < btotal; idx += kFixThreads) {
      // the warp whose sets hold tag idx, then the last of its sets whose tags
      // start at or before it
      int w = 0;
      uint32_t wo = 0;
#pragma unroll
      for (int v = 1; v < kFixThreads / 32; ++v)
        if (woff[v] <= idx) {
          w = v;
          wo = woff[v];
        }
      const uint32_t li = idx - wo;
      int lo = 0;
#pragma unroll
      for (int step = kSets / 2; step > 0; step >>= 1)
        if (pre[w][lo + step] <= li) lo += step;
      const int64_t sset = bbase + (int64_t)w * kSets + lo;
      const uint32_t tag = b.tags[p][sset * kFixCap + (li - pre[w][lo])];
      const int t = (int)(sset / kEpiWarps), ew = (int)(sset % kEpiWarps);
      const int rb = t / b.n_ct[p], ct = t % b.n_ct[p];
      const int i = rb * 128 + (ew & 3) * 32 + (int)((tag >> 8) & 31u);
      const int jg = ct * b.ncols + (ew >> 2) * kcols + 8 * (int)(tag >> 13);
      if (i >= b.d[p] || jg >= b.k[p]) continue;  // only after a timed-out update
      uint16_t* wrow = b.W[p] + (int64_t)i * b.ld_w[p];
      // the group's weights (ld_w and jg are multiples of 8), read before the
      // dot products so that the load overlaps them
      const uint4 w4 = *reinterpret_cast<const uint4*>(wrow + jg);
      const uint32_t blk[1] = {(uint32_t)i * k8 + ((uint32_t)jg >> 3)};
      uint32_t rw[1][4];
      philox4x32_10_rk_multi<1>(blk, b.step, b.layer[p], kTagSR, b.rk0, b.rk1, rw);
      const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
      const float* crow = b.C[p] + (int64_t)i * b.r;
      for (uint32_t m = tag & 0xFFu; m; m &= m - 1u) {
        const int e = __ffs(m) - 1;
        const int sh = (e & 1) * 16;
        const uint32_t w16 = (pick(wv, e >> 1) >> sh) & 0xFFFFu, r16 = (pick(rw[0], e >> 1) >> sh) & 0xFFFFu;
        fix_element(b, p, wrow, crow, jg + e, w16, r16, s, wn);
        ++done;
      }
    }
  }
  if (done != 0 && b.exact_count != nullptr) atomicAdd(&block_done, done);
  __syncthreads();
  if (threadIdx.x == 0 && block_done != 0 && b.exact_count != nullptr)
    atomicAdd(b.exact_count, (unsigned long long)block_done);
}

// After exact_fix_kernel: each layer's fixed-point total of changes added to
// its ||W_new||^2 (NaN when a change was not finite).
__global__ void __launch_bounds__(256) exact_fix_finalize_kernel(const __grid_constant__ FixBatch b) {
  for (int p = threadIdx.x; p < b.n; p += blockDim.x) {
    double* wn = b.wnorm2_out[p];
    if (wn == nullptr) continue;
    if (b.status_in[p] != nullptr && *b.status_in[p] != 0) continue;  // the update skipped the layer
    const double ref = *wn;
    if (!isfinite(ref)) continue;
    const unsigned long long acc = *b.acc[p];
    const double add = ref > 0.0 ? (double)(long long)acc / fix_to_fixed(ref) : __longlong_as_double((long long)acc);
    *wn = (*b.ticket[p] & 0x80000000u) ? __longlong_as_double(0x7FF8000000000000ll) : ref + add;
  }
}

// The fix kernel of the update launches of these problems (the same layers per
// launch as launch_update_tc).
cudaError_t launch_exact_fix(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, bool normsgd,
                             float scale_val, int ncols, uint64_t seed, uint32_t step, cudaStream_t stream) {
  unsigned long long* exact = nullptr;
  cudaError_t err = device_exact_counter(&exact);
  if (err != cudaSuccess) return err;
  static thread_local FixBatch f;
  f.r = r;
  f.ncols = ncols;
  f.scale_val = scale_val;
  philox_round_keys(seed, f.rk0, f.rk1);
  f.step = step;
  f.exact_count = exact;
  for (int base = 0; base < n; base += kMaxUpd) {
    const int m = (n - base) < kMaxUpd ? (n - base) : kMaxUpd;
    f.n = m;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      const UpdateWorkspace& w = ws[base + i];
      f.tags[i] = w.fix_tags;
      f.counts[i] = w.fix_counts;
      f.layer[i] = pr.layer;
      f.ticket[i] = w.fix_ticket;
      f.acc[i] = w.fix_acc;
      f.C[i] = pr.C;
      f.P[i] = pr.P;
      f.W[i] = pr.W;
      f.ld_w[i] = pr.ld_w;
      f.d[i] = pr.d;
      f.k[i] = pr.k;
      f.n_ct[i] = (int)ceil_div(pr.k, ncols);
      f.tiles[i] = f.n_ct[i] * (int)ceil_div(pr.d, 128);
      f.scale_dev[i] = normsgd ? w.scale : nullptr;
      f.status_in[i] = normsgd ? (pr.dev_status ? pr.dev_status : w.status) : nullptr;
      f.wnorm2_out[i] = normsgd ? pr.wnorm2_out : nullptr;
    }
    int64_t sets = 0;
    for (int i = 0; i < m; ++i) sets = std::max(sets, (int64_t)f.tiles[i] * kEpiWarps);
    count_launch();
    exact_fix_kernel<<<dim3((unsigned)ceil_div(sets, (int64_t)kFixThreads * kFixSetsPerLane), m), kFixThreads, 0,
                       stream>>>(f);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (normsgd) {
      count_launch();
      exact_fix_finalize_kernel<<<1, 256, 0, stream>>>(f);
      err = cudaGetLastError();
      if (err != cudaSuccess) return err;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_split(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, cudaStream_t stream) {
  static thread_local SplitBatch sb;
  sb.r = r;
  sb.r_pad = round16(r);
  for (int base = 0; base < n; base += kMaxAux) {
    const int m = (n - base) < kMaxAux ? (n - base) : kMaxAux;
    sb.n = 2 * m;
    sb.block_begin[0] = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      const UpdateWorkspace& w = ws[base + i];
      sb.src[2 * i] = pr.C;
      sb.rows[2 * i] = pr.d;
      sb.dst[2 * i] = w.c_split;
      sb.norm[2 * i] = w.c_norm;
      sb.unscale[2 * i] = w.c_unscale;
      sb.block_begin[2 * i + 1] = sb.block_begin[2 * i] + ceil_div(pr.d, kSplitRows);
      sb.src[2 * i + 1] = pr.P;
      sb.rows[2 * i + 1] = pr.k;
      sb.dst[2 * i + 1] = w.p_split;
      sb.norm[2 * i + 1] = w.p_norm;
      sb.unscale[2 * i + 1] = w.p_unscale;
      sb.block_begin[2 * i + 2] = sb.block_begin[2 * i + 1] + ceil_div(pr.k, kSplitRows);
      sb.fix_ticket[i] = w.fix_ticket;
      sb.fix_acc[i] = w.fix_acc;
    }
    count_launch();
    split_fp16_kernel<<<(unsigned)sb.block_begin[2 * m], 256, 0, stream>>>(sb);
  }
  return cudaGetLastError();
}

// split_done: the normalized-SGD step has already split C and P (its Grams take
// their scales from the split's row norms).
cudaError_t launch_update(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, bool normsgd,
                          float scale_val, uint64_t seed, uint32_t step, cudaStream_t stream,
                          bool split_done = false) {
  cudaError_t err = split_done ? cudaSuccess : launch_split(n, probs, ws, r, stream);
  if (err != cudaSuccess) return err;
  const int ncols = update_ncols(r);
  err = (ncols == 128) ? launch_update_tc<128>(n, probs, ws, r, normsgd, scale_val, seed, step, stream)
                       : launch_update_tc<64>(n, probs, ws, r, normsgd, scale_val, seed, step, stream);
  if (err != cudaSuccess) return err;
  return launch_exact_fix(n, probs, ws, r, normsgd, scale_val, ncols, seed, step, stream);
}

}  // namespace

size_t carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd, UpdateWorkspace* ws) {
  const size_t start = cur.offset;
  UpdateWorkspace w{};
  const int r_pad = round16(r);
  if (normsgd) {
    w.gram_partials_p = cur.take<float2>((size_t)gram_chunks_tc(k, r).nchunks * r * r);
    w.gram_partials_c = cur.take<float2>((size_t)gram_chunks_tc(d, r).nchunks * r * r);
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
  w.c_unscale = cur.take<float>((size_t)d);
  w.p_unscale = cur.take<float>((size_t)ceil_div(k, kSplitRows));
  w.c_split = cur.take<uint16_t>((size_t)d * 2 * r_pad);
  w.p_split = cur.take<uint16_t>((size_t)k * 2 * r_pad);
  // exact-path tags: a count and kFixCap tags per (tile, epilogue warp)
  const int64_t tiles = ceil_div(d, 128) * ceil_div(k, update_ncols(r));
  w.fix_ticket = cur.take<uint32_t>(1);
  w.fix_acc = cur.take<unsigned long long>(1);
  w.fix_counts = cur.take<uint8_t>((size_t)tiles * kEpiWarps);
  w.fix_tags = cur.take<uint16_t>((size_t)tiles * kEpiWarps * kFixCap);
  cur.take<char>(0);  // end on a 256-byte boundary
  if (ws) *ws = w;
  return cur.offset - start;
}

cudaError_t launch_update_normsgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float tau,
                                  uint64_t seed, uint32_t step, cudaStream_t stream) {
  static thread_local WnormBatch wb;
  static thread_local GramBatch gb;
  static thread_local FinalizeBatch fb;
  // the split first: its row norms bound each Gram chunk's largest magnitude
  cudaError_t err = launch_split(n, probs, ws, r, stream);
  if (err != cudaSuccess) return err;
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
      gb.e[2 * i].row_norms = w.p_norm;
      gb.e[2 * i + 1] = GramEntry{pr.C, pr.d, w.gram_partials_c, w.gram_c};
      gb.e[2 * i + 1].row_norms = w.c_norm;
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
  return launch_update(n, probs, ws, r, true, 0.f, seed, step, stream, true);
}

cudaError_t launch_update_sgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float alpha_eta,
                              uint64_t seed, uint32_t step, cudaStream_t stream) {
  return launch_update(n, probs, ws, r, false, alpha_eta, seed, step, stream);
}

}  // namespace rgs
