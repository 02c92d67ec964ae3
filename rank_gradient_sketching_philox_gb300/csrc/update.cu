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

constexpr int kMaxUpd = 48;     // layers per rebuild+update launch (kernel parameter table)
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
  int64_t rows[2 * kMaxAux];
  uint16_t* dst[2 * kMaxAux];   // rows x (2 r_pad): [hi | lo]
  float* norm[2 * kMaxAux];     // rows: Euclidean norm of each source row
  int r;
  int r_pad;
};

// One warp per row: x = hi + lo to 2^-17 relative (columns r..r_pad-1 zero)
// and ||row||_2.  grid (rows / 8, entries), 256 threads.
__global__ void __launch_bounds__(256) split_rows_kernel(const __grid_constant__ SplitBatch b) {
  const int en = blockIdx.y;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= b.rows[en]) return;
  const float* src = b.src[en] + row * b.r;
  uint16_t* dst = b.dst[en] + row * 2 * b.r_pad;
  float sq = 0.f;
  for (int col = lane; col < b.r_pad; col += 32) {
    const float v = (col < b.r) ? src[col] : 0.f;
    sq = fmaf(v, v, sq);
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    dst[col] = __bfloat16_as_ushort(h);
    dst[b.r_pad + col] = __bfloat16_as_ushort(l);
  }
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
  if (lane == 0) b.norm[en][row] = sqrtf(sq);
}

// ---- the rebuild + update kernel -------------------------------------------------
// Work of a launch: up to kMaxUpd layers.  Layer p is cut into units of
// (128-row block, run of up to unit_tiles column tiles of NCOLS); units of all
// layers are numbered end to end and each persistent CTA takes a contiguous
// range of them, so consecutive units usually share the row block of C.
struct UpdBatch {
  CUtensorMap tm_c[kMaxUpd];   // C split, d x (2 r_pad) BF16: [hi | lo]
  CUtensorMap tm_p[kMaxUpd];   // P split, k x (2 r_pad) BF16: [hi | lo]
  CUtensorMap tm_w[kMaxUpd];   // W, d x k BF16
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
  int n;
  int unit_tiles;
  int stages;
  float scale_val;
  uint64_t seed;
  uint32_t step;
  int r;
  int r_pad;          // r rounded up to 16 (MMA K extent)
  int kchunks;        // 64-wide chunks of r_pad
  uint32_t a_bytes;   // bytes of the C_hi (or C_lo) tile: kchunks x 16 KB
  uint32_t b_bytes;   // bytes of the P_hi (or P_lo) tile: kchunks x NCOLS x 128
  uint32_t w_bytes;   // bytes of the W tile: NCOLS/64 x 16 KB
  int* err;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

constexpr int kEpiWarps = 16;                     // warps 4..19
constexpr int kUpdThreads = (4 + kEpiWarps) * 32;
constexpr int kMaxStagesUpd = 4;

struct Unit {
  int p, rb, ct0, ct1;
};

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

__device__ __forceinline__ bool layer_skipped(const UpdBatch& a, int p) {
  return a.status_in[p] != nullptr && *a.status_in[p] != 0;
}

// Persistent rebuild + update.  Warp 0 (one lane) streams C row blocks and,
// per column tile, P_hi/P_lo rows and the W tile into a ring of stages with
// TMA; warp 1 (one lane) issues H = C_hi P_hi^T + C_hi P_lo^T + C_lo P_hi^T
// (tcgen05.mma, M=128, N=NCOLS) into one of two TMEM buffers; warps 4..19 read
// H (warp w: TMEM lanes 32(w%4).., column quarter (w-4)/4), form
// v = fmaf(-s, H, w) and stochastically round it with 16 Philox bits per weight
// in shared memory, then one thread stores the tile with TMA.
//
// Exactness where it matters: |H_tc - H| <= ||c_i|| ||p_j|| 2^-14 (three BF16
// products leave ~3 * 2^-18 per term; the bound has >4x margin).  When that
// could move v across more than one BF16 step (|v| < s ||c_i|| ||p_j|| 2^-5),
// the warp recomputes H_ij in double from fp32 C and P and uses fl32(H_ij),
// which is the value the definition rounds.
template <int NCOLS>
__global__ void __launch_bounds__(kUpdThreads, 1) update_persistent_kernel(const __grid_constant__ UpdBatch a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStagesUpd], empty_bar[kMaxStagesUpd];
  __shared__ __align__(8) uint64_t cfull_bar, cempty_bar, tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;
  __shared__ float warp_sq[kEpiWarps];

  uint8_t* smem = align1024(smem_raw);
  uint8_t* s_chi = smem;
  uint8_t* s_clo = s_chi + a.a_bytes;
  uint8_t* s_stage0 = s_clo + a.a_bytes;
  const uint32_t stage_bytes = 2 * a.b_bytes + a.w_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = a.stages;
  const int units = a.unit_begin[a.n];
  const int u_begin = (int)((int64_t)units * blockIdx.x / gridDim.x);
  const int u_end = (int)((int64_t)units * (blockIdx.x + 1) / gridDim.x);
  constexpr uint32_t kTmemCols = 2 * NCOLS;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 2);
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
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- producer ----------------
    int it = 0, cl = 0, prev_p = -1, prev_rb = -1;
    for (int u = u_begin; u < u_end && !abort_flag; ++u) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(a, x.p)) continue;
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
        const int s = it % NS;
        if (it >= NS && !tc::mbar_wait(&empty_bar[s], ((it / NS) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage))
          break;
        uint8_t* st = s_stage0 + (size_t)s * stage_bytes;
        const int j0 = ct * NCOLS;
        tc::mbar_arrive_expect_tx(&full_bar[s], stage_bytes);
        for (int c = 0; c < a.kchunks; ++c) {
          tc::tma_load_2d(st + c * NCOLS * 128, &a.tm_p[x.p], &full_bar[s], c * 64, j0);
          tc::tma_load_2d(st + a.b_bytes + c * NCOLS * 128, &a.tm_p[x.p], &full_bar[s], a.r_pad + c * 64, j0);
        }
#pragma unroll
        for (int bx = 0; bx < NCOLS / 64; ++bx)
          tc::tma_load_2d(st + 2 * a.b_bytes + bx * 16384, &a.tm_w[x.p], &full_bar[s], j0 + 64 * bx, i0);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = tc::idesc_bf16(128, NCOLS, false, false);
    int it = 0, cl = 0, prev_p = -1, prev_rb = -1;
    for (int u = u_begin; u < u_end && !abort_flag; ++u) {
      const Unit x = decode_unit(a, u);
      if (layer_skipped(a, x.p)) continue;
      if (x.p != prev_p || x.rb != prev_rb) {
        if (!tc::mbar_wait(&cfull_bar, cl & 1, &abort_flag, a.err, tc::kErrTimeoutLoad)) break;
        ++cl;
        prev_p = x.p;
        prev_rb = x.rb;
      }
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int s = it % NS, b = it & 1;
        if (!tc::mbar_wait(&full_bar[s], (it / NS) & 1, &abort_flag, a.err, tc::kErrTimeoutLoad)) break;
        if (it >= 2 && !tc::mbar_wait(&tempty_bar[b], ((it >> 1) - 1) & 1, &abort_flag, a.err, tc::kErrTimeoutStage))
          break;
        tc::tc_fence_after();
        const uint32_t st = tc::smem_u32(s_stage0 + (size_t)s * stage_bytes);
        const uint32_t d_tmem = tmem + (uint32_t)(b * NCOLS);
        uint32_t acc = 0;
        for (int c = 0; c < a.kchunks; ++c) {
          for (int kk = 0; kk < 4 && c * 64 + kk * 16 < a.r_pad; ++kk) {
            const uint32_t off_a = c * 16384 + kk * 32, off_b = c * NCOLS * 128 + kk * 32;
            const uint64_t ahi = tc::sdesc_sw128(tc::smem_u32(s_chi) + off_a, 16, 1024);
            const uint64_t alo = tc::sdesc_sw128(tc::smem_u32(s_clo) + off_a, 16, 1024);
            const uint64_t bhi = tc::sdesc_sw128(st + off_b, 16, 1024);
            const uint64_t blo = tc::sdesc_sw128(st + a.b_bytes + off_b, 16, 1024);
            tc::mma_bf16(d_tmem, ahi, bhi, idesc, acc);
            tc::mma_bf16(d_tmem, ahi, blo, idesc, 1u);
            tc::mma_bf16(d_tmem, alo, bhi, idesc, 1u);
            acc = 1u;
          }
        }
        tc::mma_commit(&empty_bar[s]);
        tc::mma_commit(&tfull_bar[b]);
      }
      // release the C row block once its last unit is issued
      bool last_of_c = (u + 1 == u_end);
      if (!last_of_c) {
        const Unit y = decode_unit(a, u + 1);
        last_of_c = (y.p != x.p || y.rb != x.rb);
      }
      if (last_of_c) tc::mma_commit(&cempty_bar);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue ----------------
    const int ew = warp - 4;
    const int quarter = warp & 3;
    constexpr int kCols = NCOLS / 4;           // columns per thread per tile
    const int col_base = (ew >> 2) * kCols;    // column quarter of the tile
    const int q = quarter * 32 + lane;         // tile row = TMEM lane
    const uint32_t key0 = (uint32_t)(a.seed & 0xFFFFFFFFull), key1 = (uint32_t)(a.seed >> 32);
    const bool storer = (ew == 0 && lane == 0);
    int it = 0;
    // Every epilogue warp runs the same loop and reaches every named barrier;
    // after a timed-out wait (abort) the work is skipped but the barriers are not.
    for (int u = u_begin; u < u_end; ++u) {
      const Unit x = decode_unit(a, u);
      const int p = x.p;
      if (layer_skipped(a, p)) continue;
      const int64_t d = a.d[p], k = a.k[p];
      const int64_t i = (int64_t)x.rb * 128 + q;
      const bool row_ok = i < d;
      const float s = a.scale_dev[p] ? *a.scale_dev[p] : a.scale_val;
      const float thr_row = row_ok ? fabsf(s) * a.c_norm[p][i] * 0x1p-5f : 0.f;
      const uint32_t layer = a.layer[p];
      const float* __restrict__ Cp = a.C[p];
      const float* __restrict__ Pp = a.P[p];
      const bool need_norm = a.wnorm2_out[p] != nullptr;
      float sq = 0.f;
      for (int ct = x.ct0; ct < x.ct1; ++ct, ++it) {
        const int st_idx = it % NS, b = it & 1;
        bool live = tc::mbar_wait(&tfull_bar[b], (it >> 1) & 1, &abort_flag, a.err, tc::kErrTimeoutMma) &&
                    tc::mbar_wait(&full_bar[st_idx], (it / NS) & 1, &abort_flag, a.err, tc::kErrTimeoutLoad);
        live = __all_sync(0xFFFFFFFFu, live);
        tc::tc_fence_after();
        uint32_t h[kCols];
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * NCOLS + col_base);
        if (live) {
          if constexpr (kCols == 32) tc::tmem_ld_32x32b_x32(taddr, h);
          else tc::tmem_ld_32x32b_x16(taddr, h);
          tc::tmem_wait_ld();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty_bar[b]);
        uint8_t* s_w = s_stage0 + (size_t)st_idx * stage_bytes + 2 * a.b_bytes;
        const int64_t j0 = (int64_t)ct * NCOLS;
#pragma unroll
        for (int g = 0; g < kCols / 8; ++g) {
          const int col = col_base + 8 * g;
          const int64_t j = j0 + col;
          const bool ok = live && row_ok && j < k;
          uint4* wp = reinterpret_cast<uint4*>(s_w + (col >> 6) * 16384 + q * 128 + ((((col & 63) >> 3) ^ (q & 7)) << 4));
          const uint4 raw = *wp;
          const uint32_t win[4] = {raw.x, raw.y, raw.z, raw.w};
          float wv[8], v[8];
          uint32_t out[8], rnd16[8];
          uint32_t flags = 0;
          if (ok) {
            const uint64_t e = (uint64_t)i * (uint64_t)k + (uint64_t)j;  // multiple of 8
            const Philox4 rnd = philox4x32_10((uint32_t)(e >> 3), a.step, layer, kTagSR, key0, key1);
            const uint32_t rw[4] = {rnd.w0, rnd.w1, rnd.w2, rnd.w3};
            const float4 pn0 = *reinterpret_cast<const float4*>(a.p_norm[p] + j);
            const float4 pn1 = *reinterpret_cast<const float4*>(a.p_norm[p] + j + 4);
            const float pn[8] = {pn0.x, pn0.y, pn0.z, pn0.w, pn1.x, pn1.y, pn1.z, pn1.w};
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              wv[t] = bf16_bits_to_float((t & 1) ? (win[t >> 1] >> 16) : (win[t >> 1] & 0xFFFFu));
              rnd16[t] = (t & 1) ? (rw[t >> 1] >> 16) : (rw[t >> 1] & 0xFFFFu);
              v[t] = fmaf(-s, __uint_as_float(h[8 * g + t]), wv[t]);
              out[t] = sr_bf16_bits(v[t], rnd16[t]);
              if (fabsf(v[t]) < thr_row * pn[t]) flags |= 1u << t;
            }
          }
          // exact recomputation of flagged elements, one warp-wide dot product each
          uint32_t pending = __ballot_sync(0xFFFFFFFFu, flags != 0);
          while (pending) {
            const int src = __ffs(pending) - 1;
            pending &= pending - 1;
            uint32_t fl = __shfl_sync(0xFFFFFFFFu, flags, src);
            const int64_t isrc = (int64_t)x.rb * 128 + quarter * 32 + src;
            while (fl) {
              const int t = __ffs(fl) - 1;
              fl &= fl - 1;
              const float* crow = Cp + isrc * a.r;
              const float* prow = Pp + (j + t) * a.r;
              double dot = 0.0;
              for (int l = lane; l < a.r; l += 32) dot = fma((double)crow[l], (double)prow[l], dot);
              for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, o);
              if (lane == src) {
#pragma unroll
                for (int tt = 0; tt < 8; ++tt) {
                  if (tt == t) {
                    v[tt] = fmaf(-s, (float)dot, wv[tt]);
                    out[tt] = sr_bf16_bits(v[tt], rnd16[tt]);
                  }
                }
              }
            }
          }
          if (ok) {
            uint32_t wout[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) wout[t] = out[2 * t] | (out[2 * t + 1] << 16);
            *wp = make_uint4(wout[0], wout[1], wout[2], wout[3]);
            if (need_norm) {
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const float nv = bf16_bits_to_float(out[t]);
                sq = fmaf(nv, nv, sq);
              }
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::named_barrier(1, kEpiWarps * 32);
        if (storer && live) {
          const int i0 = x.rb * 128;
#pragma unroll
          for (int bx = 0; bx < NCOLS / 64; ++bx)
            tc::tma_store_2d(&a.tm_w[p], s_w + bx * 16384, (int)j0 + 64 * bx, i0);
          tc::bulk_commit();
          if (NS >= 2) {
            if (it > 0) {
              tc::bulk_wait_read<1>();
              tc::mbar_arrive(&empty_bar[(it - 1) % NS]);
            }
          } else {
            tc::bulk_wait_read<0>();
            tc::mbar_arrive(&empty_bar[st_idx]);
          }
        }
      }
      if (need_norm) {
        // ||W_new||^2 of this unit, then the layer's last unit sums all units in order
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, o);
        if (lane == 0) warp_sq[ew] = sq;
        tc::named_barrier(1, kEpiWarps * 32);
        if (storer) {
          double tot = 0.0;
          for (int w = 0; w < kEpiWarps; ++w) tot += (double)warp_sq[w];
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
    if (storer) {
      tc::bulk_wait_all();
      if (NS >= 2 && it > 0) tc::mbar_arrive(&empty_bar[(it - 1) % NS]);
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
  a.step = step;
  a.r = r;
  a.r_pad = r_pad;
  a.kchunks = (r_pad + 63) / 64;
  a.a_bytes = (uint32_t)a.kchunks * 16384u;
  a.b_bytes = (uint32_t)a.kchunks * NCOLS * 128u;
  a.w_bytes = (uint32_t)(NCOLS / 64) * 16384u;
  a.err = errw;
  const size_t max_smem = 227 * 1024;
  const size_t fixed = 2 * (size_t)a.a_bytes + 1024;
  const size_t stage = 2 * (size_t)a.b_bytes + a.w_bytes;
  int stages = (int)((max_smem - fixed) / stage);
  if (stages > kMaxStagesUpd) stages = kMaxStagesUpd;
  if (stages < 1) return cudaErrorInvalidConfiguration;
  a.stages = stages;
  const size_t smem = fixed + (size_t)stages * stage;
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
    // about four units per CTA for balance, at least four tiles per unit to
    // amortize the C row block
    int64_t ut = total_tiles / (4 * (int64_t)nsm);
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
      a.ticket[i] = w.ticket;
      a.wnorm2_out[i] = normsgd ? pr.wnorm2_out : nullptr;
    }
    const int units = a.unit_begin[m];
    const int grid = units < nsm ? units : nsm;
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
    int64_t max_rows = 0;
    for (int i = 0; i < m; ++i) {
      const UpdateProblem& pr = probs[base + i];
      sb.src[2 * i] = pr.C;
      sb.rows[2 * i] = pr.d;
      sb.dst[2 * i] = ws[base + i].c_split;
      sb.norm[2 * i] = ws[base + i].c_norm;
      sb.src[2 * i + 1] = pr.P;
      sb.rows[2 * i + 1] = pr.k;
      sb.dst[2 * i + 1] = ws[base + i].p_split;
      sb.norm[2 * i + 1] = ws[base + i].p_norm;
      max_rows = pr.d > max_rows ? pr.d : max_rows;
      max_rows = pr.k > max_rows ? pr.k : max_rows;
    }
    split_rows_kernel<<<dim3((unsigned)ceil_div(max_rows, 8), (unsigned)(2 * m)), 256, 0, stream>>>(sb);
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

size_t carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd, UpdateWorkspace* ws) {
  const size_t start = cur.offset;
  UpdateWorkspace w{};
  const int r_pad = round16(r);
  if (normsgd) {
    w.gram_partials_p = cur.take<double>((size_t)gram_chunks(k).nchunks * r * r);
    w.gram_partials_c = cur.take<double>((size_t)gram_chunks(d).nchunks * r * r);
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
    if (nw > 0) wnorm_partial_kernel<<<dim3(kWnormBlocks, nw), 256, 0, stream>>>(wb);
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
    normsgd_finalize_kernel<<<m, 256, 0, stream>>>(fb);
  }
  return launch_update(n, probs, ws, r, true, 0.f, seed, step, stream);
}

cudaError_t launch_update_sgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float alpha_eta,
                              uint64_t seed, uint32_t step, cudaStream_t stream) {
  return launch_update(n, probs, ws, r, false, alpha_eta, seed, step, stream);
}

}  // namespace rgs
