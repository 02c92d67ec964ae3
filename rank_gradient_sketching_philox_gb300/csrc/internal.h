// Internal interface between the C ABI (abi.cu) and the kernel files.
// Arguments have been validated by the caller; these functions only launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rgs {

constexpr int kMaxRank = 256;
constexpr int kMaxBatch = 256;  // problems per batched launch (kernel parameter table)

// Workspace carving: every region starts on a 256-byte boundary.
struct WsCursor {
  char* base = nullptr;
  size_t offset = 0;
  template <typename T>
  T* take(size_t count) {
    size_t at = (offset + 255) & ~size_t(255);
    offset = at + count * sizeof(T);
    return base ? reinterpret_cast<T*>(base + at) : nullptr;
  }
};

// ---- runtime helpers (runtime.cu) -----------------------------------------
// BF16 2-D tensor map, 128-byte swizzle, zero fill outside the tensor.
cudaError_t make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// Device address of the current device's error word (bits from tc.cuh).
cudaError_t device_error_word(int** out);
// Device address of the current device's count of weights the update kernels
// recomputed on their exact path (instrumentation, read by
// sketch_read_exact_count).
cudaError_t device_exact_counter(unsigned long long** out);
int num_sms();
// Counts one kernel launch issued by this library (sketch_kernel_launches).
void count_launch();
uint64_t launches_issued();
// Message returned by sketch_last_error() on this thread.
void set_last_error(const char* message);

// ---- Gram matrices of tall-skinny fp32 matrices ----------------------------
// Row chunking of a partial Gram matrix over `rows` rows: at most 64 chunks.
struct GramChunks {
  int nchunks;
  int chunk_rows;
};
struct GramEntry {
  const float* A;   // rows x r, row-major
  int64_t rows;
  float2* partials; // gram_chunks_tc(rows, r).nchunks x r x r (hi, lo) pairs
  double* out;      // r x r
  // a bound on max |A| known to the caller (> 0), or the bits of max |A|
  // recorded by A's producer (NaN if A holds one); with neither (nor
  // row_norms), each chunk finds its own maximum first
  const uint32_t* amax = nullptr;
  float bound = 0.f;
  // else, when set, the rows' Euclidean norms (rows floats, >= each row's
  // largest magnitude): their maximum over a chunk is the chunk's bound
  const float* row_norms = nullptr;
};
// Each chunk's products go, 64 rows at a time, to gram_tc_accs(r) TMEM
// accumulators in turn (as many as 512 columns hold, up to 4), and each
// accumulator takes about 256 rows per chunk: the tensor cores' fp32
// accumulation drifts in proportion to the length of a chain, so longer chains
// lose measurably (QR orthogonality 7.5e-6 with 1024 rows per accumulator
// against 1.9e-6 with 256).  At most 64 chunks.
__host__ __device__ inline int gram_tc_accs(int r) {
  const int npad = (r + 15) / 16 * 16, nmh = r <= 128 ? 1 : 2;
  int a = 512 / (npad * nmh);
  if (a > 4) a = 4;
  return a >= 4 ? 4 : (a >= 2 ? 2 : 1);
}
// Chunks start on a multiple of 64 rows (one conversion step), so that a
// chunk's rows can be copied in 64-row pieces that start on 16 bytes.
__host__ __device__ inline GramChunks gram_chunks_tc(int64_t rows, int r) {
  const int64_t target = 256 * (int64_t)gram_tc_accs(r);
  int64_t n = (rows + target - 1) / target;
  if (n > 64) n = 64;
  if (n < 1) n = 1;
  int64_t per = (rows + n - 1) / n;
  per = (per + 63) / 64 * 64;
  GramChunks g;
  g.chunk_rows = (int)per;
  g.nchunks = (int)((rows + per - 1) / per);
  if (g.nchunks < 1) g.nchunks = 1;
  return g;
}
struct GramBatch {
  int n;
  int r;
  int raw_stages;  // set by launch_gram: the kernel's ring of fp32 row copies (0: none)
  GramEntry e[kMaxBatch];
  int chunk_begin[kMaxBatch + 1];  // set by launch_gram: prefix of the entries' chunk counts
};
// Partial Grams on the tensor cores (FP16 split of each chunk, an entry good to
// ~1e-6 of the entry's scale), then the fixed-order sum over the chunks.
cudaError_t launch_gram(const GramBatch& batch, cudaStream_t stream);

// ---- (a) projection -------------------------------------------------------
struct ProjProblem {
  float* P;         // k x r
  int64_t k;
  uint32_t layer;
  float scale;      // QR: sqrt(k / r) rounded to fp32; Rademacher: 1/sqrt(r)
  float2* partials; // QR: nchunks(k) x r x r (hi, lo) pairs
  double* gram;     // QR: r x r
  float* rinv;      // QR: r x r
  double* wide;     // QR with r <= k < 4r: two k x r fp64 arrays (the others unused)
  uint32_t* amax;   // QR: bits of max |P| after the first triangular product
};
struct ProjBatch {
  int n;
  int r;
  uint64_t seed;
  uint32_t rk0[10], rk1[10];  // Philox round keys of the seed (philox_round_keys)
  uint32_t step;
  int32_t* status;  // one status word for the whole batch (QR breakdown flag)
  ProjProblem p[kMaxBatch];
};
// Workspace of one QR problem.
void carve_qr_workspace(WsCursor& cur, int64_t k, int r, ProjProblem* p);
// Frames with r <= k < 4r go to the fp64 Householder kernel, the rest to CholeskyQR2.
inline bool qr_is_wide(int64_t k, int64_t r) { return 4 * r > k; }
cudaError_t launch_wide_qr(const ProjBatch& batch, cudaStream_t stream);

cudaError_t launch_rademacher(const ProjBatch& batch, int64_t max_k, cudaStream_t stream);
cudaError_t launch_gaussian_qr(const ProjBatch& batch, int64_t max_k, cudaStream_t stream);

// ---- (b) projected inputs -------------------------------------------------
struct ProjectProblem {
  const uint16_t* X;  // T x k BF16, row stride ld_x
  int64_t T, k, ld_x;
  const float* P;     // k x r fp32
  uint16_t* XP;       // T x r BF16, row stride ld_xp
  int64_t ld_xp;
  const uint16_t* P_split;  // nullable: a ready split of P (2 n_pad x k BF16)
};
size_t project_workspace_bytes(int64_t T, int64_t k, int64_t r);
// P (k x r fp32) -> [hi(P^T); lo(P^T)] (2 n_pad x k BF16) for each problem.
cudaError_t launch_split_projection(int n, const float* const* P, const int64_t* k, uint16_t* const* out, int r,
                                    cudaStream_t stream);
// A group of projections of one k that share their inputs X: their split is
// that of the k x (m r) concatenation [P_0 | ... | P_{m-1}], so one projection
// call with rank m r reads X once for all of them.
constexpr int kMaxGroup = 16;
struct SplitGroup {
  const float* P[kMaxGroup];
  int m;
  int64_t k;
  uint16_t* out;
};
cudaError_t launch_split_projection_grouped(int n, const SplitGroup* groups, int r, cudaStream_t stream);
// Workspace: the problems' regions of project_workspace_bytes, back to back.
// xp_split: write XP as a BF16 pair (hi in columns [0, r), lo = bf16(XP - hi) at
// [n_pad, n_pad + r), n_pad = r rounded up to 16) instead of one BF16 rounding.
cudaError_t launch_project_inputs(int n, const ProjectProblem* probs, int r, void* ws, cudaStream_t stream,
                                  bool xp_split = false);

// ---- (c) sketch accumulation ----------------------------------------------
struct AccumulateProblem {
  const uint16_t* D;  // T x d BF16, row stride ld_d
  int64_t T, d, ld_d;
  const uint16_t* XP; // T x r BF16, row stride ld_xp
  int64_t ld_xp;
  float* C;           // d x r fp32
};
size_t accumulate_workspace_bytes(int64_t T, int64_t d, int64_t r);
// xp_split: XP is the BF16 pair launch_project_inputs writes with xp_split.
cudaError_t launch_accumulate(int n, const AccumulateProblem* probs, int r, int overwrite, cudaStream_t stream,
                              bool xp_split = false);

// ---- (d) rebuild + update -------------------------------------------------
struct UpdateProblem {
  uint16_t* W;        // d x k BF16, row stride ld_w
  int64_t d, k, ld_w;
  const float* C;     // d x r fp32
  const float* P;     // k x r fp32
  uint32_t layer;
  const double* wnorm2_in;
  double* wnorm2_out;
  int32_t* dev_status;
};
struct UpdateWorkspace {
  float2* gram_partials_p; // gram_chunks_tc(k, r).nchunks x r x r
  float2* gram_partials_c; // gram_chunks_tc(d, r).nchunks x r x r
  double* gram_p;          // r x r
  double* gram_c;          // r x r
  float* c_norm;           // d: Euclidean norm of each row of C
  float* p_norm;           // k: Euclidean norm of each row of P
  float* c_unscale;        // d: 2^-e of each row's FP16 split of C (NaN: no usable scale)
  float* p_unscale;        // ceil(k / 128): 2^-f of each 128-row block's FP16 split of P
  double* wnorm_partials;  // kWnormBlocks
  float* scale;            // the step scale s
  int32_t* status;         // scratch status when the caller passes none
  uint32_t* ticket;        // last-block counter of the update kernel
  double* wnew_partials;   // one per update block
  uint16_t* c_split;       // d x (2 r_pad) FP16: [high | low] part of C, each row scaled by 2^e
  uint16_t* p_split;       // k x (2 r_pad) FP16: [high | low] part of P, 2^f per 128 rows
  // exact-path tags: the groups whose flagged elements the fix kernel recomputes
  uint8_t* fix_counts;     // per (tile, epilogue warp): tags written
  uint16_t* fix_tags;      // per (tile, warp): up to 128 tags (flagged elements, lane, group)
  uint32_t* fix_ticket;    // bit 31: a non-finite change; the fix kernel's block counter
  unsigned long long* fix_acc;  // fixed-point sum of the exact path's changes of ||W_new||^2
};
constexpr int kWnormBlocks = 1024;
// Carves one layer's workspace at the cursor; returns its size (a multiple of 256).
size_t carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd, UpdateWorkspace* ws);

cudaError_t launch_update_normsgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float tau,
                                  uint64_t seed, uint32_t step, cudaStream_t stream);
cudaError_t launch_update_sgd(int n, const UpdateProblem* probs, const UpdateWorkspace* ws, int r, float alpha_eta,
                              uint64_t seed, uint32_t step, cudaStream_t stream);

}  // namespace rgs
