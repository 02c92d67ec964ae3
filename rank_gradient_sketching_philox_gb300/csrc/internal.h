// Internal interface between the C ABI (abi.cu) and the kernel files.
// Arguments have been validated by the caller; these functions only launch.
#pragma once

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

// Row chunking of a partial Gram matrix over `rows` rows: at most 64 chunks.
struct GramChunks {
  int nchunks;
  int chunk_rows;
};
__host__ __device__ inline GramChunks gram_chunks(int64_t rows) {
  int64_t n = (rows + 127) / 128;
  if (n > 64) n = 64;
  if (n < 1) n = 1;
  GramChunks g;
  g.nchunks = (int)n;
  g.chunk_rows = (int)((rows + n - 1) / n);
  return g;
}

// ---- Gram matrices of tall-skinny fp32 matrices ----------------------------
struct GramEntry {
  const float* A;   // rows x r, row-major
  int64_t rows;
  float* partials;  // gram_chunks(rows).nchunks x r x r
  float* out;       // r x r
};
struct GramBatch {
  int n;
  int r;
  GramEntry e[kMaxBatch];
};
cudaError_t launch_gram(const GramBatch& batch, cudaStream_t stream);

// ---- (a) projection -------------------------------------------------------
struct ProjProblem {
  float* P;         // k x r
  int64_t k;
  uint32_t layer;
  float scale;      // QR: sqrt(k / r) rounded to fp32; Rademacher: 1/sqrt(r)
  float* partials;  // QR: nchunks(k) x r x r
  float* gram;      // QR: r x r
  float* rinv;      // QR: r x r
};
struct ProjBatch {
  int n;
  int r;
  uint64_t seed;
  uint32_t step;
  int32_t* status;  // one status word for the whole batch (QR breakdown flag)
  ProjProblem p[kMaxBatch];
};
// Workspace of one QR problem.
void carve_qr_workspace(WsCursor& cur, int64_t k, int r, ProjProblem* p);

cudaError_t launch_rademacher(const ProjBatch& batch, int64_t max_k, cudaStream_t stream);
cudaError_t launch_gaussian_qr(const ProjBatch& batch, int64_t max_k, cudaStream_t stream);

// ---- (b) projected inputs -------------------------------------------------
size_t project_workspace_bytes(int64_t T, int64_t k, int64_t r);
cudaError_t launch_project_inputs(const uint16_t* X, int64_t T, int64_t k, int64_t ld_x,
                                  const float* P, int r, uint16_t* XP, int64_t ld_xp, void* ws,
                                  cudaStream_t stream);

// ---- (c) sketch accumulation ----------------------------------------------
size_t accumulate_workspace_bytes(int64_t T, int64_t d, int64_t r);
cudaError_t launch_accumulate(const uint16_t* D, int64_t T, int64_t d, int64_t ld_d,
                              const uint16_t* XP, int64_t ld_xp, int r, float* C, int overwrite,
                              void* ws, cudaStream_t stream);

// ---- (d) rebuild + update -------------------------------------------------
struct UpdateWorkspace {
  float* gram_partials_p;  // nchunks(k) x r x r
  float* gram_partials_c;  // nchunks(d) x r x r
  float* gram_p;           // r x r
  float* gram_c;           // r x r
  double* wnorm_partials;  // kWnormBlocks
  double* wnew_partials;   // one per update block
  float* scale;            // the step scale s
  int32_t* status;         // scratch status when the caller passes none
  uint32_t* ticket;        // last-block counter of the update kernel
};
constexpr int kWnormBlocks = 1024;
void carve_update_workspace(WsCursor& cur, int64_t d, int64_t k, int r, bool normsgd,
                            UpdateWorkspace* ws);

cudaError_t launch_update_normsgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                                  const float* P, int r, float tau, uint64_t seed, uint32_t layer,
                                  uint32_t step, const double* wnorm2_in, double* wnorm2_out,
                                  int32_t* dev_status, const UpdateWorkspace& ws,
                                  cudaStream_t stream);
cudaError_t launch_update_sgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                              const float* P, int r, float alpha_eta, uint64_t seed,
                              uint32_t layer, uint32_t step, int32_t* dev_status,
                              cudaStream_t stream);

}  // namespace rgs
