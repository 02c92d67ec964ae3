// C ABI of the sketching library: argument checks, workspace carving and
// dispatch to the kernels.  Every check happens on the host before anything is
// launched; see include/sketch.h for the contract of each entry point.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "sketch.h"

namespace {

thread_local char g_last_error[512] = "";

sketch_status fail(sketch_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

sketch_status ok() {
  g_last_error[0] = '\0';
  return SKETCH_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define CHECK_PTR(p)                                                                   \
  do {                                                                                 \
    if ((p) == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "%s is NULL", #p);         \
    if (!aligned16(p)) return fail(SKETCH_ERR_INVALID_ARG, "%s is not 16-byte aligned", #p); \
  } while (0)

#define CHECK_OPT_ALIGN(p, a)                                                          \
  do {                                                                                 \
    if ((p) != nullptr && (reinterpret_cast<uintptr_t>(p) % (a)) != 0)                \
      return fail(SKETCH_ERR_INVALID_ARG, "%s is not %d-byte aligned", #p, (int)(a));  \
  } while (0)

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

sketch_status check_dim(const char* name, int64_t v) {
  if (v < 1 || v > kMaxDim) return fail(SKETCH_ERR_INVALID_ARG, "%s=%lld out of [1, 2^31)", name, (long long)v);
  return SKETCH_OK;
}

sketch_status check_rank(int64_t r) {
  if (r < 1 || r > rgs::kMaxRank)
    return fail(SKETCH_ERR_INVALID_ARG, "r=%lld out of [1, %d]", (long long)r, rgs::kMaxRank);
  return SKETCH_OK;
}

sketch_status check_ld(const char* name, int64_t ld, int64_t width) {
  if (ld < width) return fail(SKETCH_ERR_INVALID_ARG, "%s=%lld < row width %lld", name, (long long)ld, (long long)width);
  if (ld % 8 != 0) return fail(SKETCH_ERR_INVALID_ARG, "%s=%lld is not a multiple of 8", name, (long long)ld);
  if (ld > kMaxDim) return fail(SKETCH_ERR_INVALID_ARG, "%s=%lld too large", name, (long long)ld);
  return SKETCH_OK;
}

sketch_status check_k(int64_t k) {
  sketch_status st = check_dim("k", k);
  if (st) return st;
  if (k % 8 != 0) return fail(SKETCH_ERR_INVALID_ARG, "k=%lld is not a multiple of 8", (long long)k);
  return SKETCH_OK;
}

sketch_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return SKETCH_OK;
  if (ws == nullptr) return fail(SKETCH_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL", need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(SKETCH_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (ws_bytes < need) return fail(SKETCH_ERR_WORKSPACE, "workspace %zu bytes < required %zu", ws_bytes, need);
  return SKETCH_OK;
}

sketch_status launch_result(cudaError_t err, const char* what) {
  if (err != cudaSuccess) return fail(SKETCH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
  return ok();
}

#define TRY(expr)                  \
  do {                             \
    sketch_status st_ = (expr);    \
    if (st_ != SKETCH_OK) return st_; \
  } while (0)

size_t sample_ws_bytes(sketch_proj_kind kind, int64_t k, int64_t r) {
  if (kind != SKETCH_PROJ_GAUSSIAN_QR) return 0;
  rgs::WsCursor cur;
  rgs::carve_qr_workspace(cur, k, (int)r, nullptr);
  cur.take<int32_t>(1);  // scratch status word
  return cur.offset;
}

size_t update_ws_bytes(bool normsgd, int64_t d, int64_t k, int64_t r) {
  if (!normsgd) return 0;
  rgs::WsCursor cur;
  rgs::carve_update_workspace(cur, d, k, (int)r, true, nullptr);
  return cur.offset;
}

}  // namespace

extern "C" {

const char* sketch_status_string(sketch_status status) {
  switch (status) {
    case SKETCH_OK: return "ok";
    case SKETCH_ERR_INVALID_ARG: return "invalid argument";
    case SKETCH_ERR_UNSUPPORTED: return "unsupported";
    case SKETCH_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SKETCH_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* sketch_last_error(void) { return g_last_error; }

size_t sketch_workspace_bytes(sketch_op op, int64_t T, int64_t d, int64_t k, int64_t r) {
  if (r < 1 || r > rgs::kMaxRank) return 0;
  switch (op) {
    case SKETCH_OP_SAMPLE_PROJECTION:
      return (k >= 1) ? sample_ws_bytes(SKETCH_PROJ_GAUSSIAN_QR, k, r) : 0;
    case SKETCH_OP_PROJECT_INPUTS:
      return (T >= 1 && k >= 1) ? rgs::project_workspace_bytes(T, k, r) : 0;
    case SKETCH_OP_ACCUMULATE:
      return (T >= 1 && d >= 1) ? rgs::accumulate_workspace_bytes(T, d, r) : 0;
    case SKETCH_OP_UPDATE_NORMSGD:
      return (d >= 1 && k >= 1) ? update_ws_bytes(true, d, k, r) : 0;
    case SKETCH_OP_UPDATE_SGD:
      return 0;
  }
  return 0;
}

sketch_status sketch_sample_projection(sketch_proj_kind kind, uint64_t seed, uint32_t layer,
                                       uint32_t step, int64_t k, int64_t r, float* P,
                                       int32_t* dev_status, void* ws, size_t ws_bytes,
                                       void* stream) {
  if (kind != SKETCH_PROJ_RADEMACHER && kind != SKETCH_PROJ_GAUSSIAN_QR)
    return fail(SKETCH_ERR_INVALID_ARG, "unknown projection kind %d", (int)kind);
  TRY(check_k(k));
  TRY(check_rank(r));
  CHECK_PTR(P);
  CHECK_OPT_ALIGN(dev_status, 4);
  if (k * r > (int64_t(1) << 34)) return fail(SKETCH_ERR_INVALID_ARG, "k*r too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rgs::ProjBatch storage;
  rgs::ProjBatch* batch = &storage;
  batch->n = 1;
  batch->r = (int)r;
  batch->seed = seed;
  batch->step = step;
  rgs::ProjProblem& pb = batch->p[0];
  pb.P = P;
  pb.k = k;
  pb.layer = layer;
  cudaError_t err;
  if (kind == SKETCH_PROJ_RADEMACHER) {
    pb.scale = (float)(1.0 / std::sqrt((double)r));
    if (dev_status) {
      err = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s);
      if (err != cudaSuccess) return launch_result(err, "sample_projection");
    }
    err = rgs::launch_rademacher(*batch, k, s);
    return launch_result(err, "sample_projection (Rademacher)");
  }
  if (4 * r > k) {
    return fail(SKETCH_ERR_UNSUPPORTED, "Gaussian-QR projection needs 4*r <= k (k=%lld, r=%lld)",
                (long long)k, (long long)r);
  }
  const size_t need = sample_ws_bytes(kind, k, r);
  sketch_status st = check_ws(ws, ws_bytes, need);
  if (st) return st;
  rgs::WsCursor cur;
  cur.base = static_cast<char*>(ws);
  rgs::carve_qr_workspace(cur, k, (int)r, &pb);
  int32_t* scratch_status = cur.take<int32_t>(1);
  pb.scale = (float)std::sqrt((double)k / (double)r);
  batch->status = dev_status ? dev_status : scratch_status;
  err = cudaMemsetAsync(batch->status, 0, sizeof(int32_t), s);
  if (err == cudaSuccess) err = rgs::launch_gaussian_qr(*batch, k, s);
  return launch_result(err, "sample_projection (Gaussian QR)");
}

sketch_status sketch_project_inputs(const uint16_t* X, int64_t T, int64_t k, int64_t ld_x,
                                    const float* P, int64_t r, uint16_t* XP, int64_t ld_xp,
                                    void* ws, size_t ws_bytes, void* stream) {
  TRY(check_dim("T", T));
  TRY(check_k(k));
  TRY(check_rank(r));
  TRY(check_ld("ld_x", ld_x, k));
  TRY(check_ld("ld_xp", ld_xp, r));
  CHECK_PTR(X);
  CHECK_PTR(P);
  CHECK_PTR(XP);
  TRY(check_ws(ws, ws_bytes, rgs::project_workspace_bytes(T, k, r)));
  cudaError_t err = rgs::launch_project_inputs(X, T, k, ld_x, P, (int)r, XP, ld_xp, ws,
                                               static_cast<cudaStream_t>(stream));
  return launch_result(err, "project_inputs");
}

sketch_status sketch_accumulate(const uint16_t* D, int64_t T, int64_t d, int64_t ld_d,
                                const uint16_t* XP, int64_t ld_xp, int64_t r, float* C,
                                int overwrite, void* ws, size_t ws_bytes, void* stream) {
  TRY(check_dim("T", T));
  TRY(check_dim("d", d));
  TRY(check_rank(r));
  TRY(check_ld("ld_d", ld_d, d));
  TRY(check_ld("ld_xp", ld_xp, r));
  CHECK_PTR(D);
  CHECK_PTR(XP);
  CHECK_PTR(C);
  if (overwrite != 0 && overwrite != 1) return fail(SKETCH_ERR_INVALID_ARG, "overwrite must be 0 or 1");
  TRY(check_ws(ws, ws_bytes, rgs::accumulate_workspace_bytes(T, d, r)));
  cudaError_t err = rgs::launch_accumulate(D, T, d, ld_d, XP, ld_xp, (int)r, C, overwrite, ws,
                                           static_cast<cudaStream_t>(stream));
  return launch_result(err, "accumulate");
}

static sketch_status check_update_args(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                       const float* C, const float* P, int64_t r) {
  TRY(check_dim("d", d));
  TRY(check_k(k));
  TRY(check_rank(r));
  TRY(check_ld("ld_w", ld_w, k));
  CHECK_PTR(W);
  CHECK_PTR(C);
  CHECK_PTR(P);
  if (d * k >= (int64_t(1) << 40)) return fail(SKETCH_ERR_INVALID_ARG, "d*k too large");
  if ((d * k) / 8 > (int64_t)UINT32_MAX)
    return fail(SKETCH_ERR_INVALID_ARG, "d*k exceeds the 2^35 weights one rounding stream covers");
  return SKETCH_OK;
}

sketch_status sketch_apply_update_normsgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                          const float* C, const float* P, int64_t r, float tau,
                                          uint64_t seed, uint32_t layer, uint32_t step,
                                          const double* wnorm2_in, double* wnorm2_out,
                                          int32_t* dev_status, void* ws, size_t ws_bytes,
                                          void* stream) {
  TRY(check_update_args(W, d, k, ld_w, C, P, r));
  CHECK_OPT_ALIGN(wnorm2_in, 8);
  CHECK_OPT_ALIGN(wnorm2_out, 8);
  CHECK_OPT_ALIGN(dev_status, 4);
  if (!std::isfinite(tau)) return fail(SKETCH_ERR_INVALID_ARG, "tau is not finite");
  const size_t need = update_ws_bytes(true, d, k, r);
  TRY(check_ws(ws, ws_bytes, need));
  rgs::WsCursor cur;
  cur.base = static_cast<char*>(ws);
  rgs::UpdateWorkspace uw;
  rgs::carve_update_workspace(cur, d, k, (int)r, true, &uw);
  cudaError_t err = rgs::launch_update_normsgd(W, d, k, ld_w, C, P, (int)r, tau, seed, layer, step,
                                               wnorm2_in, wnorm2_out, dev_status, uw,
                                               static_cast<cudaStream_t>(stream));
  return launch_result(err, "apply_update_normsgd");
}

sketch_status sketch_apply_update_sgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                      const float* C, const float* P, int64_t r, float alpha_eta,
                                      uint64_t seed, uint32_t layer, uint32_t step,
                                      int32_t* dev_status, void* ws, size_t ws_bytes,
                                      void* stream) {
  (void)ws;
  (void)ws_bytes;
  TRY(check_update_args(W, d, k, ld_w, C, P, r));
  CHECK_OPT_ALIGN(dev_status, 4);
  if (!std::isfinite(alpha_eta)) return fail(SKETCH_ERR_INVALID_ARG, "alpha_eta is not finite");
  cudaError_t err = rgs::launch_update_sgd(W, d, k, ld_w, C, P, (int)r, alpha_eta, seed, layer, step,
                                           dev_status, static_cast<cudaStream_t>(stream));
  return launch_result(err, "apply_update_sgd");
}

}  // extern "C"
