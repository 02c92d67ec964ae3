// C ABI of the sketching library: argument checks, workspace carving and
// dispatch to the kernels.  Every check happens on the host before anything is
// launched; see include/sketch.h for the contract of each entry point.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

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

size_t qr_ws_bytes(int64_t k, int64_t r) {
  rgs::WsCursor cur;
  rgs::carve_qr_workspace(cur, k, (int)r, nullptr);
  cur.take<int32_t>(1);  // scratch status word
  cur.take<char>(0);
  return cur.offset;
}

size_t update_ws_bytes(bool normsgd, int64_t d, int64_t k, int64_t r) {
  rgs::WsCursor cur;
  return rgs::carve_update_workspace(cur, d, k, (int)r, normsgd, nullptr);
}

size_t op_ws_bytes(sketch_op op, int64_t T, int64_t d, int64_t k, int64_t r) {
  if (r < 1 || r > rgs::kMaxRank) return 0;
  switch (op) {
    case SKETCH_OP_SAMPLE_PROJECTION: return (k >= 1) ? qr_ws_bytes(k, r) : 0;
    case SKETCH_OP_PROJECT_INPUTS: return (T >= 1 && k >= 1) ? rgs::project_workspace_bytes(T, k, r) : 0;
    case SKETCH_OP_ACCUMULATE: return (T >= 1 && d >= 1) ? rgs::accumulate_workspace_bytes(T, d, r) : 0;
    case SKETCH_OP_UPDATE_NORMSGD: return (d >= 1 && k >= 1) ? update_ws_bytes(true, d, k, r) : 0;
    case SKETCH_OP_UPDATE_SGD: return (d >= 1 && k >= 1) ? update_ws_bytes(false, d, k, r) : 0;
  }
  return 0;
}

sketch_status check_n(int n) {
  if (n < 1 || n > (1 << 20)) return fail(SKETCH_ERR_INVALID_ARG, "n=%d out of [1, 2^20]", n);
  return SKETCH_OK;
}

// ---- per-problem checks ------------------------------------------------------
sketch_status check_projection(const sketch_projection_problem& p) {
  TRY(check_k(p.k));
  CHECK_PTR(p.P);
  return SKETCH_OK;
}

sketch_status check_project(const sketch_project_problem& p, int64_t r) {
  TRY(check_dim("T", p.T));
  TRY(check_k(p.k));
  TRY(check_ld("ld_x", p.ld_x, p.k));
  TRY(check_ld("ld_xp", p.ld_xp, r));
  CHECK_PTR(p.X);
  if (p.P == nullptr && p.P_split == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "P and P_split are both NULL");
  CHECK_PTR(p.XP);
  return SKETCH_OK;
}

sketch_status check_accumulate(const sketch_accumulate_problem& p, int64_t r) {
  TRY(check_dim("T", p.T));
  TRY(check_dim("d", p.d));
  TRY(check_ld("ld_d", p.ld_d, p.d));
  TRY(check_ld("ld_xp", p.ld_xp, r));
  CHECK_PTR(p.D);
  CHECK_PTR(p.XP);
  CHECK_PTR(p.C);
  return SKETCH_OK;
}

sketch_status check_update(const sketch_update_problem& p) {
  TRY(check_dim("d", p.d));
  TRY(check_k(p.k));
  TRY(check_ld("ld_w", p.ld_w, p.k));
  CHECK_PTR(p.W);
  CHECK_PTR(p.C);
  CHECK_PTR(p.P);
  CHECK_OPT_ALIGN(p.wnorm2_in, 8);
  CHECK_OPT_ALIGN(p.wnorm2_out, 8);
  CHECK_OPT_ALIGN(p.dev_status, 4);
  if (p.d * p.k >= (int64_t(1) << 40)) return fail(SKETCH_ERR_INVALID_ARG, "d*k too large");
  if ((p.d * p.k) / 8 > (int64_t)UINT32_MAX)
    return fail(SKETCH_ERR_INVALID_ARG, "d*k exceeds the 2^35 weights one rounding stream covers");
  return SKETCH_OK;
}

// ---- batched implementations --------------------------------------------------
sketch_status do_sample(sketch_proj_kind kind, uint64_t seed, uint32_t step, int n,
                        const sketch_projection_problem* probs, int64_t r, int32_t* dev_status, void* ws,
                        size_t ws_bytes, cudaStream_t s) {
  if (kind != SKETCH_PROJ_RADEMACHER && kind != SKETCH_PROJ_GAUSSIAN_QR)
    return fail(SKETCH_ERR_INVALID_ARG, "unknown projection kind %d", (int)kind);
  TRY(check_n(n));
  if (probs == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "problems is NULL");
  TRY(check_rank(r));
  CHECK_OPT_ALIGN(dev_status, 4);
  size_t need = 0;
  for (int i = 0; i < n; ++i) {
    TRY(check_projection(probs[i]));
    if (probs[i].k * r > (int64_t(1) << 34)) return fail(SKETCH_ERR_INVALID_ARG, "k*r too large");
    if (kind == SKETCH_PROJ_GAUSSIAN_QR) {
      if (r > probs[i].k)
        return fail(SKETCH_ERR_INVALID_ARG, "Gaussian-QR projection needs r <= k (k=%lld, r=%lld)",
                    (long long)probs[i].k, (long long)r);
      need += qr_ws_bytes(probs[i].k, r);
    }
  }
  if (kind == SKETCH_PROJ_GAUSSIAN_QR) TRY(check_ws(ws, ws_bytes, need));
  // Up to two batches are filled at once: CholeskyQR2 frames (and Rademacher
  // draws) in `batch`, fp64 Householder frames (r <= k < 4r) in `wide`; each is
  // launched when full and at the end.
  static thread_local rgs::ProjBatch batch, wide;
  for (rgs::ProjBatch* b : {&batch, &wide}) {
    b->n = 0;
    b->r = (int)r;
    b->seed = seed;
    rgs::philox_round_keys(seed, b->rk0, b->rk1);
    b->step = step;
  }
  rgs::WsCursor cur;
  cur.base = static_cast<char*>(ws);
  int32_t* status = dev_status;
  cudaError_t err = cudaSuccess;
  int64_t max_k = 0;
  auto flush = [&](rgs::ProjBatch& b) {
    if (b.n == 0 || err != cudaSuccess) return;
    if (kind == SKETCH_PROJ_RADEMACHER) {
      err = rgs::launch_rademacher(b, max_k, s);
    } else {
      b.status = status;
      err = (&b == &wide) ? rgs::launch_wide_qr(b, s) : rgs::launch_gaussian_qr(b, max_k, s);
    }
    if (&b == &batch) max_k = 0;
    b.n = 0;
  };
  for (int i = 0; i < n && err == cudaSuccess; ++i) {
    const sketch_projection_problem& pr = probs[i];
    const bool is_wide = kind == SKETCH_PROJ_GAUSSIAN_QR && rgs::qr_is_wide(pr.k, r);
    rgs::ProjBatch& b = is_wide ? wide : batch;
    rgs::ProjProblem& pb = b.p[b.n++];
    pb.P = pr.P;
    pb.k = pr.k;
    pb.layer = pr.layer;
    if (kind == SKETCH_PROJ_RADEMACHER) {
      pb.scale = (float)(1.0 / std::sqrt((double)r));
    } else {
      rgs::carve_qr_workspace(cur, pr.k, (int)r, &pb);
      int32_t* scratch = cur.take<int32_t>(1);
      cur.take<char>(0);
      if (status == nullptr) status = scratch;
      pb.scale = (float)std::sqrt((double)pr.k / (double)r);
      if (i == 0) err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    }
    if (!is_wide) max_k = pr.k > max_k ? pr.k : max_k;
    if (b.n == rgs::kMaxBatch) flush(b);
  }
  flush(batch);
  flush(wide);
  if (err == cudaSuccess && kind == SKETCH_PROJ_RADEMACHER && dev_status)
    err = cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s);
  return launch_result(err, "sample_projection");
}

// XP width: r columns, or the BF16 pair of the fp32-accurate form (2 * round16(r)).
int64_t xp_width(int64_t r, bool xp_split) { return xp_split ? 2 * ((r + 15) / 16 * 16) : r; }

sketch_status do_project(int n, const sketch_project_problem* probs, int64_t r, void* ws, size_t ws_bytes,
                         cudaStream_t s, bool xp_split = false) {
  TRY(check_n(n));
  if (probs == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "problems is NULL");
  TRY(check_rank(r));
  size_t need = 0;
  std::vector<rgs::ProjectProblem> v((size_t)n);
  for (int i = 0; i < n; ++i) {
    TRY(check_project(probs[i], r));
    TRY(check_ld("ld_xp", probs[i].ld_xp, xp_width(r, xp_split)));
    need += rgs::project_workspace_bytes(probs[i].T, probs[i].k, r);
    v[i] = rgs::ProjectProblem{probs[i].X, probs[i].T, probs[i].k, probs[i].ld_x, probs[i].P, probs[i].XP,
                               probs[i].ld_xp, probs[i].P_split};
  }
  TRY(check_ws(ws, ws_bytes, need));
  return launch_result(rgs::launch_project_inputs(n, v.data(), (int)r, ws, s, xp_split), "project_inputs");
}

sketch_status do_accumulate(int n, const sketch_accumulate_problem* probs, int64_t r, int overwrite, void* ws,
                            size_t ws_bytes, cudaStream_t s, bool xp_split = false) {
  TRY(check_n(n));
  if (probs == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "problems is NULL");
  TRY(check_rank(r));
  if (overwrite != 0 && overwrite != 1) return fail(SKETCH_ERR_INVALID_ARG, "overwrite must be 0 or 1");
  size_t need = 0;
  std::vector<rgs::AccumulateProblem> v((size_t)n);
  for (int i = 0; i < n; ++i) {
    TRY(check_accumulate(probs[i], r));
    TRY(check_ld("ld_xp", probs[i].ld_xp, xp_width(r, xp_split)));
    need += rgs::accumulate_workspace_bytes(probs[i].T, probs[i].d, r);
    v[i] = rgs::AccumulateProblem{probs[i].D, probs[i].T, probs[i].d, probs[i].ld_d, probs[i].XP, probs[i].ld_xp,
                                  probs[i].C};
  }
  TRY(check_ws(ws, ws_bytes, need));
  return launch_result(rgs::launch_accumulate(n, v.data(), (int)r, overwrite, s, xp_split), "accumulate");
}

sketch_status do_update(bool normsgd, int n, const sketch_update_problem* probs, int64_t r, float step_size,
                        uint64_t seed, uint32_t step, void* ws, size_t ws_bytes, cudaStream_t s) {
  TRY(check_n(n));
  if (probs == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "problems is NULL");
  TRY(check_rank(r));
  if (!std::isfinite(step_size)) return fail(SKETCH_ERR_INVALID_ARG, "%s is not finite", normsgd ? "tau" : "alpha_eta");
  size_t need = 0;
  for (int i = 0; i < n; ++i) {
    TRY(check_update(probs[i]));
    need += update_ws_bytes(normsgd, probs[i].d, probs[i].k, r);
  }
  TRY(check_ws(ws, ws_bytes, need));
  std::vector<rgs::UpdateProblem> v((size_t)n);
  std::vector<rgs::UpdateWorkspace> w((size_t)n);
  rgs::WsCursor cur;
  cur.base = static_cast<char*>(ws);
  for (int i = 0; i < n; ++i) {
    const sketch_update_problem& p = probs[i];
    v[i] = rgs::UpdateProblem{p.W, p.d, p.k, p.ld_w, p.C, p.P, p.layer,
                              normsgd ? p.wnorm2_in : nullptr, normsgd ? p.wnorm2_out : nullptr, p.dev_status};
    rgs::carve_update_workspace(cur, p.d, p.k, (int)r, normsgd, &w[i]);
  }
  cudaError_t err = normsgd ? rgs::launch_update_normsgd(n, v.data(), w.data(), (int)r, step_size, seed, step, s)
                            : rgs::launch_update_sgd(n, v.data(), w.data(), (int)r, step_size, seed, step, s);
  return launch_result(err, normsgd ? "apply_update_normsgd" : "apply_update_sgd");
}

}  // namespace

namespace rgs {
void set_last_error(const char* message) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", message);
}
}  // namespace rgs

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
  return op_ws_bytes(op, T, d, k, r);
}

size_t sketch_workspace_bytes_batched(sketch_op op, int n, const int64_t* T, const int64_t* d, const int64_t* k,
                                      int64_t r) {
  size_t total = 0;
  for (int i = 0; i < n; ++i)
    total += op_ws_bytes(op, T ? T[i] : 0, d ? d[i] : 0, k ? k[i] : 0, r);
  return total;
}

sketch_status sketch_sample_projection(sketch_proj_kind kind, uint64_t seed, uint32_t layer, uint32_t step,
                                       int64_t k, int64_t r, float* P, int32_t* dev_status, void* ws,
                                       size_t ws_bytes, void* stream) {
  const sketch_projection_problem p{P, k, layer};
  return do_sample(kind, seed, step, 1, &p, r, dev_status, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_sample_projection_batched(sketch_proj_kind kind, uint64_t seed, uint32_t step, int n,
                                               const sketch_projection_problem* problems, int64_t r,
                                               int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  return do_sample(kind, seed, step, n, problems, r, dev_status, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_project_inputs(const uint16_t* X, int64_t T, int64_t k, int64_t ld_x, const float* P,
                                    int64_t r, uint16_t* XP, int64_t ld_xp, void* ws, size_t ws_bytes,
                                    void* stream) {
  const sketch_project_problem p{X, T, k, ld_x, P, XP, ld_xp};
  return do_project(1, &p, r, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_project_inputs_batched(int n, const sketch_project_problem* problems, int64_t r, void* ws,
                                            size_t ws_bytes, void* stream) {
  return do_project(n, problems, r, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_project_inputs_fp32xp_batched(int n, const sketch_project_problem* problems, int64_t r,
                                                   void* ws, size_t ws_bytes, void* stream) {
  return do_project(n, problems, r, ws, ws_bytes, static_cast<cudaStream_t>(stream), true);
}

sketch_status sketch_accumulate_fp32xp_batched(int n, const sketch_accumulate_problem* problems, int64_t r,
                                               int overwrite, void* ws, size_t ws_bytes, void* stream) {
  return do_accumulate(n, problems, r, overwrite, ws, ws_bytes, static_cast<cudaStream_t>(stream), true);
}

size_t sketch_projection_split_elems(int64_t k, int64_t r) {
  if (k < 1 || k > kMaxDim || k % 8 != 0 || r < 1 || r > rgs::kMaxRank) return 0;
  return (size_t)2 * (size_t)((r + 15) / 16 * 16) * (size_t)k;
}

sketch_status sketch_split_projection_batched(int n, const sketch_split_problem* problems, int64_t r,
                                              void* stream) {
  TRY(check_n(n));
  if (problems == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "problems is NULL");
  TRY(check_rank(r));
  std::vector<const float*> P((size_t)n);
  std::vector<int64_t> k((size_t)n);
  std::vector<uint16_t*> out((size_t)n);
  for (int i = 0; i < n; ++i) {
    TRY(check_k(problems[i].k));
    CHECK_PTR(problems[i].P);
    CHECK_PTR(problems[i].P_split);
    P[i] = problems[i].P;
    k[i] = problems[i].k;
    out[i] = problems[i].P_split;
  }
  return launch_result(rgs::launch_split_projection(n, P.data(), k.data(), out.data(), (int)r,
                                                    static_cast<cudaStream_t>(stream)),
                       "split_projection");
}

sketch_status sketch_split_projection_grouped(int n, const sketch_split_group* groups, int64_t r, void* stream) {
  TRY(check_n(n));
  if (groups == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "groups is NULL");
  TRY(check_rank(r));
  std::vector<rgs::SplitGroup> g((size_t)n);
  for (int i = 0; i < n; ++i) {
    const sketch_split_group& gr = groups[i];
    if (gr.m < 1 || gr.m > rgs::kMaxGroup)
      return fail(SKETCH_ERR_INVALID_ARG, "group %d: m=%d out of [1, %d]", i, gr.m, rgs::kMaxGroup);
    if ((int64_t)gr.m * r > rgs::kMaxRank)
      return fail(SKETCH_ERR_INVALID_ARG, "group %d: m*r=%lld exceeds %d", i, (long long)gr.m * r, rgs::kMaxRank);
    if (gr.m > 1 && r % 8 != 0)
      return fail(SKETCH_ERR_INVALID_ARG, "group %d: r=%lld must be a multiple of 8 when m > 1", i, (long long)r);
    if (gr.P == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "group %d: P is NULL", i);
    TRY(check_k(gr.k));
    CHECK_PTR(gr.P_split);
    g[i].m = gr.m;
    g[i].k = gr.k;
    g[i].out = gr.P_split;
    for (int q = 0; q < gr.m; ++q) {
      CHECK_PTR(gr.P[q]);
      g[i].P[q] = gr.P[q];
    }
  }
  return launch_result(rgs::launch_split_projection_grouped(n, g.data(), (int)r, static_cast<cudaStream_t>(stream)),
                       "split_projection_grouped");
}

sketch_status sketch_accumulate(const uint16_t* D, int64_t T, int64_t d, int64_t ld_d, const uint16_t* XP,
                                int64_t ld_xp, int64_t r, float* C, int overwrite, void* ws, size_t ws_bytes,
                                void* stream) {
  const sketch_accumulate_problem p{D, T, d, ld_d, XP, ld_xp, C};
  return do_accumulate(1, &p, r, overwrite, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_accumulate_batched(int n, const sketch_accumulate_problem* problems, int64_t r, int overwrite,
                                        void* ws, size_t ws_bytes, void* stream) {
  return do_accumulate(n, problems, r, overwrite, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_apply_update_normsgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                                          const float* P, int64_t r, float tau, uint64_t seed, uint32_t layer,
                                          uint32_t step, const double* wnorm2_in, double* wnorm2_out,
                                          int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  const sketch_update_problem p{W, d, k, ld_w, C, P, layer, wnorm2_in, wnorm2_out, dev_status};
  return do_update(true, 1, &p, r, tau, seed, step, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_apply_update_normsgd_batched(int n, const sketch_update_problem* problems, int64_t r,
                                                  float tau, uint64_t seed, uint32_t step, void* ws,
                                                  size_t ws_bytes, void* stream) {
  return do_update(true, n, problems, r, tau, seed, step, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_apply_update_sgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w, const float* C,
                                      const float* P, int64_t r, float alpha_eta, uint64_t seed, uint32_t layer,
                                      uint32_t step, int32_t* dev_status, void* ws, size_t ws_bytes,
                                      void* stream) {
  const sketch_update_problem p{W, d, k, ld_w, C, P, layer, nullptr, nullptr, dev_status};
  return do_update(false, 1, &p, r, alpha_eta, seed, step, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

sketch_status sketch_apply_update_sgd_batched(int n, const sketch_update_problem* problems, int64_t r,
                                              float alpha_eta, uint64_t seed, uint32_t step, void* ws,
                                              size_t ws_bytes, void* stream) {
  return do_update(false, n, problems, r, alpha_eta, seed, step, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

uint64_t sketch_kernel_launches(void) { return rgs::launches_issued(); }

sketch_status sketch_read_device_errors(int32_t* flags, void* stream) {
  if (flags == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "flags is NULL");
  int* word = nullptr;
  cudaError_t err = rgs::device_error_word(&word);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (err == cudaSuccess) err = cudaMemcpyAsync(&host, word, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(word, 0, sizeof(int32_t), s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  *flags = host;
  return launch_result(err, "read_device_errors");
}

sketch_status sketch_read_exact_count(uint64_t* count, void* stream) {
  if (count == nullptr) return fail(SKETCH_ERR_INVALID_ARG, "count is NULL");
  unsigned long long* word = nullptr;
  cudaError_t err = rgs::device_exact_counter(&word);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long host = 0;
  if (err == cudaSuccess) err = cudaMemcpyAsync(&host, word, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(word, 0, sizeof(host), s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  *count = (uint64_t)host;
  return launch_result(err, "read_exact_count");
}

}  // extern "C"
