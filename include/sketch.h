/*
 * sketch.h -- C ABI of the GB300 (sm_103a) library for randomized low-rank
 * gradient sketching of linear layers (RGC / LoGRA).
 *
 * For a linear layer with weight W (d x k, out x in), input X (T x k) and
 * output derivative D (T x d), the weight gradient is G = D^T X.  The library
 * never forms G.  It
 *   (a) draws a seeded projection P (k x r),
 *   (b) forms the saved projected input XP = X P,
 *   (c) accumulates the fp32 sketch C += D^T (XP) over microbatches, and
 *   (d) rebuilds H = C P^T block by block, fused with the weight update, and
 *       writes W back to BF16 by stochastic rounding.
 * Sources (page title, section): "Randomized Gradient Compression" -- "How it
 * works" and footnote 1; "LoGRA: Scaling LLM Reinforcement Learning with
 * Low-Rank Gradient Sketches" -- Key Contributions 1 and 2; "LoGRA: Low-Rank
 * Gradient Sketches" -- "The Core Move", "Why the Sketch Can Be Accumulated
 * Without a Full Gradient", "Why the Update Is Low-Rank but Not an Exact
 * Recovery", "Why Refreshing the Projection Enables New Update Directions",
 * "Minimal Causal Code".  LoGRA's projection A (r x k) is P^T and its sketch
 * S is C.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named X, D, XP, W, C, P, ws, dev_status, wnorm2_* are DEVICE
 *   pointers on the current CUDA device.  BF16 tensors are passed as uint16_t
 *   bit patterns (the upper half of an IEEE fp32).
 * - Layouts are row-major.  P is k x r fp32 contiguous (row stride r).  C is
 *   d x r fp32 contiguous (row stride r).  X, D, XP, W have an explicit row
 *   stride in elements (ld_*), which must be >= the row width and a multiple
 *   of 8 (16 bytes); every pointer must be 16-byte aligned.
 * - Sizes: 1 <= r <= 256; k a multiple of 8; T, d, k >= 1 and < 2^31;
 *   d*k < 2^40.
 * - Ownership: the caller allocates and owns every buffer, including the
 *   workspace `ws` (query its size with sketch_workspace_bytes; pass NULL and
 *   0 when that size is 0).  The library allocates no memory and keeps no
 *   state between calls; it is safe to call from several host threads.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream).  Calls that share a workspace must be ordered on one
 *   stream.
 * - Errors: argument errors are found on the host, return a nonzero
 *   sketch_status and launch nothing.  A failed launch returns
 *   SKETCH_ERR_CUDA.  Data-dependent conditions found on the device (see
 *   SKETCH_DEV_*) are written to `dev_status`; nothing traps or spins.
 *   sketch_last_error() describes the last failure on the calling thread.
 * - Random bits: one Philox4x32-10 stream per (seed, layer, step, purpose);
 *   key = (seed low word, seed high word), counter = (block, step, layer,
 *   purpose).  Every output is a pure function of its inputs, so repeated
 *   calls and replicas produce bit-identical results.
 */
#ifndef RGS_SKETCH_H
#define RGS_SKETCH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SKETCH_API __attribute__((visibility("default")))
#else
#define SKETCH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SKETCH_OK = 0,
    SKETCH_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or stride */
    SKETCH_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels handle */
    SKETCH_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
    SKETCH_ERR_CUDA = 4          /* a CUDA call or kernel launch failed */
} sketch_status;

typedef enum {
    /* entries +-1/sqrt(r) from Philox sign bits ("LoGRA: Low-Rank Gradient
       Sketches", "Why the Sketch Can Be Accumulated Without a Full Gradient") */
    SKETCH_PROJ_RADEMACHER = 0,
    /* sqrt(k/r) * Q, Q the orthonormal factor of a k x r Gaussian matrix with
       the sign correction diag(R) > 0 ("Randomized Gradient Compression",
       footnote 1) */
    SKETCH_PROJ_GAUSSIAN_QR = 1
} sketch_proj_kind;

typedef enum {
    SKETCH_OP_SAMPLE_PROJECTION = 0,
    SKETCH_OP_PROJECT_INPUTS = 1,
    SKETCH_OP_ACCUMULATE = 2,
    SKETCH_OP_UPDATE_NORMSGD = 3,
    SKETCH_OP_UPDATE_SGD = 4
} sketch_op;

/* Bits of the device status word (int32) written by the update calls. */
#define SKETCH_DEV_H_ZERO 1        /* ||H||_F == 0: W left unchanged */
#define SKETCH_DEV_H_NONFINITE 2   /* ||H||_F is inf or NaN: W left unchanged */
#define SKETCH_DEV_W_NONFINITE 4   /* ||W||_F is inf or NaN: W left unchanged */
#define SKETCH_DEV_QR_BREAKDOWN 8  /* non-positive pivot in the QR Cholesky */

/* Workspace bytes the call `op` needs for these sizes (0 = none).  Arguments
 * that an op does not use are ignored.  Returns 0 for invalid sizes too; the
 * call itself reports those. */
SKETCH_API size_t sketch_workspace_bytes(sketch_op op, int64_t T, int64_t d, int64_t k, int64_t r);

/* (a) Draw the projection P (k x r fp32, row-major, written in full) for
 * (seed, layer, step).  A fixed projection uses a constant step; a projection
 * refreshed after every update uses the step counter ("Randomized Gradient
 * Compression", "How it works": a new random projection after every update;
 * "LoGRA: Low-Rank Gradient Sketches", "Why Refreshing the Projection
 * Enables New Update Directions").
 * SKETCH_PROJ_GAUSSIAN_QR needs r <= k (SKETCH_ERR_INVALID_ARG otherwise) and
 * a workspace.  For 4*r <= k the frame comes from CholeskyQR2 in fp32 (the
 * Gaussian matrix is then well conditioned; P^T P = (k/r) I to ~1e-6), and a
 * QR breakdown is reported in *dev_status (nullable) as
 * SKETCH_DEV_QR_BREAKDOWN.  For r <= k < 4*r, up to the square case r = k
 * where P P^T = I, it comes from Householder QR in fp64, one thread block per
 * problem (a few ms at the largest size), which cannot break down.
 * SKETCH_PROJ_RADEMACHER needs no workspace. */
SKETCH_API sketch_status sketch_sample_projection(sketch_proj_kind kind, uint64_t seed, uint32_t layer,
                                       uint32_t step, int64_t k, int64_t r, float* P,
                                       int32_t* dev_status, void* ws, size_t ws_bytes,
                                       void* stream);

/* (b) XP = X P rounded once to BF16 (round to nearest even) after fp32
 * accumulation.  X: T x k BF16 (row stride ld_x); P: k x r fp32; XP: T x r BF16
 * (row stride ld_xp), written in columns [0, r) only.  This is what the layer
 * saves for backpropagation instead of X ("Randomized Gradient Compression",
 * "How it works"). */
SKETCH_API sketch_status sketch_project_inputs(const uint16_t* X, int64_t T, int64_t k, int64_t ld_x,
                                    const float* P, int64_t r, uint16_t* XP, int64_t ld_xp,
                                    void* ws, size_t ws_bytes, void* stream);

/* (c) C = (overwrite ? 0 : C) + D^T XP in fp32, for one microbatch.  D: T x d
 * BF16 (row stride ld_d, token-major as produced by the backward pass);
 * XP: T x r BF16 (row stride ld_xp); C: d x r fp32, read (unless overwrite) and
 * written.  The dense d x k gradient is never formed ("Randomized
 * Gradient Compression", "How it works": C += D.T (X P); "LoGRA: Scaling LLM
 * Reinforcement Learning with Low-Rank Gradient Sketches", Key Contributions 1:
 * accumulated in fp32).  overwrite=1 on the first microbatch replaces zeroing
 * C ("LoGRA: Low-Rank Gradient Sketches", "Minimal Causal Code"). */
SKETCH_API sketch_status sketch_accumulate(const uint16_t* D, int64_t T, int64_t d, int64_t ld_d,
                                const uint16_t* XP, int64_t ld_xp, int64_t r, float* C,
                                int overwrite, void* ws, size_t ws_bytes, void* stream);

/* (d) Normalized SGD, W <- W - tau * ||W||_F * H / ||H||_F with H = C P^T
 * ("Randomized Gradient Compression", "How it works").  H is rebuilt 128 rows
 * at a time on chip and never stored; ||H||_F^2 = <P^T P, C^T C> comes from
 * two r x r Gram matrices.  The step scale s = fl32(tau*||W||/||H||) is
 * computed on the device (no host synchronisation).  Each weight becomes
 * v = fmaf(-s, H_ij, W_ij) and is written back by stochastic rounding with
 * 16 Philox bits of element index i*k + j.
 *   wnorm2_in  (nullable): ||W||_F^2 carried from the previous update of this
 *              W; when NULL the call reads W once more to compute it.
 *   wnorm2_out (nullable): receives ||W_new||_F^2 for the next call.
 *   dev_status (nullable): receives the SKETCH_DEV_* flags (0 = updated).
 * On a nonzero device status W is left bit-unchanged.  W: d x k BF16 (row
 * stride ld_w), updated in place; C: d x r fp32; P: k x r fp32. */
SKETCH_API sketch_status sketch_apply_update_normsgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                          const float* C, const float* P, int64_t r, float tau,
                                          uint64_t seed, uint32_t layer, uint32_t step,
                                          const double* wnorm2_in, double* wnorm2_out,
                                          int32_t* dev_status, void* ws, size_t ws_bytes,
                                          void* stream);

/* (d') LoGRA's basic SGD, W <- W - alpha_eta * S A with S = C and A = P^T
 * ("LoGRA: Low-Rank Gradient Sketches", "Why the Update Is Low-Rank but Not an
 * Exact Recovery"), with the same on-chip rebuild and stochastic rounding.
 * The receiver of a policy synchronisation applies the received factor U
 * with the received alpha_eta and the projection regenerated from the seed,
 * which gives the trainer's W bit for bit ("LoGRA: Scaling LLM Reinforcement
 * Learning with Low-Rank Gradient Sketches", Key Contributions 2).
 * dev_status (nullable) is set to 0. */
SKETCH_API sketch_status sketch_apply_update_sgd(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                      const float* C, const float* P, int64_t r, float alpha_eta,
                                      uint64_t seed, uint32_t layer, uint32_t step,
                                      int32_t* dev_status, void* ws, size_t ws_bytes,
                                      void* stream);

/* (d, without allocation) The normalized-SGD update of
 * sketch_apply_update_normsgd, same arguments and results, for callers that
 * cannot allocate device memory: a plugin handed only its input and output
 * buffers, or a process that has given all free device memory to another pool
 * (cudaMalloc would fail or stall the device there).  The method on the pages
 * has no counterpart to this entry point; it changes only where the scratch
 * lives.  The scratch is a fixed array of sketch_noalloc_scratch_bytes() (32
 * MiB) in device memory, reserved on each device that loads the library's
 * device code and held until the process exits.  Layers whose workspace,
 * sketch_workspace_bytes(SKETCH_OP_UPDATE_NORMSGD, 0, d, k, r), is larger are
 * rejected with SKETCH_ERR_WORKSPACE before anything is launched.  The first
 * call on a device looks up the array's device address (make that first call
 * before any stream capture).  All calls share the array: calls whose work
 * overlaps on the GPU race, so order them on one stream.  Nothing in the array
 * needs to start at zero.  With lazy module loading (CUDA's default) the
 * array is reserved when that first call looks up its address: a caller that
 * is about to give its free device memory to another pool should make one
 * call first (a call with d = 0 reserves the array and returns
 * SKETCH_ERR_INVALID_ARG without launching anything).  The looked-up address
 * is kept for the life of the process: after cudaDeviceReset() on a device,
 * do not call the library on that device again in the same process. */
SKETCH_API sketch_status sketch_apply_update_normsgd_noalloc(uint16_t* W, int64_t d, int64_t k, int64_t ld_w,
                                                             const float* C, const float* P, int64_t r,
                                                             float tau, uint64_t seed, uint32_t layer,
                                                             uint32_t step, const double* wnorm2_in,
                                                             double* wnorm2_out, int32_t* dev_status,
                                                             void* stream);
/* Size of the fixed scratch array of sketch_apply_update_normsgd_noalloc. */
SKETCH_API size_t sketch_noalloc_scratch_bytes(void);

/* ---- Batched forms ----------------------------------------------------------
 * One call covers many layers, one problem per layer, in a few kernel launches
 * (every layer's tiles share each launch, so small layers still fill the GPU).
 * Problems share r and, for the updates, the scale, seed and step; each
 * problem follows the contract of the single-layer call of the same name
 * (layouts, alignment, errors: a bad problem fails the whole call before
 * anything is launched).  `problems` is a HOST array of n >= 1 entries.  The
 * workspace is the concatenation of the problems' regions: its size is
 * sketch_workspace_bytes_batched, the sum of the per-problem sizes. */
typedef struct {
    float* P;          /* k x r fp32, written */
    int64_t k;
    uint32_t layer;
} sketch_projection_problem;

typedef struct {
    const uint16_t* X; /* T x k BF16 */
    int64_t T, k, ld_x;
    const float* P;    /* k x r fp32; may be NULL when P_split is given */
    uint16_t* XP;      /* T x r BF16, written */
    int64_t ld_xp;
    /* nullable: the split of P made by sketch_split_projection_batched for
     * this k and r; the call then reads it instead of splitting P again */
    const uint16_t* P_split;
} sketch_project_problem;

/* One projection to split: P (k x r fp32) into P_split, which holds
 * sketch_projection_split_elems(k, r) uint16_t, caller-owned. */
typedef struct {
    const float* P;
    int64_t k;
    uint16_t* P_split;
} sketch_split_problem;

typedef struct {
    const uint16_t* D; /* T x d BF16 */
    int64_t T, d, ld_d;
    const uint16_t* XP;/* T x r BF16 */
    int64_t ld_xp;
    float* C;          /* d x r fp32, read (unless overwrite) and written */
} sketch_accumulate_problem;

typedef struct {
    uint16_t* W;       /* d x k BF16, updated in place */
    int64_t d, k, ld_w;
    const float* C;    /* d x r fp32 */
    const float* P;    /* k x r fp32 */
    uint32_t layer;    /* Philox counter word of this layer's rounding stream */
    const double* wnorm2_in;  /* normalized SGD only, nullable */
    double* wnorm2_out;       /* normalized SGD only, nullable */
    int32_t* dev_status;      /* nullable */
} sketch_update_problem;

/* Workspace bytes of a batched call: the sum over problems i of
 * sketch_workspace_bytes(op, T[i], d[i], k[i], r).  Arrays an op does not use
 * may be NULL. */
SKETCH_API size_t sketch_workspace_bytes_batched(sketch_op op, int n, const int64_t* T, const int64_t* d,
                                                 const int64_t* k, int64_t r);
SKETCH_API sketch_status sketch_sample_projection_batched(sketch_proj_kind kind, uint64_t seed, uint32_t step,
                                                          int n, const sketch_projection_problem* problems,
                                                          int64_t r, int32_t* dev_status, void* ws,
                                                          size_t ws_bytes, void* stream);
SKETCH_API sketch_status sketch_project_inputs_batched(int n, const sketch_project_problem* problems, int64_t r,
                                                       void* ws, size_t ws_bytes, void* stream);
/* fp32-accurate saved XP.  The same calls as sketch_project_inputs_batched and
 * sketch_accumulate_batched, except that XP is kept to about 2^-17 relative
 * instead of one BF16 rounding (2^-9): XP holds, per token row, the BF16 of
 * the fp32 product in columns [0, r) and the BF16 of the remainder in columns
 * [n_pad, n_pad + r), n_pad = r rounded up to 16; so ld_xp >= 2 * n_pad, 4
 * bytes per value like fp32.  The accumulate call reads XP as the sum of the
 * two halves.  This removes the XP rounding term (~1e-3 relative) from C
 * ("Randomized Gradient Compression", "How it works": the layer saves X P; its
 * precision is this library's choice).  Columns [r, n_pad) and [n_pad + r,
 * 2 n_pad) are not written, and their contents do not affect C. */
SKETCH_API sketch_status sketch_project_inputs_fp32xp_batched(int n, const sketch_project_problem* problems,
                                                              int64_t r, void* ws, size_t ws_bytes, void* stream);
SKETCH_API sketch_status sketch_accumulate_fp32xp_batched(int n, const sketch_accumulate_problem* problems,
                                                          int64_t r, int overwrite, void* ws, size_t ws_bytes,
                                                          void* stream);

/* The BF16 split of projections as sketch_project_inputs uses them: with
 * n_pad = r rounded up to 16, rows [0, n_pad) of P_split hold the BF16 of P^T
 * (round to nearest even) and rows [n_pad, 2 n_pad) the BF16 of the remainder
 * P^T - hi, each row k values (rows r..n_pad-1 of each half are zero); the
 * tensor cores form X P as X hi + X lo.  A layer's P is split once per
 * refresh and the split passed to every sketch_project_inputs_batched call of
 * that P (the pages split nothing: this only saves work; a call without a
 * split makes its own in the workspace).  P_split must not overlap P. */
SKETCH_API size_t sketch_projection_split_elems(int64_t k, int64_t r);
SKETCH_API sketch_status sketch_split_projection_batched(int n, const sketch_split_problem* problems, int64_t r,
                                                         void* stream);

/* Layers that read the same input X (q, k and v of an attention block; gate
 * and up of an MLP) are projected together: their projections P_0 .. P_{m-1}
 * (each k x r fp32) form the k x (m r) concatenation [P_0 | ... | P_{m-1}],
 * whose split this call writes to P_split (sketch_projection_split_elems(k,
 * m r) uint16_t, caller-owned, not overlapping any P).  One
 * sketch_project_inputs_batched call with rank m r and that split then reads X
 * once and writes, per token row, XP_0 | ... | XP_{m-1}: member q's XP is
 * columns [q r, (q + 1) r) of the T x (m r) result, which sketch_accumulate
 * takes as XP = result + q r with ld_xp = the result's row stride ("LoGRA:
 * Scaling LLM Reinforcement Learning with Low-Rank Gradient Sketches", Key
 * Contributions: selected attention and MLP projections are sketched; sharing
 * their input is this library's way to read it once).  Each member column is
 * the same dot product as in a separate call.  1 <= m <= 16, m r <= 256;
 * every P 16-byte aligned; r a multiple of 8 when m > 1 (so that each
 * member's XP starts on a 16-byte boundary). */
typedef struct {
    const float* const* P; /* m pointers */
    int m;
    int64_t k;
    uint16_t* P_split;
} sketch_split_group;
SKETCH_API sketch_status sketch_split_projection_grouped(int n, const sketch_split_group* groups, int64_t r,
                                                         void* stream);
SKETCH_API sketch_status sketch_accumulate_batched(int n, const sketch_accumulate_problem* problems, int64_t r,
                                                   int overwrite, void* ws, size_t ws_bytes, void* stream);
SKETCH_API sketch_status sketch_apply_update_normsgd_batched(int n, const sketch_update_problem* problems,
                                                             int64_t r, float tau, uint64_t seed, uint32_t step,
                                                             void* ws, size_t ws_bytes, void* stream);
SKETCH_API sketch_status sketch_apply_update_sgd_batched(int n, const sketch_update_problem* problems, int64_t r,
                                                         float alpha_eta, uint64_t seed, uint32_t step, void* ws,
                                                         size_t ws_bytes, void* stream);

/* Read and clear the device error word of the current device: bits set by
 * kernels whose bounded internal waits gave up (a kernel that cannot make
 * progress records the failure and exits instead of hanging).  0 = none.
 * Synchronizes `stream`.  The outputs of a call that set a bit are undefined. */
#define SKETCH_DEVERR_TIMEOUT_LOAD 1   /* a TMA tile never arrived */
#define SKETCH_DEVERR_TIMEOUT_MMA 2    /* tensor-core work never completed */
#define SKETCH_DEVERR_TIMEOUT_STAGE 4  /* a pipeline stage was never released */
SKETCH_API sketch_status sketch_read_device_errors(int32_t* flags, void* stream);

/* Read and clear the current device's count of weights that the update calls
 * recomputed on their exact path: an element whose stochastic-rounding
 * margin lies within the error bound of the tensor-core rebuild of H_ij is
 * redone with H_ij from a compensated fp32 dot product, so that it rounds
 * exactly as the definition does.  Instrumentation for tests and benchmarks;
 * the pages have no counterpart.  Synchronizes `stream`. */
SKETCH_API sketch_status sketch_read_exact_count(uint64_t* count, void* stream);

/* Number of kernels this library has launched in this process (every device
 * and thread), counted on the host as each launch is issued.  Instrumentation
 * for benchmarks and tests; the pages have no counterpart.  Never fails. */
SKETCH_API uint64_t sketch_kernel_launches(void);

/* Static string for a status code. */
SKETCH_API const char* sketch_status_string(sketch_status status);

/* Description of the last failing call on the calling thread ("" if none). */
SKETCH_API const char* sketch_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RGS_SKETCH_H */
