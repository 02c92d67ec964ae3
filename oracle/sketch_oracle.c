/*
 * CPU oracle for randomized low-rank gradient sketching (RGC / LoGRA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant generator with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Everything is written as nested loops in double precision unless the method
 * fixes a narrower type (the stored sketch C is fp32, W and XP are BF16).
 * No blocking, fusion or reordering beyond the definitions below.
 *
 * Sources (page title, section):
 *   [RGC]   "Randomized Gradient Compression" -- "How it works", footnote 1.
 *   [LoGRA] "LoGRA: Scaling LLM Reinforcement Learning with Low-Rank Gradient
 *           Sketches" -- Key Contributions 1 and 2.
 *   [MOD]   "LoGRA: Low-Rank Gradient Sketches" -- "The Core Move", "Why the
 *           Sketch Can Be Accumulated Without a Full Gradient", "Why the Update
 *           Is Low-Rank but Not an Exact Recovery", "Minimal Causal Code".
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *           easy as 1, 2, 3", SC'11, section 3 (the Philox S-box and key
 *           schedule).
 *   Householder QR: Golub & Van Loan, Matrix Computations, section 5.2.
 *   Sign correction: Mezzadri, "How to generate random matrices from the
 *           classical compact groups", Notices AMS 2007 (R with positive
 *           diagonal makes Q Haar-distributed).
 *
 * Readings where the pages are silent (each one is a choice of this library):
 *   - Philox key = (seed low 32 bits, seed high 32 bits); counter =
 *     (block, step, layer, tag) with tag 0 = stochastic rounding, 1 = Rademacher
 *     signs, 2 = Gaussian draws.
 *   - Rademacher element (j,l) of the k x r matrix P has index e = j*r + l; its
 *     sign is bit (e % 32) of word ((e % 128) / 32) of block e / 128; a set bit
 *     means a negative sign.
 *   - Gaussian element e = j*r + l uses block e / 4; lanes 0,1 take words (0,1),
 *     lanes 2,3 take words (2,3); u = (w + 0.5) * 2^-32; even lane takes the
 *     cosine branch of Box-Muller, odd lane the sine branch.
 *   - Stochastic rounding of weight (i,j) uses e = i*k + j, the 16-bit lane
 *     e % 8 of block e / 8 (lane L is word L/2, low half when L is even).
 *   - The pre-rounding value is one fused multiply-add v = fmaf(-s, H_ij, W_ij).
 *   - A zero or non-finite norm makes the normalized-SGD update a no-op.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_TAG_SR 0u
#define ORC_TAG_RADEMACHER 1u
#define ORC_TAG_GAUSSIAN 2u

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (SC'11, section 3).                                          */
/* ------------------------------------------------------------------------- */

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    /* Multipliers and Weyl-sequence key increments as published for Philox4x32. */
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { /* the key is bumped before every round but the first */
            k0 += W0;
            k1 += W1;
        }
        uint64_t p0 = (uint64_t)M0 * (uint64_t)x0;
        uint64_t p1 = (uint64_t)M1 * (uint64_t)x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

static void stream_block(uint64_t seed, uint32_t layer, uint32_t step, uint32_t tag,
                         uint64_t block, uint32_t out[4]) {
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {(uint32_t)block, step, layer, tag};
    orc_philox4x32_10(ctr, key, out);
}

/* 16 random bits for the stochastic rounding of flat weight index e. */
uint32_t orc_sr_rand16(uint64_t seed, uint32_t layer, uint32_t step, uint64_t e) {
    uint32_t w[4];
    stream_block(seed, layer, step, ORC_TAG_SR, e / 8u, w);
    uint32_t lane = (uint32_t)(e % 8u);
    uint32_t word = w[lane / 2u];
    return (lane % 2u == 0u) ? (word & 0xFFFFu) : (word >> 16);
}

/* ------------------------------------------------------------------------- */
/* BF16 helpers (BF16 = the top 16 bits of an IEEE fp32).                     */
/* ------------------------------------------------------------------------- */

static float f32_from_bits(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

float orc_bf16_to_f32(uint16_t h) { return f32_from_bits(((uint32_t)h) << 16); }

/* Round a double to the nearest BF16 value, ties to even, in one rounding. */
uint16_t orc_bf16_from_double_rne(double x) {
    if (isnan(x)) return 0x7FC0u;
    if (isinf(x)) return x > 0 ? 0x7F80u : 0xFF80u;
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);            /* ax = m * 2^e, m in [0.5, 1) */
    int q_exp = e - 8;        /* BF16 keeps 8 significant bits */
    if (q_exp < -133) q_exp = -133; /* subnormal BF16 quantum is 2^-133 */
    double q = nearbyint(ldexp(ax, -q_exp)); /* default mode: nearest, ties even */
    double r = ldexp(q, q_exp);
    const double bf16_max = 3.3895313892515355e38; /* 0x7F7F */
    uint16_t out;
    if (r > bf16_max) out = 0x7F80u;
    else out = (uint16_t)(bits_from_f32((float)r) >> 16); /* r is exactly a BF16 value */
    return signbit(x) ? (uint16_t)(out | 0x8000u) : out;
}

/* Stochastic rounding of an fp32 value to BF16 with 16 random bits: add the
 * random bits below the BF16 mantissa and truncate.  The carry into the kept
 * bits happens with probability (dropped bits) / 2^16, which is the rounding
 * law of [RGC] "How it works" (a move of 1% of the gap happens 1% of the
 * time).  The magnitude is rounded, so negative values behave the same way. */
uint16_t orc_sr_bf16(float v, uint32_t rand16) {
    if (isnan(v)) return 0x7FC0u;
    uint32_t b = bits_from_f32(v);
    return (uint16_t)((b + (rand16 & 0xFFFFu)) >> 16);
}

/* ------------------------------------------------------------------------- */
/* (a) Projection P, k x r, fp32 row-major.                                   */
/* ------------------------------------------------------------------------- */

/* Rademacher signs scaled by 1/sqrt(r): [MOD] "Why the Sketch Can Be
 * Accumulated Without a Full Gradient" (random signs scaled by 1/sqrt(r)). */
void orc_sample_rademacher(uint64_t seed, uint32_t layer, uint32_t step, int k, int r, float* P) {
    const float scale = (float)(1.0 / sqrt((double)r));
    for (int j = 0; j < k; ++j) {
        for (int l = 0; l < r; ++l) {
            uint64_t e = (uint64_t)j * (uint64_t)r + (uint64_t)l;
            uint32_t w[4];
            stream_block(seed, layer, step, ORC_TAG_RADEMACHER, e / 128u, w);
            uint32_t bit = (uint32_t)(e % 128u);
            uint32_t set = (w[bit / 32u] >> (bit % 32u)) & 1u;
            P[(size_t)j * r + l] = set ? -scale : scale;
        }
    }
}

/* Standard normal draws by Box-Muller from the Gaussian Philox stream. */
void orc_gaussian_matrix(uint64_t seed, uint32_t layer, uint32_t step, int k, int r, double* G) {
    const double two_pi = 6.283185307179586476925286766559;
    for (int j = 0; j < k; ++j) {
        for (int l = 0; l < r; ++l) {
            uint64_t e = (uint64_t)j * (uint64_t)r + (uint64_t)l;
            uint32_t w[4];
            stream_block(seed, layer, step, ORC_TAG_GAUSSIAN, e / 4u, w);
            uint32_t lane = (uint32_t)(e % 4u);
            uint32_t wa = (lane < 2u) ? w[0] : w[2];
            uint32_t wb = (lane < 2u) ? w[1] : w[3];
            double ua = ((double)wa + 0.5) * 0x1p-32;
            double ub = ((double)wb + 0.5) * 0x1p-32;
            double radius = sqrt(-2.0 * log(ua));
            double angle = two_pi * ub;
            G[(size_t)j * r + l] = (lane % 2u == 0u) ? radius * cos(angle) : radius * sin(angle);
        }
    }
}

/* Thin Householder QR of the m x n matrix A (m >= n), row-major:
 * A = Q R with Q m x n orthonormal columns, R n x n upper triangular. */
void orc_householder_qr(int m, int n, const double* A, double* Q, double* R) {
    double* a = (double*)malloc(sizeof(double) * (size_t)m * n);
    double* vs = (double*)calloc((size_t)m * n, sizeof(double)); /* reflector j in column j */
    memcpy(a, A, sizeof(double) * (size_t)m * n);
    for (int j = 0; j < n; ++j) {
        double norm_x = 0.0;
        for (int i = j; i < m; ++i) norm_x += a[(size_t)i * n + j] * a[(size_t)i * n + j];
        norm_x = sqrt(norm_x);
        double x0 = a[(size_t)j * n + j];
        double alpha = (x0 >= 0.0) ? -norm_x : norm_x;
        double vnorm2 = 0.0;
        for (int i = j; i < m; ++i) {
            double vi = a[(size_t)i * n + j] - (i == j ? alpha : 0.0);
            vs[(size_t)i * n + j] = vi;
            vnorm2 += vi * vi;
        }
        if (vnorm2 == 0.0) continue; /* column already zero below the diagonal */
        double vnorm = sqrt(vnorm2);
        for (int i = j; i < m; ++i) vs[(size_t)i * n + j] /= vnorm;
        /* A[j:, j:] -= 2 v (v^T A[j:, j:]) */
        for (int c = j; c < n; ++c) {
            double dot = 0.0;
            for (int i = j; i < m; ++i) dot += vs[(size_t)i * n + j] * a[(size_t)i * n + c];
            for (int i = j; i < m; ++i) a[(size_t)i * n + c] -= 2.0 * vs[(size_t)i * n + j] * dot;
        }
    }
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < n; ++c) R[(size_t)i * n + c] = (c >= i) ? a[(size_t)i * n + c] : 0.0;
    /* Q = H_0 H_1 ... H_{n-1} [I_n; 0], applied right to left. */
    for (int i = 0; i < m; ++i)
        for (int c = 0; c < n; ++c) Q[(size_t)i * n + c] = (i == c) ? 1.0 : 0.0;
    for (int j = n - 1; j >= 0; --j) {
        for (int c = 0; c < n; ++c) {
            double dot = 0.0;
            for (int i = j; i < m; ++i) dot += vs[(size_t)i * n + j] * Q[(size_t)i * n + c];
            for (int i = j; i < m; ++i) Q[(size_t)i * n + c] -= 2.0 * vs[(size_t)i * n + j] * dot;
        }
    }
    free(a);
    free(vs);
}

/* Orthonormal frame by QR of a Gaussian matrix with the sign correction, scaled
 * by sqrt(input width / rank): [RGC] footnote 1.  Q_out receives the unscaled
 * frame in double (may be NULL). */
void orc_sample_qr(uint64_t seed, uint32_t layer, uint32_t step, int k, int r, float* P,
                   double* Q_out) {
    double* G = (double*)malloc(sizeof(double) * (size_t)k * r);
    double* Q = (double*)malloc(sizeof(double) * (size_t)k * r);
    double* R = (double*)malloc(sizeof(double) * (size_t)r * r);
    orc_gaussian_matrix(seed, layer, step, k, r, G);
    orc_householder_qr(k, r, G, Q, R);
    /* sign correction: make diag(R) positive by flipping columns of Q */
    for (int l = 0; l < r; ++l) {
        double sgn = (R[(size_t)l * r + l] < 0.0) ? -1.0 : 1.0;
        for (int j = 0; j < k; ++j) Q[(size_t)j * r + l] *= sgn;
    }
    const double scale = sqrt((double)k / (double)r);
    for (size_t i = 0; i < (size_t)k * r; ++i) P[i] = (float)(scale * Q[i]);
    if (Q_out) memcpy(Q_out, Q, sizeof(double) * (size_t)k * r);
    free(G);
    free(Q);
    free(R);
}

/* ------------------------------------------------------------------------- */
/* (b) Saved projected input XP = X P: [RGC] "How it works" (the layer saves  */
/* X P, not X).  Exact sum in double, one rounding to BF16.                   */
/* ------------------------------------------------------------------------- */

void orc_project_inputs(const uint16_t* X, int T, int k, int ldx, const float* P, int r,
                        uint16_t* XP, int ldxp) {
    for (int t = 0; t < T; ++t) {
        for (int l = 0; l < r; ++l) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += (double)orc_bf16_to_f32(X[(size_t)t * ldx + j]) * (double)P[(size_t)j * r + l];
            XP[(size_t)t * ldxp + l] = orc_bf16_from_double_rne(acc);
        }
    }
}

/* Same product kept in double (no rounding), for the algebraic checks. */
void orc_project_inputs_exact(const uint16_t* X, int T, int k, int ldx, const float* P, int r,
                              double* XP) {
    for (int t = 0; t < T; ++t)
        for (int l = 0; l < r; ++l) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += (double)orc_bf16_to_f32(X[(size_t)t * ldx + j]) * (double)P[(size_t)j * r + l];
            XP[(size_t)t * r + l] = acc;
        }
}

/* ------------------------------------------------------------------------- */
/* (c) Sketch accumulation C += D^T (X P), stored fp32: [RGC] "How it works"; */
/* [LoGRA] Key Contributions 1 (accumulated in fp32); [MOD] "Minimal Causal   */
/* Code" (S starts at zero, one addition per microbatch).                     */
/* ------------------------------------------------------------------------- */

void orc_accumulate(const uint16_t* D, int T, int d, int ldd, const uint16_t* XP, int ldxp, int r,
                    float* C, int overwrite) {
    for (int i = 0; i < d; ++i) {
        for (int l = 0; l < r; ++l) {
            double acc = overwrite ? 0.0 : (double)C[(size_t)i * r + l];
            for (int t = 0; t < T; ++t)
                acc += (double)orc_bf16_to_f32(D[(size_t)t * ldd + i]) *
                       (double)orc_bf16_to_f32(XP[(size_t)t * ldxp + l]);
            C[(size_t)i * r + l] = (float)acc;
        }
    }
}

/* Exact-mode accumulation with a double XP (T x r) into a double C. */
void orc_accumulate_exact(const uint16_t* D, int T, int d, int ldd, const double* XP, int r,
                          double* C) {
    for (int i = 0; i < d; ++i)
        for (int l = 0; l < r; ++l) {
            double acc = C[(size_t)i * r + l];
            for (int t = 0; t < T; ++t)
                acc += (double)orc_bf16_to_f32(D[(size_t)t * ldd + i]) * XP[(size_t)t * r + l];
            C[(size_t)i * r + l] = acc;
        }
}

/* ------------------------------------------------------------------------- */
/* (d) Rebuild H = C P^T and the norms.                                       */
/* ------------------------------------------------------------------------- */

/* H (d x k, double) = C (d x r) P^T (r x k): [RGC] "How it works" (rebuilds
 * the update H = C P.T); the LoGRA form is S A with A = P^T ([MOD]). */
void orc_rebuild(const float* C, int d, const float* P, int k, int r, double* H) {
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < k; ++j) {
            double acc = 0.0;
            for (int l = 0; l < r; ++l) acc += (double)C[(size_t)i * r + l] * (double)P[(size_t)j * r + l];
            H[(size_t)i * k + j] = acc;
        }
}

/* Frobenius norm of a BF16 matrix, in double. */
double orc_norm_w(const uint16_t* W, int d, int k, int ldw) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < k; ++j) {
            double w = (double)orc_bf16_to_f32(W[(size_t)i * ldw + j]);
            acc += w * w;
        }
    return sqrt(acc);
}

/* ||C P^T||_F by forming every element of H (the plain definition). */
double orc_norm_h_dense(const float* C, int d, const float* P, int k, int r) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < k; ++j) {
            double h = 0.0;
            for (int l = 0; l < r; ++l) h += (double)C[(size_t)i * r + l] * (double)P[(size_t)j * r + l];
            acc += h * h;
        }
    return sqrt(acc);
}

/* ||C P^T||_F^2 = sum_i c_i (P^T P) c_i^T: the same quantity through the r x r
 * Gram matrix of P, used where d*k is too large to form H. */
double orc_norm_h_gram(const float* C, int d, const float* P, int k, int r) {
    double* M = (double*)calloc((size_t)r * r, sizeof(double));
    for (int a = 0; a < r; ++a)
        for (int b = 0; b < r; ++b) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += (double)P[(size_t)j * r + a] * (double)P[(size_t)j * r + b];
            M[(size_t)a * r + b] = acc;
        }
    double total = 0.0;
    for (int i = 0; i < d; ++i) {
        const float* c = C + (size_t)i * r;
        for (int a = 0; a < r; ++a)
            for (int b = 0; b < r; ++b) total += (double)c[a] * M[(size_t)a * r + b] * (double)c[b];
    }
    free(M);
    return sqrt(total);
}

/* Status codes of the normalized-SGD step (bit flags; zero means the update ran). */
#define ORC_STATUS_H_ZERO 1
#define ORC_STATUS_H_NONFINITE 2
#define ORC_STATUS_W_NONFINITE 4

/* Step scale of normalized SGD, W <- W - tau * norm(W) * H / norm(H)
 * ([RGC] "How it works"), rounded once to fp32.  Returns the status. */
int orc_normsgd_scale(double norm_w, double norm_h, float tau, float* s_out) {
    int status = 0;
    if (!isfinite(norm_w)) status |= ORC_STATUS_W_NONFINITE;
    if (!isfinite(norm_h)) status |= ORC_STATUS_H_NONFINITE;
    else if (norm_h == 0.0) status |= ORC_STATUS_H_ZERO;
    *s_out = status ? 0.0f : (float)((double)tau * norm_w / norm_h);
    return status;
}

/* Update the given rows of W in place: v = fmaf(-s, fl32(H_ij), W_ij), then
 * stochastic rounding with the Philox bits of e = i*k + j.  rows[n] are the
 * row indices i of W (used for e and to pick the row of C); Wrows holds those
 * rows with leading dimension ldw.  v_out (nrows x k, may be NULL) receives the
 * pre-rounding fp32 values. */
void orc_update_rows(uint16_t* Wrows, const int* rows, int nrows, int k, int ldw, const float* C,
                     const float* P, int r, float s, uint64_t seed, uint32_t layer, uint32_t step,
                     float* v_out) {
    for (int n = 0; n < nrows; ++n) {
        int i = rows[n];
        const float* c = C + (size_t)i * r;
        for (int j = 0; j < k; ++j) {
            double h = 0.0;
            for (int l = 0; l < r; ++l) h += (double)c[l] * (double)P[(size_t)j * r + l];
            float hf = (float)h;
            uint16_t* wp = Wrows + (size_t)n * ldw + j;
            float v = fmaf(-s, hf, orc_bf16_to_f32(*wp));
            if (v_out) v_out[(size_t)n * k + j] = v;
            uint64_t e = (uint64_t)i * (uint64_t)k + (uint64_t)j;
            *wp = orc_sr_bf16(v, orc_sr_rand16(seed, layer, step, e));
        }
    }
}

/* Normalized SGD step on the whole matrix ([RGC] "How it works").  norm_h
 * comes from the dense definition when dense_h_norm is nonzero, otherwise from
 * the Gram route.  On a nonzero status W is left unchanged. */
int orc_update_normsgd(uint16_t* W, int d, int k, int ldw, const float* C, const float* P, int r,
                       float tau, uint64_t seed, uint32_t layer, uint32_t step, int dense_h_norm,
                       float* s_out) {
    double nw = orc_norm_w(W, d, k, ldw);
    double nh = dense_h_norm ? orc_norm_h_dense(C, d, P, k, r) : orc_norm_h_gram(C, d, P, k, r);
    float s;
    int status = orc_normsgd_scale(nw, nh, tau, &s);
    if (s_out) *s_out = s;
    if (status) return status;
    int* rows = (int*)malloc(sizeof(int) * (size_t)d);
    for (int i = 0; i < d; ++i) rows[i] = i;
    orc_update_rows(W, rows, d, k, ldw, C, P, r, s, seed, layer, step, NULL);
    free(rows);
    return 0;
}

/* LoGRA basic SGD step W <- W - alpha*eta * U A with U = S, A = P^T
 * ([MOD] "Why the Update Is Low-Rank but Not an Exact Recovery"). */
void orc_update_sgd(uint16_t* W, int d, int k, int ldw, const float* C, const float* P, int r,
                    float alpha_eta, uint64_t seed, uint32_t layer, uint32_t step) {
    int* rows = (int*)malloc(sizeof(int) * (size_t)d);
    for (int i = 0; i < d; ++i) rows[i] = i;
    orc_update_rows(W, rows, d, k, ldw, C, P, r, alpha_eta, seed, layer, step, NULL);
    free(rows);
}

/* ------------------------------------------------------------------------- */
/* Array forms of the scalar helpers above, for the Python test harness.     */
/* ------------------------------------------------------------------------- */

void orc_philox_array(const uint32_t* ctrs, int n, const uint32_t key[2], uint32_t* outs) {
    for (int i = 0; i < n; ++i) orc_philox4x32_10(ctrs + 4 * (size_t)i, key, outs + 4 * (size_t)i);
}

void orc_sr_rand16_array(uint64_t seed, uint32_t layer, uint32_t step, const uint64_t* e, int n,
                         uint32_t* out) {
    for (int i = 0; i < n; ++i) out[i] = orc_sr_rand16(seed, layer, step, e[i]);
}

void orc_sr_bf16_array(const float* v, const uint32_t* rand16, int n, uint16_t* out) {
    for (int i = 0; i < n; ++i) out[i] = orc_sr_bf16(v[i], rand16[i]);
}

void orc_bf16_from_double_array(const double* x, int n, uint16_t* out) {
    for (int i = 0; i < n; ++i) out[i] = orc_bf16_from_double_rne(x[i]);
}
