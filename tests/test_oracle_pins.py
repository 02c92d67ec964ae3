"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test checks one oracle function against a library routine (cuRAND's host
Philox generator, LAPACK QR through numpy, numpy matmul and SVD, torch's BF16
conversion), a closed form of the method, or brute force on tiny inputs.  The
method's definitions come from the pages "Randomized Gradient Compression"
("How it works", footnote 1), "LoGRA: Scaling LLM Reinforcement Learning with
Low-Rank Gradient Sketches" (Key Contributions 1) and "LoGRA: Low-Rank Gradient
Sketches" ("Why the Sketch Can Be Accumulated Without a Full Gradient", "Why
the Update Is Low-Rank but Not an Exact Recovery", "Why Refreshing the
Projection Enables New Update Directions", "What You Gain, and What You Lose").
"""
import ctypes
import ctypes.util
import glob
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from rank_gradient_sketching_philox_gb300 import synth


GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Philox4x32-10
# --------------------------------------------------------------------------

def _load_curand():
    cands = []
    found = ctypes.util.find_library("curand")
    if found:
        cands.append(found)
    for root in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
                 "/usr/local/cuda/targets/x86_64-linux/lib"):
        cands += sorted(glob.glob(os.path.join(root, "libcurand.so*")))
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


@pytest.mark.parametrize("seed", [0, 0x123456789ABCDEF, 0xFFFFFFFF00000001])
def test_philox_matches_curand_host_generator(orc, seed):
    """cuRAND's host Philox4x32-10 generator emits block b from counter
    (b // 65536, 0, b % 65536, 0) under key (seed lo, seed hi); the oracle's
    Philox must reproduce those words exactly, across the word-0 carry."""
    cur = _load_curand()
    if cur is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    assert cur.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert cur.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        nblk = 65536 + 4096
        out = np.zeros(4 * nblk, np.uint32)
        assert cur.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(out.size)) == 0
    finally:
        cur.curandDestroyGenerator(gen)
    pick = np.concatenate([np.arange(0, 2048), np.arange(65536 - 64, nblk)])
    ctrs = np.zeros((pick.size, 4), np.uint32)
    ctrs[:, 0] = pick // 65536
    ctrs[:, 2] = pick % 65536
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    mine = orc.philox_array(ctrs, key)
    ref = out.reshape(nblk, 4)[pick]
    assert np.array_equal(mine, ref)


def test_philox_counter_words_all_matter(orc):
    """Changing any counter or key word changes the block (no dead input)."""
    base = orc.philox4x32_10([1, 2, 3, 4], [5, 6])
    for w in range(4):
        c = [1, 2, 3, 4]
        c[w] ^= 1
        assert not np.array_equal(orc.philox4x32_10(c, [5, 6]), base)
    for w in range(2):
        k = [5, 6]
        k[w] ^= 1
        assert not np.array_equal(orc.philox4x32_10([1, 2, 3, 4], k), base)


def test_sr_bits_uniform(orc):
    """The 16-bit stochastic-rounding lanes are uniform (chi-square on the top
    4 bits) and bit-balanced."""
    from scipy import stats
    e = np.arange(200_000, dtype=np.uint64)
    r = orc.sr_rand16(7, 3, 11, e)
    assert r.max() < 65536
    counts = np.bincount(r >> 12, minlength=16)
    chi2 = stats.chisquare(counts)
    assert chi2.pvalue > 1e-4
    for b in range(16):
        frac = ((r >> b) & 1).mean()
        assert abs(frac - 0.5) < 5 * 0.5 / math.sqrt(r.size)


def test_sr_bits_independent_across_neighbours(orc):
    """Neighbouring weights (the 8 lanes of one Philox block and the next
    block) draw different bits: equal neighbours occur at the 2^-16 rate and
    the lanes are uncorrelated."""
    e = np.arange(400_000, dtype=np.uint64)
    r = orc.sr_rand16(1, 0, 0, e).astype(np.float64)
    for lag in (1, 2, 3, 4, 8):
        eq = np.mean(r[lag:] == r[:-lag])
        assert eq < 20.0 / 65536
        assert abs(np.corrcoef(r[lag:], r[:-lag])[0, 1]) < 5 / math.sqrt(r.size)


# --------------------------------------------------------------------------
# BF16 rounding
# --------------------------------------------------------------------------

def test_bf16_rne_matches_torch_on_fp32_values(orc):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(100_000, generator=g) * torch.exp(torch.randn(100_000, generator=g) * 20)
    special = torch.tensor([0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8,
                            2.0 ** -130, 2.0 ** -133, 3 * 2.0 ** -135, 3.3895313892515355e38,
                            3.40e38, float("inf"), float("-inf")], dtype=torch.float32)
    x = torch.cat([x, special])
    ref = _bits(x.to(torch.bfloat16))
    mine = orc.bf16_from_double(x.double().numpy())
    assert np.array_equal(mine, ref)


def test_bf16_rne_single_rounding_from_double(orc):
    """A double just above a BF16 tie must round up (rounding through fp32 first
    would land on the tie and round to even)."""
    x = 1.0 + 2 ** -8 + 2 ** -40  # fp32 would round this to the tie 1 + 2^-8
    assert orc.bf16_from_double(np.array([x]))[0] == 0x3F81
    assert orc.bf16_from_double(np.array([1.0 + 2 ** -8]))[0] == 0x3F80


# --------------------------------------------------------------------------
# Stochastic rounding
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_sr_binomial_one_percent(orc, sign):
    """A value 1% of the way across a BF16 gap rounds away from the lower
    magnitude 1% of the time, and the mean of the rounded values is the value."""
    base = 1.0
    gap = 2.0 ** -7
    f = GOLDEN["stochastic_rounding"]["fraction_of_gap"]
    v = np.float32(sign * (base + f * gap))
    n = 1_000_000
    rand16 = orc.sr_rand16(0, 0, 0, np.arange(n, dtype=np.uint64))
    out = orc.sr_bf16(np.full(n, v, np.float32), rand16)
    vals = orc.bf16_to_f32(out).astype(np.float64)
    low = sign * base
    up_frac = float(np.mean(vals != low))
    low16 = int(np.float32(v).view(np.uint32) & 0xFFFF)
    p = low16 / 65536.0
    assert abs(p - GOLDEN["stochastic_rounding"]["probability_of_moving_whole_gap"]) < 1e-4
    sigma = math.sqrt(p * (1 - p) / n)
    assert abs(up_frac - p) < 5 * sigma
    assert abs(vals.mean() - float(v)) < 5 * gap * sigma
    assert set(np.unique(vals)) <= {low, sign * (base + gap)}


def test_sr_special_values(orc):
    vals = np.array([1.0, -2.5, 0.0, -0.0, np.inf, -np.inf, np.nan, 3.3895313892515355e38],
                    np.float32)
    for rnd in (0, 1, 0x8000, 0xFFFF):
        out = orc.sr_bf16(vals, np.full(vals.size, rnd, np.uint32))
        # representable values are unchanged for every random draw
        assert list(out[:6]) == [0x3F80, 0xC020, 0x0000, 0x8000, 0x7F80, 0xFF80]
        assert out[6] == 0x7FC0
        assert out[7] == 0x7F7F
    # the largest finite fp32 lies above the largest BF16: it may round up to inf
    big = np.array([0x7F7FFFFF], np.uint32).view(np.float32)
    assert orc.sr_bf16(big, np.array([0xFFFF], np.uint32))[0] == 0x7F80
    assert orc.sr_bf16(big, np.array([0], np.uint32))[0] == 0x7F7F


# --------------------------------------------------------------------------
# Projections
# --------------------------------------------------------------------------

@pytest.mark.parametrize("k,r", [(512, 16), (24, 4), (4096, 64), (1000, 128)])
def test_rademacher_values_and_gram_diagonal(orc, k, r):
    P = orc.sample_rademacher(5, 2, 0, k, r)
    scale = np.float32(1.0 / math.sqrt(r))
    assert set(np.unique(P)) <= {scale, -scale}
    M = P.astype(np.float64).T @ P.astype(np.float64)
    assert np.allclose(np.diag(M), np.float64(scale) ** 2 * k, rtol=1e-13, atol=0)
    assert np.abs(np.diag(M) / (k / r) - 1.0).max() < 1.2e-7  # fp32 rounding of 1/sqrt(r)
    neg = float(np.mean(P < 0))
    assert abs(neg - 0.5) < 5 * 0.5 / math.sqrt(P.size)


def test_rademacher_seed_layer_step_distinct(orc):
    a = orc.sample_rademacher(1, 0, 0, 64, 16)
    assert np.array_equal(a, orc.sample_rademacher(1, 0, 0, 64, 16))
    for other in [(2, 0, 0), (1, 1, 0), (1, 0, 1)]:
        assert not np.array_equal(a, orc.sample_rademacher(other[0], other[1], other[2], 64, 16))


def test_rademacher_expectation_identity(orc):
    """E[P P^T] = I_k: off-diagonal means over N seeds are within sampling error."""
    k, r, N = 24, 4, 4000
    acc = np.zeros((k, k))
    for s in range(N):
        P = orc.sample_rademacher(s, 0, 0, k, r).astype(np.float64)
        acc += P @ P.T
    mean = acc / N
    assert np.allclose(np.diag(mean), 1.0, atol=1e-12)
    off = mean - np.diag(np.diag(mean))
    assert np.abs(off).max() < 5.0 / math.sqrt(r * N)


def test_gaussian_draws_are_standard_normal(orc):
    from scipy import stats
    G = orc.gaussian_matrix(3, 1, 2, 2000, 64).ravel()
    assert stats.kstest(G, "norm").pvalue > 1e-4
    assert abs(G.mean()) < 5 / math.sqrt(G.size)
    assert abs(G.var() - 1.0) < 5 * math.sqrt(2.0 / G.size)
    pairs = G.reshape(-1, 2)  # (cos, sin) branches of the same Box-Muller pair
    assert abs(np.corrcoef(pairs[:, 0], pairs[:, 1])[0, 1]) < 5 / math.sqrt(pairs.shape[0])


def _sign_fixed_lapack_qr(A):
    Q, R = np.linalg.qr(A)
    s = np.where(np.diag(R) < 0, -1.0, 1.0)
    return Q * s[None, :], R * s[:, None]


@pytest.mark.parametrize("m,n", [(24, 4), (200, 16), (512, 64), (64, 64)])
def test_householder_matches_lapack(orc, m, n):
    A = np.random.default_rng(m * 1000 + n).standard_normal((m, n))
    Q, R = orc.householder_qr(A)
    Qs, Rs = _sign_fixed_lapack_qr(A)
    s = np.where(np.diag(R) < 0, -1.0, 1.0)
    assert np.abs(Q * s[None, :] - Qs).max() < 1e-12
    assert np.abs(R * s[:, None] - Rs).max() < 1e-12 * np.abs(Rs).max()
    assert np.abs(Q @ R - A).max() < 1e-12 * np.abs(A).max()
    assert np.allclose(np.tril(R, -1), 0.0)


@pytest.mark.parametrize("k,r", [(512, 16), (4096, 64), (2048, 256), (24, 4)])
def test_qr_projection_frame(orc, k, r):
    """P^T P = (k/r) I_r to 1e-5 relative; Q^T G is upper triangular with a
    positive diagonal (the sign correction); Q equals LAPACK's sign-fixed Q."""
    P, Q = orc.sample_qr(9, 4, 1, k, r, return_q=True)
    M = P.astype(np.float64).T @ P.astype(np.float64)
    assert np.abs(M - (k / r) * np.eye(r)).max() / (k / r) < 1e-5
    G = orc.gaussian_matrix(9, 4, 1, k, r)
    R = Q.T @ G
    assert np.abs(np.tril(R, -1)).max() < 1e-10 * np.abs(R).max()
    assert np.all(np.diag(R) > 0)
    Qs, _ = _sign_fixed_lapack_qr(G)
    assert np.abs(Q - Qs).max() < 1e-11
    assert np.array_equal(P, (math.sqrt(k / r) * Q).astype(np.float32))


def test_qr_square_frame_is_exact_identity(orc):
    """r = k: the frame is a square orthogonal matrix, so P P^T = I and the
    rebuild returns the gradient itself."""
    k = r = 24
    _, Q = orc.sample_qr(2, 0, 0, k, r, return_q=True)
    assert np.abs(Q @ Q.T - np.eye(k)).max() < 1e-12
    G = np.random.default_rng(0).standard_normal((10, k))
    assert np.abs(G @ Q @ Q.T - G).max() < 1e-12


# --------------------------------------------------------------------------
# XP, C, H against brute force
# --------------------------------------------------------------------------

def _tiny_problem(d=40, k=24, T=17, mbs=3):
    Xs = [synth.normal_bf16((T, k), 1.0, 11 + m) for m in range(mbs)]
    Ds = [synth.normal_bf16((T, d), 1e-3, 51 + m) for m in range(mbs)]
    G = sum(D.double().T @ X.double() for D, X in zip(Ds, Xs)).numpy()
    return Xs, Ds, G


@pytest.mark.parametrize("kind", [0, 1])
def test_xp_exact_and_rounded(orc, kind):
    X = synth.normal_bf16((33, 96), 1.0, 5)
    P = orc.sample_projection(kind, 0, 0, 0, 96, 8)
    exact = X.double().numpy() @ P.astype(np.float64)
    xp_exact = orc.project_inputs_exact(_bits(X), P)
    assert np.abs(xp_exact - exact).max() < 1e-12 * np.abs(exact).max()
    xp = orc.project_inputs(_bits(X), P)
    ref = orc.bf16_from_double(exact)
    ref_torch = _bits(torch.from_numpy(exact).float().to(torch.bfloat16))
    same = np.mean(xp == ref)
    assert same >= 0.999
    # one-ulp neighbours at most, and the fp32 route agrees except near ties
    assert np.all(np.abs(xp.astype(np.int32) - ref.astype(np.int32)) <= 1)
    assert np.mean(xp == ref_torch) >= 0.99


@pytest.mark.parametrize("kind", [0, 1])
def test_sketch_equals_gradient_times_projection(orc, kind):
    """C = sum_mb D^T (X P) = G P with G = sum_mb D^T X formed densely."""
    Xs, Ds, G = _tiny_problem()
    k, d, r = 24, 40, 4
    P = orc.sample_projection(kind, 1, 0, 0, k, r)
    Ce = np.zeros((d, r))
    C = np.zeros((d, r), np.float32)
    for m, (X, D) in enumerate(zip(Xs, Ds)):
        Ce = orc.accumulate_exact(_bits(D), orc.project_inputs_exact(_bits(X), P), Ce)
        C = orc.accumulate(_bits(D), orc.project_inputs(_bits(X), P), C, overwrite=(m == 0))
    GP = G @ P.astype(np.float64)
    assert np.abs(Ce - GP).max() < 1e-12 * np.abs(GP).max()
    rel = np.linalg.norm(C - GP) / np.linalg.norm(GP)
    assert rel < 4e-3
    # accumulate without overwrite on a zero start equals overwrite
    C0 = orc.accumulate(_bits(Ds[0]), orc.project_inputs(_bits(Xs[0]), P), np.zeros((d, r)), False)
    C1 = orc.accumulate(_bits(Ds[0]), orc.project_inputs(_bits(Xs[0]), P), np.ones((d, r)), True)
    assert np.array_equal(C0, C1)


@pytest.mark.parametrize("kind", [0, 1])
def test_rebuild_equals_g_p_pt(orc, kind):
    Xs, Ds, G = _tiny_problem()
    P = orc.sample_projection(kind, 1, 0, 0, 24, 4)
    P64 = P.astype(np.float64)
    C = (G @ P64).astype(np.float32)
    H = orc.rebuild(C, P)
    assert np.abs(H - C.astype(np.float64) @ P64.T).max() < 1e-12 * np.abs(H).max()
    GPP = G @ P64 @ P64.T
    assert np.linalg.norm(H - GPP) / np.linalg.norm(GPP) < 1e-6
    assert abs(orc.norm_h_dense(C, P) - np.linalg.norm(H)) < 1e-12 * np.linalg.norm(H)
    assert abs(orc.norm_h_gram(C, P) - np.linalg.norm(H)) < 1e-12 * np.linalg.norm(H)


def test_norm_w_matches_numpy(orc):
    W = synth.normal_bf16((37, 53), 0.02, 4)
    assert abs(orc.norm_w(_bits(W)) - np.linalg.norm(W.double().numpy())) < 1e-14


@pytest.mark.parametrize("kind", [0, 1])
def test_update_rank_and_refresh(orc, kind):
    """One step's update has rank <= r; two steps with refreshed projections
    reach rank min(2r, d, k) > r."""
    d, k, r = 40, 24, 4
    G = np.random.default_rng(5).standard_normal((d, k))
    Hs = []
    for step in (0, 1):
        P = orc.sample_projection(kind, 3, 0, step, k, r)
        C = (G @ P.astype(np.float64)).astype(np.float32)
        Hs.append(orc.rebuild(C, P))
    s1 = np.linalg.svd(Hs[0], compute_uv=False)
    assert s1[r] / s1[0] < 1e-10
    s2 = np.linalg.svd(Hs[0] + Hs[1], compute_uv=False)
    assert s2[2 * r - 1] / s2[0] > 1e-6
    assert s2[2 * r] / s2[0] < 1e-10


@pytest.mark.parametrize("kind,excess", [(0, lambda k, r: (k - 1) / r), (1, lambda k, r: (k - r) / r)])
def test_monte_carlo_mean_is_unbiased(orc, kind, excess):
    """Over N seeds, ||mean(H) - G|| / ||G|| matches the closed form
    sqrt(excess / N) (Rademacher: (k-1)/r; Haar frame: (k-r)/r)."""
    d, k, r, N = 6, 24, 4, 10_000
    G = np.random.default_rng(1).standard_normal((d, k))
    acc = np.zeros((d, k))
    for s in range(N):
        P = orc.sample_projection(kind, s, 0, 0, k, r).astype(np.float64)
        acc += G @ P @ P.T
    rel = np.linalg.norm(acc / N - G) / np.linalg.norm(G)
    pred = math.sqrt(excess(k, r) / N)
    assert 0.5 * pred < rel < 1.5 * pred


# --------------------------------------------------------------------------
# Updates
# --------------------------------------------------------------------------

def _nearest_f32(x: Fraction) -> np.float32:
    """Correctly rounded fp32 of an exact rational (ties to even), by search."""
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - x),
                                     int(np.array(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_update_rows_fused_fma_and_rounding(orc):
    """W' = SR(fl32(w - s*fl32(H))) with one rounding, checked with exact
    rational arithmetic on a small block."""
    d, k, r = 6, 16, 4
    rng = np.random.default_rng(2)
    W = _bits(synth.normal_bf16((d, k), 0.02, 9))
    C = rng.standard_normal((d, r)).astype(np.float32)
    P = orc.sample_rademacher(4, 0, 0, k, r)
    s = np.float32(3.7e-4)
    rows = np.arange(d, dtype=np.int32)
    Wn, v = orc.update_rows(W, rows, C, P, float(s), 4, 2, 9, return_v=True)
    H = C.astype(np.float64) @ P.astype(np.float64).T
    e = (rows[:, None].astype(np.uint64) * k + np.arange(k, dtype=np.uint64)[None, :]).ravel()
    rnd = orc.sr_rand16(4, 2, 9, e).reshape(d, k)
    wf = orc.bf16_to_f32(W)
    for i in range(d):
        for j in range(k):
            hf = np.float32(H[i, j])
            exact = Fraction(float(wf[i, j])) - Fraction(float(s)) * Fraction(float(hf))
            vv = _nearest_f32(exact)
            assert np.array(vv).view(np.uint32) == np.array(v[i, j]).view(np.uint32)
            out = (int(np.array(vv).view(np.uint32)) + int(rnd[i, j])) >> 16
            assert out == Wn[i, j]


def test_update_sgd_is_update_rows_with_alpha_eta(orc):
    d, k, r = 8, 24, 4
    W = _bits(synth.normal_bf16((d, k), 0.02, 1))
    C = np.random.default_rng(0).standard_normal((d, r)).astype(np.float32)
    P = orc.sample_qr(0, 0, 0, k, r)
    a = orc.update_sgd(W, C, P, 1e-4, 0, 1, 2)
    b = orc.update_rows(W, np.arange(d), C, P, np.float32(1e-4), 0, 1, 2)
    assert np.array_equal(a, b)


def test_normsgd_scale_and_step_size(orc):
    """s = tau ||W|| / ||H||, so the pre-rounding step has norm tau ||W||."""
    d, k, r = 32, 48, 8
    W = _bits(synth.normal_bf16((d, k), 0.02, 2))
    C = np.random.default_rng(3).standard_normal((d, r)).astype(np.float32)
    P = orc.sample_qr(1, 0, 0, k, r)
    tau = 1e-3
    Wn, status, s = orc.update_normsgd(W, C, P, tau, 0, 0, 0)
    assert status == 0
    nw = np.linalg.norm(orc.bf16_to_f32(W).astype(np.float64))
    H = C.astype(np.float64) @ P.astype(np.float64).T
    assert abs(s - tau * nw / np.linalg.norm(H)) <= 1e-7 * s
    assert abs(np.linalg.norm(s * H) - tau * nw) < 1e-6 * tau * nw
    Wg, _, sg = orc.update_normsgd(W, C, P, tau, 0, 0, 0, dense_h_norm=False)
    assert abs(sg - s) <= 2e-7 * s


def test_normsgd_square_frame_is_dense_normalized_sgd(orc):
    """r = k with the QR frame: H = G, so the step is the textbook dense
    normalized SGD step W - tau ||W|| G / ||G||."""
    d, k = 12, 16
    r = k
    W = _bits(synth.normal_bf16((d, k), 0.02, 5))
    G = np.random.default_rng(8).standard_normal((d, k))
    P = orc.sample_qr(6, 0, 0, k, r)
    C = (G @ P.astype(np.float64)).astype(np.float32)
    nw = orc.norm_w(W)
    s, status = orc.normsgd_scale(nw, orc.norm_h_dense(C, P), 1e-3)
    assert status == 0
    _, v = orc.update_rows(W, np.arange(d), C, P, s, 0, 0, 0, return_v=True)
    wf = orc.bf16_to_f32(W).astype(np.float64)
    text = wf - 1e-3 * nw * G / np.linalg.norm(G)
    step = 1e-3 * nw * np.abs(G).max() / np.linalg.norm(G)
    assert np.abs(v - text).max() < 1e-5 * step + 2 * np.spacing(np.float32(0.1))


def test_zero_step_leaves_w_bit_identical(orc):
    d, k, r = 16, 32, 4
    W = _bits(synth.normal_bf16((d, k), 0.02, 7))
    C = np.random.default_rng(1).standard_normal((d, r)).astype(np.float32)
    P = orc.sample_rademacher(0, 0, 0, k, r)
    Wn, status, _ = orc.update_normsgd(W, C, P, 0.0, 0, 0, 0)
    assert status == 0 and np.array_equal(Wn, W)
    assert np.array_equal(orc.update_sgd(W, C, P, 0.0, 0, 0, 0), W)


def test_degenerate_norms_are_no_ops(orc):
    d, k, r = 8, 16, 4
    W = _bits(synth.normal_bf16((d, k), 0.02, 7))
    P = orc.sample_rademacher(0, 0, 0, k, r)
    Wn, status, _ = orc.update_normsgd(W, np.zeros((d, r), np.float32), P, 1e-3, 0, 0, 0)
    assert status == orc.STATUS_H_ZERO and np.array_equal(Wn, W)
    Cn = np.zeros((d, r), np.float32)
    Cn[2, 1] = np.nan
    Wn, status, _ = orc.update_normsgd(W, Cn, P, 1e-3, 0, 0, 0)
    assert status & orc.STATUS_H_NONFINITE and np.array_equal(Wn, W)
    Wi = W.copy()
    Wi[0, 0] = 0x7F80
    C = np.ones((d, r), np.float32)
    Wn, status, _ = orc.update_normsgd(Wi, C, P, 1e-3, 0, 0, 0)
    assert status & orc.STATUS_W_NONFINITE and np.array_equal(Wn, Wi)


def test_sketch_memory_is_d_times_r(orc):
    """d = k = 4096, r = 64: the fp32 sketch holds 1 MiB against 64 MiB for the
    dense fp32 gradient (LoGRA, Key Contributions 1)."""
    g = GOLDEN["sketch_memory"]
    d, k, r = g["d"], g["k"], g["r"]
    D = synth.normal_bf16((1, d), 1e-3, 1)
    XP = np.zeros((1, r), np.uint16)
    C = orc.accumulate(_bits(D), XP, np.zeros((d, r), np.float32), overwrite=True)
    assert C.nbytes == g["fp32_sketch_bytes"]
    assert np.zeros((d, k), np.float32).nbytes == g["fp32_dense_gradient_bytes"]
