"""GPU path against the CPU oracle, element by element, on seeded inputs.

Each C-ABI call is compared with the oracle on identical inputs:
  * Philox-driven outputs (Rademacher P) must be bit-exact;
  * the QR frame within 1e-5 relative Frobenius of the oracle's and
    orthonormal to 1e-5 (P^T P = (k/r) I);
  * XP within one BF16 step of the oracle (plus 1e-5 of its RMS for values
    near zero, the size of the fp32 accumulation error) and bit-identical on
    >= 99% (that error, about u*sqrt(k) relative, moves a value across a BF16
    rounding boundary on well under 1% of elements);
  * C within 2e-3 relative Frobenius, and element-wise within 1e-4 of its RMS
    (fp32 accumulation over T terms is good to a few 1e-6 relative);
  * W after an update: >= 99.99% bit-identical and every other element exactly
    one BF16 step away.
Small cases cover several tiles plus ragged edges; full-size layer shapes are
checked on sampled rows that the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
import rank_gradient_sketching_philox_gb300 as rgs
from rank_gradient_sketching_philox_gb300 import binding, diagnostics, policy_sync, synth

from gpu_util import bits, from_bits, rel_fro, w_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def bits_t(t):
    """BF16 tensor -> int16 view (bit patterns, on the device)."""
    return t.contiguous().view(torch.int16)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()
    orc.lib()


@pytest.fixture(autouse=True)
def _no_device_errors():
    binding.read_device_errors()
    yield
    assert binding.read_device_errors() == 0, "a kernel's bounded wait timed out"


# --------------------------------------------------------------------------
# (a) projections
# --------------------------------------------------------------------------

@pytest.mark.parametrize("k,r,layer,step", [(512, 16, 0, 0), (4096, 64, 3, 0), (2048, 128, 7, 5),
                                            (8192, 256, 1, 2), (24, 4, 0, 9), (16, 3, 2, 1),
                                            (8, 1, 0, 0), (1000, 50, 11, 3)])
def test_rademacher_bit_exact(k, r, layer, step):
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(rgs.PROJ_RADEMACHER, 0x5EED, layer, step, P)
    ref = orc.sample_rademacher(0x5EED, layer, step, k, r)
    assert np.array_equal(P.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("k,r,layer,step", [(512, 16, 0, 0), (4096, 64, 2, 1), (12288, 64, 5, 3),
                                            (2048, 256, 1, 0), (1000, 50, 4, 7), (64, 16, 0, 2),
                                            (8192, 4, 3, 3), (1600, 200, 2, 1), (640, 33, 0, 0),
                                            (2048, 128, 1, 2), (1000, 136, 3, 0), (4096, 192, 2, 2)])
def test_qr_projection_matches_oracle(k, r, layer, step):
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 77, layer, step, P, dev_status=status)
    assert int(status.item()) == 0
    got = P.cpu().numpy().astype(np.float64)
    ref = orc.sample_qr(77, layer, step, k, r)
    assert rel_fro(got, ref) < 1e-5
    M = got.T @ got
    assert np.abs(M - (k / r) * np.eye(r)).max() / (k / r) < 1e-5


@pytest.mark.parametrize("k,r,layer,step", [(32, 16, 0, 0), (64, 64, 1, 0), (8, 8, 2, 1), (8, 3, 0, 4),
                                            (200, 56, 3, 2), (1000, 251, 1, 1), (1016, 256, 4, 0),
                                            (256, 256, 0, 3), (520, 136, 2, 5)])
def test_wide_qr_projection_matches_oracle(k, r, layer, step):
    """Frames with r <= k < 4r (fp64 Householder on the device), up to square
    ones, whose Gaussian matrix has a condition number of order k: the frame
    matches the exact one to fp32 rounding, and P^T P = (k/r) I; for r = k the
    frame is orthogonal, so P P^T = I as well."""
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 77, layer, step, P, dev_status=status)
    assert int(status.item()) == 0
    got = P.cpu().numpy().astype(np.float64)
    ref = orc.sample_qr(77, layer, step, k, r)
    assert rel_fro(got, ref) < 1e-6
    M = got.T @ got
    assert np.abs(M - (k / r) * np.eye(r)).max() / (k / r) < 1e-6
    if r == k:
        assert np.abs(got @ got.T - np.eye(k)).max() < 1e-6


def test_qr_mixed_batch_matches_oracle():
    """One batched call over frames of both kinds (CholeskyQR2 for 4r <= k,
    Householder below), in an interleaved order."""
    r, seed, step = 64, 23, 4
    ks = [64, 1024, 200, 256, 512, 136, 4096]
    Ps = [torch.empty(k, r, dtype=torch.float32, device=DEV) for k in ks]
    layers = [5 + i for i in range(len(ks))]
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rgs.sample_projection_batched(rgs.PROJ_GAUSSIAN_QR, seed, step, Ps, layers, dev_status=status)
    assert int(status.item()) == 0
    for P, k, layer in zip(Ps, ks, layers):
        assert rel_fro(P.cpu().numpy(), orc.sample_qr(seed, layer, step, k, r)) < 1e-5, k


def test_qr_rejects_rank_above_width():
    P = torch.empty(16, 32, dtype=torch.float32, device=DEV)
    with pytest.raises(binding.SketchError) as ei:
        rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 0, 0, 0, P)
    assert ei.value.status == binding.ERR_INVALID_ARG


def test_projection_deterministic():
    a = torch.empty(4096, 64, dtype=torch.float32, device=DEV)
    b = torch.empty_like(a)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 5, 1, 1, a)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 5, 1, 1, b)
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# (b) projected inputs
# --------------------------------------------------------------------------

def _pad8(n):
    return (n + 7) // 8 * 8


def _padded_bf16(rows, cols, device=DEV, fill=float("nan")):
    """rows x cols BF16 view into a buffer whose row stride is a multiple of 8."""
    return torch.full((rows, _pad8(cols)), fill, dtype=torch.bfloat16, device=device)[:, :cols]


def _xp_check(got_bits, ref_bits):
    """One BF16 step of the oracle's value, or the fp32-accumulation slack
    (1e-5 of the RMS of XP) for values near zero; >= 99% bit-identical."""
    got = orc.bf16_to_f32(got_bits).astype(np.float64)
    ref = orc.bf16_to_f32(ref_bits).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    rms = math.sqrt(float(np.mean(ref * ref)))
    assert np.all(np.abs(got - ref) <= ulp + 1e-5 * rms)
    assert np.mean(got_bits == ref_bits) >= 0.99


@pytest.mark.parametrize("T,k,r,kind", [(128, 512, 16, 1), (300, 1024, 64, 0), (77, 104, 24, 1),
                                        (64, 256, 1, 0), (130, 2048, 256, 1), (1, 8, 3, 0)])
def test_project_inputs_matches_oracle(T, k, r, kind):
    X = synth.normal_bf16((T, k), 1.0, 31 + T)
    if kind == 0:
        P = orc.sample_rademacher(3, 0, 0, k, r)
    else:
        P = orc.sample_qr(3, 0, 0, k, r) if 4 * r <= k else orc.sample_rademacher(3, 0, 0, k, r)
    XP = _padded_bf16(T, r)
    rgs.project_inputs(X.to(DEV), torch.from_numpy(P).to(DEV), XP)
    _xp_check(bits(XP), orc.project_inputs(bits(X), P))


@pytest.mark.parametrize("r", [64, 20, 256])
def test_project_inputs_with_reused_split(r):
    """A split made once by split_projection_batched gives the same XP, bit for
    bit, as letting each call split P itself, across several microbatches and
    layers of different k; one split launch replaces one per call."""
    ks, T = [512, 1024, 136], 200
    Ps = [torch.from_numpy(orc.sample_rademacher(5, li, 0, k, r)).to(DEV) for li, k in enumerate(ks)]
    splits = rgs.split_projection_batched(Ps)
    for mb in range(2):
        Xs = [synth.normal_bf16((T, k), 1.0, 100 * mb + li).to(DEV) for li, k in enumerate(ks)]
        ref = [_padded_bf16(T, r) for _ in ks]
        got = [_padded_bf16(T, r) for _ in ks]
        rgs.project_inputs_batched(Xs, Ps, ref)
        before = rgs.kernel_launches()
        rgs.project_inputs_batched(Xs, Ps, got, splits=splits)
        assert rgs.kernel_launches() - before == 1  # the skinny GEMM only
        for li in range(len(ks)):
            assert torch.equal(bits_t(got[li]), bits_t(ref[li]))
            _xp_check(bits(got[li]), orc.project_inputs(bits(Xs[li]), Ps[li].cpu().numpy()))


def test_project_inputs_strided_rows_leave_padding():
    T, k, r, ld_x, ld_xp = 100, 320, 16, 336, 24
    X_full = synth.normal_bf16((T, ld_x), 1.0, 8).to(DEV)
    X = X_full[:, :k]
    P = orc.sample_qr(1, 0, 0, k, r)
    XP_full = torch.full((T, ld_xp), 7.0, dtype=torch.bfloat16, device=DEV)
    rgs.project_inputs(X, torch.from_numpy(P).to(DEV), XP_full[:, :r])
    _xp_check(bits(XP_full[:, :r]), orc.project_inputs(bits(X), P))
    assert torch.all(XP_full[:, r:] == 7.0)


@pytest.mark.parametrize("T,k,r,kind", [(4096, 4096, 64, 1), (16384, 8192, 256, 1), (16384, 8192, 4, 0)])
def test_project_inputs_full_size_sampled_tokens(T, k, r, kind):
    """4096 tokens x k=4096 -> r=64 (the LoGRA worked example's shape, QR P)
    and one 16384-token response of the long-response sweep (k=8192, r=256
    with QR P, r=4 with Rademacher P); compared on 64 sampled tokens."""
    X = synth.layer_x(T, k, 0, 0, device=DEV)
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(kind, 0, 0, 0, P)
    XP = _padded_bf16(T, r)
    rgs.project_inputs(X, P, XP)
    rows = np.random.default_rng(0).choice(T, 64, replace=False)
    ref = orc.project_inputs(bits(X[rows]), P.cpu().numpy())
    _xp_check(bits(XP)[rows], ref)


@pytest.mark.parametrize("r,m,k", [(64, 1, 1024), (20, 1, 1024), (64, 3, 1024), (136, 1, 1024), (72, 3, 1024),
                                   (48, 3, 128), (64, 1, 1088), (64, 1, 1000), (32, 1, 64), (40, 2, 200)])
def test_project_inputs_persistent_batch_matches_oracle(r, m, k):
    """Large batches (3 layers x 16384 tokens) run persistent CTAs, each tile
    over all of K: single layers of rank 64, 20 and 136 (ragged last column
    groups) and groups of two or three members; sampled tokens against the
    oracle, and the BF16 pair form against the exact product.  Ranks up to 64
    stage two 64-wide K chunks at a time: k = 1088 and 64 leave the last
    stage's second chunk wholly past K, k = 1000 and 200 end inside a chunk;
    k = 128 gives two K chunks, fewer than the four partial accumulators a
    tile may use."""
    T, n = 16384, 3
    Xs = [synth.layer_x(T, k, i, 0, device=DEV) for i in range(n)]
    sample = orc.sample_qr if 4 * r <= k else orc.sample_rademacher
    Ps = [[torch.from_numpy(sample(5, 3 * i + q, 0, k, r)).to(DEV) for q in range(m)] for i in range(n)]
    XPs = [_padded_bf16(T, m * r) for _ in range(n)]
    if m == 1:
        rgs.project_inputs_batched(Xs, [P[0] for P in Ps], XPs)
    else:
        splits = rgs.split_projection_grouped(Ps)
        rgs.project_inputs_grouped_batched(Xs, splits, m * r, XPs)
    rows = np.random.default_rng(5).choice(T, 48, replace=False)
    for i in range(n):
        for q in range(m):
            ref = orc.project_inputs(bits(Xs[i][rows]), Ps[i][q].cpu().numpy())
            _xp_check(bits(XPs[i][:, q * r:(q + 1) * r])[rows], ref)
    if m == 1:
        n_pad = (r + 15) // 16 * 16
        XP2 = [_padded_bf16(T, rgs.xp_split_cols(r)) for _ in range(n)]
        rgs.project_inputs_fp32xp_batched(Xs, [P[0] for P in Ps], XP2)
        for i in range(n):
            got = (XP2[i][rows, :r].float() + XP2[i][rows, n_pad:n_pad + r].float()).cpu().numpy().astype(np.float64)
            exact = orc.project_inputs_exact(bits(Xs[i][rows]), Ps[i][0].cpu().numpy())
            # P = hi + lo to 2^-17 of each entry, and fp32 sums of k terms:
            # within 2^-16 of the sum of the terms' magnitudes
            x64 = Xs[i][rows].float().cpu().numpy().astype(np.float64)
            mag = np.abs(x64) @ np.abs(Ps[i][0].cpu().numpy().astype(np.float64))
            assert np.all(np.abs(got - exact) <= 2.0 ** -16 * mag)
    assert rgs.read_device_errors() == 0


# --------------------------------------------------------------------------
# (c) accumulation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,r,m", [(300, 512, 64, 3), (129, 1024, 64, 2), (64, 256, 16, 4), (1, 8, 8, 1),
                                     (200, 4096, 32, 8)])
def test_grouped_projection_reads_x_once(T, k, r, m):
    """Members sharing X, projected in one call from the split of their
    concatenation: each member's columns equal its own projection call, bit for
    bit, and match the oracle; the accumulate reads each member's columns
    through the shared result's row stride."""
    Ps = [torch.from_numpy(orc.sample_rademacher(11, q, 2, k, r)).to(DEV) for q in range(m)]
    X = synth.normal_bf16((T, k), 1.0, 41).to(DEV)
    split = rgs.split_projection_grouped([Ps])[0]
    XPg = _padded_bf16(T, m * r)
    rgs.project_inputs_grouped_batched([X], [split], m * r, [XPg])
    D = synth.normal_bf16((T, 96), 1e-2, 42).to(DEV)
    for q in range(m):
        own = _padded_bf16(T, r)
        rgs.project_inputs(X, Ps[q], own)
        member = XPg[:, q * r:(q + 1) * r]
        assert torch.equal(bits_t(member), bits_t(own)), q
        _xp_check(bits(member), orc.project_inputs(bits(X), Ps[q].cpu().numpy()))
        C = torch.empty(96, r, dtype=torch.float32, device=DEV)
        rgs.accumulate(D, member, C, overwrite=True)
        _c_check(C.cpu().numpy(), orc.accumulate(bits(D), bits(own), np.zeros((96, r)), True))


def _c_check(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert rel_fro(got, ref) < 2e-3
    rms = math.sqrt(float(np.mean(ref * ref)))
    assert np.abs(got - ref).max() <= 1e-4 * rms


@pytest.mark.parametrize("T,d,r,mbs", [(128, 256, 16, 4), (513, 200, 64, 2), (40, 40, 4, 3),
                                       (1000, 1032, 256, 1), (17, 9, 1, 2), (64, 130, 20, 2)])
def test_accumulate_matches_oracle_same_xp(T, d, r, mbs):
    C = torch.empty(d, r, dtype=torch.float32, device=DEV)
    C_or = np.zeros((d, r), np.float32)
    for mb in range(mbs):
        D = synth.normal_bf16((T, d), 1e-3, 100 + mb)
        XPb = orc.bf16_from_double(np.random.default_rng(mb).standard_normal((T, r)) * 8)
        Dd = _padded_bf16(T, d)
        Dd.copy_(D.to(DEV))
        XPd = _padded_bf16(T, r)
        XPd.copy_(from_bits(XPb, DEV))
        rgs.accumulate(Dd, XPd, C, overwrite=(mb == 0))
        C_or = orc.accumulate(bits(D), XPb, C_or, overwrite=(mb == 0))
    _c_check(C.cpu().numpy(), C_or)


def test_accumulate_adds_to_existing_sketch():
    T, d, r = 96, 64, 8
    D = synth.normal_bf16((T, d), 1e-3, 4)
    XPb = orc.bf16_from_double(np.random.default_rng(1).standard_normal((T, r)))
    C0 = np.random.default_rng(2).standard_normal((d, r)).astype(np.float32) * 1e-3
    C = torch.from_numpy(C0).to(DEV)
    rgs.accumulate(D.to(DEV), from_bits(XPb, DEV), C, overwrite=False)
    _c_check(C.cpu().numpy(), orc.accumulate(bits(D), XPb, C0, overwrite=False))


def test_chained_sketch_matches_oracle_chain():
    """Single linear 256 x 512, r=16, 4 microbatches of 128 tokens, both
    projection kinds: GPU XP and C against the oracle's own chain."""
    d, k, r, T = 256, 512, 16, 128
    for kind in (rgs.PROJ_RADEMACHER, rgs.PROJ_GAUSSIAN_QR):
        P = torch.empty(k, r, dtype=torch.float32, device=DEV)
        rgs.sample_projection(kind, 0, 0, 0, P)
        P_or = orc.sample_projection(kind, 0, 0, 0, k, r)
        C = torch.empty(d, r, dtype=torch.float32, device=DEV)
        C_or = np.zeros((d, r), np.float32)
        for mb in range(4):
            X = synth.layer_x(T, k, 0, mb)
            D = synth.layer_d(T, d, 0, mb)
            XP = torch.empty(T, r, dtype=torch.bfloat16, device=DEV)
            rgs.project_inputs(X.to(DEV), P, XP)
            rgs.accumulate(D.to(DEV), XP, C, overwrite=(mb == 0))
            C_or = orc.accumulate(bits(D), orc.project_inputs(bits(X), P_or), C_or, overwrite=(mb == 0))
        assert rel_fro(C.cpu().numpy(), C_or) < 2e-3
        H = orc.rebuild(C.cpu().numpy(), P.cpu().numpy())
        H_or = orc.rebuild(C_or, P_or)
        assert rel_fro(H, H_or) < 2e-3


@pytest.mark.parametrize("T,d,r", [(4096, 12288, 64), (16384, 28672, 256), (16384, 8192, 4)])
def test_accumulate_full_size_sampled_rows(T, d, r):
    """d=12288 rows (the 8B stack's gate/up), 4096 tokens, r=64, and one
    16384-token response of the long-response sweep (d=28672 at r=256, d=8192
    at r=4), heavy-tailed D; 64 sampled rows of C computed by the oracle."""
    D = synth.layer_d(T, d, 5, 0, device=DEV, heavy_tail=True)
    XPb = orc.bf16_from_double(np.random.default_rng(3).standard_normal((T, r)) * 8)
    XP = _padded_bf16(T, r)
    XP.copy_(from_bits(XPb, DEV))
    C = torch.empty(d, r, dtype=torch.float32, device=DEV)
    rgs.accumulate(D, XP, C, overwrite=True)
    rows = np.sort(np.random.default_rng(1).choice(d, 64, replace=False))
    ref = orc.accumulate(bits(D[:, rows]), XPb, np.zeros((64, r), np.float32), overwrite=True)
    _c_check(C.cpu().numpy()[rows], ref)


@pytest.mark.parametrize("r", [64, 20])
def test_accumulate_many_tiles_matches_oracle(r):
    """A batched call with enough 128-row tiles of C to fill every SM twice
    (40,000 rows over five layers, one of them ragged) takes the persistent
    path; 320 tokens (five 64-token chunks), overwrite then add.  Sampled rows
    of every layer against the oracle."""
    T = 320
    ds = [12288, 12288, 8000, 4096, 3328]
    Ds = [synth.layer_d(T, d, 60 + i, 0, device=DEV) for i, d in enumerate(ds)]
    XPb = [orc.bf16_from_double(np.random.default_rng(70 + i).standard_normal((T, r)) * 4) for i in range(len(ds))]
    XPs = []
    for xb in XPb:
        XP = _padded_bf16(T, r)
        XP.copy_(from_bits(xb, DEV))
        XPs.append(XP)
    Cs = [torch.empty(d, r, dtype=torch.float32, device=DEV) for d in ds]
    rgs.accumulate_batched(Ds, XPs, Cs, overwrite=True)
    rgs.accumulate_batched(Ds, XPs, Cs, overwrite=False)
    for i, d in enumerate(ds):
        rows = np.sort(np.random.default_rng(i).choice(d, 48, replace=False))
        rows[-1] = d - 1
        Db = bits(Ds[i][:, rows])
        ref = orc.accumulate(Db, XPb[i], np.zeros((48, r), np.float32), overwrite=True)
        ref = orc.accumulate(Db, XPb[i], ref, overwrite=False)
        _c_check(Cs[i].cpu().numpy()[rows], ref)


@pytest.mark.parametrize("T,d,k,r", [(300, 136, 512, 16), (256, 256, 1024, 64), (130, 72, 256, 20),
                                     (64, 128, 1024, 256)])
def test_fp32_xp_removes_the_xp_rounding_from_c(T, d, k, r):
    """The fp32-accurate XP (a BF16 pair) is within 2^-16 of the exact X P, and
    the sketch built from it is within 5e-5 of the exact D^T (X P): the BF16
    rounding of XP (about 1e-3 in C) is gone."""
    X = synth.normal_bf16((T, k), 1.0, 90 + T)
    D = synth.normal_bf16((T, d), 1e-3, 91 + T)
    P = orc.sample_qr(6, 1, 0, k, r) if 4 * r <= k else orc.sample_rademacher(6, 1, 0, k, r)
    n_pad = (r + 15) // 16 * 16
    XP2 = _padded_bf16(T, rgs.xp_split_cols(r))
    rgs.project_inputs_fp32xp_batched([X.to(DEV)], [torch.from_numpy(P).to(DEV)], [XP2])
    got = (XP2[:, :r].float() + XP2[:, n_pad:n_pad + r].float()).cpu().numpy().astype(np.float64)
    exact = orc.project_inputs_exact(bits(X), P)
    rms = math.sqrt(float(np.mean(exact * exact)))
    assert np.all(np.abs(got - exact) <= 2.0 ** -16 * np.abs(exact) + 1e-5 * rms)
    C = torch.full((d, r), float("nan"), dtype=torch.float32, device=DEV)
    rgs.accumulate_fp32xp_batched([D.to(DEV)], [XP2], [C], overwrite=True)
    C_exact = orc.accumulate_exact(bits(D), exact, np.zeros((d, r)))
    err32 = rel_fro(C.cpu().numpy(), C_exact)
    assert err32 <= 5e-5
    # the BF16-XP path on the same inputs, for scale
    XP1 = _padded_bf16(T, r)
    rgs.project_inputs(X.to(DEV), torch.from_numpy(P).to(DEV), XP1)
    C1 = torch.empty(d, r, dtype=torch.float32, device=DEV)
    rgs.accumulate(D.to(DEV), XP1, C1, overwrite=True)
    assert err32 * 10 <= rel_fro(C1.cpu().numpy(), C_exact)


# --------------------------------------------------------------------------
# (d) updates
# --------------------------------------------------------------------------

def _w_check(got_bits, ref_bits):
    same, maxd = w_parity(got_bits, ref_bits)
    assert maxd <= 1, "an element is more than one BF16 step from the oracle"
    assert same >= 0.9999, "only %.6f of W is bit-identical" % same
    return same


def _rand_c(d, r, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal((d, r)) * scale).astype(np.float32)


@pytest.mark.parametrize("d,k,r,kind", [(256, 512, 16, 1), (256, 512, 16, 0), (40, 24, 4, 0),
                                        (130, 136, 20, 1), (1024, 2048, 128, 1), (200, 520, 96, 1),
                                        (100, 600, 136, 1), (96, 256, 48, 0),
                                        (300, 4096, 256, 1), (7, 8, 1, 0), (192, 256, 256, 1),
                                        (64, 200, 72, 1)])
def test_normsgd_matches_oracle(d, k, r, kind):
    W0 = synth.layer_weight(d, k, 3)
    P = (orc.sample_qr(2, 3, 1, k, r) if kind == 1 and r <= k
         else orc.sample_rademacher(2, 3, 1, k, r))
    C = _rand_c(d, r, d + k)
    W = W0.to(DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    out = torch.zeros(1, dtype=torch.float64, device=DEV)
    rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3,
                             0, 3, 1, wnorm2_out=out, dev_status=status)
    assert int(status.item()) == 0
    W_or, st, _ = orc.update_normsgd(bits(W0), C, P, 1e-3, 0, 3, 1, dense_h_norm=(d * k <= 1 << 22))
    assert st == 0
    _w_check(bits(W), W_or)
    assert abs(out.item() - orc.norm_w(W_or) ** 2) <= 1e-6 * orc.norm_w(W_or) ** 2


@pytest.mark.parametrize("d,k,r", [(1100, 1024, 64), (300, 2048, 128)])
def test_normsgd_rows_of_very_different_scales(d, k, r):
    """Rows of C spread over eight orders of magnitude, some of them zero: the
    Gram chunks take their scale from the largest row norm, so the small rows
    ride far below it; ||H|| and W still match the oracle."""
    W0 = synth.layer_weight(d, k, 5)
    P = orc.sample_qr(3, 1, 2, k, r)
    rng = np.random.default_rng(d + r)
    C = rng.standard_normal((d, r)) * 10.0 ** rng.uniform(-6, 2, size=(d, 1))
    C[rng.choice(d, d // 10, replace=False)] = 0.0
    C = C.astype(np.float32)
    W = W0.to(DEV)
    status = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3, 4, 1, 2,
                             dev_status=status)
    assert int(status.item()) == 0
    W_or, st, _ = orc.update_normsgd(bits(W0), C, P, 1e-3, 4, 1, 2, dense_h_norm=True)
    assert st == 0
    _w_check(bits(W), W_or)


def test_square_frame_update_is_dense_normalized_sgd():
    """r = k: the device's own orthogonal frame makes H = C P^T the gradient
    G itself, so the device update is the textbook dense normalized SGD step
    W - tau ||W|| G / ||G||, rounded stochastically: every new weight lies
    within one BF16 step of that value, and W matches the oracle's update."""
    d, k = 160, 256
    r, tau = k, 1e-2
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 31, 2, 5, P)
    Pn = P.cpu().numpy()
    G = np.random.default_rng(12).standard_normal((d, k))
    C = (G @ Pn.astype(np.float64)).astype(np.float32)
    W0 = synth.layer_weight(d, k, 4)
    W = W0.to(DEV)
    rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), P, tau, 9, 2, 5)
    W_or, st, _ = orc.update_normsgd(bits(W0), C, Pn, tau, 9, 2, 5, dense_h_norm=True)
    assert st == 0
    _w_check(bits(W), W_or)
    w0 = orc.bf16_to_f32(bits(W0)).astype(np.float64)
    text = w0 - tau * np.linalg.norm(w0) * G / np.linalg.norm(G)
    got = orc.bf16_to_f32(bits(W)).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(text), 2.0 ** -126))) - 7)
    step = tau * np.linalg.norm(w0) * np.abs(G).max() / np.linalg.norm(G)
    assert np.all(np.abs(got - text) <= ulp + 1e-5 * step)


def test_normsgd_strided_w_keeps_padding():
    d, k, r, ld = 64, 96, 8, 104
    Wf = synth.normal_bf16((d, ld), 0.02, 5).to(DEV)
    pad_before = Wf[:, k:].clone()
    P = orc.sample_rademacher(0, 0, 0, k, r)
    C = _rand_c(d, r, 9)
    W0 = bits(Wf[:, :k])
    rgs.apply_update_normsgd(Wf[:, :k], torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV),
                             1e-3, 0, 0, 0)
    W_or, _, _ = orc.update_normsgd(W0, C, P, 1e-3, 0, 0, 0)
    _w_check(bits(Wf[:, :k]), W_or)
    assert torch.equal(Wf[:, k:], pad_before)


def test_normsgd_carried_norm_chain():
    """Two refreshed steps; the second reuses the ||W||^2 the first wrote."""
    d, k, r = 512, 1024, 32
    W = synth.layer_weight(d, k, 1).to(DEV)
    W_ref = bits(W)
    carried = torch.zeros(1, dtype=torch.float64, device=DEV)
    for step in range(2):
        P = torch.empty(k, r, dtype=torch.float32, device=DEV)
        rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 9, 1, step, P)
        C = _rand_c(d, r, 40 + step)
        rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), P, 1e-3, 9, 1, step,
                                 wnorm2_in=carried if step else None, wnorm2_out=carried)
        W_ref, st, _ = orc.update_normsgd(W_ref, C, P.cpu().numpy(), 1e-3, 9, 1, step)
        assert st == 0
        _w_check(bits(W), W_ref)


def test_normsgd_degenerate_inputs_leave_w_unchanged():
    d, k, r = 64, 128, 8
    W0 = synth.layer_weight(d, k, 0).to(DEV)
    P = torch.from_numpy(orc.sample_rademacher(0, 0, 0, k, r)).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    W = W0.clone()
    rgs.apply_update_normsgd(W, torch.zeros(d, r, device=DEV), P, 1e-3, 0, 0, 0, dev_status=status)
    assert int(status.item()) == binding.DEV_H_ZERO and torch.equal(W, W0)
    C = torch.ones(d, r, device=DEV)
    C[3, 2] = float("nan")
    rgs.apply_update_normsgd(W, C, P, 1e-3, 0, 0, 0, dev_status=status)
    assert int(status.item()) & binding.DEV_H_NONFINITE and torch.equal(W, W0)
    rgs.apply_update_normsgd(W, torch.ones(d, r, device=DEV), P, 0.0, 0, 0, 0, dev_status=status)
    assert int(status.item()) == 0 and torch.equal(W, W0)


@pytest.mark.parametrize("d,k,r", [(4096, 4096, 64), (256, 512, 16), (72, 40, 5)])
def test_sgd_matches_oracle(d, k, r):
    """The LoGRA worked example shape (d = k = 4096, r = 64, alpha*eta = 1e-4)
    with a sketch of the size 8 x 4096 tokens produce."""
    W0 = synth.layer_weight(d, k, 2)
    P = orc.sample_rademacher(0, 2, 0, k, r)
    C = _rand_c(d, r, 5, scale=1.45)
    W = W0.to(DEV)
    rgs.apply_update_sgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-4, 0, 2, 0)
    _w_check(bits(W), orc.update_sgd(bits(W0), C, P, 1e-4, 0, 2, 0))


@pytest.mark.parametrize("d,k,r", [(256, 1024, 64), (200, 520, 128), (130, 136, 20)])
def test_sgd_zero_weight_uses_exact_path(d, k, r):
    """Zero W: every v is -s*H, so no weight dominates v and the tensor-core
    error of H (a few 2^-20 of ||c|| ||p||) is many fp32 steps of v; the
    elements whose rounding margin that error might cross take the exact path,
    and W matches the definition as closely as for a trained-scale W."""
    W0 = torch.zeros(d, k, dtype=torch.bfloat16)
    P = orc.sample_qr(4, 1, 0, k, r) if 4 * r <= k else orc.sample_rademacher(4, 1, 0, k, r)
    C = _rand_c(d, r, 17)
    W = W0.to(DEV)
    rgs.read_exact_count()
    rgs.apply_update_sgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-2, 4, 1, 0)
    exact = rgs.read_exact_count()
    same, maxd = w_parity(bits(W), orc.update_sgd(bits(W0), C, P, 1e-2, 4, 1, 0))
    assert maxd <= 1 and same >= 0.9999, (same, maxd)
    assert 0 < exact < d * k


@pytest.mark.parametrize("update", ["normsgd", "sgd"])
def test_update_tiny_weights_match_oracle(update):
    """W ~ N(0, 1e-4), far below the trained scale: for LoGRA's SGD the step
    (alpha*eta = 1e-3 on a unit sketch) is then as large as the weights; for
    normalized SGD it stays tau of their norm.  Both match the definition."""
    d, k, r = 512, 1024, 64
    W0 = synth.normal_bf16((d, k), 1e-4, 77)
    P = orc.sample_qr(6, 2, 3, k, r)
    C = _rand_c(d, r, 23)
    W = W0.to(DEV)
    if update == "normsgd":
        rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3, 6, 2, 3)
        ref, st, _ = orc.update_normsgd(bits(W0), C, P, 1e-3, 6, 2, 3)
        assert st == 0
    else:
        rgs.apply_update_sgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3 / 64, 6, 2, 3)
        ref = orc.update_sgd(bits(W0), C, P, 1e-3 / 64, 6, 2, 3)
    _w_check(bits(W), ref)


@pytest.mark.parametrize("update", ["normsgd", "sgd"])
def test_update_rows_of_any_scale_match_oracle(update):
    """The tensor cores see C and P scaled by powers of two (each row of C,
    each 128 rows of P); rows of C from 1e-30 to 1e6, a zero row, and a P
    far from unit scale still match the definition, and a row too small for
    any usable scale goes through the exact path whole."""
    d, k, r = 384, 640, 32
    rng = np.random.default_rng(41)
    W0 = synth.layer_weight(d, k, 12)
    P = (orc.sample_qr(7, 1, 2, k, r) * 3e-4).astype(np.float32)
    C = _rand_c(d, r, 43)
    C *= (10.0 ** rng.uniform(-30, 6, size=(d, 1))).astype(np.float32)
    C[5] = 0.0
    C[6] *= 1e-12  # about 1e-40 at most: below the normal fp32 range
    W = W0.to(DEV)
    Cd, Pd = torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV)
    if update == "normsgd":
        rgs.apply_update_normsgd(W, Cd, Pd, 1e-3, 8, 3, 4)
        ref, st, _ = orc.update_normsgd(bits(W0), C, P, 1e-3, 8, 3, 4)
        assert st == 0
    else:
        rgs.apply_update_sgd(W, Cd, Pd, 1e-4, 8, 3, 4)
        ref = orc.update_sgd(bits(W0), C, P, 1e-4, 8, 3, 4)
    _w_check(bits(W), ref)
    assert rgs.read_device_errors() == 0


def test_exact_path_is_rare_at_trained_scale():
    """At the trained scale W ~ N(0, 0.02) with tau = 1e-3 only the few
    elements with a tiny weight or a rounding sum within a few steps of a carry
    take the exact path (well under 1 in 1000)."""
    d, k, r = 1024, 2048, 64
    W0 = synth.layer_weight(d, k, 9)
    P = orc.sample_qr(1, 9, 0, k, r)
    C = _rand_c(d, r, 31)
    W = W0.to(DEV)
    rgs.read_exact_count()
    rgs.apply_update_normsgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3, 1, 9, 0)
    exact = rgs.read_exact_count()
    ref, st, _ = orc.update_normsgd(bits(W0), C, P, 1e-3, 1, 9, 0)
    _w_check(bits(W), ref)
    assert exact < 1e-3 * d * k, exact


def test_sgd_nan_sketch_row_gives_canonical_nan():
    """A NaN in row 5 of C makes row 5 of H NaN: that row of W becomes the
    canonical NaN, every other row is unaffected."""
    d, k, r = 256, 512, 16
    W0 = synth.layer_weight(d, k, 2)
    P = orc.sample_rademacher(0, 2, 0, k, r)
    C = _rand_c(d, r, 5)
    C[5, 2] = np.nan
    W = W0.to(DEV)
    rgs.apply_update_sgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-4, 0, 2, 0)
    ref = orc.update_sgd(bits(W0), C, P, 1e-4, 0, 2, 0)
    got = bits(W)
    assert np.all(ref[5] == 0x7FC0) and np.array_equal(got[5], ref[5])
    _w_check(np.delete(got, 5, 0), np.delete(ref, 5, 0))


def test_sgd_nonfinite_weights_follow_the_definition():
    """NaN weights of any payload (quiet, with a small payload, negative) give
    the canonical BF16 NaN; +-Inf weights stay +-Inf (v = Inf - s H); every
    other element is unaffected, with whole 8-column groups of NaN and Inf
    neighbours among them."""
    d, k, r = 128, 256, 16
    W0 = synth.layer_weight(d, k, 4)
    specials = {(3, 5): 0x7FC0, (3, 6): 0x7F81, (17, 200): 0xFFC0, (64, 0): 0x7F80,
                (65, 255): 0xFF80, (100, 8): 0x7FFF, (127, 129): 0xFF81}
    for (i, j), b in specials.items():
        W0[i, j] = torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)[0]
    P = orc.sample_rademacher(1, 0, 0, k, r)
    C = _rand_c(d, r, 8)
    W = W0.to(DEV)
    rgs.apply_update_sgd(W, torch.from_numpy(C).to(DEV), torch.from_numpy(P).to(DEV), 1e-3, 1, 0, 0)
    ref = orc.update_sgd(bits(W0), C, P, 1e-3, 1, 0, 0)
    got = bits(W)
    for (i, j), b in specials.items():
        expect = 0x7F80 if b == 0x7F80 else 0xFF80 if b == 0xFF80 else 0x7FC0
        assert ref[i, j] == expect and got[i, j] == expect, ((i, j), hex(got[i, j]), hex(ref[i, j]))
    _w_check(got, ref)


@pytest.mark.parametrize("kind", [rgs.PROJ_GAUSSIAN_QR, rgs.PROJ_RADEMACHER])
def test_policy_sync_receiver_matches_trainer(kind):
    """A rollout worker that receives (U, alpha*eta, seed, layer, step),
    regenerates P and applies the update ends with the trainer's W, bit for
    bit; both match the oracle's SGD update."""
    d, k, r, seed, layer, step = 512, 1024, 32, 7, 2, 5
    W0 = synth.layer_weight(d, k, 6)
    C = torch.from_numpy(_rand_c(d, r, 3)).to(DEV)
    P_t = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(kind, seed, layer, step, P_t)
    msg = policy_sync.message(C, 1e-4, seed, layer, step)
    W_t = W0.to(DEV)
    policy_sync.apply(W_t, msg, P_t)
    rx = policy_sync.Message(torch.from_numpy(msg.U.cpu().numpy().copy()).to(DEV), msg.alpha_eta, msg.seed,
                             msg.layer, msg.step)  # what travels
    P_r = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(kind, rx.seed, rx.layer, rx.step, P_r)  # regenerated, not sent
    W_r = W0.to(DEV)
    policy_sync.apply(W_r, rx, P_r)
    assert torch.equal(P_t, P_r)
    assert torch.equal(bits_t(W_t), bits_t(W_r))
    _w_check(bits(W_t), orc.update_sgd(bits(W0), C.cpu().numpy(), P_t.cpu().numpy(), 1e-4, seed, layer, step))
    assert policy_sync.payload_bytes(d, r) == 4 * d * r + 20 < 2 * d * k


@pytest.mark.parametrize("d,k,r", [(12288, 4096, 64), (2048, 6144, 256), (28672, 8192, 16)])
def test_normsgd_full_size_sampled_rows(d, k, r):
    """Full layer shapes of the Qwen3 stacks and the long-response sweep; the
    oracle computes s from the whole W and the Gram route, then the sampled
    rows one by one."""
    W = synth.layer_weight(d, k, 4, device=DEV)
    W0_bits = bits(W)
    P = torch.empty(k, r, dtype=torch.float32, device=DEV)
    rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 1, 4, 0, P)
    C = torch.from_numpy(_rand_c(d, r, 11)).to(DEV)
    rgs.apply_update_normsgd(W, C, P, 1e-3, 1, 4, 0)
    Cn, Pn = C.cpu().numpy(), P.cpu().numpy()
    s, st = orc.normsgd_scale(orc.norm_w(W0_bits), orc.norm_h_gram(Cn, Pn), 1e-3)
    assert st == 0
    rows = np.sort(np.random.default_rng(d).choice(d, 16, replace=False)).astype(np.int32)
    ref = orc.update_rows(W0_bits[rows], rows, Cn, Pn, s, 1, 4, 0)
    _w_check(bits(W)[rows], ref)


def test_update_repeatable():
    d, k, r = 512, 512, 32
    W0 = synth.layer_weight(d, k, 0).to(DEV)
    P = torch.from_numpy(orc.sample_qr(0, 0, 0, k, r)).to(DEV)
    C = torch.from_numpy(_rand_c(d, r, 0)).to(DEV)
    a, b = W0.clone(), W0.clone()
    rgs.apply_update_normsgd(a, C, P, 1e-3, 0, 0, 0)
    rgs.apply_update_normsgd(b, C, P, 1e-3, 0, 0, 0)
    assert torch.equal(a, b) and not torch.equal(a, W0)


def test_calls_on_a_side_stream():
    d, k, r, T = 128, 256, 16, 64
    s = torch.cuda.Stream()
    X = synth.normal_bf16((T, k), 1.0, 1).to(DEV)
    D = synth.normal_bf16((T, d), 1e-3, 2).to(DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        P = torch.empty(k, r, dtype=torch.float32, device=DEV)
        rgs.sample_projection(rgs.PROJ_GAUSSIAN_QR, 3, 0, 0, P, stream=s)
        XP = torch.empty(T, r, dtype=torch.bfloat16, device=DEV)
        rgs.project_inputs(X, P, XP, stream=s)
        C = torch.empty(d, r, dtype=torch.float32, device=DEV)
        rgs.accumulate(D, XP, C, overwrite=True, stream=s)
    s.synchronize()
    P_or = orc.sample_qr(3, 0, 0, k, r)
    C_or = orc.accumulate(bits(D), orc.project_inputs(bits(X), P_or), np.zeros((d, r)), True)
    assert rel_fro(C.cpu().numpy(), C_or) < 2e-3


# --------------------------------------------------------------------------
# batched calls: one call per phase for a stack of layers
# --------------------------------------------------------------------------

STACK = [(256, 512), (128, 512), (520, 256), (64, 1024), (200, 136)]  # (d, k), ragged shapes


@pytest.mark.parametrize("kind", [0, 1])
def test_batched_stack_matches_oracle(kind):
    """Projection, projected inputs, accumulation and both updates for a small
    stack of differently shaped layers, each compared with the oracle."""
    r, T, step, seed = 16, 96, 2, 11
    layers = list(range(len(STACK)))
    Ps = [torch.empty(k, r, dtype=torch.float32, device=DEV) for _, k in STACK]
    rgs.sample_projection_batched(kind, seed, step, Ps, layers)
    for li, (_, k) in enumerate(STACK):
        ref = orc.sample_projection(kind, seed, li, step, k, r)
        if kind == 0:
            assert np.array_equal(Ps[li].cpu().numpy().view(np.uint32), ref.view(np.uint32))
        else:
            assert rel_fro(Ps[li].cpu().numpy(), ref) < 1e-5
    Xs = [synth.normal_bf16((T, k), 1.0, 300 + li) for li, (_, k) in enumerate(STACK)]
    Ds = [synth.normal_bf16((T, d), 1e-3, 400 + li) for li, (d, _) in enumerate(STACK)]
    XPs = [_padded_bf16(T, r) for _ in STACK]
    rgs.project_inputs_batched([X.to(DEV) for X in Xs], Ps, XPs)
    Cs = [torch.full((d, r), 5.0, dtype=torch.float32, device=DEV) for d, _ in STACK]
    rgs.accumulate_batched([D.to(DEV) for D in Ds], XPs, Cs, overwrite=True)
    for li in layers:
        Pn = Ps[li].cpu().numpy()
        _xp_check(bits(XPs[li]), orc.project_inputs(bits(Xs[li]), Pn))
        C_or = orc.accumulate(bits(Ds[li]), bits(XPs[li]), np.zeros((STACK[li][0], r)), True)
        _c_check(Cs[li].cpu().numpy(), C_or)
    W0 = [synth.layer_weight(d, k, li) for li, (d, k) in enumerate(STACK)]
    Ws = [w.to(DEV) for w in W0]
    out = [torch.zeros(1, dtype=torch.float64, device=DEV) for _ in STACK]
    st = [torch.full((1,), -1, dtype=torch.int32, device=DEV) for _ in STACK]
    rgs.apply_update_normsgd_batched(Ws, Cs, Ps, 1e-3, seed, layers, step, wnorm2_out=out, dev_status=st)
    Ws2 = [w.to(DEV) for w in W0]
    rgs.apply_update_sgd_batched(Ws2, Cs, Ps, 1e-4, seed, layers, step)
    for li in layers:
        Cn, Pn = Cs[li].cpu().numpy(), Ps[li].cpu().numpy()
        W_or, s_or, _ = orc.update_normsgd(bits(W0[li]), Cn, Pn, 1e-3, seed, li, step)
        assert s_or == 0 and int(st[li].item()) == 0
        _w_check(bits(Ws[li]), W_or)
        assert abs(out[li].item() - orc.norm_w(W_or) ** 2) <= 1e-6 * orc.norm_w(W_or) ** 2
        _w_check(bits(Ws2[li]), orc.update_sgd(bits(W0[li]), Cn, Pn, 1e-4, seed, li, step))


def test_batched_calls_span_several_launches():
    """More layers than one launch's parameter table holds (96 GEMM problems,
    60 update problems, 128 norm problems): every layer still matches."""
    n, d, k, r, T = 140, 72, 64, 8, 40
    layers = list(range(n))
    Ps = [torch.empty(k, r, dtype=torch.float32, device=DEV) for _ in range(n)]
    rgs.sample_projection_batched(rgs.PROJ_RADEMACHER, 3, 0, Ps, layers)
    X = synth.normal_bf16((T, k), 1.0, 9).to(DEV)
    D = synth.normal_bf16((T, d), 1e-3, 10).to(DEV)
    XPs = [_padded_bf16(T, r) for _ in range(n)]
    rgs.project_inputs_batched([X] * n, Ps, XPs)
    Cs = [torch.empty(d, r, dtype=torch.float32, device=DEV) for _ in range(n)]
    rgs.accumulate_batched([D] * n, XPs, Cs, overwrite=True)
    W0 = synth.layer_weight(d, k, 0)
    Ws = [W0.to(DEV) for _ in range(n)]
    rgs.apply_update_normsgd_batched(Ws, Cs, Ps, 1e-3, 3, layers, 0)
    for li in (0, 59, 60, 95, 96, 127, 128, 139):
        Pn = Ps[li].cpu().numpy()
        assert np.array_equal(Pn.view(np.uint32), orc.sample_rademacher(3, li, 0, k, r).view(np.uint32))
        XP_or = orc.project_inputs(bits(X), Pn)
        _xp_check(bits(XPs[li]), XP_or)
        C_or = orc.accumulate(bits(D), bits(XPs[li]), np.zeros((d, r)), True)
        _c_check(Cs[li].cpu().numpy(), C_or)
        W_or, st, _ = orc.update_normsgd(bits(W0), Cs[li].cpu().numpy(), Pn, 1e-3, 3, li, 0)
        _w_check(bits(Ws[li]), W_or)


# --------------------------------------------------------------------------
# reconstruction diagnostic over ranks and projection kinds
# --------------------------------------------------------------------------

def test_reconstruction_cosine_follows_closed_forms():
    """cos(G, H) of the library's sketch against the dense gradient, for both
    projection kinds over r in {4, 16, 64, 256}: one step matches the closed
    form; averaging over 8 refreshed projections matches its closed form and
    beats a fixed projection."""
    d, k, T = 256, 1024, 256
    Ds = [synth.normal_bf16((T, d), 1.0, 70 + m).to(DEV) for m in range(2)]
    Xs = [synth.normal_bf16((T, k), 1.0, 80 + m).to(DEV) for m in range(2)]
    rows = diagnostics.sweep(Ds, Xs, ranks=(4, 16, 64, 256), steps=8)
    assert len(rows) == 16
    by = {(row["kind"], row["r"], row["refreshed"]): row for row in rows}
    for (kind, r, refreshed), row in by.items():
        if not refreshed:  # one fixed projection: the single-step closed form
            single = diagnostics.expected_cosine(
                binding.PROJ_RADEMACHER if kind == "rademacher" else binding.PROJ_GAUSSIAN_QR, k, r, 1)
            assert abs(row["cos"] - single) <= 0.15 * single, row
        else:
            assert abs(row["cos"] - row["expected_cos"]) <= 0.15 * row["expected_cos"], row
            assert row["cos"] > by[(kind, r, False)]["cos"], row


@pytest.mark.parametrize("kind,r", [(rgs.PROJ_RADEMACHER, 16), (rgs.PROJ_GAUSSIAN_QR, 64)])
def test_reconstruction_cosine_matches_oracle(kind, r):
    """One fixed projection: the diagnostic's cos(G, H) and ||H - G|| / ||G||
    from the library's sketch agree with the oracle's (its own projection,
    projected inputs, fp32 sketch and H = C P^T in double) within the sketch
    tolerance."""
    d, k, T, seed, layer = 256, 1024, 256, 0, 0
    Dh = [synth.normal_bf16((T, d), 1.0, 170 + m) for m in range(2)]
    Xh = [synth.normal_bf16((T, k), 1.0, 180 + m) for m in range(2)]
    cos, rel = diagnostics.reconstruction([D.to(DEV) for D in Dh], [X.to(DEV) for X in Xh], r, kind,
                                          steps=1, refreshed=False, seed=seed, layer=layer)
    P = orc.sample_projection(kind, seed, layer, 0, k, r)
    C = np.zeros((d, r), np.float32)
    for m in range(2):
        C = orc.accumulate(bits(Dh[m]), orc.project_inputs(bits(Xh[m]), P), C, overwrite=(m == 0))
    H = orc.rebuild(C, P)
    G = sum(np.asarray(D.float().numpy(), np.float64).T @ np.asarray(X.float().numpy(), np.float64)
            for D, X in zip(Dh, Xh))
    cos_or = float((G * H).sum() / (np.linalg.norm(G) * np.linalg.norm(H)))
    rel_or = float(np.linalg.norm(H - G) / np.linalg.norm(G))
    assert abs(cos - cos_or) <= 2e-3 * abs(cos_or), (cos, cos_or)
    assert abs(rel - rel_or) <= 2e-3 * rel_or, (rel, rel_or)
