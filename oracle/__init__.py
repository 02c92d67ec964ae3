"""CPU oracle for randomized low-rank gradient sketching -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The GPU library never imports it and shares no code with it.
The arithmetic lives in ``sketch_oracle.c`` (plain loops in double precision);
this module only marshals numpy arrays into it.

Conventions: BF16 tensors travel as ``np.uint16`` bit patterns; the projection
P is k x r fp32 row-major; the sketch C is d x r fp32 row-major; W is d x k.

Every function below follows one definition of the method (page title and
section in the C file's header):

* ``sample_rademacher`` -- random signs scaled by 1/sqrt(r)
  ("LoGRA: Low-Rank Gradient Sketches", "Why the Sketch Can Be Accumulated
  Without a Full Gradient").
* ``sample_qr`` -- QR of a Gaussian matrix with the sign correction, scaled by
  sqrt(input width / rank) ("Randomized Gradient Compression", footnote 1).
* ``project_inputs`` -- XP = X P, saved instead of X
  ("Randomized Gradient Compression", "How it works").
* ``accumulate`` -- C += D^T (X P) in fp32 ("Randomized Gradient Compression",
  "How it works"; "LoGRA: Scaling LLM Reinforcement Learning with Low-Rank
  Gradient Sketches", Key Contributions 1).
* ``update_normsgd`` -- W <- W - tau ||W|| H / ||H|| with H = C P^T and BF16
  stochastic rounding ("Randomized Gradient Compression", "How it works").
* ``update_sgd`` -- W <- W - alpha*eta S A ("LoGRA: Low-Rank Gradient Sketches",
  "Why the Update Is Low-Rank but Not an Exact Recovery").

Parity pins: every function here is checked by the ``-m "not gpu"`` tests
against library routines (cuRAND's host Philox generator, LAPACK QR, numpy
matmul and SVD), closed forms and brute force; none is unpinned.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_c = ctypes
_SIGS = {
    "orc_philox4x32_10": (None, [_u32p, _u32p, _u32p]),
    "orc_philox_array": (None, [_u32p, _c.c_int, _u32p, _u32p]),
    "orc_sr_rand16_array": (None, [_c.c_uint64, _c.c_uint32, _c.c_uint32, _u64p, _c.c_int, _u32p]),
    "orc_sr_bf16_array": (None, [_f32p, _u32p, _c.c_int, _u16p]),
    "orc_bf16_from_double_array": (None, [_f64p, _c.c_int, _u16p]),
    "orc_sample_rademacher": (None, [_c.c_uint64, _c.c_uint32, _c.c_uint32, _c.c_int, _c.c_int, _f32p]),
    "orc_gaussian_matrix": (None, [_c.c_uint64, _c.c_uint32, _c.c_uint32, _c.c_int, _c.c_int, _f64p]),
    "orc_householder_qr": (None, [_c.c_int, _c.c_int, _f64p, _f64p, _f64p]),
    "orc_sample_qr": (None, [_c.c_uint64, _c.c_uint32, _c.c_uint32, _c.c_int, _c.c_int, _f32p,
                             _c.c_void_p]),
    "orc_project_inputs": (None, [_u16p, _c.c_int, _c.c_int, _c.c_int, _f32p, _c.c_int, _u16p, _c.c_int]),
    "orc_project_inputs_exact": (None, [_u16p, _c.c_int, _c.c_int, _c.c_int, _f32p, _c.c_int, _f64p]),
    "orc_accumulate": (None, [_u16p, _c.c_int, _c.c_int, _c.c_int, _u16p, _c.c_int, _c.c_int, _f32p,
                              _c.c_int]),
    "orc_accumulate_exact": (None, [_u16p, _c.c_int, _c.c_int, _c.c_int, _f64p, _c.c_int, _f64p]),
    "orc_rebuild": (None, [_f32p, _c.c_int, _f32p, _c.c_int, _c.c_int, _f64p]),
    "orc_norm_w": (_c.c_double, [_u16p, _c.c_int, _c.c_int, _c.c_int]),
    "orc_norm_h_dense": (_c.c_double, [_f32p, _c.c_int, _f32p, _c.c_int, _c.c_int]),
    "orc_norm_h_gram": (_c.c_double, [_f32p, _c.c_int, _f32p, _c.c_int, _c.c_int]),
    "orc_normsgd_scale": (_c.c_int, [_c.c_double, _c.c_double, _c.c_float, _c.POINTER(_c.c_float)]),
    "orc_update_rows": (None, [_u16p, _i32p, _c.c_int, _c.c_int, _c.c_int, _f32p, _f32p, _c.c_int,
                               _c.c_float, _c.c_uint64, _c.c_uint32, _c.c_uint32, _c.c_void_p]),
    "orc_update_normsgd": (_c.c_int, [_u16p, _c.c_int, _c.c_int, _c.c_int, _f32p, _f32p, _c.c_int,
                                      _c.c_float, _c.c_uint64, _c.c_uint32, _c.c_uint32, _c.c_int,
                                      _c.POINTER(_c.c_float)]),
    "orc_update_sgd": (None, [_u16p, _c.c_int, _c.c_int, _c.c_int, _f32p, _f32p, _c.c_int, _c.c_float,
                              _c.c_uint64, _c.c_uint32, _c.c_uint32]),
}

STATUS_H_ZERO = 1
STATUS_H_NONFINITE = 2
STATUS_W_NONFINITE = 4


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build_oracle())
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# --------------------------------------------------------------------------
# Philox and rounding
# --------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    """One Philox4x32-10 block: ``ctr`` four uint32 words, ``key`` two."""
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def philox_array(ctrs, key):
    ctrs = np.ascontiguousarray(ctrs, np.uint32).reshape(-1, 4)
    out = np.zeros_like(ctrs)
    lib().orc_philox_array(ctrs, ctrs.shape[0], np.asarray(key, np.uint32), out)
    return out


def sr_rand16(seed, layer, step, e):
    e = np.ascontiguousarray(e, np.uint64).ravel()
    out = np.zeros(e.shape, np.uint32)
    lib().orc_sr_rand16_array(seed, layer, step, e, e.size, out)
    return out


def sr_bf16(v, rand16):
    v = _f32(v).ravel()
    rand16 = np.ascontiguousarray(rand16, np.uint32).ravel()
    out = np.zeros(v.shape, np.uint16)
    lib().orc_sr_bf16_array(v, rand16, v.size, out)
    return out


def bf16_from_double(x):
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros(x.shape, np.uint16)
    lib().orc_bf16_from_double_array(x.ravel(), x.size, out.ravel())
    return out


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# (a) projection
# --------------------------------------------------------------------------

def sample_rademacher(seed, layer, step, k, r):
    P = np.zeros((k, r), np.float32)
    lib().orc_sample_rademacher(seed, layer, step, k, r, P)
    return P


def gaussian_matrix(seed, layer, step, k, r):
    G = np.zeros((k, r), np.float64)
    lib().orc_gaussian_matrix(seed, layer, step, k, r, G)
    return G


def householder_qr(A):
    A = np.ascontiguousarray(A, np.float64)
    m, n = A.shape
    Q = np.zeros((m, n), np.float64)
    R = np.zeros((n, n), np.float64)
    lib().orc_householder_qr(m, n, A, Q, R)
    return Q, R


def sample_qr(seed, layer, step, k, r, return_q=False):
    P = np.zeros((k, r), np.float32)
    Q = np.zeros((k, r), np.float64)
    lib().orc_sample_qr(seed, layer, step, k, r, P, Q.ctypes.data)
    return (P, Q) if return_q else P


def sample_projection(kind, seed, layer, step, k, r):
    """kind 0 = Rademacher, 1 = Gaussian QR (the library's enum values)."""
    if kind == 0:
        return sample_rademacher(seed, layer, step, k, r)
    if kind == 1:
        return sample_qr(seed, layer, step, k, r)
    raise ValueError("unknown projection kind %r" % (kind,))


# --------------------------------------------------------------------------
# (b), (c) projection of inputs and accumulation
# --------------------------------------------------------------------------

def project_inputs(X_bits, P):
    X_bits = _u16(X_bits)
    P = _f32(P)
    T, k = X_bits.shape
    r = P.shape[1]
    XP = np.zeros((T, r), np.uint16)
    lib().orc_project_inputs(X_bits, T, k, k, P, r, XP, r)
    return XP


def project_inputs_exact(X_bits, P):
    X_bits = _u16(X_bits)
    P = _f32(P)
    T, k = X_bits.shape
    r = P.shape[1]
    XP = np.zeros((T, r), np.float64)
    lib().orc_project_inputs_exact(X_bits, T, k, k, P, r, XP)
    return XP


def accumulate(D_bits, XP_bits, C, overwrite=False):
    """Return a new fp32 C = (0 if overwrite else C) + D^T XP."""
    D_bits = _u16(D_bits)
    XP_bits = _u16(XP_bits)
    T, d = D_bits.shape
    r = XP_bits.shape[1]
    C = np.array(C, np.float32, copy=True, order="C").reshape(d, r)
    lib().orc_accumulate(D_bits, T, d, d, XP_bits, r, r, C, 1 if overwrite else 0)
    return C


def accumulate_exact(D_bits, XP, C):
    D_bits = _u16(D_bits)
    XP = np.ascontiguousarray(XP, np.float64)
    T, d = D_bits.shape
    r = XP.shape[1]
    C = np.array(C, np.float64, copy=True, order="C").reshape(d, r)
    lib().orc_accumulate_exact(D_bits, T, d, d, XP, r, C)
    return C


# --------------------------------------------------------------------------
# (d) rebuild, norms and updates
# --------------------------------------------------------------------------

def rebuild(C, P):
    C = _f32(C)
    P = _f32(P)
    d, r = C.shape
    k = P.shape[0]
    H = np.zeros((d, k), np.float64)
    lib().orc_rebuild(C, d, P, k, r, H)
    return H


def norm_w(W_bits):
    W_bits = _u16(W_bits)
    d, k = W_bits.shape
    return lib().orc_norm_w(W_bits, d, k, k)


def norm_h_dense(C, P):
    C = _f32(C)
    P = _f32(P)
    return lib().orc_norm_h_dense(C, C.shape[0], P, P.shape[0], C.shape[1])


def norm_h_gram(C, P):
    C = _f32(C)
    P = _f32(P)
    return lib().orc_norm_h_gram(C, C.shape[0], P, P.shape[0], C.shape[1])


def normsgd_scale(norm_w_value, norm_h_value, tau):
    s = ctypes.c_float(0.0)
    status = lib().orc_normsgd_scale(norm_w_value, norm_h_value, tau, ctypes.byref(s))
    return s.value, status


def update_rows(W_rows_bits, rows, C, P, s, seed, layer, step, return_v=False):
    """Update the listed rows of W (given as ``W_rows_bits``, one row per index)."""
    W = np.array(W_rows_bits, np.uint16, copy=True, order="C")
    rows = np.ascontiguousarray(rows, np.int32)
    C = _f32(C)
    P = _f32(P)
    nrows, k = W.shape
    r = C.shape[1]
    v = np.zeros((nrows, k), np.float32) if return_v else None
    lib().orc_update_rows(W, rows, nrows, k, k, C, P, r, s, seed, layer, step,
                          v.ctypes.data if return_v else None)
    return (W, v) if return_v else W


def update_normsgd(W_bits, C, P, tau, seed, layer, step, dense_h_norm=True):
    """Return (W_new, status, s)."""
    W = np.array(W_bits, np.uint16, copy=True, order="C")
    C = _f32(C)
    P = _f32(P)
    d, k = W.shape
    s = ctypes.c_float(0.0)
    status = lib().orc_update_normsgd(W, d, k, k, C, P, C.shape[1], tau, seed, layer, step,
                                      1 if dense_h_norm else 0, ctypes.byref(s))
    return W, status, s.value


def update_sgd(W_bits, C, P, alpha_eta, seed, layer, step):
    W = np.array(W_bits, np.uint16, copy=True, order="C")
    C = _f32(C)
    P = _f32(P)
    d, k = W.shape
    lib().orc_update_sgd(W, d, k, k, C, P, C.shape[1], alpha_eta, seed, layer, step)
    return W
