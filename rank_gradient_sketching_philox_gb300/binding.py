"""Thin Python binding of libsketch (include/sketch.h).

Argument marshalling only: every step of the method runs in the library's CUDA
kernels.  PyTorch supplies device memory (including the workspace each call
needs) and the stream.  There is no CPU fallback: if the compiled library is
missing, every call raises.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libsketch.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4

PROJ_RADEMACHER = 0
PROJ_GAUSSIAN_QR = 1

OP_SAMPLE_PROJECTION = 0
OP_PROJECT_INPUTS = 1
OP_ACCUMULATE = 2
OP_UPDATE_NORMSGD = 3
OP_UPDATE_SGD = 4

DEV_H_ZERO = 1
DEV_H_NONFINITE = 2
DEV_W_NONFINITE = 4
DEV_QR_BREAKDOWN = 8

EXPORTS = ("sketch_workspace_bytes", "sketch_sample_projection", "sketch_project_inputs",
           "sketch_accumulate", "sketch_apply_update_normsgd", "sketch_apply_update_sgd",
           "sketch_workspace_bytes_batched", "sketch_sample_projection_batched",
           "sketch_project_inputs_batched", "sketch_accumulate_batched",
           "sketch_apply_update_normsgd_batched", "sketch_apply_update_sgd_batched",
           "sketch_apply_update_normsgd_noalloc", "sketch_noalloc_scratch_bytes",
           "sketch_read_device_errors", "sketch_read_exact_count", "sketch_kernel_launches",
           "sketch_projection_split_elems",
           "sketch_split_projection_batched", "sketch_project_inputs_fp32xp_batched",
           "sketch_accumulate_fp32xp_batched", "sketch_split_projection_grouped", "sketch_status_string",
           "sketch_last_error")


class ProjectionProblem(ctypes.Structure):
    _fields_ = [("P", ctypes.c_void_p), ("k", ctypes.c_int64), ("layer", ctypes.c_uint32)]


class ProjectProblem(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("T", ctypes.c_int64), ("k", ctypes.c_int64),
                ("ld_x", ctypes.c_int64), ("P", ctypes.c_void_p), ("XP", ctypes.c_void_p),
                ("ld_xp", ctypes.c_int64), ("P_split", ctypes.c_void_p)]


class SplitProblem(ctypes.Structure):
    _fields_ = [("P", ctypes.c_void_p), ("k", ctypes.c_int64), ("P_split", ctypes.c_void_p)]


class AccumulateProblem(ctypes.Structure):
    _fields_ = [("D", ctypes.c_void_p), ("T", ctypes.c_int64), ("d", ctypes.c_int64),
                ("ld_d", ctypes.c_int64), ("XP", ctypes.c_void_p), ("ld_xp", ctypes.c_int64),
                ("C", ctypes.c_void_p)]


class UpdateProblem(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("d", ctypes.c_int64), ("k", ctypes.c_int64),
                ("ld_w", ctypes.c_int64), ("C", ctypes.c_void_p), ("P", ctypes.c_void_p),
                ("layer", ctypes.c_uint32), ("wnorm2_in", ctypes.c_void_p),
                ("wnorm2_out", ctypes.c_void_p), ("dev_status", ctypes.c_void_p)]


class SketchError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s (status %d)" % (message, status))
        self.status = status


_lib = None
_c = ctypes
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64
_SIGS = {
    "sketch_workspace_bytes": (ctypes.c_size_t, [_c.c_int, _i64, _i64, _i64, _i64]),
    "sketch_sample_projection": (_c.c_int, [_c.c_int, _u64, _u32, _u32, _i64, _i64, _vp, _vp, _vp,
                                            _c.c_size_t, _vp]),
    "sketch_project_inputs": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp,
                                         _c.c_size_t, _vp]),
    "sketch_accumulate": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _c.c_int, _vp,
                                     _c.c_size_t, _vp]),
    "sketch_apply_update_normsgd": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _c.c_float,
                                               _u64, _u32, _u32, _vp, _vp, _vp, _vp, _c.c_size_t,
                                               _vp]),
    "sketch_apply_update_sgd": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _c.c_float, _u64,
                                           _u32, _u32, _vp, _vp, _c.c_size_t, _vp]),
    "sketch_read_device_errors": (_c.c_int, [_c.POINTER(_c.c_int32), _vp]),
    "sketch_read_exact_count": (_c.c_int, [_c.POINTER(_c.c_uint64), _vp]),
    "sketch_kernel_launches": (_c.c_uint64, []),
    "sketch_projection_split_elems": (_c.c_size_t, [_i64, _i64]),
    "sketch_split_projection_batched": (_c.c_int, [_c.c_int, _vp, _i64, _vp]),
    "sketch_split_projection_grouped": (_c.c_int, [_c.c_int, _vp, _i64, _vp]),
    "sketch_project_inputs_fp32xp_batched": (_c.c_int, [_c.c_int, _vp, _i64, _vp, _c.c_size_t, _vp]),
    "sketch_accumulate_fp32xp_batched": (_c.c_int, [_c.c_int, _vp, _i64, _c.c_int, _vp, _c.c_size_t, _vp]),
    "sketch_workspace_bytes_batched": (ctypes.c_size_t, [_c.c_int, _c.c_int, _vp, _vp, _vp, _i64]),
    "sketch_sample_projection_batched": (_c.c_int, [_c.c_int, _u64, _u32, _c.c_int, _vp, _i64, _vp, _vp,
                                                    _c.c_size_t, _vp]),
    "sketch_project_inputs_batched": (_c.c_int, [_c.c_int, _vp, _i64, _vp, _c.c_size_t, _vp]),
    "sketch_accumulate_batched": (_c.c_int, [_c.c_int, _vp, _i64, _c.c_int, _vp, _c.c_size_t, _vp]),
    "sketch_apply_update_normsgd_batched": (_c.c_int, [_c.c_int, _vp, _i64, _c.c_float, _u64, _u32, _vp,
                                                       _c.c_size_t, _vp]),
    "sketch_apply_update_sgd_batched": (_c.c_int, [_c.c_int, _vp, _i64, _c.c_float, _u64, _u32, _vp,
                                                   _c.c_size_t, _vp]),
    "sketch_apply_update_normsgd_noalloc": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _c.c_float,
                                                       _u64, _u32, _u32, _vp, _vp, _vp, _vp]),
    "sketch_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "sketch_status_string": (_c.c_char_p, [_c.c_int]),
    "sketch_last_error": (_c.c_char_p, []),
}


def lib():
    """Load libsketch.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsketch.so is not built (expected at %s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(status):
    if status != OK:
        l = lib()
        raise SketchError(status, "%s: %s" % (l.sketch_status_string(status).decode(),
                                              l.sketch_last_error().decode()))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream), s


def _rows(t, dtype, name):
    """Row-major 2-D CUDA tensor of ``dtype`` with unit column stride; returns ld."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("%s must be 2-D with unit column stride" % name)
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], ((t.shape[1] + 7) // 8) * 8)


def _contig(t, dtype, name):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


def _workspace(nbytes, device, stream, given=None):
    """The caller's workspace tensor if given (checked), else a fresh one."""
    if nbytes == 0:
        return None
    if given is not None:
        if not given.is_cuda or given.numel() * given.element_size() < nbytes:
            raise ValueError("workspace needs %d bytes" % nbytes)
        return given
    with torch.cuda.stream(stream):
        return torch.empty(nbytes, dtype=torch.uint8, device=device)


def read_device_errors(stream=None, device=None):
    """Read and clear the device error word (bits of timed-out waits); syncs the stream."""
    dev = device if device is not None else torch.cuda.current_device()
    h, _ = _stream_handle(stream, dev)
    flags = ctypes.c_int32(0)
    _check(lib().sketch_read_device_errors(ctypes.byref(flags), h))
    return int(flags.value)


def read_exact_count(stream=None, device=None):
    """Read and clear the count of weights the update calls recomputed on their
    exact path (instrumentation); syncs the stream."""
    dev = device if device is not None else torch.cuda.current_device()
    h, _ = _stream_handle(stream, dev)
    n = ctypes.c_uint64(0)
    _check(lib().sketch_read_exact_count(ctypes.byref(n), h))
    return int(n.value)


def kernel_launches():
    """Kernels this library has launched in this process (counted on the host)."""
    return int(lib().sketch_kernel_launches())


def workspace_bytes(op, T=0, d=0, k=0, r=1):
    return int(lib().sketch_workspace_bytes(op, T, d, k, r))


def sample_projection(kind, seed, layer, step, P, dev_status=None, stream=None):
    """Fill P (k x r fp32) with the projection for (seed, layer, step)."""
    _contig(P, torch.float32, "P")
    k, r = P.shape
    h, s = _stream_handle(stream, P.device)
    nbytes = workspace_bytes(OP_SAMPLE_PROJECTION, 0, 0, k, r) if kind == PROJ_GAUSSIAN_QR else 0
    ws = _workspace(nbytes, P.device, s)
    _check(lib().sketch_sample_projection(kind, seed & 0xFFFFFFFFFFFFFFFF, layer, step, k, r,
                                          _ptr(P), _ptr(dev_status), _ptr(ws), nbytes, h))
    return P


def project_inputs(X, P, XP, stream=None):
    """XP[:, :r] = bf16(X P)."""
    ld_x = _rows(X, torch.bfloat16, "X")
    ld_xp = _rows(XP, torch.bfloat16, "XP")
    _contig(P, torch.float32, "P")
    T, k = X.shape
    r = P.shape[1]
    if P.shape[0] != k or XP.shape[0] != T or XP.shape[1] < r:
        raise ValueError("shape mismatch: X %s, P %s, XP %s" % (tuple(X.shape), tuple(P.shape),
                                                                tuple(XP.shape)))
    h, s = _stream_handle(stream, X.device)
    nbytes = workspace_bytes(OP_PROJECT_INPUTS, T, 0, k, r)
    ws = _workspace(nbytes, X.device, s)
    _check(lib().sketch_project_inputs(_ptr(X), T, k, ld_x, _ptr(P), r, _ptr(XP), ld_xp, _ptr(ws),
                                       nbytes, h))
    return XP


def accumulate(D, XP, C, overwrite=False, r=None, stream=None):
    """C = (0 if overwrite else C) + D^T XP[:, :r]."""
    ld_d = _rows(D, torch.bfloat16, "D")
    ld_xp = _rows(XP, torch.bfloat16, "XP")
    _contig(C, torch.float32, "C")
    T, d = D.shape
    r = C.shape[1] if r is None else r
    if C.shape[0] != d or XP.shape[0] != T or XP.shape[1] < r or C.shape[1] != r:
        raise ValueError("shape mismatch: D %s, XP %s, C %s" % (tuple(D.shape), tuple(XP.shape),
                                                                tuple(C.shape)))
    h, s = _stream_handle(stream, D.device)
    nbytes = workspace_bytes(OP_ACCUMULATE, T, d, 0, r)
    ws = _workspace(nbytes, D.device, s)
    _check(lib().sketch_accumulate(_ptr(D), T, d, ld_d, _ptr(XP), ld_xp, r, _ptr(C),
                                   1 if overwrite else 0, _ptr(ws), nbytes, h))
    return C


def apply_update_normsgd(W, C, P, tau, seed, layer, step, wnorm2_in=None, wnorm2_out=None,
                         dev_status=None, stream=None):
    """W <- SR_bf16(W - tau ||W|| H / ||H||), H = C P^T, in place."""
    ld_w = _rows(W, torch.bfloat16, "W")
    _contig(C, torch.float32, "C")
    _contig(P, torch.float32, "P")
    d, k = W.shape
    r = C.shape[1]
    if C.shape[0] != d or P.shape != (k, r):
        raise ValueError("shape mismatch: W %s, C %s, P %s" % (tuple(W.shape), tuple(C.shape),
                                                               tuple(P.shape)))
    h, s = _stream_handle(stream, W.device)
    nbytes = workspace_bytes(OP_UPDATE_NORMSGD, 0, d, k, r)
    ws = _workspace(nbytes, W.device, s)
    _check(lib().sketch_apply_update_normsgd(_ptr(W), d, k, ld_w, _ptr(C), _ptr(P), r, float(tau),
                                             seed & 0xFFFFFFFFFFFFFFFF, layer, step,
                                             _ptr(wnorm2_in), _ptr(wnorm2_out), _ptr(dev_status),
                                             _ptr(ws), nbytes, h))
    return W


def apply_update_normsgd_noalloc(W, C, P, tau, seed, layer, step, wnorm2_in=None, wnorm2_out=None,
                                 dev_status=None, stream=None):
    """apply_update_normsgd without a workspace: the library's fixed device
    scratch array is used instead (for callers that cannot allocate)."""
    ld_w = _rows(W, torch.bfloat16, "W")
    _contig(C, torch.float32, "C")
    _contig(P, torch.float32, "P")
    d, k = W.shape
    r = C.shape[1]
    if C.shape[0] != d or P.shape != (k, r):
        raise ValueError("shape mismatch: W %s, C %s, P %s" % (tuple(W.shape), tuple(C.shape),
                                                               tuple(P.shape)))
    h, _ = _stream_handle(stream, W.device)
    _check(lib().sketch_apply_update_normsgd_noalloc(_ptr(W), d, k, ld_w, _ptr(C), _ptr(P), r,
                                                     float(tau), seed & 0xFFFFFFFFFFFFFFFF, layer,
                                                     step, _ptr(wnorm2_in), _ptr(wnorm2_out),
                                                     _ptr(dev_status), h))
    return W


def apply_update_sgd(W, C, P, alpha_eta, seed, layer, step, dev_status=None, stream=None):
    """W <- SR_bf16(W - alpha_eta C P^T), in place."""
    ld_w = _rows(W, torch.bfloat16, "W")
    _contig(C, torch.float32, "C")
    _contig(P, torch.float32, "P")
    d, k = W.shape
    r = C.shape[1]
    if C.shape[0] != d or P.shape != (k, r):
        raise ValueError("shape mismatch: W %s, C %s, P %s" % (tuple(W.shape), tuple(C.shape),
                                                               tuple(P.shape)))
    h, s = _stream_handle(stream, W.device)
    nbytes = workspace_bytes(OP_UPDATE_SGD, 0, d, k, r)
    ws = _workspace(nbytes, W.device, s)
    _check(lib().sketch_apply_update_sgd(_ptr(W), d, k, ld_w, _ptr(C), _ptr(P), r,
                                         float(alpha_eta), seed & 0xFFFFFFFFFFFFFFFF, layer, step,
                                         _ptr(dev_status), _ptr(ws), nbytes, h))
    return W


# --------------------------------------------------------------------------
# Batched forms: one call per phase for a whole stack of layers
# --------------------------------------------------------------------------

def _i64_array(vals):
    return (ctypes.c_int64 * len(vals))(*vals)


def workspace_bytes_batched(op, T=None, d=None, k=None, r=1):
    n = len(next(x for x in (T, d, k) if x is not None))
    arr = [None if x is None else _i64_array(x) for x in (T, d, k)]
    return int(lib().sketch_workspace_bytes_batched(
        op, n, *[None if a is None else ctypes.cast(a, ctypes.c_void_p) for a in arr], r))


def sample_projection_batched(kind, seed, step, Ps, layers, dev_status=None, ws=None, stream=None):
    """Fill every P (k_i x r fp32) for (seed, layers[i], step)."""
    n = len(Ps)
    r = Ps[0].shape[1]
    probs = (ProjectionProblem * n)()
    for i, (P, layer) in enumerate(zip(Ps, layers)):
        _contig(P, torch.float32, "P")
        if P.shape[1] != r:
            raise ValueError("all projections of a batch share r")
        probs[i] = ProjectionProblem(P.data_ptr(), P.shape[0], layer)
    h, s = _stream_handle(stream, Ps[0].device)
    nbytes = (workspace_bytes_batched(OP_SAMPLE_PROJECTION, k=[P.shape[0] for P in Ps], r=r)
              if kind == PROJ_GAUSSIAN_QR else 0)
    wsb = _workspace(nbytes, Ps[0].device, s, ws)
    _check(lib().sketch_sample_projection_batched(kind, seed & 0xFFFFFFFFFFFFFFFF, step, n, probs, r,
                                                  _ptr(dev_status), _ptr(wsb), nbytes, h))
    return Ps


def projection_split_elems(k, r):
    return int(lib().sketch_projection_split_elems(k, r))


def split_projection_batched(Ps, splits=None, stream=None):
    """BF16 splits of the projections Ps (k x r fp32) for project_inputs_batched;
    returns the list of split buffers (uint16, allocated when not given)."""
    n = len(Ps)
    r = Ps[0].shape[1]
    if splits is None:
        splits = [torch.empty(projection_split_elems(P.shape[0], r), dtype=torch.int16, device=P.device)
                  for P in Ps]
    probs = (SplitProblem * n)()
    for i, (P, S) in enumerate(zip(Ps, splits)):
        _contig(P, torch.float32, "P")
        if P.shape[1] != r or S.numel() * S.element_size() < 2 * projection_split_elems(P.shape[0], r):
            raise ValueError("shape mismatch in problem %d" % i)
        probs[i] = SplitProblem(P.data_ptr(), P.shape[0], S.data_ptr())
    h, _ = _stream_handle(stream, Ps[0].device)
    _check(lib().sketch_split_projection_batched(n, probs, r, h))
    return splits


class SplitGroup(ctypes.Structure):
    _fields_ = [("P", ctypes.c_void_p), ("m", ctypes.c_int), ("k", ctypes.c_int64), ("P_split", ctypes.c_void_p)]


def split_projection_grouped(groups, splits=None, stream=None):
    """Splits of concatenated projections: groups is a list of lists of P
    (k x r fp32, one k per group); group g's split is that of [P_0 | ... |
    P_{m-1}] (k x m r), for project_inputs_grouped_batched.  Returns the split
    buffers (uint16, allocated when not given)."""
    n = len(groups)
    r = groups[0][0].shape[1]
    if splits is None:
        splits = [torch.empty(projection_split_elems(g[0].shape[0], len(g) * r), dtype=torch.int16,
                              device=g[0].device) for g in groups]
    probs = (SplitGroup * n)()
    keep = []
    for i, (g, S) in enumerate(zip(groups, splits)):
        k = g[0].shape[0]
        for P in g:
            _contig(P, torch.float32, "P")
            if P.shape != (k, r):
                raise ValueError("shape mismatch in group %d" % i)
        if S.numel() * S.element_size() < 2 * projection_split_elems(k, len(g) * r):
            raise ValueError("split buffer of group %d too small" % i)
        ptrs = (ctypes.c_void_p * len(g))(*[P.data_ptr() for P in g])
        keep.append(ptrs)
        probs[i] = SplitGroup(ctypes.cast(ptrs, ctypes.c_void_p), len(g), k, S.data_ptr())
    h, _ = _stream_handle(stream, groups[0][0].device)
    _check(lib().sketch_split_projection_grouped(n, probs, r, h))
    return splits


def project_inputs_grouped_batched(Xs, splits, r_total, XPs, ws=None, stream=None):
    """XP = bf16(X [P_0 | ... | P_{m-1}]) (T x r_total, r_total = m r) for each
    problem, from the splits of split_projection_grouped; member q's XP is
    XP[:, q r:(q + 1) r]."""
    n = len(Xs)
    probs = (ProjectProblem * n)()
    for i, (X, S, XP) in enumerate(zip(Xs, splits, XPs)):
        ld_x = _rows(X, torch.bfloat16, "X")
        ld_xp = _rows(XP, torch.bfloat16, "XP")
        if XP.shape[0] != X.shape[0] or XP.shape[1] < r_total:
            raise ValueError("shape mismatch in problem %d" % i)
        if S.numel() * S.element_size() < 2 * projection_split_elems(X.shape[1], r_total):
            raise ValueError("split buffer of problem %d too small" % i)
        probs[i] = ProjectProblem(X.data_ptr(), X.shape[0], X.shape[1], ld_x, None, XP.data_ptr(), ld_xp,
                                  S.data_ptr())
    h, s = _stream_handle(stream, Xs[0].device)
    nbytes = workspace_bytes_batched(OP_PROJECT_INPUTS, T=[X.shape[0] for X in Xs],
                                     k=[X.shape[1] for X in Xs], r=r_total)
    wsb = _workspace(nbytes, Xs[0].device, s, ws)
    _check(lib().sketch_project_inputs_batched(n, probs, r_total, _ptr(wsb), nbytes, h))
    return XPs


def _project_batched(Xs, Ps, XPs, ws, stream, splits, fn, xp_cols):
    n = len(Xs)
    r = Ps[0].shape[1]
    probs = (ProjectProblem * n)()
    for i, (X, P, XP) in enumerate(zip(Xs, Ps, XPs)):
        ld_x = _rows(X, torch.bfloat16, "X")
        ld_xp = _rows(XP, torch.bfloat16, "XP")
        _contig(P, torch.float32, "P")
        if P.shape != (X.shape[1], r) or XP.shape[0] != X.shape[0] or XP.shape[1] < xp_cols:
            raise ValueError("shape mismatch in problem %d" % i)
        probs[i] = ProjectProblem(X.data_ptr(), X.shape[0], X.shape[1], ld_x, P.data_ptr(),
                                  XP.data_ptr(), ld_xp, splits[i].data_ptr() if splits is not None else None)
    h, s = _stream_handle(stream, Xs[0].device)
    nbytes = workspace_bytes_batched(OP_PROJECT_INPUTS, T=[X.shape[0] for X in Xs],
                                     k=[X.shape[1] for X in Xs], r=r)
    wsb = _workspace(nbytes, Xs[0].device, s, ws)
    _check(getattr(lib(), fn)(n, probs, r, _ptr(wsb), nbytes, h))
    return XPs


def project_inputs_batched(Xs, Ps, XPs, ws=None, stream=None, splits=None):
    """XP = bf16(X P) for each problem; `splits` (from split_projection_batched
    for these Ps) skips splitting P again."""
    return _project_batched(Xs, Ps, XPs, ws, stream, splits, "sketch_project_inputs_batched", Ps[0].shape[1])


def _accumulate_batched(Ds, XPs, Cs, overwrite, ws, stream, fn, xp_cols):
    n = len(Ds)
    r = Cs[0].shape[1]
    probs = (AccumulateProblem * n)()
    for i, (D, XP, C) in enumerate(zip(Ds, XPs, Cs)):
        ld_d = _rows(D, torch.bfloat16, "D")
        ld_xp = _rows(XP, torch.bfloat16, "XP")
        _contig(C, torch.float32, "C")
        if C.shape != (D.shape[1], r) or XP.shape[0] != D.shape[0] or XP.shape[1] < xp_cols:
            raise ValueError("shape mismatch in problem %d" % i)
        probs[i] = AccumulateProblem(D.data_ptr(), D.shape[0], D.shape[1], ld_d, XP.data_ptr(), ld_xp,
                                     C.data_ptr())
    h, s = _stream_handle(stream, Ds[0].device)
    nbytes = workspace_bytes_batched(OP_ACCUMULATE, T=[D.shape[0] for D in Ds],
                                     d=[D.shape[1] for D in Ds], r=r)
    wsb = _workspace(nbytes, Ds[0].device, s, ws)
    _check(getattr(lib(), fn)(n, probs, r, 1 if overwrite else 0, _ptr(wsb), nbytes, h))
    return Cs


def accumulate_batched(Ds, XPs, Cs, overwrite=False, ws=None, stream=None):
    return _accumulate_batched(Ds, XPs, Cs, overwrite, ws, stream, "sketch_accumulate_batched", Cs[0].shape[1])


def xp_split_cols(r):
    """Columns of the fp32-accurate XP form: a BF16 pair, 2 * round16(r)."""
    return 2 * ((r + 15) // 16 * 16)


def project_inputs_fp32xp_batched(Xs, Ps, XPs, ws=None, stream=None, splits=None):
    """XP kept to ~2^-17 relative as a BF16 pair (hi in columns [0, r), lo at
    [round16(r), round16(r) + r)); each XP is T x >= xp_split_cols(r) BF16."""
    return _project_batched(Xs, Ps, XPs, ws, stream, splits, "sketch_project_inputs_fp32xp_batched",
                            xp_split_cols(Ps[0].shape[1]))


def accumulate_fp32xp_batched(Ds, XPs, Cs, overwrite=False, ws=None, stream=None):
    """C = (0 or C) + D^T (XP_hi + XP_lo) from the fp32-accurate XP form."""
    return _accumulate_batched(Ds, XPs, Cs, overwrite, ws, stream, "sketch_accumulate_fp32xp_batched",
                               xp_split_cols(Cs[0].shape[1]))


def _update_batched(normsgd, Ws, Cs, Ps, step_size, seed, layers, step, wnorm2_in, wnorm2_out,
                    dev_status, ws, stream):
    n = len(Ws)
    r = Cs[0].shape[1]
    probs = (UpdateProblem * n)()
    for i in range(n):
        W, C, P = Ws[i], Cs[i], Ps[i]
        ld_w = _rows(W, torch.bfloat16, "W")
        _contig(C, torch.float32, "C")
        _contig(P, torch.float32, "P")
        if C.shape != (W.shape[0], r) or P.shape != (W.shape[1], r):
            raise ValueError("shape mismatch in problem %d" % i)
        pick = (lambda lst: None if lst is None else lst[i])
        probs[i] = UpdateProblem(W.data_ptr(), W.shape[0], W.shape[1], ld_w, C.data_ptr(), P.data_ptr(),
                                 layers[i], _ptr(pick(wnorm2_in)), _ptr(pick(wnorm2_out)),
                                 _ptr(pick(dev_status)))
    h, s = _stream_handle(stream, Ws[0].device)
    op = OP_UPDATE_NORMSGD if normsgd else OP_UPDATE_SGD
    nbytes = workspace_bytes_batched(op, d=[W.shape[0] for W in Ws], k=[W.shape[1] for W in Ws], r=r)
    wsb = _workspace(nbytes, Ws[0].device, s, ws)
    fn = lib().sketch_apply_update_normsgd_batched if normsgd else lib().sketch_apply_update_sgd_batched
    _check(fn(n, probs, r, float(step_size), seed & 0xFFFFFFFFFFFFFFFF, step, _ptr(wsb), nbytes, h))
    return Ws


def apply_update_normsgd_batched(Ws, Cs, Ps, tau, seed, layers, step, wnorm2_in=None, wnorm2_out=None,
                                 dev_status=None, ws=None, stream=None):
    """Normalized-SGD update of every W_i (lists of per-layer tensors; the
    optional lists hold one-element device tensors or None entries)."""
    return _update_batched(True, Ws, Cs, Ps, tau, seed, layers, step, wnorm2_in, wnorm2_out,
                           dev_status, ws, stream)


def apply_update_sgd_batched(Ws, Cs, Ps, alpha_eta, seed, layers, step, dev_status=None, ws=None,
                             stream=None):
    return _update_batched(False, Ws, Cs, Ps, alpha_eta, seed, layers, step, None, None, dev_status,
                           ws, stream)
