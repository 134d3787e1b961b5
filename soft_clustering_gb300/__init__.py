"""Python binding of libgmm (include/gmm.h): the fused GMM EM step and top-m
soft assignment on one GB300.

Argument marshalling only.  Every function here has the name of the C entry
point it calls and forwards device pointers taken from torch tensors (or
plain integers) plus sizes; all arithmetic runs in the library's CUDA
kernels.  There is no CPU fallback: if ``_build/libgmm.so`` has not been
built (``python -m soft_clustering_gb300.build``) every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgmm.so")

GMM_COV_FULL, GMM_COV_DIAG, GMM_COV_ISO = 0, 1, 2
GMM_F32, GMM_F16, GMM_BF16 = 0, 1, 2
GMM_OK, GMM_ERR_INVALID_ARG, GMM_ERR_UNSUPPORTED, GMM_ERR_NOT_PD = 0, 1, 2, 3
GMM_ERR_NONFINITE, GMM_ERR_WORKSPACE, GMM_ERR_TIMEOUT, GMM_ERR_CUDA = 4, 5, 6, 7
GMM_FLAG_RIDGE, GMM_FLAG_NOT_PD, GMM_FLAG_FLOOR, GMM_FLAG_EMPTY = 1, 2, 4, 8
GMM_OPT_CUDA_CORES = 1

EXPORTS = (
    "gmm_default_opts", "gmm_status_string", "gmm_workspace_bytes", "gmm_prepared_bytes",
    "gmm_prepare", "gmm_em_step", "gmm_workspace_bytes_host", "gmm_em_step_host",
    "gmm_assign_topm", "gmm_last_device_status", "gmm_profile_enable", "gmm_profile_read",
    "gmm_profile_reset", "gmm_em_step_noalloc", "gmm_debug_tc_gemm", "gmm_ivf_lists_ws_bytes",
    "gmm_ivf_lists",
)


class gmm_params(ctypes.Structure):
    _fields_ = [("pi", ctypes.c_void_p), ("mu", ctypes.c_void_p), ("cov", ctypes.c_void_p)]


class gmm_opts(ctypes.Structure):
    _fields_ = [("ridge_rel", ctypes.c_float), ("var_floor", ctypes.c_float),
                ("min_s0", ctypes.c_float), ("flags", ctypes.c_int)]


class GmmError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__("%s: %s" % (what, status_string(status)))


_lib = None


def lib():
    """The loaded libgmm.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libgmm.so not built (%s); run python -m soft_clustering_gb300.build"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        L.gmm_default_opts.restype = gmm_opts
        L.gmm_status_string.argtypes = [i32]
        L.gmm_status_string.restype = ctypes.c_char_p
        L.gmm_workspace_bytes.argtypes = [i64, i32, i32, i32, i32]
        L.gmm_workspace_bytes.restype = sz
        L.gmm_workspace_bytes_host.argtypes = [i64, i32, i32, i32, i32, i64]
        L.gmm_workspace_bytes_host.restype = sz
        L.gmm_prepared_bytes.argtypes = [i32, i32, i32]
        L.gmm_prepared_bytes.restype = sz
        L.gmm_prepare.argtypes = [P(gmm_params), i32, i32, i32, P(gmm_opts), vp, vp, vp]
        L.gmm_em_step.argtypes = [vp, i32, i64, i32, i32, P(gmm_params), i32, P(gmm_opts), vp, sz,
                                  vp, vp, vp, vp]
        L.gmm_em_step_host.argtypes = [vp, i32, i64, i32, i32, P(gmm_params), i32, P(gmm_opts),
                                       vp, sz, i64, vp, vp, vp, vp]
        L.gmm_assign_topm.argtypes = [vp, i32, i64, i32, i32, vp, i32, i32, vp, vp, vp, vp, sz, vp]
        L.gmm_last_device_status.argtypes = [vp, vp]
        L.gmm_em_step_noalloc.argtypes = [vp, i32, i64, i32, i32, P(gmm_params), i32,
                                          P(gmm_opts), vp, vp, vp, vp]
        L.gmm_debug_tc_gemm.argtypes = [vp, vp, vp, i32, i32, vp, vp]
        L.gmm_debug_tc_gemm.restype = i32
        L.gmm_ivf_lists_ws_bytes.argtypes = [i64, i32, i32]
        L.gmm_ivf_lists_ws_bytes.restype = sz
        L.gmm_ivf_lists.argtypes = [vp, vp, i64, i32, i32, ctypes.c_float, vp, vp, vp, vp, sz, vp]
        L.gmm_profile_enable.argtypes = [i32]
        L.gmm_profile_enable.restype = None
        L.gmm_profile_read.argtypes = [P(ctypes.c_char_p), P(ctypes.c_double), P(ctypes.c_long),
                                       i32]
        L.gmm_profile_read.restype = i32
        L.gmm_profile_reset.restype = None
        for f in ("gmm_prepare", "gmm_em_step", "gmm_em_step_host", "gmm_assign_topm",
                  "gmm_last_device_status", "gmm_em_step_noalloc", "gmm_ivf_lists"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def _ptr(x):
    """Device/host address of a torch tensor, numpy array or integer (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, what, raise_on_error=True):
    if raise_on_error and status != GMM_OK:
        raise GmmError(status, what)
    return status


def status_string(status) -> str:
    return lib().gmm_status_string(int(status)).decode()


def gmm_default_opts(**overrides) -> gmm_opts:
    o = lib().gmm_default_opts()
    for k, v in overrides.items():
        setattr(o, k, v)
    return o


def gmm_workspace_bytes(N, D, K, cov, xdtype) -> int:
    return int(lib().gmm_workspace_bytes(N, D, K, cov, xdtype))


def gmm_workspace_bytes_host(N, D, K, cov, xdtype, chunk_rows) -> int:
    return int(lib().gmm_workspace_bytes_host(N, D, K, cov, xdtype, chunk_rows))


def gmm_prepared_bytes(D, K, cov) -> int:
    return int(lib().gmm_prepared_bytes(D, K, cov))


def make_params(pi, mu, cov) -> gmm_params:
    return gmm_params(_ptr(pi), _ptr(mu), _ptr(cov))


def gmm_prepare(pi, mu, cov, D, K, cov_type, prepared, flags=None, opts=None, stream=None,
                raise_on_error=True):
    p = make_params(pi, mu, cov)
    o = opts if opts is not None else gmm_default_opts()
    st = lib().gmm_prepare(ctypes.byref(p), D, K, cov_type, ctypes.byref(o), _ptr(prepared),
                           _ptr(flags), _stream(stream))
    return _check(st, "gmm_prepare", raise_on_error)


def gmm_em_step(X, xdtype, N, D, K, pi, mu, cov, cov_type, ws, ws_bytes, loglik, lse=None,
                flags=None, opts=None, stream=None, raise_on_error=True):
    p = make_params(pi, mu, cov)
    o = opts if opts is not None else gmm_default_opts()
    st = lib().gmm_em_step(_ptr(X), xdtype, N, D, K, ctypes.byref(p), cov_type, ctypes.byref(o),
                           _ptr(ws), ws_bytes, _ptr(loglik), _ptr(lse), _ptr(flags),
                           _stream(stream))
    return _check(st, "gmm_em_step", raise_on_error)


def gmm_em_step_host(X_host, xdtype, N, D, K, pi, mu, cov, cov_type, ws, ws_bytes, chunk_rows,
                     loglik, loglik_host=None, flags=None, opts=None, stream=None,
                     raise_on_error=True):
    p = make_params(pi, mu, cov)
    o = opts if opts is not None else gmm_default_opts()
    st = lib().gmm_em_step_host(_ptr(X_host), xdtype, N, D, K, ctypes.byref(p), cov_type,
                                ctypes.byref(o), _ptr(ws), ws_bytes, chunk_rows, _ptr(loglik),
                                _ptr(loglik_host), _ptr(flags), _stream(stream))
    return _check(st, "gmm_em_step_host", raise_on_error)


def gmm_assign_topm(X, xdtype, N, D, K, prepared, cov_type, m, ids, gamma, lse, ws, ws_bytes,
                    stream=None, raise_on_error=True):
    st = lib().gmm_assign_topm(_ptr(X), xdtype, N, D, K, _ptr(prepared), cov_type, m, _ptr(ids),
                               _ptr(gamma), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "gmm_assign_topm", raise_on_error)


def gmm_em_step_noalloc(X, xdtype, N, D, K, pi, mu, cov, cov_type, loglik, lse, flags=None,
                        opts=None, stream=None, raise_on_error=True):
    """The EM step without a workspace, for callers that cannot allocate
    device memory (scratch is a fixed 64 MiB array inside the library).
    Synchronises the stream; returns the call's status."""
    p = make_params(pi, mu, cov)
    o = opts if opts is not None else gmm_default_opts()
    st = lib().gmm_em_step_noalloc(_ptr(X), xdtype, N, D, K, ctypes.byref(p), cov_type,
                                   ctypes.byref(o), _ptr(loglik), _ptr(lse), _ptr(flags),
                                   _stream(stream))
    return _check(st, "gmm_em_step_noalloc", raise_on_error)


def gmm_ivf_lists_ws_bytes(N, m, K) -> int:
    return int(lib().gmm_ivf_lists_ws_bytes(N, m, K))


def gmm_ivf_lists(ids, gamma, N, m, K, gamma_min, offsets, list_pts, list_gamma, ws, ws_bytes,
                  stream=None, raise_on_error=True):
    st = lib().gmm_ivf_lists(_ptr(ids), _ptr(gamma), N, m, K, float(gamma_min), _ptr(offsets),
                             _ptr(list_pts), _ptr(list_gamma), _ptr(ws), ws_bytes, _stream(stream))
    return _check(st, "gmm_ivf_lists", raise_on_error)


def gmm_last_device_status(ws, stream=None) -> int:
    return int(lib().gmm_last_device_status(_ptr(ws), _stream(stream)))


def gmm_profile_enable(on: bool = True):
    lib().gmm_profile_enable(1 if on else 0)


def gmm_profile_reset():
    lib().gmm_profile_reset()


def gmm_profile_read(max_kernels: int = 32) -> dict:
    """{kernel name: (total ms, launches)} since the last reset (synchronises)."""
    names = (ctypes.c_char_p * max_kernels)()
    ms = (ctypes.c_double * max_kernels)()
    n_l = (ctypes.c_long * max_kernels)()
    n = lib().gmm_profile_read(names, ms, n_l, max_kernels)
    return {names[i].decode(): (ms[i], n_l[i]) for i in range(min(n, max_kernels))}


def gmm_debug_tc_gemm(A, B, C, kdim, n, status, stream=None) -> int:
    """Test-only: C = A B^T through the tensor-core building blocks."""
    return int(lib().gmm_debug_tc_gemm(_ptr(A), _ptr(B), _ptr(C), kdim, n, _ptr(status),
                                       _stream(stream)))
