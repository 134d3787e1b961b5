"""fp64 CPU oracle for the fused GMM EM step and top-m assignment.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package; the library
path (``soft_clustering_gb300``) never does, and shares no code with it.

The arithmetic lives in ``gmm_oracle.c`` (plain C, double precision, OpenMP
over points); see its header for the passages each step follows and the
readings taken where the pages are silent.  This module only builds it and
marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
COV_FULL, COV_DIAG, COV_ISO = 0, 1, 2
OK, INVALID, NOT_PD, NONFINITE, NOMEM = 0, 1, 3, 4, 8
FLAG_RIDGE, FLAG_NOT_PD, FLAG_FLOOR, FLAG_EMPTY = 1, 2, 4, 8

# Defaults of the readings: no ridge unless needed, no floor, a component is
# empty below half of one point's worth of responsibility.
DEFAULT_OPTS = dict(ridge_rel=0.0, var_floor=0.0, min_s0=0.5)


def build(src: str | None = None, out: str | None = None, extra=()) -> str:
    """Compile the oracle (gcc -O2 -fopenmp).  src/out may point at a copy
    of the source (the mutation tests build deliberately broken copies)."""
    src = src or os.path.join(_HERE, "gmm_oracle.c")
    out = out or os.path.join(_BUILD, "liboracle.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not os.path.exists(out) or os.path.getmtime(src) > os.path.getmtime(out):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               *extra, "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(lib):
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_log_joint.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, i32, dbl, vp, vp]
    lib.oracle_em_step.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                   vp, vp, vp, vp, vp]
    lib.oracle_topm.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp, i32, dbl, i32, vp, vp, vp]
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_max_threads.restype = i32
    return lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def load(path: str):
    """Load another build of the oracle (used by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _xbits(X):
    X = np.ascontiguousarray(X)
    if X.dtype == np.float32:
        return X, F32
    if X.dtype == np.float16:
        return X.view(np.uint16), F16
    raise TypeError("pass float32, float16, or (uint16, dtype) via xdtype")


def _prep_x(X, xdtype):
    if xdtype is None:
        return _xbits(X)
    return np.ascontiguousarray(X), int(xdtype)


def set_threads(n: int):
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def log_joint(X, pi, mu, cov, cov_type, xdtype=None, ridge_rel=0.0, L=None):
    """l[n, k] = log pi_k + log N(x_n | mu_k, Sigma_k) in fp64."""
    L = L or lib()
    Xb, dt = _prep_x(X, xdtype)
    N, D = Xb.shape
    K = len(pi)
    out = np.empty((N, K))
    flags = np.zeros(K, dtype=np.int32)
    st = L.oracle_log_joint(_p(Xb), dt, N, D, K, _p(_f64(pi)), _p(_f64(mu)), _p(_f64(cov)),
                            cov_type, float(ridge_rel), _p(out), _p(flags))
    return st, out, flags


def em_step(X, pi, mu, cov, cov_type, xdtype=None, opts=None, want_lse=False, L=None):
    """One EM iteration in fp64.  Returns a dict with status, pi, mu, cov,
    ll (at the input parameters), flags, s0, s1, s2c and optionally lse."""
    L = L or lib()
    o = dict(DEFAULT_OPTS)
    o.update(opts or {})
    Xb, dt = _prep_x(X, xdtype)
    N, D = Xb.shape
    K = len(pi)
    cov = _f64(cov)
    pi_o = np.empty(K)
    mu_o = np.empty((K, D))
    cov_o = np.empty_like(cov)
    ll = np.zeros(1)
    lse = np.empty(N) if want_lse else None
    s0 = np.empty(K)
    s1 = np.empty((K, D))
    s2c = np.empty((K, D, D) if cov_type == COV_FULL else (K, D))
    flags = np.zeros(K, dtype=np.int32)
    ov = np.array([o["ridge_rel"], o["var_floor"], o["min_s0"]], dtype=np.float64)
    st = L.oracle_em_step(_p(Xb), dt, N, D, K, _p(_f64(pi)), _p(_f64(mu)), _p(cov), cov_type,
                          _p(ov), _p(pi_o), _p(mu_o), _p(cov_o), _p(ll), _p(lse), _p(s0), _p(s1),
                          _p(s2c), _p(flags))
    return dict(status=st, pi=pi_o, mu=mu_o, cov=cov_o, ll=float(ll[0]), lse=lse, flags=flags,
                s0=s0, s1=s1, s2c=s2c)


def topm(X, pi, mu, cov, cov_type, m, xdtype=None, ridge_rel=0.0, L=None):
    """Top-m component ids (descending log joint, ties to lower k), their
    full-K posteriors and LSE_n."""
    L = L or lib()
    Xb, dt = _prep_x(X, xdtype)
    N, D = Xb.shape
    K = len(pi)
    ids = np.empty((N, m), dtype=np.int32)
    gam = np.empty((N, m))
    lse = np.empty(N)
    st = L.oracle_topm(_p(Xb), dt, N, D, K, _p(_f64(pi)), _p(_f64(mu)), _p(_f64(cov)), cov_type,
                       float(ridge_rel), int(m), _p(ids), _p(gam), _p(lse))
    return st, ids, gam, lse


def fit(X, pi, mu, cov, cov_type, iters, xdtype=None, opts=None):
    """Iterate em_step; returns the list of per-iteration results."""
    out = []
    for _ in range(iters):
        r = em_step(X, pi, mu, cov, cov_type, xdtype=xdtype, opts=opts)
        out.append(r)
        pi, mu, cov = r["pi"], r["mu"], r["cov"]
    return out


def ivf_lists(ids, gamma, K, gamma_min):
    """Inverted lists of an IVF index with soft multi-assignment, straight
    from the definition: walking the points in order, entry t of point n
    joins the list of component ids[n, t] when t == 0 or gamma[n, t] >=
    gamma_min (compared in float32, the type of both), ids outside [0, K)
    skipped (Flash-GMM summary, "Core insight": boundary vectors go to
    several high-responsibility clusters).  Returns (offsets [K+1] int64,
    point indices int32, gamma float32), each list in point order."""
    ids = np.asarray(ids)
    g = np.asarray(gamma, dtype=np.float32)
    N, m = ids.shape
    lists = [[] for _ in range(K)]
    gmin = np.float32(gamma_min)
    for n in range(N):
        for t in range(m):
            k = int(ids[n, t])
            if 0 <= k < K and (t == 0 or g[n, t] >= gmin):
                lists[k].append((n, g[n, t]))
    offsets = np.zeros(K + 1, dtype=np.int64)
    for k in range(K):
        offsets[k + 1] = offsets[k] + len(lists[k])
    pts = np.array([n for L in lists for (n, _) in L], dtype=np.int32)
    gam = np.array([v for L in lists for (_, v) in L], dtype=np.float32)
    return offsets, pts, gam
