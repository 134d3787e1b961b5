"""Seeded synthetic Gaussian-mixture inputs shared by the CUDA path's tests,
the benchmark and the fp64 oracle's tests.

This package only makes inputs: planted mixtures, the points drawn from them
(on the host, or straight into device memory with bit-identical results) and
the initial parameters theta_0 both sides start from.  It holds none of the
EM arithmetic (densities, responsibilities, statistics, updates).

The C sources are built on first use (gcc / nvcc) into ``datagen/_build``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_host_lib = None
_cuda_lib = None

F32, F16, BF16 = 0, 1, 2
MIX_DIAG, MIX_FULL, MIX_SPHERE, MIX_IVF = 0, 1, 2, 3
COV_FULL, COV_DIAG, COV_ISO = 0, 1, 2
_NP_STORE = {F32: np.float32, F16: np.uint16, BF16: np.uint16}
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}


class _GenMixture(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int),
        ("D", ctypes.c_int),
        ("K", ctypes.c_int),
        ("seed", ctypes.c_uint64),
        ("noise", ctypes.c_double),
        ("mid_frac", ctypes.c_double),
        ("cdf", ctypes.c_void_p),
        ("mu", ctypes.c_void_p),
        ("sd", ctypes.c_void_p),
        ("chol", ctypes.c_void_p),
    ]


def _newer(src_paths, out):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in src_paths)


def build_host() -> str:
    """Compile the host generator (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libgmmgen_host.so")
    srcs = [os.path.join(_HERE, "gen_host.c"), os.path.join(_HERE, "mixture_gen.h")]
    if _newer(srcs, out):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, srcs[0], "-lm"])
        os.replace(tmp, out)
    return out


def build_cuda() -> str:
    """Compile the device generator for sm_103a (no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, "libgmmgen_cuda.so")
    srcs = [os.path.join(_HERE, "gen_cuda.cu"), os.path.join(_HERE, "mixture_gen.h")]
    if _newer(srcs, out):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
             "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, srcs[0]])
        os.replace(tmp, out)
    return out


def host_lib():
    global _host_lib
    with _lock:
        if _host_lib is None:
            lib = ctypes.CDLL(build_host())
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.gen_planted_diag.argtypes = [u64, i32, i32, dbl, i32, dbl, dbl, dbl, vp, vp, vp, vp]
            lib.gen_planted_full.argtypes = [u64, i32, i32, dbl, dbl, dbl, vp, vp, vp, vp, vp]
            lib.gen_planted_sphere.argtypes = [u64, i32, i32, vp, vp, vp]
            lib.gen_points.argtypes = [ctypes.POINTER(_GenMixture), u64, u64, i32, vp]
            lib.gen_points_at.argtypes = [ctypes.POINTER(_GenMixture), vp, i64, i32, vp]
            lib.gen_init_indices.argtypes = [u64, i64, i32, vp]
            lib.gen_global_moments.argtypes = [vp, i32, i64, i32, vp, vp, vp]
            lib.gen_rows_to_double.argtypes = [vp, i32, i64, i32, vp]
            lib.gen_philox_block.argtypes = [vp, vp, vp]
            lib.gen_normals.argtypes = [u64, ctypes.c_uint32, u64, ctypes.c_uint32, vp]
            lib.gen_ln_host.argtypes = [dbl]
            lib.gen_ln_host.restype = dbl
            lib.gen_to_f16_host.argtypes = [dbl]
            lib.gen_to_f16_host.restype = ctypes.c_uint16
            lib.gen_to_bf16_host.argtypes = [dbl]
            lib.gen_to_bf16_host.restype = ctypes.c_uint16
            _host_lib = lib
    return _host_lib


def cuda_lib():
    global _cuda_lib
    with _lock:
        if _cuda_lib is None:
            lib = ctypes.CDLL(build_cuda())
            lib.gen_device_points.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_double,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_void_p]
            lib.gen_device_points.restype = ctypes.c_int
            _cuda_lib = lib
    return _cuda_lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Workload:
    """One synthetic workload: sizes, storage dtype, planted mixture recipe."""
    name: str
    seed: int
    N: int
    D: int
    K: int
    dtype: int
    cov_type: int
    iters: int
    kind: int
    recipe: dict
    m: int = 0            # top-m for assignment workloads (0 = EM workload)
    note: str = ""

    def with_n(self, n: int) -> "Workload":
        return Workload(self.name, self.seed, int(n), self.D, self.K, self.dtype, self.cov_type,
                        self.iters, self.kind, dict(self.recipe), self.m, self.note)


# The five workloads: sizes, dtypes and planted-mixture recipes.
WORKLOADS = {
    "tiny_diag": Workload(
        "tiny_diag", 1, 4096, 16, 8, F32, COV_DIAG, 10, MIX_DIAG,
        dict(mean_sd=4.0, sd_mode=0, lo=0.5, hi=2.0, alpha=1.0),
        note="means N(0,4^2), per-dim variance U[0.5,2], weights Dirichlet(1)"),
    "full_cov": Workload(
        "full_cov", 2, 1_000_000, 64, 16, F16, COV_FULL, 20, MIX_FULL,
        dict(mean_sd=3.0, ridge=0.1, alpha=2.0),
        note="means N(0,3^2), Sigma = A A^T/D + 0.1 I, weights Dirichlet(2)"),
    "embed_diag": Workload(
        "embed_diag", 3, 10_000_000, 128, 256, F16, COV_DIAG, 10, MIX_SPHERE,
        dict(noise=0.05),
        note="unit centres + N(0,0.05^2) noise, L2-normalised, uniform weights"),
    "large_diag": Workload(
        "large_diag", 4, 200_000_000, 128, 1024, BF16, COV_DIAG, 5, MIX_DIAG,
        dict(mean_sd=1.0, sd_mode=1, lo=0.1, hi=0.5, alpha=0.5),
        note="means N(0,1), per-component sigma U[0.1,0.5], weights Dirichlet(0.5)"),
    "ivf_assign": Workload(
        "ivf_assign", 5, 50_000_000, 128, 4096, F16, COV_DIAG, 0, MIX_IVF,
        dict(mean_sd=1.0, sd_mode=1, lo=0.1, hi=0.5, alpha=1.0, mid_frac=0.1), m=4,
        note="planted diag GMM (fp16 params), 10% midpoints of two centres, top-4"),
}


@dataclass
class Mixture:
    """A planted mixture's tables plus the workload that made it."""
    wl: Workload
    weights: np.ndarray
    cdf: np.ndarray
    mu: np.ndarray
    sd: np.ndarray | None = None
    sigma: np.ndarray | None = None
    chol: np.ndarray | None = None
    _struct: _GenMixture = field(default=None, repr=False)

    def struct(self) -> _GenMixture:
        if self._struct is None:
            r = self.wl.recipe
            s = _GenMixture()
            s.kind, s.D, s.K, s.seed = self.wl.kind, self.wl.D, self.wl.K, self.wl.seed
            s.noise = float(r.get("noise", 0.0))
            s.mid_frac = float(r.get("mid_frac", 0.0))
            s.cdf, s.mu = _ptr(self.cdf).value, _ptr(self.mu).value
            s.sd = None if self.sd is None else _ptr(self.sd).value
            s.chol = None if self.chol is None else _ptr(self.chol).value
            self._struct = s
        return self._struct


def planted(wl: Workload) -> Mixture:
    """Build the planted mixture tables for a workload (host, fp64)."""
    lib = host_lib()
    D, K, r = wl.D, wl.K, wl.recipe
    w = np.zeros(K)
    cdf = np.zeros(K)
    mu = np.zeros((K, D))
    if wl.kind in (MIX_DIAG, MIX_IVF):
        sd = np.zeros((K, D))
        rc = lib.gen_planted_diag(wl.seed, D, K, r["mean_sd"], r["sd_mode"], r["lo"], r["hi"],
                                  r["alpha"], _ptr(w), _ptr(cdf), _ptr(mu), _ptr(sd))
        mix = Mixture(wl, w, cdf, mu, sd=sd)
    elif wl.kind == MIX_FULL:
        sigma = np.zeros((K, D, D))
        chol = np.zeros((K, D, D))
        rc = lib.gen_planted_full(wl.seed, D, K, r["mean_sd"], r["ridge"], r["alpha"], _ptr(w),
                                  _ptr(cdf), _ptr(mu), _ptr(sigma), _ptr(chol))
        mix = Mixture(wl, w, cdf, mu, sigma=sigma, chol=chol)
    elif wl.kind == MIX_SPHERE:
        rc = lib.gen_planted_sphere(wl.seed, D, K, _ptr(w), _ptr(cdf), _ptr(mu))
        mix = Mixture(wl, w, cdf, mu)
    else:
        raise ValueError(wl.kind)
    if rc != 0:
        raise RuntimeError("planted mixture generation failed (%d)" % rc)
    return mix


def points(mix: Mixture, start: int, count: int) -> np.ndarray:
    """Points [start, start+count) on the host, as stored bits (N x D)."""
    wl = mix.wl
    out = np.empty((count, wl.D), dtype=_NP_STORE[wl.dtype])
    if count:
        rc = host_lib().gen_points(ctypes.byref(mix.struct()), start, count, wl.dtype, _ptr(out))
        if rc:
            raise RuntimeError("gen_points failed (%d)" % rc)
    return out


def points_at(mix: Mixture, idx) -> np.ndarray:
    """Points with the given indices, as stored bits."""
    wl = mix.wl
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty((len(idx), wl.D), dtype=_NP_STORE[wl.dtype])
    if len(idx):
        rc = host_lib().gen_points_at(ctypes.byref(mix.struct()), _ptr(idx), len(idx), wl.dtype,
                                      _ptr(out))
        if rc:
            raise RuntimeError("gen_points_at failed (%d)" % rc)
    return out


def to_double(mix_or_dtype, bits: np.ndarray) -> np.ndarray:
    """Stored values widened to float64 (generator's own decoder)."""
    dtype = mix_or_dtype.wl.dtype if isinstance(mix_or_dtype, Mixture) else int(mix_or_dtype)
    bits = np.ascontiguousarray(bits)
    n, D = bits.shape
    out = np.empty((n, D))
    host_lib().gen_rows_to_double(_ptr(bits), dtype, n, D, _ptr(out))
    return out


INIT_PREFIX = 1 << 18


def init_params(mix: Mixture, prefix_rows: np.ndarray | None = None):
    """theta_0 for an EM workload: K distinct random points as means, the
    global (co)variance of the first min(N, 2^18) points, uniform weights.

    Returns (pi[K], mu[K,D], cov) as float32, cov shaped [K,D,D] (full),
    [K,D] (diag) or [K] (iso)."""
    wl = mix.wl
    lib = host_lib()
    idx = np.zeros(wl.K, dtype=np.int64)
    if lib.gen_init_indices(wl.seed, wl.N, wl.K, _ptr(idx)):
        raise RuntimeError("gen_init_indices failed")
    mu = to_double(mix, points_at(mix, idx))
    n_pre = min(wl.N, INIT_PREFIX)
    if prefix_rows is None or len(prefix_rows) < n_pre:
        prefix_rows = points(mix, 0, n_pre)
    prefix_rows = np.ascontiguousarray(prefix_rows[:n_pre])
    mean = np.zeros(wl.D)
    var = np.zeros(wl.D)
    cov = np.zeros((wl.D, wl.D)) if wl.cov_type == COV_FULL else None
    lib.gen_global_moments(_ptr(prefix_rows), wl.dtype, n_pre, wl.D, _ptr(mean), _ptr(var),
                           _ptr(cov))
    pi = np.full(wl.K, 1.0 / wl.K)
    if wl.cov_type == COV_FULL:
        c = np.broadcast_to(cov, (wl.K, wl.D, wl.D))
    elif wl.cov_type == COV_DIAG:
        c = np.broadcast_to(var, (wl.K, wl.D))
    else:
        c = np.full(wl.K, float(var.mean()))
    return (pi.astype(np.float32), mu.astype(np.float32), np.ascontiguousarray(c, dtype=np.float32))


def em_opts(theta0, min_s0=0.5):
    """Caller-side EM options for a workload started from theta0: a variance
    floor of 1e-6 times the mean initial (global) variance, the empty
    threshold, no ridge.  Values are rounded to fp32 (the C ABI's type) so
    every side applies the same numbers."""
    cov = np.asarray(theta0[2], dtype=np.float64)
    v = np.mean(np.diagonal(cov, axis1=1, axis2=2)) if cov.ndim == 3 else np.mean(cov)
    return dict(ridge_rel=0.0, var_floor=float(np.float32(1e-6 * v)),
                min_s0=float(np.float32(min_s0)))


def planted_params_f16(mix: Mixture):
    """A trained model stored in fp16 (the assignment workload): the planted
    weights, centres and variances rounded to fp16, widened to float32."""
    pi = mix.weights.astype(np.float16).astype(np.float32)
    mu = mix.mu.astype(np.float16).astype(np.float32)
    var = (mix.sd * mix.sd).astype(np.float16).astype(np.float32)
    return pi, mu, var


def device_points(mix: Mixture, start: int, count: int, out_ptr: int, stream_ptr: int = 0,
                  dev_tables=None):
    """Draw points straight into device memory at out_ptr.  dev_tables is a
    dict of device pointers {cdf, mu, sd, chol} (see upload_tables)."""
    wl = mix.wl
    t = dev_tables
    rc = cuda_lib().gen_device_points(
        wl.kind, wl.D, wl.K, wl.seed, float(wl.recipe.get("noise", 0.0)),
        float(wl.recipe.get("mid_frac", 0.0)), t["cdf"], t["mu"], t.get("sd"), t.get("chol"),
        start, count, wl.dtype, out_ptr, stream_ptr)
    if rc:
        raise RuntimeError("gen_device_points failed (%d)" % rc)


def upload_tables(mix: Mixture, device="cuda"):
    """Copy the mixture tables to the device (torch tensors); returns
    (keepalive list, dict of pointers)."""
    import torch
    keep = []
    ptrs = {}
    for name in ("cdf", "mu", "sd", "chol"):
        a = getattr(mix, name)
        if a is None:
            ptrs[name] = None
            continue
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(device)
        keep.append(t)
        ptrs[name] = t.data_ptr()
    return keep, ptrs
