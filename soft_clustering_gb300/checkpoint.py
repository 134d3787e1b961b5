"""Checkpoint and resume of an EM run: {pi, mu, Sigma, iteration, log-likelihood history}.

The state is stored bit for bit (the fp32 parameters exactly as the library
holds them, the log-likelihoods as fp64), so a run resumed from iteration t
continues exactly as the uninterrupted run would: the EM step itself is
deterministic (every reduction has a fixed order).

File layout (little endian):
    magic        8 bytes  b"GMMCKPT1"
    version      u32      1
    D, K, cov    u32 x 3  dimensions and covariance type (0 full, 1 diag, 2 iso)
    iteration    u64      EM iterations done
    n_ll         u32      entries of the log-likelihood history
    reserved     u32      0
    pi           f32 [K]
    mu           f32 [K * D]
    cov          f32 [K * D * D | K * D | K]
    ll           f64 [n_ll]
    crc32        u32      of everything before it
Writes go to a temporary file that replaces the target in one step, so a
crash never leaves a half-written checkpoint under the target's name.
"""
from __future__ import annotations

import os
import struct
import zlib

import numpy as np

MAGIC = b"GMMCKPT1"
VERSION = 1
_HEAD = struct.Struct("<8sIIIIQII")


def _cov_count(cov_type, K, D):
    return {0: K * D * D, 1: K * D, 2: K}[int(cov_type)]


def save(path, pi, mu, cov, cov_type, iteration, ll_history=()):
    """Write a checkpoint.  pi, mu, cov are fp32 arrays (or convertible
    without change: float64 input must hold fp32 values)."""
    pi = np.ascontiguousarray(pi, dtype=np.float32)
    K = pi.size
    mu = np.ascontiguousarray(mu, dtype=np.float32).reshape(-1)
    if K < 1 or mu.size % K:
        raise ValueError("mu has %d entries for K=%d" % (mu.size, K))
    D = mu.size // K
    cov = np.ascontiguousarray(cov, dtype=np.float32).reshape(-1)
    if int(cov_type) not in (0, 1, 2) or cov.size != _cov_count(cov_type, K, D):
        raise ValueError("covariance of %d entries does not fit type %s, K=%d, D=%d"
                         % (cov.size, cov_type, K, D))
    ll = np.ascontiguousarray(ll_history, dtype=np.float64).reshape(-1)
    body = (_HEAD.pack(MAGIC, VERSION, D, K, int(cov_type), int(iteration), ll.size, 0)
            + pi.astype("<f4").tobytes() + mu.astype("<f4").tobytes()
            + cov.astype("<f4").tobytes() + ll.astype("<f8").tobytes())
    blob = body + struct.pack("<I", zlib.crc32(body) & 0xFFFFFFFF)
    tmp = "%s.tmp.%d" % (path, os.getpid())
    with open(tmp, "wb") as f:
        f.write(blob)
        f.flush()
        os.fsync(f.fileno())
    os.replace(tmp, path)


def load(path):
    """Read a checkpoint; raises ValueError on a wrong magic, version, size or
    checksum.  Returns dict(pi, mu, cov, cov_type, iteration, ll_history, D, K)
    with fp32 parameters shaped [K], [K, D] and [K, D, D] | [K, D] | [K]."""
    with open(path, "rb") as f:
        blob = f.read()
    if len(blob) < _HEAD.size + 4:
        raise ValueError("checkpoint too short")
    magic, version, D, K, cov_type, iteration, n_ll, _ = _HEAD.unpack_from(blob, 0)
    if magic != MAGIC:
        raise ValueError("not a checkpoint (magic %r)" % magic)
    if version != VERSION:
        raise ValueError("checkpoint version %d, expected %d" % (version, VERSION))
    if cov_type not in (0, 1, 2) or K < 1 or D < 1:
        raise ValueError("bad header: D=%d K=%d cov=%d" % (D, K, cov_type))
    nc = _cov_count(cov_type, K, D)
    want = _HEAD.size + 4 * (K + K * D + nc) + 8 * n_ll + 4
    if len(blob) != want:
        raise ValueError("checkpoint has %d bytes, header implies %d" % (len(blob), want))
    (crc,) = struct.unpack_from("<I", blob, want - 4)
    if zlib.crc32(blob[:want - 4]) & 0xFFFFFFFF != crc:
        raise ValueError("checkpoint checksum mismatch")
    o = _HEAD.size
    pi = np.frombuffer(blob, "<f4", K, o).astype(np.float32); o += 4 * K
    mu = np.frombuffer(blob, "<f4", K * D, o).astype(np.float32).reshape(K, D); o += 4 * K * D
    cov = np.frombuffer(blob, "<f4", nc, o).astype(np.float32); o += 4 * nc
    cov = cov.reshape({0: (K, D, D), 1: (K, D), 2: (K,)}[cov_type])
    ll = np.frombuffer(blob, "<f8", n_ll, o).astype(np.float64)
    return dict(pi=pi, mu=mu, cov=cov, cov_type=cov_type, iteration=int(iteration),
                ll_history=ll, D=D, K=K)
