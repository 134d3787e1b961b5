"""Checkpoint / resume of an EM run (host side, no GPU).

The file keeps the fp32 parameters bit for bit; a run resumed from a
checkpoint therefore continues exactly as the uninterrupted run.  That is
checked with the oracle's EM step (deterministic like the library's), with the
parameters rounded to fp32 between steps as the library holds them.
"""
import os

import numpy as np
import pytest

import datagen
import oracle
from soft_clustering_gb300 import checkpoint


def _params(rng, cov_type, K, D):
    pi = rng.dirichlet(np.ones(K)).astype(np.float32)
    mu = rng.standard_normal((K, D)).astype(np.float32)
    shape = {0: (K, D, D), 1: (K, D), 2: (K,)}[cov_type]
    cov = rng.uniform(0.1, 2.0, shape).astype(np.float32)
    # values whose bits a lossy format would change
    mu.flat[0] = -0.0
    mu.flat[1] = np.float32(1e-40)      # fp32 subnormal
    mu.flat[2] = np.float32(3.4e38)
    return pi, mu, cov


@pytest.mark.parametrize("cov_type", [0, 1, 2])
def test_round_trip_is_bit_exact(tmp_path, cov_type):
    rng = np.random.default_rng(cov_type)
    K, D = 5, 7
    pi, mu, cov = _params(rng, cov_type, K, D)
    ll = rng.standard_normal(4) * 1e6
    p = str(tmp_path / "state.ckpt")
    checkpoint.save(p, pi, mu, cov, cov_type, 17, ll)
    c = checkpoint.load(p)
    assert (c["D"], c["K"], c["cov_type"], c["iteration"]) == (D, K, cov_type, 17)
    for a, b in ((pi, c["pi"]), (mu, c["mu"]), (cov, c["cov"])):
        assert a.shape == b.shape and a.dtype == b.dtype == np.float32
        assert (a.view(np.uint32) == b.view(np.uint32)).all()
    assert (ll.view(np.uint64) == c["ll_history"].view(np.uint64)).all()
    assert not any(f.startswith("state.ckpt.tmp") for f in os.listdir(tmp_path))


def test_damaged_files_are_rejected(tmp_path):
    rng = np.random.default_rng(9)
    pi, mu, cov = _params(rng, 1, 3, 4)
    p = str(tmp_path / "a.ckpt")
    checkpoint.save(p, pi, mu, cov, 1, 2, [1.0, 2.0])
    good = open(p, "rb").read()
    cases = {
        "flipped byte": good[:60] + bytes([good[60] ^ 0x10]) + good[61:],
        "truncated": good[:-9],
        "magic": b"XXXXXXXX" + good[8:],
        "version": good[:8] + (2).to_bytes(4, "little") + good[12:],
        "empty": b"",
    }
    for name, blob in cases.items():
        q = str(tmp_path / (name.replace(" ", "_") + ".ckpt"))
        open(q, "wb").write(blob)
        with pytest.raises(ValueError):
            checkpoint.load(q)
    with pytest.raises(ValueError):
        checkpoint.save(p, pi, mu, cov[:, :3], 1, 0)       # covariance of the wrong size
    with pytest.raises(ValueError):
        checkpoint.save(p, pi, mu, cov, 3, 0)              # no such covariance type


def _f32(p):
    return tuple(np.asarray(a, dtype=np.float32) for a in p)


def _em(bits, theta, wl, opts, iters):
    lls = []
    for _ in range(iters):
        r = oracle.em_step(bits, *(np.asarray(a, np.float64) for a in theta), wl.cov_type,
                           xdtype=wl.dtype, opts=opts)
        assert r["status"] == 0
        lls.append(r["ll"])
        theta = _f32((r["pi"], r["mu"], r["cov"]))
    return theta, lls


@pytest.mark.parametrize("name,n", [("tiny_diag", None), ("full_cov", 3000)])
def test_resume_reproduces_the_uninterrupted_run(tmp_path, name, n):
    wl = datagen.WORKLOADS[name]
    if n:
        wl = wl.with_n(n)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta0 = _f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta0)
    full, ll_full = _em(bits, theta0, wl, opts, 4)
    half, ll_half = _em(bits, theta0, wl, opts, 2)
    p = str(tmp_path / "run.ckpt")
    checkpoint.save(p, *half, wl.cov_type, 2, ll_half)
    c = checkpoint.load(p)
    rest, ll_rest = _em(bits, (c["pi"], c["mu"], c["cov"]), wl, opts, 2)
    assert c["iteration"] == 2
    for a, b in zip(full, rest):
        assert (a.view(np.uint32) == b.reshape(a.shape).view(np.uint32)).all()
    assert list(c["ll_history"]) + ll_rest == ll_full
