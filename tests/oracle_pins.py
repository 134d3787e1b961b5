"""Pins for the fp64 oracle: checks against things other than the oracle.

Every check takes an oracle library handle ``L`` (``oracle.lib()`` or a
deliberately broken build from ``test_oracle_mutants.py``) and raises
AssertionError when the oracle disagrees with:
  * brute force in 40-digit arithmetic (explicit determinant by cofactor
    expansion and inverse by adjugate, direct exp/sum posteriors, explicit
    weighted sums) on tiny inputs,
  * library routines (scipy's multivariate normal log-density, numpy's
    mean / biased covariance),
  * closed forms and invariants (K=1, responsibilities summing to one,
    diag == iso and full == diag special cases, shift and permutation
    invariance, log-likelihood monotone over EM iterations),
  * hand-derived worked examples under tests/golden/ (one cites the value the
    low-precision GMM page prints for exp(-50)),
  * recovery of planted parameters of a well-separated synthetic mixture.
"""
from __future__ import annotations

import json
import math
import os

import mpmath
import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
mpmath.mp.dps = 40


# ------------------------------------------------------------ brute force

def _mp_det(M):
    n = len(M)
    if n == 1:
        return M[0][0]
    tot = mpmath.mpf(0)
    for j in range(n):
        minor = [row[:j] + row[j + 1:] for row in M[1:]]
        tot += (-1) ** j * M[0][j] * _mp_det(minor)
    return tot


def _mp_inv(M):
    """Inverse by adjugate / determinant."""
    n = len(M)
    det = _mp_det(M)
    inv = [[mpmath.mpf(0)] * n for _ in range(n)]
    for i in range(n):
        for j in range(n):
            minor = [row[:j] + row[j + 1:] for k, row in enumerate(M) if k != i]
            cof = (-1) ** (i + j) * (_mp_det(minor) if minor else mpmath.mpf(1))
            inv[j][i] = cof / det
    return inv, det


def _as_full(cov, cov_type, K, D):
    cov = np.asarray(cov, dtype=np.float64)
    if cov_type == oracle.COV_FULL:
        return cov.reshape(K, D, D)
    if cov_type == oracle.COV_DIAG:
        return np.stack([np.diag(cov[k]) for k in range(K)])
    return np.stack([np.eye(D) * cov[k] for k in range(K)])


def brute_force_step(X, pi, mu, cov, cov_type):
    """One EM step by the textbook formulas in 40-digit arithmetic."""
    X = np.asarray(X, dtype=np.float64)
    N, D = X.shape
    K = len(pi)
    S = _as_full(cov, cov_type, K, D)
    mp = mpmath.mpf
    logj = [[None] * K for _ in range(N)]
    for k in range(K):
        Sk = [[mp(float(S[k, a, b])) for b in range(D)] for a in range(D)]
        Si, det = _mp_inv(Sk)
        for n in range(N):
            y = [mp(float(X[n, d])) - mp(float(mu[k][d])) for d in range(D)]
            d2 = sum(y[a] * Si[a][b] * y[b] for a in range(D) for b in range(D))
            logj[n][k] = (mpmath.log(mp(float(pi[k]))) - d2 / 2 - mpmath.log(det) / 2
                          - mp(D) / 2 * mpmath.log(2 * mpmath.pi))
    gam = [[None] * K for _ in range(N)]
    ll = mp(0)
    for n in range(N):
        e = [mpmath.exp(v) for v in logj[n]]
        tot = sum(e)
        ll += mpmath.log(tot)
        for k in range(K):
            gam[n][k] = e[k] / tot
    s0 = [sum(gam[n][k] for n in range(N)) for k in range(K)]
    mun = [[sum(gam[n][k] * mp(float(X[n, d])) for n in range(N)) / s0[k] for d in range(D)]
           for k in range(K)]
    Sn = []
    for k in range(K):
        M = [[sum(gam[n][k] * (mp(float(X[n, a])) - mun[k][a]) * (mp(float(X[n, b])) - mun[k][b])
                  for n in range(N)) / s0[k] for b in range(D)] for a in range(D)]
        Sn.append(M)
    f = lambda v: float(v)
    out = dict(
        logj=np.array([[f(v) for v in r] for r in logj]),
        gamma=np.array([[f(v) for v in r] for r in gam]),
        ll=f(ll), pi=np.array([f(s / N) for s in s0]),
        mu=np.array([[f(v) for v in r] for r in mun]),
        S=np.array([[[f(v) for v in r] for r in M] for M in Sn]))
    return out


def _tiny_case(seed, cov_type, N=6, D=3, K=3):
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((N, D)) * 1.5).astype(np.float32)
    pi = rng.dirichlet(np.ones(K))
    mu = rng.standard_normal((K, D))
    if cov_type == oracle.COV_FULL:
        A = rng.standard_normal((K, D, D))
        cov = np.einsum("kij,klj->kil", A, A) / D + 0.3 * np.eye(D)
    elif cov_type == oracle.COV_DIAG:
        cov = rng.uniform(0.4, 2.0, (K, D))
    else:
        cov = rng.uniform(0.4, 2.0, K)
    return X, pi, mu, cov


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    bad = err > lim
    assert not bad.any(), "%s: max err %g at %s (got %r want %r)" % (
        what, float(err.max()), np.unravel_index(int(np.argmax(err - lim)), err.shape),
        a.flat[int(np.argmax(err - lim))], b.flat[int(np.argmax(err - lim))])


def pin_brute_force(L, cov_type, seed=0):
    X, pi, mu, cov = _tiny_case(seed, cov_type)
    bf = brute_force_step(X, pi, mu, cov, cov_type)
    st, lj, _ = oracle.log_joint(X, pi, mu, cov, cov_type, L=L)
    assert st == 0
    _close(lj, bf["logj"], 1e-12, 1e-12, "log joint")
    r = oracle.em_step(X, pi, mu, cov, cov_type, opts=dict(min_s0=0.0), L=L)
    assert r["status"] == 0
    _close(r["ll"], bf["ll"], 1e-12, 0, "LL")
    _close(r["pi"], bf["pi"], 1e-11, 1e-14, "pi'")
    _close(r["mu"], bf["mu"], 1e-10, 1e-12, "mu'")
    K, D = mu.shape
    if cov_type == oracle.COV_FULL:
        _close(r["cov"], bf["S"], 1e-10, 1e-12, "Sigma'")
    elif cov_type == oracle.COV_DIAG:
        _close(r["cov"], np.stack([np.diag(bf["S"][k]) for k in range(K)]), 1e-10, 1e-12, "var'")
    else:
        _close(r["cov"], np.array([np.trace(bf["S"][k]) / D for k in range(K)]), 1e-10, 1e-12,
               "iso var'")
    # top-m by exhaustive ordering of the brute-force log joints
    st, ids, gam, lse = oracle.topm(X, pi, mu, cov, cov_type, 2, L=L)
    assert st == 0
    order = np.array([sorted(range(K), key=lambda k: (-bf["logj"][n, k], k))[:2]
                      for n in range(len(X))])
    assert (ids == order).all(), (ids, order)
    _close(gam, np.take_along_axis(bf["gamma"], order, 1), 1e-11, 1e-15, "top-m gamma")


# ------------------------------------------------------ library routines

def pin_scipy_logpdf(L, cov_type, seed=1, N=200, D=16, K=4):
    from scipy.stats import multivariate_normal
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, D)).astype(np.float32)
    pi = rng.dirichlet(np.ones(K))
    mu = rng.standard_normal((K, D)) * 0.5
    if cov_type == oracle.COV_FULL:
        A = rng.standard_normal((K, D, D))
        cov = np.einsum("kij,klj->kil", A, A) / D + 0.2 * np.eye(D)
    elif cov_type == oracle.COV_DIAG:
        cov = rng.uniform(0.3, 3.0, (K, D))
    else:
        cov = rng.uniform(0.3, 3.0, K)
    S = _as_full(cov, cov_type, K, D)
    want = np.stack([np.log(pi[k]) + multivariate_normal(mu[k], S[k]).logpdf(X.astype(np.float64))
                     for k in range(K)], axis=1)
    st, lj, _ = oracle.log_joint(X, pi, mu, cov, cov_type, L=L)
    assert st == 0
    _close(lj, want, 1e-11, 1e-10, "log joint vs scipy")


def pin_k1_closed_form(L, cov_type, seed=2, N=500, D=5):
    """K = 1: every responsibility is 1, so the update is the sample mean and
    the biased sample covariance, and LL is the sum of log-densities."""
    from scipy.stats import multivariate_normal
    rng = np.random.default_rng(seed)
    X = (rng.standard_normal((N, D)) @ rng.standard_normal((D, D)) + 3.0).astype(np.float32)
    Xd = X.astype(np.float64)
    pi = np.array([1.0])
    mu = rng.standard_normal((1, D))
    if cov_type == oracle.COV_FULL:
        cov = np.cov(Xd.T)[None] + 0.5 * np.eye(D)
    elif cov_type == oracle.COV_DIAG:
        cov = rng.uniform(0.5, 2, (1, D))
    else:
        cov = np.array([1.3])
    r = oracle.em_step(X, pi, mu, cov, cov_type, L=L)
    S = _as_full(cov, cov_type, 1, D)[0]
    _close(r["ll"], multivariate_normal(mu[0], S).logpdf(Xd).sum(), 1e-12, 0, "K=1 LL")
    _close(r["pi"], [1.0], 1e-14, 0, "K=1 pi")
    _close(r["mu"][0], Xd.mean(0), 1e-13, 1e-13, "K=1 mean")
    C = np.cov(Xd.T, bias=True)
    if cov_type == oracle.COV_FULL:
        _close(r["cov"][0], C, 1e-12, 1e-13, "K=1 covariance")
    elif cov_type == oracle.COV_DIAG:
        _close(r["cov"][0], np.diag(C), 1e-12, 1e-13, "K=1 variances")
    else:
        _close(r["cov"][0], np.trace(C) / D, 1e-12, 1e-13, "K=1 iso variance")


# ------------------------------------------------ invariants, special cases

def pin_gamma_sums_to_one(L, seed=3):
    X, pi, mu, cov = _tiny_case(seed, oracle.COV_FULL, N=40, D=4, K=5)
    st, lj, _ = oracle.log_joint(X, pi, mu, cov, oracle.COV_FULL, L=L)
    r = oracle.em_step(X, pi, mu, cov, oracle.COV_FULL, want_lse=True, L=L)
    g = np.exp(lj - r["lse"][:, None])
    _close(g.sum(1), np.ones(len(X)), 1e-13, 0, "sum_k gamma")
    _close(r["s0"].sum(), len(X), 1e-13, 0, "sum_k s0")
    _close(r["pi"].sum(), 1.0, 1e-13, 0, "sum_k pi'")
    _close(r["ll"], r["lse"].sum(), 1e-13, 0, "LL = sum LSE_n")


def pin_diag_equal_var_is_iso(L, seed=4):
    X, pi, mu, _ = _tiny_case(seed, oracle.COV_ISO, N=60, D=5, K=4)
    v = np.array([0.7, 1.1, 2.0, 0.45])
    a = oracle.em_step(X, pi, mu, np.repeat(v[:, None], 5, 1), oracle.COV_DIAG, L=L)
    b = oracle.em_step(X, pi, mu, v, oracle.COV_ISO, L=L)
    _close(b["ll"], a["ll"], 1e-13, 0, "LL diag vs iso")
    _close(b["mu"], a["mu"], 1e-12, 1e-14, "mu diag vs iso")
    _close(b["cov"], a["cov"].mean(1), 1e-12, 1e-14, "iso var = mean diag var")


def pin_full_diag_sigma_is_diag(L, seed=5):
    X, pi, mu, v = _tiny_case(seed, oracle.COV_DIAG, N=60, D=4, K=3)
    S = np.stack([np.diag(v[k]) for k in range(3)])
    a = oracle.em_step(X, pi, mu, S, oracle.COV_FULL, L=L)
    b = oracle.em_step(X, pi, mu, v, oracle.COV_DIAG, L=L)
    st, la, _ = oracle.log_joint(X, pi, mu, S, oracle.COV_FULL, L=L)
    st, lb, _ = oracle.log_joint(X, pi, mu, v, oracle.COV_DIAG, L=L)
    _close(la, lb, 1e-13, 1e-13, "log joint full(diag S) vs diag")
    _close(a["ll"], b["ll"], 1e-13, 0, "LL")
    _close(np.stack([np.diag(a["cov"][k]) for k in range(3)]), b["cov"], 1e-12, 1e-14,
           "diag of full update")


def pin_shift_invariance(L, seed=6):
    rng = np.random.default_rng(seed)
    N, D, K = 80, 3, 3
    X = (np.round(rng.standard_normal((N, D)) * 256) / 256).astype(np.float32)
    c = np.array([5.0, -3.0, 17.0])
    Xs = (X.astype(np.float64) + c).astype(np.float32)
    assert (Xs.astype(np.float64) - c == X.astype(np.float64)).all()
    pi = rng.dirichlet(np.ones(K))
    mu = rng.standard_normal((K, D))
    A = rng.standard_normal((K, D, D))
    S = np.einsum("kij,klj->kil", A, A) / D + 0.3 * np.eye(D)
    a = oracle.em_step(X, pi, mu, S, oracle.COV_FULL, want_lse=True, L=L)
    b = oracle.em_step(Xs, pi, mu + c, S, oracle.COV_FULL, want_lse=True, L=L)
    _close(b["lse"], a["lse"], 1e-12, 1e-12, "LSE under shift")
    _close(b["mu"], a["mu"] + c, 1e-12, 1e-12, "mu' shifts")
    _close(b["cov"], a["cov"], 1e-9, 1e-12, "Sigma' unchanged")


def pin_permutations(L, seed=7):
    X, pi, mu, cov = _tiny_case(seed, oracle.COV_DIAG, N=50, D=4, K=4)
    a = oracle.em_step(X, pi, mu, cov, oracle.COV_DIAG, L=L)
    p = np.random.default_rng(seed).permutation(len(X))
    b = oracle.em_step(X[p], pi, mu, cov, oracle.COV_DIAG, L=L)
    _close(b["mu"], a["mu"], 1e-12, 1e-14, "point permutation: mu'")
    _close(b["cov"], a["cov"], 1e-12, 1e-14, "point permutation: var'")
    q = np.array([2, 0, 3, 1])
    c = oracle.em_step(X, pi[q], mu[q], cov[q], oracle.COV_DIAG, L=L)
    _close(c["pi"], a["pi"][q], 1e-13, 1e-15, "component permutation: pi'")
    _close(c["mu"], a["mu"][q], 1e-12, 1e-14, "component permutation: mu'")
    _close(c["ll"], a["ll"], 1e-13, 0, "component permutation: LL")


def pin_ll_monotone(L, X, pi, mu, cov, cov_type, iters, xdtype=None):
    runs = oracle.fit(X, pi, mu, cov, cov_type, iters, xdtype=xdtype, opts=None)
    lls = [r["ll"] for r in runs]
    for t in range(1, len(lls)):
        assert lls[t] >= lls[t - 1] - 1e-12 * abs(lls[t - 1]), ("LL decreased", t, lls)
    return lls


def pin_underflow(L):
    """Points 50 and 1000 standard deviations from every centre still give
    finite log-likelihoods and responsibilities summing to one."""
    X = np.array([[50.0, 0.0], [0.0, -1000.0], [2000.0, 2000.0]], dtype=np.float32)
    pi = np.array([0.3, 0.7])
    mu = np.array([[0.0, 0.0], [1.0, 1.0]])
    cov = np.array([1.0, 1.0])
    r = oracle.em_step(X, pi, mu, cov, oracle.COV_ISO, want_lse=True, L=L)
    assert r["status"] == 0 and np.isfinite(r["ll"]), r
    st, lj, _ = oracle.log_joint(X, pi, mu, cov, oracle.COV_ISO, L=L)
    g = np.exp(lj - r["lse"][:, None])
    _close(g.sum(1), np.ones(3), 1e-13, 0, "gamma sums far away")


def pin_golden(L):
    with open(os.path.join(GOLDEN, "k1_d1_three_points.json")) as f:
        g = json.load(f)
    X = np.array(g["X"], dtype=np.float32)
    r = oracle.em_step(X, g["pi"], g["mu"], g["var"], oracle.COV_DIAG, L=L)
    e = g["expected"]
    _close(r["ll"], e["ll"], g["tol"], 0, "golden K=1 LL")
    _close(r["mu"], e["mu"], g["tol"], g["tol"], "golden K=1 mu")
    _close(r["cov"], e["var"], g["tol"], g["tol"], "golden K=1 var")
    _close(r["pi"], e["pi"], g["tol"], 0, "golden K=1 pi")

    with open(os.path.join(GOLDEN, "two_symmetric_components.json")) as f:
        g = json.load(f)
    X = np.array(g["X"], dtype=np.float32)
    r = oracle.em_step(X, g["pi"], g["mu"], g["var"], oracle.COV_DIAG, want_lse=True, L=L)
    _close(r["ll"], g["expected"]["ll"], g["tol"], 0, "golden symmetric LL")
    st, ids, gam, lse = oracle.topm(X, g["pi"], g["mu"], g["var"], oracle.COV_DIAG, 2, L=L)
    _close(gam[0], g["expected"]["gamma"], g["tol"], 0, "golden symmetric gamma")
    assert ids[0, 0] == g["expected"]["top1"], ids

    with open(os.path.join(GOLDEN, "underflow_e50.json")) as f:
        g = json.load(f)
    X = np.array(g["X"], dtype=np.float32)
    st, ids, gam, lse = oracle.topm(X, g["pi"], g["mu"], g["var"], oracle.COV_DIAG, 2, L=L)
    e = g["expected"]
    _close(gam[0, 1], e["gamma1_printed"], e["gamma1_rel_tol_vs_printed"], 0, "printed e^-50")
    _close(gam[0, 1], e["gamma1"], g["tol"], 0, "gamma at a 50-nat gap")

    with open(os.path.join(GOLDEN, "ridge_rule.json")) as f:
        g = json.load(f)
    X = np.array(g["X"], dtype=np.float32)
    st, lj, flags = oracle.log_joint(X, g["pi"], g["mu"], g["cov"], oracle.COV_FULL, L=L)
    assert st == 0 and (flags[0] & oracle.FLAG_RIDGE), (st, flags)
    _close(lj[0, 0], g["expected"]["log_joint"], g["tol"], 0, "ridge rule")


def pin_planted_recovery(L, X, xdtype, true_pi, true_mu, true_var, init, iters, tol_mu):
    """From theta_0, EM recovers a well-separated planted mixture up to a
    relabelling (Hungarian matching of the means)."""
    from scipy.optimize import linear_sum_assignment
    pi, mu, cov = init
    for r in oracle.fit(X, pi, mu, cov, oracle.COV_DIAG, iters, xdtype=xdtype):
        pass
    cost = ((r["mu"][:, None, :] - true_mu[None]) ** 2).sum(-1)
    ri, ci = linear_sum_assignment(cost)
    err_mu = np.abs(r["mu"][ri] - true_mu[ci]).max()
    assert err_mu < tol_mu, err_mu
    return r, ri, ci


def pin_stored_dtypes(L, seed=8):
    """fp16 and bf16 inputs decode to the same values numpy (fp16) or a bit
    shift of float32 (bf16) gives: log joints agree with the float32 run."""
    rng = np.random.default_rng(seed)
    N, D, K = 300, 8, 3
    vals = np.concatenate([rng.standard_normal((N - 4, D)) * 3,
                           np.full((4, D), 3e-6),           # fp16 subnormal range
                           ]).astype(np.float32)
    vals[-1] = -vals[-1]
    h = vals.astype(np.float16)
    pi = rng.dirichlet(np.ones(K))
    mu = rng.standard_normal((K, D))
    cov = rng.uniform(0.5, 2.0, (K, D))
    st, la, _ = oracle.log_joint(h.view(np.uint16), pi, mu, cov, oracle.COV_DIAG,
                                 xdtype=oracle.F16, L=L)
    st, lb, _ = oracle.log_joint(h.astype(np.float32), pi, mu, cov, oracle.COV_DIAG, L=L)
    _close(la, lb, 0, 0, "fp16 decode")
    bf = (vals.view(np.uint32) >> 16).astype(np.uint16)
    back = (bf.astype(np.uint32) << 16).view(np.float32)
    st, la, _ = oracle.log_joint(bf, pi, mu, cov, oracle.COV_DIAG, xdtype=oracle.BF16, L=L)
    st, lb, _ = oracle.log_joint(back, pi, mu, cov, oracle.COV_DIAG, L=L)
    _close(la, lb, 0, 0, "bf16 decode")


ALL_QUICK_PINS = [
    ("stored_dtypes", pin_stored_dtypes),
    ("brute_full", lambda L: pin_brute_force(L, oracle.COV_FULL, 0)),
    ("brute_diag", lambda L: pin_brute_force(L, oracle.COV_DIAG, 10)),
    ("brute_iso", lambda L: pin_brute_force(L, oracle.COV_ISO, 20)),
    ("scipy_full", lambda L: pin_scipy_logpdf(L, oracle.COV_FULL)),
    ("scipy_diag", lambda L: pin_scipy_logpdf(L, oracle.COV_DIAG)),
    ("scipy_iso", lambda L: pin_scipy_logpdf(L, oracle.COV_ISO)),
    ("k1_full", lambda L: pin_k1_closed_form(L, oracle.COV_FULL)),
    ("k1_diag", lambda L: pin_k1_closed_form(L, oracle.COV_DIAG)),
    ("k1_iso", lambda L: pin_k1_closed_form(L, oracle.COV_ISO)),
    ("gamma_sum", pin_gamma_sums_to_one),
    ("diag_iso", pin_diag_equal_var_is_iso),
    ("full_diag", pin_full_diag_sigma_is_diag),
    ("shift", pin_shift_invariance),
    ("permute", pin_permutations),
    ("underflow", pin_underflow),
    ("golden", pin_golden),
]
