"""fp16-operator precision study (a CPU report; test infrastructure like the
rest of this package).

It measures, with seeded synthetic inputs, two effects the "low-precision
GMM operator" notes report for an fp16 GMM operator:

  * sec. 1.2: the squared Mahalanobis distance through an explicitly
    inverted covariance stored in fp16 errs by about 1e-2 (relative), through
    the Cholesky factor stored in fp16 by about 1e-3, both routes about 1e-6
    in fp32 (D = 64, K = 16).  Reproduced here on ill-conditioned
    covariances (condition numbers near 1e4).
  * sec. 4.1: a ridge eps = c tr(Sigma)/D added before an fp16 Cholesky
    factorisation (c = 1e-3 as the rule, 5e-4 as tried) repaired the
    components whose fp16 factorisation failed and lowered the operator's
    log-likelihood error from 0.009 to 0.003 (K = 8, D = 32).  Here: on
    near-singular covariances the ridge does make every fp16 factorisation
    succeed (a component that fails is lost to its points, which dominates
    the error); on well-conditioned ones it only adds its own bias.

The page's platform and data are not given, so the numbers are this setup's,
not the page's.  The reference values are fp64 (the oracle for the
log-likelihoods).

Emulated arithmetic (numpy, round to nearest even): a value "stored in fp16"
is rounded to fp16; "fp16 arithmetic" rounds the result of every operation
to fp16; everything else is fp32 (the page's mixed-precision rule: fp16
storage, fp32 exp / log / accumulation) or fp64 (reference).

    python -m oracle.precision_study [--seed S]
"""
from __future__ import annotations

import argparse
import json

import numpy as np

from . import COV_FULL, em_step


def planted_covariances(rng, K, D, rank=None, diag=0.1):
    """Sigma_k = A A^T / D + diag I with A_ij ~ N(0, 1) (D x rank; rank D by
    default), the recipe of the full-covariance workload."""
    r = rank or D
    A = rng.standard_normal((K, D, r))
    return np.einsum("kir,kjr->kij", A, A) / D + diag * np.eye(D)[None]


def _f16(a):
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def chol_fp16_arith(S):
    """Cholesky factor with every operation rounded to fp16 (the operands
    stored in fp16); None when a pivot is not positive."""
    D = S.shape[0]
    A = _f16(S)
    L = np.zeros((D, D), dtype=np.float16)
    for j in range(D):
        s = A[j, j]
        for k in range(j):
            s = np.float16(s - np.float16(L[j, k] * L[j, k]))
        if not s > 0:
            return None
        L[j, j] = np.float16(np.sqrt(np.float32(s)))
        for i in range(j + 1, D):
            t = A[i, j]
            for k in range(j):
                t = np.float16(t - np.float16(L[i, k] * L[j, k]))
            L[i, j] = np.float16(t / L[j, j])
    return L


def forward_solve(L, y, dtype):
    """z = L^-1 y by forward substitution, accumulating in `dtype`."""
    D = L.shape[0]
    Lc = L.astype(dtype)
    yc = y.astype(dtype)
    z = np.zeros(y.shape, dtype=dtype)
    for i in range(D):
        acc = yc[..., i]
        for j in range(i):
            acc = (acc - Lc[i, j] * z[..., j]).astype(dtype)
        z[..., i] = (acc / Lc[i, i]).astype(dtype)
    return z


def mahalanobis_routes(seed=0, D=64, K=16, n=256, rank=48, diag=1e-3):
    """Relative error of d^2 = (x - mu)^T Sigma^-1 (x - mu) per route and
    precision, against fp64, over n points per component drawn from that
    component.  The covariances (a rank-48 part plus 1e-3 I at D = 64,
    condition numbers near 1e4) are ill-conditioned enough to show the
    routes apart.  Returns {route: median relative error}."""
    rng = np.random.default_rng(seed)
    S = planted_covariances(rng, K, D, rank=rank, diag=diag)
    mu = rng.standard_normal((K, D)) * 3.0
    out = {"inverse_fp32": [], "cholesky_fp32": [], "inverse_fp16": [], "cholesky_fp16": []}
    for k in range(K):
        Lk = np.linalg.cholesky(S[k])
        x = mu[k] + rng.standard_normal((n, D)) @ Lk.T
        # x and mu are stored in fp16 (the operator's storage); the reference
        # is exact fp64 arithmetic on those stored values
        xs = _f16(x).astype(np.float64)
        ms = _f16(mu[k]).astype(np.float64)
        y = xs - ms
        ref = np.einsum("ni,ij,nj->n", y, np.linalg.inv(S[k]), y)
        P = np.linalg.inv(S[k])
        for prec, name in ((np.float32, "fp32"), (np.float16, "fp16")):
            # inverse route: the precision matrix stored in prec, the
            # quadratic form accumulated in fp32
            Pq = P.astype(prec).astype(np.float32)
            yq = y.astype(np.float32)
            d_inv = np.einsum("ni,ij,nj->n", yq, Pq, yq, dtype=np.float32).astype(np.float64)
            # Cholesky route: L stored in prec, the forward solve and z.z in fp32
            Lq = Lk.astype(prec)
            z = forward_solve(Lq, yq, np.float32)
            d_ch = (z.astype(np.float32) ** 2).sum(axis=1, dtype=np.float32).astype(np.float64)
            out["inverse_" + name] += list(np.abs(d_inv - ref) / ref)
            out["cholesky_" + name] += list(np.abs(d_ch - ref) / ref)
    return {k: float(np.median(v)) for k, v in out.items()}


def fp16_operator_ll(X, pi, mu, S, ridge_c):
    """Log-likelihood of the fp16 operator: Sigma (+ ridge_c tr/D I) factored
    with fp16 arithmetic; a component whose factorisation fails is dropped
    (its weight 0), as the operator's preprocessing flags it; z = L^-1 (x -
    mu) in fp32 with L stored in fp16; log-densities, exp, log and sums in
    fp32.  Returns (LL, number of components that failed)."""
    N, D = X.shape
    K = len(pi)
    Xs = _f16(X).astype(np.float32)
    logj = np.full((N, K), -np.inf, dtype=np.float32)
    failed = 0
    for k in range(K):
        Sk = S[k] + ridge_c * np.trace(S[k]) / D * np.eye(D)
        L = chol_fp16_arith(Sk)
        if L is None:
            failed += 1
            continue
        y = Xs - _f16(mu[k]).astype(np.float32)
        z = forward_solve(L, y, np.float32)
        d2 = (z * z).sum(axis=1, dtype=np.float32)
        logdet = np.float32(2.0) * np.log(L.astype(np.float32).diagonal()).sum(dtype=np.float32)
        logj[:, k] = (np.float32(np.log(pi[k])) - np.float32(0.5) * logdet
                      - np.float32(0.5 * D * np.log(2 * np.pi)) - np.float32(0.5) * d2)
    m = logj.max(axis=1)
    lse = m + np.log(np.exp(logj - m[:, None]).sum(axis=1, dtype=np.float32))
    return float(lse.astype(np.float64).sum()), failed


def ridge_effect(seed=0, D=32, K=8, n_per=400, rank=20, diag=1e-3):
    """LL relative error of the fp16 operator against the fp64 oracle on the
    unridged model, without a ridge and with eps = c tr/D (c = 5e-4, 1e-3),
    and the number of components whose fp16 factorisation failed.  The
    default covariances are near-singular (a rank-20 part plus 1e-3 I at
    D = 32); rank = 24, diag = 1e-2 gives well-conditioned ones.
    Returns {label: (rel err, failed)}."""
    rng = np.random.default_rng(seed)
    S = planted_covariances(rng, K, D, rank=rank, diag=diag)
    mu = rng.standard_normal((K, D)) * 2.0
    pi = np.full(K, 1.0 / K)
    X = np.concatenate([mu[k] + rng.standard_normal((n_per, D)) @ np.linalg.cholesky(S[k]).T
                        for k in range(K)])
    Xs = _f16(X)
    ref = em_step(Xs, pi, mu, S, COV_FULL)["ll"]
    out = {}
    for c in (0.0, 5e-4, 1e-3):
        ll, failed = fp16_operator_ll(X, pi, mu, S, c)
        out["ridge %g" % c] = (abs(ll - ref) / abs(ref), failed)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    fmt = lambda r: {k: dict(ll_rel_err=v[0], failed_components=v[1]) for k, v in r.items()}
    rep = dict(mahalanobis_D64_K16=mahalanobis_routes(args.seed),
               ridge_D32_K8_near_singular=fmt(ridge_effect(args.seed)),
               ridge_D32_K8_well_conditioned=fmt(ridge_effect(args.seed, rank=24, diag=1e-2)))
    print(json.dumps(rep, indent=1))


if __name__ == "__main__":
    main()
