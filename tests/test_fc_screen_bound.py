"""The error bound of the full-covariance tensor-core screen, checked on the CPU.

The screen forms, per point x and component k, z~ = s_k Z~ - b_k with
Z~ = X W~_k^T summed in fp32 (W~_k = fp16(W32_k / s_k), s_k the power of two
with max |W_k| / s_k in [2^14, 2^15), W32 the fp32 inverse Cholesky factor the
exact kernels use, b_k = W_k mu_k rounded to fp32), and claims
    |z~ - z| <= E = 1.01 ((2^-11 + 2^-16) |W_k|_F + 2^-25 s_k D) |x|
                     + 1.01 2^-18 |W_k|_F |mu_k| + 2^-15 |z~|
for the exact z = W32_k (x - mu_k).  It keeps every component whose upper
bound c - max(0, |z~| - E)^2 / 2 reaches the largest lower bound
c - (|z~| + E)^2 / 2 less 41 nats.  This test restates that arithmetic with
numpy's fp16 rounding and fp32 sums in random orders, on the full-covariance
workload's recipe and on draws chosen to stress it: tight, ill-conditioned
covariances far from the origin, and a component whose large entries push the
others toward fp16 subnormals.
"""
import numpy as np
import pytest


def _scale(W):
    """s = 2^e with max |W| / s in [2^14, 2^15)."""
    m = np.abs(W).max()
    e = int(np.frexp(m)[1]) if m > 0 else 1
    return 2.0 ** (e - 15)


def _fp32_dot_random_order(a, b, rng):
    """sum a_j b_j in fp32, the products exact (fp16 x fp16), in a random order."""
    terms = (a.astype(np.float64) * b.astype(np.float64)).astype(np.float32)
    acc = np.float32(0.0)
    for t in terms[rng.permutation(terms.size)]:
        acc = np.float32(acc + t)
    return acc


def _case(name, rng):
    D, K = 64, 8
    if name == "workload":
        mu = rng.normal(0.0, 3.0, (K, D))
        A = rng.standard_normal((K, D, D))
        S = np.einsum("kij,klj->kil", A, A) / D + 0.1 * np.eye(D)
    elif name == "tight_far_illcond":
        mu = rng.normal(0.0, 20.0, (K, D))
        A = rng.standard_normal((K, D, 40))
        S = (np.einsum("kij,klj->kil", A, A) / D + 1e-3 * np.eye(D)) * 1e-2
    else:  # subnormal: one huge entry per component's factor
        mu = rng.normal(0.0, 1.0, (K, D))
        A = rng.standard_normal((K, D, D))
        S = np.einsum("kij,klj->kil", A, A) / D + 0.5 * np.eye(D)
        S[:, 0, 0] = 1e-18  # W[0, 0] = 1e9 sets the scale: entries near 1 fall fp16-subnormal
        S[:, 0, 1:] = 0.0
        S[:, 1:, 0] = 0.0
    return D, K, mu, S


@pytest.mark.parametrize("case", ["workload", "tight_far_illcond", "subnormal"])
def test_fc_screen_error_within_bound(case):
    rng = np.random.default_rng({"workload": 11, "tight_far_illcond": 12, "subnormal": 13}[case])
    D, K, mu, S = _case(case, rng)
    L = np.linalg.cholesky(S)
    W32 = np.linalg.inv(L).astype(np.float32)
    W = np.tril(W32.astype(np.float64))
    n = 12
    worst = 0.0
    for k in range(K):
        s = _scale(W[k])
        Wt = (W[k] / s).astype(np.float16)                      # W~_k
        b = np.float32(0.0) + (W[k] @ mu[k]).astype(np.float32)  # fp32 bias (rounded once)
        F = np.sqrt((W[k] ** 2).sum())
        ex = 1.01 * ((2.0 ** -11 + 2.0 ** -16) * F + 2.0 ** -25 * s * D)
        em = 1.01 * 2.0 ** -18 * F * np.linalg.norm(mu[k])
        # points of this component and of a neighbour, stored in fp16
        for src in (k, (k + 1) % K):
            x = (mu[src] + rng.standard_normal((n, D)) @ np.linalg.cholesky(S[src]).T)
            x16 = x.astype(np.float16)
            xf = x16.astype(np.float64)
            for r in range(n):
                zt = np.empty(D, dtype=np.float32)
                for i in range(D):
                    acc = _fp32_dot_random_order(x16[r], Wt[i], rng)
                    zt[i] = np.float32(np.float32(s) * acc - b[i])
                z = W[k] @ (xf[r] - mu[k])
                nz = float(np.sqrt(np.sum(zt.astype(np.float64) ** 2)))
                E = ex * np.linalg.norm(xf[r]) + em + 2.0 ** -15 * nz
                err = float(np.linalg.norm(zt.astype(np.float64) - z))
                assert err <= E, (case, k, r, err, E)
                worst = max(worst, err / E)
    print("%s: largest error / bound = %.3g" % (case, worst))
    # the bound is not vacuous: a hundred times smaller, it would fail here
    assert worst > 0.01, worst


def test_fc_screen_window_keeps_every_component_within_40_nats():
    """The mask from the bounds contains every component whose exact log joint
    is within 40 nats of the point's best (the workload's recipe, points of
    every component and midpoints between two)."""
    rng = np.random.default_rng(21)
    D, K, mu, S = _case("workload", rng)
    L = np.linalg.cholesky(S)
    W = np.tril(np.linalg.inv(L).astype(np.float32).astype(np.float64))
    c = np.log(1.0 / K) - np.log(np.diagonal(L, axis1=1, axis2=2)).sum(1) - 0.5 * D * np.log(2 * np.pi)
    pts = [mu[k] + rng.standard_normal(D) @ L[k].T for k in range(K) for _ in range(3)]
    pts += [0.5 * (mu[k] + mu[(k + 3) % K]) for k in range(K)]
    for x in pts:
        x16 = np.asarray(x).astype(np.float16)
        xf = x16.astype(np.float64)
        lo, hi, exact = np.empty(K), np.empty(K), np.empty(K)
        for k in range(K):
            s = _scale(W[k])
            Wt = (W[k] / s).astype(np.float16).astype(np.float64)
            b = (W[k] @ mu[k]).astype(np.float32).astype(np.float64)
            zt = (s * (Wt @ xf) - b).astype(np.float32).astype(np.float64)
            F = np.sqrt((W[k] ** 2).sum())
            E = (1.01 * ((2.0 ** -11 + 2.0 ** -16) * F + 2.0 ** -25 * s * D) * np.linalg.norm(xf)
                 + 1.01 * 2.0 ** -18 * F * np.linalg.norm(mu[k]) + 2.0 ** -15 * np.linalg.norm(zt))
            nz = np.linalg.norm(zt)
            lo[k] = c[k] - 0.5 * (nz + E) ** 2
            hi[k] = c[k] - 0.5 * max(0.0, nz - E) ** 2
            exact[k] = c[k] - 0.5 * np.sum((W[k] @ (xf - mu[k])) ** 2)
        mask = hi >= lo.max() - 41.0
        within = exact >= exact.max() - 40.0
        assert np.all(mask[within]), (np.nonzero(within & ~mask)[0], exact.max())
        assert lo.max() <= exact.max() <= hi.max()
