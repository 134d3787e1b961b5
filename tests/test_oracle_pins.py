"""The fp64 oracle against its pins (no GPU)."""
import numpy as np
import pytest

import datagen
import oracle
import oracle_pins as P


@pytest.mark.parametrize("name,fn", P.ALL_QUICK_PINS, ids=[n for n, _ in P.ALL_QUICK_PINS])
def test_quick_pin(name, fn):
    fn(oracle.lib())


def test_ll_monotone_tiny_diag():
    wl = datagen.WORKLOADS["tiny_diag"]
    mix = datagen.planted(wl)
    X = datagen.points(mix, 0, wl.N)
    pi, mu, cov = datagen.init_params(mix, X)
    lls = P.pin_ll_monotone(oracle.lib(), X, pi, mu, cov, wl.cov_type, 25)
    assert lls[-1] > lls[0]


def test_ll_monotone_full_subset():
    wl = datagen.WORKLOADS["full_cov"].with_n(6000)
    mix = datagen.planted(wl)
    X = datagen.points(mix, 0, wl.N)
    pi, mu, cov = datagen.init_params(mix, X)
    P.pin_ll_monotone(oracle.lib(), X, pi, mu, cov, wl.cov_type, 6, xdtype=wl.dtype)


def test_ll_monotone_iso_bf16_subset():
    wl = datagen.WORKLOADS["large_diag"].with_n(20000)
    wl.K = 32
    wl.cov_type = oracle.COV_ISO
    mix = datagen.planted(wl)
    X = datagen.points(mix, 0, wl.N)
    pi, mu, cov = datagen.init_params(mix, X)
    P.pin_ll_monotone(oracle.lib(), X, pi, mu, cov, wl.cov_type, 5, xdtype=wl.dtype)


def test_planted_recovery_tiny_diag():
    """Well separated planted mixture (tiny_diag: 8 centres drawn N(0, 4^2)
    in 16-D, variances in [0.5, 2]): from theta_0 EM finds the centres."""
    wl = datagen.WORKLOADS["tiny_diag"].with_n(60000)
    mix = datagen.planted(wl)
    X = datagen.points(mix, 0, wl.N)
    # start from the planted parameters perturbed: one step stays within
    # sampling error of the truth
    true_var = mix.sd ** 2
    r = oracle.em_step(X, mix.weights, mix.mu, true_var, oracle.COV_DIAG)
    n_k = mix.weights * wl.N
    sig = np.sqrt(true_var)
    assert (np.abs(r["mu"] - mix.mu) < 5 * sig / np.sqrt(n_k)[:, None]).all()
    assert (np.abs(r["pi"] - mix.weights) < 5 * np.sqrt(mix.weights * (1 - mix.weights) / wl.N)).all()
    # from the centres shifted by half a standard deviation, EM walks back
    init = (np.full(wl.K, 1.0 / wl.K), mix.mu + 0.5 * sig, true_var * 1.5)
    res, ri, ci = P.pin_planted_recovery(oracle.lib(), X, None, mix.weights, mix.mu, true_var,
                                         init, 30, tol_mu=0.1)
    assert np.abs(res["pi"][ri] - mix.weights[ci]).max() < 0.01


def test_ridge_and_not_pd():
    X = np.zeros((3, 2), dtype=np.float32)
    pi = np.array([1.0])
    mu = np.zeros((1, 2))
    st, lj, flags = oracle.log_joint(X, pi, mu, np.array([[[1.0, 1.0], [1.0, 1.0]]]),
                                     oracle.COV_FULL)
    assert st == 0 and flags[0] == oracle.FLAG_RIDGE
    st, lj, flags = oracle.log_joint(X, pi, mu, np.array([[[-1.0, 0.0], [0.0, -1.0]]]),
                                     oracle.COV_FULL)
    assert st == oracle.NOT_PD and flags[0] & oracle.FLAG_NOT_PD
    st, lj, flags = oracle.log_joint(X, pi, mu, np.array([[0.0, 1.0]]), oracle.COV_DIAG)
    assert st == 0 and flags[0] == oracle.FLAG_RIDGE


def test_var_floor_and_empty_component():
    X = np.array([[0.0], [0.0], [0.0], [1e-4]], dtype=np.float32)
    pi = np.array([0.5, 0.5])
    mu = np.array([[0.0], [1e6]])
    var = np.array([[1.0], [1.0]])
    r = oracle.em_step(X, pi, mu, var, oracle.COV_DIAG, opts=dict(var_floor=1e-3, min_s0=1e-3))
    assert r["flags"][0] & oracle.FLAG_FLOOR and r["cov"][0, 0] == 1e-3
    assert r["flags"][1] & oracle.FLAG_EMPTY
    assert r["mu"][1, 0] == 1e6 and r["cov"][1, 0] == 1.0 and r["pi"][1] == 0.0


def test_sklearn_one_step_cross_check():
    """One EM step against scikit-learn's GaussianMixture update (a third
    implementation), with its covariance regulariser switched off."""
    mix_mod = pytest.importorskip("sklearn.mixture")
    rng = np.random.default_rng(11)
    N, D, K = 400, 3, 3
    X = np.concatenate([rng.standard_normal((N // 2, D)) + 3, rng.standard_normal((N // 2, D))])
    X = X.astype(np.float32)
    pi = np.array([0.2, 0.3, 0.5])
    mu = rng.standard_normal((K, D))
    A = rng.standard_normal((K, D, D))
    S = np.einsum("kij,klj->kil", A, A) / D + 0.5 * np.eye(D)
    gm = mix_mod.GaussianMixture(K, covariance_type="full", reg_covar=0.0, max_iter=1,
                                 init_params="random", tol=0.0)
    gm.weights_, gm.means_, gm.covariances_ = pi, mu, S
    gm.precisions_cholesky_ = np.stack([np.linalg.cholesky(np.linalg.inv(s)) for s in S])
    Xd = X.astype(np.float64)
    log_resp = gm._estimate_log_prob_resp(Xd)[1]
    gm._m_step(Xd, log_resp)
    r = oracle.em_step(X, pi, mu, S, oracle.COV_FULL)
    P._close(r["pi"], gm.weights_, 1e-12, 1e-14, "sklearn pi")
    P._close(r["mu"], gm.means_, 1e-10, 1e-12, "sklearn mu")
    P._close(r["cov"], gm.covariances_, 1e-9, 1e-12, "sklearn Sigma")
