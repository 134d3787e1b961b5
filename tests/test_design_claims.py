"""CPU checks of two premises the tensor-core design rests on (no GPU).

1. After the first EM iterations a point has few components within 40 nats
   of its best log joint, so exact evaluation of only those (and records
   for them) costs little next to the screening contraction.  Measured with
   the oracle on a subset of the embedding-like workload.
2. A plain fp32 running sum of the D = 128 terms w_d (x_d - mu_d)^2 errs by
   several 1e-5 nats, too much for parameters held to 2e-3 of 1e-3 of their
   scale; the kernels' order (32 partial sums of D/32 terms, then a pairwise
   tree) stays near 1e-5.
"""
import numpy as np

import datagen
import oracle


def _within(L, nats=40.0):
    return (L >= L.max(axis=1, keepdims=True) - nats).sum(axis=1)


def test_candidates_are_few_after_the_first_iterations():
    wl = datagen.WORKLOADS["embed_diag"].with_n(20_000)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = tuple(np.asarray(p, np.float32) for p in datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta)
    counts = []
    for it in range(4):
        st, L, _ = oracle.log_joint(bits, *(np.asarray(p, np.float64) for p in theta),
                                    wl.cov_type, xdtype=wl.dtype)
        assert st == 0
        counts.append(_within(L))
        r = oracle.em_step(bits, *(np.asarray(p, np.float64) for p in theta), wl.cov_type,
                           xdtype=wl.dtype, opts=opts)
        assert r["status"] == 0
        theta = tuple(np.asarray(r[k], np.float32) for k in ("pi", "mu", "cov"))
    means = [float(c.mean()) for c in counts]
    print("mean components within 40 nats, iterations 0-3:", means,
          "max:", [int(c.max()) for c in counts])
    assert means[0] > 10.0            # theta_0: dense windows (the first iteration pays)
    assert means[3] < 2.0             # iteration 3: about one per point
    assert all(c.min() >= 1 for c in counts)


def _tree32(terms):
    """The kernels' order: 32 partial sums of D/32 consecutive terms
    (sequential, fp32), then a pairwise tree over the partials."""
    D = terms.shape[1]
    per = D // 32
    p = np.zeros((terms.shape[0], 32), np.float32)
    for i in range(per):
        p = (p + terms[:, np.arange(32) * per + i]).astype(np.float32)
    w = 16
    while w >= 1:
        p = (p[:, :w] + p[:, w:2 * w]).astype(np.float32)
        w //= 2
    return p[:, 0]


def test_split_partial_sums_beat_a_running_sum():
    rng = np.random.default_rng(4)
    n, D = 4000, 128
    # terms of ~2 (a point a few sigma from a tight component)
    terms = (rng.standard_normal((n, D)) ** 2 * 2.0).astype(np.float32)
    exact = terms.astype(np.float64).sum(axis=1)
    run = np.zeros(n, np.float32)
    for d in range(D):
        run = (run + terms[:, d]).astype(np.float32)
    tree = _tree32(terms)
    e_run = np.abs(run - exact).mean() * 0.5    # l = c - d^2 / 2
    e_tree = np.abs(tree - exact).mean() * 0.5
    print("|error| in nats, mean / max: running sum %.2e / %.2e, 32-partial tree %.2e / %.2e"
          % (e_run, np.abs(run - exact).max() * 0.5, e_tree, np.abs(tree - exact).max() * 0.5))
    assert 1e-5 < e_run < 2e-4
    assert e_tree < e_run / 3
