"""GMMState.fit on the GPU: the library's EM steps driven to convergence
(Flash-GMM summary, Method: the same step repeats until the log-likelihood
converges), against the oracle driven by the same loop.

Each iteration's log-likelihood is compared with the oracle's trajectory from
the same theta_0 (relative error <= 1e-4 per iteration), the sequence must
be non-decreasing, and the stop iteration must be the oracle's unless the
oracle's relative rise at either side of it lies within 5% of the tolerance
(there the stop decision rests on rounding).
"""
import numpy as np
import pytest
import torch

import datagen
import oracle
import parity
from gpu_util import f32, make_state, set_opts, to_device
from soft_clustering_gb300 import em_loop

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from soft_clustering_gb300 import build
    build.build()


def _oracle_fit(bits, wl, theta, opts, max_iters, tol):
    """The oracle under the same loop and stop rule, fp32 parameters
    between steps (the library's parameter type)."""
    cur = {"theta": theta}

    def step():
        r = oracle.em_step(bits, *(np.asarray(p, np.float64) for p in cur["theta"]), wl.cov_type,
                           xdtype=wl.dtype, opts=opts)
        assert r["status"] == 0
        cur["theta"] = f32((r["pi"], r["mu"], r["cov"]))
        cur["ll"] = r["ll"]
    return em_loop.run_em(step, lambda: cur["ll"], max_iters, tol)


def _check(name, n, max_iters, tol):
    wl = datagen.WORKLOADS[name]
    if n:
        wl = wl.with_n(n)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta0 = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta0)
    st = make_state(wl)
    set_opts(st, opts)
    st.set_params(*theta0)
    got = st.fit(to_device(bits, wl.dtype), max_iters, tol)
    assert st.device_status() == 0
    ref = _oracle_fit(bits, wl, theta0, opts, max_iters, tol)
    assert got["monotone"], got["ll_history"]
    h_ref = ref["ll_history"]
    n_cmp = min(len(got["ll_history"]), len(h_ref))
    for t in range(n_cmp):
        g, r = got["ll_history"][t], h_ref[t]
        assert abs(g - r) <= parity.LL_RTOL * abs(r), (t, g, r)
    if got["iterations"] != ref["iterations"]:
        # only a near-threshold rise may move the stop by one iteration
        t = min(got["iterations"], ref["iterations"]) - 1
        rises = [abs(h_ref[i] - h_ref[i - 1]) / abs(h_ref[i]) for i in (t, t + 1)
                 if 1 <= i < len(h_ref)]
        assert abs(got["iterations"] - ref["iterations"]) == 1 and tol > 0, (got, ref)
        assert any(abs(x - tol) <= 0.05 * tol for x in rises), (rises, tol)
    return got, ref


def test_fit_tiny_diag_ten_iterations():
    """The 4096-point workload's 10 iterations (tol 0: every iteration runs)."""
    got, ref = _check("tiny_diag", None, 10, 0.0)
    assert got["iterations"] == 10 and not got["converged"]


def test_fit_embed_subset_to_tolerance():
    """A 20,000-point slice of the embedding workload (tensor-core path)
    iterated until the relative rise is at most 1e-6."""
    got, ref = _check("embed_diag", 20_000, 40, 1e-6)
    assert got["converged"] and ref["converged"]
