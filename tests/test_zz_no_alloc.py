"""gmm_em_step_noalloc: the EM step for callers that cannot allocate device
memory (a plugin given only its input and output buffers, code running
inside another framework's memory budget).  Its scratch is a fixed array
inside the library, so the call needs no workspace.

Checked through the C ABI on two calls in a row (two EM iterations, so the
second call finds the shared scratch holding the first call's contents):
against gmm_em_step on the same inputs, and each call against the fp64
oracle's step from that call's own input parameters, within the parity
tolerances the other GPU tests use.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import datagen
import parity
import soft_clustering_gb300 as G
from gpu_util import f32, make_state, oracle_step, set_opts, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from soft_clustering_gb300 import build
    build.build()


def _noalloc_step(wl, Xd, params, opts):
    pi, mu, cov = (torch.as_tensor(np.ascontiguousarray(p, dtype=np.float32)).cuda()
                   for p in params)
    ll = torch.zeros(1, dtype=torch.float64, device="cuda")
    lse = torch.empty(wl.N, dtype=torch.float32, device="cuda")
    flags = torch.zeros(wl.K, dtype=torch.int32, device="cuda")
    o = G.gmm_default_opts(**opts)
    st = G.gmm_em_step_noalloc(Xd, wl.dtype, wl.N, wl.D, wl.K, pi, mu, cov, wl.cov_type, ll, lse,
                               flags=flags, opts=o, raise_on_error=False)
    return st, dict(pi=pi.cpu().numpy().astype(np.float64), mu=mu.cpu().numpy().astype(np.float64),
                    cov=cov.cpu().numpy().astype(np.float64), ll=float(ll.item()),
                    lse=lse.cpu().numpy(), flags=flags.cpu().numpy())


@pytest.mark.parametrize("name,n", [("embed_diag", 20_003), ("full_cov", 9_001)])
def test_noalloc_matches_workspace_entry_point(name, n):
    wl = datagen.WORKLOADS[name].with_n(n)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta)
    Xd = to_device(bits, wl.dtype)
    ref_state = make_state(wl)
    set_opts(ref_state, opts)
    ref_state.set_params(*theta)
    lse_ref = torch.empty(wl.N, dtype=torch.float32, device="cuda")
    params = theta
    for call in range(2):
        # both entry points start every call from the same parameters (per-step
        # parity; each one's own trajectory amplifies last-bit differences)
        ref_state.set_params(*f32(params))
        ref_in = ref_state.params_numpy()
        ref_state.step(Xd, lse=lse_ref)
        assert ref_state.device_status() == G.GMM_OK
        pi, mu, cov = ref_state.params_numpy()
        ref = dict(pi=pi, mu=mu, cov=cov, ll=float(ref_state.loglik.item()))
        st, got = _noalloc_step(wl, Xd, params, opts)
        assert st == G.GMM_OK, G.status_string(st)
        fails = parity.compare_step(got, ref, "%s noalloc call %d" % (name, call))
        assert not fails, fails
        orc = oracle_step(bits, wl.dtype, params, wl.cov_type, opts=opts, want_lse=True)
        assert orc["status"] == 0
        fails = parity.compare_step(got, orc, "%s noalloc call %d vs oracle" % (name, call),
                                    opts["min_s0"])
        assert not fails, fails
        lse_ws = lse_ref.cpu().numpy()
        if wl.cov_type == datagen.COV_FULL:
            # For a few full-covariance components the workspace entry point
            # takes the candidate-mask kernels, which sum z = W (x - mu) in
            # another fp32 order than the CUDA-core kernels: both paths agree
            # with the oracle's LSE_n to fp32 evaluation error (ten times
            # inside the log-likelihood tolerance of 1e-4 relative).
            lo = orc["lse"]
            lo_ws = oracle_step(bits, wl.dtype, ref_in, wl.cov_type, opts=opts, want_lse=True)["lse"]
            scale = np.abs(lo).max()
            e_na, e_ws = np.abs(got["lse"] - lo).max(), np.abs(lse_ws - lo_ws).max()
            print("LSE_n max error vs oracle: CUDA-core %.3g, candidate-mask %.3g (scale %.1f)"
                  % (e_na, e_ws, scale))
            assert e_na <= 1e-5 * scale and e_ws <= 1e-5 * scale, (e_na, e_ws, scale)
        else:
            np.testing.assert_allclose(got["lse"], lse_ws, rtol=1e-6)
        assert (got["flags"] == ref_state.flags.cpu().numpy()).all()
        params = (got["pi"], got["mu"], got["cov"])


def test_noalloc_rejects_sizes_beyond_its_scratch():
    N, D, K = 256, 128, 60_000   # ~120 MB of statistics partials: over the 64 MiB limit
    X = torch.zeros(N * D, dtype=torch.float16, device="cuda")
    pi = torch.full((K,), 1.0 / K, device="cuda")
    mu = torch.zeros(K, D, device="cuda")
    var = torch.ones(K, D, device="cuda")
    ll = torch.zeros(1, dtype=torch.float64, device="cuda")
    lse = torch.empty(N, device="cuda")
    st = G.gmm_em_step_noalloc(X, G.GMM_F16, N, D, K, pi, mu, var, G.GMM_COV_DIAG, ll, lse,
                               raise_on_error=False)
    assert st == G.GMM_ERR_WORKSPACE
