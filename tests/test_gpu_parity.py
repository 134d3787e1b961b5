"""CUDA path vs the fp64 oracle, element by element, on seeded inputs.

Sizes are ones the oracle finishes in seconds, spanning several tiles with a
ragged tail.  Per-step parity feeds both sides the same fp32 parameters
(the oracle's own trajectory, rounded to fp32 - never values from the GPU);
a trajectory lets each side iterate on its own from theta_0 (a diagnostic:
its log-likelihood is held to the per-iteration bound, its parameters are
reported).  Multi-slab tests cross the tensor-core path's 2^21-row slabs.
"""
import numpy as np
import pytest
import torch

import datagen
import oracle
import parity
from gpu_util import f32, gpu_step, make_state, oracle_step, set_opts, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from soft_clustering_gb300 import build
    build.build()


def _workload(name, n=None, **over):
    wl = datagen.WORKLOADS[name]
    if n is not None:
        wl = wl.with_n(n)
    for k, v in over.items():
        setattr(wl, k, v)
    return wl


def _run_parity(wl, iters, trajectory=True):
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta0 = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta0)
    Xd = to_device(bits, wl.dtype)
    state = make_state(wl)
    fails = []
    # per step: both sides start each step from the oracle's (fp32-rounded) parameters
    theta = theta0
    for t in range(iters):
        ref = oracle_step(bits, wl.dtype, theta, wl.cov_type, opts=opts)
        assert ref["status"] == 0
        got = gpu_step(state, Xd, theta, opts=opts)
        assert got["status"] == 0, got["status"]
        fails += parity.compare_step(got, ref, "%s step %d" % (wl.name, t), opts["min_s0"])
        theta = f32((ref["pi"], ref["mu"], ref["cov"]))
    # trajectory: each side on its own from theta_0.  A diagnostic, not the
    # parity criterion: EM amplifies last-bit differences of an iterate
    # through components that hinge on a few boundary points, so after the
    # first step the two trajectories are different (equally valid) runs.
    # Held: the per-iteration log-likelihood bound and EM's non-decreasing
    # log-likelihood; the parameter differences are reported, not asserted.
    if trajectory:
        ref_theta = theta0
        state.set_params(*theta0)
        prev = -np.inf
        for t in range(iters):
            ref = oracle_step(bits, wl.dtype, ref_theta, wl.cov_type, opts=opts)
            state.step(Xd)
            pi, mu, cov = state.params_numpy()
            got = dict(pi=pi, mu=mu, cov=cov, ll=float(state.loglik.item()))
            tf = parity.compare_step(got, ref, "%s trajectory %d" % (wl.name, t), opts["min_s0"])
            fails += [f for f in tf if " LL " in f]
            diag = [f for f in tf if " LL " not in f]
            if diag:
                print("trajectory diagnostic:", "; ".join(d[:160] for d in diag))
            if not got["ll"] >= prev - 1e-6 * abs(prev):
                fails.append("%s trajectory %d: LL decreased %.10g -> %.10g"
                             % (wl.name, t, prev, got["ll"]))
            prev = got["ll"]
            ref_theta = (ref["pi"], ref["mu"], ref["cov"])
    if fails:
        bundle = parity.replay_bundle(wl, bits, theta0, fails)
        fails.insert(0, "replay bundle: %s" % bundle)
    assert not fails, "\n".join(fails[:10])


def test_tiny_diag_full_size():
    """N=4096, D=16, K=8, fp32 X, 10 iterations (full size)."""
    _run_parity(_workload("tiny_diag"), 10)


def test_full_cov_subset():
    _run_parity(_workload("full_cov", n=20_000 + 37), 4)


def test_embed_diag_subset():
    _run_parity(_workload("embed_diag", n=12_000 + 61), 3)


def test_large_diag_subset_bf16():
    _run_parity(_workload("large_diag", n=8_000 + 5), 2)


def test_large_iso_subset_bf16():
    _run_parity(_workload("large_diag", n=8_000 + 5, cov_type=datagen.COV_ISO, K=64), 3)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("cov", [datagen.COV_FULL, datagen.COV_DIAG, datagen.COV_ISO])
@pytest.mark.parametrize("xdtype", [datagen.F32, datagen.F16, datagen.BF16])
def test_shapes_dtypes(D, cov, xdtype):
    """Every (D, covariance, dtype) on a ragged N and a K that is not a
    multiple of any chunk."""
    kind = datagen.MIX_FULL if cov == datagen.COV_FULL else datagen.MIX_DIAG
    recipe = (dict(mean_sd=2.0, ridge=0.2, alpha=2.0) if kind == datagen.MIX_FULL else
              dict(mean_sd=2.0, sd_mode=0, lo=0.3, hi=1.5, alpha=2.0))
    wl = datagen.Workload("shape", 100 + D + 7 * cov + 31 * xdtype, 1000 + 3, D, 11, xdtype, cov,
                          1, kind, recipe)
    _run_parity(wl, 1, trajectory=False)


def test_assign_topm_subset():
    wl = _workload("ivf_assign", n=6_000 + 13)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    pi, mu, var = datagen.planted_params_f16(mix)
    st, ids_ref, gam_ref, lse_ref = oracle.topm(bits, pi, mu, var, wl.cov_type, wl.m,
                                                xdtype=wl.dtype)
    assert st == 0
    from soft_clustering_gb300.torch_api import Assigner
    a = Assigner(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, wl.m)
    a.prepare(pi, mu, var)
    a.assign(to_device(bits, wl.dtype))
    assert a.device_status() == 0
    ids = a.ids.cpu().numpy()
    gam = a.gamma.cpu().numpy().astype(np.float64)
    lse = a.lse.cpu().numpy().astype(np.float64)
    agree, kept = parity.top1_agreement(ids, ids_ref, gam_ref)
    assert agree >= parity.TOP1_MIN, (agree, kept)
    assert np.abs(lse - lse_ref).max() <= 1e-4 * np.abs(lse_ref).max()
    # every rank, in order, with its gamma
    st, L, _ = oracle.log_joint(bits, pi, mu, var, wl.cov_type, xdtype=wl.dtype)
    assert st == 0
    fails = parity.topm_compare(ids, gam, L, lse_ref, "ivf subset")
    assert not fails, fails


def test_deterministic():
    wl = _workload("embed_diag", n=5_000)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    Xd = to_device(bits, wl.dtype)
    s = make_state(wl)
    a = gpu_step(s, Xd, theta)
    b = gpu_step(s, Xd, theta)
    for k in ("pi", "mu", "cov"):
        assert (a[k] == b[k]).all(), k
    assert a["ll"] == b["ll"]


def test_no_device_allocation_in_step():
    """The library allocates nothing: free device memory is unchanged by a
    step (torch's allocator is not involved in the call)."""
    wl = _workload("embed_diag", n=50_000)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    Xd = to_device(bits, wl.dtype)
    s = make_state(wl)
    gpu_step(s, Xd, theta)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    gpu_step(s, Xd, theta)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    # no N x K buffer: past one slab of records the workspace grows by O(N)
    # bytes only (LSE_n and the hand-over bitmap and list, 8.25 bytes a
    # point), and stays below an N x K fp32 matrix
    import soft_clustering_gb300 as G
    n1, n2 = 1 << 22, 1 << 24
    w1 = G.gmm_workspace_bytes(n1, wl.D, wl.K, wl.cov_type, wl.dtype)
    w2 = G.gmm_workspace_bytes(n2, wl.D, wl.K, wl.cov_type, wl.dtype)
    assert w2 - w1 <= 9 * (n2 - n1), (w1, w2)
    assert w1 < n1 * wl.K * 4 and w2 < n2 * wl.K * 4


def test_host_streaming_matches():
    wl = _workload("embed_diag", n=30_000 + 9)
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta)
    ref = oracle_step(bits, wl.dtype, theta, wl.cov_type, opts=opts)
    s = make_state(wl, chunk_rows=7_000)
    set_opts(s, opts)
    s.set_params(*theta)
    host = torch.from_numpy(bits.view(np.int16)).pin_memory()
    ll_host = np.zeros(1)
    s.step_host(host, loglik_host=ll_host)
    assert s.device_status() == 0
    pi, mu, cov = s.params_numpy()
    fails = parity.compare_step(dict(pi=pi, mu=mu, cov=cov, ll=float(ll_host[0])), ref, "host",
                                opts["min_s0"])
    assert not fails, fails


def test_edge_cases_small():
    """N = 1, K = 1, a single tile, and K larger than N."""
    for N, K in [(1, 1), (1, 3), (5, 1), (127, 2), (129, 200)]:
        wl = datagen.Workload("edge", 77 + N + K, N, 16, K, datagen.F32, datagen.COV_DIAG, 1,
                              datagen.MIX_DIAG, dict(mean_sd=1.0, sd_mode=0, lo=0.5, hi=1.0,
                                                     alpha=1.0))
        mix = datagen.planted(wl)
        bits = datagen.points(mix, 0, N)
        pi = np.full(K, 1.0 / K, dtype=np.float32)
        mu = (mix.mu.astype(np.float32) * 0.5)
        var = np.ones((K, 16), dtype=np.float32)
        # one point has zero variance: the floor makes the update defined
        opts = dict(var_floor=1e-6, min_s0=0.5)
        ref = oracle_step(bits, wl.dtype, (pi, mu, var), wl.cov_type, opts=opts)
        got = gpu_step(make_state(wl), to_device(bits, wl.dtype), (pi, mu, var), opts=opts)
        fails = parity.compare_step(got, ref, "N=%d K=%d" % (N, K), 0.5)
        assert not fails, fails
        assert (got["flags"] == ref["flags"]).all(), (got["flags"], ref["flags"])


@pytest.mark.parametrize("D,xdtype,cov", [(128, datagen.F16, datagen.COV_DIAG),
                                          (64, datagen.BF16, datagen.COV_ISO)])
def test_tensor_core_edge_cases(D, xdtype, cov):
    """The tensor-core path at degenerate sizes: one point (one tile, 127 rows
    past the end), a partial tile, exactly one full tile, one row past it,
    and K from 1 (one chunk, 127 padding columns) to two full folded chunks.
    Against the oracle, with and without LSE_n."""
    for N, K in [(1, 1), (1, 5), (7, 3), (128, 256), (129, 200)]:
        wl = datagen.Workload("tc_edge", 300 + N + K + D, N, D, K, xdtype, cov, 1,
                              datagen.MIX_DIAG, dict(mean_sd=1.0, sd_mode=0, lo=0.5, hi=1.0,
                                                     alpha=1.0))
        mix = datagen.planted(wl)
        bits = datagen.points(mix, 0, N)
        pi = np.full(K, 1.0 / K, dtype=np.float32)
        mu = mix.mu.astype(np.float32) * 0.5
        var = np.ones((K, D) if cov == datagen.COV_DIAG else (K,), dtype=np.float32)
        opts = dict(var_floor=1e-6, min_s0=0.5)
        ref = oracle_step(bits, wl.dtype, (pi, mu, var), wl.cov_type, opts=opts, want_lse=True)
        assert ref["status"] == 0
        Xd = to_device(bits, wl.dtype)
        for want_lse in (False, True):
            got = gpu_step(make_state(wl), Xd, (pi, mu, var), want_lse=want_lse, opts=opts)
            assert got["status"] == 0, (N, K, got["status"])
            fails = parity.compare_step(got, ref, "N=%d K=%d lse=%d" % (N, K, want_lse), 0.5)
            assert not fails, fails
            assert (got["flags"] == ref["flags"]).all(), (got["flags"], ref["flags"])
            if want_lse:
                np.testing.assert_allclose(got["lse"], ref["lse"], rtol=1e-5, atol=1e-3)


def test_empty_floor_notpd_flags():
    """Empty component (mean far away), variance floor, and a covariance that
    is not positive definite: same flags and parameters as the oracle."""
    rng = np.random.default_rng(5)
    N, D, K = 2000, 16, 4
    X = (rng.standard_normal((N, D))).astype(np.float32)
    pi = np.full(K, 0.25, dtype=np.float32)
    mu = np.zeros((K, D), dtype=np.float32)
    mu[1] = 1e4  # takes no responsibility -> empty
    mu[2] = 0.5
    var = np.ones((K, D), dtype=np.float32)
    var[3, 0] = 0.0  # ridge retry (1e-3 tr/D) repairs it
    opts = dict(var_floor=0.9, min_s0=0.5)
    wl = datagen.Workload("flags", 0, N, D, K, datagen.F32, datagen.COV_DIAG, 1, 0, {})
    ref = oracle_step(X, datagen.F32, (pi, mu, var), wl.cov_type, opts=opts)
    s = make_state(wl)
    got = gpu_step(s, to_device(X, datagen.F32), (pi, mu, var), opts=opts)
    assert (got["flags"] == ref["flags"]).all(), (got["flags"], ref["flags"])
    assert got["flags"][1] & oracle.FLAG_EMPTY and got["flags"][3] & oracle.FLAG_RIDGE
    fails = parity.compare_step(got, ref, "flags")
    assert not fails, fails
    # not positive definite even after the retry: status NOT_PD, component excluded
    var2 = var.copy()
    var2[3, :] = -1.0
    got = gpu_step(s, to_device(X, datagen.F32), (pi, mu, var2))
    assert got["status"] == 3 and got["flags"][3] & oracle.FLAG_NOT_PD


@pytest.mark.parametrize("K", [200, 300])
def test_screen_wide_scales(K):
    """Screening operands with one scale per chunk (K = 200: resident and
    folded, two chunks; K = 300: streamed, three chunks; the last chunk
    ragged) under a 20:1 spread of sigma within a chunk and a component far
    from every point that sets its chunk's scale, so that small operands
    fall fp16-subnormal; with a dead component (pi = 0).  The same step as
    the oracle, with and without LSE_n, and the same top-4 assignment."""
    rng = np.random.default_rng(23 + K)
    N, D = 3001, 128
    centres = rng.standard_normal((K, D)) * 0.3
    sd = (np.exp(rng.uniform(np.log(0.05), np.log(1.0), (K, 1))) *
          np.exp(rng.uniform(-0.3, 0.3, (K, D))))
    lab = rng.integers(0, K, N)
    X = (centres[lab] + rng.standard_normal((N, D)) * sd[lab]).astype(np.float16)
    bits = X.view(np.uint16)
    pi = rng.dirichlet(np.full(K, 1.0))
    pi[7] = 0.0
    pi = (pi / pi.sum()).astype(np.float32)
    mu = (centres + 0.1 * sd * rng.standard_normal((K, D))).astype(np.float32)
    mu[13] = 300.0   # sets chunk 0's common scale: its other operands shrink
    var = (sd ** 2 * rng.uniform(0.8, 1.25, (K, D))).astype(np.float32)
    var[13] = 1.0
    opts = dict(var_floor=1e-8, min_s0=0.5)
    wl = datagen.Workload("wide", 0, N, D, K, datagen.F16, datagen.COV_DIAG, 1, 0, {})
    ref = oracle_step(bits, datagen.F16, (pi, mu, var), wl.cov_type, opts=opts, want_lse=True)
    s = make_state(wl)
    Xd = to_device(bits, datagen.F16)
    for want_lse in (False, True):
        got = gpu_step(s, Xd, (pi, mu, var), want_lse=want_lse, opts=opts)
        assert got["status"] == 0, got["status"]
        # the screen keeps most rows (the rest take the CUDA-core row list)
        handed = int(s.ws[8:12].cpu().numpy().view(np.uint32)[0])
        assert handed < N // 2, handed
        fails = parity.compare_step(got, ref, "K=%d lse=%d" % (K, want_lse), opts["min_s0"])
        assert not fails, "\n".join(fails[:10])
        if want_lse:
            assert np.abs(got["lse"] - ref["lse"]).max() <= 1e-4 * np.abs(ref["lse"]).max()
    # the same operands in assignment mode (top-4)
    m = 4
    st, ids_ref, gam_ref, lse_ref = oracle.topm(bits, pi, mu, var, wl.cov_type, m,
                                                xdtype=datagen.F16)
    assert st == 0
    from soft_clustering_gb300.torch_api import Assigner
    a = Assigner(N, D, K, wl.cov_type, datagen.F16, m)
    a.prepare(pi, mu, var)
    a.assign(Xd)
    assert a.device_status() == 0
    ids = a.ids.cpu().numpy()
    agree, kept = parity.top1_agreement(ids, ids_ref, gam_ref)
    assert agree >= parity.TOP1_MIN, (agree, kept)
    lse = a.lse.cpu().numpy().astype(np.float64)
    assert np.abs(lse - lse_ref).max() <= 1e-4 * np.abs(lse_ref).max()
    st, L, _ = oracle.log_joint(bits, pi, mu, var, wl.cov_type, xdtype=datagen.F16)
    assert st == 0
    fails = parity.topm_compare(ids, a.gamma.cpu().numpy(), L, lse_ref, "wide K=%d" % K)
    assert not fails, fails


def test_nonfinite_input_reported():
    N, D, K = 300, 16, 2
    X = np.random.default_rng(1).standard_normal((N, D)).astype(np.float32)
    X[17, 3] = np.nan
    wl = datagen.Workload("nan", 0, N, D, K, datagen.F32, datagen.COV_DIAG, 1, 0, {})
    s = make_state(wl)
    got = gpu_step(s, to_device(X, datagen.F32),
                   (np.full(K, 0.5, np.float32), np.zeros((K, D), np.float32),
                    np.ones((K, D), np.float32)))
    assert got["status"] == 4  # GMM_ERR_NONFINITE


def test_invalid_workspace_and_alignment():
    import soft_clustering_gb300 as G
    wl = _workload("tiny_diag", n=256)
    s = make_state(wl)
    X = torch.zeros(wl.N * wl.D + 1, dtype=torch.float32, device="cuda")
    st = G.gmm_em_step(X, wl.dtype, wl.N, wl.D, wl.K, s.pi, s.mu, s.cov, wl.cov_type, s.ws,
                       s.ws_bytes - 1, s.loglik, raise_on_error=False)
    assert st == G.GMM_ERR_WORKSPACE
    st = G.gmm_em_step(X.data_ptr() + 4, wl.dtype, wl.N, wl.D, wl.K, s.pi, s.mu, s.cov,
                       wl.cov_type, s.ws, s.ws_bytes, s.loglik, raise_on_error=False)
    assert st == G.GMM_ERR_INVALID_ARG


@pytest.mark.parametrize("name,n,cov", [("embed_diag", 20_011, datagen.COV_DIAG),
                                        ("large_diag", 9_003, datagen.COV_DIAG),
                                        ("large_diag", 9_003, datagen.COV_ISO)])
def test_tensor_core_path_matches_cuda_core_path(name, n, cov):
    """The tensor-core screening path and the CUDA-core path agree point by
    point (LSE_n) and on the updated parameters, at theta_0 (dense candidate
    lists, many rows handed over) and one iteration later (sparse lists)."""
    import soft_clustering_gb300 as G
    wl = _workload(name, n=n, cov_type=cov, K=min(datagen.WORKLOADS[name].K, 512))
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta)
    Xd = to_device(bits, wl.dtype)
    for it in range(2):
        tc = gpu_step(make_state(wl), Xd, theta, want_lse=True, opts=opts)
        cc = gpu_step(make_state(wl), Xd, theta, want_lse=True,
                      opts=dict(opts, flags=G.GMM_OPT_CUDA_CORES))
        assert tc["status"] == 0 and cc["status"] == 0
        np.testing.assert_allclose(tc["lse"], cc["lse"], rtol=2e-6, atol=2e-4)
        fails = parity.compare_step(tc, cc, "%s iter %d tc vs cuda cores" % (name, it))
        assert not fails, fails
        theta = f32((cc["pi"], cc["mu"], cc["cov"]))


def test_full_lists_go_to_dense_rows_and_match_oracle():
    """A point's candidate list in the screening kernel holds 13 (resident
    parameters) or 15 (streamed, per column half) components; a point with
    more goes with its candidate masks to the dense-row kernels.  24 copies of
    one component, all within every nearby point's window, force that for
    many points; none is handed to the CUDA-core row list, and the step
    matches the oracle."""
    for K in (256, 300):
        wl = _workload("embed_diag", n=20000, K=K)
        mix = datagen.planted(wl)
        bits = datagen.points(mix, 0, wl.N)
        pi, mu, cov = (np.array(p) for p in f32(datagen.init_params(mix, bits)))
        mu[1:24] = mu[0]
        cov[1:24] = cov[0]
        pi[1:24] = pi[0]
        pi /= pi.sum()
        theta = f32((pi, mu, cov))
        opts = datagen.em_opts(theta)
        state = make_state(wl)
        ref = oracle_step(bits, wl.dtype, theta, wl.cov_type, opts=opts)
        got = gpu_step(state, to_device(bits, wl.dtype), theta, opts=opts)
        assert got["status"] == 0
        # the library's status word: code, detail, rows handed to the CUDA-core path
        handed, dense = (int(v) for v in state.ws[8:16].cpu().numpy().view(np.uint32))
        assert handed < wl.N // 4, handed
        assert dense > 0, dense
        fails = parity.compare_step(got, ref, "full lists K=%d" % K, opts["min_s0"])
        assert not fails, "\n".join(fails[:10])


def test_many_candidates_take_the_dense_row_kernels():
    """K = 300 components with nearly the same mean and variance: every
    point keeps all 300 as candidates, more than the screening kernel's
    lists hold, so the points go with their candidate masks to the dense-row
    kernels (parameters staged in shared memory).  Steps from these
    parameters and from the oracle's next iterate match the oracle."""
    rng = np.random.default_rng(41)
    N, D, K = 4000, 128, 300
    # data and means away from the origin, so that every mean entry is of
    # the order of the mean array's scale (the tolerance's reference)
    X = (1.0 + rng.standard_normal((N, D)) * 0.5).astype(np.float16)
    bits = X.view(np.uint16)
    pi = np.full(K, 1.0 / K, dtype=np.float32)
    mu = (1.0 + rng.standard_normal((K, D)) * 0.01).astype(np.float32)
    var = np.full((K, D), 0.25, dtype=np.float32) * rng.uniform(0.99, 1.01, (K, 1)).astype(np.float32)
    opts = dict(var_floor=1e-6, min_s0=0.5)
    wl = datagen.Workload("dense", 0, N, D, K, datagen.F16, datagen.COV_DIAG, 1, 0, {})
    theta = (pi, mu, var)
    Xd = to_device(bits, datagen.F16)
    for step in range(2):
        ref = oracle_step(bits, datagen.F16, theta, wl.cov_type, opts=opts, want_lse=True)
        for want_lse in (False, True):
            st = make_state(wl)
            got = gpu_step(st, Xd, theta, want_lse=want_lse, opts=opts)
            assert got["status"] == 0, got["status"]
            if step == 0:
                # status word: code, detail, rows to the CUDA-core path, rows to the dense kernels
                assert int(st.ws[12:16].cpu().numpy().view(np.uint32)[0]) > N // 2
            fails = parity.compare_step(got, ref, "dense step %d lse=%d" % (step, want_lse), 0.5)
            assert not fails, "\n".join(fails[:10])
            if want_lse:
                np.testing.assert_allclose(got["lse"], ref["lse"], rtol=1e-5, atol=1e-3)
        theta = f32((ref["pi"], ref["mu"], ref["cov"]))


@pytest.mark.parametrize("K", [200, 300])
def test_nonfinite_input_reported_tensor_core(K):
    """A NaN coordinate on the tensor-core path (D = 128, fp16; resident and
    streamed parameters) gives GMM_ERR_NONFINITE."""
    rng = np.random.default_rng(K)
    N, D = 1000, 128
    X = rng.standard_normal((N, D)).astype(np.float16)
    X[517, 9] = np.nan
    wl = datagen.Workload("nan_tc", 0, N, D, K, datagen.F16, datagen.COV_DIAG, 1, 0, {})
    got = gpu_step(make_state(wl), to_device(X.view(np.uint16), datagen.F16),
                   (np.full(K, 1.0 / K, np.float32), rng.standard_normal((K, D)).astype(np.float32),
                    np.ones((K, D), np.float32)))
    assert got["status"] == 4  # GMM_ERR_NONFINITE


def test_embed_diag_full_size_sampled():
    """The bench's own launch configuration (1e7 points, 2M-row slabs): LSE_n
    of sampled points against the oracle's fp64 log-sum-exp of the same
    points, the log-likelihood against the sum of the LSE outputs, and the
    updated weights summing to one."""
    wl = datagen.WORKLOADS["embed_diag"]
    mix = datagen.planted(wl)
    keep, ptrs = datagen.upload_tables(mix, device=torch.device("cuda"))
    X = torch.empty(wl.N * wl.D, dtype=torch.float16, device="cuda")
    datagen.device_points(mix, 0, wl.N, X.data_ptr(), torch.cuda.current_stream().cuda_stream,
                          ptrs)
    theta = f32(datagen.init_params(mix))
    opts = datagen.em_opts(theta)
    state = make_state(wl)
    lse_before = None
    for it in range(2):
        got = gpu_step(state, X, theta, want_lse=True, opts=opts)
        assert got["status"] == 0
        rng = np.random.default_rng(11 + it)
        idx = np.sort(rng.choice(wl.N, 1500, replace=False))
        # include both slab edges and the last row
        idx = np.unique(np.concatenate([idx, [0, (1 << 21) - 1, 1 << 21, wl.N - 1]]))
        sample = datagen.points_at(mix, idx)
        st, L, _ = oracle.log_joint(sample, *(np.asarray(p, np.float64) for p in theta),
                                    wl.cov_type, xdtype=wl.dtype)
        assert st == 0
        m = L.max(axis=1)
        ref_lse = m + np.log(np.exp(L - m[:, None]).sum(axis=1))
        np.testing.assert_allclose(got["lse"][idx], ref_lse, rtol=1e-5, atol=2e-3)
        assert abs(got["ll"] - got["lse"].sum()) <= 1e-6 * abs(got["ll"]) + 1.0
        assert abs(got["pi"].sum() - 1.0) < 1e-5
        theta = f32((got["pi"], got["mu"], got["cov"]))
    del X, keep


def _per_step(wl, steps):
    """Per-step parity from theta_0 and from the oracle's next iterates, on
    points generated on the host (both sides read the same bits)."""
    mix = datagen.planted(wl)
    bits = datagen.points(mix, 0, wl.N)
    theta = f32(datagen.init_params(mix, bits))
    opts = datagen.em_opts(theta)
    Xd = to_device(bits, wl.dtype)
    state = make_state(wl)
    fails = []
    for t in range(steps):
        ref = oracle_step(bits, wl.dtype, theta, wl.cov_type, opts=opts)
        assert ref["status"] == 0
        got = gpu_step(state, Xd, theta, opts=opts)
        assert got["status"] == 0, got["status"]
        fails += parity.compare_step(got, ref, "%s N=%d step %d" % (wl.name, wl.N, t),
                                     opts["min_s0"])
        assert (got["flags"] == ref["flags"]).all(), (t, got["flags"], ref["flags"])
        theta = f32((ref["pi"], ref["mu"], ref["cov"]))
    if fails:
        fails.insert(0, "replay bundle: %s" % parity.replay_bundle(wl, bits, theta, fails))
    assert not fails, "\n".join(fails[:10])


def test_embed_diag_two_slabs():
    """10M-point workload's recipe at N = 2^21 + 4099: two screening slabs
    (the second ragged), statistics merged across slabs; steps 0 and 1."""
    _per_step(_workload("embed_diag", n=(1 << 21) + 4099), 2)


def test_large_diag_two_slabs_step0():
    """K = 1024, bf16 X, the streamed-parameter screen: step 0 from theta_0
    (dense responsibilities, most rows handed to the CUDA-core path) at
    N = 2^21 + 5, across two slabs."""
    _per_step(_workload("large_diag", n=(1 << 21) + 5), 1)


def test_full_cov_200k():
    """Full covariance at N = 200,000: steps 0 and 1."""
    _per_step(_workload("full_cov", n=200_000), 2)


def test_ivf_assign_full_size_sampled():
    """The assignment workload at full size (5e7 points, K = 4096, fp16,
    24 slabs) in the bench's launch configuration: every rank of the top-4
    and its gamma, and LSE_n, of 4000 sampled points (about 10% of them drawn
    as midpoints of two centres) against the oracle's log joints."""
    wl = datagen.WORKLOADS["ivf_assign"]
    mix = datagen.planted(wl)
    keep, ptrs = datagen.upload_tables(mix, device=torch.device("cuda"))
    X = torch.empty(wl.N * wl.D, dtype=torch.float16, device="cuda")
    datagen.device_points(mix, 0, wl.N, X.data_ptr(), torch.cuda.current_stream().cuda_stream,
                          ptrs)
    pi, mu, var = datagen.planted_params_f16(mix)
    from soft_clustering_gb300.torch_api import Assigner
    a = Assigner(wl.N, wl.D, wl.K, wl.cov_type, wl.dtype, wl.m)
    a.prepare(pi, mu, var)
    a.assign(X)
    assert a.device_status() == 0
    rng = np.random.default_rng(2024)
    idx = np.unique(np.concatenate([rng.choice(wl.N, 4000, replace=False),
                                    [0, (1 << 21) - 1, 1 << 21, wl.N - 1]]))
    it = torch.from_numpy(idx).cuda()
    ids = a.ids[it].cpu().numpy()
    gam = a.gamma[it].cpu().numpy().astype(np.float64)
    lse = a.lse[it].cpu().numpy().astype(np.float64)
    del X, keep
    sample = datagen.points_at(mix, idx)
    st, L, _ = oracle.log_joint(sample, pi, mu, var, wl.cov_type, xdtype=wl.dtype)
    assert st == 0
    m = L.max(axis=1)
    lse_ref = m + np.log(np.exp(L - m[:, None]).sum(axis=1))
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=2e-3)
    # boundary points are present: about 200 of the sample have a second
    # component within 40 nats of the best (73 with a share above 1e-3)
    srt = np.sort(L, axis=1)
    assert ((srt[:, -1] - srt[:, -2]) < 40).sum() >= 150
    fails = parity.topm_compare(ids, gam, L, lse_ref, "ivf full size")
    assert not fails, fails
