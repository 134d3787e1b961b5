"""The C-ABI library loads and exports every symbol include/gmm.h declares;
host-side argument checks (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

import soft_clustering_gb300 as G

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(gmm_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from soft_clustering_gb300 import build
    build.build()
    return G.lib()


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) <= set(G.EXPORTS) | {"gmm_default_opts"}


def test_default_opts_and_strings(lib):
    o = G.gmm_default_opts()
    assert o.ridge_rel == 0.0 and o.var_floor == 0.0 and o.min_s0 == 0.5
    assert G.status_string(G.GMM_ERR_NOT_PD) == "GMM_ERR_NOT_PD"


def test_sizes(lib):
    assert G.gmm_workspace_bytes(1000, 48, 4, G.GMM_COV_DIAG, G.GMM_F16) == 0  # unsupported D
    assert G.gmm_workspace_bytes(0, 64, 4, G.GMM_COV_DIAG, G.GMM_F16) == 0
    assert G.gmm_prepared_bytes(64, 16, G.GMM_COV_FULL) >= 16 * 64 * 64 * 4
    # the workspace never holds an N x K matrix: it grows like N + K*D
    for N, D, K, cov in [(10_000_000, 128, 256, G.GMM_COV_DIAG),
                         (200_000_000, 128, 1024, G.GMM_COV_DIAG),
                         (1_000_000, 64, 16, G.GMM_COV_FULL)]:
        ws = G.gmm_workspace_bytes(N, D, K, cov, G.GMM_F16)
        assert 0 < ws < N * K * 4 / 2, (N, K, ws)
        ws2 = G.gmm_workspace_bytes(2 * N, D, K, cov, G.GMM_F16)
        assert ws2 - ws <= 16 * N + 4096  # only O(N) terms grow with N


def test_invalid_args_are_synchronous(lib):
    # null pointers / bad sizes are rejected before anything is queued
    p = G.make_params(None, None, None)
    o = G.gmm_default_opts()
    st = lib.gmm_em_step(None, G.GMM_F16, 100, 64, 4, ctypes.byref(p), G.GMM_COV_DIAG,
                         ctypes.byref(o), None, 0, None, None, None, None)
    assert st == G.GMM_ERR_INVALID_ARG
    st = lib.gmm_em_step(16, G.GMM_F16, 100, 48, 4, ctypes.byref(p), G.GMM_COV_DIAG,
                         ctypes.byref(o), None, 0, None, None, None, None)
    assert st == G.GMM_ERR_UNSUPPORTED
    st = lib.gmm_assign_topm(16, G.GMM_F16, 100, 64, 4, 256, G.GMM_COV_DIAG, 9, 16, 16, None,
                             256, 256, None)
    assert st == G.GMM_ERR_INVALID_ARG  # m > 8
    st = lib.gmm_prepare(None, 64, 4, G.GMM_COV_DIAG, None, None, None, None)
    assert st == G.GMM_ERR_INVALID_ARG


def test_empty_and_degenerate_sizes_are_rejected(lib):
    """N = 0 (no points), K = 0 (no components) and D = 0 are argument errors,
    returned before anything is queued; the size queries answer 0."""
    p = G.make_params(16, 16, 16)
    o = G.gmm_default_opts()
    for N, D, K in [(0, 64, 4), (-1, 64, 4), (100, 64, 0), (100, 0, 4)]:
        st = lib.gmm_em_step(16, G.GMM_F16, N, D, K, ctypes.byref(p), G.GMM_COV_DIAG,
                             ctypes.byref(o), 256, 1 << 20, 16, None, None, None)
        assert st == G.GMM_ERR_INVALID_ARG, (N, D, K, st)
        st = lib.gmm_assign_topm(16, G.GMM_F16, N, D, K, 256, G.GMM_COV_DIAG, 1, 16, 16, None,
                                 256, 1 << 20, None)
        assert st == G.GMM_ERR_INVALID_ARG, (N, D, K, st)
        st = lib.gmm_em_step_noalloc(16, G.GMM_F16, N, D, K, ctypes.byref(p), G.GMM_COV_DIAG,
                                     ctypes.byref(o), 16, 16, None, None)
        assert st == G.GMM_ERR_INVALID_ARG, (N, D, K, st)
        assert G.gmm_workspace_bytes(N, D, K, G.GMM_COV_DIAG, G.GMM_F16) == 0
    assert G.gmm_prepared_bytes(64, 0, G.GMM_COV_DIAG) == 0


def test_host_streaming_workspace_is_bounded_by_the_chunk(lib):
    """gmm_em_step_host keeps only a chunk of rows on the device: its
    workspace does not grow with N, so a data set need not fit in HBM."""
    for D, K, cov in [(128, 1024, G.GMM_COV_DIAG), (64, 16, G.GMM_COV_FULL)]:
        chunk = 1 << 20
        small = G.gmm_workspace_bytes_host(chunk, D, K, cov, G.GMM_BF16, chunk)
        huge = G.gmm_workspace_bytes_host(10 ** 10, D, K, cov, G.GMM_BF16, chunk)  # 2.5 TB of X at D=128
        assert 0 < small == huge, (small, huge)
        assert huge < 8 << 30  # a few GiB for 2.5 TB of X
        assert G.gmm_workspace_bytes_host(10 ** 10, D, K, cov, G.GMM_BF16, 2 * chunk) > huge

