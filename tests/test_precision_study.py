"""The fp16-operator precision study (a CPU report built on the oracle):
the effects the "low-precision GMM operator" notes describe, in direction
and order of magnitude, on reduced sizes so the check runs in seconds."""
from oracle import precision_study as ps


def test_inverse_route_loses_an_order_to_cholesky_in_fp16():
    r = ps.mahalanobis_routes(seed=1, K=4, n=64)
    assert r["inverse_fp32"] < 2e-5 and r["cholesky_fp32"] < 2e-6
    assert r["inverse_fp16"] > 1e-3
    assert r["inverse_fp16"] > 5 * r["cholesky_fp16"]
    assert r["cholesky_fp16"] < 3e-3


def test_ridge_repairs_failed_fp16_factorisations():
    near = ps.ridge_effect(seed=0, n_per=100)
    assert near["ridge 0"][1] >= 1                      # some fp16 factorisation fails
    assert near["ridge 0.0005"][1] == 0 and near["ridge 0.001"][1] == 0
    assert near["ridge 0.0005"][0] < near["ridge 0"][0] / 10
    well = ps.ridge_effect(seed=0, n_per=100, rank=24, diag=1e-2)
    assert well["ridge 0"][1] == 0
    # with nothing to repair the ridge only adds its bias
    assert well["ridge 0"][0] <= well["ridge 0.0005"][0] <= well["ridge 0.001"][0]
