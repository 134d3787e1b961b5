"""The EM driver's host logic (stop rule, monotonicity, flag counts, logs),
driven by the oracle's step so that no GPU is needed."""
import io
import json

import numpy as np

import datagen
import oracle
from soft_clustering_gb300 import em_loop


class OracleStep:
    """A step function with the library's conventions: parameters updated in
    place (fp32), the log-likelihood at the step's input parameters."""

    def __init__(self, name, n=None):
        wl = datagen.WORKLOADS[name]
        self.wl = wl.with_n(n) if n else wl
        mix = datagen.planted(self.wl)
        self.bits = datagen.points(mix, 0, self.wl.N)
        self.theta = tuple(np.asarray(p, np.float32) for p in datagen.init_params(mix, self.bits))
        self.opts = datagen.em_opts(self.theta)
        self.ll = None
        self.flags = None

    def __call__(self):
        r = oracle.em_step(self.bits, *(np.asarray(p, np.float64) for p in self.theta),
                           self.wl.cov_type, xdtype=self.wl.dtype, opts=self.opts)
        assert r["status"] == 0
        self.theta = tuple(np.asarray(r[k], np.float32) for k in ("pi", "mu", "cov"))
        self.ll, self.flags = r["ll"], r["flags"]


def test_runs_to_convergence_and_logs_every_iteration():
    s = OracleStep("tiny_diag")
    buf = io.StringIO()
    out = em_loop.run_em(s, lambda: s.ll, 200, tol=1e-6, read_flags=lambda: s.flags,
                         log=em_loop.jsonl_writer(buf))
    assert out["converged"] and out["monotone"] and 2 <= out["iterations"] < 200
    lines = [json.loads(l) for l in buf.getvalue().splitlines()]
    assert [r["iter"] for r in lines] == list(range(out["iterations"]))
    assert [r["loglik"] for r in lines] == out["ll_history"]
    last = out["ll_history"]
    assert abs(last[-1] - last[-2]) <= 1e-6 * abs(last[-1])
    assert all(abs(last[i] - last[i - 1]) > 1e-6 * abs(last[i]) for i in range(1, len(last) - 1))
    assert set(lines[0]["flags"]) == {"ridge", "not_pd", "floor", "empty"}
    assert "loglik" in em_loop.table(out["records"]).splitlines()[0]


def test_tol_zero_runs_every_iteration():
    s = OracleStep("full_cov", n=2000)
    out = em_loop.run_em(s, lambda: s.ll, 4)
    assert out["iterations"] == 4 and not out["converged"] and out["monotone"]


def test_a_falling_loglik_is_reported():
    seq = iter([-100.0, -90.0, -95.0, -80.0])
    cur = {}
    out = em_loop.run_em(lambda: cur.__setitem__("ll", next(seq)), lambda: cur["ll"], 4)
    assert not out["monotone"] and [r["monotone"] for r in out["records"]] == [True, True,
                                                                                False, False]


def test_flag_counts():
    assert em_loop.flag_counts([0, 1, 8, 12, 2]) == dict(ridge=1, not_pd=1, floor=1, empty=2)
