"""EM iterations until convergence, with per-iteration metrics.

`run_em` drives any step function: it queues an iteration, reads the
log-likelihood that iteration computed (at its input parameters, so the value
read after iteration t belongs to theta_t), and stops when the relative rise
falls to `tol` or after `max_iters` iterations (the Flash-GMM summary,
Method: iterate until the log-likelihood converges).  For every iteration it
records the log-likelihood, its change, whether the sequence is still
non-decreasing (EM's own guarantee, up to fp32 rounding of the step), the
count of components per flag, and the wall time; `log` receives each record
(for example `jsonl_writer`).  No arithmetic of the method happens here.
"""
from __future__ import annotations

import json
import time

FLAG_NAMES = {1: "ridge", 2: "not_pd", 4: "floor", 8: "empty"}


def flag_counts(flags):
    """Components per flag bit (ridge / not_pd / floor / empty)."""
    out = {name: 0 for name in FLAG_NAMES.values()}
    for f in flags:
        f = int(f)
        for bit, name in FLAG_NAMES.items():
            if f & bit:
                out[name] += 1
    return out


def run_em(step, read_ll, max_iters, tol=0.0, read_flags=None, log=None, rise_slack=1e-6):
    """Iterate `step()` up to max_iters times.

    step():       queue one EM iteration (parameters updated in place);
    read_ll():    the log-likelihood the last step computed, at its input
                  parameters (waits for it);
    read_flags(): optional, the per-component flag words of the last step;
    tol:          stop once |LL_t - LL_{t-1}| <= tol |LL_t| (0: run all);
    rise_slack:   a fall of at most rise_slack |LL| still counts as monotone
                  (fp32 rounding of the statistics).
    Returns dict(iterations, ll_history, converged, monotone, records)."""
    hist, records = [], []
    monotone, converged = True, False
    for t in range(int(max_iters)):
        t0 = time.perf_counter()
        step()
        ll = float(read_ll())
        dt = time.perf_counter() - t0
        delta = ll - hist[-1] if hist else None
        if delta is not None and delta < -rise_slack * abs(ll):
            monotone = False
        hist.append(ll)
        rec = dict(iter=t, loglik=ll, delta=delta, monotone=monotone, ms=dt * 1e3)
        if read_flags is not None:
            rec["flags"] = flag_counts(read_flags())
        records.append(rec)
        if log is not None:
            log(rec)
        if tol > 0 and delta is not None and abs(delta) <= tol * abs(ll):
            converged = True
            break
    return dict(iterations=len(hist), ll_history=hist, converged=converged, monotone=monotone,
                records=records)


def jsonl_writer(f):
    """A `log` callback writing one JSON object per line to the file object f."""
    def write(rec):
        f.write(json.dumps(rec) + "\n")
        f.flush()
    return write


def table(records):
    """The records as a terse text table."""
    lines = ["%5s %22s %14s %4s %9s" % ("iter", "loglik", "delta", "mono", "ms")]
    for r in records:
        d = "" if r["delta"] is None else "%.6g" % r["delta"]
        lines.append("%5d %22.12g %14s %4s %9.3f" % (r["iter"], r["loglik"], d,
                                                      "yes" if r["monotone"] else "NO", r["ms"]))
    return "\n".join(lines)
