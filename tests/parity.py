"""Parity criteria for the CUDA path against the fp64 oracle.

Tolerances (fixed for this path):
  * log-likelihood: relative error <= 1e-4 per iteration;
  * updated means and covariance entries: |gpu - ref| / max(|ref|, 1e-3 * scale)
    <= 2e-3, scale = max |ref| over that parameter array;
  * weights: absolute error <= 1e-5;
  * top-1 assignment agreement >= 99.9%, points whose two best oracle
    responsibilities differ by less than 1e-6 excluded.
On failure the report gives the diagnostics the ops-debug page recommends
(sec. 3.2): cosine similarity, max abs error with its index and the
P50/P95/P99 of the relative error.
"""
from __future__ import annotations

import numpy as np

LL_RTOL = 1e-4
PARAM_RTOL = 2e-3
PARAM_FLOOR = 1e-3
PI_ATOL = 1e-5
TOP1_MIN = 0.999
TIE_EPS = 1e-6
# Top-m order: ranks whose oracle log joints lie within TOPM_TIE_NATS of a
# neighbouring rank are ties (either order is correct); every other rank's id
# must match the oracle's.
TOPM_TIE_NATS = 1e-4
# gamma of the top-m entries: |gpu - ref| <= GAMMA_ATOL.  gamma = exp(l - LSE)
# with l and LSE each within 1e-6 |l| of the fp64 values (|l| < 100 nats on
# these workloads) moves by at most 2e-4 gamma.
GAMMA_ATOL = 2e-4


def diagnostics(got, ref):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    err = np.abs(got - ref)
    i = int(np.argmax(err)) if err.size else 0
    rel = err / np.maximum(np.abs(ref), 1e-300)
    denom = np.linalg.norm(got) * np.linalg.norm(ref)
    cos = float(got @ ref / denom) if denom > 0 else float("nan")
    p = np.percentile(rel, [50, 95, 99]) if rel.size else [0, 0, 0]
    return dict(cosine=cos, max_abs=float(err[i]) if err.size else 0.0, argmax=i,
                got=float(got[i]) if err.size else 0.0, ref=float(ref[i]) if err.size else 0.0,
                p50=float(p[0]), p95=float(p[1]), p99=float(p[2]))


def scaled_rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    return np.abs(got - ref) / np.maximum(np.abs(ref), PARAM_FLOOR * scale + 1e-300)


def compare_step(gpu, ref, what="", min_s0=None, param_rtol=PARAM_RTOL, min_mass=None):
    """gpu/ref: dicts with pi, mu, cov, ll.  Returns a list of failure strings.
    With min_s0 (and ref['s0']), components whose oracle s0 lies within 1e-4
    (relative) of the empty threshold are left out of the mean/covariance
    check: there the empty-or-not decision rests on rounding."""
    fails = []
    keep = None
    if min_s0 is not None and "s0" in ref:
        s0 = np.asarray(ref["s0"])
        keep = np.abs(s0 - min_s0) > 1e-4 * max(min_s0, 1e-30)
        if min_mass is not None:
            keep &= s0 >= min_mass
    ll_err = abs(gpu["ll"] - ref["ll"]) / max(abs(ref["ll"]), 1e-300)
    if not ll_err <= LL_RTOL:
        fails.append("%s LL rel err %.3g (gpu %.10g ref %.10g)" % (what, ll_err, gpu["ll"], ref["ll"]))
    pe = np.abs(np.asarray(gpu["pi"]) - np.asarray(ref["pi"]))
    if not (pe <= PI_ATOL).all():
        fails.append("%s pi abs err %.3g at %d %s" % (what, pe.max(), int(pe.argmax()),
                                                     diagnostics(gpu["pi"], ref["pi"])))
    for name in ("mu", "cov"):
        e = scaled_rel_err(gpu[name], ref[name])
        if keep is not None:
            e = e * keep.reshape((-1,) + (1,) * (e.ndim - 1))
        if not (e <= param_rtol).all():
            idx = np.unravel_index(int(np.argmax(e)), e.shape)
            fails.append("%s %s scaled rel err %.3g at %s (gpu %.8g ref %.8g) %s" % (
                what, name, e.max(), idx, np.asarray(gpu[name])[idx], np.asarray(ref[name])[idx],
                diagnostics(gpu[name], ref[name])))
    return fails


def topm_compare(ids_gpu, gam_gpu, L_ref, lse_ref, what=""):
    """Every rank of the GPU's top-m against the oracle's log joints L_ref
    [n, K] (fp64) of the same points.  Rank t's id must equal the oracle's
    unless rank t's oracle value is within TOPM_TIE_NATS of rank t-1's or
    t+1's (a tie: either order is correct; then the GPU's id must still be a
    component whose value is within the tie band of rank t's, so the set is
    valid); gamma must be within GAMMA_ATOL of exp(L - LSE) of the GPU's id.
    Returns a list of failure strings."""
    ids_gpu = np.asarray(ids_gpu)
    gam_gpu = np.asarray(gam_gpu, dtype=np.float64)
    L = np.asarray(L_ref, dtype=np.float64)
    n, m = ids_gpu.shape
    order = np.lexsort((np.arange(L.shape[1])[None, :].repeat(n, 0), -L), axis=1)[:, :m]
    vals = np.take_along_axis(L, order, axis=1)
    tie = np.zeros((n, m), dtype=bool)
    gaps = vals[:, :-1] - vals[:, 1:]
    tie[:, :-1] |= gaps < TOPM_TIE_NATS
    tie[:, 1:] |= gaps < TOPM_TIE_NATS
    # the (m+1)-th value decides whether rank m-1 is tied with a component outside the list
    if L.shape[1] > m:
        nxt = np.sort(L, axis=1)[:, ::-1][:, m]
        tie[:, m - 1] |= (vals[:, m - 1] - nxt) < TOPM_TIE_NATS
    fails = []
    bad_id = (~tie) & (ids_gpu != order)
    if bad_id.any():
        i, t = np.argwhere(bad_id)[0]
        fails.append("%s top-m id mismatch at %d ranks (first: point %d rank %d gpu %d oracle %d, "
                     "oracle values %s)" % (what, int(bad_id.sum()), i, t, ids_gpu[i, t],
                                            order[i, t], vals[i]))
    valid = (ids_gpu >= 0) & (ids_gpu < L.shape[1])
    if not valid.all():
        fails.append("%s top-m: %d ids out of range" % (what, int((~valid).sum())))
        return fails
    got_vals = np.take_along_axis(L, ids_gpu, axis=1)
    band = np.abs(got_vals - vals) > TOPM_TIE_NATS
    if (tie & band).any():
        i, t = np.argwhere(tie & band)[0]
        fails.append("%s top-m tied rank holds a component outside the tie band (point %d rank %d)"
                     % (what, i, t))
    gref = np.exp(got_vals - np.asarray(lse_ref, dtype=np.float64)[:, None])
    ge = np.abs(gam_gpu - gref)
    if not (ge <= GAMMA_ATOL).all():
        i, t = np.unravel_index(int(np.argmax(ge)), ge.shape)
        fails.append("%s top-m gamma abs err %.3g at point %d rank %d (gpu %.8g ref %.8g)"
                     % (what, ge.max(), i, t, gam_gpu[i, t], gref[i, t]))
    return fails


def top1_agreement(ids_gpu, ids_ref, gamma_ref):
    """Fraction of non-tied points whose top-1 component agrees."""
    ids_gpu = np.asarray(ids_gpu)
    ids_ref = np.asarray(ids_ref)
    g = np.asarray(gamma_ref)
    if g.shape[1] >= 2:
        keep = (g[:, 0] - g[:, 1]) >= TIE_EPS
    else:
        keep = np.ones(len(g), dtype=bool)
    if not keep.any():
        return 1.0, 0
    agree = (ids_gpu[keep, 0] == ids_ref[keep, 0]).mean()
    return float(agree), int(keep.sum())


def replay_bundle(wl, bits, theta, fails, directory=None):
    """What reproduces a failed parity case (the ops-debug page, sec. 5.3):
    workload, seed, sizes and recipe, the SHA-256 of the input bits and of
    each parameter array as fp32, and the failures, as one JSON file in
    `directory` (else $GMM_REPLAY_DIR, else the temporary directory).
    Returns its path, or None if it could not be written: the failure itself
    is reported either way."""
    try:
        import hashlib
        import json
        import os
        import tempfile
        import time
        d = directory or os.environ.get("GMM_REPLAY_DIR") or tempfile.gettempdir()
        os.makedirs(d, exist_ok=True)

        def sha(a):
            return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()

        rec = dict(workload=wl.name, seed=int(wl.seed), N=int(wl.N), D=int(wl.D), K=int(wl.K),
                   x_dtype=int(wl.dtype), cov_type=int(wl.cov_type), kind=int(wl.kind),
                   recipe={k: float(v) for k, v in dict(wl.recipe).items()},
                   x_sha256=sha(bits),
                   params_sha256=[sha(np.asarray(p, dtype=np.float32)) for p in theta],
                   failures=[str(f) for f in list(fails)[:50]])
        path = os.path.join(d, "gmm_replay_%s_s%d_n%d_%d.json"
                            % (wl.name, wl.seed, wl.N, int(time.time() * 1e3)))
        with open(path, "w") as f:
            json.dump(rec, f, indent=1)
        return path
    except Exception:
        return None

