"""The error bound of the tensor-core screen, checked on the CPU.

The screen evaluates the diagonal log joint in its expanded form,
    l_k = sum_j a_j b_kj + bias_k,   a = [x, x^2],  b_k = [mu w, -w / 2],
    bias_k = log pi_k - 1/2 log|Sigma_k| - D/2 log 2pi - 1/2 sum mu^2 w,
with a and b_k / S rounded to fp16 (S a power of two per chunk) and the
products summed in fp32 in an order the hardware chooses.  Its claim: the
screened value differs from the exact log joint by at most
    kappa |a| |b_k| + 2^-20 S |a| + 1e-3 + 1e-6 |bias_k|,   kappa = 1.5e-3 + 2e-6,
(fp16 rounding of both operands 3 x 2^-11 |a_j b_j|, summed by Cauchy-Schwarz;
the fp32 accumulation; operands the common scale leaves fp16-subnormal, each
off by at most 2^-25 S; the 1e-3 + 1e-6 |bias| gap to the exact fp32 centred
form the refine computes).  This test restates that arithmetic with numpy's
fp16 rounding and fp32 sums in random orders, on draws chosen to stress it:
tight clusters far from the origin (terms of ~1e4 cancelling to ~1e2), wide
spreads of sigma within a chunk, and scales that push operands subnormal.
"""
import numpy as np
import pytest

KAPPA = 1.5e-3 + 2e-6


def _chunk_scale(b):
    """The smallest power of two with max |b| / S <= 2^14."""
    m = np.abs(b).max()
    return 2.0 ** (int(np.ceil(np.log2(m))) - 14) if m > 0 else 1.0


def _screen(x16, b, S, rng):
    """Screened log joint minus bias: fp16 operands, fp32 sum in a random order."""
    a = np.concatenate([x16.astype(np.float32),
                        (x16.astype(np.float32) * x16.astype(np.float32)).astype(np.float16)
                        .astype(np.float32)])
    bh = (b / S).astype(np.float16).astype(np.float32)
    terms = a * bh
    acc = np.float32(0.0)
    for t in terms[rng.permutation(terms.size)]:
        acc = np.float32(acc + t)
    return float(acc) * S


@pytest.mark.parametrize("case", ["tight_far", "wide_spread", "subnormal_operands"])
def test_screen_error_within_bound(case):
    rng = np.random.default_rng({"tight_far": 1, "wide_spread": 2, "subnormal_operands": 3}[case])
    D, K, n = 128, 16, 40
    if case == "tight_far":
        mu = rng.normal(0.0, 3.0, (K, D))
        var = np.full((K, D), 0.1 ** 2) * rng.uniform(0.8, 1.2, (K, D))
    elif case == "wide_spread":
        mu = rng.normal(0.0, 1.0, (K, D))
        var = (np.exp(rng.uniform(np.log(0.05), np.log(1.0), (K, 1))) ** 2 *
               rng.uniform(0.6, 1.6, (K, D)))
    else:
        mu = rng.normal(0.0, 0.3, (K, D))
        var = rng.uniform(0.5, 1.5, (K, D))
        mu[0] = 300.0   # sets the chunk's scale: the other operands shrink toward subnormal
    w = 1.0 / var
    b = np.concatenate([mu * w, -0.5 * w], axis=1)          # [K, 2D]
    S = _chunk_scale(b)
    logpi = np.log(np.full(K, 1.0 / K))
    c = logpi - 0.5 * np.log(var).sum(1) - 0.5 * D * np.log(2 * np.pi)
    bias = c - 0.5 * (mu * mu * w).sum(1)
    worst = 0.0
    for i in range(n):
        # points of the far component in the subnormal case have x^2 beyond
        # fp16: the screen hands such rows to the CUDA-core path
        k0 = rng.integers(1 if case == "subnormal_operands" else 0, K)
        x = mu[k0] + rng.standard_normal(D) * np.sqrt(var[k0]) * rng.choice([1.0, 3.0, 10.0])
        x16 = x.astype(np.float16)
        xe = x16.astype(np.float64)
        a = np.concatenate([xe, xe * xe])
        for k in range(K):
            exact = c[k] - 0.5 * (w[k] * (xe - mu[k]) ** 2).sum()
            got = _screen(x16, b[k], S, rng) + bias[k]
            na, nb = np.linalg.norm(a), np.linalg.norm(b[k])
            bound = KAPPA * na * nb + 2.0 ** -20 * S * na + 1e-3 + 1e-6 * abs(bias[k])
            err = abs(got - exact)
            assert err <= bound, (case, i, k, err, bound)
            worst = max(worst, err / bound)
    print(case, "largest error / bound: %.3g" % worst)

