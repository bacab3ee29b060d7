"""Generate the coefficients of the erf-GELU evaluation in csrc/fc_act.cuh.

The kernels evaluate the exact GELU as

    2 GELU(z) = z + |z| - |z| * erfc(|z| / sqrt 2)                          (1)

(from GELU(z) = z Phi(z), Phi(z) = erfc(-z / sqrt 2) / 2 and erfc(-x) = 2 - erfc(x)), with

    erfc(a / sqrt 2) = 2^P(a),   a = |z|,                                    (2)

P a polynomial of degree DEG.  P is log2 erfc(a / sqrt 2), fitted on [0, A_FIT] by weighted
least squares, iteratively reweighted toward the minimax solution of the error in (1): each
pass weights the residual of log erfc by a * erfc(a / sqrt 2) (the error it causes in GELU)
times the previous pass's relative error to the power POWER.  P is used without a clamp: its
leading coefficient is negative and P stays below -85 for every a > 10 (checked here up to
1e12), so 2^P vanishes there; the padding pre-activation -1e4 gives exactly 0 in fp32.

Needs numpy and scipy (scipy.special.log_ndtr for log Phi).  Run it to reprint the
constants; the kernels hold the printed values.
"""
import numpy as np
from scipy.special import log_ndtr

DEG = 5
A_FIT = 7.0
POWER = 0.7


def fit(deg=DEG, a_fit=A_FIT, power=POWER, passes=40, points=80001):
    a = np.linspace(0.0, a_fit, points)
    ln_erfc = np.log(2.0) + log_ndtr(-a)            # ln erfc(a / sqrt 2) = ln 2 Phi(-a)
    err_weight = a * np.exp(ln_erfc) + 1e-3 * np.exp(ln_erfc) + 1e-9
    extra = np.ones_like(a)
    V = np.vander(a, deg + 1, increasing=True)
    for _ in range(passes):
        w = err_weight * extra
        c, *_ = np.linalg.lstsq(V * w[:, None], ln_erfc * w, rcond=None)
        r = np.abs((V @ c - ln_erfc) * err_weight)
        extra *= (r / r.max()) ** power + 1e-3
    return (c / np.log(2.0)).astype(np.float32)   # log2 erfc(a / sqrt 2)


def tail_max(p):
    """The largest P(a) over a in (10, 1e12], evaluated in fp32 like the kernels."""
    a = np.logspace(1, 12, 20001).astype(np.float32)
    r = np.full_like(a, p[-1])
    with np.errstate(over="ignore", invalid="ignore"):
        for k in range(len(p) - 2, -1, -1):
            r = (r.astype(np.float64) * a + p[k]).astype(np.float32)
    return float(r.max())


def main():
    p = fit()
    assert p[-1] < 0 and tail_max(p) < -80, "P must decay past the fitted range"
    print(f"// P(a), fitted on [0, {A_FIT:g}], degree {DEG}: coefficients of a^0 .. a^{DEG}")
    for k, v in enumerate(p):
        print(f"constexpr float kGeluP{k} = {float(v)!r}f;")


if __name__ == "__main__":
    main()
