"""Generate the coefficients of the erf-GELU evaluation in csrc/fc_act.cuh.

The kernels evaluate the exact GELU as

    2 GELU(z) = z + |z| - |z| * erfc(|z| / sqrt 2)                          (1)

(from GELU(z) = z Phi(z), Phi(z) = erfc(-z / sqrt 2) / 2 and erfc(-x) = 2 - erfc(x)), with

    erfc(a / sqrt 2) = 2^P(min(a, A_MAX)),   a = |z|,                        (2)

P a polynomial of degree DEG.  P is log2 erfc(a / sqrt 2), fitted on [0, A_MAX] by
weighted least squares, iteratively reweighted toward the minimax solution of the error
in (1): each pass weights the residual of log erfc by a * erfc(a / sqrt 2) (the error it
causes in GELU) times the square root of the previous pass's relative error.  Beyond
A_MAX, erfc(a / sqrt 2) < 2^-74 and the clamped term is far below fp32 resolution even for
the pre-activation -1e4 that marks padding pixels.

Needs numpy and scipy (scipy.special.log_ndtr for log Phi).  Run it to reprint the
constants; the kernels hold the printed values.
"""
import numpy as np
from scipy.special import log_ndtr

DEG = 6
A_MAX = 10.0


def fit(deg=DEG, a_max=A_MAX, passes=40, points=80001):
    a = np.linspace(0.0, a_max, points)
    ln_erfc = np.log(2.0) + log_ndtr(-a)            # ln erfc(a / sqrt 2) = ln 2 Phi(-a)
    err_weight = a * np.exp(ln_erfc) + 1e-3 * np.exp(ln_erfc) + 1e-9
    extra = np.ones_like(a)
    V = np.vander(a, deg + 1, increasing=True)
    for _ in range(passes):
        w = err_weight * extra
        c, *_ = np.linalg.lstsq(V * w[:, None], ln_erfc * w, rcond=None)
        r = np.abs((V @ c - ln_erfc) * err_weight)
        extra *= np.sqrt(r / r.max()) + 1e-3
    return (c / np.log(2.0)).astype(np.float32)   # log2 erfc(a / sqrt 2)


def main():
    p = fit()
    print(f"// P(a), a in [0, {A_MAX:g}], degree {DEG}: coefficients of a^0 .. a^{DEG}")
    for k, v in enumerate(p):
        print(f"constexpr float kGeluP{k} = {float(v)!r}f;")


if __name__ == "__main__":
    main()
