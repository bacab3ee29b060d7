"""A second, independent statement of the three chains in pure Python.

TEST INFRASTRUCTURE ONLY (pins the C oracle; never used by the product path).
It shares no code with ``fc_oracle.c``: different language, the library's
``math.erf`` / ``math.exp`` / ``math.log`` rather than C's, softplus written as
log(1 + e^z) directly (no max/log1p form), tanh of it via
(e^{2s} - 1) / (e^{2s} + 1), and sums via ``math.fsum`` (exactly rounded).
Only for tiny inputs: every loop is explicit.
"""
from __future__ import annotations

import math


def gelu(v):
    return 0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0)))


def _softplus(z):
    if z > 40.0:               # log(1 + e^z) = z + log(1 + e^-z) = z to double precision
        return z
    return math.log(1.0 + math.exp(z)) if z > -30.0 else math.exp(z)


def _tanh_pos(s):
    # s = softplus(z) > 0; tanh(s) = (e^{2s} - 1) / (e^{2s} + 1)
    if s > 20.0:
        return 1.0
    e = math.exp(2.0 * s)
    return (e - 1.0) / (e + 1.0) if s > 1e-3 else math.tanh(s)


def mish(z):
    return z * _tanh_pos(_softplus(z))


def gelu_tanh(v):
    # 0.5 v (1 + tanh(u)) written as the logistic v / (1 + e^{-2u}), u = sqrt(2/pi) (v + 0.044715 v^3)
    u = math.sqrt(2.0 / math.pi) * (v + 0.044715 * v ** 3)
    if -2.0 * u > 700.0:
        return 0.0 * v
    return v / (1.0 + math.exp(-2.0 * u))


ACTS = {"gelu": gelu, "mish": mish, "mish_mish": lambda v: mish(mish(v)), "gelu_tanh": gelu_tanh,
        "none": lambda v: v}


def zero_pad(x, pad):
    """x [N][C][H][W] nested lists -> [N][C][H+2p][W+2p] with p zero rows / columns on every side."""
    out = []
    for img in x:
        planes = []
        for plane in img:
            Wp = len(plane[0]) + 2 * pad
            rows = [[0.0] * Wp for _ in range(pad)]
            rows += [[0.0] * pad + list(r) + [0.0] * pad for r in plane]
            rows += [[0.0] * Wp for _ in range(pad)]
            planes.append(rows)
        out.append(planes)
    return out


def conv3x3(x, w, b, pad=0):
    """x: nested lists [N][Cin][H][W]; w: [Cout][Cin][3][3]; b: [Cout] -> [N][Cout][H+2p-2][W+2p-2],
    padding p taken as an explicitly zero-extended input."""
    if pad:
        x = zero_pad(x, pad)
    N, Cin, H, W = len(x), len(x[0]), len(x[0][0]), len(x[0][0][0])
    Cout = len(w)
    out = []
    for n in range(N):
        planes = []
        for co in range(Cout):
            rows = []
            for oh in range(H - 2):
                row = []
                for ow in range(W - 2):
                    terms = [b[co]]
                    for ci in range(Cin):
                        for kh in range(3):
                            for kw in range(3):
                                terms.append(x[n][ci][oh + kh][ow + kw] * w[co][ci][kh][kw])
                    row.append(math.fsum(terms))
                rows.append(row)
            planes.append(rows)
        out.append(planes)
    return out


def conv3x3_act(x, w, b, act, pad=0):
    f = ACTS[act]
    return [[[[f(v) for v in row] for row in plane] for plane in img] for img in conv3x3(x, w, b, pad)]


def conv3x3_act_pool(x, w, b, act, pad=0):
    out = []
    for img in conv3x3_act(x, w, b, act, pad):
        out.append([math.fsum(v for row in plane for v in row) / (len(plane) * len(plane[0]))
                    for plane in img])
    return out


def logsumexp(t):
    m = max(t)
    return m + math.log(math.fsum(math.exp(v - m) for v in t))


def linear_lse_mish(x, Wt, b, scale, lo, hi):
    """x: [M][K]; Wt: [Nout][K]; b: [Nout] -> (y[M], lse[M])."""
    ys, ls = [], []
    for xr in x:
        t = []
        for j, wr in enumerate(Wt):
            v = math.fsum([b[j]] + [xk * wk for xk, wk in zip(xr, wr)])
            v = v * scale
            v = v + v
            t.append(min(max(v, lo), hi))
        lse = logsumexp(t)
        ls.append(lse)
        ys.append(lse * mish(lse))
    return ys, ls
