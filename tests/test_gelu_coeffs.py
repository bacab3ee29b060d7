"""The erf-GELU polynomial the kernels hold is the one its generator fits, and that fit meets
the accuracy the kernels rely on (CPU only)."""
import importlib.util
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gemm_activation_reduction_gb300")


def _kernel_coeffs():
    src = open(os.path.join(PKG, "csrc", "fc_act.cuh")).read()
    return np.array([float(re.search(rf"kGeluP{k} = ([-+0-9.eE]+)f;", src).group(1)) for k in range(6)], np.float32)


def test_kernel_constants_are_the_generated_fit():
    pytest.importorskip("scipy")
    spec = importlib.util.spec_from_file_location("gen_gelu_coeffs", os.path.join(PKG, "gen_gelu_coeffs.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    np.testing.assert_array_equal(gen.fit(), _kernel_coeffs())


def test_polynomial_form_matches_exact_gelu_in_an_fp32_model():
    """2 GELU(z) = z + |z| - |z| 2^P(|z|), evaluated with fp32 roundings (exact exponential),
    against 0.5 z (1 + erf(z / sqrt 2)) from math.erf: within 5e-7 (absolute, or relative above 1)
    on [-14, 14]; far out (to 1e12) P stays below -80, so 2^P vanishes and the result is max(z, 0);
    the padding pre-activation -1e4 gives exactly 0."""
    c = _kernel_coeffs()
    z = np.concatenate([np.linspace(-14, 14, 28001), -np.logspace(1, 12, 500), np.logspace(1, 12, 500),
                        [-1e4]]).astype(np.float32)
    a = np.abs(z)
    p = np.full_like(a, c[5])
    with np.errstate(over="ignore", invalid="ignore"):
        for k in range(4, -1, -1):
            p = (p.astype(np.float64) * a + c[k]).astype(np.float32)
    assert c[5] < 0 and np.all(p[a > 10] < -80)
    e = np.exp2(p.astype(np.float64)).astype(np.float32)
    two_g = ((z + a).astype(np.float64) - a.astype(np.float64) * e).astype(np.float32)
    got = 0.5 * two_g.astype(np.float64)
    assert np.all(np.isfinite(got))
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in z.astype(np.float64)])
    err = np.abs(got - exact) / np.maximum(1.0, np.abs(exact))
    assert err.max() < 5e-7, (err.max(), z[np.argmax(err)])
    assert got[z == -1e4][0] == 0.0
