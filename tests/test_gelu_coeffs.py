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
    return np.array([float(re.search(rf"kGeluP{k} = ([-+0-9.eE]+)f;", src).group(1)) for k in range(7)], np.float32)


def test_kernel_constants_are_the_generated_fit():
    pytest.importorskip("scipy")
    spec = importlib.util.spec_from_file_location("gen_gelu_coeffs", os.path.join(PKG, "gen_gelu_coeffs.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    np.testing.assert_array_equal(gen.fit(), _kernel_coeffs())


def test_polynomial_form_matches_exact_gelu_in_an_fp32_model():
    """2 GELU(z) = z + |z| - |z| 2^P(min(|z|, 10)), evaluated with fp32 roundings (exact exponential),
    against 0.5 z (1 + erf(z / sqrt 2)) from math.erf: within 2e-7 (absolute, or relative above 1),
    and the padding pre-activation -1e4 contributes below 1e-15."""
    c = _kernel_coeffs()
    z = np.concatenate([np.linspace(-14, 14, 28001), [-1e4, -80.0, 80.0, 1e4]]).astype(np.float32)
    a = np.abs(z)
    ac = np.minimum(a, np.float32(10))
    p = np.full_like(ac, c[6])
    for k in range(5, -1, -1):
        p = (p.astype(np.float64) * ac + c[k]).astype(np.float32)
    e = np.exp2(p.astype(np.float64)).astype(np.float32)
    two_g = ((z + a).astype(np.float64) - a.astype(np.float64) * e).astype(np.float32)
    got = 0.5 * two_g.astype(np.float64)
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in z.astype(np.float64)])
    err = np.abs(got - exact) / np.maximum(1.0, np.abs(exact))
    assert err.max() < 2e-7, (err.max(), z[np.argmax(err)])
    assert abs(got[z == -1e4][0]) < 1e-15
