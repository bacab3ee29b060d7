"""The oracle's pins reject plausible slips (CPU only).

Each test builds a mutant -- the oracle with one plausible mistake planted around it (a
flipped kernel, a transposed weight, the doubling applied once, the clamp after the
logsumexp, the wrong pool divisor, the pool and the activation swapped, the tail missing
its factor, the tanh GELU for the erf one) -- and shows that the pinned fact the pin tests
check holds for the oracle and fails for the mutant.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute
import fc_inputs


def _tolist(a):
    return np.asarray(a, dtype=np.float64).tolist()


def test_flipped_kernel_fails_the_delta_crop_pin():
    """A true convolution (kernel flipped) instead of cross-correlation."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 2, 7, 9)).astype(np.float32)
    w = np.zeros((3, 2, 3, 3), np.float32)
    w[:, 1, 0, 2] = 1.0
    b = np.zeros(3, np.float32)
    crop = x[:, 1, 0:5, 2:9].astype(np.float64)
    good = oracle.conv3x3_preact(x, w, b)
    mutant = oracle.conv3x3_preact(x, np.ascontiguousarray(w[:, :, ::-1, ::-1]), b)
    assert np.array_equal(good[:, 0], crop)
    assert not np.allclose(mutant[:, 0], crop)


def test_transposed_weight_fails_the_brute_force_pin():
    """x W instead of x W^T (square W, so both run)."""
    d = fc_inputs.linear_inputs(3, 6, 6, seeds=(61, 62, 63))
    ys, _ = brute.linear_lse_mish(_tolist(d["x"]), _tolist(d["W"]), _tolist(d["b"]), 2.0, -10.0, 10.0)
    good = oracle.linear_lse_mish(d["x"], d["W"], d["b"])
    mutant = oracle.linear_lse_mish(d["x"], np.ascontiguousarray(d["W"].T), d["b"])
    np.testing.assert_allclose(good.reshape(-1), ys, rtol=1e-12, atol=1e-13)
    assert not np.allclose(mutant.reshape(-1), ys, rtol=1e-6)


def test_doubling_applied_once_fails_the_zero_weight_closed_form():
    """t * scale without the following x + x: the closed form l = clamp(4c) + ln Nout breaks."""
    M, K, Nout = 2, 8, 4096
    x = np.random.default_rng(3).standard_normal((M, K)).astype(np.float32)
    b = np.full(Nout, 0.5, np.float32)
    expect = 2.0 + math.log(Nout)
    _, l = oracle.linear_lse_mish(x, np.zeros((Nout, K), np.float32), b, return_lse=True)
    _, l_m = oracle.linear_lse_mish(x, np.zeros((Nout, K), np.float32), b, scale=1.0, return_lse=True)
    np.testing.assert_allclose(l, expect, atol=1e-12)
    assert np.all(np.abs(l_m - expect) > 0.5)


def test_clamp_after_the_logsumexp_fails_the_bounds_pin():
    """clamp(LSE(u)) instead of LSE(clamp(u)): with every logit at 12 the pinned value is
    10 + ln Nout (about 19.01), the mutant's 10."""
    M, K, Nout = 1, 4, 8192
    x = np.zeros((M, K), np.float32)
    b = np.full(Nout, 3.0, np.float32)
    _, l = oracle.linear_lse_mish(x, np.zeros((Nout, K), np.float32), b, return_lse=True)
    # the mutant: LSE of the unclamped 4t, then the clamp
    _, l_free = oracle.linear_lse_mish(x, np.zeros((Nout, K), np.float32), b, clamp_lo=-1e30, clamp_hi=1e30,
                                       return_lse=True)
    l_m = np.clip(l_free, -10.0, 10.0)
    np.testing.assert_allclose(l, 10.0 + math.log(Nout), atol=1e-12)
    assert np.all(np.abs(l_m - (10.0 + math.log(Nout))) > 9.0)


def test_wrong_pool_divisor_fails_the_zero_weight_pool_pin():
    """Dividing by H W (the input plane) instead of (H - 2)(W - 2) (the output plane)."""
    N, Cin, H, W, Cout = 2, 3, 9, 11, 4
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, seeds=(31, 32, 33))
    y = oracle.conv3x3_act_pool(d["x"], np.zeros_like(d["w"]), d["b"], "gelu")
    y_m = y * ((H - 2) * (W - 2)) / (H * W)
    expect = np.array([oracle.gelu(float(v)) for v in d["b"]])
    np.testing.assert_allclose(y, np.broadcast_to(expect, y.shape), rtol=1e-14)
    assert not np.allclose(y_m, np.broadcast_to(expect, y.shape), rtol=1e-3)


def test_activation_of_the_mean_fails_the_brute_force_pin():
    """act(mean(v)) instead of mean(act(v))."""
    d = fc_inputs.conv_inputs(1, 2, 6, 7, 3, seeds=(21, 22, 23))
    ref = np.asarray(brute.conv3x3_act_pool(_tolist(d["x"]), _tolist(d["w"]), _tolist(d["b"]), "gelu"))
    pre = oracle.conv3x3_preact(d["x"], d["w"], d["b"])
    mutant = np.array([[oracle.gelu(float(pre[n, c].mean())) for c in range(3)] for n in range(1)])
    np.testing.assert_allclose(oracle.conv3x3_act_pool(d["x"], d["w"], d["b"], "gelu"), ref, rtol=1e-12, atol=1e-14)
    assert not np.allclose(mutant, ref, rtol=1e-4)


def test_tail_without_its_factor_fails_the_tail_pin():
    """mish(l) instead of l * mish(l): the pinned 11.68 -> 136.42 becomes about 11.68."""
    assert 11.68 * oracle.mish(11.68) == pytest.approx(136.4224, abs=1e-3)
    assert abs(oracle.mish(11.68) - 136.4224) > 100


def test_tanh_gelu_fails_the_normal_cdf_pin():
    """The tanh approximation in place of the exact erf GELU: 1.5e-4 off at x = 1, where the
    pin asks for 1e-14."""
    phi1 = 0.5 * (1.0 + math.erf(1.0 / math.sqrt(2.0)))
    assert oracle.gelu(1.0) == pytest.approx(phi1, abs=1e-15)
    assert abs(oracle.act("gelu_tanh", 1.0) - phi1) > 1e-5
