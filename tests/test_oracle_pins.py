"""Pins of the oracle to facts outside itself (CPU only).

Each test checks the fp64 oracle against something it cannot agree with by
construction: printed table values, closed forms, invariants of the
definitions, special cases that reduce to a crop of the input or to a
constant, and an independent pure-Python brute force on tiny inputs.  The
cases are chosen so that a plausible slip anywhere in the oracle (a flipped
kernel, a transposed weight, a scaling applied once, the clamp in the wrong
place, the wrong pool divisor, the tail missing its factor) fails one of them.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
import fc_inputs

pytestmark = pytest.mark.filterwarnings("ignore")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _tolist(a):
    return np.asarray(a, dtype=np.float64).tolist()


# ------------------------------------------------------------------ GELU pins

def test_gelu_matches_normal_cdf_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "normal_cdf.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) >= 8
    for xs, phis in rows:
        x, phi = float(xs), float(phis)
        assert oracle.gelu(x) == pytest.approx(x * phi, abs=1e-15, rel=1e-14)


def test_gelu_invariants():
    assert oracle.gelu(0.0) == 0.0
    for x in np.linspace(-7, 7, 57):
        # GELU(x) - GELU(-x) = x Phi(x) + x Phi(x) - x = x   (Phi(-x) = 1 - Phi(x))
        assert oracle.gelu(x) - oracle.gelu(-x) == pytest.approx(x, abs=1e-14)
    for x in (8.0, 10.0, 30.0):
        assert abs(oracle.gelu(x) - x) < 1e-14
        assert abs(oracle.gelu(-x)) < 1e-14


def test_gelu_tanh_pins():
    """The tanh-approximate GELU: odd part exactly x, limits, slope 1/2 at 0, the independent
    logistic-form statement in oracle/brute.py, and within 5e-4 of the exact GELU everywhere
    (the approximation's known accuracy) but not equal to it."""
    g = lambda v: oracle.act("gelu_tanh", v)
    assert g(0.0) == 0.0
    for x in np.linspace(-7, 7, 57):
        # 0.5 x (1 + tanh u(x)) + 0.5 x (1 + tanh u(-x)) ... u is odd, so g(x) - g(-x) = x
        assert g(x) - g(-x) == pytest.approx(x, abs=1e-14)
        assert g(x) == pytest.approx(brute.gelu_tanh(float(x)), rel=1e-13, abs=1e-15)
    for x in (8.0, 10.0, 30.0):
        assert abs(g(x) - x) < 1e-12 and abs(g(-x)) < 1e-12
    h = 1e-6
    assert (g(h) - g(-h)) / (2 * h) == pytest.approx(0.5, abs=1e-9)
    dev = max(abs(g(x) - oracle.gelu(x)) for x in np.linspace(-8, 8, 4001))
    assert 1e-4 < dev < 5e-4


# ------------------------------------------------------------------ Mish pins

def _mish_closed_form(z):
    # tanh(log(1+e^z)) = ((1+e^z)^2 - 1) / ((1+e^z)^2 + 1) = n / (n + 2), n = e^z (e^z + 2)
    ez = math.exp(z)
    n = ez * (ez + 2.0)
    return z * n / (n + 2.0)


def test_mish_closed_form_identity():
    assert oracle.mish(0.0) == 0.0
    for z in np.linspace(-20, 20, 81):
        assert oracle.mish(z) == pytest.approx(_mish_closed_form(z), rel=1e-13, abs=1e-300)


def test_mish_limits():
    for z in (25.0, 50.0, 500.0):
        assert oracle.mish(z) == pytest.approx(z, rel=1e-15)
    for z in (-30.0, -50.0, -200.0):
        # mish(z) ~ z e^z as z -> -inf (tanh(s) ~ s ~ e^z)
        assert oracle.mish(z) == pytest.approx(z * math.exp(z), rel=1e-10)
    assert oracle.act("mish_mish", 1.0) == pytest.approx(_mish_closed_form(_mish_closed_form(1.0)), rel=1e-13)


def test_softplus_stable_form():
    for z in (-800.0, -40.0, -1.0, 0.0, 1.0, 40.0, 800.0):
        ref = z + math.log1p(math.exp(-z)) if z > 0 else math.log1p(math.exp(z))
        assert oracle.softplus(z) == pytest.approx(ref, rel=1e-15, abs=1e-320)


# ------------------------------------------------------------------ TF32 rounding (diagnostic mode)

def test_tf32_round_nearest_ties_away_and_bounds():
    one = 1.0
    u = 2.0 ** -10                      # TF32's unit in the last place at 1
    cases = [(one, one), (one + u, one + u), (one + u / 2, one + u),          # tie -> away from zero
             (one + u / 4, one), (one + 3 * u / 4, one + u), (-(one + u / 2), -(one + u)),
             (0.75, 0.75), (0.0, 0.0), (2.0 - u / 2, 2.0)]                      # carry into the exponent
    for x, want in cases:
        assert float(oracle.tf32_round_nearest(np.float32(x))) == want, x
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(10000) * 10.0 ** rng.uniform(-6, 6, 10000)).astype(np.float32)
    r = oracle.tf32_round_nearest(v)
    assert np.all(r.view(np.uint32) & np.uint32(0x1FFF) == 0)
    assert np.all(np.abs(r.astype(np.float64) - v) <= np.abs(v.astype(np.float64)) * 2.0 ** -11)


def test_tf32_truncate_is_toward_zero():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(10000) * 10.0 ** rng.uniform(-6, 6, 10000)).astype(np.float32)
    t = oracle.tf32_truncate(v).astype(np.float64)
    v64 = v.astype(np.float64)
    assert np.all(np.abs(t) <= np.abs(v64)) and np.all(np.sign(t) == np.sign(v64))
    assert np.all(np.abs(v64 - t) < np.abs(v64) * 2.0 ** -10)
    assert float(oracle.tf32_truncate(np.float32(1.0 + 2.0 ** -11))) == 1.0


# ------------------------------------------------------------------ conv pins

def test_conv_delta_kernel_reproduces_shifted_crop():
    rng = np.random.default_rng(5)
    N, Cin, H, W, Cout = 2, 3, 7, 9, 4
    x = rng.standard_normal((N, Cin, H, W)).astype(np.float32)
    for (cip, a, c) in [(0, 0, 0), (1, 2, 1), (2, 1, 2), (1, 0, 2)]:
        w = np.zeros((Cout, Cin, 3, 3), np.float32)
        w[:, cip, a, c] = 1.0
        b = np.zeros(Cout, np.float32)
        pre = oracle.conv3x3_preact(x, w, b)
        crop = x[:, cip, a:a + H - 2, c:c + W - 2].astype(np.float64)
        for co in range(Cout):
            np.testing.assert_array_equal(pre[:, co], crop)


def test_conv_linear_in_weights_and_bias_only_when_w_zero():
    x, w1, _ = (fc_inputs.conv_inputs(2, 3, 8, 7, 5, seeds=(11, 12, 13))[k] for k in ("x", "w", "b"))
    w2 = fc_inputs.conv_inputs(2, 3, 8, 7, 5, seeds=(11, 14, 15))["w"]
    zb = np.zeros(5, np.float32)
    p1 = oracle.conv3x3_preact(x, w1, zb)
    p2 = oracle.conv3x3_preact(x, w2, zb)
    p12 = oracle.conv3x3_preact(x, (w1.astype(np.float64) + w2).astype(np.float32), zb)
    # w1 + w2 is rounded to fp32 once; compare against the exact fp64 sum of the two convs
    # with a bound of that rounding (|w| < 0.2, 27 taps, |x| < 6 -> 27 * 6 * 2^-24 * 0.4)
    np.testing.assert_allclose(p12, p1 + p2, atol=1e-5)
    b = np.linspace(-0.3, 0.3, 5).astype(np.float32)
    pre0 = oracle.conv3x3_preact(x, np.zeros_like(w1), b)
    for co in range(5):
        assert np.all(pre0[:, co] == np.float64(b[co]))


@pytest.mark.parametrize("shape", [(1, 2, 5, 5, 3), (2, 3, 7, 6, 4)])
@pytest.mark.parametrize("act", ["gelu", "mish", "mish_mish", "gelu_tanh"])
def test_conv_act_against_brute_force(shape, act):
    N, Cin, H, W, Cout = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, seeds=(21, 22, 23))
    x, w, b = d["x"], d["w"], d["b"]
    ref = np.array(brute.conv3x3_act(_tolist(x), _tolist(w), _tolist(b), act))
    got = oracle.conv3x3_act(x, w, b, act)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    ref_pool = np.array(brute.conv3x3_act_pool(_tolist(x), _tolist(w), _tolist(b), act))
    got_pool = oracle.conv3x3_act_pool(x, w, b, act)
    np.testing.assert_allclose(got_pool, ref_pool, rtol=1e-12, atol=1e-14)
    # sampled entry points agree with the full ones
    flat = np.arange(got.size)[::3]
    np.testing.assert_array_equal(oracle.conv3x3_act_at(x, w, b, flat, act), got.reshape(-1)[flat])
    flat_nc = np.arange(N * Cout)[::2]
    np.testing.assert_array_equal(oracle.conv3x3_act_pool_at(x, w, b, flat_nc, act), got_pool.reshape(-1)[flat_nc])


# Padding (the general-padding variant; zero padding, PyTorch's padding_mode 'zeros').

def test_conv_padding_one_with_centre_delta_is_identity():
    """'same' conv: p = 1 and w[co, ci, 1, 1] = [co == ci] reproduce the input exactly."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((2, 3, 6, 7)).astype(np.float32)
    w = np.zeros((3, 3, 3, 3), np.float32)
    for c in range(3):
        w[c, c, 1, 1] = 1.0
    pre = oracle.conv3x3_preact(x, w, np.zeros(3, np.float32), pad=1)
    np.testing.assert_array_equal(pre, x.astype(np.float64))


@pytest.mark.parametrize("pad", [1, 2, 5])
def test_conv_padding_equals_conv_of_zero_extended_input(pad):
    d = fc_inputs.conv_inputs(2, 3, 5, 7, 4, seeds=(51, 52, 53))
    x, w, b = d["x"], d["w"], d["b"]
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad)))
    got = oracle.conv3x3_act(x, w, b, "mish", pad=pad)
    assert got.shape == (2, 4, 5 + 2 * pad - 2, 7 + 2 * pad - 2)
    # the same terms in the same order apart from zero products: equal to fp64 rounding
    np.testing.assert_allclose(got, oracle.conv3x3_act(xp, w, b, "mish"), rtol=1e-15, atol=1e-16)
    np.testing.assert_allclose(oracle.conv3x3_act_pool(x, w, b, "gelu", pad=pad),
                               oracle.conv3x3_act_pool(xp, w, b, "gelu"), rtol=1e-14, atol=1e-16)


@pytest.mark.parametrize("act", ["gelu", "mish_mish"])
def test_conv_padding_against_brute_force(act):
    d = fc_inputs.conv_inputs(1, 2, 4, 5, 3, seeds=(54, 55, 56))
    x, w, b = d["x"], d["w"], d["b"]
    for pad in (1, 3):
        ref = np.array(brute.conv3x3_act(_tolist(x), _tolist(w), _tolist(b), act, pad))
        np.testing.assert_allclose(oracle.conv3x3_act(x, w, b, act, pad=pad), ref, rtol=1e-12, atol=1e-14)
        ref_pool = np.array(brute.conv3x3_act_pool(_tolist(x), _tolist(w), _tolist(b), act, pad))
        np.testing.assert_allclose(oracle.conv3x3_act_pool(x, w, b, act, pad=pad), ref_pool, rtol=1e-12,
                                   atol=1e-14)
        flat = np.arange(ref.size)[::2]
        np.testing.assert_array_equal(oracle.conv3x3_act_at(x, w, b, flat, act, pad=pad),
                                      oracle.conv3x3_act(x, w, b, act, pad=pad).reshape(-1)[flat])


def test_conv_padding_corner_sees_one_tap():
    """With p = 2 the output corner (0, 0) overlaps the input only at x[0, 0] through tap (2, 2)."""
    d = fc_inputs.conv_inputs(1, 2, 6, 6, 2, seeds=(57, 58, 59))
    x, w, b = d["x"], d["w"], d["b"]
    pre = oracle.conv3x3_preact(x, w, b, pad=2)
    for co in range(2):
        v = math.fsum([float(b[co])] + [float(x[0, ci, 0, 0]) * float(w[co, ci, 2, 2]) for ci in range(2)])
        assert pre[0, co, 0, 0] == pytest.approx(v, rel=1e-15)
        # and the far corner through tap (0, 0)
        v2 = math.fsum([float(b[co])] + [float(x[0, ci, 5, 5]) * float(w[co, ci, 0, 0]) for ci in range(2)])
        assert pre[0, co, -1, -1] == pytest.approx(v2, rel=1e-15)
    with pytest.raises(ValueError):
        oracle.conv3x3_preact(x, w, b, pad=-1)


def test_pool_with_zero_weights_is_act_of_bias():
    d = fc_inputs.conv_inputs(2, 3, 9, 11, 6, seeds=(31, 32, 33))
    y = oracle.conv3x3_act_pool(d["x"], np.zeros_like(d["w"]), d["b"], "gelu")
    for co in range(6):
        # the mean of OH*OW equal terms is that term, up to the rounding of the fp64 sum
        np.testing.assert_allclose(y[:, co], oracle.gelu(float(d["b"][co])), rtol=1e-14, atol=0)


def test_pool_of_constant_plane_is_act_of_constant_conv():
    N, Cin, H, W, Cout = 1, 2, 6, 8, 3
    x = np.full((N, Cin, H, W), 0.75, np.float32)
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, seeds=(41, 42, 43))
    w, b = d["w"], d["b"]
    y = oracle.conv3x3_act_pool(x, w, b, "gelu")
    for co in range(Cout):
        v = math.fsum([float(b[co])] + [0.75 * float(t) for t in w[co].reshape(-1)])
        assert y[0, co] == pytest.approx(oracle.gelu(v), rel=1e-13)


# ------------------------------------------------------------------- LSE pins

def test_lse_constant_row_and_shift_invariance():
    for n in (1, 7, 8192):
        for c in (-3.5, 0.0, 2.25, 10.0):
            assert oracle.logsumexp(np.full(n, c)) == pytest.approx(c + math.log(n), abs=1e-12)
    t = np.random.default_rng(1).standard_normal(1000) * 3
    for a in (-100.0, 0.5, 700.0):
        assert oracle.logsumexp(t + a) == pytest.approx(oracle.logsumexp(t) + a, rel=1e-13)
    one_hot = np.full(100, -50.0)
    one_hot[37] = 60.0
    # exactly 60 + log(1 + 99 e^-110)
    assert oracle.logsumexp(one_hot) == pytest.approx(60.0 + math.log1p(99 * math.exp(-110.0)), rel=1e-15)


def test_linear_zero_weights_closed_form():
    M, K, Nout = 3, 16, 8192
    x = np.random.default_rng(3).standard_normal((M, K)).astype(np.float32)
    for c, expect_t in [(0.5, 2.0), (3.0, 10.0), (-4.0, -10.0), (-1.25, -5.0)]:
        b = np.full(Nout, c, np.float32)
        y, l = oracle.linear_lse_mish(x, np.zeros((Nout, K), np.float32), b, return_lse=True)
        # t = clamp((c*2) + (c*2)) for every column -> l = clamp(4c) + ln Nout
        np.testing.assert_allclose(l, expect_t + math.log(Nout), rtol=0, atol=1e-12)
        np.testing.assert_allclose(y, l * np.array([_mish_closed_form(v) for v in l]), rtol=1e-13)


def test_linear_lse_bounds_and_tail():
    M, K, Nout = 4, 32, 64
    d = fc_inputs.linear_inputs(M, K, Nout, seeds=(51, 52, 53))
    x = d["x"] * 40.0           # drive |4t| far past 10 so the clamp is active
    y, l = oracle.linear_lse_mish(x, d["W"], d["b"], return_lse=True)
    assert np.all(l >= -10.0 + math.log(Nout) - 1e-12)
    assert np.all(l <= 10.0 + math.log(Nout) + 1e-12)
    # the tail is l * mish(l) (~ l^2 for large l), not mish(l)
    for v in (11.68, 15.0):
        yv = v * oracle.mish(v)
        assert yv == pytest.approx(v * v, rel=1e-9)
    assert 11.68 * oracle.mish(11.68) == pytest.approx(136.4224, abs=1e-3)


@pytest.mark.parametrize("scale_x", [1.0, 30.0])
def test_linear_against_brute_force(scale_x):
    M, K, Nout = 3, 5, 7
    d = fc_inputs.linear_inputs(M, K, Nout, seeds=(61, 62, 63))
    x = (d["x"] * scale_x).astype(np.float32)
    ys, ls = brute.linear_lse_mish(_tolist(x), _tolist(d["W"]), _tolist(d["b"]), 2.0, -10.0, 10.0)
    y, l = oracle.linear_lse_mish(x, d["W"], d["b"], return_lse=True)
    np.testing.assert_allclose(l, ls, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y, ys, rtol=1e-12, atol=1e-13)
    # row subsets agree with the full call
    y2 = oracle.linear_lse_mish(x, d["W"], d["b"], rows=[2, 0])
    np.testing.assert_array_equal(y2, y[[2, 0]])


def test_linear_is_x_times_w_transposed():
    # a non-square W with one non-zero entry W[j0, k0] selects x[:, k0] into column j0
    M, K, Nout, j0, k0 = 2, 6, 3, 2, 4
    x = np.arange(M * K, dtype=np.float32).reshape(M, K) / 10.0
    Wt = np.zeros((Nout, K), np.float32)
    Wt[j0, k0] = 1.0
    b = np.zeros(Nout, np.float32)
    _, l = oracle.linear_lse_mish(x, Wt, b, return_lse=True)
    for m in range(M):
        t = [0.0] * Nout
        t[j0] = min(max(4.0 * float(x[m, k0]), -10.0), 10.0)
        assert l[m] == pytest.approx(max(t) + math.log(sum(math.exp(v - max(t)) for v in t)), rel=1e-14)


# ---------------------------------------------------------- input generator

def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 2**-8 + 2**-20, 1.0 + 3 * 2**-8, -2.5, 3.1415927], np.float32)
    bits = fc_inputs.bf16_bits(vals)
    back = fc_inputs.bf16_bits_to_f32(bits)
    assert back[0] == 1.0
    assert back[1] == 1.0                       # tie -> even
    assert back[2] == np.float32(1.0 + 2**-7)   # above the tie -> up
    assert back[3] == np.float32(1.0 + 2**-6)   # tie -> even (up)
    assert back[4] == -2.5
    assert abs(back[5] - 3.1415927) <= 2**-7 * 2


def test_inputs_are_seeded_and_shaped():
    a = fc_inputs.conv_inputs(2, 8, 32, 32, 64)
    b = fc_inputs.conv_inputs(2, 8, 32, 32, 64)
    assert a["x"].shape == (2, 8, 32, 32) and a["w"].shape == (64, 8, 3, 3)
    np.testing.assert_array_equal(a["x"], b["x"])
    bound = 1 / math.sqrt(72)
    assert np.all(np.abs(a["w"]) <= bound) and np.all(np.abs(a["b"]) <= bound)
    assert abs(float(a["x"].mean())) < 0.05 and abs(float(a["x"].std()) - 1) < 0.05


def test_sampled_entry_points_reject_out_of_range_indices():
    d = fc_inputs.conv_inputs(1, 2, 5, 5, 3)
    with pytest.raises(IndexError):
        oracle.conv3x3_act_pool_at(d["x"], d["w"], d["b"], [3], "gelu")
    with pytest.raises(IndexError):
        oracle.conv3x3_act_at(d["x"], d["w"], d["b"], [-1], "gelu")
    dl = fc_inputs.linear_inputs(2, 4, 3)
    with pytest.raises(IndexError):
        oracle.linear_lse_mish(dl["x"], dl["W"], dl["b"], rows=[2])


# ------------------------------------------------------------ standalone epilogues

@pytest.mark.parametrize("act", ["gelu", "mish", "mish_mish", "gelu_tanh"])
def test_act_map_matches_independent_statement(act):
    v = fc_inputs.epilogue_inputs((3, 5, 7), seed=31) * np.float32(3.0)
    got = oracle.act_map(v, act)
    ref = np.array([brute.ACTS[act](float(z)) for z in v.reshape(-1)]).reshape(v.shape)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_act_mean_pins():
    # constant planes: the mean is act(c); against math.fsum of the independent statement;
    # and the pooled conv is the plane mean of its pre-activation
    for c in (-3.0, 0.0, 0.7, 9.0):
        v = np.full((2, 3, 4, 5), c, np.float32)
        np.testing.assert_allclose(oracle.act_mean(v, "gelu"), oracle.gelu(float(np.float32(c))), rtol=1e-14,
                                   atol=1e-16)
    v = fc_inputs.epilogue_inputs((2, 3, 6, 7), seed=32)
    ref = np.array([[math.fsum(brute.gelu(float(z)) for z in v[n, c].reshape(-1)) / 42.0 for c in range(3)]
                    for n in range(2)])
    np.testing.assert_allclose(oracle.act_mean(v, "gelu"), ref, rtol=1e-12, atol=1e-15)
    d = fc_inputs.conv_inputs(2, 3, 9, 8, 4, seeds=(41, 42, 43))
    pre = oracle.conv3x3_preact(d["x"], d["w"], d["b"]).astype(np.float32)
    np.testing.assert_allclose(oracle.act_mean(pre, "mish"), oracle.conv3x3_act_pool(d["x"], d["w"], d["b"], "mish"),
                               rtol=1e-6, atol=1e-7)


def test_scale_clamp_lse_mish_pins():
    N = 1000
    # a constant row c: l = clamp(4c) + ln N, y = l * mish(l)
    for c in (-5.0, -0.3, 0.0, 1.1, 4.0):
        y = oracle.scale_clamp_lse_mish(np.full((1, N), c, np.float32), 2.0, -10.0, 10.0)[0, 0]
        l = min(max(4 * float(np.float32(c)), -10.0), 10.0) + math.log(N)
        assert y == pytest.approx(l * oracle.mish(l), rel=1e-12)
    # against an independent per-row statement (math.fsum logsumexp, the brute mish)
    t = fc_inputs.epilogue_inputs((4, 257), seed=33) * np.float32(2.5)
    got = oracle.scale_clamp_lse_mish(t, 2.0, -10.0, 10.0)[:, 0]
    for m in range(4):
        u = [min(max(2.0 * float(z) + 2.0 * float(z), -10.0), 10.0) for z in t[m]]
        mx = max(u)
        l = mx + math.log(math.fsum(math.exp(q - mx) for q in u))
        assert got[m] == pytest.approx(l * brute.mish(l), rel=1e-12)
    # the Linear chain's tail: rows of x W^T + b through this function give the chain's output
    d = fc_inputs.linear_inputs(3, 16, 40, seeds=(51, 52, 53))
    t = (d["x"].astype(np.float64) @ d["W"].astype(np.float64).T + d["b"].astype(np.float64)).astype(np.float32)
    np.testing.assert_allclose(oracle.scale_clamp_lse_mish(t)[:, 0],
                               oracle.linear_lse_mish(d["x"], d["W"], d["b"], 2.0, -10.0, 10.0).reshape(-1),
                               rtol=1e-6)


def test_oracle_results_do_not_depend_on_the_thread_count():
    """Each pooled output is summed in a fixed order by one thread: 1 thread and all threads agree bit for bit."""
    d = fc_inputs.conv_inputs(2, 3, 12, 11, 5)
    n = oracle.threads()
    try:
        oracle.set_threads(1)
        one = oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], "gelu")
        full = oracle.conv3x3_act(d["x32"], d["w32"], d["b32"], "mish_mish")
    finally:
        oracle.set_threads(n)
    assert oracle.threads() == n
    assert np.array_equal(one, oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], "gelu"))
    assert np.array_equal(full, oracle.conv3x3_act(d["x32"], d["w32"], d["b32"], "mish_mish"))
