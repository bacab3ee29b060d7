"""The standalone epilogues (fc_act_map, fc_act_mean, fc_scale_clamp_lse_mish) through the C ABI,
element by element against the fp64 oracle on the same seeded inputs.

Tolerance: |gpu - ref| <= tol * (1 + |ref|), tol = 2e-6 elementwise and 2e-5 for the plane means
and row reductions (fp32 arithmetic and fp32 sums of up to 64516 terms; no TF32 here), on fp32 or
exactly upcast bf16 inputs.
"""
import ctypes

import numpy as np
import pytest

import fc_inputs
import oracle

pytestmark = pytest.mark.gpu

ACTS = ["gelu", "mish", "mish_mish", "gelu_tanh"]


def _dev(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(a):
    return fc_inputs.bf16_bits_to_f32(a) if a.dtype == np.uint16 else a


def _check(got, ref, tol, what):
    got = np.asarray(got, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert err.max() <= tol, f"{what}: max scaled error {err.max():.3e} at {int(np.argmax(err))}"


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("shape,dt", [((3, 7, 13, 17), "f32"), ((1000003,), "f32"), ((2, 5, 9, 11), "bf16"),
                                      ((5,), "f32")])
def test_act_map(cuda_lib, act, shape, dt):
    v = fc_inputs.epilogue_inputs(shape, seed=61, dtype=dt, scale=4.0)
    out = cuda_lib.fc_act_map(_dev(v), act=act).cpu().numpy()
    assert out.shape == shape
    _check(out, oracle.act_map(_host(v), act), 2e-6, f"act_map {act} {shape} {dt}")


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("shape,dt", [((2, 3, 5, 7), "f32"),       # plane of 35: misaligned planes, scalar path
                                      ((2, 4, 32, 32), "f32"),     # aligned planes, vector path
                                      ((1, 3, 254, 254), "f32"),   # the conv output plane of the pages
                                      ((2, 3, 9, 13), "bf16"),
                                      ((1, 2, 16, 16), "bf16")])
def test_act_mean(cuda_lib, act, shape, dt):
    v = fc_inputs.epilogue_inputs(shape, seed=62, dtype=dt, scale=2.0)
    y = cuda_lib.fc_act_mean(_dev(v), act=act).cpu().numpy()
    assert y.shape == shape[:2]
    _check(y, oracle.act_mean(_host(v), act), 2e-5, f"act_mean {act} {shape} {dt}")


@pytest.mark.parametrize("M,N,scale_in", [(7, 1000, 1.0), (5, 8192, 0.6), (3, 1001, 1.0), (2, 3, 1.0),
                                          (4, 4096, 12.0)])   # last: most of the row clamped
def test_scale_clamp_lse_mish(cuda_lib, M, N, scale_in):
    t = fc_inputs.epilogue_inputs((M, N), seed=63, scale=scale_in)
    y = cuda_lib.fc_scale_clamp_lse_mish(_dev(t), 2.0, -10.0, 10.0).cpu().numpy()
    _check(y, oracle.scale_clamp_lse_mish(t, 2.0, -10.0, 10.0), 2e-5, f"lse rows ({M},{N}) x{scale_in}")


def test_act_mean_full_size_sampled(cuda_lib):
    """The conv->GELU->pool page's epilogue at its size: (128, 64, 254, 254) fp32 (2.1 GB),
    sampled planes against the oracle."""
    shape = (128, 64, 254, 254)
    v = fc_inputs.epilogue_inputs(shape, seed=64, scale=0.58)
    y = cuda_lib.fc_act_mean(_dev(v), act="gelu").cpu().numpy()
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.choice(128 * 64, 48, replace=False), [0, 128 * 64 - 1]]))
    n, c = np.divmod(idx, 64)
    ref = oracle.act_mean(v[n, c][:, None], "gelu")[:, 0]
    _check(y[n, c], ref, 2e-5, "act_mean full size")


def test_epilogue_entry_points_reject_bad_arguments(cuda_lib):
    import torch
    lib = cuda_lib.load()
    v = torch.zeros(64, device="cuda")
    out = torch.zeros(64, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # misaligned pointers, negative sizes, bad enums, empty planes, inverted clamp bounds
    assert lib.fc_act_map(v.data_ptr() + 4, out.data_ptr(), 8, 0, 0, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_act_map(v.data_ptr(), out.data_ptr(), -1, 0, 0, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_act_map(v.data_ptr(), out.data_ptr(), 8, 0, 7, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_act_map(v.data_ptr(), out.data_ptr(), 0, 0, 0, s) == cuda_lib.FC_OK
    assert lib.fc_act_mean(v.data_ptr(), out.data_ptr(), 0, 8, 0, 0, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_act_mean(v.data_ptr(), out.data_ptr(), 2, 0, 0, 0, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_act_mean(v.data_ptr(), out.data_ptr(), 2, 8, 2, 0, s) == cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_scale_clamp_lse_mish(v.data_ptr(), out.data_ptr(), 2, 8, 2.0, 1.0, -1.0, s) == \
        cuda_lib.FC_ERR_INVALID_ARG
    assert lib.fc_scale_clamp_lse_mish(v.data_ptr(), out.data_ptr(), 0, 8, 2.0, -1.0, 1.0, s) == \
        cuda_lib.FC_ERR_INVALID_ARG
    torch.cuda.synchronize()
