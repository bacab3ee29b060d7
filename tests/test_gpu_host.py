"""The host-buffer conv entry points (x, w, b, y in host memory; copies overlapped with
the kernels slice by slice): parity with the fp64 oracle, bit-identity with the
device-buffer call on each slice, stream ordering, and argument errors (GPU only)."""
import numpy as np
import pytest

import fc_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-2}


def _host(arr, pinned=True):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr.view(np.int16) if arr.dtype == np.uint16 else arr))
    if arr.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.pin_memory() if pinned else t


def _check(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    assert got.shape == ref.shape
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    i = int(np.argmax(err))
    assert err[i] <= tol, f"{what}: scaled error {err[i]:.3e} > {tol} at {i}"


HOST_CASES = [
    # (N, Cin, H, W, Cout, pad, dtype, act, pool, layout, chunks)
    (7, 8, 34, 30, 64, 0, "f32", "gelu", True, "nchw", 3),      # ragged last slice (3, 3, 1)
    (5, 3, 13, 17, 3, 0, "f32", "gelu", True, "nchw", 8),       # more slices than images; odd byte sizes
    (4, 16, 18, 20, 64, 1, "bf16", "gelu", True, "nhwc", 2),
    (3, 64, 12, 140, 128, 0, "f32", "mish_mish", False, "nchw", 3),
    (5, 32, 9, 133, 64, 1, "bf16", "mish", False, "nhwc", 4),
    (2, 8, 21, 19, 40, 0, "f32", "mish_mish", False, "nchw", 1),
]


def _device_call(fc, d, N0, N1, case):
    """The device-buffer call on images [N0, N1) of the same inputs."""
    import torch
    N, Cin, H, W, Cout, pad, dt, act, pool, layout, chunks = case
    x = _host(d["x"], pinned=False)[N0:N1].clone().cuda()
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous().permute(0, 3, 1, 2)
    w, b = _host(d["w"], pinned=False).cuda(), _host(d["b"], pinned=False).cuda()
    f = fc.fc_conv3x3_act_pool if pool else fc.fc_conv3x3_act
    return f(x, w, b, act=act, pad=pad).cpu().contiguous()


@pytest.mark.parametrize("case", HOST_CASES,
                         ids=lambda c: "x".join(map(str, c[:5])) + f"-p{c[5]}-{c[6]}-{c[7]}-{'pool' if c[8] else 'act'}-{c[9]}-k{c[10]}")
def test_host_call_matches_oracle_and_the_device_call_per_slice(cuda_lib, case):
    import torch
    N, Cin, H, W, Cout, pad, dt, act, pool, layout, chunks = case
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    x = _host(d["x"])
    if layout == "nhwc":
        x = x.permute(0, 2, 3, 1).contiguous().pin_memory().permute(0, 3, 1, 2)
    f = cuda_lib.fc_conv3x3_act_pool_host if pool else cuda_lib.fc_conv3x3_act_host
    y = f(x, _host(d["w"]), _host(d["b"]), act=act, pad=pad, chunks=chunks)
    torch.cuda.synchronize()
    assert y.device.type == "cpu"
    ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x32"], d["w32"], d["b32"], act, pad=pad)
    y_np = y.contiguous().numpy()
    assert y_np.shape == ref.shape
    _check(y_np, ref, TOL[dt], f"host {case}")
    # the slices the call makes: ceil(N / chunks) images each, the last one ragged
    c = min(chunks, N)
    n0 = -(-N // c)
    for i0 in range(0, N, n0):
        i1 = min(N, i0 + n0)
        assert torch.equal(y.contiguous()[i0:i1], _device_call(cuda_lib, d, i0, i1, case)), (case, i0)
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def test_back_to_back_host_calls_share_one_staging_buffer_in_stream_order(cuda_lib):
    """The second call's copies must wait for the first call's kernels: same staging buffer,
    different inputs, no synchronization between the calls."""
    import torch
    shape = (6, 8, 40, 36, 64)
    d1 = fc_inputs.conv_inputs(*shape, seeds=(11, 12, 13))
    d2 = fc_inputs.conv_inputs(*shape, seeds=(21, 22, 23))
    nb = cuda_lib.fc_host_staging_bytes("conv3x3_act_pool", 6, 8, 40, 36, 64, chunks=3)
    assert nb > 0
    staging = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ys = []
    for d in (d1, d2, d1):
        ys.append(cuda_lib.fc_conv3x3_act_pool_host(_host(d["x"]), _host(d["w"]), _host(d["b"]),
                                                    staging=staging, chunks=3))
    torch.cuda.synchronize()
    for y, d in zip(ys, (d1, d2, d1)):
        _check(y.numpy(), oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], "gelu"), TOL["f32"], "in order")
    assert torch.equal(ys[0], ys[2])


def test_host_call_on_a_side_stream_and_with_pageable_memory(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(4, 8, 30, 22, 64)
    ref = cuda_lib.fc_conv3x3_act_pool_host(_host(d["x"]), _host(d["w"]), _host(d["b"]), chunks=2)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    y_side = cuda_lib.fc_conv3x3_act_pool_host(_host(d["x"]), _host(d["w"]), _host(d["b"]), chunks=2, stream=side)
    side.synchronize()
    y_pageable = cuda_lib.fc_conv3x3_act_pool_host(_host(d["x"], pinned=False), _host(d["w"], pinned=False),
                                                   _host(d["b"], pinned=False), chunks=2)
    torch.cuda.synchronize()
    assert torch.equal(y_side, ref) and torch.equal(y_pageable, ref)


def test_host_call_argument_errors(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(2, 8, 16, 16, 64)
    x, w, b = _host(d["x"]), _host(d["w"]), _host(d["b"])
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.FCError) as e:
        cuda_lib.fc_conv3x3_act_pool_host(x, w, b, staging=small)
    assert e.value.status == cuda_lib.FC_ERR_WORKSPACE
    with pytest.raises(cuda_lib.FCError) as e:
        cuda_lib.fc_conv3x3_act_pool_host(x, w, b, chunks=0)
    assert e.value.status == cuda_lib.FC_ERR_INVALID_ARG
    dw = fc_inputs.conv_inputs(1, 8, 16, 16, 300)
    with pytest.raises(cuda_lib.FCError) as e:
        cuda_lib.fc_conv3x3_act_pool_host(_host(dw["x"]), _host(dw["w"]), _host(dw["b"]))
    assert e.value.status == cuda_lib.FC_ERR_UNSUPPORTED
    with pytest.raises(ValueError, match="CPU tensor"):
        cuda_lib.fc_conv3x3_act_pool_host(x.cuda(), w, b)


def test_workload_B_full_size_through_the_host_buffer_call(cuda_lib):
    """The end-to-end call the benchmark times (conv3x3 + bias -> erf-GELU -> global average pool,
    x (128, 8, 256, 256) fp32 in pinned host memory, 8 slices of 16 images): sampled outputs
    against the oracle, every image of the first and last slice included."""
    import torch
    wl = fc_inputs.WORKLOADS["B"]
    d = fc_inputs.workload_inputs("B")
    y = cuda_lib.fc_conv3x3_act_pool_host(_host(d["x"]), _host(d["w"]), _host(d["b"]), act=wl.act, chunks=8)
    torch.cuda.synchronize()
    y = y.numpy()
    rng = np.random.default_rng(8)
    flat = np.unique(np.concatenate([rng.choice(wl.N * wl.Cout, 160, replace=False),
                                     np.arange(0, 16 * wl.Cout, 61), np.arange(112 * wl.Cout, 128 * wl.Cout, 59)]))
    ref = oracle.conv3x3_act_pool_at(d["x32"], d["w32"], d["b32"], flat, wl.act)
    _check(y.reshape(-1)[flat], ref, TOL["f32"], "workload B, host-buffer call")
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def _random_host_cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        pad = int(rng.choice([0, 0, 1, 2]))
        H, W = int(rng.integers(1, 40)), int(rng.integers(1, 40))
        if H + 2 * pad < 3 or W + 2 * pad < 3:
            continue
        cases.append((int(rng.integers(1, 9)), int(rng.integers(1, 33)), H, W,
                      int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 257))])), pad,
                      str(rng.choice(["f32", "bf16"])), str(rng.choice(["gelu", "mish", "mish_mish", "gelu_tanh"])),
                      bool(rng.integers(0, 2)), str(rng.choice(["nchw", "nhwc"])), int(rng.integers(1, 10))))
    return cases


@pytest.mark.parametrize("case", _random_host_cases(24),
                         ids=lambda c: "x".join(map(str, c[:5])) + f"-p{c[5]}-{c[6]}-{c[7]}-{'pool' if c[8] else 'act'}-{c[9]}-k{c[10]}")
def test_host_call_random_shapes(cuda_lib, case):
    """Seeded random shapes, slice counts (some above N), layouts and activations through the
    host-buffer call, against the oracle."""
    test_host_call_matches_oracle_and_the_device_call_per_slice(cuda_lib, case)
