"""The FC_DEBUG build: the same kernels with index checks that, instead of trapping, record
FC_ERR_BOUNDS in the device status word and skip the access.  On the CPU the debug flag's code
is compiled; on the GPU the debug library runs small shapes of every operator family and must
match the oracle with no check firing (no false positives)."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import fc_inputs
import oracle
from gemm_activation_reduction_gb300 import _build

TOL = {"f32": 2e-3, "bf16": 2e-2}


def test_debug_flag_compiles():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    for name in ("fc_conv_tf32.cu", "fc_linear.cu"):
        src = os.path.join(_build.CSRC, name)
        r = subprocess.run([nvcc, *_build.ARCH, *_build.NVCC_FLAGS, "-DFC_DEBUG", "-c", src, "-o", os.devnull],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]


def _dev(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(got, ref, tol, what):
    got = np.asarray(got, np.float64).reshape(-1)
    ref = np.asarray(ref, np.float64).reshape(-1)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert err.max() <= tol, f"{what}: scaled error {err.max():.3e}"


@pytest.mark.gpu
def test_debug_build_matches_the_oracle_and_records_nothing():
    import torch
    lib = ctypes.CDLL(_build.build(debug=True))
    P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    for nm in ("fc_conv3x3_act_pool_ex", "fc_conv3x3_act_ex"):
        getattr(lib, nm).argtypes = [P, P, P, P, I, I, I, I, I, I, I, I, I, P, S, P]
    lib.fc_workspace_bytes_ex.restype = S
    lib.fc_workspace_bytes_ex.argtypes = [I] * 9
    lib.fc_linear_lse_mish.argtypes = [P, P, P, P, I, I, I, F, F, F, I, P, S, P]
    lib.fc_workspace_bytes.restype = S
    lib.fc_workspace_bytes.argtypes = [I] * 7
    lib.fc_device_status.argtypes = [I]
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fc_device_status(1) == 0

    acts = {"gelu": 0, "mish": 1, "mish_mish": 2, "gelu_tanh": 3}
    conv_cases = [  # (N, Cin, H, W, Cout, dtype, act, pool, layout)
        (2, 8, 40, 70, 64, "f32", "gelu", True, 0),      # 16 x 32 pooled tiles, ragged edges
        (1, 13, 20, 37, 96, "f32", "gelu", True, 0),     # 16 x 8 pooled tiles
        (1, 40, 17, 19, 256, "bf16", "gelu_tanh", True, 0),   # CTA pairs
        (1, 16, 13, 150, 64, "f32", "mish_mish", False, 0),   # two-row full-output tiles
        (1, 16, 9, 133, 250, "f32", "mish", False, 0),        # CTA pairs, padded Cout
        (1, 32, 12, 40, 64, "bf16", "mish_mish", False, 1),   # NHWC
    ]
    for N, Cin, H, W, Cout, dt, act, pool, nhwc in conv_cases:
        d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
        xa = np.transpose(d["x"], (0, 2, 3, 1)) if nhwc else d["x"]
        x, w, b = _dev(xa), _dev(d["w"]), _dev(d["b"])
        dtype = 1 if dt == "bf16" else 0
        nb = lib.fc_workspace_bytes_ex(0 if pool else 1, N, Cin, H, W, Cout, 0, nhwc, dtype)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
        OH, OW = H - 2, W - 2
        y = torch.empty((N, Cout) if pool else ((N, OH, OW, Cout) if nhwc else (N, Cout, OH, OW)), device="cuda")
        fn = lib.fc_conv3x3_act_pool_ex if pool else lib.fc_conv3x3_act_ex
        st = fn(x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), N, Cin, H, W, Cout, 0, nhwc, dtype,
                acts[act], ws.data_ptr(), nb, stream)
        assert st == 0, (N, Cin, H, W, Cout, dt, act, pool, nhwc, st)
        got = y.cpu().numpy()
        if nhwc:
            got = np.transpose(got, (0, 3, 1, 2))
        ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x32"], d["w32"], d["b32"], act)
        _check(got, ref, TOL[dt], f"debug conv {(N, Cin, H, W, Cout, dt, act, pool, nhwc)}")
        assert lib.fc_device_status(1) == 0
    for M, K, Nout in ((96, 512, 1200), (300, 260, 3000)):   # single CTAs, then CTA pairs
        d = fc_inputs.linear_inputs(M, K, Nout)
        x, W, b = _dev(d["x"]), _dev(d["W"]), _dev(d["b"])
        nb = lib.fc_workspace_bytes(2, M, K, 1, 1, Nout, 0)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
        y = torch.empty((M, 1), device="cuda")
        assert lib.fc_linear_lse_mish(x.data_ptr(), W.data_ptr(), b.data_ptr(), y.data_ptr(), M, K, Nout,
                                      2.0, -10.0, 10.0, 0, ws.data_ptr(), nb, stream) == 0
        _check(y.cpu().numpy(), oracle.linear_lse_mish(d["x"], d["W"], d["b"]), TOL["f32"], f"debug linear {(M, K, Nout)}")
        assert lib.fc_device_status(1) == 0
