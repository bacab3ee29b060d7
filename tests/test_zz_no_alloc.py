"""fc_linear_lse_mish_noalloc, called through the C ABI, against fc_linear_lse_mish.

The allocation-free entry point exists for callers that cannot allocate
device memory (their memory belongs to another allocator or a fixed budget,
or a cudaMalloc and its possible device-wide synchronization is not
acceptable where they call from).  It keeps its scratch in the library's own
static device array.  This file is collected last so that a run stopping at
its first failure has already run every other test; it also passes alone in
a fresh process, where its first call does the one-time set-up.
"""
import ctypes

import numpy as np
import pytest

import fc_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3  # |gpu - ref| <= TOL * (1 + |ref|), the fp32-on-TF32 tolerance of the parity tests


def _noalloc_fn(lib):
    fn = lib.fc_linear_lse_mish_noalloc
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_float] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(cuda_lib):
    """Two calls in a row, the larger first, so the second reads an array the first filled further:
    each result equals the workspace entry point's bit for bit (same plan, same kernels), and the
    smaller one also matches the oracle within the fp32-on-TF32 tolerance."""
    import torch
    import oracle
    lib = cuda_lib.load()
    fn = _noalloc_fn(lib)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [((300, 260, 3000), (201, 202, 203), 20.0),   # larger first, clamp mostly active
             ((96, 512, 1200), (101, 102, 103), 1.0)]     # then fewer rows and column tiles
    for i, ((M, K, Nout), seeds, sx) in enumerate(cases):
        d = fc_inputs.linear_inputs(M, K, Nout, seeds=seeds)
        xh = (d["x"] * np.float32(sx)).astype(np.float32)
        x = torch.from_numpy(xh).cuda()
        W = torch.from_numpy(d["W"]).cuda()
        b = torch.from_numpy(d["b"]).cuda()
        y = torch.empty((M, 1), dtype=torch.float32, device="cuda")
        st = fn(x.data_ptr(), W.data_ptr(), b.data_ptr(), y.data_ptr(), M, K, Nout, 2.0, -10.0, 10.0, stream)
        assert st == cuda_lib.FC_OK, cuda_lib.fc_status_string(st)
        ref = cuda_lib.fc_linear_lse_mish(x, W, b, 2.0, -10.0, 10.0)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"case {(M, K, Nout)}: differs from fc_linear_lse_mish"
        if i == 1:
            want = oracle.linear_lse_mish(xh, d["W"], d["b"], 2.0, -10.0, 10.0).reshape(-1)
            got = y.cpu().numpy().astype(np.float64).reshape(-1)
            err = np.abs(got - want) / (1.0 + np.abs(want))
            assert err.max() <= TOL, f"case {(M, K, Nout)}: scaled error {err.max():.3e} against the oracle"
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def test_noalloc_rejects_requests_beyond_its_static_scratch(cuda_lib):
    import torch
    fn = _noalloc_fn(cuda_lib.load())
    M, K, Nout = 1024, 4, 40000          # >= 1024 * ceil(40000 / 256) = 160768 pairs of 8 B > 1 MiB
    x = torch.zeros((M, K), device="cuda")
    W = torch.zeros((Nout, K), device="cuda")
    b = torch.zeros(Nout, device="cuda")
    y = torch.zeros((M, 1), device="cuda")
    st = fn(x.data_ptr(), W.data_ptr(), b.data_ptr(), y.data_ptr(), M, K, Nout, 2.0, -10.0, 10.0, None)
    assert st == cuda_lib.FC_ERR_UNSUPPORTED
