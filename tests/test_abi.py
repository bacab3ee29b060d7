"""The C-ABI library builds for sm_103a, loads, exports every symbol the public
header declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import gemm_activation_reduction_gb300 as fc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(fc_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_fused_ops():
    names = declared_functions()
    for n in ("fc_conv3x3_act_pool", "fc_conv3x3_act", "fc_linear_lse_mish", "fc_workspace_bytes"):
        assert n in names
    assert set(names) == set(fc.EXPORTS)


def test_library_builds_and_exports_every_declared_symbol():
    lib = fc.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
    # dynamic symbol table of the shared object, read with nm
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fc.library_path()], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


def test_status_strings_and_version():
    assert fc.fc_status_string(fc.FC_OK) == "ok"
    assert "timed out" in fc.fc_status_string(fc.FC_ERR_TIMEOUT)
    assert "index check" in fc.fc_status_string(fc.FC_ERR_BOUNDS)
    assert fc.fc_version() >= 100


def _call_pool(lib, x=16, w=16, b=16, y=16, N=1, Cin=8, H=8, W=8, Cout=64, dtype=0, act=0, ws=None, wsb=0):
    return lib.fc_conv3x3_act_pool(x, w, b, y, N, Cin, H, W, Cout, dtype, act, ws, wsb, None)


def test_host_validation_rejects_bad_arguments_before_any_launch():
    lib = fc.load()
    assert _call_pool(lib, x=None) == fc.FC_ERR_INVALID_ARG
    assert _call_pool(lib, y=0) == fc.FC_ERR_INVALID_ARG
    assert _call_pool(lib, x=0x1004) == fc.FC_ERR_INVALID_ARG           # not 16-byte aligned
    assert _call_pool(lib, H=2) == fc.FC_ERR_INVALID_ARG
    assert _call_pool(lib, N=0) == fc.FC_ERR_INVALID_ARG
    assert _call_pool(lib, dtype=7) == fc.FC_ERR_INVALID_ARG
    assert _call_pool(lib, act=9) == fc.FC_ERR_INVALID_ARG
    assert lib.fc_conv3x3_act(16, 16, 16, 16, 1, 8, 2, 8, 64, 0, 2, None, 0, None) == fc.FC_ERR_INVALID_ARG
    lin = lib.fc_linear_lse_mish
    assert lin(16, 16, 16, 16, 4, 8, 8, 2.0, 1.0, -1.0, 0, None, 0, None) == fc.FC_ERR_INVALID_ARG  # lo > hi
    assert lin(16, 16, 16, 16, 4, 8, 8, 2.0, float("nan"), 1.0, 0, None, 0, None) == fc.FC_ERR_INVALID_ARG
    assert lin(16, 16, 16, 16, 0, 8, 8, 2.0, -1.0, 1.0, 0, None, 0, None) == fc.FC_ERR_INVALID_ARG
    assert lin(16, 16, 16, 16, 4, 6, 8, 2.0, -1.0, 1.0, 0, None, 0, None) == fc.FC_ERR_UNSUPPORTED  # K % 4
    assert lin(16, 16, 16, 16, 4, 4, 8, 2.0, -1.0, 1.0, 1, None, 0, None) == fc.FC_ERR_UNSUPPORTED  # bf16, K % 8


def test_without_a_device_calls_report_cuda_errors_not_crashes():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = fc.load()
    assert _call_pool(lib) == fc.FC_ERR_CUDA
    assert lib.fc_workspace_bytes(0, 1, 8, 8, 8, 64, 0) == 0


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 8, 8, 8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fc.fc_conv3x3_act_pool(x, torch.zeros(64, 8, 3, 3), torch.zeros(64))
    with pytest.raises(ValueError, match="CUDA tensor"):
        fc.fc_linear_lse_mish(torch.zeros(4, 8), torch.zeros(8, 8), torch.zeros(8))


def test_host_buffer_entry_points_validate_before_any_copy():
    import torch
    lib = fc.load()
    host = lib.fc_conv3x3_act_pool_host

    def call(x=16, y=16, N=2, chunks=4, staging=None, nb=0):
        return host(x, 16, 16, y, N, 8, 8, 8, 64, 0, fc.FC_NCHW, fc.FC_F32, 0, chunks, staging, nb, None)

    assert call(x=None) == fc.FC_ERR_INVALID_ARG
    assert call(y=None) == fc.FC_ERR_INVALID_ARG
    assert call(chunks=0) == fc.FC_ERR_INVALID_ARG
    assert call(N=0) == fc.FC_ERR_INVALID_ARG
    assert lib.fc_conv3x3_act_host(16, 16, 16, 16, 1, 8, 2, 2, 64, 0, fc.FC_NCHW, fc.FC_F32, 2, 1, None, 0,
                                   None) == fc.FC_ERR_INVALID_ARG          # a 2 x 2 input with no padding
    assert lib.fc_host_staging_bytes(0, 2, 8, 8, 8, 64, 0, fc.FC_NCHW, fc.FC_F32, 0) == 0
    if not torch.cuda.is_available():
        # a well-formed call with no device reports a CUDA error and copies nothing
        assert call() == fc.FC_ERR_CUDA
        assert lib.fc_host_staging_bytes(0, 2, 8, 8, 8, 64, 0, fc.FC_NCHW, fc.FC_F32, 4) == 0


def test_python_host_binding_refuses_device_tensors():
    import torch
    with pytest.raises(ValueError, match="CPU tensor"):
        fc.fc_conv3x3_act_pool_host(torch.zeros(1, 8, 8, 8, device="meta"), torch.zeros(64, 8, 3, 3),
                                    torch.zeros(64))


def _compile_c_client(out_path):
    """Build tests/c_abi_client.c as plain C99 against include/fc.h and the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(fc.library_path())
    lib = os.path.basename(fc.library_path())[3:-3]
    # C11: the CUDA runtime's own headers use anonymous unions; fc.h alone is checked as C99 below
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-o", out_path,
           os.path.join(ROOT, "tests", "c_abi_client.c"), "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-l" + lib, "-Wl,-rpath," + libdir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


def test_plain_c_client_compiles_and_links(tmp_path):
    """The header is valid C99 and the library links into a C program with the CUDA runtime alone."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    fc.load()
    _compile_c_client(str(tmp_path / "c_abi_client"))
    assert os.path.exists(tmp_path / "c_abi_client")


@pytest.mark.gpu
def test_plain_c_client_runs_the_tiny_workload(tmp_path):
    """The C client on a GPU: the tiny conv -> GELU -> pool workload (2, 8, 32, 32) -> 64 channels
    through the C ABI from C, against the oracle."""
    import subprocess
    import numpy as np
    import fc_inputs
    import oracle
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fc.load()
    exe = str(tmp_path / "c_abi_client")
    _compile_c_client(exe)
    N, Cin, H, W, Cout = 2, 8, 32, 32, 64
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout)
    paths = {}
    for k in ("x", "w", "b"):
        paths[k] = str(tmp_path / f"{k}.bin")
        np.ascontiguousarray(d[k], dtype="<f4").tofile(paths[k])
    y_path = str(tmp_path / "y.bin")
    r = subprocess.run([exe, str(N), str(Cin), str(H), str(W), str(Cout), paths["x"], paths["w"], paths["b"], y_path],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    y = np.fromfile(y_path, dtype="<f4").reshape(N, Cout).astype(np.float64)
    ref = oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], "gelu")
    err = np.abs(y - ref) / (1.0 + np.abs(ref))
    assert err.max() <= 2e-3, err.max()


def test_python_host_binding_validates_before_any_cuda_call():
    import torch
    x = torch.zeros(2, 8, 8, 8)
    w = torch.zeros(64, 8, 3, 3)
    b = torch.zeros(64)
    with pytest.raises(ValueError, match="share one dtype"):
        fc.fc_conv3x3_act_pool_host(x, w.to(torch.bfloat16), b)
    with pytest.raises(ValueError, match="expected x"):
        fc.fc_conv3x3_act_pool_host(x, torch.zeros(64, 8, 5, 5), b)
    with pytest.raises(ValueError, match="contiguous"):
        fc.fc_conv3x3_act_host(x.transpose(2, 3), w, b, layout="nchw")
    with pytest.raises(ValueError, match="out must be"):
        fc.fc_conv3x3_act_pool_host(x, w, b, out=torch.zeros(2, 63))
