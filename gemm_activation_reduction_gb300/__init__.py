"""GB300 (sm_103a) fused contraction + activation + reduction kernels.

Thin ctypes binding over the C ABI in ``include/fc.h``: the functions below
carry the C names, check that the torch tensors they are given are CUDA,
contiguous and of the right dtype, allocate the output and the workspace
with torch (device memory only), and pass raw pointers plus the current
CUDA stream.  Every step of the computation runs in the library's CUDA
kernels; there is no CPU or eager-PyTorch fallback, and calling any op
without the built library raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import _build

__all__ = [
    "FCError", "load", "build", "library_path",
    "fc_conv3x3_act_pool", "fc_conv3x3_act", "fc_linear_lse_mish", "fc_linear_lse_mish_noalloc",
    "fc_conv3x3_act_pool_host", "fc_conv3x3_act_host", "fc_host_staging_bytes",
    "fc_act_map", "fc_act_mean", "fc_scale_clamp_lse_mish", "fc_workspace_bytes", "fc_status_string", "fc_device_status", "fc_last_device_status", "fc_selftest_watchdog", "fc_version",
    "FC_OK", "FC_ERR_INVALID_ARG", "FC_ERR_UNSUPPORTED", "FC_ERR_WORKSPACE", "FC_ERR_CUDA", "FC_ERR_TIMEOUT",
    "FC_ERR_BOUNDS",
    "FC_F32", "FC_BF16", "FC_F32_3XTF32", "FC_NCHW", "FC_NHWC", "ACTS", "OPS",
]

FC_OK, FC_ERR_INVALID_ARG, FC_ERR_UNSUPPORTED, FC_ERR_WORKSPACE, FC_ERR_CUDA, FC_ERR_TIMEOUT, FC_ERR_BOUNDS = range(7)
FC_F32, FC_BF16, FC_F32_3XTF32 = 0, 1, 2
FC_NCHW, FC_NHWC = 0, 1
ACTS = {"gelu": 0, "mish": 1, "mish_mish": 2, "gelu_tanh": 3}
OPS = {"conv3x3_act_pool": 0, "conv3x3_act": 1, "linear_lse_mish": 2}

# Every symbol include/fc.h declares.
EXPORTS = ("fc_conv3x3_act_pool", "fc_conv3x3_act", "fc_conv3x3_act_pool_ex", "fc_conv3x3_act_ex",
           "fc_linear_lse_mish", "fc_linear_lse_mish_noalloc",
           "fc_conv3x3_act_pool_host", "fc_conv3x3_act_host", "fc_host_staging_bytes",
           "fc_act_map", "fc_act_mean", "fc_scale_clamp_lse_mish", "fc_workspace_bytes", "fc_workspace_bytes_ex",
           "fc_status_string", "fc_device_status", "fc_last_device_status", "fc_selftest_watchdog", "fc_version")

_lock = threading.Lock()
_lib = None


class FCError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fc_status_string(status)} (status {status})")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree for sm_103a; returns its path."""
    return _build.build(force=force)


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the CUDA library (building it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        lib = ctypes.CDLL(path)
        P, I, F, S, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_ulonglong
        conv = [P, P, P, P, I, I, I, I, I, I, I, P, S, P]
        lib.fc_conv3x3_act_pool.argtypes = conv
        lib.fc_conv3x3_act_pool.restype = I
        lib.fc_conv3x3_act.argtypes = conv
        lib.fc_conv3x3_act.restype = I
        conv_ex = [P, P, P, P, I, I, I, I, I, I, I, I, I, P, S, P]
        lib.fc_conv3x3_act_pool_ex.argtypes = conv_ex
        lib.fc_conv3x3_act_pool_ex.restype = I
        lib.fc_conv3x3_act_ex.argtypes = conv_ex
        lib.fc_conv3x3_act_ex.restype = I
        conv_host = [P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, S, P]
        lib.fc_conv3x3_act_pool_host.argtypes = conv_host
        lib.fc_conv3x3_act_pool_host.restype = I
        lib.fc_conv3x3_act_host.argtypes = conv_host
        lib.fc_conv3x3_act_host.restype = I
        lib.fc_host_staging_bytes.argtypes = [I, I, I, I, I, I, I, I, I, I]
        lib.fc_host_staging_bytes.restype = S
        lib.fc_linear_lse_mish.argtypes = [P, P, P, P, I, I, I, F, F, F, I, P, S, P]
        lib.fc_linear_lse_mish.restype = I
        L = ctypes.c_longlong
        lib.fc_act_map.argtypes = [P, P, L, I, I, P]
        lib.fc_act_map.restype = I
        lib.fc_act_mean.argtypes = [P, P, L, L, I, I, P]
        lib.fc_act_mean.restype = I
        lib.fc_scale_clamp_lse_mish.argtypes = [P, P, I, I, F, F, F, P]
        lib.fc_scale_clamp_lse_mish.restype = I
        lib.fc_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
        lib.fc_workspace_bytes.restype = S
        lib.fc_workspace_bytes_ex.argtypes = [I, I, I, I, I, I, I, I, I]
        lib.fc_workspace_bytes_ex.restype = S
        lib.fc_status_string.argtypes = [I]
        lib.fc_status_string.restype = ctypes.c_char_p
        lib.fc_device_status.argtypes = [I]
        lib.fc_device_status.restype = I
        lib.fc_last_device_status.argtypes = [P]
        lib.fc_last_device_status.restype = I
        lib.fc_selftest_watchdog.argtypes = [Z, P]
        lib.fc_selftest_watchdog.restype = I
        lib.fc_version.restype = I
        _lib = lib
        return lib


def fc_status_string(status: int) -> str:
    return load().fc_status_string(int(status)).decode()


def fc_version() -> int:
    return load().fc_version()


def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtypes, device=None, channels_last=False):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if channels_last:
        if not t.is_contiguous(memory_format=torch.channels_last):
            raise ValueError(f"{name} must be contiguous in the channels_last memory format")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _dtype_code(t, precision=None):
    """The fc_dtype of a call: the storage dtype, and for fp32 the tensor-core precision
    ("tf32", the default, or "3xtf32" for split-TF32 products)."""
    torch = _torch()
    if t.dtype == torch.bfloat16:
        if precision not in (None, "bf16"):
            raise ValueError(f"precision {precision!r} needs fp32 inputs")
        return FC_BF16
    if precision in (None, "tf32"):
        return FC_F32
    if precision == "3xtf32":
        return FC_F32_3XTF32
    raise ValueError(f"unknown precision {precision!r} (expected 'tf32' or '3xtf32')")


def _raise(status, where):
    if status != FC_OK:
        raise FCError(status, where)


def fc_workspace_bytes(op: str, n_or_m: int, cin_or_k: int, h: int, w: int, cout_or_nout: int,
                       dtype: int = FC_F32) -> int:
    """Workspace bytes a call needs on the current device (0 when the arguments are invalid)."""
    return int(load().fc_workspace_bytes(OPS[op], n_or_m, cin_or_k, h, w, cout_or_nout, dtype))


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        # the library itself checks the size (FC_ERR_WORKSPACE)
        _check(workspace, "workspace", (torch.uint8,), device)
        return workspace, workspace.numel()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def _layout_of(x, layout):
    """"nchw" / "nhwc" for x [N, C, H, W]: given, or "nhwc" when x is stored channels_last
    (and not also plainly contiguous)."""
    torch = _torch()
    if layout is None:
        cl = x.dim() == 4 and x.is_contiguous(memory_format=torch.channels_last) and not x.is_contiguous()
        return "nhwc" if cl else "nchw"
    if layout not in ("nchw", "nhwc"):
        raise ValueError(f"unknown layout {layout!r} (expected 'nchw' or 'nhwc')")
    return layout


def _conv(cname, op, x, w, b, act, out, workspace, stream, precision=None, pad=0, layout=None):
    torch = _torch()
    lib = load()
    dts = (torch.float32, torch.bfloat16)
    layout = _layout_of(x, layout)
    nhwc = layout == "nhwc"
    _check(x, "x", dts, channels_last=nhwc)
    _check(w, "w", (x.dtype,), x.device)
    _check(b, "b", (x.dtype,), x.device)
    if x.dim() != 4 or w.dim() != 4 or tuple(w.shape[1:]) != (x.shape[1], 3, 3) or b.shape != (w.shape[0],):
        raise ValueError("expected x [N,Cin,H,W], w [Cout,Cin,3,3], b [Cout]")
    N, Cin, H, W = (int(s) for s in x.shape)
    Cout = int(w.shape[0])
    pad = int(pad)
    pooled = op == "conv3x3_act_pool"
    shape = (N, Cout) if pooled else (N, Cout, H + 2 * pad - 2, W + 2 * pad - 2)
    # the full output of an NHWC call is channels_last too (logical shape N, Cout, OH, OW)
    out_cl = nhwc and not pooled
    if out is None:
        out = torch.empty(shape, dtype=torch.float32, device=x.device,
                          memory_format=torch.channels_last if out_cl else torch.contiguous_format)
    else:
        _check(out, "out", (torch.float32,), x.device, channels_last=out_cl)
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    dt = _dtype_code(x, precision)
    lay = FC_NHWC if nhwc else FC_NCHW
    with torch.cuda.device(x.device):
        nbytes = int(lib.fc_workspace_bytes_ex(OPS[op], N, Cin, H, W, Cout, pad, lay, dt))
        ws, wsb = _workspace(nbytes, x.device, workspace)
        st = getattr(lib, cname + "_ex")(x.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(), N, Cin, H, W,
                                         Cout, pad, lay, dt, ACTS[act], None if ws is None else ws.data_ptr(), wsb,
                                         _stream_handle(stream))
    _raise(st, cname)
    return out


def fc_conv3x3_act_pool(x, w, b, act: str = "gelu", out=None, workspace=None, stream=None, precision=None,
                        pad: int = 0, layout=None):
    """y[N, Cout] = mean over the OH x OW plane of act(conv3x3(x, w, padding=pad) + b), OH = H + 2 pad - 2,
    OW = W + 2 pad - 2; fp32 output.  precision (fp32 inputs): "tf32" (default) or "3xtf32".
    layout: "nchw", "nhwc" (x stored channels_last), or None to follow x's memory format."""
    return _conv("fc_conv3x3_act_pool", "conv3x3_act_pool", x, w, b, act, out, workspace, stream, precision, pad,
                 layout)


def fc_conv3x3_act(x, w, b, act: str = "mish_mish", out=None, workspace=None, stream=None, precision=None,
                   pad: int = 0, layout=None):
    """y[N, Cout, OH, OW] = act(conv3x3(x, w, padding=pad) + b), OH = H + 2 pad - 2, OW = W + 2 pad - 2;
    fp32 output, channels_last when x is.  precision (fp32 inputs): "tf32" (default) or "3xtf32".
    layout: "nchw", "nhwc" (x stored channels_last), or None to follow x's memory format."""
    return _conv("fc_conv3x3_act", "conv3x3_act", x, w, b, act, out, workspace, stream, precision, pad, layout)


def _conv_host(cname, op, x, w, b, act, out, staging, stream, precision, pad, layout, chunks, device):
    """The host-buffer conv call: x, w, b and out are CPU tensors (pinned for overlapped copies)."""
    torch = _torch()
    lib = load()
    dts = (torch.float32, torch.bfloat16)
    layout = _layout_of(x, layout)
    nhwc = layout == "nhwc"
    for t, name in ((x, "x"), (w, "w"), (b, "b")):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{name} must be a CPU tensor (host memory) for {cname}")
    if not (x.is_contiguous(memory_format=torch.channels_last) if nhwc else x.is_contiguous()):
        raise ValueError("x must be contiguous" + (" in the channels_last memory format" if nhwc else ""))
    if x.dtype not in dts or w.dtype != x.dtype or b.dtype != x.dtype or not w.is_contiguous() \
            or not b.is_contiguous():
        raise ValueError("x, w, b must be contiguous and share one dtype (float32 or bfloat16)")
    if x.dim() != 4 or w.dim() != 4 or tuple(w.shape[1:]) != (x.shape[1], 3, 3) or b.shape != (w.shape[0],):
        raise ValueError("expected x [N,Cin,H,W], w [Cout,Cin,3,3], b [Cout]")
    N, Cin, H, W = (int(s) for s in x.shape)
    Cout = int(w.shape[0])
    pad = int(pad)
    pooled = op == "conv3x3_act_pool"
    shape = (N, Cout) if pooled else (N, Cout, H + 2 * pad - 2, W + 2 * pad - 2)
    out_cl = nhwc and not pooled
    fmt = torch.channels_last if out_cl else torch.contiguous_format
    if out is None:
        if out_cl:
            n_, c_, oh_, ow_ = shape
            out = torch.empty((n_, oh_, ow_, c_), dtype=torch.float32, pin_memory=True).permute(0, 3, 1, 2)
        else:
            out = torch.empty(shape, dtype=torch.float32, pin_memory=True)
    elif out.device.type != "cpu" or out.dtype != torch.float32 or tuple(out.shape) != shape or \
            not out.is_contiguous(memory_format=fmt):
        raise ValueError(f"out must be a contiguous float32 CPU tensor of shape {shape}")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    dt = _dtype_code(x, precision)
    lay = FC_NHWC if nhwc else FC_NCHW
    with torch.cuda.device(dev):
        nbytes = int(lib.fc_host_staging_bytes(OPS[op], N, Cin, H, W, Cout, pad, lay, dt, int(chunks)))
        if staging is None:
            staging = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
        else:
            _check(staging, "staging", (torch.uint8,), dev)
        st = getattr(lib, cname + "_host")(x.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(), N, Cin, H, W,
                                           Cout, pad, lay, dt, ACTS[act], int(chunks), staging.data_ptr(),
                                           staging.numel(), _stream_handle(stream))
    _raise(st, cname + "_host")
    return out


def fc_host_staging_bytes(op: str, n: int, cin: int, h: int, w: int, cout: int, pad: int = 0, layout: str = "nchw",
                          dtype: int = FC_F32, chunks: int = 8) -> int:
    """Device staging bytes a host-buffer conv call needs on the current device (0 for invalid arguments)."""
    lay = {"nchw": FC_NCHW, "nhwc": FC_NHWC}[layout]
    return int(load().fc_host_staging_bytes(OPS[op], n, cin, h, w, cout, pad, lay, dtype, int(chunks)))


def fc_conv3x3_act_pool_host(x, w, b, act: str = "gelu", out=None, staging=None, stream=None, precision=None,
                             pad: int = 0, layout=None, chunks: int = 8, device=None):
    """fc_conv3x3_act_pool for inputs in host memory: x, w, b are CPU tensors (pinned for overlapped
    copies), the result is a CPU tensor (pinned when allocated here), valid once `stream` (default: the
    current stream of `device`, default the current device) has synchronized.  The batch moves in
    `chunks` slices whose copies overlap the kernels; `staging` is an optional uint8 device buffer of
    fc_host_staging_bytes(...) bytes."""
    return _conv_host("fc_conv3x3_act_pool", "conv3x3_act_pool", x, w, b, act, out, staging, stream, precision,
                      pad, layout, chunks, device)


def fc_conv3x3_act_host(x, w, b, act: str = "mish_mish", out=None, staging=None, stream=None, precision=None,
                        pad: int = 0, layout=None, chunks: int = 8, device=None):
    """fc_conv3x3_act for inputs in host memory (see fc_conv3x3_act_pool_host)."""
    return _conv_host("fc_conv3x3_act", "conv3x3_act", x, w, b, act, out, staging, stream, precision, pad, layout,
                      chunks, device)


def fc_linear_lse_mish(x, W, b, scale: float = 2.0, clamp_lo: float = -10.0, clamp_hi: float = 10.0,
                       out=None, workspace=None, stream=None, precision=None):
    """y[M, 1] = l * mish(l), l = logsumexp_j clamp(u + u), u = (x W^T + b) * scale.
    precision (fp32 inputs): "tf32" (default) or "3xtf32" (split TF32, fp32-level error)."""
    torch = _torch()
    lib = load()
    _check(x, "x", (torch.float32, torch.bfloat16))
    _check(W, "W", (x.dtype,), x.device)
    _check(b, "b", (x.dtype,), x.device)
    if x.dim() != 2 or W.dim() != 2 or W.shape[1] != x.shape[1] or b.shape != (W.shape[0],):
        raise ValueError("expected x [M,K], W [Nout,K], b [Nout]")
    M, K = (int(s) for s in x.shape)
    Nout = int(W.shape[0])
    if out is None:
        out = torch.empty((M, 1), dtype=torch.float32, device=x.device)
    else:
        _check(out, "out", (torch.float32,), x.device)
        if out.numel() != M:
            raise ValueError(f"out must hold {M} values")
    dt = _dtype_code(x, precision)
    with torch.cuda.device(x.device):
        nbytes = int(lib.fc_workspace_bytes(OPS["linear_lse_mish"], M, K, 1, 1, Nout, dt))
        ws, wsb = _workspace(nbytes, x.device, workspace)
        st = lib.fc_linear_lse_mish(x.data_ptr(), W.data_ptr(), b.data_ptr(), out.data_ptr(), M, K, Nout,
                                    float(scale), float(clamp_lo), float(clamp_hi), dt,
                                    None if ws is None else ws.data_ptr(), wsb, _stream_handle(stream))
    _raise(st, "fc_linear_lse_mish")
    return out


def fc_device_status(clear: bool = True) -> int:
    """Synchronize the current device and return (and by default clear) its watchdog word."""
    return int(load().fc_device_status(1 if clear else 0))


def fc_last_device_status(stream=None) -> int:
    """The watchdog word once `stream`'s enqueued work has finished (other streams are not waited
    for, and the word is not cleared)."""
    return int(load().fc_last_device_status(_stream_handle(stream)))


def fc_selftest_watchdog(budget_cycles: int, stream=None) -> None:
    """Enqueue the watchdog self-test kernel (a wait that must time out)."""
    _raise(load().fc_selftest_watchdog(int(budget_cycles), _stream_handle(stream)), "fc_selftest_watchdog")


def fc_linear_lse_mish_noalloc(x, W, b, scale: float = 2.0, clamp_lo: float = -10.0, clamp_hi: float = 10.0,
                               out=None, stream=None):
    """fc_linear_lse_mish for callers that cannot allocate device memory: the
    library's own static 1 MiB device scratch replaces the workspace.  Only
    `out` is allocated here when not given; pass `out` to allocate nothing.
    Calls that overlap on the GPU share that scratch and race."""
    torch = _torch()
    lib = load()
    fn = lib.fc_linear_lse_mish_noalloc
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_float] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    _check(x, "x", (torch.float32,))
    _check(W, "W", (torch.float32,), x.device)
    _check(b, "b", (torch.float32,), x.device)
    if x.dim() != 2 or W.dim() != 2 or W.shape[1] != x.shape[1] or b.shape != (W.shape[0],):
        raise ValueError("expected x [M,K], W [Nout,K], b [Nout]")
    M, K = (int(s) for s in x.shape)
    Nout = int(W.shape[0])
    if out is None:
        out = torch.empty((M, 1), dtype=torch.float32, device=x.device)
    else:
        _check(out, "out", (torch.float32,), x.device)
        if out.numel() != M:
            raise ValueError(f"out must hold {M} values")
    with torch.cuda.device(x.device):
        st = fn(x.data_ptr(), W.data_ptr(), b.data_ptr(), out.data_ptr(), M, K, Nout, float(scale),
                float(clamp_lo), float(clamp_hi), _stream_handle(stream))
    _raise(st, "fc_linear_lse_mish_noalloc")
    return out


def fc_act_map(v, act: str = "mish_mish", out=None, stream=None):
    """out = act(v) elementwise, fp32 (the elementwise epilogue over a computed conv output)."""
    torch = _torch()
    lib = load()
    _check(v, "v", (torch.float32, torch.bfloat16))
    if out is None:
        out = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    else:
        _check(out, "out", (torch.float32,), v.device)
        if out.numel() != v.numel():
            raise ValueError(f"out must hold {v.numel()} values")
    with torch.cuda.device(v.device):
        st = lib.fc_act_map(v.data_ptr(), out.data_ptr(), v.numel(), _dtype_code(v), ACTS[act],
                            _stream_handle(stream))
    _raise(st, "fc_act_map")
    return out


def fc_act_mean(v, act: str = "gelu", out=None, stream=None):
    """y[..] = mean over the last two dims of act(v): v (N, C, H, W) -> (N, C) fp32."""
    torch = _torch()
    lib = load()
    _check(v, "v", (torch.float32, torch.bfloat16))
    if v.dim() < 2:
        raise ValueError("expected at least two dims (the plane is the last two)")
    lead = tuple(int(s) for s in v.shape[:-2])
    planes = 1
    for s in lead:
        planes *= s
    plane = int(v.shape[-2]) * int(v.shape[-1])
    if out is None:
        out = torch.empty(lead, dtype=torch.float32, device=v.device)
    else:
        _check(out, "out", (torch.float32,), v.device)
        if out.numel() != planes:
            raise ValueError(f"out must hold {planes} values")
    with torch.cuda.device(v.device):
        st = lib.fc_act_mean(v.data_ptr(), out.data_ptr(), planes, plane, _dtype_code(v), ACTS[act],
                             _stream_handle(stream))
    _raise(st, "fc_act_mean")
    return out


def fc_scale_clamp_lse_mish(t, scale: float = 2.0, clamp_lo: float = -10.0, clamp_hi: float = 10.0, out=None,
                            stream=None):
    """y[M, 1] = l * mish(l), l = logsumexp_j clamp(t * scale + t * scale) for a computed t [M, N] fp32."""
    torch = _torch()
    lib = load()
    _check(t, "t", (torch.float32,))
    if t.dim() != 2:
        raise ValueError("expected t [M, N]")
    M, N = (int(s) for s in t.shape)
    if out is None:
        out = torch.empty((M, 1), dtype=torch.float32, device=t.device)
    else:
        _check(out, "out", (torch.float32,), t.device)
        if out.numel() != M:
            raise ValueError(f"out must hold {M} values")
    with torch.cuda.device(t.device):
        st = lib.fc_scale_clamp_lse_mish(t.data_ptr(), out.data_ptr(), M, N, float(scale), float(clamp_lo),
                                         float(clamp_hi), _stream_handle(stream))
    _raise(st, "fc_scale_clamp_lse_mish")
    return out
