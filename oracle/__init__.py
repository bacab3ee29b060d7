"""The oracle: plain fp64 CPU implementation of the three fused chains.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``gemm_activation_reduction_gb300``) never imports it and has no
CPU fallback.

``fc_oracle.c`` holds the arithmetic; this module compiles it with gcc
(``-O2``, OpenMP, no fast-math) and wraps it with ctypes.  ``brute.py`` is a
second, independent pure-Python statement used only to pin the C oracle on
tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

ACT = {"none": -1, "gelu": 0, "mish": 1, "mish_mish": 2, "gelu_tanh": 3}


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (skipped when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        for name in ("oracle_gelu", "oracle_softplus", "oracle_mish"):
            getattr(lib, name).argtypes = [D]
            getattr(lib, name).restype = D
        lib.oracle_act.argtypes = [I, D]
        lib.oracle_act.restype = D
        lib.oracle_act_map.argtypes = [P, P, L, I]
        lib.oracle_act_map.restype = None
        lib.oracle_act_mean.argtypes = [P, P, L, L, I]
        lib.oracle_act_mean.restype = None
        lib.oracle_scale_clamp_lse_mish_rows.argtypes = [P, I, I, D, D, D, P]
        lib.oracle_scale_clamp_lse_mish_rows.restype = I
        lib.oracle_conv3x3_point.argtypes = [P, P, P, I, I, I, I, I, I, I, I]
        lib.oracle_conv3x3_point.restype = D
        lib.oracle_conv3x3_preact.argtypes = [P, P, P, P, I, I, I, I, I, I]
        lib.oracle_conv3x3_act.argtypes = [P, P, P, P, I, I, I, I, I, I, I]
        lib.oracle_conv3x3_act_at.argtypes = [P, P, P, I, I, I, I, I, I, I, P, L, P]
        lib.oracle_conv3x3_act_pool.argtypes = [P, P, P, P, I, I, I, I, I, I, I]
        lib.oracle_conv3x3_act_pool_at.argtypes = [P, P, P, I, I, I, I, I, I, I, P, L, P]
        lib.oracle_logsumexp.argtypes = [P, L]
        lib.oracle_logsumexp.restype = D
        lib.oracle_linear_lse_mish_rows.argtypes = [P, P, P, I, I, I, D, D, D, P, L, P, P]
        lib.oracle_linear_lse_mish_rows.restype = I
        lib.oracle_threads.restype = I
        _lib = lib
        return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _indices(idx, limit, what):
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= limit):
        raise IndexError(f"{what} index out of range [0, {limit})")
    return idx


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return _load().oracle_threads()


def set_threads(n: int) -> None:
    """Use n OpenMP threads from now on (results do not depend on it)."""
    lib = _load()
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_set_threads(int(n))


def gelu(v: float) -> float:
    return _load().oracle_gelu(float(v))


def softplus(v: float) -> float:
    return _load().oracle_softplus(float(v))


def mish(v: float) -> float:
    return _load().oracle_mish(float(v))


def act(name: str, v: float) -> float:
    return _load().oracle_act(ACT[name], float(v))


def act_map(v, act: str) -> np.ndarray:
    """act applied elementwise (the Conv->Mish->Mish page's elementwise epilogue), fp64."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.float64)
    _load().oracle_act_map(_p(v), _p(out), v.size, ACT[act])
    return out


def act_mean(v, act: str) -> np.ndarray:
    """Mean of act over each trailing (H, W) plane of v (N, C, H, W) -> (N, C), fp64 (the
    Conv->GELU->pool page's fused GELU + global-average-pool epilogue)."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    planes = int(np.prod(v.shape[:-2]))
    plane = int(v.shape[-2] * v.shape[-1])
    out = np.empty(v.shape[:-2], np.float64)
    _load().oracle_act_mean(_p(v), _p(out), planes, plane, ACT[act])
    return out


def scale_clamp_lse_mish(y, scale=2.0, lo=-10.0, hi=10.0) -> np.ndarray:
    """The Linear page's row kernel on a computed (M, N) output: t = clamp(2 scale y, lo, hi),
    l = logsumexp_row(t), out (M, 1) = l * mish(l), fp64."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    M, N = y.shape
    out = np.empty((M, 1), np.float64)
    if _load().oracle_scale_clamp_lse_mish_rows(_p(y), M, N, float(scale), float(lo), float(hi), _p(out)) != 0:
        raise MemoryError("oracle scratch")
    return out


def logsumexp(t) -> float:
    t = np.ascontiguousarray(t, dtype=np.float64)
    return _load().oracle_logsumexp(_p(t), t.size)


def tf32_round_nearest(a) -> np.ndarray:
    """fp32 values rounded to TF32 (10 stored mantissa bits) to nearest, ties away from zero:
    add half a TF32 unit in the last place to the magnitude bits and drop the 13 low bits (a carry
    into the exponent is the correct rounding up).  Diagnostic mode: an oracle run on operands
    rounded this way differs from a contraction that rounds its operands the same way only by the
    order and precision of its accumulation.  Finite inputs."""
    u = np.array(a, dtype=np.float32).view(np.uint32)   # a copy, any shape (0-d included)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def tf32_truncate(a) -> np.ndarray:
    """fp32 values with the 13 low mantissa bits dropped: TF32 rounded toward zero."""
    u = np.array(a, dtype=np.float32).view(np.uint32)
    return (u & np.uint32(0xFFFFE000)).view(np.float32)


def _out_hw(H, W, pad):
    if pad < 0 or H + 2 * pad < 3 or W + 2 * pad < 3:
        raise ValueError("padding must be >= 0 and leave an output of at least 1 x 1")
    return H + 2 * pad - 2, W + 2 * pad - 2


def conv3x3_preact(x, w, b, pad=0):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    OH, OW = _out_hw(H, W, pad)
    out = np.empty((N, Cout, OH, OW), dtype=np.float64)
    _load().oracle_conv3x3_preact(_p(x), _p(w), _p(b), _p(out), N, Cin, H, W, Cout, pad)
    return out


def conv3x3_act(x, w, b, act="mish_mish", pad=0):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    OH, OW = _out_hw(H, W, pad)
    out = np.empty((N, Cout, OH, OW), dtype=np.float64)
    _load().oracle_conv3x3_act(_p(x), _p(w), _p(b), _p(out), N, Cin, H, W, Cout, pad, ACT[act])
    return out


def conv3x3_act_at(x, w, b, flat_idx, act="mish_mish", pad=0):
    """act(conv) at flat indices into the (N, Cout, H+2p-2, W+2p-2) output."""
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    OH, OW = _out_hw(H, W, pad)
    idx = _indices(flat_idx, N * Cout * OH * OW, "output")
    out = np.empty(idx.size, dtype=np.float64)
    _load().oracle_conv3x3_act_at(_p(x), _p(w), _p(b), N, Cin, H, W, Cout, pad, ACT[act],
                                  _p(idx), idx.size, _p(out))
    return out


def conv3x3_act_pool(x, w, b, act="gelu", pad=0):
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    _out_hw(H, W, pad)
    y = np.empty((N, Cout), dtype=np.float64)
    _load().oracle_conv3x3_act_pool(_p(x), _p(w), _p(b), _p(y), N, Cin, H, W, Cout, pad, ACT[act])
    return y


def conv3x3_act_pool_at(x, w, b, flat_nc, act="gelu", pad=0):
    """Pooled output at flat (n * Cout + co) indices."""
    x, w, b = _f32(x), _f32(w), _f32(b)
    N, Cin, H, W = x.shape
    Cout = w.shape[0]
    _out_hw(H, W, pad)
    idx = _indices(flat_nc, N * Cout, "pooled output")
    out = np.empty(idx.size, dtype=np.float64)
    _load().oracle_conv3x3_act_pool_at(_p(x), _p(w), _p(b), N, Cin, H, W, Cout, pad, ACT[act],
                                       _p(idx), idx.size, _p(out))
    return out


def linear_lse_mish(x, Wt, b, scale=2.0, clamp_lo=-10.0, clamp_hi=10.0, rows=None,
                    return_lse=False):
    """y[m] = l * mish(l), l = logsumexp_j clamp(2 * (scale * (x W^T + b)))[m, j]."""
    x, Wt, b = _f32(x), _f32(Wt), _f32(b)
    M, K = x.shape
    Nout = Wt.shape[0]
    if rows is None:
        r, count = None, M
    else:
        r = _indices(rows, M, "row")
        count = r.size
    y = np.empty(count, dtype=np.float64)
    lse = np.empty(count, dtype=np.float64)
    rc = _load().oracle_linear_lse_mish_rows(
        _p(x), _p(Wt), _p(b), M, K, Nout, float(scale), float(clamp_lo), float(clamp_hi),
        None if r is None else _p(r), count, _p(y), _p(lse))
    if rc != 0:
        raise MemoryError("oracle: row scratch allocation failed")
    return (y, lse) if return_lse else y
