"""Parity of the CUDA path with the fp64 oracle, element by element, on the
same seeded inputs (GPU only; every call goes through the C ABI).

Tolerance (the one the fused-op contract states): |gpu - ref| <= tol * (1 + |ref|)
with tol = 2e-3 for fp32 inputs on TF32 tensor cores and 2e-2 for bf16 inputs.
Small and ragged shapes are checked in full; the five workloads at full size
are checked in the launch configuration the benchmark times, on outputs the
oracle computes one by one (random samples plus every border row/column of
a few planes).
"""
import ctypes
import math

import numpy as np
import pytest

import fc_inputs
import oracle

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-3, "bf16": 2e-2}


def _dev(arr):
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def _check(got, ref, tol, what):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    i = int(np.argmax(err))
    assert err[i] <= tol, f"{what}: scaled error {err[i]:.3e} > {tol} at {i} (gpu {got[i]!r}, ref {ref[i]!r})"
    return float(err[i])


# ------------------------------------------------------------------ conv + pool

POOL_SHAPES = [
    # (N, Cin, H, W, Cout, dtype, act)
    (2, 8, 32, 32, 64, "f32", "gelu"),       # the tiny workload, exhaustively
    (1, 1, 3, 3, 32, "f32", "gelu"),         # degenerate: a 1x1 output plane
    (3, 3, 19, 13, 32, "f32", "gelu"),       # ragged rows and columns, Cin < one K block
    (2, 13, 20, 37, 96, "f32", "gelu"),      # Cin not a multiple of 8, Cout = 96
    (1, 8, 40, 17, 256, "f32", "gelu"),      # Cout = 256, resident weights
    (1, 64, 21, 18, 128, "f32", "gelu"),     # streamed weights
    (2, 8, 23, 29, 64, "f32", "mish"),
    (2, 16, 18, 20, 64, "bf16", "gelu"),
    (1, 128, 12, 12, 256, "bf16", "gelu"),   # streamed bf16 weights
    (1, 24, 35, 9, 32, "bf16", "gelu"),      # Cin not a multiple of 16
    (2, 5, 21, 26, 48, "f32", "gelu"),       # Cout = 48 (a multiple of 16, not of 32)
    (1, 16, 19, 30, 16, "bf16", "gelu"),     # the smallest Cout, 16
    (2, 8, 33, 30, 64, "f32", "gelu_tanh"),  # tanh-approximate GELU
    (1, 40, 17, 19, 256, "bf16", "gelu_tanh"),
    # output channel counts that are not multiples of 16 (run padded to the next one)
    (2, 8, 21, 19, 40, "f32", "gelu"),
    (3, 5, 13, 17, 3, "f32", "gelu"),
    (1, 3, 10, 9, 1, "bf16", "mish"),
    (2, 12, 18, 22, 200, "f32", "gelu"),     # CTA pairs, 104 channels each
    (1, 24, 15, 16, 145, "bf16", "gelu_tanh"),
    # CTA pairs whose column-strip count is a multiple of 4 (the pair's two tiles at strips j and
    # j + CS/2), with a ragged last strip or row block, and the neighbouring counts that keep the
    # plain order
    (2, 16, 34, 34, 256, "bf16", "gelu"),    # OW 32: 4 strips
    (1, 16, 21, 61, 144, "bf16", "mish"),    # OW 59: 8 strips, the last one 3 wide
    (3, 8, 19, 50, 160, "f32", "gelu"),      # OW 48: 6 strips
    (1, 8, 40, 66, 256, "f32", "gelu"),      # OW 64: 8 strips, 3 row blocks (the last 6 rows)
]


@pytest.mark.parametrize("shape", POOL_SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-{s[5]}-{s[6]}")
def test_conv_pool_small(cuda_lib, shape):
    N, Cin, H, W, Cout, dt, act = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    y = cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act).cpu().numpy()
    ref = oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], act)
    _check(y, ref, TOL[dt], f"pool {shape}")


ACT_SHAPES = [
    (1, 3, 11, 13, 32, "f32", "mish_mish"),
    (2, 64, 20, 19, 128, "f32", "mish_mish"),
    (1, 8, 34, 34, 64, "f32", "mish_mish"),
    (1, 5, 17, 21, 96, "f32", "gelu"),
    (1, 32, 14, 12, 64, "bf16", "mish_mish"),
    (2, 16, 19, 10, 256, "bf16", "mish"),
    (1, 7, 9, 140, 80, "f32", "mish_mish"),  # Cout = 80; rows wider than one 128-pixel tile
    (1, 9, 13, 150, 64, "f32", "gelu_tanh"),
    (2, 8, 12, 140, 40, "f32", "mish_mish"),   # Cout not a multiple of 16
    (1, 6, 11, 21, 7, "bf16", "gelu"),
    (1, 16, 9, 133, 250, "f32", "mish"),       # CTA pairs, padded to 256
]


@pytest.mark.parametrize("shape", ACT_SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-{s[5]}-{s[6]}")
def test_conv_act_small(cuda_lib, shape):
    N, Cin, H, W, Cout, dt, act = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    y = cuda_lib.fc_conv3x3_act(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act).cpu().numpy()
    ref = oracle.conv3x3_act(d["x32"], d["w32"], d["b32"], act)
    _check(y, ref, TOL[dt], f"act {shape}")


# ------------------------------------------------------------------ split TF32 (FC_F32_3XTF32)

# Tolerance: each product of TF32 parts misses only lo*lo and the parts' own rounding (about
# 3 * 2^-22 of |x w|), the fp32 accumulation of K <= 1152 terms adds about 2^-24 of the running
# sum per addition, and the activations' approximate exponential / reciprocal about 1e-6: the
# outputs land within a few 1e-6.  2e-5 (1 + |ref|) is 100x tighter than the TF32 bar and 5x
# tighter than the pages' own atol = rtol = 1e-4, which their TF32-backed results missed.
TOL_X3 = 2e-5

X3_SHAPES = [
    # (N, Cin, H, W, Cout, act, pool)
    (2, 8, 32, 32, 64, "gelu", True),          # the tiny workload
    (1, 13, 20, 37, 96, "gelu", True),         # Cin not a multiple of 8, ragged edges
    (1, 64, 21, 18, 128, "mish", True),        # 24 K stages, streamed weights
    (1, 8, 40, 17, 256, "gelu", True),         # CTA pairs
    (1, 3, 11, 13, 40, "gelu_tanh", True),     # row pitch not a 16-byte multiple: plain-load staging
    (2, 5, 13, 150, 64, "mish_mish", False),   # two-row tiles, rows wider than one tile
    (1, 64, 12, 140, 128, "mish_mish", False), # the Mish->Mish page's channel counts
    (1, 16, 9, 133, 200, "mish", False),       # CTA pairs, padded Cout
    (1, 3, 9, 13, 40, "gelu", False),          # plain-load staging, full output
]


@pytest.mark.parametrize("shape", X3_SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"-{s[5]}-{'pool' if s[6] else 'act'}")
def test_conv_split_tf32_small(cuda_lib, shape):
    N, Cin, H, W, Cout, act, pool = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout)
    f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
    y = f(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act, precision="3xtf32").cpu().numpy()
    ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x"], d["w"], d["b"], act)
    _check(y, ref, TOL_X3, f"3xtf32 {shape}")


def test_split_tf32_is_far_more_accurate_than_tf32(cuda_lib):
    """Same inputs, both precisions: the split-TF32 error is at least 30x below the TF32 error
    (TF32 rounds each operand to 11 significant bits, so its error is ~2^-11 of sum |x w|)."""
    d = fc_inputs.conv_inputs(1, 64, 12, 140, 128)
    x, w, b = _dev(d["x"]), _dev(d["w"]), _dev(d["b"])
    ref = oracle.conv3x3_act(d["x"], d["w"], d["b"], "mish")
    e1 = np.abs(cuda_lib.fc_conv3x3_act(x, w, b, act="mish").cpu().numpy() - ref).max()
    e3 = np.abs(cuda_lib.fc_conv3x3_act(x, w, b, act="mish", precision="3xtf32").cpu().numpy() - ref).max()
    assert e3 * 30 < e1, (e1, e3)


def test_split_tf32_rejects_bf16_inputs(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(1, 8, 16, 16, 64, "bf16")
    with pytest.raises(ValueError):
        cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), precision="3xtf32")
    lib = cuda_lib.load()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    v = torch.zeros(1024, device="cuda")
    # split TF32 needs fp32 rows with a 16-byte pitch (K % 4 == 0)
    assert lib.fc_linear_lse_mish(v.data_ptr(), v.data_ptr(), v.data_ptr(), v.data_ptr(), 4, 6, 8, 2.0, -1.0, 1.0,
                                  cuda_lib.FC_F32_3XTF32, None, 0, s) == cuda_lib.FC_ERR_UNSUPPORTED
    dl = fc_inputs.linear_inputs(8, 64, 32, dtype="bf16")
    with pytest.raises(ValueError):
        cuda_lib.fc_linear_lse_mish(_dev(dl["x"]), _dev(dl["W"]), _dev(dl["b"]), precision="3xtf32")


LIN_X3_SHAPES = [
    # (M, K, Nout, input scale)
    (1, 4, 1, 1.0),            # degenerate
    (100, 132, 300, 1.0),      # one 128-row block: single CTAs; K not a multiple of 32
    (263, 212, 6, 8.0),        # heavy cancellation: TF32 alone misses the N(0, 1) tolerance here
    (300, 520, 700, 1.0),      # CTA pairs, ragged rows and columns
    (129, 64, 513, 40.0),      # the clamp active on most logits
]


@pytest.mark.parametrize("shape", LIN_X3_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linear_split_tf32_small(cuda_lib, shape):
    """Split TF32 for the Linear chain: fp32-level agreement with the exact oracle (2e-5), where
    plain TF32 misses it by orders of magnitude on the scaled cases."""
    M, K, Nout, sx = shape
    d = fc_inputs.linear_inputs(M, K, Nout)
    x = (d["x32"] * np.float32(sx)).astype(np.float32)
    ref = oracle.linear_lse_mish(x, d["W32"], d["b32"])
    y = cuda_lib.fc_linear_lse_mish(_dev(x), _dev(d["W"]), _dev(d["b"]), precision="3xtf32").cpu().numpy()
    _check(y, ref, TOL_X3, f"linear 3xtf32 {shape}")


# ------------------------------------------------------------------ zero padding

PAD_SHAPES = [
    # (N, Cin, H, W, Cout, pad, dtype, act, pool)
    (2, 8, 32, 32, 64, 1, "f32", "gelu", True),        # 'same' conv, TMA staging, column shift 3
    (1, 13, 20, 36, 96, 2, "f32", "gelu", True),       # shift 2, ragged edges
    (1, 5, 17, 24, 32, 3, "f32", "mish", True),        # shift 1
    (1, 6, 15, 20, 48, 4, "f32", "gelu", True),        # shift 0: the unshifted kernel, negative start
    (1, 3, 9, 11, 40, 5, "f32", "gelu_tanh", True),    # plain-load staging, wide border
    (2, 16, 18, 24, 64, 1, "bf16", "gelu", True),      # bf16, shift 7
    (1, 8, 40, 16, 256, 1, "f32", "gelu", True),       # CTA pairs
    (1, 40, 12, 32, 256, 2, "bf16", "gelu", True),     # CTA pairs, bf16, streamed weights
    (1, 2, 1, 2, 16, 1, "f32", "gelu", True),          # input smaller than the kernel: 1 x 2 output
    (2, 8, 12, 140, 64, 1, "f32", "mish_mish", False), # two-row tiles, rows wider than one tile
    (1, 64, 9, 132, 128, 1, "f32", "mish_mish", False),# the Mish->Mish page's channel counts
    (1, 16, 9, 136, 64, 3, "bf16", "mish", False),     # bf16, shift 5
    (1, 16, 7, 128, 200, 1, "f32", "mish", False),     # CTA pairs, padded Cout
    (1, 3, 5, 7, 24, 2, "f32", "gelu", False),         # plain-load staging, full output
    (1, 16, 20, 62, 256, 1, "bf16", "gelu", True),     # CTA pairs at strips j and j + 4 (8 strips), shift 7
    (2, 8, 18, 30, 160, 1, "f32", "mish", True),       # CTA pairs at strips j and j + 2 (4 strips), shift 3
]


@pytest.mark.parametrize("shape", PAD_SHAPES,
                         ids=lambda s: "x".join(map(str, s[:5])) + f"-p{s[5]}-{s[6]}-{s[7]}-{'pool' if s[8] else 'act'}")
def test_conv_padded_small(cuda_lib, shape):
    N, Cin, H, W, Cout, pad, dt, act, pool = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
    y = f(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act, pad=pad).cpu().numpy()
    ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x32"], d["w32"], d["b32"], act, pad=pad)
    assert y.shape == ref.shape
    _check(y, ref, TOL[dt], f"pad {shape}")


def test_conv_padded_split_tf32(cuda_lib):
    d = fc_inputs.conv_inputs(1, 12, 14, 24, 64)
    for pool, pad in ((True, 1), (False, 2)):
        f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
        y = f(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act="gelu", pad=pad, precision="3xtf32").cpu().numpy()
        ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x"], d["w"], d["b"], "gelu", pad=pad)
        _check(y, ref, TOL_X3, f"pad {pad} 3xtf32")


def test_conv_pad_zero_matches_unpadded_entry_point_bit_for_bit(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(2, 8, 20, 36, 64)
    x, w, b = _dev(d["x"]), _dev(d["w"]), _dev(d["b"])
    lib = cuda_lib.load()
    y0 = torch.empty((2, 64), device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    nb = lib.fc_workspace_bytes(0, 2, 8, 20, 36, 64, 0)
    assert nb == lib.fc_workspace_bytes_ex(0, 2, 8, 20, 36, 64, 0, cuda_lib.FC_NCHW, 0)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert lib.fc_conv3x3_act_pool(x.data_ptr(), w.data_ptr(), b.data_ptr(), y0.data_ptr(), 2, 8, 20, 36, 64, 0, 0,
                                   ws.data_ptr(), nb, s) == 0
    y1 = cuda_lib.fc_conv3x3_act_pool(x, w, b, pad=0)
    assert torch.equal(y0, y1)


def test_conv_pad_arguments_are_checked(cuda_lib):
    import torch
    lib = cuda_lib.load()
    v = torch.zeros(4096, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = v.data_ptr()
    call = lambda H, W, pad, lay=0: lib.fc_conv3x3_act_ex(p, p, p, p, 1, 1, H, W, 16, pad, lay, 0, 0, None, 0, s)
    assert call(4, 4, -1) == cuda_lib.FC_ERR_INVALID_ARG
    assert call(4, 4, 65) == cuda_lib.FC_ERR_INVALID_ARG
    assert call(1, 1, 0) == cuda_lib.FC_ERR_INVALID_ARG       # no output
    assert call(4, 4, 0, 2) == cuda_lib.FC_ERR_INVALID_ARG    # unknown layout
    assert lib.fc_workspace_bytes_ex(1, 1, 1, 4, 4, 16, -1, 0, 0) == 0
    assert lib.fc_workspace_bytes_ex(2, 1, 1, 4, 4, 16, 1, 0, 0) == 0   # not a conv op
    assert lib.fc_workspace_bytes_ex(1, 1, 1, 4, 4, 16, 1, 5, 0) == 0   # unknown layout
    torch.cuda.synchronize()


# ------------------------------------------------------------------ NHWC (channels_last) input

NHWC_SHAPES = [
    # (N, Cin, H, W, Cout, pad, dtype, act, pool, precision)
    (2, 8, 32, 32, 64, 0, "f32", "gelu", True, None),        # TMA channel boxes straight into the strip
    (1, 13, 20, 37, 96, 0, "f32", "gelu", True, None),       # 13 channels: not 16-byte rows, plain loads
    (2, 16, 18, 20, 64, 0, "bf16", "gelu", True, None),
    (1, 8, 40, 17, 256, 0, "f32", "gelu", True, None),       # CTA pairs
    (2, 8, 21, 19, 64, 1, "f32", "mish", True, None),        # padding: negative box origins
    (1, 12, 14, 24, 64, 2, "f32", "gelu", True, "3xtf32"),   # split TF32 with padding
    (2, 64, 12, 140, 128, 0, "f32", "mish_mish", False, None),  # two-row tiles
    (1, 32, 9, 133, 64, 1, "bf16", "mish_mish", False, None),
    (1, 16, 9, 131, 40, 0, "f32", "mish", False, None),      # Cout 40: a partial last slice
    (1, 8, 7, 30, 7, 1, "f32", "gelu", False, None),         # Cout 7: scalar stores
    (1, 16, 9, 130, 200, 1, "f32", "mish", False, None),     # CTA pairs
    (1, 3, 11, 13, 32, 1, "f32", "gelu_tanh", False, None),  # 3 channels: plain loads
    (1, 24, 10, 40, 64, 0, "f32", "mish_mish", False, "3xtf32"),
    (1, 16, 20, 34, 256, 0, "bf16", "gelu", True, None),     # CTA pairs at strips j and j + 2 (4 strips)
    (1, 8, 19, 64, 160, 1, "f32", "gelu", True, None),       # CTA pairs at strips j and j + 4, padding
]


def _nhwc(arr):
    """A CUDA tensor of logical shape [N, C, H, W] stored channels_last, from an NCHW array."""
    import torch
    t = _dev(np.ascontiguousarray(np.transpose(arr, (0, 2, 3, 1))))
    return t.permute(0, 3, 1, 2)


@pytest.mark.parametrize("shape", NHWC_SHAPES,
                         ids=lambda s: "x".join(map(str, s[:5])) + f"-p{s[5]}-{s[6]}-{s[7]}-{'pool' if s[8] else 'act'}-{s[9]}")
def test_conv_nhwc_small(cuda_lib, shape):
    import torch
    N, Cin, H, W, Cout, pad, dt, act, pool, prec = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    x = _nhwc(d["x"])
    assert x.is_contiguous(memory_format=torch.channels_last) and not x.is_contiguous()
    f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
    y = f(x, _dev(d["w"]), _dev(d["b"]), act=act, pad=pad, precision=prec)
    if not pool:
        assert y.is_contiguous(memory_format=torch.channels_last)
    y = y.cpu().numpy()
    ref = (oracle.conv3x3_act_pool if pool else oracle.conv3x3_act)(d["x32"], d["w32"], d["b32"], act, pad=pad)
    assert y.shape == ref.shape
    _check(y, ref, TOL_X3 if prec == "3xtf32" else TOL[dt], f"nhwc {shape}")


def test_conv_nhwc_matches_nchw_bit_for_bit_where_the_arithmetic_is_the_same(cuda_lib):
    """bf16 NHWC and NCHW calls stage the same operands and sum in the same order."""
    import torch
    d = fc_inputs.conv_inputs(2, 32, 12, 136, 64, "bf16")
    w, b = _dev(d["w"]), _dev(d["b"])
    y_nchw = cuda_lib.fc_conv3x3_act(_dev(d["x"]), w, b, act="mish")
    y_nhwc = cuda_lib.fc_conv3x3_act(_nhwc(d["x"]), w, b, act="mish")
    assert torch.equal(y_nchw, y_nhwc.contiguous())
    p_nchw = cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), w, b)
    p_nhwc = cuda_lib.fc_conv3x3_act_pool(_nhwc(d["x"]), w, b)
    assert torch.equal(p_nchw, p_nhwc)


# ------------------------------------------------------------------ randomized sweep

def _random_conv_cases(n, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        pad = int(rng.choice([0, 0, 1, 2, 3]))
        H, W = int(rng.integers(1, 41)), int(rng.integers(1, 41))
        if H + 2 * pad < 3 or W + 2 * pad < 3:
            continue
        cases.append(dict(N=int(rng.integers(1, 4)), Cin=int(rng.integers(1, 41)), H=H, W=W,
                          Cout=int(rng.choice([int(rng.integers(1, 129)), int(rng.integers(129, 257))])), pad=pad,
                          prec=str(rng.choice(["tf32", "tf32", "bf16", "3xtf32"])),
                          layout=str(rng.choice(["nchw", "nhwc"])), pool=bool(rng.integers(0, 2)),
                          act=str(rng.choice(["gelu", "mish", "mish_mish", "gelu_tanh"]))))
    return cases


@pytest.mark.parametrize("case", _random_conv_cases(120), ids=lambda c: "{N}x{Cin}x{H}x{W}-c{Cout}-p{pad}-{prec}-{layout}-{act}-{p}".format(p="pool" if c["pool"] else "act", **c))
def test_conv_random_shapes(cuda_lib, case):
    """Seeded random shapes, paddings, channel counts (single CTAs and pairs), precisions, layouts and
    activations against the oracle: the plan and kernels have no unexercised combination."""
    c = case
    bf16 = c["prec"] == "bf16"
    d = fc_inputs.conv_inputs(c["N"], c["Cin"], c["H"], c["W"], c["Cout"], "bf16" if bf16 else "f32")
    x = _nhwc(d["x"]) if c["layout"] == "nhwc" else _dev(d["x"])
    f = cuda_lib.fc_conv3x3_act_pool if c["pool"] else cuda_lib.fc_conv3x3_act
    y = f(x, _dev(d["w"]), _dev(d["b"]), act=c["act"], pad=c["pad"], precision=None if bf16 else c["prec"])
    y = y.cpu().numpy()
    o = oracle.conv3x3_act_pool if c["pool"] else oracle.conv3x3_act
    ref = o(d["x32"], d["w32"], d["b32"], c["act"], pad=c["pad"])
    assert y.shape == ref.shape
    tol = TOL["bf16"] if bf16 else (TOL_X3 if c["prec"] == "3xtf32" else TOL["f32"])
    _check(y, ref, tol, f"random {c}")


# ------------------------------------------------------------------ linear chain

LIN_SHAPES = [
    # (M, K, Nout, x scale)
    (1, 4, 1, 1.0),
    (3, 36, 17, 1.0),
    (130, 520, 300, 1.0),     # ragged in M, K and Nout
    (129, 64, 513, 30.0),     # clamp active on most entries
    (256, 1024, 2048, 1.0),
]


@pytest.mark.parametrize("shape", LIN_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_linear_small(cuda_lib, shape):
    M, K, Nout, sx = shape
    d = fc_inputs.linear_inputs(M, K, Nout)
    x = (d["x"] * np.float32(sx)).astype(np.float32)
    y = cuda_lib.fc_linear_lse_mish(_dev(x), _dev(d["W"]), _dev(d["b"])).cpu().numpy()
    ref = oracle.linear_lse_mish(x, d["W"], d["b"])
    _check(y, ref, TOL["f32"], f"linear {shape}")


LIN_SHAPES_BF16 = [
    # (M, K, Nout, x scale): single CTAs (M <= 128) and CTA pairs, ragged sizes, clamp active
    (3, 40, 17, 1.0),
    (100, 264, 300, 1.0),
    (129, 64, 513, 30.0),
    (300, 1032, 1000, 1.0),
]


@pytest.mark.parametrize("shape", LIN_SHAPES_BF16, ids=lambda s: "x".join(map(str, s)))
def test_linear_small_bf16(cuda_lib, shape):
    M, K, Nout, sx = shape
    d = fc_inputs.linear_inputs(M, K, Nout, dtype="bf16")
    xs = fc_inputs.bf16_bits(d["x32"] * np.float32(sx))
    y = cuda_lib.fc_linear_lse_mish(_dev(xs), _dev(d["W"]), _dev(d["b"])).cpu().numpy()
    ref = oracle.linear_lse_mish(fc_inputs.bf16_bits_to_f32(xs), d["W32"], d["b32"])
    _check(y, ref, TOL["bf16"], f"linear bf16 {shape}")


# ------------------------------------------------------------------ TF32 diagnostic mode

# With the oracle fed the operands the tensor cores actually multiply -- the tensor core drops the
# 13 low mantissa bits of the raw fp32 it is handed (x of both ops, W of the linear op), the conv
# path's weight re-layout rounds w to nearest TF32 (ties away from zero) -- the products are exact
# in fp32 and what remains is the fp32
# accumulation of K <= 1024 terms (about 2^-24 of the running sum per addition) and the
# activations' approximate exponential / reciprocal (about 1e-6): 1e-5 (conv) and 2e-5 (linear,
# whose logsumexp sums 2048 exponentials and whose l * mish(l) tail doubles relative error)
# of (1 + |ref|).  Observed on GB300: <= 2e-6 and <= 4e-6.  Against the raw operands the same
# calls are 100-1000x further off, so these pin each path's operand rounding.
DIAG_CONV = [(2, 8, 32, 32, 64, "gelu", True), (1, 64, 12, 140, 128, "mish_mish", False),
             (1, 13, 20, 37, 96, "mish", False), (2, 5, 19, 13, 32, "gelu_tanh", True)]


@pytest.mark.parametrize("shape", DIAG_CONV, ids=lambda s: "x".join(map(str, s[:5])) + f"-{s[5]}")
def test_conv_equals_oracle_on_its_tf32_operands(cuda_lib, shape):
    N, Cin, H, W, Cout, act, pool = shape
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout)
    f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
    o = oracle.conv3x3_act_pool if pool else oracle.conv3x3_act
    y = f(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act).cpu().numpy()
    xt, wr = oracle.tf32_truncate(d["x"]), oracle.tf32_round_nearest(d["w"])
    _check(y, o(xt, wr, d["b"], act), 1e-5, f"conv tf32 operands {shape}")


@pytest.mark.parametrize("shape", [(130, 520, 300, 1.0), (256, 1024, 2048, 1.0), (129, 64, 513, 30.0)],
                         ids=lambda s: "x".join(map(str, s)))
def test_linear_equals_oracle_on_tf32_truncated_operands(cuda_lib, shape):
    M, K, Nout, sx = shape
    d = fc_inputs.linear_inputs(M, K, Nout)
    x = (d["x"] * np.float32(sx)).astype(np.float32)
    y = cuda_lib.fc_linear_lse_mish(_dev(x), _dev(d["W"]), _dev(d["b"])).cpu().numpy()
    ref = oracle.linear_lse_mish(oracle.tf32_truncate(x), oracle.tf32_truncate(d["W"]), d["b"])
    _check(y, ref, 2e-5, f"linear tf32-truncated {shape}")


def _check_linear_tf32_bound(y, ref, x, W, b, what):
    """|y - y_exact| within the worst-case error of TF32 operands: each operand truncated to 10
    mantissa bits (relative error < 2^-10), so |dt_j| <= 2^-9 sum_k |x_k W_jk| (plus fp32
    accumulation, K 2^-24 of the same sum); u = clamp(4 t) moves by at most 4 |dt|; the row
    logsumexp l by at most max_j |du_j|; y = l mish(l) has |dy/dl| <= 2.2 |l| + 1 (mish' <= 1.1,
    |mish(l)| <= max(l, 0.31)).  l itself (for the slope only) comes from fp64 numpy."""
    x64, W64 = x.astype(np.float64), W.astype(np.float64)
    K = x.shape[1]
    dl = 4.0 * (2.0 ** -9 + K * 2.0 ** -24) * (np.abs(x64) @ np.abs(W64).T).max(axis=1)
    u = np.clip(4.0 * (x64 @ W64.T + b.astype(np.float64)), -10.0, 10.0)
    m = u.max(axis=1)
    l = m + np.log(np.exp(u - m[:, None]).sum(axis=1))
    bound = (2.2 * (np.abs(l) + dl) + 1.0) * dl + 1e-6
    err = np.abs(np.asarray(y, dtype=np.float64).reshape(-1) - np.asarray(ref, dtype=np.float64).reshape(-1))
    i = int(np.argmax(err - bound))
    assert err[i] <= bound[i], f"{what}: error {err[i]:.3e} above the TF32 bound {bound[i]:.3e} at {i}"


def _random_linear_cases(n, seed=2025):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        bf16 = bool(rng.integers(0, 2))
        step = 8 if bf16 else 4
        cases.append(dict(M=int(rng.integers(1, 400)), K=int(rng.integers(1, 160)) * step,
                          Nout=int(rng.integers(1, 1500)), sx=float(rng.choice([1.0, 1.0, 8.0, 40.0])), bf16=bf16))
    return cases


@pytest.mark.parametrize("case", _random_linear_cases(50), ids=lambda c: "{M}x{K}x{Nout}-s{sx:g}-{t}".format(t="bf16" if c["bf16"] else "f32", **c))
def test_linear_random_shapes(cuda_lib, case):
    """Seeded random (M, K, Nout) -- single CTAs and CTA pairs, ragged tiles, clamp on or off -- in fp32
    and bf16 against the oracle."""
    c = case
    dt = "bf16" if c["bf16"] else "f32"
    d = fc_inputs.linear_inputs(c["M"], c["K"], c["Nout"], dtype=dt)
    x32 = (d["x32"] * np.float32(c["sx"])).astype(np.float32)
    xs = fc_inputs.bf16_bits(x32) if c["bf16"] else x32
    xo = fc_inputs.bf16_bits_to_f32(xs) if c["bf16"] else x32
    y = cuda_lib.fc_linear_lse_mish(_dev(xs), _dev(d["W"]), _dev(d["b"])).cpu().numpy()
    ref = oracle.linear_lse_mish(xo, d["W32"], d["b32"])
    if c["bf16"] or c["sx"] == 1.0:
        # bf16 products are exact in fp32; N(0, 1) inputs are the workloads' distribution
        _check(y, ref, TOL[dt], f"random linear {c}")
    else:
        # Inputs scaled up: TF32 operands (10 mantissa bits) give an absolute error that grows with
        # the scale and with cancellation in the dot products, beyond the tolerance stated for the
        # workloads' N(0, 1) inputs.  The kernel is pinned to the oracle on the operands the tensor
        # core sees, and the exact result must lie within the TF32 error bound.
        _check(y, oracle.linear_lse_mish(oracle.tf32_truncate(x32), oracle.tf32_truncate(d["W32"]), d["b32"]),
               2e-5, f"random linear {c}, TF32 operands")
        _check_linear_tf32_bound(y, ref, x32, d["W32"], d["b32"], f"random linear {c}")


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("key", ["B", "Bt", "B3", "Bp", "Bn"])
def test_workload_B_full_size_sampled(cuda_lib, key):
    wl = fc_inputs.WORKLOADS[key]
    d = fc_inputs.workload_inputs(key)
    x = _nhwc(d["x"]) if wl.layout == "nhwc" else _dev(d["x"])
    y = cuda_lib.fc_conv3x3_act_pool(x, _dev(d["w"]), _dev(d["b"]), act=wl.act,
                                     precision=wl.precision, pad=wl.pad).cpu().numpy()
    rng = np.random.default_rng(7)
    flat = np.unique(np.concatenate([rng.choice(wl.N * wl.Cout, 192, replace=False),
                                     np.arange(wl.Cout), np.arange((wl.N - 1) * wl.Cout, wl.N * wl.Cout)]))
    ref = oracle.conv3x3_act_pool_at(d["x32"], d["w32"], d["b32"], flat, wl.act, pad=wl.pad)
    _check(y.reshape(-1)[flat], ref, TOL_X3 if wl.precision == "3xtf32" else TOL["f32"], f"workload {key}")


@pytest.mark.parametrize("key", ["C", "Cb", "C3", "Cp", "Cn", "Cbn"])
def test_workload_C_full_size_sampled(cuda_lib, key):
    import torch
    wl = fc_inputs.WORKLOADS[key]
    d = fc_inputs.workload_inputs(key)
    x = _nhwc(d["x"]) if wl.layout == "nhwc" else _dev(d["x"])
    y = cuda_lib.fc_conv3x3_act(x, _dev(d["w"]), _dev(d["b"]), act=wl.act,
                                precision=None if wl.dtype == "bf16" else wl.precision, pad=wl.pad)
    del x
    y = y.contiguous()   # logical NCHW order for the flat sample indices
    OH, OW = wl.OH, wl.OW
    rng = np.random.default_rng(8)
    total = wl.N * wl.Cout * OH * OW
    samples = [rng.choice(total, 1 << 20, replace=False)]
    for (n, co) in [(0, 0), (wl.N - 1, wl.Cout - 1), (17, 77)]:
        base = (n * wl.Cout + co) * OH * OW
        rows = np.concatenate([np.arange(OW), (OH - 1) * OW + np.arange(OW)])
        cols = np.concatenate([np.arange(OH) * OW, np.arange(OH) * OW + OW - 1])
        samples.append(base + np.concatenate([rows, cols]))
    flat = np.unique(np.concatenate(samples))
    got = y.view(-1)[torch.from_numpy(flat).cuda()].cpu().numpy()
    del y
    ref = oracle.conv3x3_act_at(d["x32"], d["w32"], d["b32"], flat, wl.act, pad=wl.pad)
    _check(got, ref, TOL_X3 if wl.precision == "3xtf32" else TOL[wl.dtype], f"workload {key}")


@pytest.mark.parametrize("key", ["D", "Db", "D3"])
def test_workload_D_full_size_sampled(cuda_lib, key):
    wl = fc_inputs.WORKLOADS[key]
    d = fc_inputs.workload_inputs(key)
    y = cuda_lib.fc_linear_lse_mish(_dev(d["x"]), _dev(d["W"]), _dev(d["b"]), wl.scale, wl.clamp_lo,
                                    wl.clamp_hi, precision=None if wl.dtype == "bf16" else wl.precision)
    y = y.cpu().numpy().reshape(-1)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(wl.M - 8, wl.M),
                                     np.random.default_rng(9).choice(wl.M, 112, replace=False)]))
    ref = oracle.linear_lse_mish(d["x32"], d["W32"], d["b32"], wl.scale, wl.clamp_lo, wl.clamp_hi, rows=rows)
    # Split TF32 removes the operands' TF32 error (7.9e-4 at this size with TF32 alone); what is left
    # over K = 8192 (3K = 24576 products, 3072 MMA steps per logit) is the rounding of the tensor
    # core's fp32 accumulator at every step, measured 9.8e-5 -- hence 2e-4 here, while the short
    # dot products of the small split-TF32 cases meet 2e-5.
    tol = 2e-4 if wl.precision == "3xtf32" else TOL[wl.dtype]
    _check(y[rows], ref, tol, f"workload {key}")
    # clamped logsumexp bound: l in [lo + ln n, hi + ln n] -> y = l mish(l) within the image of that range
    lo_l, hi_l = wl.clamp_lo + math.log(wl.Nout), wl.clamp_hi + math.log(wl.Nout)
    f = lambda l: l * oracle.mish(l)
    assert np.all(y >= min(f(lo_l), 0.0) - 1e-3) and np.all(y <= f(hi_l) + 1e-2)


@pytest.mark.parametrize("key", ["E", "En"])
def test_workload_E_full_size_sampled(cuda_lib, key):
    wl = fc_inputs.WORKLOADS[key]
    d = fc_inputs.workload_inputs(key)
    x = _nhwc(d["x"]) if wl.layout == "nhwc" else _dev(d["x"])
    y = cuda_lib.fc_conv3x3_act_pool(x, _dev(d["w"]), _dev(d["b"]), act="gelu").cpu().numpy()
    rng = np.random.default_rng(10)
    flat = np.unique(np.concatenate([rng.choice(wl.N * wl.Cout, 96, replace=False), np.arange(wl.Cout)]))
    ref = oracle.conv3x3_act_pool_at(d["x32"], d["w32"], d["b32"], flat, "gelu")
    _check(y.reshape(-1)[flat], ref, TOL["bf16"], f"workload {key}")


# ------------------------------------------------------------------ properties, errors, watchdog

def test_calls_on_a_side_stream_and_in_a_cuda_graph_match_direct_calls(cuda_lib):
    """Each op is several kernels with programmatic dependent launch between them; on a non-default
    stream and captured into a CUDA graph (programmatic edges) the results are the same bits."""
    import torch
    d = fc_inputs.conv_inputs(2, 8, 40, 36, 64)
    x, w, b = _dev(d["x"]), _dev(d["w"]), _dev(d["b"])
    dl = fc_inputs.linear_inputs(200, 256, 700)
    xl, Wl, bl = _dev(dl["x"]), _dev(dl["W"]), _dev(dl["b"])
    ref_pool = cuda_lib.fc_conv3x3_act_pool(x, w, b)
    ref_act = cuda_lib.fc_conv3x3_act(x, w, b, act="mish")
    ref_lin = cuda_lib.fc_linear_lse_mish(xl, Wl, bl)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        y_pool = cuda_lib.fc_conv3x3_act_pool(x, w, b, stream=side)
        y_act = cuda_lib.fc_conv3x3_act(x, w, b, act="mish", stream=side)
        y_lin = cuda_lib.fc_linear_lse_mish(xl, Wl, bl, stream=side)
    side.synchronize()
    assert torch.equal(y_pool, ref_pool) and torch.equal(y_act, ref_act) and torch.equal(y_lin, ref_lin)
    # graph capture: outputs and workspaces allocated up front, the calls captured and replayed
    o_pool, o_act, o_lin = torch.empty_like(ref_pool), torch.empty_like(ref_act), torch.empty_like(ref_lin)
    nb_pool = cuda_lib.fc_workspace_bytes("conv3x3_act_pool", 2, 8, 40, 36, 64)
    nb_act = cuda_lib.fc_workspace_bytes("conv3x3_act", 2, 8, 40, 36, 64)
    nb_lin = cuda_lib.fc_workspace_bytes("linear_lse_mish", 200, 256, 1, 1, 700)
    ws = [torch.empty(max(n, 1), dtype=torch.uint8, device="cuda") for n in (nb_pool, nb_act, nb_lin)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cuda_lib.fc_conv3x3_act_pool(x, w, b, out=o_pool, workspace=ws[0])
        cuda_lib.fc_conv3x3_act(x, w, b, act="mish", out=o_act, workspace=ws[1])
        cuda_lib.fc_linear_lse_mish(xl, Wl, bl, out=o_lin, workspace=ws[2])
    for _ in range(3):
        o_pool.zero_(); o_act.zero_(); o_lin.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o_pool, ref_pool) and torch.equal(o_act, ref_act) and torch.equal(o_lin, ref_lin)
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def test_results_are_bit_identical_run_to_run(cuda_lib):
    d = fc_inputs.conv_inputs(4, 8, 64, 64, 64)
    x, w, b = _dev(d["x"]), _dev(d["w"]), _dev(d["b"])
    y1 = cuda_lib.fc_conv3x3_act_pool(x, w, b).cpu().numpy()
    y2 = cuda_lib.fc_conv3x3_act_pool(x, w, b).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    dl = fc_inputs.linear_inputs(200, 256, 700)
    xl, Wl, bl = _dev(dl["x"]), _dev(dl["W"]), _dev(dl["b"])
    z1 = cuda_lib.fc_linear_lse_mish(xl, Wl, bl).cpu().numpy()
    z2 = cuda_lib.fc_linear_lse_mish(xl, Wl, bl).cpu().numpy()
    assert np.array_equal(z1.view(np.uint32), z2.view(np.uint32))


def test_zero_weights_give_activation_of_bias(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(2, 8, 30, 22, 64)
    w0 = torch.zeros(64, 8, 3, 3, device="cuda")
    y = cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), w0, _dev(d["b"])).cpu().numpy()
    ref = np.array([oracle.gelu(float(v)) for v in d["b"]])
    _check(y, np.broadcast_to(ref, y.shape), TOL["f32"], "w = 0")


def test_workspace_too_small_is_rejected(cuda_lib):
    import torch
    d = fc_inputs.conv_inputs(1, 8, 16, 16, 64)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.FCError) as e:
        cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), workspace=small)
    assert e.value.status in (cuda_lib.FC_ERR_WORKSPACE,)


def test_unsupported_cout_is_reported(cuda_lib):
    d = fc_inputs.conv_inputs(1, 8, 16, 16, 272)   # more than 256 output channels
    with pytest.raises(cuda_lib.FCError) as e:
        cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]))
    assert e.value.status == cuda_lib.FC_ERR_UNSUPPORTED


def test_watchdog_times_out_and_context_stays_usable(cuda_lib):
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK
    cuda_lib.fc_selftest_watchdog(2_000_000)   # ~1 ms: nothing ever arrives on the barrier
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_ERR_TIMEOUT
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK
    d = fc_inputs.conv_inputs(2, 8, 32, 32, 64)
    y = cuda_lib.fc_conv3x3_act_pool(_dev(d["x"]), _dev(d["w"]), _dev(d["b"])).cpu().numpy()
    ref = oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], "gelu")
    _check(y, ref, TOL["f32"], "after watchdog")
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def test_stream_scoped_status_sees_a_timeout_on_its_stream(cuda_lib):
    """fc_last_device_status(stream) waits for that stream only and reads the word without
    clearing it."""
    import torch
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK
    s = torch.cuda.Stream()
    assert cuda_lib.fc_last_device_status(s) == cuda_lib.FC_OK
    cuda_lib.fc_selftest_watchdog(2_000_000, stream=s)
    assert cuda_lib.fc_last_device_status(s) == cuda_lib.FC_ERR_TIMEOUT
    assert cuda_lib.fc_last_device_status(s) == cuda_lib.FC_ERR_TIMEOUT   # not cleared
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_ERR_TIMEOUT
    assert cuda_lib.fc_last_device_status(s) == cuda_lib.FC_OK


def test_outputs_are_nan_while_a_timeout_is_recorded(cuda_lib):
    """A recorded timeout (made by the watchdog self-test's bounded wait, no fault) means some
    kernel's partial results may be missing: the pooled conv and the Linear chain then write NaN
    instead of combining them, and are exact again once the status is cleared."""
    import torch
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK
    dc = fc_inputs.conv_inputs(2, 8, 32, 32, 64)
    dl = fc_inputs.linear_inputs(64, 256, 512)
    conv = lambda: cuda_lib.fc_conv3x3_act_pool(_dev(dc["x"]), _dev(dc["w"]), _dev(dc["b"])).cpu().numpy()
    lin = lambda: cuda_lib.fc_linear_lse_mish(_dev(dl["x"]), _dev(dl["W"]), _dev(dl["b"])).cpu().numpy()
    cuda_lib.fc_selftest_watchdog(2_000_000)
    torch.cuda.synchronize()
    assert np.all(np.isnan(conv())) and np.all(np.isnan(lin()))
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_ERR_TIMEOUT
    _check(conv(), oracle.conv3x3_act_pool(dc["x32"], dc["w32"], dc["b32"], "gelu"), TOL["f32"], "after clearing")
    _check(lin(), oracle.linear_lse_mish(dl["x"], dl["W"], dl["b"]), TOL["f32"], "after clearing")
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


def test_real_operators_give_up_through_their_bounded_waits(cuda_lib):
    """A short wait budget (set through the library's testing hook, which fc.h does not declare)
    makes the single-CTA pooled conv kernel and the single-CTA Linear kernel give up mid-pipeline:
    every role stops at its next wait, drains its own copies and MMAs in flight, and the CTA frees
    its tensor memory and returns.  The status word then reads FC_ERR_TIMEOUT and the outputs are
    NaN; with the default budget back, the next calls match the oracle and leave no status."""
    import torch
    lib = cuda_lib.load()
    set_budget = lib.fc_testing_set_wait_budget
    set_budget.argtypes = [ctypes.c_longlong]
    set_budget.restype = ctypes.c_longlong
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK
    dc = fc_inputs.conv_inputs(16, 8, 128, 128, 64)   # 16 x 32 pooled tiles on single CTAs
    dl = fc_inputs.linear_inputs(128, 1024, 4096)     # M <= 128: the single-CTA Linear kernel
    xc, wc, bc = _dev(dc["x"]), _dev(dc["w"]), _dev(dc["b"])
    xl, wl, bl = _dev(dl["x"]), _dev(dl["W"]), _dev(dl["b"])
    torch.cuda.synchronize()
    prev = set_budget(64)   # SM cycles: far below the first TMA load's latency
    try:
        yc = cuda_lib.fc_conv3x3_act_pool(xc, wc, bc).cpu().numpy()
        st_conv = cuda_lib.fc_device_status(clear=True)
        yl = cuda_lib.fc_linear_lse_mish(xl, wl, bl).cpu().numpy()
        st_lin = cuda_lib.fc_device_status(clear=True)
    finally:
        set_budget(0)
    assert prev > 10 ** 9
    assert st_conv == cuda_lib.FC_ERR_TIMEOUT and st_lin == cuda_lib.FC_ERR_TIMEOUT
    assert np.all(np.isnan(yc)) and np.all(np.isnan(yl))
    _check(cuda_lib.fc_conv3x3_act_pool(xc, wc, bc).cpu().numpy(),
           oracle.conv3x3_act_pool(dc["x32"], dc["w32"], dc["b32"], "gelu"), TOL["f32"], "conv after the timeout")
    _check(cuda_lib.fc_linear_lse_mish(xl, wl, bl).cpu().numpy(), oracle.linear_lse_mish(dl["x"], dl["W"], dl["b"]),
           TOL["f32"], "linear after the timeout")
    assert cuda_lib.fc_device_status(clear=True) == cuda_lib.FC_OK


@pytest.mark.parametrize("act", ["gelu", "mish", "mish_mish", "gelu_tanh"])
def test_activation_accuracy_through_a_delta_kernel(cuda_lib, act):
    """A delta 3x3 kernel makes the pre-activation equal to the input (values on a
    1/64 grid are exact in TF32), so the output is the kernel's activation of
    known points: checked against the oracle's fp64 activation to fp32-level
    absolute error over [-12, 12] plus large-magnitude points."""
    import torch
    pts = np.concatenate([np.arange(-768, 769) / 64.0, [-80.0, -40.0, -20.0, 20.0, 40.0, 80.0]]).astype(np.float32)
    W = pts.size + 2
    x = np.zeros((1, 1, 3, W), np.float32)
    x[0, 0, 0, :pts.size] = pts
    w = np.zeros((32, 1, 3, 3), np.float32)
    w[:, 0, 0, 0] = 1.0
    b = np.zeros(32, np.float32)
    y = cuda_lib.fc_conv3x3_act(_dev(x), _dev(w), _dev(b), act=act).cpu().numpy()[0, :, 0, :pts.size]
    ref = np.array([oracle.act(act, float(v)) for v in pts])
    err = np.abs(y - ref[None, :]) / np.maximum(1.0, np.abs(ref[None, :]))
    assert err.max() <= 2e-6, f"{act}: max error {err.max():.3e} at x = {pts[int(np.argmax(err.max(0)))]}"


# ------------------------------------------------------------------ extreme but valid shapes

EXTREME_CONV = [
    # (N, Cin, H, W, Cout, dtype, act, pool, pad)
    (2048, 3, 34, 34, 64, "f32", "gelu", True, 0),       # thousands of small images: many records per CTA
    (1, 8, 2050, 2050, 64, "f32", "gelu", True, 0),      # one large image: 32k tiles of one plane
    (1, 16, 5, 4100, 128, "f32", "mish_mish", False, 1),  # very wide rows
    (512, 128, 10, 10, 256, "bf16", "gelu", True, 0),    # CTA pairs over many small images
    (4096, 1, 3, 3, 16, "f32", "gelu", True, 0),         # 1 x 1 output planes
]


@pytest.mark.parametrize("case", EXTREME_CONV, ids=lambda c: "x".join(map(str, c[:5])) + f"-{c[5]}-{c[6]}-p{c[8]}")
def test_conv_extreme_shapes_sampled(cuda_lib, case):
    N, Cin, H, W, Cout, dt, act, pool, pad = case
    d = fc_inputs.conv_inputs(N, Cin, H, W, Cout, dt)
    f = cuda_lib.fc_conv3x3_act_pool if pool else cuda_lib.fc_conv3x3_act
    y = f(_dev(d["x"]), _dev(d["w"]), _dev(d["b"]), act=act, pad=pad).cpu().numpy().reshape(-1)
    rng = np.random.default_rng(11)
    idx = np.unique(np.concatenate([rng.choice(y.size, min(y.size, 300), replace=False), [0, y.size - 1]]))
    at = oracle.conv3x3_act_pool_at if pool else oracle.conv3x3_act_at
    _check(y[idx], at(d["x32"], d["w32"], d["b32"], idx, act, pad=pad), TOL[dt], f"extreme {case}")


@pytest.mark.parametrize("shape", [(65536, 64, 16), (1, 65536, 1), (3, 4, 70000)], ids=lambda s: "x".join(map(str, s)))
def test_linear_extreme_shapes_sampled(cuda_lib, shape):
    M, K, Nout = shape
    d = fc_inputs.linear_inputs(M, K, Nout)
    y = cuda_lib.fc_linear_lse_mish(_dev(d["x"]), _dev(d["W"]), _dev(d["b"])).cpu().numpy().reshape(-1)
    rows = np.unique(np.concatenate([np.random.default_rng(12).choice(M, min(M, 64), replace=False), [0, M - 1]]))
    _check(y[rows], oracle.linear_lse_mish(d["x32"], d["W32"], d["b32"], rows=rows), TOL["f32"], f"extreme {shape}")
