"""Seeded synthetic inputs and the named workloads.

This module is shared by the oracle-side tests, the CUDA-side tests and
``bench.py``.  It holds NO arithmetic of the fused operators: it only draws
random numbers (numpy's PCG64 ``default_rng``), casts them to the storage type
and names the workload shapes.  Keeping it free of the method means the oracle
and the CUDA path share nothing but their inputs.

Distributions: activations are N(0, 1); weights and biases are
U(-1/sqrt(fan_in), +1/sqrt(fan_in)) -- the default ``nn.Conv2d`` / ``nn.Linear``
initialisation the pages rely on (Linear page, Kimi-K2.6 l2_p22, discussion of
the module's parameter initialisation).  Seeds: x <- 0, w <- 1, b <- 2.
bf16 values are the round-to-nearest-even bf16 of the fp32 draws.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_X, SEED_W, SEED_B = 0, 1, 2


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(shape, seed):
    return np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)


def _uniform(shape, bound, seed):
    return np.random.default_rng(seed).uniform(-bound, bound, size=shape).astype(np.float32)


@dataclasses.dataclass(frozen=True)
class ConvWorkload:
    name: str
    N: int
    Cin: int
    H: int
    W: int
    Cout: int
    dtype: str          # "f32" or "bf16"
    act: str            # "gelu" | "mish" | "mish_mish" | "gelu_tanh"
    pool: bool          # True: global mean to (N, Cout); False: full output
    precision: str = "tf32"   # fp32 storage: "tf32" or "3xtf32" (split-TF32 products); bf16: "bf16"
    pad: int = 0              # zero padding on every side
    layout: str = "nchw"      # "nchw", or "nhwc": x stored [N][H][W][Cin], full output [N][OH][OW][Cout]

    @property
    def OH(self):
        return self.H + 2 * self.pad - 2

    @property
    def OW(self):
        return self.W + 2 * self.pad - 2

    def flops(self) -> float:
        """Contraction flops only: 2 * outputs * (Cin * 9)."""
        return 2.0 * self.N * self.Cout * self.OH * self.OW * self.Cin * 9

    def compulsory_bytes(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        out = self.N * self.Cout * (1 if self.pool else self.OH * self.OW) * 4
        return (self.N * self.Cin * self.H * self.W + self.Cout * self.Cin * 9 + self.Cout) * es + out


@dataclasses.dataclass(frozen=True)
class LinearWorkload:
    name: str
    M: int
    K: int
    Nout: int
    scale: float = 2.0
    clamp_lo: float = -10.0
    clamp_hi: float = 10.0
    dtype: str = "f32"
    precision: str = "tf32"   # fp32 inputs: "tf32" or "3xtf32" (split TF32)

    def flops(self) -> float:
        return 2.0 * self.M * self.K * self.Nout

    def compulsory_bytes(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        return (self.M * self.K + self.Nout * self.K + self.Nout) * es + self.M * 4


@dataclasses.dataclass(frozen=True)
class EpilogueWorkload:
    """A standalone epilogue over a computed contraction output (the pages' own kernels):
    kind "act_mean" (act, then the mean of each trailing (H, W) plane), "act_map" (act
    elementwise) or "lse_row" (scale, x + x, clamp, row logsumexp, l * mish(l))."""
    name: str
    kind: str
    shape: tuple
    act: str = "gelu"
    dtype: str = "f32"

    def flops(self) -> float:
        return 0.0   # no contraction: these are HBM-bound

    def elements(self) -> int:
        return int(np.prod(self.shape))

    def compulsory_bytes(self) -> int:
        es = 4 if self.dtype == "f32" else 2
        if self.kind == "act_map":
            return self.elements() * (es + 4)
        if self.kind == "act_mean":
            return self.elements() * es + int(np.prod(self.shape[:-2])) * 4
        return self.elements() * 4 + self.shape[0] * 4


# The five workloads of the pages, with the shapes each page states.
WORKLOADS = {
    # Conv2d->GELU->global-average-pool page (Kimi-K2.6 l2_p67), problem statement,
    # at a tiny batch/size for exhaustive checks.
    "A": ConvWorkload("conv3x3_gelu_avgpool_tiny_f32_2x8x32x32_c64", 2, 8, 32, 32, 64, "f32", "gelu", True),
    # Same page, full problem size.
    "B": ConvWorkload("conv3x3_gelu_avgpool_f32_128x8x256x256_c64", 128, 8, 256, 256, 64, "f32", "gelu", True),
    # Conv2d->Mish->Mish page (Kimi-K2.6 l2_p4), problem statement.
    "C": ConvWorkload("conv3x3_mish_mish_f32_64x64x256x256_c128", 64, 64, 256, 256, 128, "f32", "mish_mish", False),
    # Linear->x2->x+x->clamp->logsumexp->x*mish(x) page (Kimi-K2.6 l2_p22), problem statement.
    "D": LinearWorkload("linear_lse_mish_f32_1024x8192x8192", 1024, 8192, 8192),
    # bf16 variants of the Linear and Mish->Mish chains at the same sizes (precision variants)
    "Db": LinearWorkload("linear_lse_mish_bf16_1024x8192x8192", 1024, 8192, 8192, dtype="bf16"),
    # split-TF32 (fp32-level error) variant of the Linear chain at the same size
    "D3": LinearWorkload("linear_lse_mish_3xtf32_1024x8192x8192", 1024, 8192, 8192, precision="3xtf32"),
    "Cb": ConvWorkload("conv3x3_mish_mish_bf16_64x64x256x256_c128", 64, 64, 256, 256, 128, "bf16", "mish_mish", False),
    # bf16 variant of the conv->GELU->pool chain at a tensor-core-bound size.
    "E": ConvWorkload("conv3x3_gelu_avgpool_bf16_32x128x128x128_c256", 32, 128, 128, 128, 256, "bf16", "gelu", True),
    # The conv->GELU->pool page's tanh-approximate GELU (the variant its trace weighs against
    # the exact form), at the full problem size.
    "Bt": ConvWorkload("conv3x3_gelu_tanh_avgpool_f32_128x8x256x256_c64", 128, 8, 256, 256, 64, "f32", "gelu_tanh",
                       True),
    # Split-TF32 (3 products per term, fp32-level contraction error) at the fp32 conv pages' sizes.
    "B3": ConvWorkload("conv3x3_gelu_avgpool_f32x3_128x8x256x256_c64", 128, 8, 256, 256, 64, "f32", "gelu", True,
                       "3xtf32"),
    "C3": ConvWorkload("conv3x3_mish_mish_f32x3_64x64x256x256_c128", 64, 64, 256, 256, 128, "f32", "mish_mish",
                       False, "3xtf32"),
    # Zero padding 1 ('same' convs: 256 x 256 outputs) at the fp32 conv pages' sizes.
    "Bp": ConvWorkload("conv3x3_gelu_avgpool_pad1_f32_128x8x256x256_c64", 128, 8, 256, 256, 64, "f32", "gelu", True,
                       pad=1),
    "Cp": ConvWorkload("conv3x3_mish_mish_pad1_f32_64x64x256x256_c128", 64, 64, 256, 256, 128, "f32", "mish_mish",
                       False, pad=1),
    # NHWC (channels_last) input and output at the Mish->Mish page's size, fp32 and bf16.
    "Cn": ConvWorkload("conv3x3_mish_mish_nhwc_f32_64x64x256x256_c128", 64, 64, 256, 256, 128, "f32", "mish_mish",
                       False, layout="nhwc"),
    "Cbn": ConvWorkload("conv3x3_mish_mish_nhwc_bf16_64x64x256x256_c128", 64, 64, 256, 256, 128, "bf16",
                        "mish_mish", False, "bf16", layout="nhwc"),
    # NHWC input for the pooled chains at B's and E's sizes.
    "Bn": ConvWorkload("conv3x3_gelu_avgpool_nhwc_f32_128x8x256x256_c64", 128, 8, 256, 256, 64, "f32", "gelu", True,
                       layout="nhwc"),
    "En": ConvWorkload("conv3x3_gelu_avgpool_nhwc_bf16_32x128x128x128_c256", 32, 128, 128, 128, 256, "bf16", "gelu",
                       True, "bf16", layout="nhwc"),
    # Profiling-size cases of B and C (inputs still larger than L2, a fraction of the device memory):
    # what a many-pass ncu capture runs instead of the full workloads.
    "B64": ConvWorkload("conv3x3_gelu_avgpool_f32_64x8x256x256_c64", 64, 8, 256, 256, 64, "f32", "gelu", True),
    "C8": ConvWorkload("conv3x3_mish_mish_f32_8x64x256x256_c128", 8, 64, 256, 256, 128, "f32", "mish_mish", False),
    # The pages' epilogue-only kernels at their sizes: over the conv output of the GELU->pool page,
    # the conv output of the Mish->Mish page, and the Linear output of the Linear page.
    "K1e": EpilogueWorkload("gelu_avgpool_epilogue_f32_128x64x254x254", "act_mean", (128, 64, 254, 254), "gelu"),
    "K2e": EpilogueWorkload("mish_mish_epilogue_f32_64x128x254x254", "act_map", (64, 128, 254, 254), "mish_mish"),
    "K3e": EpilogueWorkload("scale_clamp_lse_mish_rows_f32_1024x8192", "lse_row", (1024, 8192)),
}


def epilogue_inputs(shape, seed=SEED_X, dtype="f32", scale=1.0):
    """A computed contraction output for the standalone epilogues: N(0, scale^2) fp32 (or its
    bf16 bits), seeded.  The conv outputs of the workloads are close to N(0, 1/3) before the
    bias (unit-variance inputs, U(+-1/sqrt(fan_in)) weights), the Linear output likewise."""
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)).astype(np.float32)
    return bf16_bits(v) if dtype == "bf16" else v


def conv_inputs(N, Cin, H, W, Cout, dtype="f32", seeds=(SEED_X, SEED_W, SEED_B)):
    """x (N,Cin,H,W) ~ N(0,1); w (Cout,Cin,3,3), b (Cout) ~ U(+-1/sqrt(Cin*9)).

    Returns a dict with the storage arrays (``x``, ``w``, ``b``: float32, or
    uint16 bf16 bit patterns when dtype == "bf16") and their exact fp32 values
    (``x32``, ``w32``, ``b32``) for the oracle.
    """
    bound = 1.0 / math.sqrt(Cin * 9)
    x = _normal((N, Cin, H, W), seeds[0])
    w = _uniform((Cout, Cin, 3, 3), bound, seeds[1])
    b = _uniform((Cout,), bound, seeds[2])
    if dtype == "f32":
        return dict(x=x, w=w, b=b, x32=x, w32=w, b32=b)
    if dtype == "bf16":
        xb, wb, bb = bf16_bits(x), bf16_bits(w), bf16_bits(b)
        return dict(x=xb, w=wb, b=bb, x32=bf16_bits_to_f32(xb), w32=bf16_bits_to_f32(wb),
                    b32=bf16_bits_to_f32(bb))
    raise ValueError(f"unknown dtype {dtype!r}")


def linear_inputs(M, K, Nout, seeds=(SEED_X, SEED_W, SEED_B), dtype="f32"):
    """x (M,K) ~ N(0,1); W (Nout,K), b (Nout) ~ U(+-1/sqrt(K)).  For dtype "bf16" the arrays are
    uint16 bf16 bit patterns (round to nearest even of the fp32 draws) and x32 / W32 / b32 hold
    their exact fp32 values for the oracle."""
    bound = 1.0 / math.sqrt(K)
    x = _normal((M, K), seeds[0])
    Wt = _uniform((Nout, K), bound, seeds[1])
    b = _uniform((Nout,), bound, seeds[2])
    if dtype == "bf16":
        xb, wb, bb = bf16_bits(x), bf16_bits(Wt), bf16_bits(b)
        return dict(x=xb, W=wb, b=bb, x32=bf16_bits_to_f32(xb), W32=bf16_bits_to_f32(wb), b32=bf16_bits_to_f32(bb))
    return dict(x=x, W=Wt, b=b, x32=x, W32=Wt, b32=b)


def workload_inputs(key: str):
    wl = WORKLOADS[key]
    if isinstance(wl, EpilogueWorkload):
        # conv / Linear outputs of the workloads have a standard deviation near 0.58
        return {"v": epilogue_inputs(wl.shape, seed=SEED_X, dtype=wl.dtype, scale=0.58)}
    if isinstance(wl, ConvWorkload):
        return conv_inputs(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, wl.dtype)
    return linear_inputs(wl.M, wl.K, wl.Nout, dtype=wl.dtype)
