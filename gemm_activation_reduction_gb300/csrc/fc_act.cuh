// fc_act.cuh -- the pointwise activations of the three chains, evaluated for two
// values per paired-FP32 (f32x2) instruction: the conv epilogue and the standalone
// epilogue kernels share them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fc {
namespace convk {

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- packed activations
// The epilogue evaluates two accumulator columns per instruction with Blackwell's paired
// FP32 arithmetic (fma/mul/add.rn.f32x2: two results per issued instruction, same
// rounding as the scalar forms); only the SFU steps (reciprocal, exponential) and the
// absolute value / clamp stay per lane.  The epilogue is issue-bound, so this cuts its
// instruction count by about 40 %.
__device__ __forceinline__ float2 splat2(float c) { return make_float2(c, c); }

// 2 GELU(z) for two lanes, GELU the exact (erf) form z Phi(z).  With Phi(z) = erfc(-z / sqrt 2) / 2
// and erfc(-x) = 2 - erfc(x):  2 GELU(z) = z + |z| - |z| erfc(|z| / sqrt 2).  The erfc factor is
// 2^P(|z|), P the degree-5 polynomial below: log2 erfc(a / sqrt 2) fitted on [0, 7] by weighted
// least squares iteratively reweighted toward minimax of the GELU error (gen_gelu_coeffs.py
// prints these values); GELU's error stays below 5e-7 (absolute, or relative above 1) before the
// exponential's own rounding.  P's leading coefficient is negative and P < -85 for every
// |z| > 10, so no clamp is needed: 2^P vanishes there (the padding pre-activation -1e4 gives
// exactly 0).  Per pair: five paired FMAs (Horner), one paired add and one paired FMA for the
// result, two exponentials -- no reciprocal, no clamp.  The factor 1/2 is applied by the caller
// (once per pooled sum, or per stored value).
constexpr float kGeluP0 = -3.733664925675839e-05f;
constexpr float kGeluP1 = -1.1507893800735474f;
constexpr float kGeluP2 = -0.4599895775318146f;
constexpr float kGeluP3 = -0.05182963237166405f;
constexpr float kGeluP4 = 0.007085344288498163f;
constexpr float kGeluP5 = -0.0004734089015983045f;

__device__ __forceinline__ float2 gelu2(float2 z)
{
    const float2 a = make_float2(fabsf(z.x), fabsf(z.y));
    float2 p = __ffma2_rn(splat2(kGeluP5), a, splat2(kGeluP4));
    p = __ffma2_rn(p, a, splat2(kGeluP3));
    p = __ffma2_rn(p, a, splat2(kGeluP2));
    p = __ffma2_rn(p, a, splat2(kGeluP1));
    p = __ffma2_rn(p, a, splat2(kGeluP0));
    const float2 e = make_float2(ex2_approx(p.x), ex2_approx(p.y));   // erfc(|z| / sqrt 2)
    return __ffma2_rn(make_float2(-a.x, -a.y), e, __fadd2_rn(z, a));
}

// Mish(z) = z tanh(softplus(z)) for two lanes, with tanh(log(1 + e^z)) = n / (n + 2),
// n = e^z (e^z + 2), so Mish(z) = z - 2 z / (n + 2) and n + 2 = (e^z + 1)^2 + 1.  With
// v = (e^z + 1) / sqrt 2 that is z - z / h, h = v^2 + 1/2 = (n + 2) / 2 >= 1: two paired FMAs
// for h, one reciprocal, one paired FMA for the result.  The exponent is clamped at 15, where
// n / (n + 2) is already 1 in fp32, so that nothing overflows and no select is needed.  (The
// difference z - z / h cancels for very negative z, where Mish is near 0: the absolute error stays
// near 2^-24 |z|, e.g. 1e-6 at z = -20.)
__device__ __forceinline__ float2 mish2(float2 z)
{
    constexpr float kInvSqrt2 = 0.70710678118654752f;
    const float2 s = __fmul2_rn(make_float2(fminf(z.x, 15.0f), fminf(z.y, 15.0f)), splat2(1.4426950408889634f));
    const float2 e = make_float2(ex2_approx(s.x), ex2_approx(s.y));
    const float2 v = __ffma2_rn(e, splat2(kInvSqrt2), splat2(kInvSqrt2));
    const float2 h = __ffma2_rn(v, v, splat2(0.5f));
    const float2 r = make_float2(rcp_approx(h.x), rcp_approx(h.y));
    return __ffma2_rn(make_float2(-r.x, -r.y), z, z);
}

// tanh-approximate GELU for two lanes: 0.5 z (1 + tanh(u)) = z sigma(2u) = z / (1 + e^{-2u}),
// u = sqrt(2/pi) (z + 0.044715 z^3), with 2u log2 e = z (k + k 0.044715 z^2), k = 2 sqrt(2/pi) log2 e.
// Far below zero e^{-2u} overflows to inf and the result is -0; far above it is z.
__device__ __forceinline__ float2 gelu_tanh2(float2 z)
{
    constexpr float kK = 2.302208198144325f;
    constexpr float kK3 = 0.1029432395800235f;   // k * 0.044715
    const float2 w = __fmul2_rn(__ffma2_rn(__fmul2_rn(z, z), splat2(kK3), splat2(kK)), z);   // 2u log2 e
    const float2 e = make_float2(ex2_approx(-w.x), ex2_approx(-w.y));
    const float2 d = __fadd2_rn(e, splat2(1.0f));
    return __fmul2_rn(z, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Activation codes follow fc_act: 0 erf-GELU, 1 Mish, 2 Mish twice, 3 tanh-GELU.  act2
// returns kActScale<ACT>^-1 times the activation: the caller multiplies by kActScale.
template <int ACT>
__device__ __forceinline__ float2 act2(float2 z)
{
    if constexpr (ACT == 0) return gelu2(z);
    else if constexpr (ACT == 1) return mish2(z);
    else if constexpr (ACT == 2) return mish2(mish2(z));
    else return gelu_tanh2(z);
}
template <int ACT>
constexpr float kActScale = ACT == 0 ? 0.5f : 1.0f;

}  // namespace convk
}  // namespace fc
