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

// 2 GELU(z) for two lanes, GELU the exact (erf) form 0.5 z (1 + erf(z / sqrt 2)).
// erf is Hastings' rational approximation as printed in Abramowitz & Stegun, Handbook of
// Mathematical Functions, eq. 7.1.26: for u >= 0, erf(u) = 1 - t q(t) e^{-u^2} with
// q(t) = a1 + t (a2 + t (a3 + t (a4 + t a5))), t = 1 / (1 + p u), |error| <= 1.5e-7.
// With u = |z| / sqrt 2: p u = (p / sqrt 2) |z| and e^{-u^2} = 2^{-(log2 e / 2) z^2}.
// erf is odd, so z erf(z / sqrt 2) = |z| erf(u) and 2 GELU(z) = z + |z| erf(u): one
// fused multiply-add after erf.  The factor 1/2 is applied by the caller (once per
// pooled sum, or per stored value).
__device__ __forceinline__ float2 gelu2(float2 z)
{
    const float2 a = make_float2(fabsf(z.x), fabsf(z.y));
    const float2 d = __ffma2_rn(a, splat2(0.3275911f * 0.70710678118654752f), splat2(1.0f));
    const float2 t = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 q = __ffma2_rn(splat2(1.061405429f), t, splat2(-1.453152027f));
    q = __ffma2_rn(q, t, splat2(1.421413741f));
    q = __ffma2_rn(q, t, splat2(-0.284496736f));
    q = __ffma2_rn(q, t, splat2(0.254829592f));
    const float2 w = __fmul2_rn(__fmul2_rn(z, z), splat2(0.72134752044448170f));   // (log2 e / 2) z^2
    const float2 e = make_float2(ex2_approx(-w.x), ex2_approx(-w.y));
    const float2 tq = __fmul2_rn(q, t);
    const float2 erfv = __ffma2_rn(make_float2(-tq.x, -tq.y), e, splat2(1.0f));   // erf(|z| / sqrt 2)
    return __ffma2_rn(a, erfv, z);
}

// Mish(z) = z tanh(softplus(z)) for two lanes, with tanh(log(1 + e^z)) = n / (n + 2),
// n = e^z (e^z + 2).  The exponent is clamped at 15, where n / (n + 2) is already 1 in
// fp32, so that n cannot overflow (it would near z = 44) and no select is needed.
__device__ __forceinline__ float2 mish2(float2 z)
{
    const float2 s = __fmul2_rn(make_float2(fminf(z.x, 15.0f), fminf(z.y, 15.0f)), splat2(1.4426950408889634f));
    const float2 e = make_float2(ex2_approx(s.x), ex2_approx(s.y));
    const float2 n = __fmul2_rn(__fadd2_rn(e, splat2(2.0f)), e);
    const float2 d = __fadd2_rn(n, splat2(2.0f));
    const float2 r = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    return __fmul2_rn(__fmul2_rn(z, n), r);
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
