// fc_epilogue.cu -- the pages' epilogue-only kernels, as HBM-streaming GB300 kernels over an
// already computed contraction output:
//   act_map        out = act(v) elementwise          (Conv->Mish->Mish page, elementwise kernel)
//   act_mean       y[p] = mean of act over plane p   (Conv->GELU->pool page, fused epilogue kernel)
//   lse_row        y[m] = l * mish(l), l = logsumexp_j clamp(2 scale t[m, j], lo, hi)
//                                                    (Linear page, row kernel)
// Each reads its input once (and act_map writes its output once); the activation arithmetic
// is the conv epilogue's (fc_act.cuh).  Reductions are fixed-order (deterministic).
#include <algorithm>

#include <cuda_bf16.h>

#include "fc_act.cuh"
#include "fc_internal.h"

namespace fc {
namespace {

using convk::act2;
using convk::kActScale;

// 8 consecutive inputs as floats: two 16-byte loads (fp32) or one (bf16), streaming.
template <bool BF16>
__device__ __forceinline__ void load8(const void* base, long long i8, float (&v)[8])
{
    if constexpr (BF16) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(base) + i8);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    } else {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(base) + 2 * i8);
        const float4 b = __ldcs(reinterpret_cast<const float4*>(base) + 2 * i8 + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

template <bool BF16>
__device__ __forceinline__ float load1(const void* base, long long i)
{
    if constexpr (BF16) {
        const unsigned short h = reinterpret_cast<const unsigned short*>(base)[i];
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return reinterpret_cast<const float*>(base)[i];
    }
}

template <int ACT>
__device__ __forceinline__ float act1(float z)
{
    return act2<ACT>(make_float2(z, z)).x * kActScale<ACT>;
}

// out[i] = act(v[i]); v and out 16-byte aligned.  Grid-stride over groups of 8 elements,
// kInFlight groups loaded per thread before any is evaluated (enough bytes in flight for
// HBM latency); the n % 8 tail by the first threads.
constexpr int kInFlight = 4;

template <int ACT, bool BF16>
__global__ void __launch_bounds__(256) act_map_kernel(const void* v, float* out, long long n)
{
    const long long groups = n / 8;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    float4* o = reinterpret_cast<float4*>(out);
    for (long long g0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; g0 < groups;
         g0 += kInFlight * stride) {
        float x[kInFlight][8];
#pragma unroll
        for (int h = 0; h < kInFlight; ++h)
            if (g0 + h * stride < groups) load8<BF16>(v, g0 + h * stride, x[h]);
#pragma unroll
        for (int h = 0; h < kInFlight; ++h) {
            const long long g = g0 + h * stride;
            if (g >= groups) break;
            float r[8];
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                float2 y = act2<ACT>(make_float2(x[h][k], x[h][k + 1]));
                if constexpr (ACT == 0) y = __fmul2_rn(y, convk::splat2(kActScale<ACT>));
                r[k] = y.x;
                r[k + 1] = y.y;
            }
            __stcs(o + 2 * g, make_float4(r[0], r[1], r[2], r[3]));
            __stcs(o + 2 * g + 1, make_float4(r[4], r[5], r[6], r[7]));
        }
    }
    const long long tail = n - groups * 8;
    const long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
    if (t < tail) out[groups * 8 + t] = act1<ACT>(load1<BF16>(v, groups * 8 + t));
}

constexpr int kRedThreads = 256;

// Block sum of one float per thread in a fixed order: warp butterflies, then warp 0 over the
// eight warp totals.  The result is valid in thread 0.
__device__ __forceinline__ float block_sum(float s, float* red)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = s;
    __syncthreads();
    float t = 0.0f;
    if (warp == 0) {
        t = lane < kRedThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    return t;
}

// y[p] = kActScale * sum act(v[p * plane + i]) / plane; one CTA per plane.  The vector path
// needs the plane's start 16-byte aligned; otherwise (or for the tail) scalar loads.
template <int ACT, bool BF16>
__global__ void __launch_bounds__(kRedThreads) act_mean_kernel(const void* v, float* y, long long plane)
{
    __shared__ float red[kRedThreads / 32];
    constexpr int kEs = BF16 ? 2 : 4;
    const long long p = blockIdx.x;
    const long long first = p * plane;
    const uint8_t* base = reinterpret_cast<const uint8_t*>(v) + first * kEs;
    float2 acc = make_float2(0.0f, 0.0f);
    long long done = 0;
    if ((reinterpret_cast<uintptr_t>(base) & 15u) == 0) {
        const long long groups = plane / 8;
        for (long long g = threadIdx.x; g < groups; g += kRedThreads) {
            float x[8];
            load8<BF16>(base, g, x);
#pragma unroll
            for (int k = 0; k < 8; k += 2) acc = __fadd2_rn(acc, act2<ACT>(make_float2(x[k], x[k + 1])));
        }
        done = groups * 8;
    }
    float s = acc.x + acc.y;
    for (long long i = done + threadIdx.x; i < plane; i += kRedThreads) {
        const float z = load1<BF16>(base, i);
        s += act2<ACT>(make_float2(z, 0.0f)).x;
    }
    const float tot = block_sum(s, red);
    if (threadIdx.x == 0) y[p] = tot * kActScale<ACT> / static_cast<float>(plane);
}

// Three-input maximum (one instruction on sm_100 and later); NaN inputs are ignored.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Merge two online (max, sum of 2^(x - max)) pairs of base-2 logsumexp.
__device__ __forceinline__ void lse2_merge(float& m, float& s, float m2, float s2)
{
    const float nm = fmaxf(m, m2);
    if (nm == -INFINITY) return;
    s = s * convk::ex2_approx(m - nm) + s2 * convk::ex2_approx(m2 - nm);
    m = nm;
}

constexpr float kLn2 = 0.69314718055994531f;

// One CTA per row.  The row's logsumexp of u = clamp(y * scale + y * scale, lo, hi) is taken in
// base 2: w = y * k2 with k2 = 2 scale log2(e), clamped to [lo2, hi2] = [lo, hi] log2(e), and
// l = ln 2 (max w + log2 sum 2^(w - max w)).  Since clamping is monotone, the max is taken over
// the unclamped w (three at a time) and clamped once; each term is then 2^-d with
// d = clamp(cm - w, 0, cm - lo2), which equals cm - clamp(w, lo2, hi2) exactly (a NaN input
// counts as lo, as clamp(NaN) = lo does for fminf / fmaxf).  Per element that is a paired
// multiply, a third of a max, a paired subtract, two min/max, one ex2 and half a paired add:
// the ex2 unit (16 per clock per SM) is the arithmetic bound, below the HBM time at 8192
// columns.  Up to 8 of a thread's 16-byte chunks are loaded before any is reduced; missing
// chunks of a short batch add nothing.  out[m] = l * mish(l) = l^2 tanh(softplus(l)).
// Launched as a programmatic dependent: the wait comes before the first read of t.
__global__ void __launch_bounds__(kRedThreads) lse_row_kernel(const float* t, float* out, int N, float k2, float lo2,
                                                           float hi2)
{
    __shared__ float red_m[kRedThreads / 32], red_s[kRedThreads / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float* row = t + static_cast<long long>(blockIdx.x) * N;
    float m = -INFINITY, s = 0.0f;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
        const int quads = N / 4;
        for (int q0 = threadIdx.x; q0 < quads; q0 += 8 * kRedThreads) {
            float2 w[16];
            bool have[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                have[h] = q0 + h * kRedThreads < quads;
                float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (have[h]) v = __ldcs(reinterpret_cast<const float4*>(row) + q0 + h * kRedThreads);
                w[2 * h] = __fmul2_rn(make_float2(v.x, v.y), make_float2(k2, k2));
                w[2 * h + 1] = __fmul2_rn(make_float2(v.z, v.w), make_float2(k2, k2));
                if (!have[h]) w[2 * h] = w[2 * h + 1] = make_float2(-INFINITY, -INFINITY);
            }
            float a0 = max3(w[0].x, w[0].y, w[1].x), a1 = max3(w[1].y, w[2].x, w[2].y);
#pragma unroll
            for (int k = 3; k < 15; k += 3) {
                a0 = max3(a0, w[k].x, w[k].y);
                a1 = max3(a1, w[k + 1].x, w[k + 1].y);
                a0 = max3(a0, w[k + 2].x, w[k + 2].y);
            }
            const float cm = fminf(fmaxf(max3(a0, a1, fmaxf(w[15].x, w[15].y)), lo2), hi2);
            const float dl = cm - lo2;
            float2 acc0 = make_float2(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float2 d = __fadd2_rn(make_float2(cm, cm), make_float2(-w[2 * h + j].x, -w[2 * h + j].y));
                    d.x = fmaxf(fminf(d.x, dl), 0.0f);
                    d.y = fmaxf(fminf(d.y, dl), 0.0f);
                    float2 e = make_float2(convk::ex2_approx(-d.x), convk::ex2_approx(-d.y));
                    if (!have[h]) e = make_float2(0.0f, 0.0f);
                    if (j == 0)
                        acc0 = __fadd2_rn(acc0, e);
                    else
                        acc1 = __fadd2_rn(acc1, e);
                }
            }
            const float2 acc = __fadd2_rn(acc0, acc1);
            lse2_merge(m, s, cm, acc.x + acc.y);
        }
        done = quads * 4;
    }
    // rows that are not 16-byte aligned, and the N % 4 tail: one element at a time
    for (int j = done + threadIdx.x; j < N; j += kRedThreads) {
        const float w = fminf(fmaxf(row[j] * k2, lo2), hi2);
        if (w > m) {
            s = s * convk::ex2_approx(m - w) + 1.0f;
            m = w;
        } else {
            s += convk::ex2_approx(w - m);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        lse2_merge(m, s, m2, s2);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red_m[warp] = m;
        red_s[warp] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float M = red_m[0], S = red_s[0];
        for (int w = 1; w < kRedThreads / 32; ++w) lse2_merge(M, S, red_m[w], red_s[w]);
        const float l = (M + log2f(S)) * kLn2;
        const float sp = fmaxf(l, 0.0f) + log1pf(expf(-fabsf(l)));
        out[blockIdx.x] = l * (l * tanhf(sp));
    }
}

template <bool BF16>
cudaError_t act_map_dispatch(const void* v, float* out, long long n, int act, int blocks, cudaStream_t st)
{
    switch (act) {
    case 0: act_map_kernel<0, BF16><<<blocks, 256, 0, st>>>(v, out, n); break;
    case 1: act_map_kernel<1, BF16><<<blocks, 256, 0, st>>>(v, out, n); break;
    case 2: act_map_kernel<2, BF16><<<blocks, 256, 0, st>>>(v, out, n); break;
    case 3: act_map_kernel<3, BF16><<<blocks, 256, 0, st>>>(v, out, n); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t act_mean_dispatch(const void* v, float* y, long long planes, long long plane, int act, cudaStream_t st)
{
    const dim3 grid(static_cast<unsigned>(planes));
    switch (act) {
    case 0: act_mean_kernel<0, BF16><<<grid, kRedThreads, 0, st>>>(v, y, plane); break;
    case 1: act_mean_kernel<1, BF16><<<grid, kRedThreads, 0, st>>>(v, y, plane); break;
    case 2: act_mean_kernel<2, BF16><<<grid, kRedThreads, 0, st>>>(v, y, plane); break;
    case 3: act_mean_kernel<3, BF16><<<grid, kRedThreads, 0, st>>>(v, y, plane); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t act_map_launch(const void* v, float* out, long long n, int bf16, int act, int sm_count, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    // enough 16-byte loads in flight to cover HBM latency: 8 CTAs of 256 threads per SM
    const long long groups = (n + 7) / 8;
    const int blocks = static_cast<int>(std::max<long long>(1, std::min<long long>((groups + 255) / 256, 8LL * sm_count)));
    return bf16 ? act_map_dispatch<true>(v, out, n, act, blocks, st) : act_map_dispatch<false>(v, out, n, act, blocks, st);
}

cudaError_t act_mean_launch(const void* v, float* y, long long planes, long long plane, int bf16, int act,
                            cudaStream_t st)
{
    if (planes <= 0) return cudaSuccess;
    return bf16 ? act_mean_dispatch<true>(v, y, planes, plane, act, st)
                : act_mean_dispatch<false>(v, y, planes, plane, act, st);
}

cudaError_t lse_row_launch(const float* t, float* out, int M, int N, float scale, float lo, float hi, cudaStream_t st)
{
    if (M <= 0) return cudaSuccess;
    // the base-2 constants, each rounded once from double
    const double log2e = 1.4426950408889634;
    const float k2 = static_cast<float>(2.0 * static_cast<double>(scale) * log2e);
    const float lo2 = static_cast<float>(static_cast<double>(lo) * log2e);
    const float hi2 = static_cast<float>(static_cast<double>(hi) * log2e);
    // a programmatic dependent launch: the CTAs may be scheduled while the previous kernel on
    // the stream finishes; each waits for its results before reading t
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(kRedThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lse_row_kernel, t, out, N, k2, lo2, hi2);
}

}  // namespace fc
