// fc_conv_kernel.cuh -- fused conv3x3 (stride 1, padding 0) + bias + activation, with
// either a global-mean epilogue (Conv2d -> GELU -> adaptive_avg_pool2d(1) page,
// "Kimi-K2.6 l2_p67") or a full-output epilogue (Conv2d -> Mish -> Mish page,
// "Kimi-K2.6 l2_p4"), as an implicit GEMM on tcgen05 tensor cores.
//
// GEMM view (the Mish page's implicit-GEMM sizing: M x N x K =
// pixels x Cout x Cin*9):  D[pixel, co] = sum_{ci, kh, kw} x[ci, oh+kh, ow+kw] * w[co, ci, kh, kw].
//
// Tile: M = 128 output pixels arranged as a 16-row x 8-column patch, N = Cout
// (<= 256), K stepped as (K block of 8 fp32 / 16 bf16 input channels) x (9 taps).
//
// The operand trick that makes shifted windows free: the producer warps stage
// the input patch plus its halo (18 rows x 10 columns) in shared memory as
// "channel-blocked pixels": for every staged pixel one 16-byte row holding 4
// fp32 (or 8 bf16) consecutive channels.  In the tensor core's K-major,
// no-swizzle canonical layout a core matrix is 8 rows x 16 bytes, so 8
// consecutive staged pixels of one row form a core matrix, the next output row
// is SBO = 10 pixels * 16 B = 160 B further, and the second channel group of
// the K step is LBO = one group plane further.  A tap (kh, kw) is then just the
// start address moved by (kh * 10 + kw) * 16 bytes -- 16-byte aligned for every
// tap, so all nine taps read the one staged strip with no copies and no
// extra FLOPs.  Weights are re-laid once per call into the same form
// ([K block][tap][channel half][co][4 or 8 channels]) and copied with bulk
// async copies (resident in shared memory when they fit, else streamed per K
// block).
//
// Warp roles (416 threads, one CTA per SM, persistent over a contiguous tile range):
//   warps 0-7  epilogue: tcgen05.ld of the accumulator (lane quarter = warp % 4,
//              column half = warp / 4), bias + activation, then either a
//              warp-transpose sum over the 32 pixels (pool) or coalesced stores.
//   warps 8-11 producers: one shared-memory stage slot each.
//   warp 12    tensor-memory allocator and single-thread MMA issuer.
#pragma once

#include "fc_ptx.cuh"

namespace fc {
namespace convk {

constexpr int kConvThreads = 13 * 32;
constexpr int kEpiWarps = 8;
constexpr int kProdWarp0 = 8;
constexpr int kNumProd = 4;
constexpr int kMmaWarp = 12;
constexpr int kPatchRows = 16;
constexpr int kPatchCols = 8;
constexpr int kStripCols = kPatchCols + 2;               // 10
constexpr int kStripRows = kPatchRows + 2;               // 18
constexpr int kStripPos = kStripRows * kStripCols;       // 180 staged pixels
constexpr int kStripIters = (kStripPos + 31) / 32;       // 6 per lane
constexpr uint32_t kStripPlane = kStripPos * 16;         // one channel group: 2880 B
constexpr uint32_t kStripBytes = 2 * kStripPlane;        // one K block: 5760 B
constexpr uint32_t kResidentMax = 96 * 1024;
constexpr uint32_t kSmemBudget = 200 * 1024;

struct ConvArgs {
    const void* x;
    const void* wr;      // re-laid weights (workspace)
    const void* bias;
    float* out;          // full output (store) or pool partials (pool)
    int N, Cin, H, W, Cout, OH, OW;
    int ncb, CS;
    long long tpi, base;
    int rem, J, stages, resident, nacc, tmem_cols;
    uint32_t w_block_bytes, w_total_bytes, strip_off, w_off, bar_off;
    int* status;
    long long budget;
};

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

__device__ __forceinline__ float softplus_stable(float z) { return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z))); }

__device__ __forceinline__ float mish(float z) { return z * tanhf(softplus_stable(z)); }

// Activation codes follow fc_act: 0 erf-GELU, 1 Mish, 2 Mish twice.
template <int ACT>
__device__ __forceinline__ float apply_act(float z)
{
    if constexpr (ACT == 0) return gelu_erf(z);
    else if constexpr (ACT == 1) return mish(z);
    else return mish(mish(z));
}

template <bool BF16>
__device__ __forceinline__ float load_bias(const void* b, int co)
{
    if constexpr (BF16) {
        const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(b) + co);
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    } else {
        return __ldg(reinterpret_cast<const float*>(b) + co);
    }
}

// After the call lane L holds sum over the warp's 32 lanes of v[L] (v is clobbered).
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane)
{
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = upper ? v[i] : v[i + w];
            const float keep = upper ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// Tile t of the flattened (image, row block, column strip) grid.
struct TileCoord {
    int n, oh0, ow0;
};

__device__ __forceinline__ TileCoord tile_coord(long long t, long long tpi, int CS)
{
    TileCoord c;
    c.n = static_cast<int>(t / tpi);
    const int r = static_cast<int>(t - static_cast<long long>(c.n) * tpi);
    const int rb = r / CS;
    c.oh0 = rb * kPatchRows;
    c.ow0 = (r - rb * CS) * kPatchCols;
    return c;
}

// Stage one K block of the 18 x 10 halo patch as [group][pixel][16 B].
template <bool BF16>
__device__ __forceinline__ void fill_strip(uint32_t strip, const void* xv, int n, int cb, int oh0, int ow0,
                                           int Cin, int H, int W, int lane)
{
    const size_t HW = static_cast<size_t>(H) * W;
    if constexpr (!BF16) {
        const float* x = reinterpret_cast<const float*>(xv);
        const int ci0 = cb * 8;
        float v[kStripIters][8];
#pragma unroll
        for (int i = 0; i < kStripIters; ++i) {
            const int s = lane + 32 * i;
            const int rr = s / kStripCols, cc = s - (s / kStripCols) * kStripCols;
            const int ih = oh0 + rr, iw = ow0 + cc;
            const bool ok = (s < kStripPos) && ih < H && iw < W;
            const size_t off = ok ? ((static_cast<size_t>(n) * Cin + ci0) * HW + static_cast<size_t>(ih) * W + iw) : 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = (ok && ci0 + e < Cin) ? __ldg(x + off + e * HW) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kStripIters; ++i) {
            const int s = lane + 32 * i;
            if (s < kStripPos) {
                const uint32_t a = strip + static_cast<uint32_t>(s) * 16u;
                st_shared_v4(a, __float_as_uint(to_tf32(v[i][0])), __float_as_uint(to_tf32(v[i][1])),
                             __float_as_uint(to_tf32(v[i][2])), __float_as_uint(to_tf32(v[i][3])));
                st_shared_v4(a + kStripPlane, __float_as_uint(to_tf32(v[i][4])), __float_as_uint(to_tf32(v[i][5])),
                             __float_as_uint(to_tf32(v[i][6])), __float_as_uint(to_tf32(v[i][7])));
            }
        }
    } else {
        const unsigned short* x = reinterpret_cast<const unsigned short*>(xv);
        const int ci0 = cb * 16;
        uint32_t v[kStripIters][8];
#pragma unroll
        for (int i = 0; i < kStripIters; ++i) {
            const int s = lane + 32 * i;
            const int rr = s / kStripCols, cc = s - (s / kStripCols) * kStripCols;
            const int ih = oh0 + rr, iw = ow0 + cc;
            const bool ok = (s < kStripPos) && ih < H && iw < W;
            const size_t off = ok ? ((static_cast<size_t>(n) * Cin + ci0) * HW + static_cast<size_t>(ih) * W + iw) : 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t lo = (ok && ci0 + 2 * e < Cin) ? __ldg(x + off + (2 * e) * HW) : 0u;
                const uint32_t hi = (ok && ci0 + 2 * e + 1 < Cin) ? __ldg(x + off + (2 * e + 1) * HW) : 0u;
                v[i][e] = lo | (hi << 16);
            }
        }
#pragma unroll
        for (int i = 0; i < kStripIters; ++i) {
            const int s = lane + 32 * i;
            if (s < kStripPos) {
                const uint32_t a = strip + static_cast<uint32_t>(s) * 16u;
                st_shared_v4(a, v[i][0], v[i][1], v[i][2], v[i][3]);
                st_shared_v4(a + kStripPlane, v[i][4], v[i][5], v[i][6], v[i][7]);
            }
        }
    }
}

// Wait with no abort check and no status write: used to drain this warp's own
// copies in flight before the CTA exits after an abort.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, long long budget)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) break;
    }
}

template <bool BF16, bool POOL, int ACT>
__global__ void __launch_bounds__(kConvThreads, 1) conv3x3_fused_kernel(const ConvArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* full = bars;        // [4] strip (+ streamed weights) ready
    uint64_t* empty = bars + 4;   // [4] stage consumed by the MMA
    uint64_t* wfull = bars + 8;   // resident weights landed
    uint64_t* tfull = bars + 9;   // [4] accumulator ready for the epilogue
    uint64_t* tempty = bars + 13; // [4] accumulator drained by the epilogue
    uint64_t* mdone = bars + 17;  // every MMA issued by this CTA completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const long long t_begin = static_cast<long long>(blockIdx.x) * a.base + min(static_cast<int>(blockIdx.x), a.rem);
    const long long n_tiles = a.base + (static_cast<int>(blockIdx.x) < a.rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&full[s], 33);
            mbar_init(&empty[s], 1);
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], kEpiWarps * 32);
        }
        mbar_init(wfull, 1);
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, static_cast<uint32_t>(a.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kProdWarp0 && warp < kProdWarp0 + kNumProd) {
        // ------------------------------------------------------------ producers
        const int pw = warp - kProdWarp0;
        if (pw < a.stages) {
            const uint32_t slot = static_cast<uint32_t>(pw);
            const uint32_t strip = smem_u32(smem + a.strip_off) + slot * kStripBytes;
            uint8_t* wslot = smem + a.w_off + (a.resident ? 0u : slot * a.w_block_bytes);
            if (a.resident && pw == 0 && lane == 0) {
                mbar_arrive_expect_tx(wfull, a.w_total_bytes);
                bulk_g2s(smem + a.w_off, a.wr, a.w_total_bytes, wfull);
            }
            const long long total = n_tiles * a.ncb;
            uint32_t use = 0;
            for (long long g = pw; g < total; g += a.stages, ++use) {
                bool ok = mbar_wait(&empty[slot], (use & 1u) ^ 1u, abort_flag, a.status, a.budget);
                if (!__all_sync(0xffffffffu, ok)) break;
                fence_proxy_async_smem();
                const long long lt = g / a.ncb;
                const int cb = static_cast<int>(g - lt * a.ncb);
                const TileCoord tc = tile_coord(t_begin + lt, a.tpi, a.CS);
                if (lane == 0) {
                    if (!a.resident) {
                        mbar_arrive_expect_tx(&full[slot], a.w_block_bytes);
                        bulk_g2s(wslot, reinterpret_cast<const uint8_t*>(a.wr) + static_cast<size_t>(cb) * a.w_block_bytes,
                                 a.w_block_bytes, &full[slot]);
                    } else {
                        mbar_arrive(&full[slot]);
                    }
                }
                fill_strip<BF16>(strip, a.x, tc.n, cb, tc.oh0, tc.ow0, a.Cin, a.H, a.W, lane);
                fence_proxy_async_smem();
                mbar_arrive(&full[slot]);
            }
            if (*abort_flag && lane == 0) {
                if (!a.resident && use > 0) drain_wait(&full[slot], (use - 1u) & 1u, a.budget);
                if (a.resident && pw == 0) drain_wait(wfull, 0, a.budget);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(BF16 ? kFmtBF16 : kFmtTF32, 128, a.Cout);
            const uint32_t strip0 = smem_u32(smem + a.strip_off);
            const uint32_t w0 = smem_u32(smem + a.w_off);
            const uint32_t wtap = 2u * static_cast<uint32_t>(a.Cout) * 16u;
            const uint32_t w_lbo = static_cast<uint32_t>(a.Cout) * 16u;
            bool ok = true;
            if (a.resident) ok = mbar_wait(wfull, 0, abort_flag, a.status, a.budget);
            long long g = 0;
            for (long long lt = 0; ok && lt < n_tiles; ++lt) {
                const int acc = static_cast<int>(lt % a.nacc);
                const uint32_t aph = static_cast<uint32_t>((lt / a.nacc) & 1);
                if (!(ok = mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.budget))) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * a.Cout);
                for (int cb = 0; cb < a.ncb; ++cb, ++g) {
                    const uint32_t slot = static_cast<uint32_t>(g % a.stages);
                    const uint32_t use = static_cast<uint32_t>(g / a.stages);
                    if (!(ok = mbar_wait(&full[slot], use & 1u, abort_flag, a.status, a.budget))) break;
                    tc_fence_after();
                    const uint32_t abase = strip0 + slot * kStripBytes;
                    const uint32_t bbase = w0 + (a.resident ? static_cast<uint32_t>(cb) : slot) * a.w_block_bytes;
#pragma unroll
                    for (int tap = 0; tap < 9; ++tap) {
                        const int kh = tap / 3, kw = tap - (tap / 3) * 3;
                        const uint64_t ad =
                            smem_desc(abase + static_cast<uint32_t>(kh * kStripCols + kw) * 16u, kStripPlane,
                                      kStripCols * 16u, kLayoutNone);
                        const uint64_t bd = smem_desc(bbase + static_cast<uint32_t>(tap) * wtap, w_lbo, 128u, kLayoutNone);
                        const uint32_t accum = (cb | tap) != 0 ? 1u : 0u;
                        if constexpr (BF16) mma_f16(d, ad, bd, idesc, accum);
                        else mma_tf32(d, ad, bd, idesc, accum);
                    }
                    mma_commit(&empty[slot]);
                }
                if (ok) mma_commit(&tfull[acc]);
            }
            mma_commit(mdone);
            drain_wait(mdone, 0, a.budget);
        }
        __syncwarp();
    } else if (warp < kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int h = warp >> 2;
        const int nchunks = a.Cout / 32;
        const int r = q * 32 + lane;
        const int pr = r >> 3, pc = r & 7;
        const long long n_first = t_begin / a.tpi;
        float psum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int cur_n = -1;
        bool ok = true;

        auto flush = [&](int n_img) {
            float* dst = a.out + ((static_cast<size_t>(blockIdx.x) * a.J + static_cast<size_t>(n_img - n_first)) * 4 + q) *
                                     static_cast<size_t>(a.Cout);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = h + 2 * k;
                if (c < nchunks) dst[c * 32 + lane] = psum[k];
                psum[k] = 0.0f;
            }
        };

        for (long long lt = 0; lt < n_tiles; ++lt) {
            const TileCoord tc = tile_coord(t_begin + lt, a.tpi, a.CS);
            if constexpr (POOL) {
                if (tc.n != cur_n) {
                    if (cur_n >= 0) flush(cur_n);
                    cur_n = tc.n;
                }
            }
            const int acc = static_cast<int>(lt % a.nacc);
            const uint32_t aph = static_cast<uint32_t>((lt / a.nacc) & 1);
            ok = mbar_wait(&tfull[acc], aph, abort_flag, a.status, a.budget);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int oh = tc.oh0 + pr, ow = tc.ow0 + pc;
            const bool valid = oh < a.OH && ow < a.OW;
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * a.Cout);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = h + 2 * k;
                if (c < nchunks) {
                    float v[32];
                    tmem_ld32(tbase + static_cast<uint32_t>(c * 32), v);
                    if constexpr (POOL) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float z = v[j] + load_bias<BF16>(a.bias, c * 32 + j);
                            v[j] = valid ? apply_act<ACT>(z) : 0.0f;
                        }
                        psum[k] += warp_transpose_sum(v, lane);
                    } else {
                        if (valid) {
                            float* o = a.out + ((static_cast<size_t>(tc.n) * a.Cout + c * 32) * a.OH + oh) *
                                                   static_cast<size_t>(a.OW) + ow;
                            const size_t plane = static_cast<size_t>(a.OH) * a.OW;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float z = v[j] + load_bias<BF16>(a.bias, c * 32 + j);
                                o[j * plane] = apply_act<ACT>(z);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
        }
        if constexpr (POOL) {
            if (ok && cur_n >= 0) flush(cur_n);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, static_cast<uint32_t>(a.tmem_cols));
    }
}

template <bool BF16, bool POOL, int ACT>
cudaError_t launch_variant(const ConvArgs& a, int grid, uint32_t smem_bytes, cudaStream_t stream)
{
    auto kern = conv3x3_fused_kernel<BF16, POOL, ACT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
    if (e != cudaSuccess) return e;
    kern<<<grid, kConvThreads, smem_bytes, stream>>>(a);
    return cudaGetLastError();
}

// One instantiation per (pool, activation) for the given operand type; defined
// in fc_conv_tf32.cu and fc_conv_bf16.cu so the variants compile in parallel.
cudaError_t launch_main_tf32(const ConvArgs& a, int pool, int act, int grid, uint32_t smem_bytes, cudaStream_t stream);
cudaError_t launch_main_bf16(const ConvArgs& a, int pool, int act, int grid, uint32_t smem_bytes, cudaStream_t stream);

}  // namespace convk
}  // namespace fc
