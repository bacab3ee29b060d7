// fc_linear.cu -- fused Linear + bias -> x*scale -> x+x -> clamp -> row logsumexp
// -> x*mish(x) (page "Kimi-K2.6 l2_p22": the module's forward; the stable
// logsumexp and the streaming "running max with rescaled sum" it weighs).
//
// Main kernel: persistent TF32 (fp32 inputs) or BF16 GEMM on tcgen05.  Tile
// 128 x 256 x (one 128-byte row of K: 32 fp32 or 64 bf16); both operands are K-major (x [M][K] rows and nn.Linear's W [Nout][K] rows are
// contiguous in K), loaded by TMA with 128-byte swizzle into a 4-stage
// shared-memory ring; the accumulator lives in tensor memory, double-buffered
// (2 x 256 columns) so the epilogue of tile i overlaps the MMAs of tile i+1.
// The epilogue reads each accumulator row, applies bias, the two scalings and
// the clamp, and reduces the 256 columns to one (max, sum exp(t - max)) pair
// with the online rescaling update; the pairs of all column tiles of a row are
// merged by a second, one-thread-per-row kernel in fixed order, which also
// applies the x * mish(x) tail.  The (M x Nout) intermediate never exists.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 tensor-memory
// allocator + MMA issuer, warps 2-5 epilogue (lane quarter = warp % 4).
#include "fc_ptx.cuh"

#include <cudaTypedefs.h>

#include <algorithm>

namespace fc {
namespace {

constexpr int kBM = 128, kBN = 256, kStages = 4;
constexpr int kKRowBytes = 128;                       // K per stage: one 128-byte swizzle row
template <bool BF16>
constexpr int kKElems = BF16 ? kKRowBytes / 2 : kKRowBytes / 4;   // its elements: 32 fp32 or 64 bf16
constexpr uint32_t kABytes = kBM * kKRowBytes;        // 16 KB
constexpr uint32_t kBBytes = kBN * kKRowBytes;        // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kBarOff = kStages * (kABytes + kBBytes);
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;

struct LinArgs {
    const void* bias;   // fp32 or bf16, as x and W
    float2* partials;   // [n_blocks][M]
    int M, N, K;
    int m_blocks, n_blocks, k_blocks, num_tiles;
    int kseg;           // split TF32: K blocks per segment (k_blocks = 3 kseg), else 0
    float scale, lo, hi;
    int* status;
    long long budget;
};

template <bool BF16>
__device__ __forceinline__ float bias_at(const void* b, int n)
{
    if constexpr (BF16) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(b) + n);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        return __ldg(reinterpret_cast<const float*>(b) + n);
    }
}

// The four 32-byte K steps of one stage: kind::tf32 (K = 8) or kind::f16 with bf16 (K = 16).
template <bool BF16, bool PAIR>
__device__ __forceinline__ void mma_kstep(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    if constexpr (BF16 && PAIR) mma_f16_pair(d, ad, bd, idesc, acc);
    else if constexpr (BF16) mma_f16(d, ad, bd, idesc, acc);
    else if constexpr (PAIR) mma_tf32_pair(d, ad, bd, idesc, acc);
    else mma_tf32(d, ad, bd, idesc, acc);
}

// Split TF32 runs the K loop over three segments of K blocks: (x, W), (x, W_lo), (x_lo, W).
// The tensor core truncates the raw fp32 x and W to TF32 (their high parts); x_lo and W_lo
// hold the TF32-rounded remainders.  Returns the K block within its segment and sets the maps.
__device__ __forceinline__ int k_segment(int kb, int kseg, const CUtensorMap* tmx, const CUtensorMap* tmw,
                                         const CUtensorMap* tmx_lo, const CUtensorMap* tmw_lo,
                                         const CUtensorMap** mx, const CUtensorMap** mw)
{
    *mx = tmx;
    *mw = tmw;
    if (kseg == 0) return kb;
    const int seg = kb / kseg;
    if (seg == 1) *mw = tmw_lo;
    else if (seg == 2) *mx = tmx_lo;
    return kb - seg * kseg;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, long long budget)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > budget) break;
    }
}

// POLL: the waits poll instead of suspending (see mbar_wait); only launched while a test has
// shortened the wait budget.
template <bool BF16, bool POLL = false>
__global__ void __launch_bounds__(kThreads, 1)
    linear_lse_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                      const __grid_constant__ CUtensorMap tmx_lo, const __grid_constant__ CUtensorMap tmw_lo,
                      const LinArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kStages * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);
    uint64_t* full = bars;         // [4]
    uint64_t* empty = bars + 4;    // [4]
    uint64_t* tfull = bars + 8;    // [2]
    uint64_t* tempty = bars + 10;  // [2]
    uint64_t* mdone = bars + 12;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();   // the row combine may start its set-up; it waits for the partials

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], 4);   // lane 0 of each epilogue warp
        }
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
        if (a.kseg > 0) {
            prefetch_tmap(&tmx_lo);
            prefetch_tmap(&tmw_lo);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // x's row blocks are re-read by every column tile while W streams through the L2 once:
            // W's lines go first when the L2 needs room, so x's stay
            const uint64_t stream_ = l2_policy_evict_first();
            for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x) {
                const int mb = t % a.m_blocks, nb = t / a.m_blocks;
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!(ok = mbar_wait<POLL>(&empty[stage], phase ^ 1u, abort_flag, a.status, a.budget))) break;
                    mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes);
                    const CUtensorMap* mx;
                    const CUtensorMap* mw;
                    const int kk = k_segment(kb, a.kseg, &tmx, &tmw, &tmx_lo, &tmw_lo, &mx, &mw);
                    tma_load_2d(sA + stage * kABytes, mx, &full[stage], kk * kKElems<BF16>, mb * kBM);
                    tma_load_2d_hint(sB + stage * kBBytes, mw, &full[stage], kk * kKElems<BF16>, nb * kBN, stream_);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // after an abort, wait for the most recent fill of each slot to land
                const long long first = issued > kStages ? issued - kStages : 0;
                for (long long i = first; i < issued; ++i)
                    drain_wait(&full[i % kStages], static_cast<uint32_t>((i / kStages) & 1), kDrainBudgetCycles);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(BF16 ? kFmtBF16 : kFmtTF32, kBM, kBN);
            // Descriptors built once; stages and K steps only move the start-address
            // field (16-byte units; addresses stay below 256 KB, so no carry).
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(smem_u32(sB), 16, 1024, kLayoutSw128);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>((it >> 1) & 1);
                if (!(ok = mbar_wait<POLL>(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.budget))) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!(ok = mbar_wait<POLL>(&full[stage], phase, abort_flag, a.status, a.budget))) break;
                    const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage) * (kABytes >> 4);
                    const uint64_t bd = b_desc0 + static_cast<uint32_t>(stage) * (kBBytes >> 4);
#pragma unroll
                    for (int k = 0; k < kKRowBytes / 32; ++k)   // 32-byte K steps inside the 128-byte swizzle row
                        mma_kstep<BF16, false>(d, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit(&tfull[acc]);
            }
            mma_commit(mdone);
            drain_wait(mdone, 0, kDrainBudgetCycles);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++it) {
            const int mb = t % a.m_blocks, nb = t / a.m_blocks;
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>((it >> 1) & 1);
            const bool ok = mbar_wait<POLL>(&tfull[acc], aph, abort_flag, a.status, a.budget);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kBN);
            float run_m = -INFINITY, run_s = 0.0f;
#pragma unroll 1
            for (int c = 0; c < kBN / 32; ++c) {
                float v[32];
                tmem_ld32(tbase + static_cast<uint32_t>(c * 32), v);
                const int n0 = nb * kBN + c * 32;
                float cm = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = n0 + j;
                    if (n < a.N) {
                        float u = (v[j] + bias_at<BF16>(a.bias, n)) * a.scale;
                        u = u + u;
                        v[j] = fminf(fmaxf(u, a.lo), a.hi);
                    } else {
                        v[j] = -INFINITY;
                    }
                    cm = fmaxf(cm, v[j]);
                }
                if (cm > -INFINITY) {
                    const float nm = fmaxf(run_m, cm);
                    float s = 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) s += __expf(v[j] - nm);
                    run_s = run_s * __expf(run_m - nm) + s;
                    run_m = nm;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            const int m = mb * kBM + row;
            if (m < a.M && FC_DEBUG_OK(nb < a.n_blocks, a.status))
                a.partials[static_cast<size_t>(nb) * a.M + m] = make_float2(run_m, run_s);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}


// ---------------------------------------------------------------- CTA-pair variant
//
// Two CTAs of a cluster compute one 256 x 256 tile with M = 256 MMAs
// (tcgen05 cta_group::2): CTA r holds rows 128r..128r+127 of the x tile and rows
// 128r..128r+127 of the W tile (half of N), so per SM the operand fetch per MMA
// halves for W while the MMA's work per SM is unchanged.  Both CTAs' TMA loads
// signal the leader's (rank 0) stage barrier; the leader issues the MMAs and
// multicasts its commits to both CTAs' barriers; each CTA's epilogue reads its
// own 128 accumulator rows and tells the leader through a remote arrive.
constexpr int kPBM = 128;                                  // rows per CTA (256 per pair)
constexpr int kPBN = 256;                                  // most columns per pair tile
constexpr int kPStages = 6;
constexpr uint32_t kPABytes = kPBM * kKRowBytes;           // 16 KB
constexpr uint32_t kPBBytes = (kPBN / 2) * kKRowBytes;     // 16 KB: stage slot for this CTA's half of W
constexpr uint32_t kPBarOff = kPStages * (kPABytes + kPBBytes);
constexpr uint32_t kPSmemBytes = kPBarOff + 256 + 1024;

struct LinPairArgs {
    const void* bias;   // fp32 or bf16, as x and W
    float2* partials;   // [n_blocks][M]
    int M, N, K;
    int m_pairs, n_blocks, k_blocks, num_tiles;
    int kseg;           // split TF32: K blocks per segment (k_blocks = 3 kseg), else 0
    int bn;             // columns per pair tile: a multiple of 32, <= kPBN
    float scale, lo, hi;
    int* status;
    long long budget;
};

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    linear_lse_pair_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                           const __grid_constant__ CUtensorMap tmx_lo, const __grid_constant__ CUtensorMap tmw_lo,
                           const LinPairArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + kPStages * kPABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPBarOff);
    uint64_t* full = bars;            // [6] leader: both CTAs' stage bytes landed
    uint64_t* empty = bars + 6;       // [6] both: stage consumed (multicast commit)
    uint64_t* tfull = bars + 12;      // [2] both: accumulator ready (multicast commit)
    uint64_t* tempty = bars + 14;     // [2] leader: both CTAs' epilogues drained it
    uint64_t* mdone = bars + 16;      // leader: every MMA completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    pdl_launch_dependents();   // the row combine may start its set-up; it waits for the partials

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], 8);   // lane 0 of the 4 epilogue warps of each CTA
        }
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
        if (a.kseg > 0) {
            prefetch_tmap(&tmx_lo);
            prefetch_tmap(&tmw_lo);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();   // barriers of both CTAs initialised before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // x's row blocks are re-read by every column tile while W streams through the L2 once:
            // W's lines go first when the L2 needs room, so x's stay
            const uint64_t stream_ = l2_policy_evict_first();
            for (int t = cluster; ok && t < a.num_tiles; t += nclusters) {
                const int mp = t % a.m_pairs, nb = t / a.m_pairs;
                const int m0 = mp * 2 * kPBM + static_cast<int>(rank) * kPBM;
                const int n0 = nb * a.bn + static_cast<int>(rank) * (a.bn / 2);
                const uint32_t b_bytes = static_cast<uint32_t>(a.bn / 2) * kKRowBytes;
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!(ok = mbar_wait_cluster(&empty[stage], phase ^ 1u, abort_flag, a.status, a.budget))) break;
                    const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (kPABytes + b_bytes));
                    const CUtensorMap* mx;
                    const CUtensorMap* mw;
                    const int kk = k_segment(kb, a.kseg, &tmx, &tmw, &tmx_lo, &tmw_lo, &mx, &mw);
                    tma_load_2d_pair(sA + stage * kPABytes, mx, fbar, kk * kKElems<BF16>, m0);
                    tma_load_2d_pair_hint(sB + stage * kPBBytes, mw, fbar, kk * kKElems<BF16>, n0, stream_);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // after an abort, give copies already issued time to land before the CTA exits
                const long long t0 = clock64();
                while (clock64() - t0 < kDrainBudgetCycles / 8) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader only)
        if (leader && lane == 0) {
            const uint32_t idesc = make_idesc(BF16 ? kFmtBF16 : kFmtTF32, 2 * kPBM, a.bn);
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024, kLayoutSw128);
            const uint64_t b_desc0 = smem_desc(smem_u32(sB), 16, 1024, kLayoutSw128);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int t = cluster; ok && t < a.num_tiles; t += nclusters, ++it) {
                const int acc = it & 1;
                const uint32_t aph = static_cast<uint32_t>((it >> 1) & 1);
                if (!(ok = mbar_wait_cluster(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.budget))) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kPBN);
                for (int kb = 0; kb < a.k_blocks; ++kb) {
                    if (!(ok = mbar_wait_cluster(&full[stage], phase, abort_flag, a.status, a.budget))) break;
                    const uint64_t ad = a_desc0 + static_cast<uint32_t>(stage) * (kPABytes >> 4);
                    const uint64_t bd = b_desc0 + static_cast<uint32_t>(stage) * (kPBBytes >> 4);
#pragma unroll
                    for (int k = 0; k < kKRowBytes / 32; ++k)
                        mma_kstep<BF16, true>(d, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) mma_commit_pair_multicast(&tfull[acc], 0x3);
            }
            mma_commit_pair_multicast(mdone, 0x1);
            const long long t0 = clock64();
            while (!mbar_try_wait(mdone, 0) && clock64() - t0 < kDrainBudgetCycles) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int it = 0;
        for (int t = cluster; t < a.num_tiles; t += nclusters, ++it) {
            const int mp = t % a.m_pairs, nb = t / a.m_pairs;
            const int acc = it & 1;
            const uint32_t aph = static_cast<uint32_t>((it >> 1) & 1);
            const bool ok = mbar_wait_cluster(&tfull[acc], aph, abort_flag, a.status, a.budget);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kPBN);
            float run_m = -INFINITY, run_s = 0.0f;
#pragma unroll 1
            for (int c = 0; c < a.bn / 32; ++c) {
                float v[32];
                tmem_ld32(tbase + static_cast<uint32_t>(c * 32), v);
                const int n0 = nb * a.bn + c * 32;
                float cm = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = n0 + j;
                    if (n < a.N) {
                        float u = (v[j] + bias_at<BF16>(a.bias, n)) * a.scale;
                        u = u + u;
                        v[j] = fminf(fmaxf(u, a.lo), a.hi);
                    } else {
                        v[j] = -INFINITY;
                    }
                    cm = fmaxf(cm, v[j]);
                }
                if (cm > -INFINITY) {
                    const float nm = fmaxf(run_m, cm);
                    float s = 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) s += __expf(v[j] - nm);
                    run_s = run_s * __expf(run_m - nm) + s;
                    run_m = nm;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
            const int m = mp * 2 * kPBM + static_cast<int>(rank) * kPBM + row;
            if (m < a.M && FC_DEBUG_OK(nb < a.n_blocks, a.status))
                a.partials[static_cast<size_t>(nb) * a.M + m] = make_float2(run_m, run_s);
        }
    }

    tc_fence_before();
    cluster_sync();   // the leader's MMAs into both CTAs' tensor memory are complete
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// Merge the per-column-tile (max, sum) pairs of each row in fixed order, then
// lse = M + log S and y = lse * mish(lse), mish(l) = l * tanh(softplus(l)).
__global__ void lse_combine_kernel(const float2* partials, float* y, int M, int n_blocks, int* status)
{
    pdl_wait();   // the GEMM's partials are complete and visible
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m >= M) return;
    // a bounded wait that gave up (or a failed index check of a debug build) leaves partials the
    // GEMM never wrote: say so in the output
    if (*reinterpret_cast<const volatile int*>(status) != 0) {
        y[m] = __int_as_float(0x7fc00000);
        return;
    }
    float mx = -INFINITY;
    for (int i = 0; i < n_blocks; ++i) mx = fmaxf(mx, partials[static_cast<size_t>(i) * M + m].x);
    float s = 0.0f;
    for (int i = 0; i < n_blocks; ++i) {
        const float2 p = partials[static_cast<size_t>(i) * M + m];
        s += p.y * expf(p.x - mx);
    }
    const float l = mx + logf(s);
    const float sp = fmaxf(l, 0.0f) + log1pf(expf(-fabsf(l)));
    y[m] = l * (l * tanhf(sp));
}

// The row combine, launched so that it may start while the GEMM finishes (it waits for the
// partials itself).
cudaError_t launch_lse_combine(const float2* partials, float* y, int M, int n_blocks, int* status,
                               cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>((M + 127) / 128));
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lse_combine_kernel, partials, y, M, n_blocks, status);
}

// Row-major [rows][cols] fp32 or bf16 matrix, box = box_rows x one 128-byte row of K, 128-byte swizzle.
bool make_kmajor_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows, bool bf16)
{
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
    if (enc == nullptr) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * es};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kKRowBytes / es), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                     const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Split-TF32 operands (the FC_F32_3XTF32 precision of the Linear op).  The tensor core reads
// raw fp32 operands as TF32 by dropping their 13 low mantissa bits, so the high part of a value
// v is hi = v with those bits cleared, and the GEMM reads it straight from x and W.  This kernel
// writes the remainders lo = (v - hi) rounded to TF32 (v - hi is exact in fp32): |lo| < 2^-10
// |v|, and lo's own rounding error is below 2^-22 |v|.  The GEMM's three K segments then sum
// hi*hi + hi*lo + lo*hi for every term -- the product less lo*lo (< 2^-20 of it).
__global__ void tf32_remainder_kernel(const float4* __restrict__ src, float4* __restrict__ dst, long long n4)
{
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 v = src[i];
        float4 l;
        l.x = to_tf32(v.x - __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u));
        l.y = to_tf32(v.y - __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u));
        l.z = to_tf32(v.z - __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u));
        l.w = to_tf32(v.w - __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u));
        dst[i] = l;
    }
}

size_t align256_sz(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t linear_split_bytes(int M, int K, int Nout)
{
    return align256_sz(static_cast<size_t>(M) * K * sizeof(float)) +
           align256_sz(static_cast<size_t>(Nout) * K * sizeof(float));
}

cudaError_t linear_split_launch(const float* x, const float* W, int M, int K, int Nout, void* dst, int sm_count,
                                cudaStream_t stream, const float** x_lo, const float** W_lo)
{
    float* a = static_cast<float*>(dst);
    float* w = reinterpret_cast<float*>(static_cast<char*>(dst) +
                                        align256_sz(static_cast<size_t>(M) * K * sizeof(float)));
    const unsigned blocks = static_cast<unsigned>(std::max(sm_count, 1) * 8);
    tf32_remainder_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(x), reinterpret_cast<float4*>(a),
                                                      static_cast<long long>(M) * K / 4);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    tf32_remainder_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(W), reinterpret_cast<float4*>(w),
                                                      static_cast<long long>(Nout) * K / 4);
    e = cudaGetLastError();
    *x_lo = a;
    *W_lo = w;
    return e;
}

void* tensor_map_encoder()
{
    static void* fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    }
    return fn;
}

int linear_plan(LinearPlan* p, int M, int K, int Nout, int bf16, int sm_count, int split)
{
    *p = LinearPlan{};
    // TMA needs a 16-byte row pitch: K a multiple of 4 fp32 or 8 bf16
    if (K % (bf16 ? 8 : 4) != 0) return 2;
    if (split && bf16) return 2;
    p->M = M; p->K = K; p->Nout = Nout; p->bf16 = bf16;
    p->m_blocks = (M + kBM - 1) / kBM;
    p->n_blocks = (Nout + kBN - 1) / kBN;
    const int kelems = bf16 ? kKElems<true> : kKElems<false>;
    p->k_blocks = (K + kelems - 1) / kelems;
    // split TF32: three segments of K blocks, (x, W), (x, W_lo), (x_lo, W)
    p->kseg = split ? p->k_blocks : 0;
    if (split) p->k_blocks *= 3;
    const long long tiles = static_cast<long long>(p->m_blocks) * p->n_blocks;
    if (tiles > 0x7FFFFFFFLL) return 2;
    p->num_tiles = static_cast<int>(tiles);
    p->grid = std::min(p->num_tiles, std::max(sm_count, 1));
    p->smem_bytes = kSmemBytes;
    // CTA pairs (M = 256 MMAs) once there is more than one 128-row block
    p->use_pair = M > kBM && sm_count >= 2;
    if (p->use_pair) {
        // Tile width: the multiple of 32 in [128, 256] that minimises waves x width (ties go to
        // the wider tile), so that the last wave of pair tiles leaves few clusters idle.
        p->m_pairs = (M + 2 * kPBM - 1) / (2 * kPBM);
        const long long clusters = std::max(sm_count / 2, 1);
        long long best = -1;
        for (int bn = kPBN; bn >= 128; bn -= 32) {
            const long long tiles = static_cast<long long>(p->m_pairs) * ((Nout + bn - 1) / bn);
            const long long cost = (tiles + clusters - 1) / clusters * bn;
            if (best < 0 || cost < best) {
                best = cost;
                p->bn = bn;
            }
        }
        p->n_blocks = (Nout + p->bn - 1) / p->bn;
        const long long ptiles = static_cast<long long>(p->m_pairs) * p->n_blocks;
        if (ptiles > 0x7FFFFFFFLL) return 2;
        p->num_tiles = static_cast<int>(ptiles);
        p->grid = 2 * static_cast<int>(std::min<long long>(p->num_tiles, clusters));
        p->smem_bytes = kPSmemBytes;
    }
    p->ws_bytes = (static_cast<size_t>(p->n_blocks) * M * sizeof(float2) + 255) & ~static_cast<size_t>(255);
    return 0;
}

cudaError_t linear_launch(const LinearPlan& p, const void* x, const void* W, const void* b, float* y, float scale,
                          float lo, float hi, void* workspace, cudaStream_t stream, int* status, long long budget,
                          const void* x_lo, const void* W_lo)
{
    CUtensorMap tmx, tmw, tmxl, tmwl;
    const bool bf16 = p.bf16 != 0;
    // split TF32 reads the remainders through their own maps; otherwise those maps repeat x and W
    if (p.kseg > 0 && (x_lo == nullptr || W_lo == nullptr)) return cudaErrorInvalidValue;
    const void* xl = p.kseg > 0 ? x_lo : x;
    const void* wl = p.kseg > 0 ? W_lo : W;
    if (p.use_pair) {
        if (polling_budget(budget)) return cudaErrorNotSupported;   // no polling instantiation of the pair kernel
        if (!make_kmajor_map(&tmx, x, p.M, p.K, kPBM, bf16) || !make_kmajor_map(&tmw, W, p.Nout, p.K, p.bn / 2, bf16) ||
            !make_kmajor_map(&tmxl, xl, p.M, p.K, kPBM, bf16) ||
            !make_kmajor_map(&tmwl, wl, p.Nout, p.K, p.bn / 2, bf16))
            return cudaErrorInvalidValue;
        LinPairArgs a{};
        a.bias = b;
        a.partials = reinterpret_cast<float2*>(workspace);
        a.M = p.M; a.N = p.Nout; a.K = p.K;
        a.m_pairs = p.m_pairs; a.n_blocks = p.n_blocks; a.k_blocks = p.k_blocks; a.num_tiles = p.num_tiles;
        a.kseg = p.kseg;
        a.bn = p.bn;
        a.scale = scale; a.lo = lo; a.hi = hi;
        a.status = status; a.budget = budget;
        auto kern = bf16 ? linear_lse_pair_kernel<true> : linear_lse_pair_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(p.smem_bytes));
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = p.smem_bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, tmx, tmw, tmxl, tmwl, a);
        if (e != cudaSuccess) return e;
        return launch_lse_combine(a.partials, y, p.M, p.n_blocks, status, stream);
    }
    if (!make_kmajor_map(&tmx, x, p.M, p.K, kBM, bf16) || !make_kmajor_map(&tmw, W, p.Nout, p.K, kBN, bf16) ||
        !make_kmajor_map(&tmxl, xl, p.M, p.K, kBM, bf16) || !make_kmajor_map(&tmwl, wl, p.Nout, p.K, kBN, bf16))
        return cudaErrorInvalidValue;
    LinArgs a{};
    a.bias = b;
    a.partials = reinterpret_cast<float2*>(workspace);
    a.M = p.M; a.N = p.Nout; a.K = p.K;
    a.m_blocks = p.m_blocks; a.n_blocks = p.n_blocks; a.k_blocks = p.k_blocks; a.num_tiles = p.num_tiles;
    a.kseg = p.kseg;
    a.scale = scale; a.lo = lo; a.hi = hi;
    a.status = status; a.budget = budget;
    if (polling_budget(budget) && bf16) return cudaErrorNotSupported;
    auto kern = bf16 ? linear_lse_kernel<true> : (polling_budget(budget) ? linear_lse_kernel<false, true> : linear_lse_kernel<false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(p.smem_bytes));
    if (e != cudaSuccess) return e;
    kern<<<p.grid, kThreads, p.smem_bytes, stream>>>(tmx, tmw, tmxl, tmwl, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_lse_combine(a.partials, y, p.M, p.n_blocks, status, stream);
}

}  // namespace fc
