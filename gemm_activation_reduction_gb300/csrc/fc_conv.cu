// fc_conv.cu -- host side of the fused conv3x3 operators: the launch plan
// (tiling, pipeline depth, tensor-memory buffers, workspace layout), the
// once-per-call weight re-layout kernel, the fixed-order pool combine kernel,
// and the launch sequence.  The fused kernel itself is in fc_conv_kernel.cuh.
#include "fc_conv_kernel.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

namespace fc {
using namespace convk;
namespace {

// Re-lay w [Co][Cin][3][3] for `halves` CTAs of a group (2 for a CTA pair, else 1) as
// Cout >= Co channels (Cout a multiple of 16; channels past Co get zero weights and bias):
// CTA r holds output channels [r hc, (r+1) hc), hc = Cout / halves.  Layout
// [r][K stage][tap][half][co'][G]
// (G = 4 fp32 rounded to TF32, or 8 bf16; co' the channel within the half),
// zero-padding channels past Cin.  With parts = 3 (split TF32) every K block of
// channels is three consecutive K stages whose B operands are the TF32 high part,
// the TF32 remainder w - hi, and the high part again (the A side stages x_hi, x_hi,
// x_lo), so the stages sum hi*hi + hi*lo + lo*hi.  Then the B operands of the bias K step,
// [r][half][co'][G]: half 0 holds the bias (fp32: its TF32 high part in k 0 and
// the TF32 remainder in k 2; bf16: the bias in k 0) and the padding value in k 1;
// half 1 is zero.
template <bool BF16>
__global__ void conv_weight_relayout_kernel(const void* w, const void* b, void* wr, int Cin, int Co, int Cout,
                                            int ncb, int halves, int parts)
{
    // the fused kernel may start its set-up now; it waits for these writes before reading them
    pdl_launch_dependents();
    // 32-bit index arithmetic: the plan keeps the re-laid tensor at 2^30 elements at most
    constexpr int G = BF16 ? 8 : 4;
    const int hc = Cout / halves;
    const int wtotal = halves * ncb * 9 * 2 * hc * G;
    const int total = wtotal + halves * 2 * hc * G;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        int f = i < wtotal ? i : i - wtotal;
        const int e = f % G;
        f /= G;
        const int col = f % hc;
        f /= hc;
        const int half = f % 2;
        f /= 2;
        if (i >= wtotal) {
            // f = rank
            const int co = f * hc + col;
            if constexpr (BF16) {
                const unsigned short bv = co < Co ? reinterpret_cast<const unsigned short*>(b)[co] : 0;
                const unsigned short pad = static_cast<unsigned short>(__float_as_uint(kPadValue) >> 16);
                unsigned short v = 0;
                if (half == 0 && e == 0) v = bv;
                if (half == 0 && e == 1) v = pad;
                reinterpret_cast<unsigned short*>(wr)[i] = v;
            } else {
                const float bv = co < Co ? reinterpret_cast<const float*>(b)[co] : 0.0f;
                const float hi = to_tf32(bv);
                float v = 0.0f;
                if (half == 0 && e == 0) v = hi;
                if (half == 0 && e == 1) v = kPadValue;
                if (half == 0 && e == 2) v = to_tf32(bv - hi);
                reinterpret_cast<float*>(wr)[i] = v;
            }
            continue;
        }
        const int tap = f % 9;
        f /= 9;
        const int kb = f % ncb;
        const int rank = f / ncb;
        const int co = rank * hc + col;
        const int cb = kb / parts;
        const bool lo_part = parts == 3 && kb - cb * parts == 1;
        const int ci = cb * 2 * G + half * G + e;
        const size_t src = (static_cast<size_t>(co) * Cin + ci) * 9 + tap;
        const bool real = ci < Cin && co < Co;
        if constexpr (BF16) {
            const unsigned short* ws = reinterpret_cast<const unsigned short*>(w);
            reinterpret_cast<unsigned short*>(wr)[i] = real ? ws[src] : static_cast<unsigned short>(0);
        } else {
            const float* ws = reinterpret_cast<const float*>(w);
            const float v = real ? ws[src] : 0.0f;
            const float hi = to_tf32(v);
            reinterpret_cast<float*>(wr)[i] = lo_part ? to_tf32(v - hi) : hi;
        }
    }
}

// y[n, co] = (fixed-order sum of every image-n record of the CTAs whose tiles can touch
// image n) / (OH * OW), for co < Co; records hold Cout >= Co channels.  Cluster c handles tile
// groups [P(c), P(c+1)) of `step` tiles (2 for CTA pairs, else 1); its CTA r handles tiles
// step * g + r.  Records a CTA never reached hold zeros.  One warp per 4 consecutive channels of
// an image: record k of the image's list (cluster, CTA of the cluster, record) goes to lane
// k % 32, which loads the 4 channels with one 16-byte load (Cout is a multiple of 16) and sums
// its records in order; a fixed shuffle tree adds the lanes -- the same order on every run.
// The sums are fp32: a few dozen partial sums per output, each already a sum over thousands of
// values, so the rounding stays near 1e-6 relative, far inside every tolerance; fp64 adds and
// shuffles took about a third of this kernel's time on this GPU.
__global__ void conv_pool_combine_kernel(const float* ws, float* y, int N, int Co, int Cout, long long tpi,
                                         long long pbase, int prem, int J, int step, int recs, double inv_count,
                                         int* status, int grid)
{
    pdl_wait();   // the fused kernel's records are complete and visible
    const int quads = (Co + 3) / 4;
    const long long wid = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= static_cast<long long>(N) * quads) return;   // whole warps leave together
    const int n = static_cast<int>(wid / quads);
    const int co0 = 4 * static_cast<int>(wid - static_cast<long long>(n) * quads);
    const int nco = Co - co0 < 4 ? Co - co0 : 4;
    float* yo = y + static_cast<long long>(n) * Co + co0;
    // a bounded wait that gave up (or a failed index check of a debug build) leaves records the
    // fused kernel never wrote: say so in the output
    if (*reinterpret_cast<const volatile int*>(status) != 0) {
        if (lane < nco) yo[lane] = __int_as_float(0x7fc00000);
        return;
    }
    const long long big = static_cast<long long>(prem) * (pbase + 1);
    auto cluster_of = [&](long long p) -> long long { return p < big ? p / (pbase + 1) : prem + (p - big) / pbase; };
    auto start_of = [&](long long c) -> long long { return c * pbase + (c < prem ? c : prem); };
    const long long t0 = static_cast<long long>(n) * tpi;
    const long long c0 = cluster_of(t0 / step), c1 = cluster_of((t0 + tpi - 1) / step);
    const int per_cluster = step * recs;
    const long long total = (c1 - c0 + 1) * per_cluster;
    float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (long long k = lane; k < total; k += 32) {
        const long long c = c0 + k / per_cluster;
        const int rq = static_cast<int>(k - (k / per_cluster) * per_cluster);
        const int r = rq / recs, q = rq - (rq / recs) * recs;
        const long long cta = step * c + r;
        const long long nf = (step * start_of(c) + r) / tpi;
        const long long slot = n - nf;
        if (slot < 0 || slot >= J) continue;
        if (FC_DEBUG_OK(cta >= 0 && cta < grid && q < recs && co0 + 4 <= Cout, status)) {
            const float4 v = *reinterpret_cast<const float4*>(ws + ((cta * J + slot) * recs + q) * static_cast<long long>(Cout) + co0);
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        s.x += __shfl_xor_sync(0xffffffffu, s.x, off);
        s.y += __shfl_xor_sync(0xffffffffu, s.y, off);
        s.z += __shfl_xor_sync(0xffffffffu, s.z, off);
        s.w += __shfl_xor_sync(0xffffffffu, s.w, off);
    }
    if (lane < nco) {
        const float v = lane == 0 ? s.x : (lane == 1 ? s.y : (lane == 2 ? s.z : s.w));
        yo[lane] = static_cast<float>(static_cast<double>(v) * inv_count);
    }
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Tile geometry of one call: the pooled ops use the 16 x 8 patch, the full-output op the 1 x 128 row.
struct Geometry {
    int PR, PC, SR, box_cols, box_ch;
    uint32_t strip_bytes, raw_bytes;
};

template <bool BF16, bool WIDE, int ROWS, int XP, bool NHWC = false, int UPW = 1>
Geometry geometry_of()
{
    using S = Shape<WIDE, ROWS, XP, NHWC, UPW>;
    using R = RawBox<BF16, WIDE, ROWS, XP, UPW>;
    // NHWC: one box per K block, [SR][SC][32 B of channels]
    if (NHWC) return Geometry{S::PR, S::PC, S::SR, S::SC, 32 / (BF16 ? 2 : 4), S::STRIP, S::RAW_NHWC};
    return Geometry{S::PR, S::PC, S::SR, R::kCols, R::kCh, S::STRIP, R::kBytes};
}

// The kernel's tile shape: 16 x 8 patches or 16 x 32 patches of four units (pool), two rows
// of 128 (full output, single CTAs) or one row of 128 (full output, CTA pairs).
template <int XPF, int XPB>
Geometry geometry_xp(int bf16, int pool, int pair, int upw)
{
    if (pool && upw == 4)
        return bf16 ? geometry_of<true, false, 1, XPB, false, 4>()
                    : geometry_of<false, false, 1, staged_xp(false, false, 1, 4, XPF != 0, false), false, 4>();
    if (pool) return bf16 ? geometry_of<true, false, 1, XPB>() : geometry_of<false, false, 1, XPF>();
    if (pair) return bf16 ? geometry_of<true, true, 1, XPB>() : geometry_of<false, true, 1, XPF>();
    return bf16 ? geometry_of<true, true, 2, XPB>() : geometry_of<false, true, 2, staged_xp(false, true, 2, 1, XPF != 0, false)>();
}

// padx: the padding's column shift needs XP = 4 (fp32) / 8 (bf16) extra staged columns
Geometry geometry(int bf16, int pool, int pair, int padx, int nhwc, int upw)
{
    if (nhwc) {
        if (pool && upw == 4)
            return bf16 ? geometry_of<true, false, 1, 0, true, 4>() : geometry_of<false, false, 1, 0, true, 4>();
        if (pool) return bf16 ? geometry_of<true, false, 1, 0, true>() : geometry_of<false, false, 1, 0, true>();
        if (pair) return bf16 ? geometry_of<true, true, 1, 0, true>() : geometry_of<false, true, 1, 0, true>();
        return bf16 ? geometry_of<true, true, 2, 0, true>() : geometry_of<false, true, 2, 0, true>();
    }
    return padx ? geometry_xp<4, 8>(bf16, pool, pair, upw) : geometry_xp<0, 0>(bf16, pool, pair, upw);
}

}  // namespace

int conv_plan(ConvPlan* p, int N, int Cin, int H, int W, int Cout, int pad, int nhwc, int dtype, int pool,
              int sm_count)
{
    *p = ConvPlan{};
    if (dtype < 0 || dtype > 2) return 2;
    if (pad < 0 || pad > kMaxPad || H + 2 * pad < 3 || W + 2 * pad < 3) return 2;
    const int bf16 = dtype == 1 ? 1 : 0;
    p->parts = dtype == 2 ? 3 : 1;
    if (Cout < 1 || Cout > 256) return 2;
    p->N = N; p->Cin = Cin; p->H = H; p->W = W; p->Co = Cout;
    // the MMA's N: whole 16-column slices; the padded channels are computed and dropped
    Cout = (Cout + 15) / 16 * 16;
    p->Cout = Cout;
    p->pad = pad;
    p->OH = H + 2 * pad - 2; p->OW = W + 2 * pad - 2;
    p->bf16 = bf16; p->pool = pool;
    p->esize = bf16 ? 2 : 4;
    // TMA boxes start on 16-byte boundaries: the staged patch begins dcol columns before the
    // padded window, dcol = (-pad) mod (elements per 16 B)
    const int align = 16 / p->esize;
    p->nhwc = nhwc ? 1 : 0;
    // NHWC boxes start at any column (channels are the 16-byte-aligned dimension)
    p->dcol = p->nhwc ? 0 : (align - pad % align) % align;
    p->padx = p->dcol != 0 ? 1 : 0;
    p->cb_ch = bf16 ? 16 : 8;
    p->ncb = (Cin + p->cb_ch - 1) / p->cb_ch * p->parts;
    // CTA pairs (M = 256 MMAs, each CTA holding half of the weights) for Cout > 128, where
    // a warp would otherwise hold more than 8 accumulator slices; single CTAs otherwise
    // (cheaper per-tile hand-offs between the MMA issuer and the epilogue).
    p->pair = (Cout > 128 && sm_count >= 2) ? 1 : 0;
    // Pooled single-CTA tiles of up to 64 channels: four 16 x 8 units side by side share one
    // staged strip (one TMA box, one re-layout, one stage hand-off per 512 outputs); the eight
    // accumulators still hold two such tiles.  Wider channel counts keep one unit per tile.
    p->upw = (pool && !p->pair && Cout <= 64) ? 4 : 1;
    const Geometry geo = geometry(bf16, pool, p->pair, p->padx, p->nhwc, p->upw);
    p->RB = (p->OH + geo.PR - 1) / geo.PR;
    p->CS = (p->OW + geo.PC - 1) / geo.PC;
    p->tpi = static_cast<long long>(p->RB) * p->CS;
    // pooled CTA pairs stage strips j and j + CS / 2 (strip_col) when CS is a multiple of 4
    p->split_cs = (p->pair && pool && p->CS % 4 == 0) ? 1 : 0;
    p->num_tiles = static_cast<long long>(N) * p->tpi;
    const int step = p->pair ? 2 : 1;
    // cluster c (a CTA pair, or one CTA) takes a contiguous range of tile groups
    const long long groups = (p->num_tiles + step - 1) / step;
    const int clusters = static_cast<int>(std::min<long long>(groups, std::max(sm_count / step, 1)));
    p->grid = step * clusters;
    p->pbase = groups / clusters;
    p->prem = static_cast<int>(groups % clusters);
    // a CTA's tiles span at most step * (pbase + 1) - 1 consecutive tiles
    p->J = static_cast<int>((step * (p->pbase + 1) + p->tpi - 1) / p->tpi) + 1;
    // per CTA of a group: Cout / step output channels
    p->w_block_bytes = 9u * 2u * static_cast<uint32_t>(Cout / step) * 16u;
    const unsigned long long wtot = static_cast<unsigned long long>(p->w_block_bytes) * p->ncb;
    // the re-layout kernel indexes elements with 32-bit integers (grid stride included)
    if (static_cast<unsigned long long>(step) * (wtot + 2ull * (Cout / step) * 16ull) / p->esize > (1ull << 30)) return 2;
    p->w_total_bytes = static_cast<uint32_t>(wtot);
    p->bias_block_bytes = 2u * static_cast<uint32_t>(Cout / step) * 16u;
    p->raw_bytes = geo.raw_bytes;
    p->strip_bytes = geo.strip_bytes;
    // TMA needs 16-byte multiples for every global stride: the row pitch W * esize decides
    // (NCHW), or the pixel pitch Cin * esize (NHWC)
    p->use_tma = (static_cast<long long>(nhwc ? Cin : W) * p->esize) % 16 == 0;
    p->resident = p->w_total_bytes <= kResidentMax;
    // Shared memory: strips and (streamed) weight blocks per stage, kNumProd x raw_depth
    // TMA boxes, the indicator planes, the (resident) weights and the bias block.
    const uint32_t fixed = ind_bytes(pool != 0) + p->bias_block_bytes + 128u + (p->resident ? p->w_total_bytes : 0u);
    const uint32_t per_stage = p->strip_bytes + (p->resident ? 0u : p->w_block_bytes);
    const uint32_t per_depth = static_cast<uint32_t>(kNumProd) * p->raw_bytes;
    const uint32_t boxes_min = p->use_tma ? per_depth : 0u;
    // At least one strip slot per producer warp: producer w fills stages w, w + P, ... and
    // waits on empty[slot] by phase parity, which is only unambiguous while the slot's
    // previous user (stage g - stages) is at most one phase ahead of that producer's own
    // previous stage (g - P), i.e. stages >= P.
    if (fixed + static_cast<uint32_t>(kNumProd) * per_stage + boxes_min > kSmemBudget) return 2;
    p->stages = static_cast<int>(std::min<uint32_t>(kMaxStages, (kSmemBudget - fixed - boxes_min) / per_stage));
    if (p->stages < kNumProd) return 2;
    // the shared memory left buys TMA look-ahead
    p->raw_depth = 1;
    if (p->use_tma)
        p->raw_depth = static_cast<int>(std::min<uint32_t>(
            kMaxRawDepth, (kSmemBudget - fixed - static_cast<uint32_t>(p->stages) * per_stage) / per_depth));
    p->nacc = std::min(kMaxAcc, 512 / Cout);
    // Epilogue tile groups: as many as keep each warp at most four 16-column slices per tile
    // (the registers its running pool sums or its pipelined loads take) and fit the
    // accumulator ring.
    const int nsub = Cout / 16;
    const int max_slices = 4;
    p->egroups = 1;
    for (int g : {4, 2})
        if ((nsub + 4 / g - 1) / (4 / g) <= max_slices && g <= p->nacc) {
            p->egroups = g;
            break;
        }
    // the four-unit kernel folds these as constants
    if (p->upw == 4 && (p->nacc != 8 || p->egroups != 4)) return 2;
    int cols = 32;
    while (cols < p->nacc * Cout) cols <<= 1;
    p->tmem_cols = cols;
    p->strip_off = 0;
    p->raw_off = p->strip_off + static_cast<uint32_t>(p->stages) * p->strip_bytes;
    p->ind_off = p->raw_off + (p->use_tma ? static_cast<uint32_t>(kNumProd * p->raw_depth) * p->raw_bytes : 0u);
    p->w_off = p->ind_off + ind_bytes(pool != 0);
    p->bb_off = p->w_off + (p->resident ? p->w_total_bytes : static_cast<uint32_t>(p->stages) * p->w_block_bytes);
    p->bar_off = p->bb_off + p->bias_block_bytes;
    p->bar_off = (p->bar_off + 127u) & ~127u;
    // barriers + tmem slot + abort flag, plus 1 KB for aligning the base
    p->smem_bytes = p->bar_off + kBarBytes + 1024u;
    p->ws_weights_bytes = align256(step * (static_cast<size_t>(p->w_total_bytes) + p->bias_block_bytes));
    p->ws_pool_bytes = pool ? align256(static_cast<size_t>(p->grid) * p->J * p->egroups * 4 * Cout * sizeof(float)) : 0;
    return 0;
}

cudaError_t conv_launch(const ConvPlan& p, const void* x, const void* w, const void* b, float* y, int act,
                        void* workspace, cudaStream_t stream, int* status, long long budget)
{
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    void* wr = ws;
    float* pool_ws = reinterpret_cast<float*>(ws + p.ws_weights_bytes);

    {
        const long long total = (static_cast<long long>(p.ncb) * 9 + 1) * 2 * p.Cout * (p.bf16 ? 8 : 4);
        const int threads = 256;
        const int blocks = static_cast<int>(std::min<long long>((total + threads - 1) / threads, 4096));
        const int halves = p.pair ? 2 : 1;
        if (p.bf16)
            conv_weight_relayout_kernel<true><<<blocks, threads, 0, stream>>>(w, b, wr, p.Cin, p.Co, p.Cout, p.ncb,
                                                                               halves, p.parts);
        else
            conv_weight_relayout_kernel<false><<<blocks, threads, 0, stream>>>(w, b, wr, p.Cin, p.Co, p.Cout, p.ncb,
                                                                                halves, p.parts);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    // NCHW x as a 4-D tensor (W, H, Cin, N), one box = [K-block channels][staged rows][staged
    // columns]; NHWC x as (Cin, W, H, N), one box = [staged rows][staged columns][one channel group]
    CUtensorMap tmx;
    std::memset(&tmx, 0, sizeof(tmx));
    if (p.use_tma) {
        auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
        if (enc == nullptr) return cudaErrorNotSupported;
        const cuuint64_t es = static_cast<cuuint64_t>(p.esize);
        const Geometry geo = geometry(p.bf16, p.pool, p.pair, p.padx, p.nhwc, p.upw);
        cuuint64_t dims[4];
        cuuint32_t box[4];
        if (p.nhwc) {
            dims[0] = static_cast<cuuint64_t>(p.Cin); dims[1] = static_cast<cuuint64_t>(p.W);
            dims[2] = static_cast<cuuint64_t>(p.H); dims[3] = static_cast<cuuint64_t>(p.N);
            box[0] = static_cast<cuuint32_t>(geo.box_ch); box[1] = static_cast<cuuint32_t>(geo.box_cols);
            box[2] = static_cast<cuuint32_t>(geo.SR); box[3] = 1u;
        } else {
            dims[0] = static_cast<cuuint64_t>(p.W); dims[1] = static_cast<cuuint64_t>(p.H);
            dims[2] = static_cast<cuuint64_t>(p.Cin); dims[3] = static_cast<cuuint64_t>(p.N);
            box[0] = static_cast<cuuint32_t>(geo.box_cols); box[1] = static_cast<cuuint32_t>(geo.SR);
            box[2] = static_cast<cuuint32_t>(geo.box_ch); box[3] = 1u;
        }
        cuuint64_t strides[3] = {dims[0] * es, dims[0] * dims[1] * es, dims[0] * dims[1] * dims[2] * es};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = enc(&tmx, p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                         const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE,
                         // 256-byte L2 promotion for NCHW wide rows and CTA pairs (measured 0.6-2 %
                         // faster); pooled single-CTA tiles and NHWC boxes keep 128 bytes (faster there)
                         (p.nhwc || (p.pool && !p.pair)) ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                         : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }

    ConvArgs a{};
    a.x = x; a.wr = wr;
    a.out = p.pool ? pool_ws : y;
    a.N = p.N; a.Cin = p.Cin; a.H = p.H; a.W = p.W; a.Cout = p.Cout; a.Co = p.Co; a.OH = p.OH; a.OW = p.OW;
    a.ncb = p.ncb; a.parts = p.parts; a.pad = p.pad; a.dcol = p.dcol; a.RB = p.RB; a.CS = p.CS; a.tpi = p.tpi; a.num_tiles = p.num_tiles;
    a.pbase = p.pbase; a.prem = p.prem; a.J = p.J; a.pair = p.pair; a.split_cs = p.split_cs;
    a.stages = p.stages; a.raw_depth = p.raw_depth; a.resident = p.resident; a.nacc = p.nacc; a.egroups = p.egroups; a.tmem_cols = p.tmem_cols;
    a.upw = p.upw;
    a.poll = polling_budget(budget) ? 1 : 0;
    a.w_block_bytes = p.w_block_bytes; a.w_total_bytes = p.w_total_bytes; a.bias_block_bytes = p.bias_block_bytes;
    a.strip_off = p.strip_off; a.ind_off = p.ind_off; a.w_off = p.w_off; a.bb_off = p.bb_off; a.raw_off = p.raw_off;
    a.bar_off = p.bar_off; a.use_tma = p.use_tma;
    a.status = status; a.budget = budget;

    cudaError_t e;
    if (p.nhwc) {
        if (p.bf16)
            e = p.pair ? launch_main_bf16_pair_nhwc(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                       : launch_main_bf16_nhwc(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
        else
            e = p.pair ? launch_main_tf32_pair_nhwc(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                       : launch_main_tf32_nhwc(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
    } else if (p.padx) {
        if (p.bf16)
            e = p.pair ? launch_main_bf16_pair_padx(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                       : launch_main_bf16_padx(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
        else
            e = p.pair ? launch_main_tf32_pair_padx(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                       : launch_main_tf32_padx(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
    } else if (p.bf16) {
        e = p.pair ? launch_main_bf16_pair(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                   : launch_main_bf16(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
    } else {
        e = p.pair ? launch_main_tf32_pair(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream)
                   : launch_main_tf32(tmx, a, p.pool, act, p.grid, p.smem_bytes, stream);
    }
    if (e != cudaSuccess) return e;

    if (p.pool) {
        const long long outs = static_cast<long long>(p.N) * ((p.Co + 3) / 4);   // one warp per 4 channels
        const int threads = 256;
        const int blocks = static_cast<int>((outs * 32 + threads - 1) / threads);
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(blocks));
        cfg.blockDim = dim3(threads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the fused kernel's tail
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, conv_pool_combine_kernel, static_cast<const float*>(pool_ws), y, p.N, p.Co,
                               p.Cout, p.tpi, p.pbase, p.prem, p.J, p.pair ? 2 : 1, 4 * p.egroups,
                               1.0 / (static_cast<double>(p.OH) * p.OW), status, p.grid);
    }
    return e;
}

}  // namespace fc
