// fc_conv_kernel.cuh -- fused conv3x3 (stride 1, padding 0) + bias + activation, with
// either a global-mean epilogue (Conv2d -> GELU -> adaptive_avg_pool2d(1) page,
// "Kimi-K2.6 l2_p67") or a full-output epilogue (Conv2d -> Mish -> Mish page,
// "Kimi-K2.6 l2_p4"), as an implicit GEMM on tcgen05 tensor cores.
//
// GEMM view (the Mish page's implicit-GEMM sizing: M x N x K =
// pixels x Cout x Cin*9):  D[pixel, co] = sum_{ci, kh, kw} x[ci, oh+kh, ow+kw] * w[co, ci, kh, kw].
//
// Unit: M = 128 output pixels arranged as a 16-row x 8-column patch, N = Cout
// (<= 256), K stepped as (K block of 8 fp32 / 16 bf16 input channels) x (9 taps).  A pooled
// single-CTA tile of up to 64 channels holds four such units side by side (16 x 32 outputs):
// they share one staged strip, so one TMA box, one re-layout and one stage hand-off serve 512
// outputs.
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
// Bias and the ragged-edge mask ride on the tensor core too: every tile starts
// with one extra K step whose A operand is a per-tile "indicator" tile (column
// 0 and 2: 1 for an output pixel inside the image; column 1: 1 for a pixel of
// the tile past the image edge) and whose B operand holds, per output channel,
// the bias split into two TF32 halves (columns 0 and 2) and -1e4 (column 1).
// The accumulator therefore starts at bias for real pixels and near -1e4 for
// padding pixels, whose GELU / Mish is exactly -0: the epilogue needs no bias
// loads and no masking.
//
// Warp roles (640 threads, one CTA per SM, persistent over a contiguous tile range;
// 20 warps leave 96 registers per thread):
//   warps 0-15 epilogue: tcgen05.ld of the accumulator (lane quarter = warp % 4; the
//              column groups h = warp / 4 form 1, 2 or 4 tile groups that take
//              alternate tiles), activation, then either a running per-thread sum
//              (pool; reduced across the warp's 32 pixels only when the image
//              changes) or coalesced stores.
//   warps 16-18 producers: stage g goes to warp g % 3 and strip slot g % S; x arrives
//              as TMA boxes (channel-major, zero-filled past the image), several in
//              flight per warp, that the warp re-lays into the staged strip.
//   warp 19    tensor-memory allocator and single-thread MMA issuer.
#pragma once

#include "fc_act.cuh"
#include "fc_ptx.cuh"

namespace fc {
namespace convk {

constexpr int kEpiWarps = 16;                 // 4 per TMEM lane quarter
constexpr int kEpiCols = 16;                  // accumulator columns per TMEM load
constexpr int kProdWarp0 = kEpiWarps;
constexpr int kNumProd = 3;
constexpr int kMmaWarp = kProdWarp0 + kNumProd;
constexpr int kConvThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kIndPlane = 128 * 16;                 // one indicator plane: 2048 B
// Pooled units: 6 edge variants + a zero plane.  Full-output tiles store only pixels inside
// the output, so every tile uses the all-inside plane: 1 variant + the zero plane.
// Pooled units: (full rows, last row block) x (8 valid columns, OW % 8, none) = 6 variants.
__host__ __device__ constexpr int ind_variants(bool pool) { return pool ? 6 : 1; }
__host__ __device__ constexpr uint32_t ind_bytes(bool pool) { return (ind_variants(pool) + 1) * kIndPlane; }
constexpr float kPadValue = -1.0e4f;                     // pre-activation of padding pixels
constexpr uint32_t kResidentMax = 96 * 1024;
constexpr int kMaxAcc = 8;                               // tensor-memory accumulator ring depth
constexpr int kMaxRawDepth = 4;                          // raw x boxes per producer warp
constexpr int kMaxStages = 6;                            // staged strip slots
// barrier block: 2 kMaxStages + 2 kMaxAcc + kNumProd kMaxRawDepth + 3 barriers, slot, flag
constexpr uint32_t kBarBytes = 512;
static_assert((2 * kMaxStages + 2 * kMaxAcc + kNumProd * kMaxRawDepth + 3) * 8 + 8 <= kBarBytes, "barrier block");
static_assert(kMaxStages >= kNumProd, "one strip slot per producer warp at least (parity waits on empty[])");
// everything the plan places, below the 227 KB per-CTA opt-in limit less the barrier
// block and the 1 KB base alignment
constexpr uint32_t kSmemBudget = 227 * 1024 - kBarBytes - 1024 - 128;

// Output pixels of one staged tile.  The pooled ops use UPW 16-row x 8-column
// units side by side, each one 128-row MMA tile (18 x 10 staged pixels for one unit,
// 18 x 34 for four); the full-output op uses ROWS rows of 128 columns so that each warp
// stores 32 consecutive pixels of a row (128 contiguous bytes) per output
// channel.  Each row of a wide tile is one M = 128 MMA "unit" with its own
// accumulator; the rows share the staged strip (row u starts u * SC pixels
// further) and every streamed weight block, so two rows halve the weight
// traffic per output and stage 4 input rows per 2 output rows instead of 3 per 1.
// Either way the 8-pixel core-matrix groups of a unit lie at one constant stride
// in the staged strip (SBO): the next patch row (16 x 8), or the next 8 pixels (1 x 128).
//
// With zero padding p the staged patch starts p rows above and p + d columns left of the
// tile, d = (-p) mod (16 B / element size), so that the TMA box starts on a 16-byte
// boundary; XP = 4 (fp32) or 8 (bf16) extra staged columns hold the d-column shift and
// every MMA operand starts d staged pixels further (XP = 0 when d is always 0).  fp32 two-row
// full-output tiles and fp32 pooled four-unit tiles stage an odd number of columns instead
// (XP = 1, or 5 with the shift: 131 / 135, or 35 / 39): the re-layout then maps a quarter-warp to
// 4 rows x 2 column quads whose 16-byte strip stores, 16 * SC bytes per row apart, fall in 8
// different bank groups.
//
// NHWC input: a K block lands as one TMA box [SR rows][SC columns][32 B of channels] and is
// split into the two planes; NHWC planes are 64 bytes past a 128-byte multiple apart so that
// the split's 128-bit stores of one phase (4 pixels x 2 planes) cover all banks.
__host__ __device__ constexpr bool fp32_quarter_map(bool bf16, bool wide, int rows, int upw)
{
    return !bf16 && ((wide && rows == 2) || (!wide && upw == 4));
}

__host__ __device__ constexpr int staged_xp(bool bf16, bool wide, int rows, int upw, bool padx, bool nhwc)
{
    return nhwc ? 0 : fp32_quarter_map(bf16, wide, rows, upw) ? (padx ? 5 : 1) : (padx ? (bf16 ? 8 : 4) : 0);
}

template <bool WIDE, int ROWS = 1, int XP = 0, bool NHWC = false, int UPW = 1>
struct Shape {
    static constexpr int UNITS = WIDE ? ROWS : UPW;        // M = 128 MMA units per tile
    static constexpr int PR = WIDE ? ROWS : 16;            // output rows per tile
    static constexpr int PC = WIDE ? 128 : 8 * UPW;        // output columns per tile
    static constexpr int SR = PR + 2;                      // staged rows (halo)
    static constexpr int SC = PC + 2 + XP;                 // staged columns (halo + shift room)
    static constexpr int SPOS = SR * SC;                   // staged pixels
    static constexpr uint32_t PLANE = NHWC ? (SPOS * 16 + 127) / 128 * 128 + 64 : SPOS * 16;   // one channel group
    static constexpr uint32_t RAW_NHWC = (SPOS * 32 + 127) / 128 * 128;   // one NHWC box: [SPOS][32 B]
    static constexpr uint32_t STRIP = (2 * PLANE + 127) / 128 * 128;  // one K block, slot pitch
    static constexpr uint32_t SBO = WIDE ? 128u : SC * 16u;
    // staged pixels between consecutive units' A operands: the next output row (wide rows) or
    // the next 8 columns (pooled units side by side)
    static constexpr int UOFF = WIDE ? SC : 8;
};

// Raw TMA box of one K block: [channel][SR rows][cols] in x's own (channel-major)
// order; cols covers the SC staged columns and keeps each box row a 16-byte multiple.  The
// fp32 boxes of the quarter map are 8 columns past a multiple of 32 wide (136 for 131 or 135
// staged columns, 40 for 35 or 39), so that the re-layout's 16-byte reads of a quarter-warp
// (4 rows x 2 column quads) fall in 8 different bank groups too.
template <bool BF16, bool WIDE, int ROWS = 1, int XP = 0, int UPW = 1>
struct RawBox {
    using S = Shape<WIDE, ROWS, XP, false, UPW>;
    static constexpr bool kQuarterMap = fp32_quarter_map(BF16, WIDE, ROWS, UPW);
    static constexpr int kCh = BF16 ? 16 : 8;
    static constexpr int kCols = BF16 ? (S::SC + 7) / 8 * 8
                                      : (kQuarterMap ? (S::SC - 8 + 31) / 32 * 32 + 8 : (S::SC + 3) / 4 * 4);
    static constexpr uint32_t kChPlane = S::SR * kCols * (BF16 ? 2 : 4);
    static constexpr uint32_t kBytes = (kCh * kChPlane + 127) / 128 * 128;
};

struct ConvArgs {
    const void* x;
    const void* wr;      // re-laid weights, then the bias block (workspace)
    float* out;          // full output (store) or pool partials (pool)
    int N, Cin, H, W, OH, OW;
    int Cout;            // tile width: output channels rounded up to 16
    int Co;              // output channels stored (<= Cout)
    int ncb;             // K stages per tile (K blocks x parts)
    int parts;           // 1, or 3 for split TF32: stages hi*hi, hi*lo, lo*hi of each K block (no other values)
    int pad;             // zero padding p on every side (output = input + 2p - 2)
    int dcol;            // (-pad) mod (16 B / element size): staged columns before the first tap column
    int RB, CS;
    long long tpi;
    long long num_tiles;  // tiles of the whole call
    long long pbase;      // tile groups per cluster (the first `prem` clusters take one more)
    int prem, J, stages, raw_depth, resident, nacc, tmem_cols;
    int egroups;          // epilogue tile groups G (1, 2, 4): group g takes every G-th tile
    int upw;              // pooled single-CTA tiles: 1 (16 x 8) or 4 units side by side (16 x 32)
    int poll;             // a test shortened the wait budget: launch the polling instantiation
    int pair;             // 1: CTA pairs with M = 256 MMAs (group = 2 tiles); 0: single CTAs
    int split_cs;         // pooled CTA pairs: the pair's two tiles at strips j and j + CS / 2 (strip_col)
    uint32_t w_block_bytes, w_total_bytes, bias_block_bytes;   // per CTA of the pair (its half of Cout)
    uint32_t strip_off, ind_off, w_off, bb_off, raw_off, bar_off;
    int use_tma;         // x staged by TMA boxes + in-warp transpose (else plain loads)
    int* status;
    long long budget;
};

// Start loading 16 accumulator columns of this warp's 32 TMEM lanes into r; the
// registers are valid only after tmem_ld16_wait(r).
__device__ __forceinline__ void tmem_ld16_start(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// One 16-column accumulator slice of this warp's 32 TMEM lanes in the 16x256b fragment
// shape: two loads (lane bases +0 and +16) of 16 lanes x 16 columns.  Thread t receives, for
// lane base L in {0, 16}, r[8L/16 + k]: k = 0, 1 lane L + t/4, columns 2(t%4) + {0, 1};
// k = 2, 3 lane L + t/4 + 8, the same columns; k = 4..7 the same with columns + 8.  So a
// thread holds 4 pixels x 4 channels, and can pre-sum its pixels per channel.
__device__ __forceinline__ void tmem_ld_slice16x256_start(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
                 : "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr + (16u << 16))
                 : "memory");
}

// Wait for this thread's TMEM loads into two 16-register sets (see tmem_ld16_wait).
__device__ __forceinline__ void tmem_ld16x2_wait(uint32_t (&r)[16], uint32_t (&u)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(u[0]), "+r"(u[1]), "+r"(u[2]), "+r"(u[3]), "+r"(u[4]), "+r"(u[5]), "+r"(u[6]),
                   "+r"(u[7]), "+r"(u[8]), "+r"(u[9]), "+r"(u[10]), "+r"(u[11]), "+r"(u[12]), "+r"(u[13]),
                   "+r"(u[14]), "+r"(u[15])
                 :
                 : "memory");
}

// Wait for this thread's TMEM loads.  The registers are read-write operands here, so
// that the compiler cannot read them between the load and this wait.
__device__ __forceinline__ void tmem_ld16_wait(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

// Tile t of the flattened (image, row block, column strip) grid.
struct TileCoord {
    int n, rb, cs;
};

__device__ __forceinline__ TileCoord tile_coord(long long t, long long tpi, int CS)
{
    TileCoord c;
    c.n = static_cast<int>(t / tpi);
    const int r = static_cast<int>(t - static_cast<long long>(c.n) * tpi);
    c.rb = r / CS;
    c.cs = r - c.rb * CS;
    return c;
}

// Column strip of tile c.  CTA pairs take the even (rank 0) and odd (rank 1) tiles of the tile
// order.  With split_cs (pooled pairs, CS a multiple of 4) tile cs of a row block sits at strip
// cs / 2 (even cs) or CS / 2 + cs / 2 (odd cs), so that the two CTAs of a pair stage strips j and
// j + CS / 2 of one row block: both x boxes of a stage then start at the same 32-byte parity, and
// the pair's stages alternate between boxes of one and of two sectors per row instead of one CTA
// always fetching two (its 16-byte-aligned strip starting mid-sector).
template <bool PAIR>
__device__ __forceinline__ int strip_col(const TileCoord& c, const ConvArgs& a)
{
    if constexpr (PAIR) return a.split_cs ? (c.cs >> 1) + (c.cs & 1) * (a.CS >> 1) : c.cs;
    else return c.cs;
}

// Next tile in (image, row block, column strip) order.
__device__ __forceinline__ void next_tile(TileCoord& c, int RB, int CS)
{
    if (++c.cs == CS) {
        c.cs = 0;
        if (++c.rb == RB) {
            c.rb = 0;
            ++c.n;
        }
    }
}

// Raw TMA box of one K block: [channel][18 rows][kRawCols columns], channel-major as in x.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* map, uint64_t* bar, int c0, int c1, int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// The same with the destination as a shared-memory address.
__device__ __forceinline__ void tma_load_4d_s(uint32_t dst, const void* map, uint64_t* bar, int c0, int c1, int c2,
                                              int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint2 ld_shared_u2(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float2 ld_shared_f2(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}

// Re-lay a landed raw box into the staged strip [group][SPOS pixels][16 B].
// The TF32 operand of x for one split-TF32 part.  The high part is x as stored: the tensor core
// reads an fp32 word as TF32 by dropping its 13 low mantissa bits (as the Linear op's operands,
// which TMA hands to the MMA untouched); with LO, the remainder x - trunc(x) rounded to TF32.
template <bool LO>
__device__ __forceinline__ uint32_t tf32_part(float v)
{
    if constexpr (LO) return __float_as_uint(to_tf32(v - __uint_as_float(__float_as_uint(v) & 0xFFFFE000u)));
    else return __float_as_uint(v);
}

template <bool BF16, bool WIDE, int ROWS, int XP, bool LO, int UPW>
__device__ __forceinline__ void transpose_raw(uint32_t raw, uint32_t strip, int lane)
{
    using S = Shape<WIDE, ROWS, XP, false, UPW>;
    using RB_ = RawBox<BF16, WIDE, ROWS, XP, UPW>;
    static_assert(!(BF16 && LO), "split TF32 is an fp32 mode");
    if constexpr (RB_::kQuarterMap) {
        // fp32 two-row full-output tiles (4 staged rows) and pooled four-unit tiles (18 staged
        // rows, taken in row groups of 4, the last one holding 2): item = (group g, staged row,
        // column quad), 4 channels x 4 pixels -> four 16-byte rows; a quarter-warp takes the 4
        // rows of one row group x 2 adjacent quads of one (g, row group, quad pair), so that
        // with SC odd and the box 8 columns past a multiple of 32 wide both its 16-byte reads
        // and its 16-byte stores hit 8 different bank groups
        static_assert(S::SC % 2 == 1 && RB_::kCols % 32 == 8 && RB_::kCols >= S::SC, "quarter map");
        constexpr int kQuads = (S::SC + 3) / 4;
        constexpr int kPairs = (kQuads + 1) / 2;
        constexpr int kSlots = (S::SR + 3) / 4 * kPairs;   // quarter-warp slots per channel group
        const int cq_lo = (lane >> 2) & 1;
#pragma unroll 2
        for (int qs = lane >> 3; qs < 2 * kSlots; qs += 4) {
            const int g = qs >= kSlots ? 1 : 0;
            const int rem = qs - g * kSlots;
            // one row group (the two-row tiles): no division, no row bound
            const int rg = S::SR == 4 ? 0 : rem / kPairs;
            const int cq = 2 * (rem - rg * kPairs) + cq_lo;
            const int row = 4 * rg + (lane & 3);
            if (cq < kQuads && (S::SR % 4 == 0 || row < S::SR)) {
                const uint32_t src = raw + static_cast<uint32_t>(4 * g) * RB_::kChPlane +
                                     static_cast<uint32_t>(row * RB_::kCols + 4 * cq) * 4u;
                float4 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = ld_shared_f4(src + static_cast<uint32_t>(c) * RB_::kChPlane);
                const uint32_t dst = strip + static_cast<uint32_t>(g) * S::PLANE +
                                     static_cast<uint32_t>(row * S::SC + 4 * cq) * 16u;
                st_shared_v4(dst, tf32_part<LO>(v[0].x), tf32_part<LO>(v[1].x), tf32_part<LO>(v[2].x),
                             tf32_part<LO>(v[3].x));
                st_shared_v4(dst + 16u, tf32_part<LO>(v[0].y), tf32_part<LO>(v[1].y), tf32_part<LO>(v[2].y),
                             tf32_part<LO>(v[3].y));
                if (4 * cq + 2 < S::SC)
                    st_shared_v4(dst + 32u, tf32_part<LO>(v[0].z), tf32_part<LO>(v[1].z), tf32_part<LO>(v[2].z),
                                 tf32_part<LO>(v[3].z));
                if (4 * cq + 3 < S::SC)
                    st_shared_v4(dst + 48u, tf32_part<LO>(v[0].w), tf32_part<LO>(v[1].w), tf32_part<LO>(v[2].w),
                                 tf32_part<LO>(v[3].w));
            }
        }
    } else if constexpr (!BF16) {
        // item = (group g, staged row, column quad): 4 channels x 4 pixels -> four 16-byte rows
        // (the last quad of a row holds SC % 4 staged pixels; the raw box is wider)
        static_assert(RB_::kCols % 4 == 0 && RB_::kChPlane % 16 == 0, "16-byte raw reads");
        static_assert(S::SC % 4 == 0 || S::SC % 4 == 2, "a row's last quad holds 4 or 2 staged pixels");
        constexpr int kQuads = (S::SC + 3) / 4;
        constexpr int kHalf = S::SR * kQuads;
#pragma unroll 2
        for (int i = lane; i < 2 * kHalf; i += 32) {
            const int g = i >= kHalf ? 1 : 0;
            const int r = i - g * kHalf;
            const int row = r / kQuads, cq = r - (r / kQuads) * kQuads;
            const uint32_t src = raw + static_cast<uint32_t>(4 * g) * RB_::kChPlane +
                                 static_cast<uint32_t>(row * RB_::kCols + 4 * cq) * 4u;
            float4 v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) v[c] = ld_shared_f4(src + static_cast<uint32_t>(c) * RB_::kChPlane);
            const uint32_t dst = strip + static_cast<uint32_t>(g) * S::PLANE +
                                 static_cast<uint32_t>(row * S::SC + 4 * cq) * 16u;
            st_shared_v4(dst, tf32_part<LO>(v[0].x), tf32_part<LO>(v[1].x), tf32_part<LO>(v[2].x),
                         tf32_part<LO>(v[3].x));
            st_shared_v4(dst + 16u, tf32_part<LO>(v[0].y), tf32_part<LO>(v[1].y), tf32_part<LO>(v[2].y),
                         tf32_part<LO>(v[3].y));
            if (4 * cq + 2 < S::SC) {
                st_shared_v4(dst + 32u, tf32_part<LO>(v[0].z), tf32_part<LO>(v[1].z), tf32_part<LO>(v[2].z),
                             tf32_part<LO>(v[3].z));
                st_shared_v4(dst + 48u, tf32_part<LO>(v[0].w), tf32_part<LO>(v[1].w), tf32_part<LO>(v[2].w),
                             tf32_part<LO>(v[3].w));
            }
        }
    } else if constexpr (!WIDE) {
        // pooled patches (an even number of staged columns): item = (group g, staged row, column pair):
        // 8 channels x 2 columns -> two 16-byte rows
        constexpr int kPairs = S::SC / 2;
        constexpr int kHalf = S::SR * kPairs;
#pragma unroll 2
        for (int i = lane; i < 2 * kHalf; i += 32) {
            const int g = i >= kHalf ? 1 : 0;
            const int r = i - g * kHalf;
            const int row = r / kPairs, cp = r - (r / kPairs) * kPairs;
            const uint32_t src = raw + static_cast<uint32_t>(8 * g) * RB_::kChPlane +
                                 static_cast<uint32_t>(row * RB_::kCols + 2 * cp) * 2u;
            uint32_t w[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) w[c] = ld_shared_u32(src + static_cast<uint32_t>(c) * RB_::kChPlane);
            const uint32_t dst = strip + static_cast<uint32_t>(g) * S::PLANE +
                                 static_cast<uint32_t>(row * S::SC + 2 * cp) * 16u;
            st_shared_v4(dst, __byte_perm(w[0], w[1], 0x5410), __byte_perm(w[2], w[3], 0x5410),
                         __byte_perm(w[4], w[5], 0x5410), __byte_perm(w[6], w[7], 0x5410));
            st_shared_v4(dst + 16u, __byte_perm(w[0], w[1], 0x7632), __byte_perm(w[2], w[3], 0x7632),
                         __byte_perm(w[4], w[5], 0x7632), __byte_perm(w[6], w[7], 0x7632));
        }
    } else {
        // wide rows (130 or 138 staged columns): item = (group g, staged row, column quad):
        // 8 channels x 4 columns, one 64-bit read per channel -> four 16-byte rows (the last quad
        // of a row holds SC % 4 = 2 staged pixels; the raw box is wider)
        static_assert(RB_::kCols % 8 == 0 && RB_::kChPlane % 16 == 0, "8-byte raw reads");
        static_assert(S::SC % 4 == 2, "a row's last quad holds 2 staged pixels");
        constexpr int kQuads = (S::SC + 3) / 4;
        constexpr int kHalf = S::SR * kQuads;
#pragma unroll 2
        for (int i = lane; i < 2 * kHalf; i += 32) {
            const int g = i >= kHalf ? 1 : 0;
            const int r = i - g * kHalf;
            const int row = r / kQuads, cq = r - (r / kQuads) * kQuads;
            const uint32_t src = raw + static_cast<uint32_t>(8 * g) * RB_::kChPlane +
                                 static_cast<uint32_t>(row * RB_::kCols + 4 * cq) * 2u;
            uint2 w[8];   // channel c: .x = columns 0, 1; .y = columns 2, 3
#pragma unroll
            for (int c = 0; c < 8; ++c) w[c] = ld_shared_u2(src + static_cast<uint32_t>(c) * RB_::kChPlane);
            const uint32_t dst = strip + static_cast<uint32_t>(g) * S::PLANE +
                                 static_cast<uint32_t>(row * S::SC + 4 * cq) * 16u;
            st_shared_v4(dst, __byte_perm(w[0].x, w[1].x, 0x5410), __byte_perm(w[2].x, w[3].x, 0x5410),
                         __byte_perm(w[4].x, w[5].x, 0x5410), __byte_perm(w[6].x, w[7].x, 0x5410));
            st_shared_v4(dst + 16u, __byte_perm(w[0].x, w[1].x, 0x7632), __byte_perm(w[2].x, w[3].x, 0x7632),
                         __byte_perm(w[4].x, w[5].x, 0x7632), __byte_perm(w[6].x, w[7].x, 0x7632));
            if (4 * cq + 2 < S::SC) {
                st_shared_v4(dst + 32u, __byte_perm(w[0].y, w[1].y, 0x5410), __byte_perm(w[2].y, w[3].y, 0x5410),
                             __byte_perm(w[4].y, w[5].y, 0x5410), __byte_perm(w[6].y, w[7].y, 0x5410));
                st_shared_v4(dst + 48u, __byte_perm(w[0].y, w[1].y, 0x7632), __byte_perm(w[2].y, w[3].y, 0x7632),
                             __byte_perm(w[4].y, w[5].y, 0x7632), __byte_perm(w[6].y, w[7].y, 0x7632));
            }
        }
    }
}

// Fallback staging with plain loads (when x's row pitch is not a 16-byte
// multiple and TMA cannot address it): one K block of the halo patch as
// [group][SPOS pixels][16 B], zero past the image and past Cin; `lo` stages the
// split-TF32 remainder instead of the high part (fp32 only).
template <bool BF16, bool WIDE, int ROWS, int XP, int UPW>
__device__ __forceinline__ void fill_strip(uint32_t strip, const void* xv, int n, int cb, int oh0, int ow0,
                                           int Cin, int H, int W, int lane, bool lo)
{
    using S = Shape<WIDE, ROWS, XP, false, UPW>;
    const size_t HW = static_cast<size_t>(H) * W;
    for (int s = lane; s < S::SPOS; s += 32) {
        const int rr = s / S::SC, cc = s - (s / S::SC) * S::SC;
        const int ih = oh0 + rr, iw = ow0 + cc;   // negative above / left of the image (padding)
        const bool ok = ih >= 0 && ih < H && iw >= 0 && iw < W;
        const uint32_t a = strip + static_cast<uint32_t>(s) * 16u;
        if constexpr (!BF16) {
            const float* x = reinterpret_cast<const float*>(xv);
            const int ci0 = cb * 8;
            const size_t off = ok ? ((static_cast<size_t>(n) * Cin + ci0) * HW + static_cast<size_t>(ih) * W + iw) : 0;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = (ok && ci0 + e < Cin) ? __ldg(x + off + e * HW) : 0.0f;
            uint32_t t[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) t[e] = lo ? tf32_part<true>(v[e]) : tf32_part<false>(v[e]);
            st_shared_v4(a, t[0], t[1], t[2], t[3]);
            st_shared_v4(a + S::PLANE, t[4], t[5], t[6], t[7]);
        } else {
            const unsigned short* x = reinterpret_cast<const unsigned short*>(xv);
            const int ci0 = cb * 16;
            const size_t off = ok ? ((static_cast<size_t>(n) * Cin + ci0) * HW + static_cast<size_t>(ih) * W + iw) : 0;
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t lo = (ok && ci0 + 2 * e < Cin) ? __ldg(x + off + (2 * e) * HW) : 0u;
                const uint32_t hi = (ok && ci0 + 2 * e + 1 < Cin) ? __ldg(x + off + (2 * e + 1) * HW) : 0u;
                v[e] = lo | (hi << 16);
            }
            st_shared_v4(a, v[0], v[1], v[2], v[3]);
            st_shared_v4(a + S::PLANE, v[4], v[5], v[6], v[7]);
        }
    }
}

// NHWC fallback staging with plain loads (when Cin's row of channels is not a 16-byte
// multiple and TMA cannot address it): x [N][H][W][Cin]; one staged pixel's K block is
// 8 fp32 / 16 bf16 consecutive channels, zero past the image and past Cin.
template <bool BF16, bool WIDE, int ROWS, int UPW>
__device__ __forceinline__ void fill_strip_nhwc(uint32_t strip, const void* xv, int n, int cb, int oh0, int ow0,
                                                int Cin, int H, int W, int lane, bool lo)
{
    using S = Shape<WIDE, ROWS, 0, true, UPW>;
    for (int s = lane; s < S::SPOS; s += 32) {
        const int rr = s / S::SC, cc = s - (s / S::SC) * S::SC;
        const int ih = oh0 + rr, iw = ow0 + cc;
        const bool ok = ih >= 0 && ih < H && iw >= 0 && iw < W;
        const size_t pix = ok ? ((static_cast<size_t>(n) * H + ih) * W + iw) * static_cast<size_t>(Cin) : 0;
        const uint32_t a = strip + static_cast<uint32_t>(s) * 16u;
        if constexpr (!BF16) {
            const float* x = reinterpret_cast<const float*>(xv) + pix;
            const int ci0 = cb * 8;
            uint32_t t[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float v = (ok && ci0 + e < Cin) ? __ldg(x + ci0 + e) : 0.0f;
                t[e] = lo ? tf32_part<true>(v) : tf32_part<false>(v);
            }
            st_shared_v4(a, t[0], t[1], t[2], t[3]);
            st_shared_v4(a + S::PLANE, t[4], t[5], t[6], t[7]);
        } else {
            const unsigned short* x = reinterpret_cast<const unsigned short*>(xv) + pix;
            const int ci0 = cb * 16;
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t l = (ok && ci0 + 2 * e < Cin) ? __ldg(x + ci0 + 2 * e) : 0u;
                const uint32_t h = (ok && ci0 + 2 * e + 1 < Cin) ? __ldg(x + ci0 + 2 * e + 1) : 0u;
                v[e] = l | (h << 16);
            }
            st_shared_v4(a, v[0], v[1], v[2], v[3]);
            st_shared_v4(a + S::PLANE, v[4], v[5], v[6], v[7]);
        }
    }
}

// NHWC: a landed box holds each staged pixel's K block of channels as 32 contiguous bytes;
// split them into the strip's two group planes -- fp32 rounded to the TF32 operand (the high
// part, or with LO the split-TF32 remainder), bf16 as they are.  Item i is half i % 2 of pixel
// i / 2: consecutive lanes read consecutive 16 bytes.
template <bool BF16, bool WIDE, int ROWS, bool LO, int UPW>
__device__ __forceinline__ void copy_raw_nhwc(uint32_t raw, uint32_t strip, int lane)
{
    using S = Shape<WIDE, ROWS, 0, true, UPW>;
#pragma unroll 4
    for (int i = lane; i < 2 * S::SPOS; i += 32) {
        const uint32_t px = static_cast<uint32_t>(i >> 1), h = static_cast<uint32_t>(i & 1);
        const float4 v = ld_shared_f4(raw + static_cast<uint32_t>(i) * 16u);
        const uint32_t dst = strip + h * S::PLANE + px * 16u;
        if constexpr (BF16)
            st_shared_v4(dst, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
        else
            st_shared_v4(dst, tf32_part<LO>(v.x), tf32_part<LO>(v.y), tf32_part<LO>(v.z), tf32_part<LO>(v.w));
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

// A operand of the bias K step, one 128-row plane per edge variant of a pooled unit (16 rows x 8
// columns): v = 3 re + cc, re = 1 for a unit in the last row block (rows past the image are
// padding), cc = 0 for 8 columns inside the image, 1 for the first OW % 8 columns only (the unit
// that straddles the right edge), 2 for none (a unit wholly past the edge); then a zero plane
// (the second K core matrix).  A pixel inside the output gets a 1 in the bias columns (fp32: k 0
// and k 2 for the two TF32 halves; bf16: k 0); a padding pixel gets a 1 in k 1, whose B entry is
// the padding value, so its accumulator starts near -1e4 and activates to exactly -0.  CTA pairs
// share one descriptor for two tiles, so they use plane 0 (all inside) and mask in the epilogue
// instead.  Full-output tiles store only the pixels inside the output and use the all-inside
// plane alone (plane 0, then the zero plane).
template <bool BF16, bool WIDE, int ROWS, int UPW>
__device__ __forceinline__ void build_indicator_planes(uint8_t* ind, int OH, int OW, int RB, int tid, int nthreads)
{
    using S = Shape<WIDE, ROWS, 0, false, UPW>;
    constexpr int NV = ind_variants(!WIDE);
    const int rows_last = OH - (RB - 1) * S::PR;   // valid rows in the last row block
    const int cols_part = OW % 8;                  // valid columns of a unit on the right edge
    for (int i = tid; i < (NV + 1) * 128; i += nthreads) {
        const int v = i >> 7, r = i & 127;
        const int pr = r >> 3, pc = r & 7;           // a pooled unit's pixel r
        const int re = v / 3, cc = v - (v / 3) * 3;
        const bool in = v < NV && (re == 0 || pr < rows_last) && (cc == 0 || (cc == 1 && pc < cols_part));
        const bool pad = v < NV && !in;
        uint32_t w0, w1, w2;
        if constexpr (BF16) {
            w0 = (in ? 0x3F80u : 0u) | ((pad ? 0x3F80u : 0u) << 16);   // bf16 1.0 in k 0 / k 1
            w1 = 0u;
            w2 = 0u;
        } else {
            w0 = in ? 0x3F800000u : 0u;      // k 0: bias high half
            w1 = pad ? 0x3F800000u : 0u;     // k 1: padding value
            w2 = in ? 0x3F800000u : 0u;      // k 2: bias low half
        }
        st_shared_v4(smem_u32(ind) + static_cast<uint32_t>(v) * kIndPlane + static_cast<uint32_t>(r) * 16u, w0, w1,
                     w2, 0u);
    }
}

// One MMA of the tile group: M = 256 over the CTA pair, or M = 128 in this CTA.
// (A kernel may use only one of the two tcgen05 CTA-group forms.)
template <bool BF16, bool PAIR>
__device__ __forceinline__ void issue_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    // Executed by the whole MMA warp: one elected lane issues, and the operands stay
    // warp-uniform, which keeps the issue loop short when other warps compete for
    // this sub-partition's issue slots.
#define FC_MMA_ELECT(GROUP, KIND)                                                                  \
    asm volatile("{\n\t.reg .pred e, p;\n\t"                                                  \
                 "elect.sync _|e, 0xffffffff;\n\t"                                              \
                 "setp.ne.b32 p, %4, 0;\n\t"                                                     \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], %1, %2, %3, p;\n\t}\n" \
                 ::"r"(d), "l"(ad), "l"(bd), "r"(idesc), "r"(acc)                                  \
                 : "memory")
    if constexpr (BF16 && PAIR) FC_MMA_ELECT("2", "f16");
    else if constexpr (BF16) FC_MMA_ELECT("1", "f16");
    else if constexpr (PAIR) FC_MMA_ELECT("2", "tf32");
    else FC_MMA_ELECT("1", "tf32");
#undef FC_MMA_ELECT
}

// The nine accumulating MMAs of one K block (the 3 x 3 taps) from one asm block, by one
// elected lane of the MMA warp: tap (kh, kw) reads A (the staged strip) at start
// a + (kh * SC + kw) * 16 B and B (this tap's weights) at b + tap * bstep * 16 B.  Issuing
// them back to back, with all descriptor arithmetic done first, keeps the MMA issue rate
// close to the tensor rate while the epilogue warps compete for this sub-partition.
template <bool BF16, bool PAIR, int SC>
__device__ __forceinline__ void issue_mma9(uint32_t d, uint64_t a, uint64_t b, uint64_t bstep, uint32_t idesc)
{
#define FC_MMA9(GROUP, KIND)                                                                              \
    asm volatile("{\n\t.reg .pred e, p;\n\t"                                                              \
                 ".reg .b64 a1, a2, a3, a4, a5, a6, a7, a8, b1, b2, b3, b4, b5, b6, b7, b8;\n\t"           \
                 "setp.ne.b32 p, 1, 0;\n\t"                                                               \
                 "add.s64 a1, %1, 1;\n\tadd.s64 a2, %1, 2;\n\tadd.s64 a3, %1, %5;\n\tadd.s64 a4, %1, %6;\n\t" \
                 "add.s64 a5, %1, %7;\n\tadd.s64 a6, %1, %8;\n\tadd.s64 a7, %1, %9;\n\tadd.s64 a8, %1, %10;\n\t" \
                 "add.s64 b1, %2, %4;\n\tadd.s64 b2, b1, %4;\n\tadd.s64 b3, b2, %4;\n\tadd.s64 b4, b3, %4;\n\t"  \
                 "add.s64 b5, b4, %4;\n\tadd.s64 b6, b5, %4;\n\tadd.s64 b7, b6, %4;\n\tadd.s64 b8, b7, %4;\n\t"  \
                 "elect.sync _|e, 0xffffffff;\n\t"                                                        \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], %1, %2, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a1, b1, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a2, b2, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a3, b3, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a4, b4, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a5, b5, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a6, b6, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a7, b7, %3, p;\n\t"            \
                 "@e tcgen05.mma.cta_group::" GROUP ".kind::" KIND " [%0], a8, b8, %3, p;\n\t}\n"         \
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "l"(bstep), "n"(SC), "n"(SC + 1), "n"(SC + 2),       \
                 "n"(2 * SC), "n"(2 * SC + 1), "n"(2 * SC + 2)                                              \
                 : "memory")
    if constexpr (BF16 && PAIR) FC_MMA9("2", "f16");
    else if constexpr (BF16) FC_MMA9("1", "f16");
    else if constexpr (PAIR) FC_MMA9("2", "tf32");
    else FC_MMA9("1", "tf32");
#undef FC_MMA9
}

// Bounded wait; barriers that the peer CTA signals need cluster-scope acquire.  POLL: see mbar_wait.
template <bool PAIR, bool POLL = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                         long long budget)
{
    static_assert(!(PAIR && POLL), "CTA pairs have no polling instantiation");
    if constexpr (PAIR) return mbar_wait_cluster(bar, parity, abort_flag, status, budget);
    else return mbar_wait<POLL>(bar, parity, abort_flag, status, budget);
}

// Commit this thread's MMAs to `bar` in the CTAs of `mask` (pair) or in this CTA.
template <bool PAIR>
__device__ __forceinline__ void commit_to(uint64_t* bar, uint16_t mask)
{
    // whole MMA warp; one elected lane commits (its MMAs are the warp's MMAs)
    if constexpr (PAIR) {
        asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                     "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}\n"
                     ::"r"(smem_u32(bar)), "h"(mask)
                     : "memory");
    } else {
        asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                     "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n"
                     ::"r"(smem_u32(bar))
                     : "memory");
    }
}

// POLL: the waits poll instead of suspending (see mbar_wait); only launched while a test has
// shortened the wait budget.
template <bool BF16, bool POOL, int ACT, bool PAIR, bool PADX, bool NHWC, int UPW, bool POLL = false>
__global__ void __launch_bounds__(kConvThreads, 1)
    conv3x3_fused_kernel(const __grid_constant__ CUtensorMap tmx, const ConvArgs a)
{
    constexpr bool WIDE = !POOL;
    // full output on single CTAs: two-row tiles (two MMA units sharing each staged strip
    // and weight block); CTA pairs keep one row per CTA
    constexpr int ROWS = (WIDE && !PAIR) ? 2 : 1;
    // room for the padding's column shift a.dcol (< 16 B of elements) when it is not 0
    constexpr int XP = staged_xp(BF16, WIDE, ROWS, UPW, PADX, NHWC);
    static_assert(!(PADX && NHWC), "NHWC boxes start at any column: no shift room needed");
    static_assert(UPW == 1 || (POOL && !PAIR), "side-by-side units: single-CTA pooled tiles only");
    using S = Shape<WIDE, ROWS, XP, NHWC, UPW>;
    using RBox = RawBox<BF16, WIDE, ROWS, XP, UPW>;
    // one raw buffer: an NCHW box, or (NHWC) the two channel-group boxes in the strip's layout
    constexpr uint32_t kRawBytes = NHWC ? S::RAW_NHWC : RBox::kBytes;
    constexpr int UPT = S::UNITS;   // accumulator units per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + a.bar_off);
    uint64_t* full = bars;                  // [kMaxStages] leader: both CTAs' stage ready; peer: its own
    uint64_t* empty = bars + kMaxStages;    // [kMaxStages] both: stage consumed (multicast commit)
    uint64_t* wfull = bars + 2 * kMaxStages;   // both: own bias block (+ resident weights) landed
    uint64_t* tfull = wfull + 1;               // [kMaxAcc] both: accumulator ready (multicast commit)
    uint64_t* tempty = tfull + kMaxAcc;        // [kMaxAcc] leader: both CTAs' epilogues drained it
    uint64_t* mdone = tempty + kMaxAcc;        // leader: every MMA completed
    uint64_t* rawfull = mdone + 1;                      // [kNumProd kMaxRawDepth] a raw x box landed (warp-major)
    uint64_t* wpeer = rawfull + kNumProd * kMaxRawDepth;   // leader: the peer's bias block (+ resident weights) landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wpeer + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool pair = PAIR;
    const uint32_t rank = pair ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int step = pair ? 2 : 1;                      // tiles per group
    const int cluster = static_cast<int>(blockIdx.x) / step;
    const long long p_begin = static_cast<long long>(cluster) * a.pbase + min(cluster, a.prem);
    const int n_pairs = static_cast<int>(a.pbase + (cluster < a.prem ? 1 : 0));   // groups of this CTA
    const long long t_first = step * p_begin + rank;   // this CTA's tiles: t_first, t_first + step, ...

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            // leader: lane 0 before (weight bytes) and after its fill, plus the peer's forward
            mbar_init(&full[s], (pair && leader) ? 3 : 2);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kNumProd * kMaxRawDepth; ++s) mbar_init(&rawfull[s], 1);
        for (int s = 0; s < kMaxAcc; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], step * kEpiWarps / a.egroups);   // lane 0 of every epilogue warp of the tile group
        }
        mbar_init(wfull, 1);
        mbar_init(wpeer, 1);
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (a.use_tma) prefetch_tmap(&tmx);
    }
    if (warp < kEpiWarps) {
        build_indicator_planes<BF16, WIDE, ROWS, UPW>(smem + a.ind_off, a.OH, a.OW, a.RB, threadIdx.x, kEpiWarps * 32);
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        if constexpr (PAIR) {
            tmem_alloc_pair(tmem_slot, static_cast<uint32_t>(a.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, static_cast<uint32_t>(a.tmem_cols));
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync();   // both CTAs' barriers exist before any remote arrive
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const TileCoord first = tile_coord(t_first, a.tpi, a.CS);
    // The set-up above overlaps the previous kernel (the weight re-layout); only the producers
    // read its output (the re-laid weights and bias), so only they wait for it, after requesting
    // their first boxes of x.  The next kernel (the pool combine) may start its own set-up now.
    pdl_launch_dependents();

    if (warp >= kProdWarp0 && warp < kProdWarp0 + kNumProd) {
        // ------------------------------------------------------------ producers (both CTAs)
        const int pw = warp - kProdWarp0;
        const uint8_t* wmine = reinterpret_cast<const uint8_t*>(a.wr) + static_cast<size_t>(rank) * a.w_total_bytes;
        {
            // This warp handles stages g = pw, pw + P, ... of the (tile group, K block)
            // sequence (P producer warps); stage g fills strip slot g % S.  Its x boxes
            // rotate through a.raw_depth raw buffers of its own, so that many TMA loads
            // are in flight ahead of the re-layout.
            const uint32_t S_ = static_cast<uint32_t>(a.stages);
            const uint32_t strip0 = smem_u32(smem + a.strip_off);
            const int rd = a.raw_depth;
            auto advance = [&](TileCoord& c, int& l, int& kb, int k) {
                kb += k;
                while (kb >= a.ncb) {
                    kb -= a.ncb;
                    ++l;
                    next_tile(c, a.RB, a.CS);
                    if (pair) next_tile(c, a.RB, a.CS);
                }
            };
            // raw buffer (and its rawfull barrier) of this warp's i-th stage
            auto raw_buf = [&](uint32_t i) { return static_cast<uint32_t>(pw * rd) + i % static_cast<uint32_t>(rd); };
            TileCoord tc = first;
            int lt = 0, cb = 0;
            advance(tc, lt, cb, pw);
            // the issue-ahead position: the next of this warp's stages whose box is not yet requested
            TileCoord atc = tc;
            int alt = lt, acb = cb;
            uint32_t issued = 0;
            // a tile past the end (the peer's half of a last, odd pair) is staged as zeros by TMA
            auto issue_next = [&]() {
                const uint32_t r = raw_buf(issued);
                if (NHWC && lane == 0) {
                    // x [N][H][W][Cin]: the K block is one box [SR rows][SC columns][32 B of
                    // channels] (zeros outside x: padding, channels past Cin, a tile past the end)
                    constexpr int kCh = BF16 ? 16 : 8;   // channels per K block (32 B)
                    mbar_arrive_expect_tx(&rawfull[r], static_cast<uint32_t>(S::SPOS) * 32u);
                    tma_load_4d_s(smem_u32(smem + a.raw_off) + r * kRawBytes, &tmx, &rawfull[r],
                                  (a.parts == 1 ? acb : acb / 3) * kCh, strip_col<PAIR>(atc, a) * S::PC - a.pad, atc.rb * S::PR - a.pad,
                                  atc.n);
                } else if (lane == 0) {
                    mbar_arrive_expect_tx(&rawfull[r], RBox::kBytes);
                    // the patch starts pad rows above and pad + dcol columns left of the tile: a
                    // 16-byte-aligned column, possibly negative (TMA fills zeros outside x)
                    tma_load_4d(smem + a.raw_off + r * RBox::kBytes, &tmx, &rawfull[r],
                                strip_col<PAIR>(atc, a) * S::PC - a.pad - a.dcol, atc.rb * S::PR - a.pad,
                                (a.parts == 1 ? acb : acb / 3) * RBox::kCh, atc.n);
                }
                ++issued;
                advance(atc, alt, acb, kNumProd);
            };
            if (a.use_tma)
                while (static_cast<int>(issued) < rd && alt < n_pairs) issue_next();
            pdl_wait();   // the re-laid weights and bias are complete and visible from here on
            if (pw == 0 && lane == 0) {
                // own bias block, plus the own half of the weights when they stay resident
                // workspace: [weights of CTA 0 .. step-1][bias blocks of CTA 0 .. step-1]
                const uint8_t* bias_src = reinterpret_cast<const uint8_t*>(a.wr) +
                                          static_cast<size_t>(step) * a.w_total_bytes +
                                          static_cast<size_t>(rank) * a.bias_block_bytes;
                mbar_arrive_expect_tx(wfull, a.bias_block_bytes + (a.resident ? a.w_total_bytes : 0u));
                bulk_g2s(smem + a.bb_off, bias_src, a.bias_block_bytes, wfull);
                if (a.resident) bulk_g2s(smem + a.w_off, wmine, a.w_total_bytes, wfull);
                if (pair && !leader && mbar_wait(wfull, 0, abort_flag, a.status, a.budget))
                    mbar_arrive_remote(mapa_shared(smem_u32(wpeer), 0));
            }
            uint32_t use = 0;                         // this warp's stages whose box was waited for
            uint32_t g = static_cast<uint32_t>(pw);   // global stage index
            long long last_w = -1;                    // stage of this warp's last weight copy
            // The strip of stage `slot` is complete: arrive on its full barrier; a pair's peer then
            // forwards "my half is complete" to the leader once its own barrier has completed.
            // Returns false (for the whole warp) when that wait gave up.
            auto hand_over = [&](uint32_t slot, uint32_t par) -> bool {
                bool fok = true;
                if (lane == 0) {
                    mbar_arrive(&full[slot]);
                    if (pair && !leader) {
                        fok = mbar_wait(&full[slot], par, abort_flag, a.status, a.budget);
                        if (fok) mbar_arrive_remote(mapa_shared(smem_u32(&full[slot]), 0));
                    }
                }
                return __shfl_sync(0xffffffffu, fok ? 1 : 0, 0) != 0;
            };
            while (lt < n_pairs) {
                const uint32_t slot = g % S_;
                const uint32_t par = (g / S_) & 1u;
                bool ok = wait_bar<PAIR, POLL>(&empty[slot], par ^ 1u, abort_flag, a.status, a.budget);
                if (!__all_sync(0xffffffffu, ok)) break;
                fence_proxy_async_smem();
                if (lane == 0) {
                    if (!a.resident) {
                        last_w = g;
                        mbar_arrive_expect_tx(&full[slot], a.w_block_bytes);
                        bulk_g2s(smem + a.w_off + slot * a.w_block_bytes, wmine + static_cast<size_t>(cb) * a.w_block_bytes,
                                 a.w_block_bytes, &full[slot]);
                    } else {
                        mbar_arrive(&full[slot]);
                    }
                }
                if (!FC_DEBUG_OK(slot < S_ && cb < a.ncb, a.status)) {
                    *abort_flag = 1;   // the other roles stop at their next wait, the status kept
                    break;
                }
                const uint32_t strip = strip0 + slot * S::STRIP;
                if (NHWC && !a.use_tma) {
                    fill_strip_nhwc<BF16, WIDE, ROWS, UPW>(strip, a.x, tc.n < a.N ? tc.n : 0, a.parts == 1 ? cb : cb / 3,
                                                      tc.rb * S::PR - a.pad, strip_col<PAIR>(tc, a) * S::PC - a.pad, a.Cin,
                                                      tc.n < a.N ? a.H : 0, a.W, lane, a.parts == 3 && cb % 3 == 2);
                    fence_proxy_async_smem();
                    __syncwarp();
                } else if (a.use_tma) {
                    const uint32_t r = raw_buf(use);
                    ok = mbar_wait<POLL>(&rawfull[r], (use / static_cast<uint32_t>(rd)) & 1u, abort_flag, a.status, a.budget);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    if (!FC_DEBUG_OK(r < static_cast<uint32_t>(kNumProd * rd), a.status)) {
                        *abort_flag = 1;
                        break;
                    }
                    const uint32_t raw = smem_u32(smem + a.raw_off) + r * kRawBytes;
                    // split TF32: the third stage of each K block stages x's remainder
                    if constexpr (NHWC) {
                        if (!BF16 && a.parts == 3 && cb % 3 == 2) copy_raw_nhwc<BF16, WIDE, ROWS, true, UPW>(raw, strip, lane);
                        else copy_raw_nhwc<BF16, WIDE, ROWS, false, UPW>(raw, strip, lane);
                    } else if constexpr (!BF16) {
                        if (a.parts == 3 && cb % 3 == 2) transpose_raw<BF16, WIDE, ROWS, XP, true, UPW>(raw, strip, lane);
                        else transpose_raw<BF16, WIDE, ROWS, XP, false, UPW>(raw, strip, lane);
                    } else {
                        transpose_raw<BF16, WIDE, ROWS, XP, false, UPW>(raw, strip, lane);
                    }
                    fence_proxy_async_smem();   // order the raw reads before the next box overwrites it
                    __syncwarp();
                    if (alt < n_pairs) issue_next();   // reuses buffer r: issued - use == rd
                } else {
                    fill_strip<BF16, WIDE, ROWS, XP, UPW>(strip, a.x, tc.n < a.N ? tc.n : 0, a.parts == 1 ? cb : cb / 3,
                                                     tc.rb * S::PR - a.pad, strip_col<PAIR>(tc, a) * S::PC - a.pad - a.dcol, a.Cin,
                                                     tc.n < a.N ? a.H : 0, a.W, lane, a.parts == 3 && cb % 3 == 2);
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                // every lane fenced its strip writes and the warp has synchronised
                if (!hand_over(slot, par)) break;
                advance(tc, lt, cb, kNumProd);
                ++use;
                g += kNumProd;
            }
            if (*abort_flag && lane == 0) {
                if (last_w >= 0) {
                    // the weight copy of this warp's last stage
                    const uint32_t gl = static_cast<uint32_t>(last_w);
                    drain_wait(&full[gl % S_], (gl / S_) & 1u, kDrainBudgetCycles);
                }
                // boxes requested but not yet waited for
                for (uint32_t i = use; i < issued; ++i)
                    drain_wait(&rawfull[raw_buf(i)], (i / static_cast<uint32_t>(rd)) & 1u, kDrainBudgetCycles);
            }
        }
        if (pw == 0 && lane == 0 && *abort_flag) drain_wait(wfull, 0, kDrainBudgetCycles);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (leader) {
            const uint32_t idesc = make_idesc(BF16 ? kFmtBF16 : kFmtTF32, pair ? 256 : 128, a.Cout);
            // Descriptors are built once; each MMA only moves the start-address field
            // (bits 0-13, 16-byte units).  Every address stays below 256 KB, so the
            // field never carries into the LBO bits above it.  B holds Cout / 2 rows
            // in each CTA of a pair (all Cout rows for a single CTA).
            const uint32_t half_co = static_cast<uint32_t>(a.Cout / step);
            const uint64_t a_desc0 = smem_desc(smem_u32(smem + a.strip_off), S::PLANE, S::SBO, kLayoutNone);
            const uint64_t i_desc0 = smem_desc(smem_u32(smem + a.ind_off), 0u, 128u, kLayoutNone);
            constexpr uint32_t kInd16 = kIndPlane >> 4;
            constexpr uint32_t kZeroPlane = static_cast<uint32_t>(ind_variants(!WIDE));
            // indicator plane of unit u of a tile (see build_indicator_planes); LBO points at the zero plane
            auto unit_ind = [&](const TileCoord& c, int u) -> uint64_t {
                uint32_t v = 0u;
                if constexpr (!PAIR && !WIDE) {
                    const int valid = a.OW - (strip_col<PAIR>(c, a) * S::PC + 8 * u);
                    v = (c.rb == a.RB - 1 ? 3u : 0u) + (valid >= 8 ? 0u : (valid > 0 ? 1u : 2u));
                }
                return i_desc0 + v * kInd16 + (static_cast<uint64_t>((kZeroPlane - v) * kInd16) << 16);
            };
            const uint64_t b_desc0 = smem_desc(smem_u32(smem + a.w_off), half_co * 16u, 128u, kLayoutNone);
            const uint64_t bb_desc = smem_desc(smem_u32(smem + a.bb_off), half_co * 16u, 128u, kLayoutNone);
            const uint32_t wtap16 = 2u * half_co;   // one tap of this CTA's weights, 16-byte units
            const uint32_t wblk16 = a.w_block_bytes >> 4;
            constexpr uint32_t kStrip16 = S::STRIP >> 4;
            bool ok = mbar_wait<POLL>(wfull, 0, abort_flag, a.status, a.budget) &&
                      (!pair || mbar_wait_cluster(wpeer, 0, abort_flag, a.status, a.budget));
            ok = __all_sync(0xffffffffu, ok);
            int acc = 0;   // accumulator ring position of the next unit
            uint32_t aph = 0, slot = 0, sph = 0;
            TileCoord tc = first;
            for (int lt = 0; ok && lt < n_pairs && UPT == 1; ++lt) {
                // one accumulator per tile (pooled tiles, CTA pairs)
                ok = wait_bar<PAIR, POLL>(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.budget);
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc_fence_after();
                ok = FC_DEBUG_OK((acc + 1) * a.Cout <= a.tmem_cols && slot < static_cast<uint32_t>(a.stages), a.status);
                if (!ok) {
                    *abort_flag = 1;
                    break;
                }
                const uint32_t d = tmem + static_cast<uint32_t>(acc * a.Cout);
                // bias (+ padding) K step, overwriting the accumulator
                issue_mma<BF16, PAIR>(d, unit_ind(tc, 0), bb_desc, idesc, 0u);
                for (int cb = 0; cb < a.ncb; ++cb) {
                    ok = wait_bar<PAIR, POLL>(&full[slot], sph, abort_flag, a.status, a.budget);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
                    const uint64_t ab = a_desc0 + slot * kStrip16 + static_cast<uint32_t>(a.dcol);
                    const uint64_t bbase = b_desc0 + (a.resident ? static_cast<uint32_t>(cb) : slot) * wblk16;
                    issue_mma9<BF16, PAIR, S::SC>(d, ab, bbase, wtap16, idesc);
                    commit_to<PAIR>(&empty[slot], 0x3);
                    if (++slot == static_cast<uint32_t>(a.stages)) {
                        slot = 0;
                        sph ^= 1u;
                    }
                }
                if (ok) commit_to<PAIR>(&tfull[acc], 0x3);
                if (++acc == a.nacc) {
                    acc = 0;
                    aph ^= 1u;
                }
                next_tile(tc, a.RB, a.CS);
                if constexpr (PAIR) next_tile(tc, a.RB, a.CS);
            }
            for (int lt = 0; ok && lt < n_pairs && UPT > 1; ++lt) {
                // the tile's UPT units take the next UPT accumulators of the ring
                uint32_t d[UPT];
                int accu[UPT];
#pragma unroll
                for (int u = 0; u < UPT; ++u) {
                    accu[u] = acc;
                    if (!FC_DEBUG_OK((acc + 1) * a.Cout <= a.tmem_cols, a.status)) {
                        ok = false;
                        *abort_flag = 1;
                    }
                    d[u] = tmem + static_cast<uint32_t>(acc * a.Cout);
                    ok = ok && wait_bar<PAIR, POLL>(&tempty[acc], aph ^ 1u, abort_flag, a.status, a.budget);
                    if (++acc == a.nacc) {
                        acc = 0;
                        aph ^= 1u;
                    }
                }
                if (!(ok = __all_sync(0xffffffffu, ok))) break;
                tc_fence_after();
                // bias (+ padding) K step of every unit, overwriting its accumulator
#pragma unroll
                for (int u = 0; u < UPT; ++u) issue_mma<BF16, PAIR>(d[u], unit_ind(tc, u), bb_desc, idesc, 0u);
                for (int cb = 0; cb < a.ncb; ++cb) {
                    ok = wait_bar<PAIR, POLL>(&full[slot], sph, abort_flag, a.status, a.budget);
                    if (!(ok = __all_sync(0xffffffffu, ok))) break;
                    tc_fence_after();
                    const uint64_t ab = a_desc0 + slot * kStrip16 + static_cast<uint32_t>(a.dcol);
                    const uint64_t bbase = b_desc0 + (a.resident ? static_cast<uint32_t>(cb) : slot) * wblk16;
                    // unit u reads the strip u * UOFF staged pixels (16 B each) further.  In the last K
                    // block each unit's accumulator is committed right after its own MMAs (a commit
                    // tracks every MMA issued before it), so the tile groups start staggered.
                    const bool last = cb == a.ncb - 1;
#pragma unroll
                    for (int u = 0; u < UPT; ++u) {
                        issue_mma9<BF16, PAIR, S::SC>(d[u], ab + static_cast<uint64_t>(u * S::UOFF), bbase, wtap16, idesc);
                        if (last) commit_to<PAIR>(&tfull[accu[u]], 0x3);
                    }
                    commit_to<PAIR>(&empty[slot], 0x3);
                    if (++slot == static_cast<uint32_t>(a.stages)) {
                        slot = 0;
                        sph ^= 1u;
                    }
                }
                next_tile(tc, a.RB, a.CS);
                if constexpr (PAIR) next_tile(tc, a.RB, a.CS);
            }
            commit_to<PAIR>(mdone, 0x1);
            drain_wait(mdone, 0, kDrainBudgetCycles);
        }
        __syncwarp();
    } else if (warp < kEpiWarps) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        // warp = (lane quarter q, column group h): this warp owns TMEM lanes 32q..32q+31
        // (tile pixels) and the 16-column accumulator slices c = h, h + 4, h + 8, h + 12.
        const int q = warp & 3;
        const int h = warp >> 2;
        // The four column groups h split into G tile groups: group gi = h / hw takes the
        // tiles lt = gi, gi + G, ... of this CTA's sequence (G = 1, 2 or 4; hw = 4 / G),
        // and within a tile this warp owns the slices c = hh + hw k.  More columns per
        // warp and tile amortise the per-tile hand-offs; groups on different tiles keep
        // the pipes busy while others wait.
        // four side-by-side units: the plan always gives 4 tile groups and 8 accumulators (Cout <= 64),
        // constants the compiler folds into the ring and tile arithmetic below
        const int G = UPW == 4 ? 4 : a.egroups;
        const int nacc = UPW == 4 ? 8 : a.nacc;
        const int hw = 4 / G;
        const int gi = h / hw;
        const int hh = h - gi * hw;
        const int nsub = a.Cout / kEpiCols;
        const int ms = nsub > hh ? min(4, (nsub - hh + hw - 1) / hw) : 0;   // slices of this warp
        const int r = q * 32 + lane;
        const int pr = r / S::PC, pc = r - (r / S::PC) * S::PC;
        const int n_first = first.n;
        // pool: running per-thread sums over the tiles of one image.  The 16x256b load shape
        // gives each thread 4 pixels x 4 channels of a slice, so it keeps 4 sums per slice --
        // sums[k][0] for channels 2(lane%4) + {0, 1} and sums[k][1] for 8 + 2(lane%4) + {0, 1}
        // of slice c = hh + hw k -- reduced across the 8 lanes that share lane%4 only when the
        // image changes.
        float2 sums[4][2];
#pragma unroll
        for (int k = 0; k < 4; ++k) sums[k][0] = sums[k][1] = make_float2(0.0f, 0.0f);
        int cur_n = -1;
        int slots_written = 0;
        bool ok = true;

        // pool records: [CTA][image slot][tile group][lane quarter][Cout]
        auto record = [&](int slot_index) {
            return a.out +
                   (((static_cast<size_t>(blockIdx.x) * a.J + static_cast<size_t>(slot_index)) * G + gi) * 4 + q) *
                       static_cast<size_t>(a.Cout);
        };
        auto zero_slot = [&](int sl) {
            if (!FC_DEBUG_OK(sl >= 0 && sl < a.J, a.status)) return;
            float* dst = record(sl);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = hh + hw * k;
                if (k < ms && lane < kEpiCols) dst[c * kEpiCols + lane] = 0.0f;
            }
        };
        auto flush = [&](int n_img) {
            // images this warp's every-G-th-tile sequence stepped over get zero records
            for (int sl = slots_written; sl < n_img - n_first; ++sl) zero_slot(sl);
            float* dst = record(n_img - n_first);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = hh + hw * k;
                if (k < ms) {
                    {
                        float v4[4] = {sums[k][0].x, sums[k][0].y, sums[k][1].x, sums[k][1].y};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v4[e] += __shfl_xor_sync(0xffffffffu, v4[e], 4);
                            v4[e] += __shfl_xor_sync(0xffffffffu, v4[e], 8);
                            v4[e] += __shfl_xor_sync(0xffffffffu, v4[e], 16);
                        }
                        if (lane < 4 && FC_DEBUG_OK(n_img - n_first >= 0 && n_img - n_first < a.J, a.status)) {
                            float* o = dst + c * kEpiCols + 2 * lane;
                            o[0] = v4[0] * kActScale<ACT>;
                            o[1] = v4[1] * kActScale<ACT>;
                            o[8] = v4[2] * kActScale<ACT>;
                            o[9] = v4[3] * kActScale<ACT>;
                        }
                        sums[k][0] = sums[k][1] = make_float2(0.0f, 0.0f);
                    }
                }
            }
            slots_written = n_img - n_first + 1;
        };

        // Units: the UPT accumulators of every tile of this CTA, in order (unit lt is row
        // us = lt % UPT of tile lt / UPT); group gi takes units gi, gi + G, ...
        const int n_units = n_pairs * UPT;
        TileCoord tc = first;
        int us = 0;
        auto advance_units = [&](int k) {
            if constexpr (UPT == 1) {
                for (int i = 0; i < k * step; ++i) next_tile(tc, a.RB, a.CS);
            } else {
                us += k;
                while (us >= UPT) {
                    us -= UPT;
                    for (int i = 0; i < step; ++i) next_tile(tc, a.RB, a.CS);
                }
            }
        };
        advance_units(gi);
        int lt = gi;
        int acc = gi % nacc;
        uint32_t aph = static_cast<uint32_t>(gi / nacc) & 1u;
        auto taddr = [&](int acc_i, int k) {
            return tmem + (static_cast<uint32_t>(q * 32) << 16) +
                   static_cast<uint32_t>(acc_i * a.Cout + (hh + hw * k) * kEpiCols);
        };
        if constexpr (POOL) {
            // Pooled sums in registers: the slices of this warp's tiles stream through one
            // pipeline -- the load of the next slice (of this tile, or slice 0 of the next
            // tile once this one's accumulator is released) is in flight while the current
            // slice is evaluated.  One barrier hand-off per tile of up to four slices.
            auto slice_addr = [&](int acc_i, int k) {
                return tmem + (static_cast<uint32_t>(q * 32) << 16) +
                       static_cast<uint32_t>(acc_i * a.Cout + (hh + hw * k) * kEpiCols);
            };
            // pixels of this thread in the tile: rows (lane / 4) + {0, 8, 16, 24} of the warp's quarter
            auto pixel_valid = [&](const TileCoord& c, int j) {
                const int rr = q * 32 + (lane >> 2) + 8 * j;
                const int pr_ = rr / S::PC, pc_ = rr - (rr / S::PC) * S::PC;
                return c.rb * S::PR + pr_ < a.OH && strip_col<PAIR>(c, a) * S::PC + pc_ < a.OW;
            };
            // two load buffers, used alternately (slice k of a tile in buf[k & 1]); a tile with an
            // odd number of slices leaves the next tile's slice 0 in buf[1], moved after its wait
            uint32_t buf[2][kEpiCols];
            if (lt < n_units) {
                ok = wait_bar<PAIR, POLL>(&tfull[acc], aph, abort_flag, a.status, a.budget);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok && ms > 0) tmem_ld_slice16x256_start(slice_addr(acc, 0), buf[0]);
            }
            while (ok && lt < n_units) {
                const bool real = t_first + static_cast<long long>(step) * (lt / UPT) < a.num_tiles;   // the peer's half of a last, odd pair is not
                if (real && tc.n != cur_n) {
                    if (cur_n >= 0) flush(cur_n);
                    cur_n = tc.n;
                }
                // padding pixels of a single CTA's tile already activate to -0 (padding K column);
                // CTA pairs mask the edge tiles here
                float m4[4] = {1.0f, 1.0f, 1.0f, 1.0f};
                if (PAIR && (!real || tc.rb == a.RB - 1 || strip_col<PAIR>(tc, a) == a.CS - 1)) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) m4[j] = (real && pixel_valid(tc, j)) ? 1.0f : 0.0f;
                }
                const int nlt = lt + G;
                int nacc_i = acc + G;
                uint32_t naph = aph;
                while (nacc_i >= nacc) {
                    nacc_i -= nacc;
                    naph ^= 1u;
                }
                auto release_and_next = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (pair) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
                        else mbar_arrive(&tempty[acc]);
                    }
                    if (nlt < n_units) {
                        ok = wait_bar<PAIR, POLL>(&tfull[nacc_i], naph, abort_flag, a.status, a.budget);
                        ok = __all_sync(0xffffffffu, ok);
                        tc_fence_after();
                        if (ok && ms > 0) {
                            if (ms & 1) tmem_ld_slice16x256_start(slice_addr(nacc_i, 0), buf[1]);
                            else tmem_ld_slice16x256_start(slice_addr(nacc_i, 0), buf[0]);
                        }
                    }
                };
                if (ms == 0) release_and_next();   // no columns here, but the group's phases are kept
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k < ms) {
                        uint32_t(&cur)[kEpiCols] = buf[k & 1];
                        tmem_ld16_wait(cur);
                        if (k + 1 < ms) tmem_ld_slice16x256_start(slice_addr(acc, k + 1), buf[(k + 1) & 1]);
                        else release_and_next();
                        // cur[8h + 4u + 2p + e]: lane base 16h, pixel (lane / 4) + 16h + 8p, channel
                        // 8u + 2(lane % 4) + e
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
#pragma unroll
                            for (int hp = 0; hp < 4; ++hp) {
                                const int base = 8 * (hp >> 1) + 4 * u + 2 * (hp & 1);
                                float2 g = act2<ACT>(make_float2(__uint_as_float(cur[base]), __uint_as_float(cur[base + 1])));
                                if constexpr (PAIR) g = __fmul2_rn(g, splat2(m4[hp]));
                                sums[k][u] = __fadd2_rn(sums[k][u], g);
                            }
                        }
                    }
                }
                if ((ms & 1) && ok && nlt < n_units) {
                    tmem_ld16_wait(buf[1]);
#pragma unroll
                    for (int j = 0; j < kEpiCols; ++j) buf[0][j] = buf[1][j];
                }
                acc = nacc_i;
                aph = naph;
                lt = nlt;
                advance_units(G);
            }
        }
        if constexpr (!POOL && NHWC) {
            // NHWC full output y [N][OH][OW][Co]: the slices are read in the 16x256b shape, so the
            // four threads that share a pixel hold its 16 channels as 4 pairs each, and one
            // 8-byte store per thread writes 8 pixels x 32 contiguous bytes per instruction (whole
            // sectors).  Same pipeline as the pooled loop: the next slice (or the next tile's
            // first one, once this accumulator is released) loads while this one is stored.
            auto slice_addr = [&](int acc_i, int k) {
                return tmem + (static_cast<uint32_t>(q * 32) << 16) +
                       static_cast<uint32_t>(acc_i * a.Cout + (hh + hw * k) * kEpiCols);
            };
            const bool pairs_ok = (a.Co & 1) == 0;   // 8-byte-aligned channel pairs
            uint32_t buf[2][kEpiCols];
            if (lt < n_units) {
                ok = wait_bar<PAIR, POLL>(&tfull[acc], aph, abort_flag, a.status, a.budget);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (ok && ms > 0) tmem_ld_slice16x256_start(slice_addr(acc, 0), buf[0]);
            }
            while (ok && lt < n_units) {
                const bool real = t_first + static_cast<long long>(step) * (lt / UPT) < a.num_tiles;
                const int nlt = lt + G;
                int nacc_i = acc + G;
                uint32_t naph = aph;
                while (nacc_i >= nacc) {
                    nacc_i -= nacc;
                    naph ^= 1u;
                }
                auto release_and_next = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (pair) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
                        else mbar_arrive(&tempty[acc]);
                    }
                    if (nlt < n_units) {
                        ok = wait_bar<PAIR, POLL>(&tfull[nacc_i], naph, abort_flag, a.status, a.budget);
                        ok = __all_sync(0xffffffffu, ok);
                        tc_fence_after();
                        if (ok && ms > 0) {
                            if (ms & 1) tmem_ld_slice16x256_start(slice_addr(nacc_i, 0), buf[1]);
                            else tmem_ld_slice16x256_start(slice_addr(nacc_i, 0), buf[0]);
                        }
                    }
                };
                if (ms == 0) release_and_next();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (k < ms) {
                        uint32_t(&cur)[kEpiCols] = buf[k & 1];
                        tmem_ld16_wait(cur);
                        if (k + 1 < ms) tmem_ld_slice16x256_start(slice_addr(acc, k + 1), buf[(k + 1) & 1]);
                        else release_and_next();
                        const int c = hh + hw * k;
                        // cur[8hb + 4u + 2p + e]: pixel (lane / 4) + 16hb + 8p of the warp's quarter,
                        // channel 16c + 8u + 2(lane % 4) + e
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
                            for (int pp = 0; pp < 2; ++pp) {
                                const int rr = q * 32 + (lane >> 2) + 16 * hb + 8 * pp;
                                const int oh = tc.rb * S::PR + us + rr / S::PC, ow = strip_col<PAIR>(tc, a) * S::PC + rr % S::PC;
                                const bool valid = real && oh < a.OH && ow < a.OW;
#pragma unroll
                                for (int u = 0; u < 2; ++u) {
                                    const int base = 8 * hb + 4 * u + 2 * pp;
                                    float2 g = act2<ACT>(make_float2(__uint_as_float(cur[base]), __uint_as_float(cur[base + 1])));
                                    if constexpr (ACT == 0) g = __fmul2_rn(g, splat2(kActScale<ACT>));
                                    const int ch = c * kEpiCols + 8 * u + 2 * (lane & 3);
                                    if (valid && ch < a.Co && FC_DEBUG_OK(tc.n < a.N && oh >= 0 && ow >= 0, a.status)) {
                                        float* o = a.out + ((static_cast<size_t>(tc.n) * a.OH + oh) * a.OW + ow) *
                                                               static_cast<size_t>(a.Co) + ch;
                                        if (pairs_ok) {
                                            __stcs(reinterpret_cast<float2*>(o), g);
                                        } else {
                                            __stcs(o, g.x);
                                            if (ch + 1 < a.Co) __stcs(o + 1, g.y);
                                        }
                                    }
                                }
                            }
                        }
                    }
                }
                if ((ms & 1) && ok && nlt < n_units) {
                    tmem_ld16_wait(buf[1]);
#pragma unroll
                    for (int j = 0; j < kEpiCols; ++j) buf[0][j] = buf[1][j];
                }
                acc = nacc_i;
                aph = naph;
                lt = nlt;
                advance_units(G);
            }
        }
        // Full output: the next slice's TMEM load is in flight while the current one is
        // activated and stored; a tile's accumulator is released as soon as its last slice
        // is in registers.
        uint32_t rnext[kEpiCols];
        if (!POOL && !NHWC && lt < n_units) {
            ok = wait_bar<PAIR, POLL>(&tfull[acc], aph, abort_flag, a.status, a.budget);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (ok && ms > 0) tmem_ld16_start(taddr(acc, 0), rnext);
        }
        while (!POOL && !NHWC && ok && lt < n_units) {
            const bool real = t_first + static_cast<long long>(step) * (lt / UPT) < a.num_tiles;   // the peer's half of a last, odd pair is not
            const int oh = tc.rb * S::PR + us + pr, ow = strip_col<PAIR>(tc, a) * S::PC + pc;
            const bool valid = real && oh < a.OH && ow < a.OW;
            const int nlt = lt + G;
            int nacc_i = acc + G;
            uint32_t naph = aph;
            while (nacc_i >= nacc) {
                nacc_i -= nacc;
                naph ^= 1u;
            }
            auto release_and_next = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (pair) mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
                    else mbar_arrive(&tempty[acc]);
                }
                if (nlt < n_units) {
                    ok = wait_bar<PAIR, POLL>(&tfull[nacc_i], naph, abort_flag, a.status, a.budget);
                    ok = __all_sync(0xffffffffu, ok);
                    tc_fence_after();
                    if (ok && ms > 0) tmem_ld16_start(taddr(nacc_i, 0), rnext);
                }
            };
            if (ms == 0) release_and_next();   // no columns here, but the group's phases are kept
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (k < ms) {
                    const int c = hh + hw * k;
                    tmem_ld16_wait(rnext);
                    float v[kEpiCols];
#pragma unroll
                    for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(rnext[j]);
                    if (k + 1 < ms) tmem_ld16_start(taddr(acc, k + 1), rnext);
                    else release_and_next();
                    if constexpr (!POOL) {
                        if (valid && FC_DEBUG_OK(tc.n < a.N && c * kEpiCols < a.Co && oh >= 0 && ow >= 0, a.status)) {
                            float* o = a.out + ((static_cast<size_t>(tc.n) * a.Co + c * kEpiCols) * a.OH + oh) *
                                                   static_cast<size_t>(a.OW) + ow;
                            const size_t plane = static_cast<size_t>(a.OH) * a.OW;
                            const int jmax = a.Co - c * kEpiCols;   // < 16 only in a padded last slice
                            // streaming stores: the output is written once and not re-read here
#pragma unroll
                            for (int j = 0; j < kEpiCols; j += 2) {
                                float2 g = act2<ACT>(make_float2(v[j], v[j + 1]));
                                if constexpr (ACT == 0) g = __fmul2_rn(g, splat2(kActScale<ACT>));
                                if (j < jmax) __stcs(o + j * plane, g.x);
                                if (j + 1 < jmax) __stcs(o + (j + 1) * plane, g.y);
                            }
                        }
                    }
                }
            }
            acc = nacc_i;
            aph = naph;
            lt = nlt;
            advance_units(G);
        }
        if constexpr (POOL) {
            if (ok) {
                if (cur_n >= 0) flush(cur_n);
                // records of image slots this warp never reached are zero, so the
                // combine may add every slot a CTA could have written
                for (int sl = slots_written; sl < a.J; ++sl) zero_slot(sl);
            }
        }
    }

    tc_fence_before();
    if constexpr (PAIR) cluster_sync();   // the leader's MMAs into both CTAs' tensor memory have completed
    else __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem, static_cast<uint32_t>(a.tmem_cols));
        else tmem_dealloc(tmem, static_cast<uint32_t>(a.tmem_cols));
    }
}

template <bool BF16, bool POOL, int ACT, bool PAIR, bool PADX, bool NHWC, int UPW = 1, bool POLL = false>
cudaError_t launch_variant(const CUtensorMap& tmx, const ConvArgs& a, int grid, uint32_t smem_bytes,
                           cudaStream_t stream)
{
    auto kern = conv3x3_fused_kernel<BF16, POOL, ACT, PAIR, PADX, NHWC, UPW, POLL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kConvThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the re-layout's tail
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, tmx, a);
}

// One instantiation per (pool or full output) x activation for each operand type and CTA
// grouping; defined in fc_conv_{tf32,bf16}{,_pair}.cu so the variants compile in parallel.
#define FC_CONV_LAUNCH_DECL(name)                                                                                  \
    cudaError_t name(const CUtensorMap& tmx, const ConvArgs& a, int pool, int act, int grid, uint32_t smem_bytes, \
                     cudaStream_t stream)

// Single-CTA pooled tiles of four side-by-side units (a.upw == 4); CTA pairs have none.
// With a shortened (test) wait budget, only the fp32 erf-GELU variant has a polling instantiation.
template <bool BF16, int ACT, bool PAIR, bool PADX, bool NHWC>
cudaError_t launch_units4(const CUtensorMap& tmx, const ConvArgs& a, int grid, uint32_t smem_bytes, cudaStream_t stream)
{
    if constexpr (PAIR) {
        return cudaErrorInvalidValue;
    } else if constexpr (!BF16 && ACT == 0 && !PADX && !NHWC) {
        if (a.poll) return launch_variant<BF16, true, ACT, false, PADX, NHWC, 4, true>(tmx, a, grid, smem_bytes, stream);
        return launch_variant<BF16, true, ACT, false, PADX, NHWC, 4>(tmx, a, grid, smem_bytes, stream);
    } else {
        if (a.poll) return cudaErrorNotSupported;
        return launch_variant<BF16, true, ACT, false, PADX, NHWC, 4>(tmx, a, grid, smem_bytes, stream);
    }
}

// The variant switch shared by the translation units.
#define FC_CONV_LAUNCH_BODY(BF16, PAIR, PADX, NHWC)                                                      \
    if (a.poll && !(pool && a.upw == 4)) return cudaErrorNotSupported;                                 \
    switch ((pool ? (a.upw == 4 ? 2 : 0) : 1) * 4 + act) {                                              \
    case 0: return launch_variant<BF16, true, 0, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);    \
    case 1: return launch_variant<BF16, true, 1, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);    \
    case 2: return launch_variant<BF16, true, 2, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);    \
    case 3: return launch_variant<BF16, true, 3, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);    \
    case 4: return launch_variant<BF16, false, 0, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);   \
    case 5: return launch_variant<BF16, false, 1, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);   \
    case 6: return launch_variant<BF16, false, 2, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);   \
    case 7: return launch_variant<BF16, false, 3, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);   \
    case 8: return launch_units4<BF16, 0, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);          \
    case 9: return launch_units4<BF16, 1, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);          \
    case 10: return launch_units4<BF16, 2, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);         \
    case 11: return launch_units4<BF16, 3, PAIR, PADX, NHWC>(tmx, a, grid, smem_bytes, stream);         \
    default: return cudaErrorInvalidValue;                                                             \
    }
FC_CONV_LAUNCH_DECL(launch_main_tf32);
FC_CONV_LAUNCH_DECL(launch_main_tf32_pair);
FC_CONV_LAUNCH_DECL(launch_main_bf16);
FC_CONV_LAUNCH_DECL(launch_main_bf16_pair);
// the same with room for a padding column shift (PADX)
FC_CONV_LAUNCH_DECL(launch_main_tf32_padx);
FC_CONV_LAUNCH_DECL(launch_main_tf32_pair_padx);
FC_CONV_LAUNCH_DECL(launch_main_bf16_padx);
FC_CONV_LAUNCH_DECL(launch_main_bf16_pair_padx);
// the same for NHWC (channels-last) input and full output
FC_CONV_LAUNCH_DECL(launch_main_tf32_nhwc);
FC_CONV_LAUNCH_DECL(launch_main_tf32_pair_nhwc);
FC_CONV_LAUNCH_DECL(launch_main_bf16_nhwc);
FC_CONV_LAUNCH_DECL(launch_main_bf16_pair_nhwc);

}  // namespace convk
}  // namespace fc
