// fc_internal.h -- declarations shared by the library's translation units
// (never installed, never part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

// Value a kernel writes into the device status word when a bounded wait runs
// out; equal to FC_ERR_TIMEOUT of the public header.
#define FC_DEVICE_TIMEOUT 5
// Value a kernel of an FC_DEBUG build writes there when one of its index checks fails (the
// checked access is then skipped); equal to FC_ERR_BOUNDS of the public header.
#define FC_DEVICE_BOUNDS 6

// FC_DEBUG_OK(cond, status): true when `cond` holds.  In an FC_DEBUG build a false `cond`
// records FC_DEVICE_BOUNDS in the status word and the caller skips the guarded access; in
// other builds the check compiles to `true` and costs nothing.
#ifdef FC_DEBUG
#define FC_DEBUG_OK(cond, status) ((cond) || (atomicExch((status), FC_DEVICE_BOUNDS), false))
#else
#define FC_DEBUG_OK(cond, status) true
#endif

namespace fc {

// Default spin budget of every mbarrier wait, in SM clock cycles (~1 s at 2 GHz).
constexpr long long kWaitBudgetCycles = 2000000000LL;
// Budget of the drains that run after a wait gave up (a kernel waiting for its own copies and
// MMAs in flight before it frees shared and tensor memory): always the full one, whatever
// budget the call's waits have.
constexpr long long kDrainBudgetCycles = kWaitBudgetCycles;
// The wait budget kernels are launched with: kWaitBudgetCycles, unless a test shortened it
// through the library's testing hook.
long long wait_budget();
// A budget this short comes only from a test; the kernels launched with it poll their barriers
// (see mbar_wait), and only the single-CTA fp32 pooled erf-GELU conv with 16 x 32 tiles and the
// single-CTA fp32 Linear chain have such instantiations (other calls then fail with an error).
constexpr long long kPollBelowCycles = 2000000;
constexpr bool polling_budget(long long budget) { return budget < kPollBelowCycles; }

// ---------------------------------------------------------------- conv

// Geometry and resources of one fused conv3x3 call; computed on the host by
// conv_plan() and passed by value to the kernel.
struct ConvPlan {
    int N, Cin, H, W, OH, OW;   // OH = H + 2 pad - 2, OW = W + 2 pad - 2
    int pad;              // zero padding on every side
    int dcol;             // staged columns before the padded window: (-pad) mod (16 B / esize)
    int padx;             // dcol != 0: the kernel variant with room for that shift
    int nhwc;             // x is [N][H][W][Cin] and the full output [N][OH][OW][Cout]
    int Co;               // output channels of the call (any count in 1 .. 256)
    int Cout;             // Co rounded up to 16: the MMA tile width; channels >= Co carry zero
                          // weights and bias and are never stored
    int bf16, pool;
    int parts;            // products per K block: 1, or 3 for split TF32 (hi*hi, hi*lo, lo*hi)
    int esize;            // bytes per stored element (4 or 2)
    int cb_ch;            // input channels per K block (8 fp32, 16 bf16)
    int ncb;              // K stages per tile = ceil(Cin / cb_ch) * parts
    int RB, CS;           // output row blocks and column strips per image (tiles of 16 x 8, or 1 x 128)
    long long tpi;        // tiles per image = RB * CS
    long long num_tiles;  // N * tpi
    int grid;             // CTAs (persistent)
    int pair;             // CTA pairs (clusters of 2, M = 256 MMAs) instead of single CTAs
    int split_cs;         // pooled pairs: the pair's tiles at column strips j and j + CS / 2
    long long pbase;      // tile groups per cluster (the first `prem` clusters take one more)
    int prem;
    int J;                // image slots per CTA in the pool partial buffer
    int stages;           // shared-memory pipeline depth (staged strips, one producer warp each)
    int raw_depth;        // TMA boxes of x in flight per producer warp (1 .. 4)
    int resident;         // whole re-laid weight tensor kept in shared memory
    int nacc;             // tensor-memory accumulator buffers
    int egroups;          // epilogue tile groups (1, 2, 4): each takes every egroups-th tile
    int upw;              // pooled single-CTA tiles: units side by side (1: 16 x 8, 4: 16 x 32)
    int tmem_cols;        // tensor-memory columns allocated
    uint32_t w_block_bytes;   // one CTA's re-laid weights of one K block: 9 taps * 2 halves * (Cout/2) * 16 B
    uint32_t w_total_bytes;   // ncb * w_block_bytes (one CTA of the pair)
    uint32_t bias_block_bytes;  // one CTA's B operand of the bias K step: 2 halves * (Cout/2) * 16 B
    uint32_t raw_bytes;       // one TMA box of x per K block (channel-major)
    uint32_t strip_bytes;     // one staged K block, channel-blocked
    int use_tma;              // x rows are 16-byte multiples: stage x with TMA boxes
    uint32_t strip_off, raw_off, ind_off, w_off, bb_off, bar_off, smem_bytes;
    size_t ws_weights_bytes;  // re-laid weights + bias block in the workspace
    size_t ws_pool_bytes;     // pool partial sums in the workspace
};

// Fills `plan`; returns 0 on success, 2 (unsupported) when the shape is outside
// what the kernels cover.
// dtype: 0 fp32 (TF32 products), 1 bf16, 2 fp32 with split-TF32 products (the fc_dtype codes);
// pad: zero padding, 0 .. kMaxPad.
constexpr int kMaxPad = 64;
int conv_plan(ConvPlan* plan, int N, int Cin, int H, int W, int Cout, int pad, int nhwc, int dtype, int pool,
              int sm_count);

cudaError_t conv_launch(const ConvPlan& plan, const void* x, const void* w, const void* b, float* y, int act,
                        void* workspace, cudaStream_t stream, int* status, long long budget);

// ---------------------------------------------------------------- linear

struct LinearPlan {
    int M, K, Nout;
    int m_blocks, n_blocks, k_blocks;
    int num_tiles, grid;
    int bf16;             // operands bf16 (kind::f16 MMAs) instead of fp32 (kind::tf32)
    int use_pair;         // CTA pairs with M = 256 MMAs (tcgen05 cta_group::2)
    int m_pairs;          // 256-row blocks in pair mode
    int bn;               // pair mode: columns per tile (a multiple of 32, <= 256)
    int kseg;             // split TF32: K blocks per segment (k_blocks = 3 kseg), else 0
    uint32_t smem_bytes;
    size_t ws_bytes;      // (max, sum-exp) partial per row and column tile
};

// Standalone epilogues over a computed contraction output (fc_epilogue.cu).
cudaError_t act_map_launch(const void* v, float* out, long long n, int bf16, int act, int sm_count, cudaStream_t st);
cudaError_t act_mean_launch(const void* v, float* y, long long planes, long long plane, int bf16, int act,
                            cudaStream_t st);
cudaError_t lse_row_launch(const float* t, float* out, int M, int N, float scale, float lo, float hi, cudaStream_t st);

// split != 0: split TF32 (fp32 only), the K loop over three segments (x, W), (x, W_lo), (x_lo, W).
int linear_plan(LinearPlan* plan, int M, int K, int Nout, int bf16, int sm_count, int split = 0);

// x_lo, W_lo: the TF32 remainders of x and W (split plans only; nullptr otherwise).
cudaError_t linear_launch(const LinearPlan& plan, const void* x, const void* W, const void* b, float* y,
                          float scale, float lo, float hi, void* workspace, cudaStream_t stream, int* status,
                          long long budget, const void* x_lo = nullptr, const void* W_lo = nullptr);

// Split-TF32 Linear: bytes of the TF32 remainders of x [M][K] and W [Nout][K] (fp32, each array
// 256-byte aligned), and the kernels that write them into `dst` (K % 4 == 0); *x_lo and *W_lo
// receive the two arrays' addresses.
size_t linear_split_bytes(int M, int K, int Nout);
cudaError_t linear_split_launch(const float* x, const float* W, int M, int K, int Nout, void* dst, int sm_count,
                                cudaStream_t stream, const float** x_lo, const float** W_lo);

// ---------------------------------------------------------------- misc

cudaError_t watchdog_selftest_launch(long long budget, cudaStream_t stream, int* status);

// cuTensorMapEncodeTiled from the driver (as a PFN_cuTensorMapEncodeTiled_v12000), or null.
void* tensor_map_encoder();

// SM count and device address of the watchdog word of the current device.
cudaError_t current_device_info(int* sm_count, int** status);

}  // namespace fc
