/*
 * fc.h -- C ABI of the GB300 (sm_103a) fused contraction + activation +
 * reduction library.
 *
 * Three fused operators, each a dense contraction on the 5th-generation
 * tensor cores (tcgen05, accumulators in tensor memory) with its pointwise
 * activation and its reduction done in the epilogue, so the contraction's
 * full-size result never goes to HBM (it is written out only where the
 * operator's output IS the full result, fc_conv3x3_act).
 *
 * The three source pages are reasoning traces, each titled by its problem:
 *   "Kimi-K2.6 l2_p67": Conv2d(3x3) -> GELU -> adaptive_avg_pool2d(1) -> squeeze
 *   "Kimi-K2.6 l2_p4" : Conv2d(3x3) -> Mish -> Mish
 *   "Kimi-K2.6 l2_p22": Linear -> x*scale -> x+x -> clamp -> logsumexp(dim 1) -> x*mish(x)
 *
 * Conventions shared by every entry point
 *   - Every data pointer is caller-owned DEVICE memory, contiguous, row-major
 *     (C order), at least 16-byte aligned.  The library allocates nothing and
 *     keeps no state between calls apart from per-device launch attributes.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream).  A
 *     FC_OK return means the work was enqueued; the outputs are fully
 *     overwritten (never accumulated into).
 *   - Argument errors (null pointer, misalignment, non-positive or too-small
 *     sizes, clamp_lo > clamp_hi, workspace too small, unknown enum) return an
 *     error BEFORE anything is enqueued.  Shapes the kernels do not cover
 *     return FC_ERR_UNSUPPORTED; there is no CPU or library fallback.
 *   - `workspace` is caller-owned device scratch of at least
 *     fc_workspace_bytes(...) bytes (256-byte aligned); its contents on entry
 *     do not matter.  Two calls that share a workspace must not overlap.
 *   - Floating point: fp32 inputs run on TF32 tensor cores (the tensor core
 *     reads x, and the Linear op's W, as stored, dropping 13 low mantissa
 *     bits; the conv ops' weights are rounded to nearest TF32 by their per-call
 *     weight re-layout), bf16 inputs on BF16 tensor cores; accumulation, activation and
 *     reduction are fp32; outputs are fp32.  FC_F32_3XTF32 takes the same fp32
 *     inputs but splits each operand into a TF32 high part and a TF32
 *     remainder and sums three products per term (hi*hi + hi*lo + lo*hi),
 *     which brings the contraction's error to fp32 level at three times the
 *     tensor-core work.
 */
#ifndef FC_H_
#define FC_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fc_stream_t;

typedef enum {
    FC_OK = 0,
    FC_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or enum value */
    FC_ERR_UNSUPPORTED = 2,   /* valid request outside the shapes the kernels cover */
    FC_ERR_WORKSPACE = 3,     /* workspace missing or smaller than fc_workspace_bytes() */
    FC_ERR_CUDA = 4,          /* a CUDA runtime/driver call or a launch failed */
    FC_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (see fc_device_status) */
    FC_ERR_BOUNDS = 6         /* FC_DEBUG builds only: a kernel's index check failed and the
                                 access was skipped (see fc_device_status) */
} fc_status;

typedef enum {
    FC_F32 = 0,          /* fp32 storage, TF32 tensor-core products */
    FC_BF16 = 1,         /* bf16 storage, BF16 tensor-core products */
    FC_F32_3XTF32 = 2    /* fp32 storage, split TF32 (3 products per term) */
} fc_dtype;

typedef enum {
    FC_ACT_GELU_ERF = 0,      /* 0.5 v (1 + erf(v / sqrt 2)), torch's exact GELU */
    FC_ACT_MISH = 1,          /* v tanh(softplus(v)) */
    FC_ACT_MISH_MISH = 2,     /* mish(mish(v)) */
    FC_ACT_GELU_TANH = 3      /* 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), torch's
                                 approximate='tanh' GELU, the variant the Conv->GELU->pool
                                 page weighs against the exact form */
} fc_act;

/* Memory layout of the conv ops' x (and of the full output y): NCHW, or NHWC
 * (channels last, PyTorch's channels_last memory format). */
typedef enum { FC_NCHW = 0, FC_NHWC = 1 } fc_layout;

typedef enum {
    FC_OP_CONV3X3_ACT_POOL = 0,
    FC_OP_CONV3X3_ACT = 1,
    FC_OP_LINEAR_LSE_MISH = 2
} fc_op;

/*
 * y[n, co] = mean_{oh < H-2, ow < W-2} act( b[co] + sum_{ci, kh<3, kw<3}
 *                                   x[n, ci, oh+kh, ow+kw] * w[co, ci, kh, kw] )
 *
 * Page "Kimi-K2.6 l2_p67", problem statement: Conv2d(Cin -> Cout, kernel 3,
 * stride 1, padding 0, bias) then GELU then adaptive_avg_pool2d(1) then
 * squeeze, i.e. the mean of the activated conv output over its whole
 * (H-2) x (W-2) plane; the trace fixes GELU to the exact erf form.
 *
 *   x   [N, Cin, H, W]     fp32 or bf16 (dtype), NCHW
 *   w   [Cout, Cin, 3, 3]  same dtype, OIHW
 *   b   [Cout]             same dtype
 *   y   [N, Cout]          fp32 output
 *   dtype FC_F32 or FC_F32_3XTF32 (fp32 x, w, b) or FC_BF16 (bf16 x, w, b).
 *   Requires N, Cin >= 1; H, W >= 3; 1 <= Cout <= 256 (else FC_ERR_UNSUPPORTED).
 *   A Cout that is not a multiple of 16 runs as the next multiple with the
 *   extra channels zero and unstored.  The mean is a fixed-order two-stage sum:
 *   results are bit-identical run to run on the same GPU model.
 */
fc_status fc_conv3x3_act_pool(const void* x, const void* w, const void* b, float* y,
                              int N, int Cin, int H, int W, int Cout,
                              fc_dtype dtype, fc_act act,
                              void* workspace, size_t workspace_bytes, fc_stream_t stream);

/*
 * y[n, co, oh, ow] = act( b[co] + sum_{ci, kh, kw} x[n, ci, oh+kh, ow+kw] * w[co, ci, kh, kw] )
 *
 * Page "Kimi-K2.6 l2_p4", problem statement: Conv2d(Cin -> Cout, kernel 3,
 * stride 1, padding 0, bias) then Mish then Mish (act = FC_ACT_MISH_MISH);
 * the full output is written.
 *
 *   x, w, b as for fc_conv3x3_act_pool;  y [N, Cout, H-2, W-2] fp32, NCHW.
 *   Same shape limits as fc_conv3x3_act_pool.
 */
fc_status fc_conv3x3_act(const void* x, const void* w, const void* b, float* y,
                         int N, int Cin, int H, int W, int Cout,
                         fc_dtype dtype, fc_act act,
                         void* workspace, size_t workspace_bytes, fc_stream_t stream);

/*
 * The two conv operators with zero padding p on every side and a choice of
 * memory layout.  Padding is PyTorch's Conv2d(padding=p), padding_mode 'zeros',
 * the general-padding variant of the pages' padding-0 convs (the Conv2d -> GELU
 * -> pool page raises padded convs as the general case):
 *   v[n, co, oh, ow] = b[co] + sum_{ci, kh, kw} x[n, ci, oh+kh-p, ow+kw-p] * w[co, ci, kh, kw],
 * terms outside the input omitted; output plane OH x OW = (H+2p-2) x (W+2p-2),
 * so p = 1 keeps H x W.  fc_conv3x3_act_pool_ex: y [N, Cout], the mean over
 * the OH x OW plane; fc_conv3x3_act_ex: the full output.
 *   layout FC_NCHW: x [N, Cin, H, W], full y [N, Cout, OH, OW];
 *   layout FC_NHWC: x [N, H, W, Cin], full y [N, OH, OW, Cout] (channels last);
 *   w is [Cout, Cin, 3, 3] (OIHW) and b [Cout] in both layouts.
 *   Requires 0 <= pad <= 64, H, W >= 1 with H + 2 pad >= 3 and W + 2 pad >= 3
 *   (FC_ERR_INVALID_ARG otherwise); the rest as for the pad-0 NCHW entry points
 *   (pad = 0, FC_NCHW gives exactly their results).  The workspace size comes
 *   from fc_workspace_bytes_ex.
 */
fc_status fc_conv3x3_act_pool_ex(const void* x, const void* w, const void* b, float* y,
                                 int N, int Cin, int H, int W, int Cout, int pad, fc_layout layout,
                                 fc_dtype dtype, fc_act act,
                                 void* workspace, size_t workspace_bytes, fc_stream_t stream);
fc_status fc_conv3x3_act_ex(const void* x, const void* w, const void* b, float* y,
                            int N, int Cin, int H, int W, int Cout, int pad, fc_layout layout,
                            fc_dtype dtype, fc_act act,
                            void* workspace, size_t workspace_bytes, fc_stream_t stream);

/*
 * t[m, j] = clamp( u + u, clamp_lo, clamp_hi ),  u = (b[j] + sum_k x[m, k] W[j, k]) * scale
 * l[m]    = log sum_j exp(t[m, j])
 * y[m]    = l[m] * mish(l[m])
 *
 * Page "Kimi-K2.6 l2_p22", problem statement (the module's forward):
 * nn.Linear(K -> Nout) then x * scale_factor then x + x then torch.clamp then
 * torch.logsumexp(dim=1, keepdim=True) then x * mish(x).  The row logsumexp
 * is taken as per-tile (max, sum of exp) pairs combined across column tiles.
 *
 *   x [M, K], W [Nout, K] (nn.Linear weight layout), b [Nout]: all fp32 (TF32
 *   tensor-core products) or all bf16 (dtype FC_BF16); y [M] fp32 (the (M, 1)
 *   output, contiguous); fp32 accumulation and epilogue either way.
 *   Requires M, Nout >= 1, a 16-byte row pitch (K % 4 == 0 for fp32, K % 8 == 0
 *   for bf16; FC_ERR_UNSUPPORTED otherwise), clamp_lo <= clamp_hi.
 *   dtype FC_F32_3XTF32 (fp32 x, W, b): split TF32 for fp32-level product
 *   error.  The tensor core reads raw fp32 as TF32 by dropping 13 low mantissa
 *   bits (the high part hi); a small kernel writes the remainders
 *   lo = (v - hi) rounded to TF32 of x and W into the workspace, and the GEMM's
 *   K loop runs three times -- over (x, W), (x, W_lo), (x_lo, W) -- summing
 *   hi*hi + hi*lo + lo*hi.  The workspace then also holds the remainders
 *   ((M + Nout) K fp32 values, see fc_workspace_bytes).  Inputs must be finite.
 */
fc_status fc_linear_lse_mish(const void* x, const void* W, const void* b, float* y,
                             int M, int K, int Nout, float scale, float clamp_lo, float clamp_hi,
                             fc_dtype dtype,
                             void* workspace, size_t workspace_bytes, fc_stream_t stream);

/*
 * The pages' epilogue-only kernels, for a contraction computed elsewhere (each
 * page's own deliverable is such a kernel run after cuDNN / cuBLAS).  Inputs are
 * the contraction's output with the bias already added; fp32 or bf16 input (for
 * fc_scale_clamp_lse_mish fp32), fp32 output; all pointers device memory, 16-byte
 * aligned, caller-owned; asynchronous on `stream`; no workspace.
 *
 * fc_act_map: out[i] = act(v[i]) for i < n (Conv->Mish->Mish page, its
 *   elementwise Mish-twice kernel; any fc_act).  n == 0 does nothing.
 * fc_act_mean: y[p] = mean over i < plane_size of act(v[p * plane_size + i]) for
 *   p < planes: the (H, W) plane mean of an NCHW tensor with planes = N * C
 *   (Conv->GELU->pool page, its fused GELU + global-average-pool kernel).
 *   Requires 1 <= planes <= 2^31 - 1, plane_size >= 1.
 * fc_scale_clamp_lse_mish: for each row m < M of t (M x N, row-major),
 *   u = clamp(t * scale + t * scale, clamp_lo, clamp_hi), l = logsumexp_j u_j,
 *   y[m] = l * mish(l) (Linear page, its row kernel).  Requires 1 <= M <= 2^31 - 1,
 *   N >= 1, clamp_lo <= clamp_hi.
 * Errors: FC_ERR_INVALID_ARG for null or misaligned pointers, bad sizes or
 * enums; FC_ERR_CUDA if a launch fails.
 */
fc_status fc_act_map(const void* v, float* out, long long n, fc_dtype dtype, fc_act act, fc_stream_t stream);
fc_status fc_act_mean(const void* v, float* y, long long planes, long long plane_size, fc_dtype dtype, fc_act act,
                      fc_stream_t stream);
fc_status fc_scale_clamp_lse_mish(const float* t, float* y, int M, int N, float scale, float clamp_lo,
                                  float clamp_hi, fc_stream_t stream);

/*
 * fc_linear_lse_mish without a workspace argument, for callers that cannot
 * allocate device memory: code whose device memory belongs to another
 * allocator or a fixed budget, C hosts with no allocator of their own, or
 * loops where a cudaMalloc (which may synchronize the device) is not
 * acceptable.  The pages have no counterpart to this entry point; it is an
 * interface convenience, not part of the method.
 *
 * Same operator, arguments, limits and errors as fc_linear_lse_mish (fp32
 * only).  Its scratch is a 1 MiB array in device memory that the library
 * holds on every device that loads it, until the process exits; requests
 * whose scratch (8 bytes per row and column tile: what fc_workspace_bytes
 * reports for the same shape) exceeds 1 MiB return FC_ERR_UNSUPPORTED.
 * The call allocates nothing.  The first call on a device looks up that
 * array's device address (a one-time set-up); make that first call before
 * any stream capture (a look-up that fails returns FC_ERR_CUDA and is tried
 * again by the next call).  All calls share the one array: calls that
 * overlap on the GPU (other streams, or other host threads) race on it and
 * give wrong results.  Nothing in it needs to start at zero.
 */
fc_status fc_linear_lse_mish_noalloc(const void* x, const void* W, const void* b, float* y,
                                     int M, int K, int Nout, float scale, float clamp_lo, float clamp_hi,
                                     fc_stream_t stream);

/*
 * Workspace bytes the given call needs on the CURRENT device (0 is possible).
 * Argument order follows the call: (N, Cin, H, W, Cout) for the conv ops,
 * (M, K, -, -, Nout) for the linear op.  Returns 0 for invalid arguments.
 */
size_t fc_workspace_bytes(fc_op op, int n_or_m, int cin_or_k, int h, int w, int cout_or_nout,
                          fc_dtype dtype);

/* The same for the conv _ex entry points (op = one of the two conv ops). */
size_t fc_workspace_bytes_ex(fc_op op, int n, int cin, int h, int w, int cout, int pad, fc_layout layout,
                             fc_dtype dtype);

/*
 * Host-buffer forms of the two conv operators: the _ex operators (same
 * arguments, limits and results) with x, w, b and y in HOST memory.  The call
 * copies w and b to the device, then the batch in `chunks` slices of whole
 * images (1 .. 64; fewer when N is smaller); each slice's kernels start as
 * soon as that slice has arrived and each slice's result is copied back as
 * soon as it is computed, so the host<->device copies of one slice overlap
 * the kernels of another.  Per image the result is that of the device-buffer
 * call on the slice holding it (bit-identical to a device-buffer call on the
 * same slice).  The pages have no counterpart to this entry point; it is the
 * end-to-end interface for data that starts in host memory.
 *
 *   x, w, b, y   host pointers, no alignment needed.  Page-locked (pinned)
 *                memory gives asynchronous, overlapped copies; pageable memory
 *                works but its copies are not overlapped.
 *   chunks       slices of the batch (the overlap granularity).
 *   staging      device memory of at least fc_host_staging_bytes(...) bytes,
 *                256-byte aligned, caller-owned: the device copies of x, w, b,
 *                y and the operator's workspace.
 *   stream       the call is asynchronous and ordered as if all of it ran on
 *                `stream`: the copies start after the work already enqueued
 *                there, and work enqueued there later starts after the last
 *                result has reached y.  y is valid after `stream` has
 *                synchronized.  The copies run on two library-owned streams
 *                per device (created on the first call); concurrent calls on
 *                one device are serialised by a lock while they enqueue.
 * Errors: FC_ERR_INVALID_ARG / FC_ERR_UNSUPPORTED as for the _ex operators
 * (and for chunks < 1), FC_ERR_WORKSPACE for a missing, misaligned or short
 * staging buffer (checked before anything is enqueued), FC_ERR_CUDA if a copy
 * or launch fails (earlier slices may then already be enqueued; `stream` still
 * waits for every copy that was, so the buffers stay in use until then).
 */
fc_status fc_conv3x3_act_pool_host(const void* x, const void* w, const void* b, float* y,
                                   int N, int Cin, int H, int W, int Cout, int pad, fc_layout layout,
                                   fc_dtype dtype, fc_act act, int chunks,
                                   void* staging, size_t staging_bytes, fc_stream_t stream);
fc_status fc_conv3x3_act_host(const void* x, const void* w, const void* b, float* y,
                              int N, int Cin, int H, int W, int Cout, int pad, fc_layout layout,
                              fc_dtype dtype, fc_act act, int chunks,
                              void* staging, size_t staging_bytes, fc_stream_t stream);

/* Staging bytes for the host-buffer conv operators on the CURRENT device
 * (op = one of the two conv ops); 0 for invalid arguments. */
size_t fc_host_staging_bytes(fc_op op, int n, int cin, int h, int w, int cout, int pad, fc_layout layout,
                             fc_dtype dtype, int chunks);

/* Static English text for a status code. */
const char* fc_status_string(fc_status status);

/*
 * Watchdog word of the current device.  Every spin-wait in the kernels is
 * bounded; on expiry a kernel records FC_ERR_TIMEOUT here, stops its loops,
 * drains its own copies and returns (the context stays usable).  While the
 * word holds FC_ERR_TIMEOUT (or FC_ERR_BOUNDS), the pooled conv and Linear operators write NaN
 * to their outputs (their partial results cannot be trusted); a full-output
 * conv whose kernel gave up leaves its output undefined.  This call
 * synchronizes the device, returns the recorded status (FC_OK if none) and,
 * when clear != 0, resets it.
 */
fc_status fc_device_status(int clear);

/*
 * The same word read after the work enqueued on `stream` so far has finished,
 * without synchronizing the rest of the device, and without clearing it (the
 * word is shared by every stream of the device; fc_device_status(1) clears it).
 * Returns FC_OK, FC_ERR_TIMEOUT, or FC_ERR_CUDA if the stream or the read fails.
 */
fc_status fc_last_device_status(fc_stream_t stream);

/*
 * Self-test of the watchdog path: enqueues one tiny kernel that waits on an
 * mbarrier nothing will ever arrive on, with a budget of `budget_cycles`
 * SM clock cycles.  The wait must give up, record FC_ERR_TIMEOUT and return.
 * Read the result with fc_device_status().  Faults and hangs nothing.
 */
fc_status fc_selftest_watchdog(unsigned long long budget_cycles, fc_stream_t stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int fc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FC_H_ */
