// fc_host.cu -- host-buffer forms of the two conv operators.  The batch goes to the
// device in slices of whole images on a copy stream; each slice's kernels run on the
// caller's stream as soon as that slice has landed, and each slice's result goes back
// on a second copy stream.  The host<->device link (a few hundred GB/s) is far slower
// than the kernels, so overlapping the copies with the kernels is what an end-to-end
// call from host memory can gain.  No arithmetic happens here: every slice is one call
// of the device-buffer entry point.
#include "../../include/fc.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;

// Per-device copy streams and events, created on first use and kept for the process.
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr;    // host -> device copies
    cudaStream_t out = nullptr;   // device -> host copies
    cudaEvent_t start = nullptr, params_in = nullptr, y_out = nullptr;
    cudaEvent_t x_in[kMaxChunks] = {};
    cudaEvent_t done[kMaxChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

cudaError_t pipe_init(HostPipe& p)
{
    if (p.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
    const unsigned fl = cudaEventDisableTiming;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, fl);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.params_in, fl);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.y_out, fl);
    for (int i = 0; i < kMaxChunks && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&p.x_in[i], fl);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done[i], fl);
    }
    p.ready = e == cudaSuccess;
    return e;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Where everything lives in the caller's staging buffer (offsets in bytes, each 256-byte
// aligned): the weights and bias, the operator's workspace (one, reused slice after slice
// since the slices run in order on one stream), then one result slot and one input slot
// per slice.
struct StagingPlan {
    int n0 = 0, chunks = 0;            // images per slice (the last may hold fewer), slices
    size_t img_x = 0, img_y = 0;       // bytes of one image's input / result
    size_t w_bytes = 0, b_bytes = 0, ws_bytes = 0;
    size_t off_b = 0, off_ws = 0, off_y = 0, y_slot = 0, off_x = 0, x_slot = 0, total = 0;
};

// False when the arguments are invalid (the workspace query answers 0 for those: every
// valid conv call needs workspace for its re-laid-out weights).
bool staging_plan(StagingPlan* s, fc_op op, int N, int Cin, int H, int W, int Cout, int pad, fc_layout layout,
                  fc_dtype dtype, int chunks)
{
    if (op != FC_OP_CONV3X3_ACT_POOL && op != FC_OP_CONV3X3_ACT) return false;
    if (N < 1 || Cin < 1 || Cout < 1 || H < 1 || W < 1 || pad < 0 || chunks < 1) return false;
    if (dtype != FC_F32 && dtype != FC_BF16 && dtype != FC_F32_3XTF32) return false;
    const size_t es = dtype == FC_BF16 ? 2 : 4;
    int c = chunks < kMaxChunks ? chunks : kMaxChunks;
    if (c > N) c = N;
    s->n0 = (N + c - 1) / c;
    s->chunks = (N + s->n0 - 1) / s->n0;
    const int last = N - (s->chunks - 1) * s->n0;
    const size_t ws0 = fc_workspace_bytes_ex(op, s->n0, Cin, H, W, Cout, pad, layout, dtype);
    const size_t ws1 = fc_workspace_bytes_ex(op, last, Cin, H, W, Cout, pad, layout, dtype);
    if (ws0 == 0 || ws1 == 0) return false;
    const size_t OH = static_cast<size_t>(H) + 2 * pad - 2, OW = static_cast<size_t>(W) + 2 * pad - 2;
    s->img_x = static_cast<size_t>(Cin) * H * W * es;
    s->img_y = (op == FC_OP_CONV3X3_ACT_POOL ? static_cast<size_t>(Cout) : Cout * OH * OW) * sizeof(float);
    s->w_bytes = static_cast<size_t>(Cout) * Cin * 9 * es;
    s->b_bytes = static_cast<size_t>(Cout) * es;
    s->ws_bytes = ws0 > ws1 ? ws0 : ws1;
    s->off_b = align256(s->w_bytes);
    s->off_ws = s->off_b + align256(s->b_bytes);
    s->off_y = s->off_ws + align256(s->ws_bytes);
    s->y_slot = align256(s->n0 * s->img_y);
    s->off_x = s->off_y + s->chunks * s->y_slot;
    s->x_slot = align256(s->n0 * s->img_x);
    s->total = s->off_x + s->chunks * s->x_slot;
    return true;
}

fc_status host_call(fc_op op, const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W,
                    int Cout, int pad, fc_layout layout, fc_dtype dtype, fc_act act, int chunks, void* staging,
                    size_t staging_bytes, fc_stream_t stream)
{
    if (!x || !w || !b || !y) return FC_ERR_INVALID_ARG;
    if (chunks < 1) return FC_ERR_INVALID_ARG;
    StagingPlan s;
    if (!staging_plan(&s, op, N, Cin, H, W, Cout, pad, layout, dtype, chunks)) {
        // The device-buffer entry point tells a malformed call (FC_ERR_INVALID_ARG) from a
        // shape its kernels do not cover (FC_ERR_UNSUPPORTED) or a missing device
        // (FC_ERR_CUDA).  With no workspace it cannot launch anything: every conv plan
        // needs workspace for its re-laid-out weights.
        void* const dummy = reinterpret_cast<void*>(static_cast<uintptr_t>(256));
        const fc_status st =
            op == FC_OP_CONV3X3_ACT_POOL
                ? fc_conv3x3_act_pool_ex(dummy, dummy, dummy, static_cast<float*>(dummy), N, Cin, H, W, Cout, pad,
                                         layout, dtype, act, nullptr, 0, stream)
                : fc_conv3x3_act_ex(dummy, dummy, dummy, static_cast<float*>(dummy), N, Cin, H, W, Cout, pad, layout,
                                    dtype, act, nullptr, 0, stream);
        return st == FC_OK || st == FC_ERR_WORKSPACE ? FC_ERR_INVALID_ARG : st;
    }
    if (!staging || staging_bytes < s.total || (reinterpret_cast<uintptr_t>(staging) & 255u)) return FC_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FC_ERR_CUDA;
    HostPipe& p = g_pipe[dev];
    std::lock_guard<std::mutex> lock(p.mu);
    if (pipe_init(p) != cudaSuccess) return FC_ERR_CUDA;

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // On a failure after copies were enqueued, the caller's stream still waits for them, so that
    // the staging buffer and the host buffers stay in use until they have finished.
    auto fail = [&](fc_status st) {
        if (cudaEventRecord(p.params_in, p.in) == cudaSuccess) cudaStreamWaitEvent(cs, p.params_in, 0);
        if (cudaEventRecord(p.y_out, p.out) == cudaSuccess) cudaStreamWaitEvent(cs, p.y_out, 0);
        return st;
    };
    char* base = static_cast<char*>(staging);
    char* w_d = base;
    char* b_d = base + s.off_b;
    void* ws_d = base + s.off_ws;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    const char* xh = static_cast<const char*>(x);
    char* yh = reinterpret_cast<char*>(y);

    // The copies start only after the work already on the caller's stream: an earlier call
    // may still be reading this staging buffer.
    cudaError_t e = cudaEventRecord(p.start, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.in, p.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.start, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(w_d, w, s.w_bytes, h2d, p.in);
    if (e == cudaSuccess) e = cudaMemcpyAsync(b_d, b, s.b_bytes, h2d, p.in);
    if (e == cudaSuccess) e = cudaEventRecord(p.params_in, p.in);
    for (int i = 0; i < s.chunks && e == cudaSuccess; ++i) {
        const int n = i + 1 < s.chunks ? s.n0 : N - i * s.n0;
        e = cudaMemcpyAsync(base + s.off_x + i * s.x_slot, xh + static_cast<size_t>(i) * s.n0 * s.img_x,
                            n * s.img_x, h2d, p.in);
        if (e == cudaSuccess) e = cudaEventRecord(p.x_in[i], p.in);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p.params_in, 0);
    if (e != cudaSuccess) return fail(FC_ERR_CUDA);
    for (int i = 0; i < s.chunks; ++i) {
        const int n = i + 1 < s.chunks ? s.n0 : N - i * s.n0;
        void* x_d = base + s.off_x + i * s.x_slot;
        float* y_d = reinterpret_cast<float*>(base + s.off_y + i * s.y_slot);
        if (cudaStreamWaitEvent(cs, p.x_in[i], 0) != cudaSuccess) return fail(FC_ERR_CUDA);
        const fc_status st =
            op == FC_OP_CONV3X3_ACT_POOL
                ? fc_conv3x3_act_pool_ex(x_d, w_d, b_d, y_d, n, Cin, H, W, Cout, pad, layout, dtype, act, ws_d,
                                         s.ws_bytes, stream)
                : fc_conv3x3_act_ex(x_d, w_d, b_d, y_d, n, Cin, H, W, Cout, pad, layout, dtype, act, ws_d,
                                    s.ws_bytes, stream);
        if (st != FC_OK) return fail(st);
        e = cudaEventRecord(p.done[i], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.done[i], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(yh + static_cast<size_t>(i) * s.n0 * s.img_y, y_d, n * s.img_y, d2h, p.out);
        if (e != cudaSuccess) return fail(FC_ERR_CUDA);
    }
    // The caller's stream ends after the last result has reached the host.
    e = cudaEventRecord(p.y_out, p.out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p.y_out, 0);
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t fc_host_staging_bytes(fc_op op, int n, int cin, int h, int w, int cout, int pad, fc_layout layout,
                             fc_dtype dtype, int chunks)
{
    StagingPlan s;
    return staging_plan(&s, op, n, cin, h, w, cout, pad, layout, dtype, chunks) ? s.total : 0;
}

fc_status fc_conv3x3_act_pool_host(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H,
                                   int W, int Cout, int pad, fc_layout layout, fc_dtype dtype, fc_act act,
                                   int chunks, void* staging, size_t staging_bytes, fc_stream_t stream)
{
    return host_call(FC_OP_CONV3X3_ACT_POOL, x, w, b, y, N, Cin, H, W, Cout, pad, layout, dtype, act, chunks,
                     staging, staging_bytes, stream);
}

fc_status fc_conv3x3_act_host(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W,
                              int Cout, int pad, fc_layout layout, fc_dtype dtype, fc_act act, int chunks,
                              void* staging, size_t staging_bytes, fc_stream_t stream)
{
    return host_call(FC_OP_CONV3X3_ACT, x, w, b, y, N, Cin, H, W, Cout, pad, layout, dtype, act, chunks, staging,
                     staging_bytes, stream);
}

}  // extern "C"
