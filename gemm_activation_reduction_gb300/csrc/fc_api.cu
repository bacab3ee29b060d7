// fc_api.cu -- the C ABI: argument validation, workspace sizing, the device
// status word, and dispatch to the fused kernels.  No entry point allocates
// memory or falls back to anything but its CUDA kernels.
#include "../../include/fc.h"
#include "fc_internal.h"
#include "fc_ptx.cuh"

#include <atomic>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;

__device__ int g_fc_status = 0;

// Wait budget of the next launches (see fc::wait_budget); only the testing hook below changes it.
std::atomic<long long> g_wait_budget{fc::kWaitBudgetCycles};

struct DeviceState {
    std::atomic<bool> ready{false};   // set once sm_count and status hold this device's values
    int sm_count = 0;
    int* status = nullptr;            // device address of g_fc_status on this device
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mutex;

// SM count and status-word address of the current device.  Only a successful look-up is kept:
// a failed one (say, a first call made while a stream capture forbids it) is tried again on the
// next call.
fc_status device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FC_ERR_CUDA;
    DeviceState& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            int* st = nullptr;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaGetSymbolAddress(reinterpret_cast<void**>(&st), g_fc_status) != cudaSuccess || st == nullptr)
                return FC_ERR_CUDA;
            d.sm_count = sms;
            d.status = st;
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return FC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by the conv entry points and the workspace query: a padded input of
// at least 3 x 3 (an output of at least 1 x 1) and a padding in 0 .. kMaxPad.
bool conv_shape_ok(int N, int Cin, int H, int W, int Cout, int pad)
{
    return N >= 1 && Cin >= 1 && Cout >= 1 && H >= 1 && W >= 1 && pad >= 0 && pad <= fc::kMaxPad &&
           H + 2 * pad >= 3 && W + 2 * pad >= 3;
}

fc_status conv_common(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W, int Cout,
                      int pad, fc_layout layout, fc_dtype dtype, fc_act act, void* workspace,
                      size_t workspace_bytes, fc_stream_t stream, int pool)
{
    if (!x || !w || !b || !y) return FC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(b) || !aligned16(y)) return FC_ERR_INVALID_ARG;
    if (!conv_shape_ok(N, Cin, H, W, Cout, pad)) return FC_ERR_INVALID_ARG;
    if (layout != FC_NCHW && layout != FC_NHWC) return FC_ERR_INVALID_ARG;
    if (dtype != FC_F32 && dtype != FC_BF16 && dtype != FC_F32_3XTF32) return FC_ERR_INVALID_ARG;
    if (act != FC_ACT_GELU_ERF && act != FC_ACT_MISH && act != FC_ACT_MISH_MISH && act != FC_ACT_GELU_TANH)
        return FC_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    fc::ConvPlan plan;
    if (fc::conv_plan(&plan, N, Cin, H, W, Cout, pad, layout == FC_NHWC, static_cast<int>(dtype), pool,
                      d->sm_count) != 0)
        return FC_ERR_UNSUPPORTED;
    const size_t need = plan.ws_weights_bytes + plan.ws_pool_bytes;
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return FC_ERR_WORKSPACE;
    cudaError_t e = fc::conv_launch(plan, x, w, b, y, static_cast<int>(act), workspace,
                                    reinterpret_cast<cudaStream_t>(stream), d->status, fc::wait_budget());
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

__global__ void watchdog_kernel(long long budget, int* status)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        fc::mbar_init(&bar, 1);
        abort_flag = 0;
        fc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the bounded wait must give up and record the timeout.
        fc::mbar_wait(&bar, 0, &abort_flag, status, budget);
    }
    __syncthreads();
}

}  // namespace

namespace fc {
cudaError_t watchdog_selftest_launch(long long budget, cudaStream_t stream, int* status)
{
    watchdog_kernel<<<1, 32, 0, stream>>>(budget, status);
    return cudaGetLastError();
}

long long wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }

cudaError_t current_device_info(int* sm_count, int** status)
{
    DeviceState* d = nullptr;
    if (device_state(&d) != FC_OK) return cudaErrorInvalidDevice;
    *sm_count = d->sm_count;
    *status = d->status;
    return cudaSuccess;
}
}  // namespace fc

extern "C" {

fc_status fc_conv3x3_act_pool(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W,
                              int Cout, fc_dtype dtype, fc_act act, void* workspace, size_t workspace_bytes,
                              fc_stream_t stream)
{
    if (H < 3 || W < 3) return FC_ERR_INVALID_ARG;
    return conv_common(x, w, b, y, N, Cin, H, W, Cout, 0, FC_NCHW, dtype, act, workspace, workspace_bytes, stream, 1);
}

fc_status fc_conv3x3_act(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W, int Cout,
                         fc_dtype dtype, fc_act act, void* workspace, size_t workspace_bytes, fc_stream_t stream)
{
    if (H < 3 || W < 3) return FC_ERR_INVALID_ARG;
    return conv_common(x, w, b, y, N, Cin, H, W, Cout, 0, FC_NCHW, dtype, act, workspace, workspace_bytes, stream, 0);
}

fc_status fc_conv3x3_act_pool_ex(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H,
                                 int W, int Cout, int pad, fc_layout layout, fc_dtype dtype, fc_act act,
                                 void* workspace, size_t workspace_bytes, fc_stream_t stream)
{
    return conv_common(x, w, b, y, N, Cin, H, W, Cout, pad, layout, dtype, act, workspace, workspace_bytes, stream,
                       1);
}

fc_status fc_conv3x3_act_ex(const void* x, const void* w, const void* b, float* y, int N, int Cin, int H, int W,
                            int Cout, int pad, fc_layout layout, fc_dtype dtype, fc_act act, void* workspace,
                            size_t workspace_bytes, fc_stream_t stream)
{
    return conv_common(x, w, b, y, N, Cin, H, W, Cout, pad, layout, dtype, act, workspace, workspace_bytes, stream,
                       0);
}

fc_status fc_linear_lse_mish(const void* x, const void* W, const void* b, float* y, int M, int K, int Nout,
                             float scale, float clamp_lo, float clamp_hi, fc_dtype dtype, void* workspace,
                             size_t workspace_bytes, fc_stream_t stream)
{
    if (!x || !W || !b || !y) return FC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(b) || !aligned16(y)) return FC_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || Nout < 1) return FC_ERR_INVALID_ARG;
    if (!(clamp_lo <= clamp_hi)) return FC_ERR_INVALID_ARG;   // also rejects NaN bounds
    if (dtype != FC_F32 && dtype != FC_BF16 && dtype != FC_F32_3XTF32) return FC_ERR_INVALID_ARG;
    if (K % (dtype == FC_BF16 ? 8 : 4) != 0) return FC_ERR_UNSUPPORTED;   // 16-byte row pitch for TMA
    const bool split = dtype == FC_F32_3XTF32;
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    fc::LinearPlan plan;
    if (fc::linear_plan(&plan, M, K, Nout, dtype == FC_BF16, d->sm_count, split) != 0) return FC_ERR_UNSUPPORTED;
    const size_t part = (plan.ws_bytes + 255) & ~static_cast<size_t>(255);
    const size_t need = part + (split ? fc::linear_split_bytes(M, K, Nout) : 0);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return FC_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float* x_lo = nullptr;
    const float* W_lo = nullptr;
    if (split) {
        cudaError_t e = fc::linear_split_launch(static_cast<const float*>(x), static_cast<const float*>(W), M, K,
                                                Nout, static_cast<char*>(workspace) + part, d->sm_count, s, &x_lo,
                                                &W_lo);
        if (e != cudaSuccess) return FC_ERR_CUDA;
    }
    cudaError_t e = fc::linear_launch(plan, x, W, b, y, scale, clamp_lo, clamp_hi, workspace, s, d->status,
                                      fc::wait_budget(), x_lo, W_lo);
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

namespace {
bool valid_act(fc_act act)
{
    return act == FC_ACT_GELU_ERF || act == FC_ACT_MISH || act == FC_ACT_MISH_MISH || act == FC_ACT_GELU_TANH;
}
}  // namespace

fc_status fc_act_map(const void* v, float* out, long long n, fc_dtype dtype, fc_act act, fc_stream_t stream)
{
    if (!v || !out || !aligned16(v) || !aligned16(out)) return FC_ERR_INVALID_ARG;
    if (n < 0 || (dtype != FC_F32 && dtype != FC_BF16) || !valid_act(act)) return FC_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    cudaError_t e = fc::act_map_launch(v, out, n, dtype == FC_BF16, static_cast<int>(act), d->sm_count,
                                       reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

fc_status fc_act_mean(const void* v, float* y, long long planes, long long plane_size, fc_dtype dtype, fc_act act,
                      fc_stream_t stream)
{
    if (!v || !y || !aligned16(v) || !aligned16(y)) return FC_ERR_INVALID_ARG;
    if (planes < 1 || planes > 0x7FFFFFFFLL || plane_size < 1) return FC_ERR_INVALID_ARG;
    if ((dtype != FC_F32 && dtype != FC_BF16) || !valid_act(act)) return FC_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    cudaError_t e = fc::act_mean_launch(v, y, planes, plane_size, dtype == FC_BF16, static_cast<int>(act),
                                        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

fc_status fc_scale_clamp_lse_mish(const float* t, float* y, int M, int N, float scale, float clamp_lo,
                                  float clamp_hi, fc_stream_t stream)
{
    if (!t || !y || !aligned16(t) || !aligned16(y)) return FC_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || !(clamp_lo <= clamp_hi)) return FC_ERR_INVALID_ARG;
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    cudaError_t e = fc::lse_row_launch(t, y, M, N, scale, clamp_lo, clamp_hi, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

size_t fc_workspace_bytes_ex(fc_op op, int n, int cin, int h, int w, int cout, int pad, fc_layout layout,
                             fc_dtype dtype)
{
    if (op != FC_OP_CONV3X3_ACT_POOL && op != FC_OP_CONV3X3_ACT) return 0;
    if (layout != FC_NCHW && layout != FC_NHWC) return 0;
    DeviceState* d = nullptr;
    if (device_state(&d) != FC_OK) return 0;
    if (dtype != FC_F32 && dtype != FC_BF16 && dtype != FC_F32_3XTF32) return 0;
    if (!conv_shape_ok(n, cin, h, w, cout, pad)) return 0;
    fc::ConvPlan plan;
    if (fc::conv_plan(&plan, n, cin, h, w, cout, pad, layout == FC_NHWC, static_cast<int>(dtype),
                      op == FC_OP_CONV3X3_ACT_POOL, d->sm_count) != 0)
        return 0;
    return plan.ws_weights_bytes + plan.ws_pool_bytes;
}

size_t fc_workspace_bytes(fc_op op, int n_or_m, int cin_or_k, int h, int w, int cout_or_nout, fc_dtype dtype)
{
    DeviceState* d = nullptr;
    if (device_state(&d) != FC_OK) return 0;
    if (dtype != FC_F32 && dtype != FC_BF16 && dtype != FC_F32_3XTF32) return 0;
    if (op == FC_OP_CONV3X3_ACT_POOL || op == FC_OP_CONV3X3_ACT) {
        if (h < 3 || w < 3) return 0;
        return fc_workspace_bytes_ex(op, n_or_m, cin_or_k, h, w, cout_or_nout, 0, FC_NCHW, dtype);
    }
    if (op == FC_OP_LINEAR_LSE_MISH) {
        if (n_or_m < 1 || cin_or_k < 1 || cout_or_nout < 1) return 0;
        const bool split = dtype == FC_F32_3XTF32;
        fc::LinearPlan plan;
        if (fc::linear_plan(&plan, n_or_m, cin_or_k, cout_or_nout, dtype == FC_BF16, d->sm_count, split) != 0)
            return 0;
        if (!split) return plan.ws_bytes;
        return ((plan.ws_bytes + 255) & ~static_cast<size_t>(255)) +
               fc::linear_split_bytes(n_or_m, cin_or_k, cout_or_nout);
    }
    return 0;
}

const char* fc_status_string(fc_status s)
{
    switch (s) {
    case FC_OK: return "ok";
    case FC_ERR_INVALID_ARG: return "invalid argument";
    case FC_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case FC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case FC_ERR_CUDA: return "CUDA error";
    case FC_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case FC_ERR_BOUNDS: return "a kernel's index check failed (FC_DEBUG build)";
    default: return "unknown status";
    }
}

fc_status fc_device_status(int clear)
{
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return FC_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FC_ERR_CUDA;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FC_ERR_CUDA;
    }
    return v == 0 ? FC_OK : static_cast<fc_status>(v);
}

fc_status fc_last_device_status(fc_stream_t stream)
{
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    // read on the stream itself: ordered after its enqueued work, and only that stream waits
    if (cudaMemcpyAsync(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FC_ERR_CUDA;
    return v == 0 ? FC_OK : static_cast<fc_status>(v);
}

fc_status fc_selftest_watchdog(unsigned long long budget_cycles, fc_stream_t stream)
{
    DeviceState* d = nullptr;
    fc_status st = device_state(&d);
    if (st != FC_OK) return st;
    if (budget_cycles > 4000000000ull) return FC_ERR_INVALID_ARG;
    cudaError_t e = fc::watchdog_selftest_launch(static_cast<long long>(budget_cycles),
                                                 reinterpret_cast<cudaStream_t>(stream), d->status);
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}

int fc_version(void) { return 100; }

// Testing hook, deliberately not declared in fc.h: sets the spin budget (SM clock cycles) that
// every later launch's bounded waits get, so that a test can make a real operator's waits give
// up.  cycles <= 0 restores the default.  Drains after a wait gives up keep the full budget.
// Returns the previous budget.  Affects every thread of the process; for tests only.
long long fc_testing_set_wait_budget(long long cycles)
{
    return g_wait_budget.exchange(cycles > 0 ? cycles : fc::kWaitBudgetCycles);
}

}  // extern "C"
