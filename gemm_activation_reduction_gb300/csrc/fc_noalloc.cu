// fc_noalloc.cu -- fc_linear_lse_mish_noalloc: the Linear + logsumexp + x*mish(x)
// operator for callers that cannot allocate device memory.
//
// fc_linear_lse_mish needs caller-provided scratch for its per-tile
// (max, sum-exp) pairs.  Some callers have no way to provide it: code whose
// device memory is owned by somebody else's allocator or a fixed budget,
// plain C hosts with no allocator of their own, or loops where a cudaMalloc
// (which can synchronize the whole device) is not acceptable.  This entry
// point keeps that scratch in a file-scope device array instead, so a call
// needs only its inputs and outputs and performs no allocation.
#include "../../include/fc.h"
#include "fc_internal.h"

#include <atomic>
#include <mutex>

namespace {

// 1 MiB of scratch, resident on every device that loads the library until the
// process exits: room for 131072 (max, sum-exp) pairs of 8 bytes, one per row and
// column tile, i.e. M * ceil(Nout / bn) <= 131072 with bn the planned tile width
// (128 to 256 columns; M = 1024 with Nout = 8192 needs 37 tiles of 224).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch per device; only a successful look-up is kept, so a
// failed first call (for instance one made during a stream capture) is retried on the next.
std::atomic<void*> g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fc_status fc_linear_lse_mish_noalloc(const void* x, const void* W, const void* b, float* y, int M, int K,
                                                int Nout, float scale, float clamp_lo, float clamp_hi,
                                                fc_stream_t stream)
{
    if (!x || !W || !b || !y) return FC_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W) || !aligned16(b) || !aligned16(y)) return FC_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || Nout < 1) return FC_ERR_INVALID_ARG;
    if (!(clamp_lo <= clamp_hi)) return FC_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FC_ERR_CUDA;
    // Host code cannot use g_noalloc_scratch's name as a device address: look the
    // address up once per device, with that device current (it is: this call runs
    // on the caller's current device).
    void* scratch = g_scratch[dev].load(std::memory_order_acquire);
    if (scratch == nullptr) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        scratch = g_scratch[dev].load(std::memory_order_relaxed);
        if (scratch == nullptr) {
            if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || scratch == nullptr)
                return FC_ERR_CUDA;
            g_scratch[dev].store(scratch, std::memory_order_release);
        }
    }
    int sm_count = 0;
    int* status = nullptr;
    if (fc::current_device_info(&sm_count, &status) != cudaSuccess) return FC_ERR_CUDA;
    fc::LinearPlan plan;
    if (fc::linear_plan(&plan, M, K, Nout, 0, sm_count) != 0) return FC_ERR_UNSUPPORTED;
    if (plan.ws_bytes > kNoAllocScratchBytes) return FC_ERR_UNSUPPORTED;
    // Every (max, sum-exp) pair the combine kernel reads is written by the main kernel of the
    // same call, so the array needs no clearing between calls -- unless a bounded wait of that
    // kernel gives up, in which case the combine writes NaN instead of reading the array.
    cudaError_t e = fc::linear_launch(plan, static_cast<const float*>(x), static_cast<const float*>(W),
                                      static_cast<const float*>(b), y, scale, clamp_lo, clamp_hi, scratch,
                                      reinterpret_cast<cudaStream_t>(stream), status, fc::wait_budget());
    return e == cudaSuccess ? FC_OK : FC_ERR_CUDA;
}
