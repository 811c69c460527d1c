// static_scratch.cu -- the layer forward for callers that cannot allocate
// device memory.
//
// Some callers have no way to get a device buffer for the forward's
// workspace: code that runs inside a host framework which owns every device
// allocation and hands out only the tensors it manages, or a latency-bound
// decode loop where a cudaMalloc would synchronise the device.  For them the
// workspace lives in one file-scope device array of fixed size, reserved on
// every GPU that loads this library until the process exits.
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = MOE_W4A16_STATIC_SCRATCH_BYTES;  // 16 MiB
constexpr int kMaxDevices = 64;

// In host code this name is only a stand-in for the symbol; its device
// address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_lock;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up once per
// device, with that device current).
moe_status_t scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MOE_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_w4a16_forward_static(const uint16_t *hidden, const int32_t *topk_ids,
                                                 const float *topk_w, const void *w13,
                                                 const void *w2, uint16_t *out, int M, int k, int E, int H, int I,
                                                 moe_stream_t stream) {
    const size_t need = moe_w4a16_workspace_size(M, k, E, H, I);
    if (need == 0) return MOE_ERR_INVALID_ARG;
    if (need > moe::kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    const moe_status_t st = moe::scratch_address(&scratch);
    if (st != MOE_OK) return st;
    return moe::forward_on_scratch(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I,
                                   scratch, moe::kStaticScratchBytes, stream);
}
