// route.cu -- router front-end over many tokens: one warp per token (the
// routine of route.cuh), eight tokens per CTA, for batches too large for the
// single-CTA alignment kernel to route by itself.
#include "route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) route_kernel(RouteArgs a) {
    const int lane = threadIdx.x & 31;
    const int vpl = route_vpl(a.E);
    for (int t = blockIdx.x * kWarps + (threadIdx.x >> 5); t < a.M; t += gridDim.x * kWarps) {
        const bool bad = route_row_any<kRouteMaxVpl>(vpl, a.logits + (size_t)t * a.E, a.E, a.k, lane,
                                       a.ids + (size_t)t * a.k, a.w + (size_t)t * a.k);
        if (bad && lane == 0) set_status(a.ctrl, MOE_ERR_DEVICE_BAD_LOGIT, t);
    }
}

}  // namespace

cudaError_t launch_route(const RouteArgs &a, cudaStream_t s) {
    int64_t blocks = ((int64_t)a.M + kWarps - 1) / kWarps;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    route_kernel<<<(int)blocks, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
