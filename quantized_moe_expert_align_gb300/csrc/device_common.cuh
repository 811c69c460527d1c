// device_common.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

// Record the first device-side error of the current call; never traps.
__device__ __forceinline__ void set_status(Ctrl *ctrl, int code, int detail) {
    if (atomicCAS(&ctrl->status, 0, code) == 0) atomicExch(&ctrl->detail, detail);
}

// Programmatic dependent launch: wait until the previous kernel in the stream
// has completed and its writes are visible.  Every block of every kernel
// launched with the programmatic-serialization attribute executes this
// before it reads a predecessor's output and before it exits, so completion
// of a kernel implies completion of all kernels before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to be scheduled early.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

// Validate a prepacked buffer header against the expected geometry.
__device__ __forceinline__ bool header_ok(const uint8_t *buf, uint32_t kind, int E, int N, int K) {
    const PackHeader *h = reinterpret_cast<const PackHeader *>(buf);
    return h->magic == kPackMagic && h->version == kPackVersion && h->kind == kind &&
           h->block_bytes == (uint32_t)kBlockBytes && h->E == E && h->N == N && h->K == K &&
           h->group == kGroup && h->status == MOE_OK;
}

// Index of the expert owning tile `tile`: the largest e with prefix[e] <= tile
// (prefix is non-decreasing, prefix[0] = 0, tile < prefix[E]).
__device__ __forceinline__ int find_segment(const int32_t *prefix, int E, int tile) {
    int lo = 0, hi = E;  // invariant: prefix[lo] <= tile < prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(prefix + mid) <= tile) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace moe
