// prep_small.cu -- the alignment and the hidden-row gather of a small batch
// (at most kSmallAlignSlots routed slots) in one kernel.
//
// For decode-sized batches the one-CTA alignment kernel spent most of its
// time in fixed costs (a 32 x E shared table, five block barriers, a scan of
// E counts), and the gather kernel then waited for it.  Here every CTA of
// one launch aligns the few slots itself, in shared memory (small_align.cuh:
// the same stable counting sort), and converts its share of the hidden rows
// to fp16 straight into their sorted positions; CTA 0 also writes the
// alignment, both token-tile prefixes and the status word for the GEMMs and
// for inspection.  The hidden loads go out before the alignment is done.
//
// Status: only CTA 0 writes the status word (this kernel starts the call:
// it clears the word, then reports out-of-range ids).  A hidden value beyond
// fp16 range is recorded in this CTA's own overflow slot, which every call
// writes, and the gate+up GEMM reports it after its launch wait.
#include "device_common.cuh"
#include "elementwise.h"
#include "small_align.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
static_assert(kThreads >= kSmallAlignSlots && kThreads % 32 == 0, "one thread per slot");

__device__ __forceinline__ uint32_t half_bits(float v) {
    return (uint32_t)__half_as_ushort(__float2half_rn(v));
}

__global__ void __launch_bounds__(kThreads) align_gather_small_kernel(SmallPrepArgs a) {
    __shared__ SmallAlign sa;
    __shared__ int32_t tp[kSmallAlignSlots + 1], tp2[kSmallAlignSlots + 1];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, g = blockIdx.x, n = a.M * a.k;
    // the next kernel (the gate+up GEMM) may start its set-up; it waits for
    // this one to complete before it reads anything written here
    pdl_trigger();

    // this thread's first 16-byte piece of the hidden rows (the call's input)
    const int vecs = a.H / 8;
    const int64_t work = (int64_t)a.M * vecs, gthreads = (int64_t)G * kThreads;
    const int64_t gi = (int64_t)g * kThreads + tid;
    uint4 first = make_uint4(0, 0, 0, 0);
    if (gi < work)
        first = __ldg(reinterpret_cast<const uint4 *>(a.hidden + (size_t)(gi / vecs) * a.H) + gi % vecs);
    // the split-K tickets of both GEMMs
    for (int64_t i = gi; i < a.clear.n / 4; i += gthreads)
        reinterpret_cast<int4 *>(a.clear.tickets)[i] = make_int4(0, 0, 0, 0);

    small_align(&sa, a.ids, n, a.E);
    if (g == 0) {
        if (warp == 0) small_tile_prefix(&sa, a.nt, tp, lane);
        if (warp == 1) small_tile_prefix(&sa, a.nt2, tp2, lane);
        __syncthreads();
        // counts, offsets and the tile prefixes for every expert (e = E: the
        // totals), perm and inv_perm
        const int n_valid = sa.n_valid, n_act = sa.n_act;
        for (int e = tid; e <= a.E; e += kThreads) {
            const int lo = small_first_at_least(&sa, e);
            a.offsets[e] = sa.act_off[lo];
            a.tile_prefix[e] = tp[lo];
            a.tile_prefix2[e] = tp2[lo];
            if (e < a.E)
                a.counts[e] = (lo < n_act && sa.act_e[lo] == e) ? sa.act_off[lo + 1] - sa.act_off[lo] : 0;
        }
        for (int p = tid; p < n; p += kThreads) {
            a.perm[p] = p < n_valid ? sa.perm[p] : -1;
            if (a.inv_perm) a.inv_perm[p] = sa.inv[p];
        }
        if (tid == 0) {
            a.ctrl->status = 0;
            a.ctrl->detail = 0;
            a.ctrl->n_invalid = n - n_valid;
            if (n_valid < n) set_status(a.ctrl, MOE_ERR_DEVICE_BAD_EXPERT_ID, sa.raw[sa.first_bad_slot]);
        }
    }

    // hidden rows -> fp16, each piece written to the sorted rows of its
    // token's valid slots
    bool overflow = false;
    for (int64_t i = gi; i < work; i += gthreads) {
        const int t = (int)(i / vecs), v = (int)(i % vecs);
        const uint4 in = (i == gi) ? first
                                   : __ldg(reinterpret_cast<const uint4 *>(a.hidden + (size_t)t * a.H) + v);
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16);
            const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
            overflow |= (fabsf(lo) > 65504.0f && !isinf(lo)) || (fabsf(hi) > 65504.0f && !isinf(hi));
            o[j] = half_bits(lo) | (half_bits(hi) << 16);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        for (int j = 0; j < a.k; ++j) {
            const int p = sa.inv[t * a.k + j];
            if (p >= 0) reinterpret_cast<uint4 *>(a.xs + (size_t)p * a.H)[v] = ov;
        }
    }
    const int any = __syncthreads_or(overflow);
    if (tid == 0) a.ovf[g] = any;
}

}  // namespace

int small_prep_grid(int M, int H) {
    const int64_t blocks = ((int64_t)M * (H / 8) + kThreads - 1) / kThreads;
    return (int)(blocks < 1 ? 1 : (blocks > kSmallPrepMaxGrid ? kSmallPrepMaxGrid : blocks));
}

cudaError_t launch_align_gather_small(const SmallPrepArgs &a, int grid, cudaStream_t s) {
    // The first kernel of a call: ordinary stream order (no early launch),
    // so it never overlaps the previous call's kernels on the same workspace.
    align_gather_small_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
