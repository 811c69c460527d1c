// elementwise.cu -- the two HBM-bound row kernels around the expert GEMMs:
//   gather_hidden: xs[inv_perm[t*k + j]] = fp16(hidden[t]) for every slot j
//                  of token t, the hidden rows in expert-sorted order as
//                  the gate+up GEMM's token operand (each hidden row is
//                  read once and written to its k sorted positions); it
//                  also zeroes the two GEMMs' split-K tickets;
//   combine:       out[t] = bf16(sum_{j ascending} topk_w[t][j] * y[inv_perm[t*k+j]]),
//                  the fixed-order top-k combine back to token rows (the
//                  "direct/scatter" row writes of "perf(exl3): accelerate
//                  fat-expert prefill - #77", "Engagement and fallback proof").
#include "device_common.cuh"
#include "elementwise.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

// One thread per 16-byte chunk (8 elements) of a token row: one read, one
// conversion, k writes (slots whose id was invalid are skipped).
__global__ void __launch_bounds__(kThreads) gather_hidden_kernel(GatherArgs a, TicketClear z) {
    const int vecs = a.H / 8;
    const int64_t total = (int64_t)a.M * vecs;
    const int64_t i0 = blockIdx.x * (int64_t)kThreads + threadIdx.x;
    // The tickets are used only by the two GEMMs' epilogue warps, and
    // nothing earlier in the call touches them, so they are zeroed before
    // the wait.  An epilogue warp's first ticket update follows its CTA's
    // first accumulator, which follows the producers' griddepcontrol.wait
    // (through the stage and accumulator mbarriers), and that wait returns
    // only once this kernel has completed.  A change that lets the GEMMs
    // touch a ticket before that chain would race with these stores.
    for (int64_t i = i0; i < z.n / 4; i += (int64_t)gridDim.x * kThreads)
        reinterpret_cast<int4 *>(z.tickets)[i] = make_int4(0, 0, 0, 0);
    // The hidden rows are the call's input, complete before its first
    // kernel started, so the first load goes out before waiting for the
    // alignment (inv_perm is read only after the wait).
    uint4 first = make_uint4(0, 0, 0, 0);
    if (i0 < total)
        first = __ldg(reinterpret_cast<const uint4 *>(a.hidden + (size_t)(i0 / vecs) * a.H) +
                      i0 % vecs);
    pdl_wait();
    pdl_trigger();
    bool overflow = false;
    for (int64_t i = i0; i < total; i += (int64_t)gridDim.x * kThreads) {
        const int t = (int)(i / vecs), v = (int)(i % vecs);
        const uint4 in = (i == i0) ? first
                                   : __ldg(reinterpret_cast<const uint4 *>(a.hidden + (size_t)t * a.H) + v);
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(w[j] << 16);
            const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
            overflow |= (fabsf(lo) > 65504.0f && !isinf(lo)) || (fabsf(hi) > 65504.0f && !isinf(hi));
            const __half2 h = __floats2half2_rn(lo, hi);
            o[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
        for (int j = 0; j < a.k; ++j) {
            const int p = __ldg(a.inv_perm + (size_t)t * a.k + j);
            if (p >= 0) reinterpret_cast<uint4 *>(a.xs + (size_t)p * a.H)[v] = ov;
        }
    }
    if (overflow) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 0);
}

// One thread per 4 consecutive outputs of one token row.
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineArgs a) {
    const int quads = a.H / 4;
    const int64_t total = (int64_t)a.M * quads;
    const int64_t i0 = blockIdx.x * (int64_t)kThreads + threadIdx.x;
    // Decode-sized batches (one output quad per thread, at most 8 slots):
    // inv_perm (from the alignment, which had completed before the first
    // GEMM could start) and topk_w (the call's input) are read before
    // waiting for the down GEMM, so only the y loads wait.
    constexpr int kPre = 8;
    if (a.k <= kPre && total <= (int64_t)gridDim.x * kThreads && total <= 16384) {
        int pos[kPre];
        float w[kPre];
        const int t = (int)(i0 / quads), q = (int)(i0 % quads);
        if (i0 < total) {
#pragma unroll
            for (int j = 0; j < kPre; ++j) {
                pos[j] = j < a.k ? __ldg(a.inv_perm + (size_t)t * a.k + j) : -1;
                w[j] = j < a.k ? __ldg(a.topk_w + (size_t)t * a.k + j) : 0.f;
            }
        }
        pdl_wait();
        pdl_trigger();
        if (i0 >= total) return;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
            if (pos[j] < 0) continue;
            const float4 v = __ldg(reinterpret_cast<const float4 *>(a.y + (size_t)pos[j] * a.H) + q);
            acc.x = fmaf(w[j], v.x, acc.x);
            acc.y = fmaf(w[j], v.y, acc.y);
            acc.z = fmaf(w[j], v.z, acc.z);
            acc.w = fmaf(w[j], v.w, acc.w);
        }
        const __nv_bfloat162 b01 = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 b23 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t *>(&b01);
        o.y = *reinterpret_cast<const uint32_t *>(&b23);
        reinterpret_cast<uint2 *>(a.out + (size_t)t * a.H)[q] = o;
        return;
    }
    pdl_wait();
    pdl_trigger();
    for (int64_t i = i0; i < total; i += (int64_t)gridDim.x * kThreads) {
        const int t = (int)(i / quads), q = (int)(i % quads);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.k; ++j) {
            const int pos = __ldg(a.inv_perm + (size_t)t * a.k + j);
            if (pos < 0) continue;
            const float w = __ldg(a.topk_w + (size_t)t * a.k + j);
            const float4 v = __ldg(reinterpret_cast<const float4 *>(a.y + (size_t)pos * a.H) + q);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        const __nv_bfloat162 b01 = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 b23 = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t *>(&b01);
        o.y = *reinterpret_cast<const uint32_t *>(&b23);
        reinterpret_cast<uint2 *>(a.out + (size_t)t * a.H)[q] = o;
    }
}

template <typename Kernel, typename... Args>
cudaError_t launch(Kernel k, int blocks, cudaStream_t s, bool pdl, const Args &...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks > 0 ? blocks : 1);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace

cudaError_t launch_gather_hidden(const GatherArgs &a, const TicketClear &clear, cudaStream_t s,
                                 bool pdl) {
    int64_t blocks = ((int64_t)a.M * (a.H / 8) + kThreads - 1) / kThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch(gather_hidden_kernel, (int)blocks, s, pdl, a, clear);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s, bool pdl) {
    int64_t blocks = ((int64_t)a.M * (a.H / 4) + kThreads - 1) / kThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch(combine_kernel, (int)blocks, s, pdl, a);
}

}  // namespace moe
