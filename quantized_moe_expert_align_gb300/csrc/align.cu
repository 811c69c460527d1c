// align.cu -- top-k routed token alignment: per-expert histogram, warp-shuffle
// prefix scan, stable permutation.
//
// "perf(exl3): accelerate fat-expert prefill - #77" ("Rollout") groups routed
// tokens by expert ("sorted routing"); "DeepSeek-V4.1-Flash-EXL3 ... Detailed
// results" ("Nsight Compute on the stock kernel") found the serial scan over
// 384 expert counts to be the hottest spot of decode.  Here the scan is a
// two-level warp-shuffle scan over one count per thread.
//
// One CTA of 1024 threads (batches of more than kAlignLargeSlots slots: the
// same algorithm over kAlignSegs CTAs, below).  The M*k flat slots are cut
// into 32 contiguous segments, one per warp.  Each warp builds its segment's histogram with
// __match_any_sync (no atomics decide any order), the block turns the 32 x E
// table into per-(warp, expert) starting positions, and each warp walks its
// segment again in order, so the permutation is the stable counting sort by
// expert of the flat index f = t*k + j.
#include "device_common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Exclusive scan of one int per thread over the whole block; returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int *warp_buf, int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_buf[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = warp_buf[lane];
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        warp_buf[lane] = incl - s;
        if (lane == 31) warp_buf[32] = incl;
    }
    __syncthreads();
    int excl = warp_buf[w] + x - v;
    *total = warp_buf[32];
    __syncthreads();
    return excl;
}

// Per-warp histogram of the flat slots [lo, hi) into row[E] (the warp's
// row of the table); out-of-range ids are counted, not placed.
__device__ __forceinline__ void warp_histogram(const AlignArgs &a, int32_t *row, int lo, int hi,
                                               int lane, int &invalid, int &first_bad) {
    for (int base = lo; base < hi; base += 32) {
        const int f = base + lane;
        int id = -1;
        if (f < hi) {
            id = a.ids[f];
            if (id < 0 || id >= a.E) {
                if (invalid == 0) first_bad = id;
                ++invalid;
                id = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && lane == __ffs(peers) - 1) row[id] += __popc(peers);
        __syncwarp();
    }
}

// Stable placement of the flat slots [lo, hi), walked in order; row[e] holds
// the sorted position of the warp's next slot of expert e.
__device__ __forceinline__ void warp_place(const AlignArgs &a, int32_t *row, int lo, int hi,
                                           int lane) {
    for (int base = lo; base < hi; base += 32) {
        const int f = base + lane;
        int id = -1;
        if (f < hi) {
            id = a.ids[f];
            if (id < 0 || id >= a.E) id = -1;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        int pos = -1;
        if (id >= 0) pos = row[id] + __popc(peers & ((1u << lane) - 1u));
        __syncwarp();
        if (id >= 0 && lane == __ffs(peers) - 1) row[id] += __popc(peers);
        __syncwarp();
        if (f < hi) {
            if (pos >= 0) a.perm[pos] = f;
            if (a.inv_perm) a.inv_perm[f] = pos;
        }
    }
}

// From each expert's count c (thread e < E): counts, offsets (the
// warp-shuffle scan), both token-tile prefixes, and the zeroed split-K
// tickets.  Returns the thread's offset; *total = offsets[E].
__device__ int write_prefixes(const AlignArgs &a, int c, int *warp_buf, int *total) {
    const int tid = threadIdx.x, E = a.E;
    const int off = block_exclusive_scan(c, warp_buf, total);
    if (tid < E) {
        a.counts[tid] = c;
        a.offsets[tid] = off;
    }
    if (tid == 0) a.offsets[E] = *total;
    if (a.token_tile > 0) {
        const int tiles = (tid < E) ? (c + a.token_tile - 1) / a.token_tile : 0;
        int ttotal = 0;
        const int toff = block_exclusive_scan(tiles, warp_buf, &ttotal);
        if (tid < E) a.tile_prefix[tid] = toff;
        if (tid == 0) a.tile_prefix[E] = ttotal;
        const int tiles2 = (tid < E) ? (c + a.token_tile2 - 1) / a.token_tile2 : 0;
        int ttotal2 = 0;
        const int toff2 = block_exclusive_scan(tiles2, warp_buf, &ttotal2);
        if (tid < E) a.tile_prefix2[tid] = toff2;
        if (tid == 0) a.tile_prefix2[E] = ttotal2;
        if (a.tickets) {
            for (int i = tid; i < ttotal * a.r1; i += kThreads) a.tickets[i] = 0;
            for (int i = tid; i < ttotal2 * a.r2; i += kThreads) a.tickets[a.off2 + i] = 0;
        }
    }
    return off;
}

__global__ void __launch_bounds__(kThreads, 1) align_kernel(AlignArgs a) {
    extern __shared__ int32_t table[];  // [kWarps][E]
    __shared__ int warp_buf[33];
    __shared__ int s_invalid;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int E = a.E, n = a.n;

    if (tid == 0) {
        if (a.reset_status) {
            a.ctrl->status = 0;
            a.ctrl->detail = 0;
        }
        s_invalid = 0;
    }
    for (int i = tid; i < kWarps * E; i += kThreads) table[i] = 0;
    __syncthreads();
    pdl_trigger();

    // Optional router front-end: warp w routes tokens w, w + 32, ...; the ids
    // it writes are read back below by other warps of this CTA, after the
    // barrier, with ordinary (coherent) loads.
    if (a.logits) {
        const int vpl = route_vpl(E);
        for (int t = w; t < a.route_M; t += kWarps) {
            const bool bad = route_row_any<kAlignRouteMaxVpl>(vpl, a.logits + (size_t)t * E, E, a.route_k, lane,
                                           a.route_ids + (size_t)t * a.route_k,
                                           a.route_w + (size_t)t * a.route_k);
            if (bad && lane == 0) set_status(a.ctrl, MOE_ERR_DEVICE_BAD_LOGIT, t);
        }
        __syncthreads();
    }

    const int per = (n + kWarps - 1) / kWarps;
    const int seg_lo = min(n, w * per), seg_hi = min(n, seg_lo + per);
    int32_t *row = table + w * E;

    // Phase A: per-warp histogram of its segment.
    int my_invalid = 0, first_bad = 0;
    warp_histogram(a, row, seg_lo, seg_hi, lane, my_invalid, first_bad);
    if (my_invalid) {
        atomicAdd(&s_invalid, my_invalid);
        set_status(a.ctrl, MOE_ERR_DEVICE_BAD_EXPERT_ID, first_bad);
    }
    __syncthreads();

    // Counts, then the warp-shuffle scan into offsets and tile prefixes.
    int c = 0;
    if (tid < E) {
#pragma unroll 8
        for (int ww = 0; ww < kWarps; ++ww) c += table[ww * E + tid];
    }
    int total = 0;
    const int off = write_prefixes(a, c, warp_buf, &total);
    if (tid < E) {
        // Phase B: starting position of (warp, expert) = offsets[e] + the
        // expert's slots in earlier segments.
        int run = off;
        for (int ww = 0; ww < kWarps; ++ww) {
            int t = table[ww * E + tid];
            table[ww * E + tid] = run;
            run += t;
        }
    }
    __syncthreads();

    // Phase C: stable placement, walking each segment in order.
    warp_place(a, row, seg_lo, seg_hi, lane);
    __syncthreads();
    for (int p = total + tid; p < n; p += kThreads) a.perm[p] = -1;
    if (tid == 0) a.ctrl->n_invalid = s_invalid;
}

// ---- large batches: the same stable counting sort over kAlignSegs CTAs.
// The slots are cut into kAlignSegs contiguous segments (one per CTA), each
// into 32 warp segments as above.  (1) Each CTA counts its segment per
// expert; (2) one CTA turns the [E][kAlignSegs] counts into, per expert, the
// exclusive prefix over segments, plus counts, offsets and tile prefixes;
// (3) each CTA places its segment from offsets[e] + that prefix.  Every
// slot lands where the single-CTA kernel puts it.

__device__ __forceinline__ void cta_segment(int n, int b, int &lo, int &hi) {
    const int per = (n + kAlignSegs - 1) / kAlignSegs;
    lo = min(n, b * per);
    hi = min(n, lo + per);
}

__global__ void __launch_bounds__(kThreads) align_count_kernel(AlignArgs a, int32_t *seg_counts) {
    extern __shared__ int32_t table[];  // [kWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = a.E;
    for (int i = tid; i < kWarps * E; i += kThreads) table[i] = 0;
    __syncthreads();
    pdl_trigger();
    int lo, hi;
    cta_segment(a.n, blockIdx.x, lo, hi);
    const int per = (hi - lo + kWarps - 1) / kWarps;
    const int wlo = min(hi, lo + w * per), whi = min(hi, wlo + per);
    int invalid = 0, first_bad = 0;
    warp_histogram(a, table + w * E, wlo, whi, lane, invalid, first_bad);
    if (invalid) {
        atomicAdd(&a.ctrl->n_invalid, invalid);
        set_status(a.ctrl, MOE_ERR_DEVICE_BAD_EXPERT_ID, first_bad);
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int c = 0;
#pragma unroll 8
        for (int ww = 0; ww < kWarps; ++ww) c += table[ww * E + e];
        seg_counts[e * kAlignSegs + blockIdx.x] = c;
    }
}

__global__ void __launch_bounds__(kThreads, 1) align_scan_kernel(AlignArgs a,
                                                                 const int32_t *seg_counts,
                                                                 int32_t *seg_base) {
    __shared__ int warp_buf[33];
    __shared__ int32_t s_count[1024];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = a.E;
    pdl_wait();
    pdl_trigger();
    static_assert(kAlignSegs == 32, "one segment per lane");
    // warp w scans experts w, w + 32, ... over their kAlignSegs segment
    // counts, one per lane, 8 experts' loads in flight at a time
    constexpr int kBatch = 8;
    for (int e0 = w; e0 < E; e0 += kBatch * kWarps) {
        int v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = e0 + i * kWarps;
            v[i] = e < E ? seg_counts[e * kAlignSegs + lane] : 0;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = e0 + i * kWarps;
            int x = v[i];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (e < E) {
                seg_base[e * kAlignSegs + lane] = x - v[i];
                if (lane == 31) s_count[e] = x;
            }
        }
    }
    __syncthreads();
    const int c = tid < E ? s_count[tid] : 0;
    int total = 0;
    write_prefixes(a, c, warp_buf, &total);
    for (int p = total + tid; p < a.n; p += kThreads) a.perm[p] = -1;
}

__global__ void __launch_bounds__(kThreads) align_place_kernel(AlignArgs a,
                                                               const int32_t *seg_base) {
    extern __shared__ int32_t table[];  // [kWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, E = a.E;
    for (int i = tid; i < kWarps * E; i += kThreads) table[i] = 0;
    __syncthreads();
    int lo, hi;
    cta_segment(a.n, blockIdx.x, lo, hi);
    const int per = (hi - lo + kWarps - 1) / kWarps;
    const int wlo = min(hi, lo + w * per), whi = min(hi, wlo + per);
    int invalid = 0, first_bad = 0;
    warp_histogram(a, table + w * E, wlo, whi, lane, invalid, first_bad);
    pdl_wait();  // offsets and segment bases come from the scan kernel
    pdl_trigger();
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        int run = a.offsets[e] + seg_base[e * kAlignSegs + blockIdx.x];
        for (int ww = 0; ww < kWarps; ++ww) {
            const int t = table[ww * E + e];
            table[ww * E + e] = run;
            run += t;
        }
    }
    __syncthreads();
    warp_place(a, table + w * E, wlo, whi, lane);
}

template <typename... Args>
cudaError_t launch_pdl(void (*k)(Args...), int blocks, size_t smem, cudaStream_t s, bool pdl,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace

cudaError_t launch_align(const AlignArgs &a, cudaStream_t s) {
    // The first kernel of a call: ordinary stream order (no early launch), so
    // it never overlaps the previous call's kernels on the same workspace.
    const size_t smem = (size_t)kWarps * a.E * sizeof(int32_t);
    if (a.seg_counts) {
        // large batch (the caller has cleared the status word and routed)
        cudaError_t err = cudaFuncSetAttribute(align_count_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(align_place_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        align_count_kernel<<<kAlignSegs, kThreads, smem, s>>>(a, a.seg_counts);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if ((err = launch_pdl(align_scan_kernel, 1, 0, s, true, a,
                              static_cast<const int32_t *>(a.seg_counts), a.seg_base)) !=
            cudaSuccess)
            return err;
        return launch_pdl(align_place_kernel, kAlignSegs, smem, s, true, a,
                          static_cast<const int32_t *>(a.seg_base));
    }
    cudaError_t err = cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    align_kernel<<<1, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
