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

// Exclusive scan of three ints per thread over the whole block at once (the
// counts and the two token-tile counts): one warp-shuffle pass, then warps
// 0..2 scan the 32 warp totals of x, y and z.  Returns the thread's
// exclusive prefixes and writes the block totals to *total.  buf holds
// 3 * 33 ints; the block has exactly 32 warps.
__device__ int3 block_exclusive_scan3(int3 v, int *buf, int3 *total) {
    static_assert(kWarps == 32, "warps 0..2 scan one warp total per lane");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int3 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yx = __shfl_up_sync(0xffffffffu, x.x, o);
        const int yy = __shfl_up_sync(0xffffffffu, x.y, o);
        const int yz = __shfl_up_sync(0xffffffffu, x.z, o);
        if (lane >= o) {
            x.x += yx;
            x.y += yy;
            x.z += yz;
        }
    }
    if (lane == 31) {
        buf[w] = x.x;
        buf[33 + w] = x.y;
        buf[66 + w] = x.z;
    }
    __syncthreads();
    if (w < 3) {  // warps 0, 1, 2 scan the warp totals of x, y, z
        const int s = buf[33 * w + lane];
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        buf[33 * w + lane] = incl - s;
        if (lane == 31) buf[33 * w + 32] = incl;
    }
    __syncthreads();
    const int3 excl = make_int3(buf[w] + x.x - v.x, buf[33 + w] + x.y - v.y,
                                buf[66 + w] + x.z - v.z);
    *total = make_int3(buf[32], buf[65], buf[98]);
    __syncthreads();
    return excl;
}

// From each expert's count c (thread e < E): counts, offsets (the
// warp-shuffle scan) and both token-tile prefixes (scanned together with the
// counts).  Returns the thread's offset; *total = offsets[E].
__device__ int write_prefixes(const AlignArgs &a, int c, int *scan_buf, int *total) {
    const int tid = threadIdx.x, E = a.E;
    const bool tiled = a.token_tile > 0;
    int3 v = make_int3(c, 0, 0);
    if (tiled && tid < E) {
        v.y = (c + a.token_tile - 1) / a.token_tile;
        v.z = (c + a.token_tile2 - 1) / a.token_tile2;
    }
    int3 tot;
    const int3 ex = block_exclusive_scan3(v, scan_buf, &tot);
    *total = tot.x;
    if (tid < E) {
        a.counts[tid] = c;
        a.offsets[tid] = ex.x;
    }
    if (tid == 0) a.offsets[E] = tot.x;
    if (tiled) {
        if (tid < E) {
            a.tile_prefix[tid] = ex.y;
            a.tile_prefix2[tid] = ex.z;
        }
        if (tid == 0) {
            a.tile_prefix[E] = tot.y;
            a.tile_prefix2[E] = tot.z;
        }
    }
    return ex.x;
}

__global__ void __launch_bounds__(kThreads, 1) align_kernel(AlignArgs a) {
    extern __shared__ int32_t table[];  // [kWarps][E]
    __shared__ int scan_buf[3 * 33];
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
    const int off = write_prefixes(a, c, scan_buf, &total);
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
    __shared__ int scan_buf[3 * 33];
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
    write_prefixes(a, c, scan_buf, &total);
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
