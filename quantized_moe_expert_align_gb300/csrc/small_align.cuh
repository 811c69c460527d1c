// small_align.cuh -- the stable counting sort by expert of at most
// kSmallAlignSlots routed slots, computed by one CTA in its shared memory.
//
// The same result as the alignment kernels (align.cu): slot f = t*k + j of
// expert e lands at offsets[e] + (number of earlier slots of e), slots with
// an id outside [0, E) are left out.  For so few slots each slot simply
// ranks itself against all the others, so every CTA of a kernel can align
// the batch on its own, with no global memory round trip and no kernel of
// its own.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kSmallAlignSlots = 128;

struct SmallAlign {
    int first_bad_slot;          // lowest slot with an id outside [0, E), else kSmallAlignSlots
    int warp_starts[4];
    int n_valid, n_act;          // placed slots, active experts
    int32_t raw[kSmallAlignSlots];   // the slot's id as given
    int32_t sid[kSmallAlignSlots];   // the slot's id, or -1 outside [0, E)
    int32_t perm[kSmallAlignSlots];  // sorted row -> slot
    int32_t inv[kSmallAlignSlots];   // slot -> sorted row, or -1
    int32_t act_e[kSmallAlignSlots + 1];    // active experts, ascending
    int32_t act_off[kSmallAlignSlots + 1];  // their first sorted row; act_off[n_act] = n_valid
};

// Every thread of the block calls it (at least kSmallAlignSlots threads, in
// whole warps; n <= kSmallAlignSlots).  Returns after a block barrier with
// *sa filled in.
__device__ __forceinline__ void small_align(SmallAlign *sa, const int32_t *ids, int n, int E) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) sa->first_bad_slot = kSmallAlignSlots;
    int id = -1;
    if (tid < n) {
        const int raw = __ldg(ids + tid);
        id = (raw >= 0 && raw < E) ? raw : -1;
        sa->raw[tid] = raw;
        sa->sid[tid] = id;
    }
    const int n_valid = __syncthreads_count(tid < n && id >= 0);
    if (tid < n) {
        if (id >= 0) {
            // rank: slots of lower experts, then earlier slots of this one
            int pos = 0;
            for (int f = 0; f < n; ++f) {
                const int o = sa->sid[f];
                pos += (o >= 0) & ((o < id) | ((o == id) & (f < tid)));
            }
            sa->inv[tid] = pos;
            sa->perm[pos] = tid;
        } else {
            sa->inv[tid] = -1;
            atomicMin(&sa->first_bad_slot, tid);
        }
    }
    __syncthreads();
    // active experts: the sorted rows where the expert changes, ranked by a
    // ballot over the first four warps
    bool start = false;
    int e_here = -1;
    if (tid < n_valid) {
        e_here = sa->sid[sa->perm[tid]];
        start = (tid == 0) || (sa->sid[sa->perm[tid - 1]] != e_here);
    }
    unsigned ballot = 0;
    if (warp < 4) {
        ballot = __ballot_sync(0xffffffffu, start);
        if (lane == 0) sa->warp_starts[warp] = __popc(ballot);
    }
    __syncthreads();
    const int n_act = sa->warp_starts[0] + sa->warp_starts[1] + sa->warp_starts[2] + sa->warp_starts[3];
    if (warp < 4) {
        int rank = __popc(ballot & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) rank += sa->warp_starts[w];
        if (start) {
            sa->act_e[rank] = e_here;
            sa->act_off[rank] = tid;
        }
    }
    if (tid == 0) {
        sa->act_off[n_act] = n_valid;
        sa->n_valid = n_valid;
        sa->n_act = n_act;
    }
    __syncthreads();
}

// Exclusive prefix, over the active experts, of their token tiles of `nt`
// rows: tp[a] for a < n_act and tp[n_act] = the total, which every lane
// returns.  Executed by one whole warp (four experts per lane).
__device__ __forceinline__ int small_tile_prefix(const SmallAlign *sa, int nt, int32_t *tp, int lane) {
    const int n_act = sa->n_act;
    int cnt[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ai = lane * 4 + i;
        cnt[i] = ai < n_act ? (sa->act_off[ai + 1] - sa->act_off[ai] + nt - 1) / nt : 0;
        sum += cnt[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int ai = lane * 4 + i;
        if (ai < n_act) tp[ai] = run;
        run += cnt[i];
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) tp[n_act] = total;
    return total;
}

// First active index whose expert is >= e (n_act if none): where expert e's
// rows and tiles start in the prefixes above (e = E gives the totals).
__device__ __forceinline__ int small_first_at_least(const SmallAlign *sa, int e) {
    int lo = 0, hi = sa->n_act;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (sa->act_e[mid] < e) lo = mid + 1; else hi = mid;
    }
    return lo;
}

}  // namespace moe
