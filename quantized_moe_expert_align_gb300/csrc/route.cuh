// route.cuh -- router front-end on one warp per token: the k experts of
// largest logit (lower index first on ties) and their softmax weights
// renormalised over the k, from one row of fp32 router logits.
//
// The pages leave the router open; the layer's inputs are defined as a
// softmax over all E logits, its top k, weights renormalised to sum 1.  The
// softmax is monotone, so the order is taken on the logits, and
// p_j / sum_{i<k} p_i = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0) with l_0
// the largest logit: the normaliser over all E cancels and only the k
// selected logits are exponentiated.
//
// Order of logits (a total order, as 32-bit keys, larger first): numbers by
// value with -0 == +0, then NaN; equal keys go to the lower expert index.  A
// row holding a NaN or +inf gets zero weights and is reported; -inf logits
// get weight 0; a row of only -inf gets zero weights.
#pragma once

#include "device_common.cuh"

namespace moe {

// Largest number of values one lane holds: E <= 32 * kRouteMaxVpl.  The
// alignment kernel (1024 threads, at most 64 registers each) routes only up
// to kAlignRouteMaxVpl values per lane.
constexpr int kRouteMaxVpl = 32;
constexpr int kAlignRouteMaxVpl = 16;

// Key of a logit: larger key ranks first.  Numbers map monotonically onto
// [0x007FFFFF (-inf), 0xFF800000 (+inf)], both zeros onto 0x80000000, NaN
// onto 1; 0 is left for "taken" and for padding lanes.
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v != v) return 1u;
    const uint32_t b = (v == 0.0f) ? 0u : __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of logit_key for keys > 1 (NaN for key 1).
__device__ __forceinline__ float key_logit(uint32_t key) {
    if (key <= 1u) return __uint_as_float(0x7FC00000u);
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Routes one token.  All 32 lanes of the warp call it with the same row;
// lane j (and j + 32) writes slot j (j + 32) of ids and w.  VPL logits per
// lane (lane + 32 i), VPL * 32 >= E.  Returns true (on every lane) when the
// row holds a NaN or +inf.
template <int VPL>
__device__ __forceinline__ bool route_row(const float *row, int E, int k, int lane, int32_t *ids,
                                          float *w) {
    uint32_t key[VPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0u;
        if (e < E) {
            const float v = row[e];
            bad |= (v != v) || (v == INFINITY);
            key[i] = logit_key(v);
        }
    }
    bad = __any_sync(0xffffffffu, bad);

    // k rounds of a warp arg-max over (key, -index): the largest key of the
    // warp (one warp reduction), then the lowest index among the lanes that
    // hold it (another); the winner is cleared in its lane.  Slot j ends up
    // in lane j % 32 (register a or b).
    float la = 0.f, lb = 0.f;
    int ia = -1, ib = -1;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (key[i] > bk) {  // ascending e inside the lane: strict keeps the lower index
                bk = key[i];
                be = lane + 32 * i;
            }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        be = __reduce_min_sync(0xffffffffu, bk == mk ? be : 0x7FFFFFFF);
        bk = mk;
        // (a select per register: an indexed store would put key[] in
        // local memory)
#pragma unroll
        for (int i = 0; i < VPL; ++i) key[i] = (lane + 32 * i == be) ? 0u : key[i];
        if (j == lane) {
            ia = be;
            la = key_logit(bk);
        } else if (j == lane + 32) {
            ib = be;
            lb = key_logit(bk);
        }
    }

    // weights: exp(l_j - l_0) over their sum (every lane ends with the same
    // sum: the butterfly adds the same two values on both partners)
    const float l0 = __shfl_sync(0xffffffffu, la, 0);
    const bool ha = lane < k, hb = lane + 32 < k;
    const float ea = (ha && !bad && la > -INFINITY) ? expf(la - l0) : 0.f;
    const float eb = (hb && !bad && lb > -INFINITY) ? expf(lb - l0) : 0.f;
    float sum = ea + eb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (ha) {
        ids[lane] = ia;
        w[lane] = sum > 0.f ? ea / sum : 0.f;
    }
    if (hb) {
        ids[lane + 32] = ib;
        w[lane + 32] = sum > 0.f ? eb / sum : 0.f;
    }
    return bad;
}

// Lane count class for E: the smallest supported VPL with 32 * VPL >= E.
__host__ __device__ inline int route_vpl(int E) {
    const int need = (E + 31) / 32;
    return need <= 2 ? need : need <= 4 ? 4 : need <= 8 ? 8 : need <= 12 ? 12 : need <= 16 ? 16
         : need <= 24 ? 24 : need <= 32 ? 32 : 0;
}

// route_row for the VPL class of E (one branch per class, uniform per
// warp), for classes up to MAXV.
template <int MAXV>
__device__ __forceinline__ bool route_row_any(int vpl, const float *row, int E, int k, int lane,
                                              int32_t *ids, float *w) {
    switch (vpl) {
        case 1: return route_row<1>(row, E, k, lane, ids, w);
        case 2: return route_row<2>(row, E, k, lane, ids, w);
        case 4: return route_row<4>(row, E, k, lane, ids, w);
        case 8: return route_row<8>(row, E, k, lane, ids, w);
        case 12: return route_row<12>(row, E, k, lane, ids, w);
        default:
            if (MAXV <= 16 || vpl == 16) return route_row<(MAXV < 16 ? MAXV : 16)>(row, E, k, lane, ids, w);
            if (vpl == 24) return route_row<(MAXV < 24 ? MAXV : 24)>(row, E, k, lane, ids, w);
            return route_row<MAXV>(row, E, k, lane, ids, w);
    }
}

}  // namespace moe
