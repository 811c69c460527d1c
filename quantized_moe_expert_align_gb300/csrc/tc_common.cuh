// tc_common.cuh -- device pieces shared by the tensor-core expert GEMM
// (gemm_tc.cu) and the fused small-batch layer kernel (decode.cu): bounded
// mbarrier waits, the stream-K partition, the INT4 -> fp16 dequantisation of
// one code word and the SiLU(gate)*up epilogue of one accumulator pair.
#pragma once

#include <cuda_fp16.h>

#include "device_common.cuh"
#include "sm100.cuh"

namespace moe {
namespace tc {

using namespace sm100;

constexpr long long kWaitCycles = 1ll << 31;  // bounded waits give up after ~1-2 s
constexpr uint32_t kSleepNs = 20000;          // longest sleep of one poll of a wait

// Bounded wait that also gives up as soon as another role has aborted.  The
// limit is measured with the SM's own cycle counter, which never runs
// backwards.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int *abort, Ctrl *ctrl,
                                         int who) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
        if (*(volatile int *)abort) return false;
        if (clock64() - t0 > kWaitCycles) {
            atomicExch(abort, 1);
            set_status(ctrl, MOE_ERR_DEVICE_TIMEOUT, who);
            return false;
        }
    }
}

// All lanes of a warp wait; the warp goes on only if every lane saw the
// phase complete, so later warp-wide (.sync.aligned) instructions stay
// convergent even when an abort races with completion.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, int *abort,
                                              Ctrl *ctrl, int who) {
    const bool ok = wait_bar(bar, parity, abort, ctrl, who);
    return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (used while winding down).
__device__ __forceinline__ bool wait_bar_final(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Stream-K partition of W chunk-units over G CTAs.
__device__ __forceinline__ int64_t range_begin(int g, int64_t W, int G) {
    return (int64_t)g * W / G;
}
__device__ __forceinline__ int unit_owner(int64_t u, int64_t W, int G) {
    return (int)(((u + 1) * (int64_t)G - 1) / W);
}
// Number of CTAs whose (non-empty) ranges cover units [u0, u1].
__device__ __forceinline__ int contributors(int64_t u0, int64_t u1, int64_t W, int G) {
    int n = 0;
    for (int g = unit_owner(u0, W, G);; g = unit_owner(range_begin(g + 1, W, G), W, G)) {
        ++n;
        if (range_begin(g + 1, W, G) > u1) break;
    }
    return n;
}

// Dequantisation of one 32-bit code word: the 8 weights (q - 8) * scale,
// exactly, as 4 fp16 pairs in element order (elements 2j, 2j+1 -> o[j]).
// Element i's code sits at bit nibble_pos(i) = 6, 22, 10, 26, 14, 30, 18, 2
// (the one at 30 wraps to bits 0-1), so that
//  * w & 0x03C003C0 holds elements 0 and 1 at bits 6-9 of each half, and a
//    rotation by 4 brings elements 2 and 3 there: OR-ing the exponent of 16
//    makes the fp16 values 16 + q, and one fused multiply-add with the
//    scale s and -24 s gives (16 + q) s - 24 s = (q - 8) s, rounded once
//    from the exact value, which is itself an fp16 number (s has at most 8
//    significant bits, q - 8 at most 4);
//  * a rotation by 14 brings elements 4, 5 to bits 0-3 and 6, 7 to bits
//    4-7 of each half: OR-ing the exponent of 1024 makes 1024 + q (or
//    1024 + 16 q), minus 1032 (or times 1/16 minus 72) is q - 8 exactly,
//    then a product with s.
// The fused form needs -24 s in fp16 (|s| <= 65504/24); buffers with wider
// or infinite scales use exact_pairs for elements 0-3 as well.  The two
// ways split the work evenly between the integer and the fp16 pipes.
__device__ __forceinline__ uint32_t rotr(uint32_t x, int n) { return __funnelshift_r(x, x, n); }

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// The two exponent patterns OR-ed onto the codes (fp16 16 and 1024 in both
// halves).  An AND-OR takes one of its two constants as an immediate and
// the other from a register; given two immediates the compiler emits two
// instructions.  The kernels therefore keep these two in shared memory and
// load them into registers once (a loaded value is not folded back into an
// immediate), which takes the dequantisation from 10 to 6 integer
// instructions per code word.
struct DqMagic {
    uint32_t m16, m1024;
};
constexpr uint32_t kMagic16 = 0x4C004C00u, kMagic1024 = 0x64006400u;
// p: 8-byte aligned shared-memory pair holding {kMagic16, kMagic1024}
__device__ __forceinline__ DqMagic load_dq_magic(const uint32_t *p) {
    DqMagic m;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(m.m16), "=r"(m.m1024) : "r"(smem_u32(p)));
    return m;
}

// (1024 + q) and (1024 + 16 q) at bits 0-3 / 4-7 of each half of x -> 2 pairs
__device__ __forceinline__ void exact_pairs(uint32_t x, __half2 s2, uint32_t m1024, uint32_t &lo,
                                            uint32_t &hi) {
    uint32_t r0 = (x & 0x000F000Fu) | m1024;
    uint32_t r1 = (x & 0x00F000F0u) | m1024;
    lo = h2u(__hmul2(__hsub2(*reinterpret_cast<__half2 *>(&r0), __floats2half2_rn(1032.f, 1032.f)),
                     s2));
    hi = h2u(__hmul2(__hfma2(*reinterpret_cast<__half2 *>(&r1), __floats2half2_rn(0.0625f, 0.0625f),
                             __floats2half2_rn(-72.f, -72.f)),
                     s2));
}

// s2 = (s, s); c2 = (-24 s, -24 s) when FUSED
template <bool FUSED>
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 c2, DqMagic m,
                                             uint32_t (&o)[4]) {
    if (FUSED) {
        const uint32_t mask = 0x03C003C0u;
        uint32_t r0 = (w & mask) | m.m16;
        uint32_t r1 = (rotr(w, 4) & mask) | m.m16;
        o[0] = h2u(__hfma2(*reinterpret_cast<__half2 *>(&r0), s2, c2));
        o[1] = h2u(__hfma2(*reinterpret_cast<__half2 *>(&r1), s2, c2));
    } else {
        exact_pairs(rotr(w, 6), s2, m.m1024, o[0], o[1]);
    }
    exact_pairs(rotr(w, 14), s2, m.m1024, o[2], o[3]);
}

// SiLU(gate) * up of one gate/up lane pair, as the fp16 pair hi + lo of
// the lane's parity: hi = fp16(a) for even lanes, lo = fp16(a - hi) for odd
// ones.  Both lanes compute a (no divergent branch); v is the lane's
// accumulator value, the partner's comes over a shuffle.  __expf and
// __fdividef (relative error ~1e-6) are far inside the layer tolerance.
// Sets *overflow when a finite a is beyond fp16 range.
__device__ __forceinline__ uint16_t silu_mul_half(float v, int lane, bool &overflow) {
    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
    const float gte = (lane & 1) ? other : v;
    const float up = (lane & 1) ? v : other;
    const float act = __fdividef(gte * up, 1.0f + __expf(-gte));
    const __half hi = __float2half_rn(act);
    const __half lo = __float2half_rn(act - __half2float(hi));
    overflow |= fabsf(act) > 65504.0f && fabsf(act) < INFINITY;
    return __half_as_ushort((lane & 1) ? lo : hi);
}

}  // namespace tc
}  // namespace moe
