// decode.cu -- the whole MoE layer forward for small batches in one kernel.
//
// For decode-sized batches (at most kDecodeMaxSlots routed slots) the layer's
// time is set by streaming the active experts' weights ("The MoE Throughput
// Lever: Quantifying the INT4 Marlin GEMM on Blackwell PRO 6000", "The Two
// Regimes: Weight-Streaming vs. Compute-Bound", and the M = 1 ... 9 rows of
// "The Benchmark: What Was Measured").  Five launches (alignment, hidden
// gather, gate+up GEMM, down GEMM, combine) each pay a start-up and a
// pipeline fill and drain around a few tens of microseconds of streaming;
// here one persistent CTA per SM runs all of them:
//
//  1. every CTA aligns the <= 128 slots itself, in shared memory (the stable
//     counting sort by expert of the flat slot index, as the alignment
//     kernel does; CTA 0 also writes it to the workspace);
//  2. the grid converts the hidden rows to fp16 in expert-sorted order and
//     zeroes the call's tickets and flags, while each CTA's weight producers
//     already issue their first weight copies; one grid-wide barrier (a
//     cooperative launch) ends this prologue;
//  3. each CTA streams its share of the gate+up chunks and then of the down
//     chunks through one ring of shared-memory stages: weight blocks and
//     token rows arrive on separate barriers, so the down GEMM's weights
//     (dequantised as soon as they land) stream while the gate+up GEMM's
//     last tiles finish anywhere on the GPU;
//  4. a gate+up tile's epilogue writes its 64 activation columns and counts
//     them into a per-(token tile, 128-column K chunk) flag; the token
//     producer issues a down-GEMM chunk's activation copy only once its flag
//     is complete (a bounded wait on memory that other CTAs of this grid
//     write -- all of them are resident, the launch being cooperative);
//  5. a down tile's epilogue writes y rows and counts them into a per
//     (128-row output slice, epilogue warp) ticket; the last tile to arrive
//     sums the k slots of every token for its 32 output columns in ascending
//     slot order and writes the bf16 output (the combine of "perf(exl3):
//     accelerate fat-expert prefill - #77", direct row writes).
// The tile schedule, dequantisation, MMAs and split-tile reduction are those
// of the grouped GEMM kernel (gemm_tc.cu).  Every wait is bounded; a wait
// that gives up records MOE_ERR_DEVICE_TIMEOUT and the CTA winds down.
#include <cooperative_groups.h>

#include "decode.h"
#include "device_common.cuh"
#include "sm100.cuh"
#include "small_align.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

using namespace sm100;
using namespace tc;
namespace cg = cooperative_groups;

constexpr int kNT = kDecodeTokenTile;                 // token rows per tile
constexpr int kStages = 12;
constexpr int kDqGroups = 4;
constexpr int kWProd = 2;                             // producer warps (alternate chunks)
constexpr int kMmaWarps = 2;
constexpr int kEpiWarps = 4;
constexpr int kAB = 4;                                // TMEM A buffers
constexpr int kACols = kChunkK / 2;                   // 64 columns per A buffer
constexpr int kTokBox = kNT * 128;                    // one 64-column box of kNT rows
constexpr int kTokBytes = 4 * kTokBox;                // down GEMM: [hi | lo] x 2 K halves
constexpr int kStageBytes = kTokBytes + kBlockBytes;  // token rows, then the weight block
constexpr int kAccCols = 2 * kNT;                     // down GEMM: hi and lo rows stacked
constexpr int kAccBase = kAB * kACols;
constexpr uint32_t kTmemCols = 512;
constexpr int kWarpDq = kEpiWarps;
constexpr int kWarpWProd = kWarpDq + 4 * kDqGroups;
constexpr int kWarpMma = kWarpWProd + kWProd;
constexpr int kWarps = kWarpMma + kMmaWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxSlots = kDecodeMaxSlots;
static_assert(kMaxSlots == kSmallAlignSlots, "the alignment of a small batch");
// a down-GEMM chunk (128 activation columns) is ready once both gate+up
// tiles that write them have had all four epilogue warps count it
constexpr int kFlagTarget = 2 * kEpiWarps;

static_assert(kStages % kDqGroups == 0 && kAB % kDqGroups == 0, "stages and A buffers per dequant group");
static_assert(kStages % kWProd == 0, "stages per weight producer");
static_assert(kStages % kMmaWarps == 0 && kAB % kMmaWarps == 0, "stages and A buffers per MMA warp");
static_assert(kStages >= kAB, "a stage must outlive its A buffer's reuse distance");
static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
static_assert(kAccBase + 2 * kMmaWarps * kAccCols <= (int)kTmemCols, "tensor memory budget");
static_assert(kMaxSlots <= kThreads && kMaxSlots <= 128, "one thread per slot; four warps rank");

// One GEMM of the layer as this CTA sees it: geometry and its schedule (the
// rules of gemm_tc.cu: whole tiles round-robin with at least 8 tiles per
// CTA, else the chunks of the first `rem` tiles split evenly (stream-K) and
// then `q_whole` whole tiles per CTA).
struct Gemm {
    const uint8_t *w;
    int R, KC, T;
    bool rr;
    int q_whole, rem;
    int64_t W, u_begin;
    int sk, my;  // this CTA's stream-K chunks, all its chunks
};

struct Smem {
    uint64_t full[kStages];      // weight block and token rows landed
    uint64_t consumed[kStages];  // MMAs of the stage's chunk done
    uint64_t a_full[kAB];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t done;
    uint32_t dq_magic[2];  // {kMagic16, kMagic1024}, loaded by the dequant warps
    uint32_t tmem_base;
    int abort;
    int bad;                     // a prepacked header does not match
    int wide[2];                 // per matrix: scales beyond the fused dequantisation
    int overflow;                // a hidden value beyond fp16 range
    int n_tt;
    Gemm gm[2];                  // this CTA's view of the gate+up and the down GEMM
    SmallAlign al;               // the batch's alignment
    int32_t act_tp[kMaxSlots + 1];   // active experts' first token tile (act_tp[n_act] = n_tt)
};

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(int32_t *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders this thread's earlier (generic) accesses of global memory with its
// later tensor-copy (async proxy) reads of it.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void make_gemm(Gemm &m, const uint8_t *w, int R, int KC, int n_tt, int G,
                                          int g) {
    m.w = w;
    m.R = R;
    m.KC = KC;
    m.T = n_tt * R;
    m.rr = m.T >= 8 * G;
    m.q_whole = m.rr ? 0 : m.T / G;
    m.rem = m.rr ? 0 : m.T - m.q_whole * G;
    m.W = (int64_t)m.rem * KC;
    m.u_begin = range_begin(g, m.W, G);
    m.sk = (int)(range_begin(g + 1, m.W, G) - m.u_begin);
    m.my = m.rr ? (g < m.T ? (m.T - g + G - 1) / G : 0) * KC : m.sk + m.q_whole * KC;
}

// tile and K chunk of this CTA's chunk c of GEMM m
__device__ __forceinline__ void locate(const Gemm &m, int g, int G, int c, int &tile, int &kc) {
    if (m.rr) {
        tile = g + (c / m.KC) * G;
        kc = c % m.KC;
    } else if (c < m.sk) {
        tile = (int)((m.u_begin + c) / m.KC);
        kc = (int)((m.u_begin + c) % m.KC);
    } else {
        tile = m.rem + g + ((c - m.sk) / m.KC) * G;
        kc = (c - m.sk) % m.KC;
    }
}

// end (exclusive) of the run of chunks from c that stays in one tile and one
// part of the schedule
__device__ __forceinline__ int seg_end(const Gemm &m, int c, int kc) {
    const int limit = (c < m.sk) ? m.sk : m.my;
    return c + min(m.KC - kc, limit - c);
}

struct Tile {
    int e, rt, v, p0, rows;
};

__device__ __forceinline__ Tile decode_tile(const Smem *sm, int R, int tile) {
    Tile t;
    t.v = tile / R;
    t.rt = tile - t.v * R;
    int lo = 0, hi = sm->al.n_act;  // largest a with act_tp[a] <= v
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm->act_tp[mid] <= t.v) lo = mid; else hi = mid;
    }
    t.e = sm->al.act_e[lo];
    t.p0 = sm->al.act_off[lo] + (t.v - sm->act_tp[lo]) * kNT;
    t.rows = min(kNT, sm->al.act_off[lo + 1] - t.p0);
    return t;
}

// Walks a producer's chunks over both GEMMs (gate+up first), `step` chunks
// at a time: within a tile it only moves the weight pointer; a round-robin
// walk steps to the tile G further on without a division; only the start,
// the stream-K part and the change of GEMM use the full lookup.  It keeps
// its own copy of the current GEMM (a runtime index into a pair would put
// the pair in local memory).
struct Walker {
    Gemm cur;
    int ph, c, kc, end, tile;
    const uint8_t *wp;  // the weight block of the current chunk
    int p0, v;          // the current tile's first sorted row and token tile

    __device__ __forceinline__ void at_tile(const Smem *sm) {
        const Tile t = decode_tile(sm, cur.R, tile);
        p0 = t.p0;
        v = t.v;
        wp = cur.w + kHeaderBytes + (((int64_t)t.e * cur.R + t.rt) * cur.KC + kc) * kBlockBytes;
    }
    __device__ __forceinline__ bool settle(const Gemm &m0, const Gemm &m1, const Smem *sm, int g,
                                           int G) {
        if (ph == 0 && c >= m0.my) {
            c -= m0.my;
            ph = 1;
            cur = m1;
        }
        if (c >= cur.my) return false;
        locate(cur, g, G, c, tile, kc);
        end = seg_end(cur, c, kc);
        at_tile(sm);
        return true;
    }
    __device__ __forceinline__ bool start(int gc, const Gemm &m0, const Gemm &m1, const Smem *sm,
                                          int g, int G) {
        ph = 0;
        cur = m0;
        c = gc;
        return settle(m0, m1, sm, g, G);
    }
    __device__ __forceinline__ bool advance(int step, const Gemm &m0, const Gemm &m1, const Smem *sm,
                                            int g, int G) {
        c += step;
        if (c < end) {
            kc += step;
            wp += (int64_t)step * kBlockBytes;
            return true;
        }
        if (cur.rr && c < cur.my) {
            kc += step;
            do {
                kc -= cur.KC;
                tile += G;
            } while (kc >= cur.KC);
            end = c - kc + cur.KC;
            at_tile(sm);
            return true;
        }
        return settle(m0, m1, sm, g, G);
    }
};

__device__ __forceinline__ uint32_t half_bits(float v) {
    return (uint32_t)__half_as_ushort(__float2half_rn(v));
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_x,
                  const __grid_constant__ CUtensorMap map_act) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem *sm = reinterpret_cast<Smem *>(base + kStages * kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, g = blockIdx.x;
    const int n = a.M * a.k;
    const int R1 = 2 * a.I / kTileRows, KC1 = a.H / kChunkK;  // gate+up
    const int R2 = a.H / kTileRows, KC2 = a.I / kChunkK;      // down

    // ---------------- set-up
    if (warp == kWarpMma) {
        tmem_alloc(&sm->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->consumed[s], 1);
        }
        for (int b = 0; b < kAB; ++b) mbar_init(&sm->a_full[b], 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm->acc_full[b], kMmaWarps);
            mbar_init(&sm->acc_empty[b], 128);
        }
        mbar_init(&sm->done, kMmaWarps);
        sm->dq_magic[0] = kMagic16;
        sm->dq_magic[1] = kMagic1024;
        sm->abort = 0;
        sm->bad = !header_ok(a.w13, MOE_PACK_W13, a.E, 2 * a.I, a.H) ||
                  !header_ok(a.w2, MOE_PACK_W2, a.E, a.H, a.I);
        sm->wide[0] = reinterpret_cast<const PackHeader *>(a.w13)->wide_scales != 0;
        sm->wide[1] = reinterpret_cast<const PackHeader *>(a.w2)->wide_scales != 0;
        sm->overflow = 0;
        fence_barrier_init();
    }
    if (warp == kWarpWProd && lane == 0) {
        prefetch_tensormap(&map_x);
        prefetch_tensormap(&map_act);
    }

    // The hidden rows are the call's input: this thread's first 16-byte
    // piece of them goes out now, before the alignment says where it goes.
    const int64_t gthreads = (int64_t)G * kThreads, gi = (int64_t)g * kThreads + tid;
    const int vecs = a.H / 8;
    const int64_t hwork = (int64_t)a.M * vecs;
    uint4 hv0 = make_uint4(0, 0, 0, 0);
    if (gi < hwork)
        hv0 = __ldg(reinterpret_cast<const uint4 *>(a.hidden + (size_t)(gi / vecs) * a.H) + gi % vecs);

    // ---------------- alignment of the <= 128 slots, in shared memory
    small_align(&sm->al, a.ids, n, a.E);
    const int n_valid = sm->al.n_valid, n_act = sm->al.n_act;
    if (warp == 0) {
        const int tt = small_tile_prefix(&sm->al, kNT, sm->act_tp, lane);
        if (lane == 0) sm->n_tt = tt;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const int n_tt_all = sm->n_tt;
    const int n_tt = sm->bad ? 0 : n_tt_all;  // a mismatched buffer: no GEMM work
    // the two GEMMs' schedules live in shared memory: every role reads the
    // fields it needs instead of holding both in registers
    if (tid == 0) make_gemm(sm->gm[0], a.w13, R1, KC1, n_tt, G, g);
    if (tid == 32) make_gemm(sm->gm[1], a.w2, R2, KC2, n_tt, G, g);
    __syncthreads();
    const Gemm *m = sm->gm;
    const int total = m[0].my + m[1].my;  // this CTA's chunks over both GEMMs
    // the sync region: tickets of both GEMMs (per tile and epilogue warp),
    // activation-ready flags (per token tile and 128-column K chunk of the
    // down GEMM), combine tickets (per 128-row output slice and warp)
    int32_t *tick1 = a.sync;
    int32_t *tick2 = tick1 + (int64_t)m[0].T * kEpiWarps;
    int32_t *flags = tick2 + (int64_t)m[1].T * kEpiWarps;
    int32_t *comb = flags + (int64_t)n_tt * KC2;
    const int64_t sync_used = (int64_t)(comb - a.sync) + (int64_t)R2 * kEpiWarps;

    // ---------------- prologue across the grid
    if (sync_used <= a.sync_ints)
        for (int64_t i = gi; i < sync_used; i += gthreads) a.sync[i] = 0;
    {
        // hidden rows -> fp16, each piece written to the sorted rows of its
        // token's valid slots
        bool overflow = false;
        for (int64_t i = gi; i < hwork; i += gthreads) {
            const int t = (int)(i / vecs), v = (int)(i % vecs);
            const uint4 in = (i == gi) ? hv0
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
                const int p = sm->al.inv[t * a.k + j];
                if (p >= 0) reinterpret_cast<uint4 *>(a.xs + (size_t)p * a.H)[v] = ov;
            }
        }
        if (overflow) sm->overflow = 1;
        // no token tile at all (every id out of range): the output is zero
        if (n_tt_all == 0) {
            const int64_t ovec = (int64_t)a.M * a.H / 8;
            for (int64_t i = gi; i < ovec; i += gthreads)
                reinterpret_cast<uint4 *>(a.out)[i] = make_uint4(0, 0, 0, 0);
        }
    }
    if (g == 0 && tid == 0) {
        if (a.reset_status) {
            a.ctrl->status = 0;
            a.ctrl->detail = 0;
        }
        a.ctrl->n_invalid = n - n_valid;
    }

    // ---------------- producers, set-up.  Producer pw copies the weight
    // block and the token rows of chunks pw, pw + 2, ... (global order: the
    // gate+up chunks, then the down chunks) into the chunk's stage, both
    // counted on the stage's `full` barrier.  The weights are the call's
    // input, so the copies into the first (free) stages go out now; their
    // token rows follow the grid barrier below.
    const bool producer = warp >= kWarpWProd && warp < kWarpMma;
    const int pw = warp - kWarpWProd;
    Walker wk;           // the next chunk whose copies are not issued
    int wgc = pw;        // its global index
    bool more = false;
    const uint64_t pol_w = policy_evict_first();
    auto issue_weights = [&](int s) {
        if (elect_one()) {
            mbar_arrive_expect_tx(&sm->full[s], kBlockBytes + (wk.ph ? 4 : 2) * kTokBox);
            bulk_g2s_hint(base + s * kStageBytes + kTokBytes, wk.wp, kBlockBytes, &sm->full[s], pol_w);
        }
        __syncwarp();
    };
    auto issue_tokens = [&](const Walker &w, int s) {
        if (elect_one()) {
            uint8_t *st = base + s * kStageBytes;
            if (w.ph == 0)
                tma_load_3d(st, &map_x, 0, w.p0, 2 * w.kc, &sm->full[s]);
            else
                tma_load_4d(st, &map_act, 0, w.p0, 0, 2 * w.kc, &sm->full[s]);
        }
        __syncwarp();
    };
    // Down-GEMM chunks need the gate+up tiles that write their activation
    // rows to be done.  The producer reads the flags of 32 K chunks of one
    // token tile with one warp-wide load (lane i: chunk base + i) and keeps
    // which of them were complete (flags only grow), so a flag costs an L2
    // round trip only when the producer reaches a chunk whose flag it has
    // not yet seen complete.  Waits are bounded.
    int ready_v = -1, ready_base = 0;
    unsigned ready_mask = 0;  // bit i: flag (ready_v, ready_base + i) seen complete
    auto wait_flag = [&](const Walker &w) {
        const int base32 = w.kc & ~31, bit = w.kc - base32;
        if (w.v == ready_v && base32 == ready_base && ((ready_mask >> bit) & 1u)) return true;
        const long long t0 = clock64();
        for (;;) {
            const int kc = base32 + lane;
            const bool ok = kc < KC2 && ld_acquire(flags + (int64_t)w.v * KC2 + kc) >= kFlagTarget;
            ready_v = w.v;
            ready_base = base32;
            ready_mask = __ballot_sync(0xffffffffu, ok);
            if ((ready_mask >> bit) & 1u) {
                // the lane that issues the copy follows every lane's acquire
                __syncwarp();
                fence_proxy_async_global();
                return true;
            }
            if (*(volatile int *)&sm->abort) return false;
            if (clock64() - t0 > kWaitCycles) {
                if (lane == 0) {
                    atomicExch(&sm->abort, 1);
                    set_status(a.ctrl, MOE_ERR_DEVICE_TIMEOUT, 7);
                }
                __syncwarp();
                return false;
            }
            __nanosleep(256);
        }
    };
    if (producer && !a.test_no_copies) {
        more = wk.start(pw, m[0], m[1], sm, g, G);
        while (more && wgc < kStages) {  // fresh stages: free
            issue_weights(wgc);
            wgc += kWProd;
            more = wk.advance(kWProd, m[0], m[1], sm, g, G);
        }
    }

    // grid-wide barrier: xs, the zeroed tickets and flags are complete.
    // Only a cooperative launch has one; without it the kernel reports a
    // device error and does no GEMM work rather than wait on CTAs that may
    // never run.
    cg::grid_group grid = cg::this_grid();
    const bool have_grid = grid.is_valid();
    if (have_grid) grid.sync();
    if (tid == 0 && !have_grid) {
        set_status(a.ctrl, MOE_ERR_DEVICE_TIMEOUT, 8);
        atomicExch(&sm->abort, 1);
    }
    __syncthreads();
    if (tid == 0) {
        if (g == 0 && sm->bad) set_status(a.ctrl, MOE_ERR_BAD_LAYOUT, 0);
        if (g == 0 && n_valid < n) set_status(a.ctrl, MOE_ERR_DEVICE_BAD_EXPERT_ID, sm->al.raw[sm->al.first_bad_slot]);
        if (sm->overflow) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 0);
        if (sync_used > a.sync_ints) {
            set_status(a.ctrl, MOE_ERR_DEVICE_TIMEOUT, 0);  // cannot happen: sized on the host
            atomicExch(&sm->abort, 1);
        }
    }
    const uint32_t tb = sm->tmem_base;
    __syncthreads();
    // a set-up failure found above: only the weight copies already issued
    // are waited for
    const bool run = !*(volatile int *)&sm->abort;

    if (producer) {
        // ---------------- producers.  First the token rows of the chunks
        // whose weights went out before the barrier (each stage's
        // transaction count includes them, so they are issued even after a
        // failure), then one chunk at a time: wait for its stage, copy its
        // weights, and copy its token rows -- for a down-GEMM chunk once the
        // gate+up tiles that write them are done.
        if (!a.test_no_copies) {
            fence_proxy_async_global();
            bool ok = run;
            if (pw < wgc) {
                Walker tk;
                tk.start(pw, m[0], m[1], sm, g, G);
                for (int tgc = pw; tgc < wgc; tgc += kWProd) {
                    if (tk.ph == 1 && ok) ok = wait_flag(tk);
                    issue_tokens(tk, tgc % kStages);
                    tk.advance(kWProd, m[0], m[1], sm, g, G);
                }
            }
            // stage and its phase parity kept incrementally (no division per chunk)
            int s = wgc % kStages;
            uint32_t par = ((wgc / kStages) & 1) ^ 1;
            while (ok && more) {
                if (!warp_wait_bar(&sm->consumed[s], par, &sm->abort, a.ctrl, 1)) break;
                const bool known = wk.ph == 0 || (wk.v == ready_v && (wk.kc & ~31) == ready_base &&
                                                  ((ready_mask >> (wk.kc & 31)) & 1u));
                if (known) {
                    // the common case: both copies from one elected lane
                    if (elect_one()) {
                        uint8_t *st = base + s * kStageBytes;
                        mbar_arrive_expect_tx(&sm->full[s], kBlockBytes + (wk.ph ? 4 : 2) * kTokBox);
                        bulk_g2s_hint(st + kTokBytes, wk.wp, kBlockBytes, &sm->full[s], pol_w);
                        if (wk.ph == 0)
                            tma_load_3d(st, &map_x, 0, wk.p0, 2 * wk.kc, &sm->full[s]);
                        else
                            tma_load_4d(st, &map_act, 0, wk.p0, 0, 2 * wk.kc, &sm->full[s]);
                    }
                    __syncwarp();
                } else {
                    // the weights go out first; the activation rows once ready
                    issue_weights(s);
                    ok = wait_flag(wk);
                    issue_tokens(wk, s);
                }
                wgc += kWProd;
                s += kWProd;
                if (s >= kStages) {
                    s -= kStages;
                    par ^= 1;
                }
                more = wk.advance(kWProd, m[0], m[1], sm, g, G);
            }
        }
        // every copy issued must land before the CTA exits
        for (int j = (wgc > kStages ? wgc - kStages : 0); j < wgc; ++j)
            if (j % kWProd == pw) wait_bar_final(&sm->full[j % kStages], (j / kStages) & 1);
        __syncwarp();
    } else if (!run) {
        // nothing to do
    } else if (warp >= kWarpMma) {
        // ---------------- MMA issuers (alternate chunks, own accumulators)
        const int mw = warp - kWarpMma;
        const uint64_t desc_base = sdesc_k_sw128(smem_u32(base));
        int seg = 0;
        bool ok = true;
        // stage, A buffer and A-buffer phase of this warp's next chunk, kept
        // incrementally (kStages and kAB are multiples of kMmaWarps)
        int s = mw, b = mw;
        uint32_t bph = 0;
#pragma unroll
        for (int ph = 0; ph < 2; ++ph) {
            if (!ok) break;
            const Gemm &G_ = m[ph];
            const int gbase = ph ? m[0].my : 0;
            const uint32_t idesc = idesc_f16_m128(ph ? 2 * kNT : kNT);
            for (int c = 0; c < G_.my && ok; ++seg) {
                int tile, k0;
                locate(G_, g, G, c, tile, k0);
                const int c_end = seg_end(G_, c, k0);
                const int acc = seg & 1;
                if (!warp_wait_bar(&sm->acc_empty[acc], ((seg >> 1) & 1) ^ 1, &sm->abort, a.ctrl, 2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tb + kAccBase + (acc * kMmaWarps + mw) * kAccCols;
                bool first = true;
                int gc = gbase + c;
                gc += ((mw - gc % kMmaWarps) + kMmaWarps) % kMmaWarps;
                for (; gc < gbase + c_end; gc += kMmaWarps) {
                    // the dequant warps arrive on a_full after their wait on the
                    // stage's full barrier, which also counted the token rows
                    if (!warp_wait_bar(&sm->a_full[b], bph, &sm->abort, a.ctrl, 3)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) {
                        const uint64_t desc0 = desc_base + (uint64_t)((s * kStageBytes) >> 4);
                        const uint32_t a_tmem = tb + b * kACols;
#pragma unroll
                        for (int j = 0; j < kChunkK / 16; ++j) {
                            const uint32_t boff = ph ? (j >> 2) * 2 * kTokBox + (j & 3) * 32
                                                     : (j >> 2) * kTokBox + (j & 3) * 32;
                            mma_f16_ts(d_tmem, a_tmem + j * 8, desc0 + (boff >> 4), idesc,
                                       (!first || j > 0) ? 1u : 0u);
                        }
                        tc_commit(&sm->consumed[s]);
                    }
                    __syncwarp();
                    first = false;
                    s += kMmaWarps;
                    if (s >= kStages) s -= kStages;
                    b += kMmaWarps;
                    if (b >= kAB) {
                        b -= kAB;
                        bph ^= 1;
                    }
                }
                if (!ok) break;
                if (elect_one()) tc_commit(&sm->acc_full[acc]);
                __syncwarp();
                c = c_end;
            }
        }
        if (elect_one()) {
            tc_commit(&sm->done);
            wait_bar_final(&sm->done, 0);
        }
        __syncwarp();
    } else if (warp >= kWarpDq) {
        // ---------------- dequantisation warpgroups (every fourth chunk)
        const int grp = (warp - kWarpDq) / 4;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const int my0 = m[0].my;
        const DqMagic mg = load_dq_magic(sm->dq_magic);
        const bool wide0 = sm->wide[0] != 0, wide1 = sm->wide[1] != 0;
        // stage, its phase and the A buffer of this group's next chunk, kept
        // incrementally (kStages and kAB are multiples of kDqGroups)
        int s = grp, b = grp;
        uint32_t ph = 0;
        for (int gc = grp; gc < total; gc += kDqGroups) {
            if (!warp_wait_bar(&sm->full[s], ph, &sm->abort, a.ctrl, 4)) break;
            if (gc >= kAB) {
                // A buffer b was last read by the MMAs of chunk gc - kAB,
                // whose stage is kAB stages back
                const int sp = s >= kAB ? s - kAB : s - kAB + kStages;
                const uint32_t pp = s >= kAB ? ph : ph ^ 1;
                if (!warp_wait_bar(&sm->consumed[sp], pp, &sm->abort, a.ctrl, 5)) break;
            }
            tc_fence_after();
            const uint32_t st_s = smem_u32(base + s * kStageBytes + kTokBytes);
            uint2 sc;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(sc.x), "=r"(sc.y) : "r"(st_s + kCodeBlockBytes + r * 8));
            const uint32_t scw[2] = {sc.x, sc.y};
            const uint32_t a_addr = tb + lane_off + b * kACols;
            auto pieces = [&](auto fused) {
                constexpr bool kFused = decltype(fused)::value;
#pragma unroll
                for (int pc = 0; pc < 4; ++pc) {
                    uint4 q;
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                                 : "r"(st_s + (pc * kTileRows + r) * 16));
                    const uint32_t sbits = (scw[pc >> 1] >> ((pc & 1) * 16)) & 0xFFFFu;
                    const __half hs = __ushort_as_half((unsigned short)sbits);
                    const __half2 s2 = __halves2half2(hs, hs);
                    const __half2 c2 = kFused ? __hmul2(s2, __floats2half2_rn(-24.f, -24.f)) : s2;
                    uint32_t v[16], o[4];
                    dequant_word<kFused>(q.x, s2, c2, mg, o);
                    v[0] = o[0]; v[1] = o[1]; v[2] = o[2]; v[3] = o[3];
                    dequant_word<kFused>(q.y, s2, c2, mg, o);
                    v[4] = o[0]; v[5] = o[1]; v[6] = o[2]; v[7] = o[3];
                    dequant_word<kFused>(q.z, s2, c2, mg, o);
                    v[8] = o[0]; v[9] = o[1]; v[10] = o[2]; v[11] = o[3];
                    dequant_word<kFused>(q.w, s2, c2, mg, o);
                    v[12] = o[0]; v[13] = o[1]; v[14] = o[2]; v[15] = o[3];
                    tmem_st16(a_addr + pc * 16, v);
                }
            };
            if (gc < my0 ? wide0 : wide1)
                pieces(std::false_type{});
            else
                pieces(std::true_type{});
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&sm->a_full[b]);
            s += kDqGroups;
            if (s >= kStages) {
                s -= kStages;
                ph ^= 1;
            }
            b += kDqGroups;
            if (b >= kAB) b -= kAB;
        }
    } else {
        // ---------------- epilogue warpgroup (warps 0-3)
        if (g == 0) {
            // the alignment, for inspection (the views of the workspace),
            // written while the first tiles are still being computed
            for (int e = tid; e < a.E; e += (32 * kEpiWarps)) {
                const int lo = small_first_at_least(&sm->al, e);
                a.offsets[e] = sm->al.act_off[lo];
                a.counts[e] = (lo < n_act && sm->al.act_e[lo] == e)
                                  ? sm->al.act_off[lo + 1] - sm->al.act_off[lo] : 0;
            }
            if (tid == 0) a.offsets[a.E] = n_valid;
            for (int p = tid; p < n; p += (32 * kEpiWarps)) {
                a.perm[p] = p < n_valid ? sm->al.perm[p] : -1;
                a.inv_perm[p] = sm->al.inv[p];
            }
        }
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int seg = 0;
        bool ok = true;
#pragma unroll
        for (int ph = 0; ph < 2; ++ph) {
            if (!ok) break;
            const Gemm &G_ = m[ph];
            const int gbase = ph ? m[0].my : 0;
            int32_t *tickets = ph ? tick2 : tick1;
            float *part = a.partials + (size_t)ph * G * 2 * kNT * kTileRows;
            for (int c = 0; c < G_.my; ++seg) {
                int tile, k0;
                locate(G_, g, G, c, tile, k0);
                const int c_end = seg_end(G_, c, k0);
                const int k1 = k0 + (c_end - c);
                const Tile t = decode_tile(sm, G_.R, tile);
                const int acc = seg & 1;
                if (!warp_wait_bar(&sm->acc_full[acc], (seg >> 1) & 1, &sm->abort, a.ctrl, 6)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t acc_addr = tb + lane_off + kAccBase + acc * kMmaWarps * kAccCols;
                bool has[2] = {true, true};
                if (c_end - c == 1) {
                    has[0] = ((gbase + c) % 2 == 0);
                    has[1] = !has[0];
                }
                // the issuers' accumulators (and, in the down GEMM, the lo
                // half of each, kNT columns on) added one 16-column slice at
                // a time, always in the same order
                float v[16];
                bool any = false;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) {
                    if (!has[w]) continue;
#pragma unroll
                    for (int half = 0; half < (ph ? 2 : 1); ++half) {
                        uint32_t x[16];
                        tmem_ld16(acc_addr + w * kAccCols + half * kNT, x);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[j] = any ? v[j] + __uint_as_float(x[j]) : __uint_as_float(x[j]);
                        any = true;
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm->acc_empty[acc]);

                const bool whole = (k0 == 0 && k1 == G_.KC);
                bool finish = whole;  // this warp writes the tile's rows
                if (!whole) {
                    // partial sums; the last CTA to finish the tile adds all
                    // of them in CTA order
                    const int which = (c == 0) ? 0 : 1;
                    float *slot = part + ((size_t)g * 2 + which) * kNT * kTileRows;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j >= t.rows) break;
                        slot[(size_t)j * kTileRows + r] = v[j];
                    }
                    const int64_t tu0 = (int64_t)tile * G_.KC, tu1 = tu0 + G_.KC - 1;
                    const int ncontrib = contributors(tu0, tu1, G_.W, G);
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0) last = (atomicAdd(tickets + (size_t)tile * kEpiWarps + warp, 1) == ncontrib - 1);
                    finish = __shfl_sync(0xffffffffu, last, 0) != 0;
                    if (finish) {
                        __threadfence();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (j >= t.rows) break;
                            float sum = 0.f;
                            for (int gg = unit_owner(tu0, G_.W, G);; gg = unit_owner(range_begin(gg + 1, G_.W, G), G_.W, G)) {
                                const int wh = (range_begin(gg, G_.W, G) >= tu0) ? 0 : 1;
                                sum += __ldcg(part + ((size_t)gg * 2 + wh) * kNT * kTileRows +
                                              (size_t)j * kTileRows + r);
                                if (range_begin(gg + 1, G_.W, G) > tu1) break;
                            }
                            v[j] = sum;
                        }
                    }
                }
                if (finish) {
                    if (ph == 0) {
                        // SiLU(gate)*up: even lanes write hi, odd lanes lo, of
                        // activation column rt*64 + r/2; then count the rows
                        // into the flag of their 128-column K chunk
                        uint16_t *dst = ((lane & 1) ? a.act_lo : a.act_hi) + (size_t)t.p0 * a.I +
                                        t.rt * (kTileRows / 2) + (r >> 1);
                        bool overflow = false;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (j >= t.rows) break;
                            dst[(size_t)j * a.I] = silu_mul_half(v[j], lane, overflow);
                        }
                        if (overflow) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 1);
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) red_release_add(flags + (int64_t)t.v * KC2 + (t.rt >> 1), 1);
                    } else {
                        // y rows of the 128-row output slice rt, then the
                        // combine ticket of (slice, warp)
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            if (j >= t.rows) break;
                            a.y[(size_t)(t.p0 + j) * a.H + t.rt * kTileRows + r] = v[j];
                        }
                        __threadfence();
                        __syncwarp();
                        int last = 0;
                        if (lane == 0) last = (atomicAdd(comb + t.rt * kEpiWarps + warp, 1) == n_tt - 1);
                        if (__shfl_sync(0xffffffffu, last, 0)) {
                            // every token's k slots for output column h, in
                            // ascending slot order (the flat slot order),
                            // one bf16 rounding; the y loads of 8 slots go
                            // out together
                            __threadfence();
                            const int h = t.rt * kTileRows + r;
                            float sum = 0.f;
                            for (int f0 = 0; f0 < n; f0 += 8) {
                                float yv[8], wv[8];
                                int pv[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int f = f0 + i;
                                    pv[i] = f < n ? sm->al.inv[f] : -1;
                                    wv[i] = pv[i] >= 0 ? __ldg(a.topk_w + f) : 0.f;
                                    yv[i] = pv[i] >= 0 ? __ldcg(a.y + (size_t)pv[i] * a.H + h) : 0.f;
                                }
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int f = f0 + i;
                                    if (f >= n) break;
                                    if (pv[i] >= 0) sum = fmaf(wv[i], yv[i], sum);
                                    if ((f + 1) % a.k == 0) {
                                        a.out[(size_t)(f / a.k) * a.H + h] =
                                            __bfloat16_as_ushort(__float2bfloat16_rn(sum));
                                        sum = 0.f;
                                    }
                                }
                            }
                        }
                    }
                }
                c = c_end;
            }
        }
    }

    // ---------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tb, kTmemCols);
    }
}

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + sizeof(Smem) + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

}  // namespace

int64_t decode_sync_ints(int max_tiles, int H, int I) {
    const int R1 = 2 * I / kTileRows, R2 = H / kTileRows, KC2 = I / kChunkK;
    const int64_t n = (int64_t)max_tiles * (R1 + R2) * kEpiWarps + (int64_t)max_tiles * KC2 +
                      (int64_t)R2 * kEpiWarps;
    return (n + 3) / 4 * 4;
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &map_x, const CUtensorMap &map_act,
                          int grid, cudaStream_t s) {
    cudaError_t err = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel, a, map_x, map_act);
}

}  // namespace moe
