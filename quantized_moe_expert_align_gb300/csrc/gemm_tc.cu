// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores.
//
// Both expert contractions of the layer run here:
//   gate+up (MOE_PACK_W13): for every expert-sorted token row p of expert e,
//       g = xs[p] . Wg[n], u = xs[p] . Wu[n], a[p][n] = silu(g) * u  (the
//       stacked gate+up GEMM of "perf(exl3): accelerate fat-expert prefill -
//       #77", "Summary", with SiLU(gate)*up fused into the epilogue);
//   down    (MOE_PACK_W2):  y[p][h] = (a_hi + a_lo)[p] . W2[h].
// Weights are INT4 with one scale per 32 elements along K, as in the MoE
// GEMM of "The MoE Throughput Lever: Quantifying the INT4 Marlin GEMM on
// Blackwell PRO 6000" ("The Benchmark: What Was Measured").
//
// Design (weights as the MMA's M side, tokens as its N side):
//  * One persistent CTA per SM.  The work is the list of tiles (expert,
//    128-row weight tile, token tile of NT sorted rows) times 128-element K
//    chunks.  With many tiles each CTA takes whole tiles round-robin; with
//    few, the chunks of the first tiles are cut into equal contiguous shares
//    (stream-K), which each CTA does before its whole tiles, so the weight
//    stream is spread evenly over all SMs even when only a few experts are
//    active.  A tile cut between CTAs leaves fp32 partials in the workspace;
//    the last CTA to finish it (an atomic ticket, no waiting) sums them in
//    CTA order and runs the epilogue, so results do not depend on timing.
//  * Two TMA producer warps (alternate chunks) stream each chunk's 9 KiB
//    weight block (codes and scales, one bulk copy) and the chunk's token
//    rows (one tensor copy, 128-byte swizzle) into a ring of shared-memory
//    stages.
//  * Dequantisation warpgroups (four, or six in the gate+up GEMM with small
//    token tiles, three with the 160/80-row pair tiles; each takes every
//    fourth, sixth or third chunk) turn codes into
//    exact fp16 weights, (q - 8) * scale, one weight row per thread, and
//    write them straight into tensor memory with tcgen05.st.  That tensor
//    memory is the A operand of tcgen05.mma, so dequantised weights never
//    touch shared memory.
//  * One or two MMA warps (alternate chunks, each with its own accumulator,
//    or on the gate+up GEMM's CTA pairs taking turns on one) issue
//    tcgen05.mma (kind::f16, M = 128, N = token rows of the tile rounded up
//    to 16, K = 16) from one elected thread, accumulating in tensor memory;
//    the down GEMM multiplies the hi and the lo halves of a (stacked into
//    one B operand for small token tiles: 8 rows at decode, whose stages
//    leave room for 16 of them).
//  * An epilogue warpgroup drains the (double-buffered) accumulators while
//    the next tile is being computed.
//  * Large token tiles (128/160 rows in the gate+up GEMM, 64/80 in the down
//    GEMM) run on CTA pairs (clusters of two, tcgen05 cta_group::2): a work tile
//    is two neighbouring weight tiles, one per CTA, and one M = 256 MMA
//    covers both, so each SM loads only half of the token operand.  One SM
//    alone could not take in its 32 KiB of token rows per chunk as fast as
//    its tensor core used them (E = 128 M = 2048: one chunk every ~740
//    cycles against 512 of MMA work; as pairs the layer takes 898 instead of
//    973 us, Zipf prefill M = 16384 11.2 instead of 13.8 ms).
// Every mbarrier wait is bounded; a wait that gives up records
// MOE_ERR_DEVICE_TIMEOUT and the CTA winds down without hanging.
#include <cstring>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "gemm_tc.h"

namespace moe {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kEpiWarps = 4;
// Warps: 4 epilogue, 4 per dequantisation warpgroup, one or two TMA
// producers and one or two MMA issuers.
__host__ __device__ constexpr int threads_for(int dq_groups, int producers, int mma_warps) {
    return 32 * (kEpiWarps + 4 * dq_groups + producers + mma_warps);
}
constexpr int kMaxABufs = 6;                  // TMEM A buffers (64 columns each)
// TMEM A buffers of a configuration: one per dequant group, at least four
// (160-column accumulators -- 160-row gate+up tiles, 80-row down tiles with
// hi and lo stacked: three, next to two accumulators).
__host__ __device__ constexpr int a_buffers(int nt, int stages, int dq) {
    return (nt == 160 || nt == 80) ? 3 : (stages >= 4 ? (dq > 4 ? dq : 4) : 2);
}
constexpr int kACols = kChunkK / 2;           // 64 fp16 pairs per row per chunk
constexpr uint32_t kTmemCols = 512;

struct Smem {
    uint64_t full[kMaxStages];      // stage loaded (TMA transaction bytes)
    uint64_t consumed[kMaxStages];  // MMAs of the stage's chunk done (stage and A buffer free)
    uint64_t a_full[kMaxABufs];     // A buffer written by the dequant warps
    uint64_t acc_full[2], acc_empty[2];
    uint64_t done;
    uint64_t turn[2];  // CTA pairs: MMA issuer w may issue its next chunk
    uint32_t dq_magic[2];  // {kMagic16, kMagic1024}, loaded by the dequant warps
    uint32_t tmem_base;
    int abort;
    int bad;
    int wide;  // the weights have scales beyond the fused dequantisation's range
    // per-expert token-tile prefix and sorted-row offsets, copied once so
    // that decoding a tile is a search in shared, not global, memory
    int32_t tile_prefix[1025];
    int32_t offsets[1025];
};

struct Tile {
    int e, rt, p0, rows;
};

// MMA N of a gate+up tile of `rows` token rows on a CTA pair: a multiple of
// 32, so that each CTA's half of the token rows is a multiple of 16.
__device__ __forceinline__ int pair_n(int rows) { return max(32, (rows + 31) & ~31); }

// Work tile -> expert, first 128-row weight tile, token tile.  With CTA
// pairs (CG = 2) a work tile is two neighbouring weight tiles, one per CTA.
template <int NT, int CG>
__device__ __forceinline__ Tile decode_tile(const TcArgs &a, const Smem *sm, int tile) {
    Tile t;
    const int R = a.N / kTileRows / CG;
    const int v = tile / R;
    int lo = 0, hi = a.E;  // largest e with tile_prefix[e] <= v (tile_prefix[E] > v)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm->tile_prefix[mid] <= v) lo = mid; else hi = mid;
    }
    t.e = lo;
    const int tp0 = sm->tile_prefix[lo], tp1 = sm->tile_prefix[lo + 1];
    // within an expert, tiles run over the 128-row weight tiles of one token
    // tile before moving to the next token tile
    const int local = tile - R * tp0;
    (void)tp1;
    t.rt = (local % R) * CG;
    const int tt = local / R;
    t.p0 = sm->offsets[lo] + tt * NT;
    t.rows = min(NT, sm->offsets[lo + 1] - t.p0);
    return t;
}

// CG = 2: the kernel runs on clusters of two CTAs (CTA pairs, on the two SMs
// of a TPC) that share each MMA (cta_group::2, M = 256): the even CTA issues
// the pair's MMAs, each CTA dequantises its own 128-row weight tile into its
// own tensor memory and holds its own 128 rows of the accumulators, and each
// loads half of the token operand (the N side of the MMA): the first / second
// half of the token rows (gate+up) or the hi / lo rows (down).
template <int KIND, int NT, int STAGES, int DQG, int NPROD, int MMAW, int CG>
__global__ void __launch_bounds__(threads_for(DQG, NPROD, MMAW), 1)
    gemm_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tok) {
    constexpr int kDqGroups = DQG;
    constexpr int kThreads = threads_for(DQG, NPROD, MMAW);
    constexpr int kProducerWarp = kEpiWarps + 4 * DQG;
    constexpr int kMmaWarp = kProducerWarp + NPROD;
    constexpr bool kPair = CG == 2;
    constexpr int kTokRows = (kPair && KIND == MOE_PACK_W13) ? NT / 2 : NT;  // rows per box here
    constexpr int kTokBox = kTokRows * 128;                   // one 64-column box
    constexpr int kTokBoxes = (KIND == MOE_PACK_W2 && !kPair) ? 4 : 2;  // hi(+lo) x 2 boxes
    constexpr int kStageBytes = kTokBoxes * kTokBox + kBlockBytes;
    // Down GEMM with small token tiles: the hi and lo rows of a are stacked
    // into one B operand of 2*NT rows, so one MMA (whose cost does not grow
    // with N up to 128) covers both; the epilogue adds the two halves.
    constexpr bool kCat = (KIND == MOE_PACK_W2) && (NT <= 64 || NT == 80);  // == stacked_hi_lo(NT)
    constexpr int kAB = a_buffers(NT, STAGES, DQG);  // TMEM A buffers in use
    constexpr int kAccBase = kAB * kACols;
    // columns per accumulator (at least 32 stacked ones: the epilogue reads
    // 16-column blocks, the lo block of an 8-row tile from column 8)
    // (8-row gate+up tiles: the MMA's N is 16)
    constexpr int kAccCols = kCat ? (2 * NT > 32 ? 2 * NT : 32) : (NT < 16 ? 16 : NT);
    // CTA pairs with two MMA issuers: tensor memory holds one accumulator
    // pair (double-buffered), not one per issuer, so the issuers take the
    // chunks in turns and accumulate into the same one (below)
    constexpr bool kTurns = kPair && MMAW == 2;
    constexpr int kAccSets = kTurns ? 1 : MMAW;
    static_assert(kAccBase + 2 * kAccSets * kAccCols <= 512, "tensor memory budget");
    static_assert(STAGES >= kAB, "a stage must outlive its A buffer's reuse distance");
    static_assert(kStageBytes % 1024 == 0, "stage size must keep 1024-byte alignment");
    static_assert(STAGES % kDqGroups == 0, "each stage must belong to one dequant group");
    static_assert(kAB % kDqGroups == 0, "each A buffer must belong to one dequant group");
    static_assert(STAGES % NPROD == 0, "each stage must belong to one producer");
    // Each A buffer and each stage must also stay with one MMA issuer: an
    // issuer that took turns on a buffer with the other could wait on its
    // a_full barrier a whole phase ahead, where the parity test passes early
    // (a down-GEMM build with 5 A buffers and 2 issuers ran into exactly
    // that: its bounded waits gave up and reported MOE_ERR_DEVICE_TIMEOUT).
    // (Issuers that take turns never run ahead of each other.)
    static_assert(kTurns || (kAB % MMAW == 0 && STAGES % MMAW == 0),
                  "each A buffer must belong to one MMA warp");
    static_assert(!kPair || KIND == MOE_PACK_W13 || kCat,
                  "CTA pairs: the down GEMM's hi and lo rows split between the CTAs");
    // mbarrier arrivals: every dequant / epilogue thread of this CTA, or, on
    // CTA pairs, one per warp of both CTAs (on the even CTA's barriers)
    constexpr uint32_t kArrive = kPair ? 8u : 128u;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem *sm = reinterpret_cast<Smem *>(base + STAGES * kStageBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, g = blockIdx.x;
    const int R = a.N / kTileRows, KC = a.K / kChunkK;
    // CTA pairs: rank in the pair (0 issues the MMAs), pair index, pairs
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int gs = kPair ? g >> 1 : g, GS = kPair ? G >> 1 : G;

    // ---------------- setup
    if (warp == kMmaWarp) {
        if (kPair) {
            tmem_alloc_pair(&sm->tmem_base, kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&sm->tmem_base, kTmemCols);
            tmem_relinquish();
        }
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm->full[s], 1);
            mbar_init(&sm->consumed[s], 1);
        }
        for (int b = 0; b < kAB; ++b) mbar_init(&sm->a_full[b], kArrive);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm->acc_full[b], MMAW);
            mbar_init(&sm->acc_empty[b], kArrive);
        }
        mbar_init(&sm->done, MMAW);
        mbar_init(&sm->turn[0], 1);
        mbar_init(&sm->turn[1], 1);
        sm->dq_magic[0] = kMagic16;
        sm->dq_magic[1] = kMagic1024;
        sm->abort = 0;
        sm->bad = !header_ok(a.w, KIND, a.E, a.N, a.K);
        sm->wide = reinterpret_cast<const PackHeader *>(a.w)->wide_scales != 0;
        if (sm->bad && g == 0) set_status(a.ctrl, MOE_ERR_BAD_LAYOUT, KIND);
        fence_barrier_init();
    }
    if (warp == kProducerWarp && lane == 0) prefetch_tensormap(&tok);
    // The tile tables come from an earlier kernel of the call.  When that is
    // the kernel right before this one, wait for it to complete first.
    // Either way this kernel lets the next one start only after reading
    // them, and that one reads the same tables in its own set-up: every
    // kernel's early start follows the completion of all kernels before its
    // predecessor.
    if (a.tables_after_wait) pdl_wait();
    for (int i = tid; i <= a.E; i += kThreads) {
        sm->tile_prefix[i] = __ldg(a.tile_prefix + i);
        sm->offsets[i] = __ldg(a.offsets + i);
    }
    if (a.n_ovf > 0 && g == 0 && warp == 0) {
        int any = 0;
        for (int i = lane; i < a.n_ovf; i += 32) any |= a.ovf[i];
        if (__any_sync(0xffffffffu, any) && lane == 0) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 0);
    }
    tc_fence_before();
    __syncthreads();
    // the other CTA of a pair arrives on this one's barriers from now on
    if (kPair) cluster_sync();
    tc_fence_after();
    pdl_trigger();

    const uint32_t tb = sm->tmem_base;
    // Schedule.  With many tiles (at least 8 per CTA) each CTA takes whole
    // tiles g, g + G, g + 2G, ...: the CTAs then work on neighbouring tiles
    // at the same time, which share token rows (tiles of one token tile are
    // consecutive), so the token rows are read from L2, not DRAM.  With few
    // tiles, T = q G + rem: the chunks of tiles [0, rem) are cut into equal
    // contiguous shares (stream-K), which each CTA does first, and then it
    // takes q whole tiles rem + g, rem + g + G, ...  Every CTA thus ends on
    // a whole tile, whose epilogue needs no fix-up: the ticketed reductions
    // of split tiles happen while the other CTAs are still streaming.
    // (CTA pairs: work tiles of two weight tiles, always whole tiles
    // round-robin over the pairs)
    const int T = sm->bad ? 0 : sm->tile_prefix[a.E] * (R / CG);
    const bool rr = kPair || T >= 8 * G;
    const int q_whole = rr ? 0 : T / G;
    const int rem = rr ? 0 : T - q_whole * G;
    const int64_t W = (int64_t)rem * KC;  // stream-K units (tile * KC + chunk)
    const int64_t u_begin = range_begin(g, W, G), u_end = range_begin(g + 1, W, G);
    const int sk_chunks = (int)(u_end - u_begin);  // this CTA's stream-K chunks
    const int my_chunks = rr ? (gs < T ? (T - gs + GS - 1) / GS : 0) * KC : sk_chunks + q_whole * KC;
    // tile and K chunk of this CTA's chunk number c
    auto locate_chunk = [&](int c, int &tile, int &kc) {
        if (rr) {
            tile = gs + (c / KC) * GS;
            kc = c % KC;
        } else if (c < sk_chunks) {
            tile = (int)((u_begin + c) / KC);
            kc = (int)((u_begin + c) % KC);
        } else {
            tile = rem + g + ((c - sk_chunks) / KC) * G;
            kc = (c - sk_chunks) % KC;
        }
    };
    // end (exclusive) of the run of chunks that starts at c and stays in one
    // tile and one part of the schedule
    auto segment_end = [&](int c, int kc) {
        const int limit = (c < sk_chunks) ? sk_chunks : my_chunks;
        return c + min(KC - kc, limit - c);
    };

    if (warp >= kProducerWarp && warp < kMmaWarp) {
        // ---------------- TMA producers (the whole warp runs the loop, one
        // elected lane issues; a converged warp keeps the loop's values in
        // uniform registers, which the copy and MMA instructions want).
        // Every mbarrier wait costs a round trip of well over a hundred
        // cycles even when the phase is already complete, so one warp
        // alone cannot keep the HBM stream going; with two, producer pw
        // takes the chunks c with c % 2 == pw (and thereby its own stages).
        const int pw = warp - kProducerWarp;
        pdl_wait();  // token rows come from the previous kernel
        // Walk this producer's own chunks c = pw, pw + NPROD, ... keeping the
        // tile, K chunk, stage and stage phase incrementally: under the
        // dequantisation warps' load every instruction of this loop is slow
        // to issue, so it carries no per-chunk division or tile search.
        // An expert whose rows fit one token tile has its weights read once:
        // they go through L2 as evict-first, so that the token rows, which
        // every 128-row weight tile of their expert reads again, stay in L2
        // (without the hint, at M = 1024 on E = 384 the gate+up GEMM read
        // 1.86x its weight bytes from DRAM).  An expert with several token
        // tiles has its weights streamed again for each of them, by CTAs
        // working on its neighbouring tiles: those weights are kept in L2
        // (evict-last) for the next token tile (Zipf prefill M = 16384
        // 14.09 -> 13.35 ms, E = 128 M = 2048 979 -> 954 us in an A/B on one
        // GPU; decode and plateau batches unchanged).
        const uint64_t pol_first = policy_evict_first(), pol_keep = policy_evict_last();
        uint64_t pol_w = pol_first;
        int c = pw, kc = 0, s = pw, p0 = 0, tile = 0;
        uint32_t phase = 0;
        int64_t blk0 = 0;
        auto locate = [&]() {
            const Tile t = decode_tile<NT, CG>(a, sm, tile);
            // (a CTA pair: this CTA's weight tile of the two and, gate+up,
            // its half of the token rows)
            blk0 = ((int64_t)t.e * R + t.rt + (int)rank) * KC;
            p0 = t.p0 + ((kPair && KIND == MOE_PACK_W13) ? (int)rank * (pair_n(t.rows) / 2) : 0);
            pol_w = (sm->tile_prefix[t.e + 1] - sm->tile_prefix[t.e] > 1) ? pol_keep : pol_first;
        };
        if (c < my_chunks) {
            locate_chunk(c, tile, kc);
            locate();
        }
        // The loop is compiled once per schedule (a round-robin walk steps
        // to the tile G further on without a lookup).
        auto walk = [&](auto round_robin) {
            constexpr bool kRR = decltype(round_robin)::value;
            for (; c < my_chunks; c += NPROD) {
                if (!warp_wait_bar(&sm->consumed[s], phase ^ 1, &sm->abort, a.ctrl, 1)) break;
                if (elect_one()) {
                    // two copies per chunk: the weight block (codes and
                    // scales, contiguous) and the chunk's token rows
                    uint8_t *st = base + s * kStageBytes;
                    mbar_arrive_expect_tx(&sm->full[s], kStageBytes);
                    bulk_g2s_hint(st + kTokBoxes * kTokBox,
                                  a.w + kHeaderBytes + (blk0 + kc) * kBlockBytes, kBlockBytes,
                                  &sm->full[s], pol_w);
                    if (KIND == MOE_PACK_W13)
                        tma_load_3d(st, &tok, 0, p0, 2 * kc, &sm->full[s]);
                    else if (kPair)  // this CTA's hi (rank 0) or lo rows, K 0-63 then 64-127
                        tma_load_4d(st, &tok, 0, p0, (int)rank, 2 * kc, &sm->full[s]);
                    else if (kCat)  // [hi | lo] for K 0-63, then for K 64-127
                        tma_load_4d(st, &tok, 0, p0, 0, 2 * kc, &sm->full[s]);
                    else            // [hi K0-63 | hi K64-127 | lo K0-63 | lo K64-127]
                        tma_load_4d(st, &tok, 0, p0, 2 * kc, 0, &sm->full[s]);
                }
                __syncwarp();
                s += NPROD;
                if (s >= STAGES) {
                    s -= STAGES;
                    phase ^= 1;
                }
                // next chunk: K chunk + NPROD in the same tile unless that
                // leaves the tile or (stream-K) the stream-K part
                kc += NPROD;
                if constexpr (kRR) {
                    if (kc >= KC) {
                        do {
                            kc -= KC;
                            tile += GS;
                        } while (kc >= KC);
                        if (c + NPROD < my_chunks) locate();
                    }
                } else {
                    const int cn = c + NPROD;
                    if ((kc >= KC || (c < sk_chunks && cn >= sk_chunks)) && cn < my_chunks) {
                        locate_chunk(cn, tile, kc);
                        locate();
                    }
                }
            }
        };
        if (a.test_no_copies) {
            // failure-path test: no copy is issued (c stays below every
            // chunk of this producer, so nothing is left in flight)
        } else if (rr) {
            walk(std::true_type{});
        } else {
            walk(std::false_type{});
        }
        // Before the CTA exits, every copy issued must have landed; after an
        // abort elsewhere some were never consumed.  The last copy into each
        // stage is the only one that can be pending.  Chunks below c with
        // c % NPROD == pw are this producer's.
        for (int j = (c > STAGES ? c - STAGES : 0); j < c; ++j)
            if (j % NPROD == pw) wait_bar_final(&sm->full[j % STAGES], (j / STAGES) & 1);
        __syncwarp();
    } else if (warp >= kMmaWarp) {
        // ---------------- MMA issuers (converged warps, one elected lane
        // issues; the same lane every time, so its commits track its MMAs).
        // With two issuers, warp mw takes the chunks c with c % 2 == mw and
        // accumulates into its own accumulator; the epilogue adds the two.
        // A single issuer is limited by the issue rate of tcgen05.mma at
        // small N, not by the tensor pipe, so two of them go about twice
        // as fast there.  On CTA pairs the two issuers share one
        // accumulator and take turns: warp mw issues chunk c only after the
        // other one has issued chunk c - 1 (its arrival on turn[mw], after
        // a tcgen05 fence, orders those MMAs before these).  The waits and
        // the loop of one issuer then overlap the other one's MMA issue,
        // which a single issuer on a pair could not keep up with the
        // tensor pipe.
        const int mw = warp - kMmaWarp;
        // stage, A buffer and A-buffer phase of this warp's next chunk, kept
        // incrementally (STAGES and kAB are multiples of MMAW, or the
        // issuers take turns: a step of MMAW <= kAB chunks wraps b at most
        // once)
        int s = mw, b = mw;
        uint32_t bph = 0, tph = 0;
        const uint64_t desc_base = sdesc_k_sw128(smem_u32(base));
        int c = 0, seg = 0;  // c: CTA-local index of the segment's first chunk
        bool ok = true;
        // (the odd CTA of a pair issues nothing: the even one's MMAs cover both)
        while (c < my_chunks && ok && rank == 0) {
            int tile, k0;
            locate_chunk(c, tile, k0);
            const int k1 = k0 + (segment_end(c, k0) - c);
            const Tile t = decode_tile<NT, CG>(a, sm, tile);
            const int n_mma = kCat ? 2 * NT : (kPair ? pair_n(t.rows) : max(16, (t.rows + 15) & ~15));
            const uint32_t idesc = idesc_f16(kTileRows * CG, (uint32_t)n_mma);
            const int acc = seg & 1;
            if (!warp_wait_bar(&sm->acc_empty[acc], ((seg >> 1) & 1) ^ 1, &sm->abort, a.ctrl, 2))
                break;
            tc_fence_after();
            const uint32_t d_tmem = tb + kAccBase + (acc * kAccSets + (kTurns ? 0 : mw)) * kAccCols;
            const int c_end = c + (k1 - k0);
            bool first = true;
            for (int cc = c + ((mw - c % MMAW) + MMAW) % MMAW; cc < c_end; cc += MMAW) {
                if (!warp_wait_bar(&sm->a_full[b], bph, &sm->abort, a.ctrl, 3)) {
                    ok = false;
                    break;
                }
                if (kTurns && cc > 0) {
                    if (!warp_wait_bar(&sm->turn[mw], tph, &sm->abort, a.ctrl, 3)) {
                        ok = false;
                        break;
                    }
                    tph ^= 1;
                }
                tc_fence_after();
                if (elect_one()) {
                    // 8 MMAs (K = 16 each) over the chunk's A buffer and
                    // stage; a byte offset of the B start address adds
                    // offset >> 4 to the descriptor.  One commit then frees
                    // both.
                    const uint64_t desc0 = desc_base + (uint64_t)((s * kStageBytes) >> 4);
                    const uint32_t a_tmem = tb + b * kACols;
#pragma unroll
                    for (int j = 0; j < kChunkK / 16; ++j) {
                        // (taking turns, the tile's first chunk starts the
                        // shared accumulator)
                        const uint32_t acc_flag = (kTurns ? cc != c : !first) || j > 0 ? 1u : 0u;
                        if (kPair) {  // each CTA's stage: its token rows, K 0-63 then 64-127
                            const uint32_t boff = (j >> 2) * kTokBox + (j & 3) * 32;
                            mma_f16_ts_pair(d_tmem, a_tmem + j * 8, desc0 + (boff >> 4), idesc,
                                            acc_flag);
                        } else if (kCat) {
                            const uint32_t boff = (j >> 2) * 2 * kTokBox + (j & 3) * 32;
                            mma_f16_ts(d_tmem, a_tmem + j * 8, desc0 + (boff >> 4), idesc,
                                       acc_flag);
                        } else {
                            const uint32_t boff = (j >> 2) * kTokBox + (j & 3) * 32;
                            mma_f16_ts(d_tmem, a_tmem + j * 8, desc0 + (boff >> 4), idesc,
                                       acc_flag);
                            if (KIND == MOE_PACK_W2)
                                mma_f16_ts(d_tmem, a_tmem + j * 8,
                                           desc0 + ((2 * kTokBox + boff) >> 4), idesc, 1u);
                        }
                    }
                    if (kPair)
                        tc_commit_pair(&sm->consumed[s]);
                    else
                        tc_commit(&sm->consumed[s]);
                    if (kTurns) {
                        tc_fence_before();
                        mbar_arrive(&sm->turn[mw ^ 1]);
                    }
                }
                __syncwarp();
                first = false;
                s += MMAW;
                if (s >= STAGES) s -= STAGES;
                b += MMAW;
                if (b >= kAB) {
                    b -= kAB;
                    bph ^= 1;
                }
            }
            if (!ok) break;
            // an issuer with no chunk in this segment still arrives (its
            // accumulator is then not read; taking turns, the commit of
            // each issuer covers its own MMAs of the shared one)
            if (elect_one()) {
                if (kPair)
                    tc_commit_pair(&sm->acc_full[acc]);
                else
                    tc_commit(&sm->acc_full[acc]);
            }
            __syncwarp();
            c = c_end;
            ++seg;
        }
        // Every MMA issued has completed once `done` fires (on CTA pairs the
        // even CTA's commit arrives in both).
        if (elect_one()) {
            if (!kPair)
                tc_commit(&sm->done);
            else if (rank == 0)
                tc_commit_pair(&sm->done);
            wait_bar_final(&sm->done, 0);
        }
        __syncwarp();
    } else if (warp >= kEpiWarps) {
        // ---------------- dequantisation warpgroups
        const int grp = (warp - kEpiWarps) / 4;
        const bool wide = sm->wide != 0;
        const int r = (warp & 3) * 32 + lane;  // weight row of the tile = TMEM lane
        const DqMagic mg = load_dq_magic(sm->dq_magic);
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        // stage, its phase and the A buffer of this group's next chunk, kept
        // incrementally (STAGES and kAB are multiples of kDqGroups)
        int s = grp, b = grp;
        uint32_t ph = 0;
        for (int c = grp; c < my_chunks; c += kDqGroups) {
            if (!warp_wait_bar(&sm->full[s], ph, &sm->abort, a.ctrl, 4)) break;
            // A buffer b was last read by the MMAs of chunk c - kAB, whose
            // stage is kAB stages back
            if (c >= kAB) {
                const int sp = s >= kAB ? s - kAB : s - kAB + STAGES;
                const uint32_t pp = s >= kAB ? ph : ph ^ 1;
                if (!warp_wait_bar(&sm->consumed[sp], pp, &sm->abort, a.ctrl, 5)) break;
            }
            tc_fence_after();
            const uint8_t *st = base + s * kStageBytes + kTokBoxes * kTokBox;
            const uint32_t st_s = smem_u32(st);
            uint2 sc;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(sc.x), "=r"(sc.y) : "r"(st_s + kCodeBlockBytes + r * 8));
            const uint32_t scw[2] = {sc.x, sc.y};
            const uint32_t a_addr = tb + lane_off + b * kACols;
            // one 32-element scale group per piece: load, dequantise, store
            // the piece's 16 columns of the A buffer
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
                    uint32_t v[16];
                    uint32_t o[4];
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
            if (wide)
                pieces(std::false_type{});
            else
                pieces(std::true_type{});
            tc_wait_st();
            tc_fence_before();
            if (kPair) {
                // one arrival per warp, on the even CTA's barrier
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive(&sm->a_full[b]);
                    else
                        mbar_arrive_remote(&sm->a_full[b], 0);
                }
            } else {
                mbar_arrive(&sm->a_full[b]);
            }
            s += kDqGroups;
            if (s >= STAGES) {
                s -= STAGES;
                ph ^= 1;
            }
            b += kDqGroups;
            if (b >= kAB) b -= kAB;
        }
    } else {
        // ---------------- epilogue warpgroup (warps 0-3)
        const int r = warp * 32 + lane;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        float *part = a.partials;
        int seg = 0;
        for (int c_seg = 0; c_seg < my_chunks; ++seg) {
            int tile, k0;
            locate_chunk(c_seg, tile, k0);
            const int k1 = k0 + (segment_end(c_seg, k0) - c_seg);
            const Tile t = decode_tile<NT, CG>(a, sm, tile);
            const int acc = seg & 1;
            if (!warp_wait_bar(&sm->acc_full[acc], (seg >> 1) & 1, &sm->abort, a.ctrl, 6)) break;
            const int rt = t.rt + (int)rank;  // this CTA's weight tile
            tc_fence_after();
            const uint32_t acc_addr = tb + lane_off + kAccBase + acc * kAccSets * kAccCols;
            // with two issuers, the second one had a chunk here unless the
            // segment is a single chunk that fell to the first (and vice versa)
            bool has[2] = {true, true};
            if (kAccSets == 2 && k1 - k0 == 1) {
                has[0] = (c_seg % 2 == 0);
                has[1] = !has[0];
            }
            const bool whole = (k0 == 0 && k1 == KC);
            const int which = (c_seg == 0) ? 0 : 1;  // first or last segment of this CTA
            float *slot = part + ((size_t)g * 2 + which) * (size_t)NT * kTileRows;
#pragma unroll 1
            for (int c0 = 0; c0 < t.rows; c0 += 16) {
                // valid token columns of this block of 16 (warp-uniform); the
                // loops below stop there, so a tile with a few rows costs a
                // few columns of work
                const int nval = min(16, t.rows - c0);
                // Sum of the issuers' accumulators (and, with stacked hi/lo
                // rows, of both halves), always in the same order.
                uint32_t v[16];
                bool any = false;
#pragma unroll
                for (int w = 0; w < kAccSets; ++w) {
                    if (!has[w]) continue;
                    uint32_t x[16];
                    tmem_ld16(acc_addr + w * kAccCols + c0, x);
                    if (kCat) {  // add the lo half, NT columns further on
                        uint32_t lo[16];
                        tmem_ld16(acc_addr + w * kAccCols + NT + c0, lo);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            x[j] = __float_as_uint(__uint_as_float(x[j]) + __uint_as_float(lo[j]));
                    } else {
                        tc_wait_ld();
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = any ? __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(x[j])) : x[j];
                    any = true;
                }
                if (whole) {
                    {
                        if (KIND == MOE_PACK_W13) {
                            // even lanes write hi, odd lanes lo, of act
                            // column rt*64 + r/2
                            uint16_t *dst = ((lane & 1) ? a.act_lo : a.act_hi) +
                                            (size_t)(t.p0 + c0) * a.I + rt * (kTileRows / 2) +
                                            (r >> 1);
                            bool overflow = false;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if (j >= nval) break;
                                dst[(size_t)j * a.I] =
                                    silu_mul_half(__uint_as_float(v[j]), lane, overflow);
                            }
                            if (overflow) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 1);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if (j >= nval) break;
                                a.y[(size_t)(t.p0 + c0 + j) * a.N + rt * kTileRows + r] =
                                    __uint_as_float(v[j]);
                            }
                        }
                    }
                } else {
                    // partial sums of the valid columns (the reduction reads
                    // no others)
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j >= nval) break;
                        slot[(size_t)(c0 + j) * kTileRows + r] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            if (kPair) {
                // one arrival per warp, on the even CTA's barrier
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0)
                        mbar_arrive(&sm->acc_empty[acc]);
                    else
                        mbar_arrive_remote(&sm->acc_empty[acc], 0);
                }
            } else {
                mbar_arrive(&sm->acc_empty[acc]);
            }

            if (!whole) {
                // Fixed-order reduction by whichever CTA finishes the tile
                // last; each warp handles its own 32 rows with its own ticket.
                // An earlier kernel of the call (the hidden-row gather)
                // zeroes the tickets: this atomic must stay ordered after the
                // producers' griddepcontrol.wait, which it is through the
                // full -> MMA -> acc_full chain that led here.
                const int64_t tu0 = (int64_t)tile * KC, tu1 = tu0 + KC - 1;
                const int ncontrib = contributors(tu0, tu1, W, G);
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = (atomicAdd(a.tickets + (size_t)tile * 4 + warp, 1) == ncontrib - 1);
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
#pragma unroll 1
                    for (int col = 0; col < t.rows; ++col) {
                        float sum = 0.f;
                        for (int gg = unit_owner(tu0, W, G);; gg = unit_owner(range_begin(gg + 1, W, G), W, G)) {
                            const int wh = (range_begin(gg, W, G) >= tu0) ? 0 : 1;
                            const float *sl = part + ((size_t)gg * 2 + wh) * (size_t)NT * kTileRows;
                            sum += __ldcg(sl + (size_t)col * kTileRows + r);
                            if (range_begin(gg + 1, W, G) > tu1) break;
                        }
                        if (KIND == MOE_PACK_W13) {
                            bool overflow = false;
                            const uint16_t val = silu_mul_half(sum, lane, overflow);
                            ((lane & 1) ? a.act_lo : a.act_hi)[(size_t)(t.p0 + col) * a.I +
                                                               t.rt * (kTileRows / 2) + (r >> 1)] = val;
                            if (overflow) set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 1);
                        } else {
                            a.y[(size_t)(t.p0 + col) * a.N + t.rt * kTileRows + r] = sum;
                        }
                    }
                }
            }
            c_seg += k1 - k0;
        }
    }

    // ---------------- teardown
    tc_fence_before();
    __syncthreads();
    // no arrival of one CTA of a pair may reach the other after it exits
    if (kPair) cluster_sync();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tb, kTmemCols);
        else
            tmem_dealloc(tb, kTmemCols);
    }
}

using KernelFn = void (*)(const TcArgs, const CUtensorMap);

template <int KIND, int NT, int CG = 1>
struct Config {
    // (CTA pairs: this CTA's half of the token operand per stage)
    static constexpr bool kPair = CG == 2;
    static constexpr int kTokRows = (kPair && KIND == MOE_PACK_W13) ? NT / 2 : NT;
    static constexpr int kTokBoxes = (KIND == MOE_PACK_W2 && !kPair) ? 4 : 2;
    static constexpr int kStage = kTokBoxes * kTokRows * 128 + kBlockBytes;
    static constexpr int kBudget = 210 * 1024;
    // An even stage count keeps every shared-memory stage with one dequant
    // warpgroup (chunk c and chunk c + kStages have the same parity), so a
    // warpgroup always waits on the phase right after the one it consumed
    // and the parity test of the mbarrier cannot alias an older phase.
    static constexpr int kFit = (kBudget / kStage) < kMaxStages ? (kBudget / kStage) : kMaxStages;
    // Gate+up GEMM with small token tiles: 6 dequant warpgroups (1024
    // threads, 64 registers each) over 12 stages.  The dequantisation is
    // instruction-issue bound there, and 24 instead of 16 dequant warps issue
    // more of the time (decode M = 90: 1026 -> 976 us); the down GEMM, whose
    // epilogue needs more registers, spilled at 64 and stays at 4 groups.
    static constexpr bool kWide = KIND == MOE_PACK_W13 && NT <= 32 && kFit >= 12;
    // 160-column accumulators (160-row gate+up, 80-row down tiles, CTA
    // pairs): 6 stages of 29 KiB, 3 dequant warpgroups, whose 3 A buffers
    // leave room for the two accumulators
    static constexpr bool k160 = NT == 160 || NT == 80;
    // (18 stages of the 8-row gate+up tiles' 11 KiB)
    static constexpr int kStages = kWide ? (kFit >= 18 ? 18 : 12) : (k160 ? 6 : (kFit & ~1));
    // Warp roles.  Each mbarrier wait costs a shared-memory round trip of
    // over a hundred cycles even when the phase is complete, and every
    // instruction of the small control loops waits behind the dequantisation
    // warps' arithmetic, so the control roles are split over several warps
    // whose waits overlap:
    //  * four dequantisation warpgroups (each stage stays with one of them,
    //    which needs a stage count divisible by four), else two, or six over
    //    12 stages in the gate+up GEMM with small token tiles (below);
    //  * two TMA producers (each owns every other stage);
    //  * two MMA issuers where N is small enough for the issue rate of
    //    tcgen05.mma, not the tensor pipe, to limit, and their
    //    accumulators fit next to the A buffers in tensor memory; for the
    //    gate+up GEMM on CTA pairs two issuers that take turns on one
    //    accumulator (E128 M = 2048 gate+up 360 -> 352 us, Zipf prefill
    //    M = 4096 / 16384 -1% to -5%; on the down GEMM's pairs the extra
    //    warp cost 1-2%, so it keeps one issuer there).
    static constexpr int kDq = kWide ? 6 : (k160 ? 3 : ((kStages % 4 == 0) ? 4 : 2));
    static constexpr int kAB = a_buffers(NT, kStages, kDq);
    static constexpr int kAccCols = (KIND == MOE_PACK_W2 && (NT <= 64 || NT == 80))
                                        ? (2 * NT > 32 ? 2 * NT : 32) : (NT < 16 ? 16 : NT);
    // (two issuers with accumulators of their own need the A buffers and
    // stages to split evenly between them)
    static constexpr int kMma = (CG == 2) ? (KIND == MOE_PACK_W13 ? 2 : 1)
                                          : ((kAccCols <= 64 &&
                                              kAB * kACols + 4 * kAccCols <= (int)kTmemCols &&
                                              kAB % 2 == 0 && kStages % 2 == 0)
                                                 ? 2 : 1);
    static constexpr int kProd = 2;
    static constexpr int kThreads = threads_for(kDq, kProd, kMma);
    static_assert(kStages >= 2 && kStages % kDq == 0, "stage count must be a multiple of the dequant groups");
    // The kernel is persistent with one CTA per SM and allocates all of
    // tensor memory: asking for more than half of an SM's shared memory
    // keeps the scheduler from ever placing two of its CTAs on one SM (the
    // second would stall in tcgen05.alloc until the first finished).
    static constexpr size_t kMinSmem = 120 * 1024;
    static constexpr size_t kNeed = (size_t)kStages * kStage + sizeof(Smem) + 1024;
    static constexpr size_t kSmem = kNeed > kMinSmem ? kNeed : kMinSmem;
    static KernelFn fn() { return gemm_tc_kernel<KIND, NT, kStages, kDq, kProd, kMma, CG>; }
};

template <int KIND, int NT, int CG>
bool pick_cfg(KernelFn *fn, size_t *smem, int *threads) {
    *fn = Config<KIND, NT, CG>::fn();
    *smem = Config<KIND, NT, CG>::kSmem;
    *threads = Config<KIND, NT, CG>::kThreads;
    return true;
}

// (the CTA-pair kernels exist for the tile widths tc_pair_mode names)
template <int KIND, int NT>
bool pick_nt(bool pair, KernelFn *fn, size_t *smem, int *threads) {
    if constexpr ((KIND == MOE_PACK_W13 && NT >= 128) || (KIND == MOE_PACK_W2 && NT == 64)) {
        if (pair) return pick_cfg<KIND, NT, 2>(fn, smem, threads);
    }
    return pick_cfg<KIND, NT, 1>(fn, smem, threads);
}

template <int KIND>
bool pick(int nt, bool pair, KernelFn *fn, size_t *smem, int *threads) {
    switch (nt) {
        case 8: return pick_cfg<KIND, 8, 1>(fn, smem, threads);  // decode batches
        case 16: return pick_nt<KIND, 16>(pair, fn, smem, threads);
        case 32: return pick_nt<KIND, 32>(pair, fn, smem, threads);
        case 64: return pick_nt<KIND, 64>(pair, fn, smem, threads);
        case 128: return pick_nt<KIND, 128>(pair, fn, smem, threads);
        case 80:  // down only, always on CTA pairs
            if constexpr (KIND == MOE_PACK_W2) {
                if (pair) return pick_cfg<KIND, 80, 2>(fn, smem, threads);
            }
            return false;
        case 160:  // gate+up only, always on CTA pairs
            if constexpr (KIND == MOE_PACK_W13) {
                if (pair) return pick_cfg<KIND, 160, 2>(fn, smem, threads);
            }
            return false;
    }
    return false;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool make_token_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)(rows > 0 ? rows : 1), (cuuint64_t)cols / 64};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_act_map(CUtensorMap *map, const void *hi, const void *lo, int rows, int cols,
                  int box_rows, bool stacked, bool one_half) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const uintptr_t h = reinterpret_cast<uintptr_t>(hi), l = reinterpret_cast<uintptr_t>(lo);
    if (l <= h || (l - h) % 16) return false;
    const cuuint64_t r = (cuuint64_t)(rows > 0 ? rows : 1), kh = (cuuint64_t)cols / 64;
    const cuuint64_t row_b = (cuuint64_t)cols * 2, half_b = l - h;
    // dimension 0: 64 columns; 1: rows; then (hi/lo, K half) or (K half, hi/lo)
    cuuint64_t dims[4] = {64, r, stacked ? 2 : kh, stacked ? kh : 2};
    cuuint64_t strides[3] = {row_b, stacked ? half_b : 128, stacked ? 128 : half_b};
    cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (one_half && stacked) ? 1u : 2u, 2};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(hi), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int tc_grid(int device) {
    static int sms[64] = {0};
    if (device < 0 || device >= 64) return 0;
    if (!sms[device]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        sms[device] = v;
    }
    return sms[device];
}

cudaError_t launch_gemm_tc(const TcArgs &args, const CUtensorMap &tok, int grid, cudaStream_t s,
                           bool pdl) {
    KernelFn fn = nullptr;
    size_t smem = 0;
    int threads = 0;
    const bool pair = tc_pair_mode(args.kind, args.nt, args.N);
    const bool ok = (args.kind == MOE_PACK_W13)
                        ? pick<MOE_PACK_W13>(args.nt, pair, &fn, &smem, &threads)
                        : pick<MOE_PACK_W2>(args.nt, pair, &fn, &smem, &threads);
    if (!ok) return cudaErrorInvalidValue;
    if (pair) grid &= ~1;  // whole CTA pairs
    if (grid < 1) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (pdl) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    if (pair) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 2;
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, fn, args, tok);
}

}  // namespace moe
