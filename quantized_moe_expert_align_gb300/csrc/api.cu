// api.cu -- the C ABI: argument validation, workspace carving and the
// stream-ordered launch sequence of the MoE layer forward.
#include <climits>
#include <cstdlib>
#include <cstring>

#include "decode.h"
#include "elementwise.h"
#include "gemm_tc.h"
#include "moe_internal.h"
#include "route.cuh"
#include "small_align.cuh"

namespace moe {

constexpr int kMaxGrid = 256;  // bound on the GEMM grid used to size workspaces

static bool decode_kernel_enabled();

// Rows per active expert if routing spreads the n slots evenly (rounded up).
static int rows_per_active_expert(int64_t n, int E) {
    const int64_t active = n < E ? (n > 0 ? n : 1) : E;
    return (int)((n + active - 1) / active);
}

int pick_token_tile(int n, int E) {
    // Test override: MOE_W4A16_TOKEN_TILE = 16, 32, 64, 128 or 160.
    static const int forced = [] {
        const char *v = std::getenv("MOE_W4A16_TOKEN_TILE");
        const int t = v ? std::atoi(v) : 0;
        return (t == 16 || t == 32 || t == 64 || t == 128 || t == 160) ? t : 0;
    }();
    if (forced) return forced;
    // At most 3 rows per active expert (decode batches) and at least 32
    // slots: 8-row tiles, whose 11 KiB stages (2 KiB of token rows next to
    // the 9 KiB weight block) leave room for 18 stages where 16-row tiles
    // fit 12, so more weight bytes stay in flight (E = 384 M = 90 gate+up
    // GEMM 858 -> 827 us, M = 9 180 -> 178 us; at M = 1, 8 slots, 34.8 ->
    // 36.8 us, so the smallest batches keep 16 rows).  (The opt-in single
    // small-batch kernel takes 16-row tiles.)
    if (n >= 32 && rows_per_active_expert(n, E) <= 3 &&
        !(decode_kernel_enabled() && n <= kDecodeMaxSlots))
        return 8;
    // Rows per active expert if routing spreads the slots evenly.  The tile
    // is sized for about 1.25x that, so that most experts' rows fit in one
    // tile (every extra token tile streams the expert's weights again), but
    // stays at 64 rows below 256 rows per expert: 128-row token tiles leave
    // room for only four (gate+up) or two (down) shared-memory stages, and
    // one 128-row tile per SM no longer fits in L2 at once.  Measured on the
    // E = 128 / E = 384 workloads: 32 beats 16 at 16 rows per expert, 64
    // beats 128 at 85 and 128 rows, 128 wins at 341; at 22 rows 32 beats 64.
    const int avg = rows_per_active_expert(n, E);
    const int want = avg + avg / 4;
    int nt = 16;
    while (nt < want && nt < 128) nt <<= 1;
    // Beyond 128 rows the gate+up GEMM takes 160-row tiles (on CTA pairs,
    // 80 rows in each SM): at E = 128 M = 2048 (128 +- 11 rows per expert)
    // a third of the 128-row tiles were second tiles of a few rows, each
    // dequantising the expert's whole weight tile for a narrow MMA.
    if (nt == 128 && want > 128) nt = 160;
    return nt;
}

// Failure-path test switch, read once per process:
// MOE_W4A16_TEST_NO_COPIES=1 makes the gate+up GEMM issue no copies, so its
// bounded waits run out and the call reports MOE_ERR_DEVICE_TIMEOUT.
static int test_no_copies() {
    static const int v = [] {
        const char *e = std::getenv("MOE_W4A16_TEST_NO_COPIES");
        return (e && std::atoi(e) == 1) ? 1 : 0;
    }();
    return v;
}

// Opt-in switch, read once per process: MOE_W4A16_DECODE_FUSED=1 runs
// batches of at most kDecodeMaxSlots slots (16-row token tiles) as the single
// small-batch kernel.  Off by default: on one GB300 that kernel measured
// slower than the four kernels of the small-batch path (E = 384, M = 1 / 9:
// 74 / 330 us against 62 / 285 us), its prologue and grid barrier costing
// about 10 us and its weight stream running slower per 128-element chunk
// than the separate GEMMs'.
static bool decode_kernel_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("MOE_W4A16_DECODE_FUSED");
        return v && std::atoi(v) == 1;
    }();
    return on;
}

bool use_decode_kernel(int64_t n, int nt) {
    return decode_kernel_enabled() && n > 0 && n <= kDecodeMaxSlots && nt == kDecodeTokenTile;
}

// The down GEMM's stage holds both halves (hi, lo) of its token rows, so a
// 128-row tile leaves room for only two stages.  Under 128- and 160-row
// gate+up tiles it takes 80-row tiles on CTA pairs (each CTA the hi or the
// lo rows) when its weight tiles come in pairs, else 64-row tiles.  On one
// GB300, 80 against 64 rows: E = 128 M = 1024 (64 rows per expert) down
// GEMM 206 -> 168 us, M = 2048 332 -> 315 us, Zipf prefill M = 16384
// 5.32 -> 5.02 ms, E = 384 M = 4096 1.78 -> 1.76 ms.
int down_token_tile(int nt, int H, int64_t n, int E) {
    static const bool forced = std::getenv("MOE_W4A16_TOKEN_TILE") != nullptr;
    if (nt == 160 || (nt == 128 && !forced)) return tc_pair_mode(MOE_PACK_W2, 80, H) ? 80 : 64;
    // At most 3 rows per active expert (decode batches): 8-row down tiles.
    // A stage then holds 4 KiB of hi and lo rows next to the 9 KiB weight
    // block, so 16 stages fit where the 16-row tiles' 17 KiB stages left
    // room for 12, and the weight stream keeps more bytes in flight (12 -> 8
    // stages of the 16-row tiles cost 7% at decode M = 9 and 90).
    if (!forced && nt <= 16 && rows_per_active_expert(n, E) <= 3) return 8;
    return (forced || nt <= 64) ? nt : 64;
}

AlignLayout align_layout(int M, int k, int E) {
    AlignLayout l;
    l.ctrl = 0;
    l.seg_counts = l.seg_base = 0;
    size_t off = sizeof(Ctrl);
    if (align_large((int64_t)M * k)) {
        const size_t seg = (size_t)E * kAlignSegs * 4;
        l.seg_counts = off;
        off = align_up(off + seg, 256);
        l.seg_base = off;
        off = align_up(off + seg, 256);
    }
    l.total = off;
    return l;
}

FwdLayout fwd_layout(int M, int k, int E, int H, int I) {
    const size_t n = (size_t)M * k;
    FwdLayout l;
    l.nt = pick_token_tile((int)n, E);
    l.fused = use_decode_kernel((int64_t)n, l.nt);
    // (the single small-batch kernel takes 16-row tiles in both GEMMs)
    l.nt2 = l.fused ? l.nt : down_token_tile(l.nt, H, (int64_t)n, E);
    l.max_tok_tiles = (int)(n / l.nt) + (n < (size_t)E ? (int)n : E) + 1;
    l.max_tok_tiles2 = (int)(n / l.nt2) + (n < (size_t)E ? (int)n : E) + 1;
    l.grid = kMaxGrid;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    l.ctrl = take(sizeof(Ctrl));
    l.seg_counts = l.seg_base = 0;
    if (align_large((int64_t)n)) {
        l.seg_counts = take((size_t)E * kAlignSegs * 4);
        l.seg_base = take((size_t)E * kAlignSegs * 4);
    }
    l.counts = take((size_t)E * 4);
    l.offsets = take((size_t)(E + 1) * 4);
    l.tile_prefix = take((size_t)(E + 1) * 4);
    l.tile_prefix2 = take((size_t)(E + 1) * 4);
    l.perm = take(n * 4);
    l.inv_perm = take(n * 4);
    // one ticket per (tile, epilogue warp); the single small-batch kernel
    // also keeps its activation-ready flags and combine tickets there, and
    // the partials of both GEMMs
    l.tickets = l.fused ? take((size_t)decode_sync_ints(l.max_tok_tiles, H, I) * 4)
                        : take(((size_t)l.max_tok_tiles * (2 * I / kTileRows) +
                                (size_t)l.max_tok_tiles2 * (H / kTileRows)) * 4 * 4);
    l.partials = take((size_t)(l.fused ? 2 : 1) * l.grid * 2 * l.nt * kTileRows * 4);
    l.ovf = take((size_t)kMaxGrid * 4);
    l.xs = take(n * H * 2);
    l.act_hi = take(n * I * 2);
    l.act_lo = take(n * I * 2);
    l.y = take(n * H * 4);
    l.total = off;
    return l;
}

namespace {

// Per host thread: calls from several threads (or for several devices from
// several threads) never write the same record.
thread_local moe_diag_t g_diag = {2, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t check_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_UNSUPPORTED_DEVICE;
    }
    static int support[64] = {0};  // 0 unknown, 1 supported, 2 not
    if (dev >= 0 && dev < 64 && support[dev]) return support[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_UNSUPPORTED_DEVICE;
    }
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < 64) support[dev] = ok ? 1 : 2;
    return ok ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

bool routing_sizes_ok(int M, int k, int E) {
    return M >= 0 && k >= 1 && k <= 64 && E >= 1 && E <= 1024 && (int64_t)M * k < INT_MAX;
}

// What precedes the alignment kernel(s) of `a` (whose ids must be topk_ids
// when logits are given).  The single-CTA alignment kernel clears the status
// word itself and routes small batches; otherwise the status word is cleared
// by a memset first, then route_kernel routes (if logits are given), and the
// alignment leaves the word alone.  Sets *route_kernel when it launched one.
cudaError_t begin_call(AlignArgs &a, const float *logits, int M, int k, int32_t *topk_ids,
                       float *topk_w, cudaStream_t s, bool *route_kernel = nullptr) {
    const bool large = a.seg_counts != nullptr;
    if (route_kernel) *route_kernel = false;
    a.logits = nullptr;
    if (!large && (!logits || (M <= kFusedRouteMaxM && route_vpl(a.E) <= kAlignRouteMaxVpl))) {
        if (logits) {
            a.logits = logits;
            a.route_M = M;
            a.route_k = k;
            a.route_ids = topk_ids;
            a.route_w = topk_w;
        }
        a.reset_status = 1;
        return cudaSuccess;
    }
    a.reset_status = 0;
    cudaError_t err = cudaMemsetAsync(a.ctrl, 0, 4 * sizeof(int32_t), s);
    if (err != cudaSuccess || !logits) return err;
    if (route_kernel) *route_kernel = true;
    RouteArgs r = {logits, M, a.E, k, topk_ids, topk_w, a.ctrl};
    return launch_route(r, s);
}

// The large-batch workspace arrays of an alignment, when it takes that path.
void set_segments(AlignArgs &a, uint8_t *ws, size_t seg_counts, size_t seg_base) {
    const bool large = align_large(a.n);
    a.seg_counts = large ? reinterpret_cast<int32_t *>(ws + seg_counts) : nullptr;
    a.seg_base = large ? reinterpret_cast<int32_t *>(ws + seg_base) : nullptr;
}

bool layer_sizes_ok(int M, int k, int E, int H, int I) {
    return routing_sizes_ok(M, k, E) && H > 0 && I > 0 && H % kChunkK == 0 &&
           I % kChunkK == 0 && H <= (1 << 20) && I <= (1 << 20) &&
           (int64_t)M * k * H < ((int64_t)1 << 40);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer or size out of range";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: pointer below its required alignment";
        case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
        case MOE_ERR_BAD_LAYOUT: return "MOE_ERR_BAD_LAYOUT: prepacked buffer header does not match";
        case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE: needs an sm_103 GPU";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA runtime call failed";
        case MOE_ERR_DEVICE_BAD_EXPERT_ID: return "MOE_ERR_DEVICE_BAD_EXPERT_ID: expert id outside [0, E)";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
        case MOE_ERR_DEVICE_FP16_RANGE: return "MOE_ERR_DEVICE_FP16_RANGE: value not representable in fp16";
        case MOE_ERR_DEVICE_BAD_LOGIT: return "MOE_ERR_DEVICE_BAD_LOGIT: a router logit is NaN or +inf";
    }
    return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_w4a16_prepack_size(int kind, int E, int N, int K, int group, size_t *bytes) {
    if (bytes) *bytes = 0;
    if (!bytes) return MOE_ERR_INVALID_ARG;
    if ((kind != MOE_PACK_W13 && kind != MOE_PACK_W2) ||
        (group != 32 && group != 64 && group != 128) || E < 1 || N <= 0 ||
        K <= 0 || N % kTileRows || K % kChunkK || N > (1 << 20) || K > (1 << 20))
        return MOE_ERR_INVALID_ARG;
    *bytes = packed_bytes(E, N, K);
    return MOE_OK;
}

moe_status_t moe_w4a16_prepack(int kind, const uint8_t *q_canon, const uint16_t *scales, int E,
                               int N, int K, int group, void *dst, size_t dst_bytes,
                               moe_stream_t stream) {
    size_t need = 0;
    moe_status_t st = moe_w4a16_prepack_size(kind, E, N, K, group, &need);
    if (st != MOE_OK) return st;
    if (!q_canon || !scales || !dst) return MOE_ERR_INVALID_ARG;
    if (!aligned(q_canon, 16) || !aligned(scales, 16) || !aligned(dst, 256))
        return MOE_ERR_MISALIGNED;
    if (dst_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((st = check_device()) != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    PackHeader h;
    std::memset(&h, 0, sizeof h);
    h.magic = kPackMagic;
    h.version = kPackVersion;
    h.kind = (uint32_t)kind;
    h.block_bytes = kBlockBytes;
    h.E = E;
    h.N = N;
    h.K = K;
    h.group = kGroup;  // the packed blocks always hold one scale per 32 elements
    h.source_group = group;
    h.status = MOE_OK;
    uint8_t *d = static_cast<uint8_t *>(dst);
    // a scale outside the exact range sets the header's status, which makes
    // every later forward reject the buffer
    int32_t *flag = &reinterpret_cast<PackHeader *>(d)->status;
    int32_t *wide = &reinterpret_cast<PackHeader *>(d)->wide_scales;
    if (cudaMemcpyAsync(d, &h, sizeof h, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        launch_prepack_codes(kind, q_canon, E, N, K, d, s) != cudaSuccess ||
        launch_prepack_scales(kind, scales, E, N, K, group, d, flag, wide, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    int32_t dev_status = 0;
    if (cudaMemcpy(&dev_status, flag, sizeof dev_status, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return dev_status == MOE_OK ? MOE_OK : MOE_ERR_DEVICE_FP16_RANGE;
}

size_t moe_align_workspace_size(int M, int k, int E) {
    if (!routing_sizes_ok(M, k, E)) return 0;
    return align_layout(M, k, E).total;
}

moe_status_t moe_align(const int32_t *ids, int M, int k, int E, int32_t *counts, int32_t *offsets,
                       int32_t *perm, int32_t *inv_perm, void *workspace, size_t ws_bytes,
                       moe_stream_t stream) {
    if (!routing_sizes_ok(M, k, E)) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !workspace || (M > 0 && (!ids || !perm))) return MOE_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4) ||
        !aligned(inv_perm, 4) || !aligned(workspace, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < align_layout(M, k, E).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    moe_status_t st = check_device();
    if (st != MOE_OK) return st;
    AlignArgs a = {};
    a.ids = ids;
    a.n = M * k;
    a.E = E;
    a.reset_status = 1;
    a.token_tile = 0;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.inv_perm = inv_perm;
    a.tile_prefix = nullptr;
    const AlignLayout L = align_layout(M, k, E);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.ctrl = reinterpret_cast<Ctrl *>(ws + L.ctrl);
    set_segments(a, ws, L.seg_counts, L.seg_base);
    if (begin_call(a, nullptr, M, k, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream)) !=
            cudaSuccess ||
        launch_align(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status_t moe_route_align(const float *logits, int M, int k, int E, int32_t *topk_ids,
                             float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm,
                             int32_t *inv_perm, void *workspace, size_t ws_bytes,
                             moe_stream_t stream) {
    if (!routing_sizes_ok(M, k, E) || k > E) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !workspace ||
        (M > 0 && (!logits || !topk_ids || !topk_w || !perm)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) ||
        !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4) ||
        !aligned(inv_perm, 4) || !aligned(workspace, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < align_layout(M, k, E).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    moe_status_t st = check_device();
    if (st != MOE_OK) return st;
    const AlignLayout L = align_layout(M, k, E);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(ws + L.ctrl);
    AlignArgs a = {};
    a.ids = topk_ids;
    a.n = M * k;
    a.E = E;
    a.counts = counts;
    a.offsets = offsets;
    a.perm = perm;
    a.inv_perm = inv_perm;
    a.ctrl = ctrl;
    set_segments(a, ws, L.seg_counts, L.seg_base);
    if (begin_call(a, logits, M, k, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream)) !=
            cudaSuccess ||
        launch_align(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

size_t moe_w4a16_workspace_size(int M, int k, int E, int H, int I) {
    if (!layer_sizes_ok(M, k, E, H, I)) return 0;
    return fwd_layout(M, k, E, H, I).total;
}

// The forward; with `logits` non-null the router front-end first writes ids
// and topk_w (then caller-owned outputs) from the logits.
static moe_status_t forward_impl(const uint16_t *hidden, const int32_t *ids, const float *topk_w,
                                 const void *w13, const void *w2, uint16_t *out, int M, int k,
                                 int E, int H, int I, void *workspace, size_t ws_bytes,
                                 moe_stream_t stream, cudaEvent_t *ev,
                                 const float *logits = nullptr) {
    if (!layer_sizes_ok(M, k, E, H, I)) return MOE_ERR_INVALID_ARG;
    if (logits && k > E) return MOE_ERR_INVALID_ARG;
    if (!w13 || !w2 || !workspace) return MOE_ERR_INVALID_ARG;
    if (M > 0 && (!hidden || !ids || !topk_w || !out)) return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(out, 16) || !aligned(ids, 4) || !aligned(topk_w, 4) ||
        !aligned(logits, 4) || !aligned(w13, 256) || !aligned(w2, 256) ||
        !aligned(workspace, 256))
        return MOE_ERR_MISALIGNED;
    const FwdLayout L = fwd_layout(M, k, E, H, I);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    moe_status_t st = check_device();
    if (st != MOE_OK) return st;
    if (M == 0) return MOE_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    int grid = tc_grid(dev);
    if (grid <= 0) return MOE_ERR_CUDA;
    if (grid > L.grid) grid = L.grid;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(ws + L.ctrl);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(ws + L.tile_prefix);
    int32_t *tile_prefix2 = reinterpret_cast<int32_t *>(ws + L.tile_prefix2);
    int32_t *perm = reinterpret_cast<int32_t *>(ws + L.perm);
    int32_t *inv_perm = reinterpret_cast<int32_t *>(ws + L.inv_perm);
    int32_t *tickets = reinterpret_cast<int32_t *>(ws + L.tickets);
    float *partials = reinterpret_cast<float *>(ws + L.partials);
    uint16_t *xs = reinterpret_cast<uint16_t *>(ws + L.xs);
    uint16_t *act_hi = reinterpret_cast<uint16_t *>(ws + L.act_hi);
    uint16_t *act_lo = reinterpret_cast<uint16_t *>(ws + L.act_lo);
    float *y = reinterpret_cast<float *>(ws + L.y);
    const int n = M * k;
    const int r1 = 4 * (2 * I / kTileRows), r2 = 4 * (H / kTileRows);  // tickets per token tile

    AlignArgs al = {};
    al.ids = ids;
    al.n = n;
    al.E = E;
    al.reset_status = 1;
    al.token_tile = L.nt;
    al.token_tile2 = L.nt2;
    al.counts = counts;
    al.offsets = offsets;
    al.perm = perm;
    al.inv_perm = inv_perm;
    al.tile_prefix = tile_prefix;
    al.tile_prefix2 = tile_prefix2;
    al.ctrl = ctrl;
    // The gather kernel (hundreds of CTAs) zeroes both GEMMs' split-K
    // tickets, not the one-CTA alignment.
    GatherArgs ga = {hidden, inv_perm, M, k, H, xs, ctrl};
    // every ticket of both GEMMs (the workspace's whole ticket region)
    const TicketClear clear = {tickets, (int64_t)L.max_tok_tiles * r1 + (int64_t)L.max_tok_tiles2 * r2};
    TcArgs g1 = {};
    g1.w = static_cast<const uint8_t *>(w13);
    g1.offsets = offsets;
    g1.tile_prefix = tile_prefix;
    g1.tickets = tickets;
    g1.partials = partials;
    g1.E = E;
    g1.N = 2 * I;
    g1.K = H;
    g1.I = I;
    g1.kind = MOE_PACK_W13;
    g1.nt = L.nt;
    g1.act_hi = act_hi;
    g1.act_lo = act_lo;
    g1.ctrl = ctrl;
    g1.test_no_copies = test_no_copies();
    TcArgs g2 = g1;
    g2.test_no_copies = 0;
    g2.w = static_cast<const uint8_t *>(w2);
    g2.tickets = tickets + (int64_t)L.max_tok_tiles * r1;
    g2.tile_prefix = tile_prefix2;
    g2.nt = L.nt2;
    g2.N = H;
    g2.K = I;
    g2.kind = MOE_PACK_W2;
    g2.y = y;
    CombineArgs cb = {y, inv_perm, topk_w, M, k, H, out};

    CUtensorMap map_x, map_act;
    // CTA pairs load half of the token rows (gate+up) or one of hi / lo (down)
    const bool pair1 = tc_pair_mode(MOE_PACK_W13, L.nt, 2 * I);
    const bool pair2 = tc_pair_mode(MOE_PACK_W2, L.nt2, H);
    if (!make_token_map(&map_x, xs, n, H, pair1 ? L.nt / 2 : L.nt) ||
        !make_act_map(&map_act, act_hi, act_lo, n, I, L.nt2, stacked_hi_lo(L.nt2), pair2))
        return MOE_ERR_CUDA;

    auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], s) : cudaSuccess; };

    if (L.fused) {
        // The whole layer in one cooperative kernel; with logits the router
        // runs first (after the status word is cleared), and the kernel then
        // leaves the word alone.
        DecodeArgs d = {};
        d.hidden = hidden;
        d.ids = ids;
        d.topk_w = topk_w;
        d.w13 = g1.w;
        d.w2 = g2.w;
        d.out = out;
        d.M = M;
        d.k = k;
        d.E = E;
        d.H = H;
        d.I = I;
        d.reset_status = logits ? 0 : 1;
        d.ctrl = ctrl;
        d.counts = counts;
        d.offsets = offsets;
        d.perm = perm;
        d.inv_perm = inv_perm;
        d.sync = tickets;
        d.sync_ints = decode_sync_ints(L.max_tok_tiles, H, I);
        d.partials = partials;
        d.xs = xs;
        d.act_hi = act_hi;
        d.act_lo = act_lo;
        d.y = y;
        d.test_no_copies = test_no_copies();
        bool routed = false;
        if (logits) {
            RouteArgs r = {logits, M, E, k, const_cast<int32_t *>(ids), const_cast<float *>(topk_w), ctrl};
            if (cudaMemsetAsync(ctrl, 0, 4 * sizeof(int32_t), s) != cudaSuccess ||
                launch_route(r, s) != cudaSuccess) {
                cudaGetLastError();
                return MOE_ERR_CUDA;
            }
            routed = true;
        }
        if (mark(0) != cudaSuccess || launch_decode(d, map_x, map_act, grid, s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        for (int i = 1; i < 6; ++i)
            if (mark(i) != cudaSuccess) {
                cudaGetLastError();
                return MOE_ERR_CUDA;
            }
        g_diag.M = M;
        g_diag.k = k;
        g_diag.E = E;
        g_diag.H = H;
        g_diag.I = I;
        g_diag.token_tile = L.nt;
        g_diag.token_tile2 = L.nt2;
        g_diag.grid_gemm1 = grid;
        g_diag.grid_gemm2 = grid;
        g_diag.kernels_launched = 1 + (routed ? 1 : 0);
        g_diag.workspace_bytes = (int64_t)L.total;
        g_diag.calls += 1;
        return MOE_OK;
    }
    const bool pdl = (ev == nullptr);
    if (!logits && n <= kSmallAlignSlots) {
        // Small batch: one kernel aligns (in every CTA) and gathers, then the
        // two GEMMs and the combine.
        const int pg = small_prep_grid(M, H);
        SmallPrepArgs sp = {ids, hidden, M, k, E, H, L.nt, L.nt2, counts, offsets, tile_prefix,
                            tile_prefix2, perm, inv_perm, xs, ctrl, clear,
                            reinterpret_cast<int32_t *>(ws + L.ovf)};
        g1.ovf = sp.ovf;
        g1.n_ovf = pg;
        g1.tables_after_wait = 1;
        if (mark(0) != cudaSuccess || launch_align_gather_small(sp, pg, s) != cudaSuccess ||
            mark(1) != cudaSuccess || mark(2) != cudaSuccess ||
            launch_gemm_tc(g1, map_x, grid, s, pdl) != cudaSuccess || mark(3) != cudaSuccess ||
            launch_gemm_tc(g2, map_act, grid, s, pdl) != cudaSuccess || mark(4) != cudaSuccess ||
            launch_combine(cb, s, pdl) != cudaSuccess || mark(5) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_diag.M = M;
        g_diag.k = k;
        g_diag.E = E;
        g_diag.H = H;
        g_diag.I = I;
        g_diag.token_tile = L.nt;
        g_diag.token_tile2 = L.nt2;
        g_diag.grid_gemm1 = grid;
        g_diag.grid_gemm2 = grid;
        g_diag.kernels_launched = 4;
        g_diag.workspace_bytes = (int64_t)L.total;
        g_diag.calls += 1;
        return MOE_OK;
    }
    bool route_kernel = false;
    set_segments(al, ws, L.seg_counts, L.seg_base);
    if (begin_call(al, logits, M, k, const_cast<int32_t *>(ids), const_cast<float *>(topk_w), s,
                   &route_kernel) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (mark(0) != cudaSuccess || launch_align(al, s) != cudaSuccess || mark(1) != cudaSuccess ||
        launch_gather_hidden(ga, clear, s, pdl) != cudaSuccess || mark(2) != cudaSuccess ||
        launch_gemm_tc(g1, map_x, grid, s, pdl) != cudaSuccess || mark(3) != cudaSuccess ||
        launch_gemm_tc(g2, map_act, grid, s, pdl) != cudaSuccess || mark(4) != cudaSuccess ||
        launch_combine(cb, s, pdl) != cudaSuccess || mark(5) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    g_diag.M = M;
    g_diag.k = k;
    g_diag.E = E;
    g_diag.H = H;
    g_diag.I = I;
    g_diag.token_tile = L.nt;
    g_diag.token_tile2 = L.nt2;
    g_diag.grid_gemm1 = grid;
    g_diag.grid_gemm2 = grid;
    g_diag.kernels_launched = 5 + (route_kernel ? 1 : 0) + (al.seg_counts ? 2 : 0);
    g_diag.workspace_bytes = (int64_t)L.total;
    g_diag.calls += 1;
    return MOE_OK;
}

moe_status_t moe_w4a16_forward(const uint16_t *hidden, const int32_t *ids, const float *topk_w,
                               const void *w13, const void *w2,
                               uint16_t *out, int M, int k, int E, int H, int I, void *workspace,
                               size_t ws_bytes, moe_stream_t stream) {
    return forward_impl(hidden, ids, topk_w, w13, w2, out, M, k, E, H, I, workspace,
                        ws_bytes, stream, nullptr);
}

moe_status_t moe_w4a16_forward_routed(const uint16_t *hidden, const float *logits,
                                      const void *w13, const void *w2, uint16_t *out,
                                      int32_t *topk_ids, float *topk_w, int M, int k, int E,
                                      int H, int I, void *workspace, size_t ws_bytes,
                                      moe_stream_t stream) {
    if (M > 0 && !logits) return MOE_ERR_INVALID_ARG;
    return forward_impl(hidden, topk_ids, topk_w, w13, w2, out, M, k, E, H, I, workspace,
                        ws_bytes, stream, nullptr, M > 0 ? logits : nullptr);
}

moe_status_t moe_w4a16_forward_profiled(const uint16_t *hidden, const int32_t *ids,
                                        const float *topk_w, const void *w13, const void *w2, uint16_t *out, int M,
                                        int k, int E, int H, int I, void *workspace,
                                        size_t ws_bytes, moe_stream_t stream, void **events,
                                        int n_events) {
    if (!events || n_events < 6) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    return forward_impl(hidden, ids, topk_w, w13, w2, out, M, k, E, H, I, workspace,
                        ws_bytes, stream, reinterpret_cast<cudaEvent_t *>(events));
}

moe_status_t moe_w4a16_get_device_status(const void *workspace, moe_stream_t stream,
                                         int32_t *detail) {
    if (detail) *detail = 0;
    if (!workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return MOE_ERR_MISALIGNED;
    Ctrl c;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaMemcpy(&c, workspace, 2 * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    if (detail) *detail = c.detail;
    return static_cast<moe_status_t>(c.status);
}

moe_status_t moe_w4a16_workspace_views(int M, int k, int E, int H, int I, moe_ws_views_t *v) {
    if (!v || !layer_sizes_ok(M, k, E, H, I)) return MOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(M, k, E, H, I);
    v->counts = L.counts;
    v->offsets = L.offsets;
    v->perm = L.perm;
    v->inv_perm = L.inv_perm;
    v->act_hi = L.act_hi;
    v->act_lo = L.act_lo;
    v->y = L.y;
    return MOE_OK;
}

moe_status_t moe_w4a16_get_diag(moe_diag_t *diag) {
    if (!diag) return MOE_ERR_INVALID_ARG;
    *diag = g_diag;
    return MOE_OK;
}

}  // extern "C"

namespace moe {

// The forward on a caller-chosen scratch buffer (used by the entry point
// whose scratch is a static device array).
moe_status_t forward_on_scratch(const uint16_t *hidden, const int32_t *ids, const float *topk_w,
                                const void *w13, const void *w2, uint16_t *out, int M, int k, int E, int H, int I, void *scratch,
                                size_t scratch_bytes, moe_stream_t stream) {
    return forward_impl(hidden, ids, topk_w, w13, w2, out, M, k, E, H, I, scratch,
                        scratch_bytes, stream, nullptr);
}

}  // namespace moe
