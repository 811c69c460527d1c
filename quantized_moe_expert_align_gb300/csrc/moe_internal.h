// moe_internal.h -- layouts and launchers shared by the library's .cu files.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "moe_w4a16.h"

namespace moe {

// ---------------------------------------------------------------------------
// Prepacked weight layout.
//
// A prepacked buffer starts with a 256-byte header, then blocks of 9216 B.
// A block covers one 128-row tile of one expert and one 128-element K chunk:
//   bytes [0, 8192)    codes: 4 pieces x 128 rows x 16 B; piece pc of row r
//                      at byte (pc*128 + r)*16 holds K elements
//                      [32pc, 32pc+32) of the chunk as 4 words; word w
//                      covers elements 8w..8w+7, element i's 4-bit code
//                      starting at bit nibble_pos(i) and wrapping past bit
//                      31 to bit 0 (see the dequantisation in gemm_tc.cu).
//   bytes [8192, 9216) scales: 128 rows x 4 groups of fp16, row r group g
//                      at byte 8192 + (r*4 + g)*2.
// Block index = (e * tiles_per_expert + tile) * k_chunks + chunk.
// For w13, tile t holds gate rows 64t..64t+63 at even tile rows (row 2j =
// gate row 64t+j) and the matching up rows at odd tile rows (2j+1).
// ---------------------------------------------------------------------------
constexpr int kTileRows = 128;
constexpr int kChunkK = 128;
constexpr int kGroup = 32;
constexpr int kCodeBlockBytes = kTileRows * kChunkK / 2;       // 8192
constexpr int kScaleBlockBytes = kTileRows * (kChunkK / kGroup) * 2;  // 1024
constexpr int kBlockBytes = kCodeBlockBytes + kScaleBlockBytes;       // 9216
constexpr int kHeaderBytes = 256;
// Bit offset of element i's code inside its 32-bit word: 6, 22, 10, 26, 14,
// 30, 18, 2 for i = 0..7.
__host__ __device__ constexpr int nibble_pos(int i) {
    return (((i & 1) ? 22 : 6) + 4 * (i >> 1)) & 31;
}

constexpr uint32_t kPackMagic = 0x5034574Du;  // "MW4P"
constexpr uint32_t kPackVersion = 3;  // 3: one block per chunk, codes at nibble_pos

struct PackHeader {
    uint32_t magic;
    uint32_t version;
    uint32_t kind;    // MOE_PACK_W13 / MOE_PACK_W2
    uint32_t block_bytes;  // kBlockBytes
    int32_t E, N, K, group;
    int32_t status;   // MOE_OK once the prepack finished and validated
    int32_t wide_scales;  // nonzero: some |scale| > 65504/24 or infinite
    int32_t source_group; // elements per scale of the source (32, 64, 128)
    int32_t pad;
};
static_assert(sizeof(PackHeader) <= kHeaderBytes, "header too large");

inline size_t packed_bytes(int E, int N, int K) {
    return kHeaderBytes + (size_t)E * (N / kTileRows) * (K / kChunkK) * kBlockBytes;
}

// ---------------------------------------------------------------------------
// Workspace control block (first 256 bytes of every workspace).
// ---------------------------------------------------------------------------
struct Ctrl {
    int32_t status;   // first device-side error of the current call
    int32_t detail;
    int32_t n_invalid;  // slots whose id was out of range
    int32_t pad[61];
};
static_assert(sizeof(Ctrl) == 256, "ctrl block is 256 bytes");

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Carving of the align workspace.
struct AlignLayout {
    size_t ctrl, seg_counts, seg_base, total;  // seg_*: large batches only
};
AlignLayout align_layout(int M, int k, int E);

// Carving of the forward workspace.
struct FwdLayout {
    bool fused;         // the whole layer in one kernel (small batches, decode.cu)
    int nt;             // token rows per MMA tile of the gate+up GEMM
    int nt2;            // token rows per MMA tile of the down GEMM (<= nt)
    int max_tok_tiles;  // bound on sum_e ceil(count_e / nt)
    int max_tok_tiles2; // bound on sum_e ceil(count_e / nt2)
    int grid;           // most CTAs the GEMM kernels may use (partials are sized for it)
    size_t ctrl, counts, offsets, tile_prefix, tile_prefix2, perm, inv_perm;
    size_t seg_counts, seg_base;  // int32 [E][kAlignSegs] each, large batches only
    size_t tickets;     // int32 [max_tok_tiles * 4 * 2I/128 + max_tok_tiles2 * 4 * H/128];
                        // fused: the single kernel's sync region (decode_sync_ints)
    size_t partials;    // fp32 [grid][2][nt][128], fused: [2][grid][2][nt][128]
    size_t ovf;         // int32 [grid]: per-CTA fp16-overflow flags of the small-batch kernel
    size_t xs;          // [n][H] fp16 hidden rows in sorted order
    size_t act_hi;      // [n][I] fp16
    size_t act_lo;      // [n][I] fp16
    size_t y;           // [n][H] fp32
    size_t total;
};
// Token rows per tile for a batch of n = M*k slots over E experts: for the
// gate+up GEMM, and for the down GEMM given the former.
int pick_token_tile(int n, int E);
int down_token_tile(int nt, int H, int64_t n, int E);
// Whether a batch of n slots with gate+up token tiles of nt rows runs as the
// single small-batch kernel.
bool use_decode_kernel(int64_t n, int nt);
FwdLayout fwd_layout(int M, int k, int E, int H, int I);

// moe_w4a16_forward on a scratch buffer the caller of this function chose.
moe_status_t forward_on_scratch(const uint16_t *hidden, const int32_t *ids, const float *topk_w,
                                const void *w13, const void *w2,
                                uint16_t *out, int M, int k, int E, int H, int I, void *scratch,
                                size_t scratch_bytes, moe_stream_t stream);

// ---------------------------------------------------------------------------
// Launchers (each returns the cudaError_t of its launch).
// ---------------------------------------------------------------------------
struct AlignArgs {
    const int32_t *ids;
    int n;            // M * k
    int E;
    int reset_status; // nonzero: this kernel starts the call (clears the status word)
    // Routing inside the alignment kernel (logits non-null): the kernel first
    // writes route_ids / route_w for route_M tokens of route_k slots from
    // logits [route_M][E], then aligns route_ids (ids must equal route_ids).
    const float *logits;
    int route_M, route_k;
    int32_t *route_ids;
    float *route_w;
    int token_tile;   // >0: also write tile_prefix for this tile width,
    int token_tile2;  //     and tile_prefix2 for this one
    int32_t *counts, *offsets, *perm, *inv_perm, *tile_prefix, *tile_prefix2;
    Ctrl *ctrl;
    // Large batches (align_large): per-(expert, segment) counts and their
    // exclusive prefixes, [E][kAlignSegs] int32 each; null for one CTA.  The
    // caller clears the status word (and routes) before such a call.
    int32_t *seg_counts, *seg_base;
};
cudaError_t launch_align(const AlignArgs &a, cudaStream_t s);
// Batches of more than kAlignLargeSlots slots are aligned by kAlignSegs CTAs
// (three kernels) instead of one.  One CTA's time grows with the slots it
// walks (13 us at 2048 slots, 25 at 8192, 42 at 16384 on one GB300); the
// three kernels take 13-15 us at 8192-16384 slots and 17 at 32768, so the
// switch is at 2048 (E = 128 M = 2048: 893 -> 866 us per layer call).
constexpr int kAlignSegs = 32;
constexpr int kAlignLargeSlots = 2048;
inline bool align_large(int64_t n) { return n > kAlignLargeSlots; }

// Router front-end: topk ids / weights from fp32 logits, one warp per token.
struct RouteArgs {
    const float *logits;  // [M][E]
    int M, E, k;
    int32_t *ids;         // [M][k]
    float *w;             // [M][k]
    Ctrl *ctrl;
};
cudaError_t launch_route(const RouteArgs &a, cudaStream_t s);
// Batches up to this many tokens are routed inside the alignment kernel
// (32 warps, at most two tokens each); larger ones by route_kernel first.
constexpr int kFusedRouteMaxM = 64;

// Both write into the blocks after the header of a prepacked buffer `dst`.
cudaError_t launch_prepack_codes(int kind, const uint8_t *q, int E, int N, int K,
                                 uint8_t *dst, cudaStream_t s);
// `group`: elements of K per source scale (32, 64 or 128).
cudaError_t launch_prepack_scales(int kind, const uint16_t *sc, int E, int N, int K, int group,
                                  uint8_t *dst, int32_t *bad_flag, int32_t *wide_flag,
                                  cudaStream_t s);

struct GatherArgs {
    const uint16_t *hidden;    // [M][H] bf16
    const int32_t *inv_perm;   // [M*k]: sorted row of each slot, -1 if invalid
    int M, k, H;
    uint16_t *xs;              // [n][H] fp16
    Ctrl *ctrl;
};

struct CombineArgs {
    const float *y;           // [n][H]
    const int32_t *inv_perm;  // [M*k]
    const float *topk_w;      // [M][k]
    int M, k, H;
    uint16_t *out;            // [M][H] bf16
};
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t s, bool pdl);

}  // namespace moe
