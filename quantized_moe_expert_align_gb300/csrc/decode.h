// decode.h -- host interface of the single-kernel layer forward for small
// batches (decode.cu).
#pragma once

#include <cuda.h>

#include "moe_internal.h"

namespace moe {

// Batches of at most this many slots (M*k) whose token tile is
// kDecodeTokenTile rows run as one kernel.
constexpr int kDecodeMaxSlots = 128;
constexpr int kDecodeTokenTile = 16;

struct DecodeArgs {
    const uint16_t *hidden;     // [M][H] bf16
    const int32_t *ids;         // [M][k]
    const float *topk_w;        // [M][k]
    const uint8_t *w13, *w2;    // prepacked (headers included)
    uint16_t *out;              // [M][H] bf16
    int M, k, E, H, I;
    int reset_status;           // nonzero: the kernel clears the status word first
    Ctrl *ctrl;
    // the alignment, written for inspection (one CTA writes them)
    int32_t *counts, *offsets, *perm, *inv_perm;
    // int32 region the kernel zeroes before its grid-wide barrier and then
    // uses for the split-K tickets of both GEMMs, the activation-ready flags
    // and the combine tickets; `sync_ints` bounds it
    int32_t *sync;
    int64_t sync_ints;
    float *partials;            // [2][grid][2][kDecodeTokenTile][128] fp32
    uint16_t *xs;               // [M*k][H] fp16 sorted hidden rows
    uint16_t *act_hi, *act_lo;  // [M*k][I] fp16
    float *y;                   // [M*k][H] fp32
    int test_no_copies;         // failure-path test: no weight copies are issued
};

// int32 entries of the sync region for a batch whose token tiles (of
// kDecodeTokenTile rows, over all experts) number at most max_tiles.
int64_t decode_sync_ints(int max_tiles, int H, int I);

// Launch as a cooperative grid of `grid` CTAs (one per SM); the token maps
// are those of the regular path with kDecodeTokenTile-row boxes (the hidden
// rows, and the stacked hi/lo activation).
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &map_x, const CUtensorMap &map_act,
                          int grid, cudaStream_t s);

}  // namespace moe
