// elementwise.h -- host interface of the row kernels around the GEMMs: the
// gather kernel's second duty (elementwise.cu: it also zeroes the split-K
// tickets of both GEMMs of a forward call, spread over its whole grid), and
// the small-batch kernel that aligns and gathers at once (prep_small.cu).
#pragma once

#include "moe_internal.h"

namespace moe {

// `n` int32 tickets at `tickets` (16-byte aligned, n a multiple of 4) to
// zero; n = 0: none.
struct TicketClear {
    int32_t *tickets;
    int64_t n;
};

cudaError_t launch_gather_hidden(const GatherArgs &a, const TicketClear &clear, cudaStream_t s,
                                 bool pdl);

// The alignment and the hidden-row gather of a batch of at most
// kSmallAlignSlots slots in one kernel (prep_small.cu).
constexpr int kSmallPrepMaxGrid = 152;
struct SmallPrepArgs {
    const int32_t *ids;        // [M][k]
    const uint16_t *hidden;    // [M][H] bf16
    int M, k, E, H;
    int nt, nt2;               // token-tile widths of the gate+up and the down GEMM
    int32_t *counts, *offsets, *tile_prefix, *tile_prefix2, *perm, *inv_perm;
    uint16_t *xs;              // [M*k][H] fp16, sorted rows
    Ctrl *ctrl;
    TicketClear clear;         // both GEMMs' split-K tickets
    int32_t *ovf;              // [grid] per-CTA fp16-overflow flags, written every call
};
int small_prep_grid(int M, int H);
cudaError_t launch_align_gather_small(const SmallPrepArgs &a, int grid, cudaStream_t s);

}  // namespace moe
