// elementwise.h -- host interface of the gather kernel's second duty
// (elementwise.cu): it also zeroes the split-K tickets of both GEMMs of a
// forward call, spread over its whole grid.
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

}  // namespace moe
