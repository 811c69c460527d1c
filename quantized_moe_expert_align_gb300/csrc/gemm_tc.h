// gemm_tc.h -- host interface of the tensor-core expert GEMMs (gemm_tc.cu).
#pragma once

#include <cuda.h>

#include "moe_internal.h"

namespace moe {

constexpr int kMaxStages = 16;

struct TcArgs {
    const uint8_t *w_codes;      // prepacked codes (header included)
    const uint8_t *w_scales;     // prepacked scales (header included)
    const int32_t *offsets;      // [E+1] sorted-row offsets per expert
    const int32_t *tile_prefix;  // [E+1] token-tile prefix per expert (tile width nt)
    int32_t *tickets;            // per (expert tile x weight tile); zeroed by align
    float *partials;             // [grid][2][nt][128] fp32 split-tile partial sums
    int E, N, K, I;              // N, K of this matrix; I for the gate+up epilogue
    int kind;                    // MOE_PACK_W13 or MOE_PACK_W2
    int nt;                      // token rows per tile: 16, 32, 64 or 128
    uint16_t *act_hi, *act_lo;   // gate+up output [n][I] fp16
    float *y;                    // down output [n][H] fp32
    Ctrl *ctrl;
};

// 2-D fp16 tensor map over [rows][cols] (row-major), box {64, box_rows},
// 128-byte swizzle, zero fill out of bounds.
bool make_token_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows);
int tc_grid(int device);
cudaError_t launch_gemm_tc(const TcArgs &args, const CUtensorMap &hi, const CUtensorMap &lo,
                           int grid, cudaStream_t s, bool pdl);

}  // namespace moe
