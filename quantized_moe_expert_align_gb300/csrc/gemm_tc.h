// gemm_tc.h -- host interface of the tensor-core expert GEMMs (gemm_tc.cu).
#pragma once

#include <cuda.h>

#include "moe_internal.h"

namespace moe {

constexpr int kMaxStages = 18;

struct TcArgs {
    const uint8_t *w;            // prepacked weights (header included)
    const int32_t *offsets;      // [E+1] sorted-row offsets per expert
    const int32_t *tile_prefix;  // [E+1] token-tile prefix per expert (tile width nt)
    int32_t *tickets;            // per (expert tile x weight tile); zeroed before the call's GEMMs
    float *partials;             // [grid][2][nt][128] fp32 split-tile partial sums
    int E, N, K, I;              // N, K of this matrix; I for the gate+up epilogue
    int kind;                    // MOE_PACK_W13 or MOE_PACK_W2
    int nt;                      // token rows per tile: 16, 32, 64 or 128
    uint16_t *act_hi, *act_lo;   // gate+up output [n][I] fp16
    float *y;                    // down output [n][H] fp32
    Ctrl *ctrl;
    // Per-CTA fp16-overflow flags of the small-batch alignment-and-gather
    // kernel (n_ovf of them, null otherwise); the gate+up GEMM reports any.
    const int32_t *ovf;
    int n_ovf;
    // Nonzero: the kernel right before this one wrote the tile tables (the
    // small-batch kernel before the gate+up GEMM), so the set-up waits for it
    // before reading them; otherwise the tables are older and the set-up
    // reads them at once, overlapping the previous kernel.
    int tables_after_wait;
    // Failure-path test switch: nonzero makes the producers issue no copies,
    // so the other roles' bounded waits run out (MOE_ERR_DEVICE_TIMEOUT) and
    // the CTA winds down; zero in normal use.
    int test_no_copies;
};

// Whether the down GEMM stacks the hi and lo rows of its activation into one
// B operand (small token tiles); the kernel and its tensor map agree on it.
inline bool stacked_hi_lo(int nt) { return nt <= 64 || nt == 80; }

// Whether the GEMM of `kind` (MOE_PACK_W13 / W2) with nt-row token tiles over
// an N-row weight matrix runs on CTA pairs: two SMs share each MMA
// (tcgen05 cta_group::2, 256 weight rows, 128 in each SM's tensor memory)
// and each loads only half of the token operand -- half of the token rows
// (gate+up) or one of the hi / lo halves (down).  That is done where a chunk
// of token rows is 32 KiB (128-row gate+up tiles, 64-row down tiles), which
// one SM cannot take in as fast as its tensor core uses it, and needs the
// 128-row weight tiles of an expert to come in pairs (N a multiple of 256).
// The kernel choice and the token maps follow it.
inline bool tc_pair_mode(int kind, int nt, int N) {
    const bool big = (kind == MOE_PACK_W13) ? nt >= 128 : (nt == 64 || nt == 80);
    return big && N % (2 * kTileRows) == 0;
}

// Token operand of the gate+up GEMM: fp16 [rows][cols] (row-major) seen as
// 3-D (64 columns, rows, cols/64) so that one copy brings a 128-column K
// chunk of box_rows rows, stored as two 64-column slabs of box_rows x 128 B
// (128-byte swizzle, zero fill beyond the last row).
bool make_token_map(CUtensorMap *map, const void *ptr, int rows, int cols, int box_rows);
// Token operand of the down GEMM: the hi and lo fp16 halves of the
// activation (lo at a fixed byte distance after hi) as one 4-D map, so that
// one copy brings both halves of a K chunk: slabs in the order
// [K half][hi, lo] when `stacked`, [hi, lo][K half] otherwise.  With
// `one_half` (CTA pairs, stacked) a copy brings only the hi or only the lo
// rows (the third coordinate picks which) of both K halves.
bool make_act_map(CUtensorMap *map, const void *hi, const void *lo, int rows, int cols,
                  int box_rows, bool stacked, bool one_half = false);
int tc_grid(int device);
cudaError_t launch_gemm_tc(const TcArgs &args, const CUtensorMap &tok, int grid, cudaStream_t s,
                           bool pdl);

}  // namespace moe
