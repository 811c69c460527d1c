// prepack.cu -- one-time repack of canonical INT4 codes and bf16 scales into
// the library's block layout (see moe_internal.h for the layout).
//
// The MoE GEMM sweep of "The MoE Throughput Lever: Quantifying the INT4
// Marlin GEMM on Blackwell PRO 6000" ("The Benchmark: What Was Measured")
// drives a repack path that turns checkpoint weights into the kernel's own
// layout once, before any timed call; this is that step for this library.
#include "device_common.cuh"

namespace moe {
namespace {

// Canonical row of tile-row r of tile `tile` (w13 interleaves gate and up).
__device__ __forceinline__ int canonical_row(int kind, int N, int tile, int r) {
    if (kind == MOE_PACK_W13) {
        const int half = N / 2, j = r >> 1;
        return (r & 1) ? half + tile * (kTileRows / 2) + j : tile * (kTileRows / 2) + j;
    }
    return tile * kTileRows + r;
}

// One thread per output 32-bit word of codes (the first 8 KiB of a block).
__global__ void prepack_codes_kernel(int kind, const uint32_t *__restrict__ q, int E, int N,
                                     int K, uint8_t *__restrict__ blocks) {
    const int tiles = N / kTileRows, chunks = K / kChunkK;
    const int64_t words_per_block = kCodeBlockBytes / 4;
    const int64_t total = (int64_t)E * tiles * chunks * words_per_block;
    const int64_t row_words = K / 8;  // canonical row length in 32-bit words
    for (int64_t wd = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; wd < total;
         wd += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = wd / words_per_block;
        const int wib = (int)(wd % words_per_block);
        const int pc = wib / (kTileRows * 4), r = (wib / 4) % kTileRows, wi = wib % 4;
        const int chunk = (int)(b % chunks);
        const int tile = (int)((b / chunks) % tiles);
        const int64_t e = b / ((int64_t)chunks * tiles);
        const int n = canonical_row(kind, N, tile, r);
        const int kk0 = chunk * kChunkK + pc * 32 + wi * 8;
        const uint32_t c = __ldg(q + (e * N + n) * row_words + kk0 / 8);
        // canonical nibble i holds element i; it moves to bit nibble_pos(i)
        // (a rotation, so the code at bit 30 wraps into bits 0-1)
        uint32_t o = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t v = (c >> (4 * i)) & 0xFu;
            o |= __funnelshift_l(v, v, nibble_pos(i));
        }
        reinterpret_cast<uint32_t *>(blocks + b * kBlockBytes)[wib] = o;
    }
}

// One thread per output fp16 scale (the last 1 KiB of a block).  The block
// holds one scale per 32 elements of K; a source with wider groups (64 or
// 128 elements per scale) repeats each of its scales into the 32-element
// slots it covers.  A scale must be zero, NaN, infinite or of magnitude in
// [2^-14, 8188] so that (q - 8) * scale is exact in fp16.  Scales above
// 65504/24 in magnitude or infinite set *wide_flag: the one-instruction
// dequantisation needs -24 * s in fp16.
__global__ void prepack_scales_kernel(int kind, const uint16_t *__restrict__ s, int E, int N,
                                      int K, int group, uint8_t *__restrict__ blocks,
                                      int32_t *bad_flag, int32_t *wide_flag) {
    const int tiles = N / kTileRows, chunks = K / kChunkK, groups = K / group;
    const int per_block = kTileRows * (kChunkK / kGroup);
    const int64_t total = (int64_t)E * tiles * chunks * per_block;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / per_block;
        const int within = (int)(i % per_block);
        const int r = within / 4, g = within % 4;
        const int chunk = (int)(b % chunks);
        const int tile = (int)((b / chunks) % tiles);
        const int64_t e = b / ((int64_t)chunks * tiles);
        const int n = canonical_row(kind, N, tile, r);
        const int src = (chunk * kChunkK + g * kGroup) / group;
        const float f = bf16_bits_to_float(__ldg(s + (e * N + n) * groups + src));
        const float a = fabsf(f);
        const bool ok = (f == 0.0f) || isnan(f) || isinf(f) ||
                        (a >= 6.103515625e-05f && a <= 8188.0f);
        if (!ok) atomicExch(bad_flag, 1);
        if (isinf(f) || 24.0f * a > 65504.0f) atomicExch(wide_flag, 1);
        reinterpret_cast<__half *>(blocks + b * kBlockBytes + kCodeBlockBytes)[within] =
            __float2half_rn(f);
    }
}

int grid_for(int64_t work) {
    int64_t blocks = (work + 255) / 256;
    return (int)(blocks < 152 * 16 ? (blocks > 0 ? blocks : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_prepack_codes(int kind, const uint8_t *q, int E, int N, int K, uint8_t *dst,
                                 cudaStream_t s) {
    const int64_t words = (int64_t)E * (N / kTileRows) * (K / kChunkK) * (kCodeBlockBytes / 4);
    prepack_codes_kernel<<<grid_for(words), 256, 0, s>>>(
        kind, reinterpret_cast<const uint32_t *>(q), E, N, K, dst + kHeaderBytes);
    return cudaGetLastError();
}

cudaError_t launch_prepack_scales(int kind, const uint16_t *sc, int E, int N, int K, int group,
                                  uint8_t *dst, int32_t *bad_flag, int32_t *wide_flag,
                                  cudaStream_t s) {
    const int64_t n = (int64_t)E * (N / kTileRows) * (K / kChunkK) * (kScaleBlockBytes / 2);
    prepack_scales_kernel<<<grid_for(n), 256, 0, s>>>(kind, sc, E, N, K, group,
                                                      dst + kHeaderBytes, bad_flag, wide_flag);
    return cudaGetLastError();
}

}  // namespace moe
