// gemm_simple.cu -- straightforward CUDA-core grouped expert GEMMs over the
// prepacked layout.  One warp computes one output column for up to 16
// expert-sorted token rows; the weights of that column are read once per
// 16 rows.  This is the first, correctness-first path of the library.
//
//  gate+up (MOE_PACK_W13): a[p][n] = silu(g) * u with g, u the dot products
//      of xs[p] with gate row n and up row n; a is stored as fp16 hi + lo.
//  down    (MOE_PACK_W2):  y[p][h] = (a_hi + a_lo)[p] . W2[h]   (fp32)
// Weights are dequantised exactly ((q - 8) * fp16 scale), products and sums
// are fp32.
#include "device_common.cuh"

namespace moe {
namespace {

constexpr int kRowsPerWarp = 16;
constexpr int kWarps = 8;

__device__ __forceinline__ void decode_word(uint32_t word, float scale, float (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int slot = (i & 1) ? 4 + (i >> 1) : (i >> 1);
        v[i] = (float)((int)((word >> (4 * slot)) & 0xFu) - 8) * scale;
    }
}

__device__ __forceinline__ void load_half8(const uint16_t *p, float (&x)[8]) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        const float2 f = __half22float2(h);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

template <int KIND>
__global__ void __launch_bounds__(kWarps * 32) gemm_simple_kernel(GemmArgs a,
                                                                  const int32_t *tile_prefix) {
    pdl_wait();
    pdl_trigger();
    const int tile = blockIdx.x;
    if (tile >= __ldg(tile_prefix + a.E)) return;
    if (!header_ok(a.w_codes, KIND, kPartCodes, a.E, a.N, a.K) ||
        !header_ok(a.w_scales, KIND, kPartScales, a.E, a.N, a.K)) {
        if (threadIdx.x == 0) set_status(a.ctrl, MOE_ERR_BAD_LAYOUT, KIND);
        return;
    }
    const int e = find_segment(tile_prefix, a.E, tile);
    const int p0 = __ldg(a.offsets + e) + (tile - __ldg(tile_prefix + e)) * kRowsPerWarp;
    const int rows = min(kRowsPerWarp, __ldg(a.offsets + e + 1) - p0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = blockIdx.y * kWarps + warp;
    const int tiles = a.N / kTileRows, chunks = a.K / kChunkK;
    const uint32_t *codes = reinterpret_cast<const uint32_t *>(a.w_codes + kHeaderBytes);
    const __half *scales = reinterpret_cast<const __half *>(a.w_scales + kHeaderBytes);

    int rt, r, chunk0, chunk_step;
    if (KIND == MOE_PACK_W13) {
        rt = col / (kTileRows / 2);
        r = 2 * (col % (kTileRows / 2)) + (lane >> 4);
        chunk0 = 0;
        chunk_step = 1;
    } else {
        rt = col / kTileRows;
        r = col % kTileRows;
        chunk0 = lane >> 4;
        chunk_step = 2;
    }
    const int pc = (lane & 15) >> 2, wi = lane & 3;

    float acc[kRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) acc[j] = 0.f;

    for (int c = chunk0; c < chunks; c += chunk_step) {
        const int64_t blk = ((int64_t)e * tiles + rt) * chunks + c;
        const uint32_t word = __ldg(codes + blk * (kCodeBlockBytes / 4) + (pc * kTileRows + r) * 4 + wi);
        const float sc = __half2float(scales[blk * (kScaleBlockBytes / 2) + r * 4 + pc]);
        float w[8];
        decode_word(word, sc, w);
        const int kk = c * kChunkK + pc * 32 + wi * 8;
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            if (j < rows) {
                float x[8];
                load_half8(a.in_hi + (size_t)(p0 + j) * a.K + kk, x);
                if (KIND == MOE_PACK_W2) {
                    float xl[8];
                    load_half8(a.in_lo + (size_t)(p0 + j) * a.K + kk, xl);
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] += xl[i];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j] = fmaf(w[i], x[i], acc[j]);
            }
        }
    }

#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        float v = acc[j];
        if (KIND == MOE_PACK_W13) {
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            const float u = __shfl_sync(0xffffffffu, v, 16);
            if (lane == 0 && j < rows) {
                const float g = v;
                const float act = g / (1.0f + expf(-g)) * u;
                if (fabsf(act) > 65504.0f && !isinf(act) && !isnan(act))
                    set_status(a.ctrl, MOE_ERR_DEVICE_FP16_RANGE, 1);
                const __half hi = __float2half_rn(act);
                const __half lo = __float2half_rn(act - __half2float(hi));
                const size_t o = (size_t)(p0 + j) * a.I + col;
                a.act_hi[o] = *reinterpret_cast<const uint16_t *>(&hi);
                a.act_lo[o] = *reinterpret_cast<const uint16_t *>(&lo);
            }
        } else {
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && j < rows) a.y[(size_t)(p0 + j) * a.N + col] = v;
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simple(const GemmArgs &a, const int32_t *tile_prefix, cudaStream_t s,
                               bool pdl) {
    // Upper bound on the tile count: sum_e ceil(c_e / 16) <= n / 16 + E.
    const int64_t max_tiles = (int64_t)a.n / kRowsPerWarp + a.E;
    const int cols = (a.kind == MOE_PACK_W13) ? a.I : a.N;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)max_tiles, (unsigned)(cols / kWarps));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (a.kind == MOE_PACK_W13) return cudaLaunchKernelEx(&cfg, gemm_simple_kernel<MOE_PACK_W13>, a, tile_prefix);
    return cudaLaunchKernelEx(&cfg, gemm_simple_kernel<MOE_PACK_W2>, a, tile_prefix);
}

int simple_token_tile() { return kRowsPerWarp; }

}  // namespace moe
