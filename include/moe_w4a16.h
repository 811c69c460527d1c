/*
 * moe_w4a16.h -- C ABI of the GB300 (sm_103a) weight-only-INT4 MoE layer
 * forward: top-k routed token alignment, grouped gate+up GEMM with a fused
 * SiLU(gate)*up epilogue, grouped down GEMM, fixed-order top-k combine.
 *
 * The operation (page title, section):
 *  - "The MoE Throughput Lever: Quantifying the INT4 Marlin GEMM on Blackwell
 *    PRO 6000", "The Benchmark: What Was Measured": an MoE GEMM with INT4
 *    weights in groups of 32, 16-bit activations, top-8 routing over E=384
 *    experts, hidden 7168, intermediate 2048, weights repacked once into the
 *    kernel's own layout before use.
 *  - "perf(exl3): accelerate fat-expert prefill - #77", "Rollout" and
 *    "Summary": routed tokens are sorted by expert and each expert's rows run
 *    as one batch through a stacked gate+up GEMM; results are written back to
 *    token rows ("direct"/"scatter" writes).
 *  - "DeepSeek-V4.1-Flash-EXL3 ... Detailed results", "Nsight Compute on the
 *    stock kernel": the per-expert count scan, serial there, is done here
 *    with warp shuffles.
 * Definition used (the pages give no formula):
 *   W[e][n][kk] = (q - 8) * scale[e][n][kk / 32],  q in [0, 15]
 *   a = silu(x W13_gate^T) * (x W13_up^T)   with rows [0, I) of w13 = gate
 *   y = a W2^T,   out[t] = bf16( sum_{j=0..k-1 ascending} topk_w[t][j] * y(t,j) )
 *
 * Conventions for every entry point:
 *  - The caller owns every buffer; the library allocates no device memory.
 *  - Device pointers must be device-accessible; the library never reads them
 *    on the host.  Calls taking a stream are asynchronous on that stream
 *    (except moe_w4a16_prepack and moe_w4a16_get_device_status, which wait).
 *  - Host-detectable errors (null or misaligned pointers, bad sizes, small
 *    workspace, no sm_103 device) return before anything is launched.
 *  - Errors found on the device (an expert id outside [0, E), a prepacked
 *    buffer whose header does not match, an activation beyond fp16 range,
 *    a NaN or +inf router logit, a bounded wait that ran out) never trap:
 *    the kernels record the first one in the workspace's status word and
 *    skip the affected work.
 *    moe_w4a16_get_device_status() reads it back.  Each forward or align
 *    call resets the word when it starts.
 *  - A workspace must not be used by two calls that overlap on the GPU.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,          /* null pointer, size out of range */
    MOE_ERR_MISALIGNED = 2,           /* pointer below its required alignment */
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,
    MOE_ERR_BAD_LAYOUT = 4,           /* prepacked header does not match */
    MOE_ERR_UNSUPPORTED_DEVICE = 5,   /* current device is not sm_103 */
    MOE_ERR_CUDA = 6,                 /* a CUDA runtime call failed */
    MOE_ERR_DEVICE_BAD_EXPERT_ID = 7, /* an id outside [0, E) was seen */
    MOE_ERR_DEVICE_TIMEOUT = 8,       /* a bounded device wait gave up */
    MOE_ERR_DEVICE_FP16_RANGE = 9,    /* a value is not representable in fp16 */
    MOE_ERR_DEVICE_BAD_LOGIT = 10     /* a router logit is NaN or +inf */
} moe_status_t;

/* Which matrix a prepacked buffer holds. */
typedef enum {
    MOE_PACK_W13 = 1, /* gate+up, canonical [E][2I][H/2]: N = 2I, K = H */
    MOE_PACK_W2 = 2   /* down,    canonical [E][H][I/2]:  N = H,  K = I */
} moe_pack_kind_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *moe_status_string(moe_status_t status);

/*
 * Bytes of the prepacked buffer for one matrix: a 256-byte header, then
 * 9 KiB per (expert, 128-row tile, 128-element K chunk), whatever the
 * group.  Requires group in {32, 64, 128}, N % 128 == 0, K % 128 == 0,
 * E >= 1; otherwise returns MOE_ERR_INVALID_ARG and sets *bytes to 0.
 */
moe_status_t moe_w4a16_prepack_size(int kind, int E, int N, int K, int group,
                                    size_t *bytes);

/*
 * Repack canonical weights into the library's layout (done once per layer at
 * load time, ahead of any forward).  The weight repack step corresponds to
 * the repack path the MoE GEMM sweep drives before timing ("The MoE
 * Throughput Lever", "The Benchmark: What Was Measured").
 *
 *  q_canon [E][N][K/2] uint8, device: element kk of row n sits in byte kk/2,
 *          in the low nibble when kk is even, the high nibble when odd.
 *  scales  [E][N][K/group] bf16 bit patterns, device: one scale per `group`
 *          consecutive elements of K.  The pages' layer uses group = 32;
 *          64 and 128 (a variant this library adds) are stored in the same
 *          packed layout, each scale repeated into the 32-element slots it
 *          covers, so the forward is the same for all three.
 *  dst     device buffer of at least moe_w4a16_prepack_size bytes,
 *          256-byte aligned; the caller owns it.
 * Layout written: per expert, 128-row tiles (for w13 each tile holds 64 gate
 * rows interleaved with the 64 matching up rows), per 128-element K chunk one
 * 9 KiB block: 8 KiB of codes, reordered for a cheap 4-bit -> fp16
 * conversion, followed by the chunk's 1 KiB of scales as fp16, so that one
 * contiguous copy brings a chunk's weights on chip.
 *
 * Every scale must be zero, NaN, infinite or of magnitude in
 * [2^-14, 8188] so that every (q - 8) * scale is exact in fp16; otherwise the
 * call returns MOE_ERR_DEVICE_FP16_RANGE and marks the buffer invalid.
 * This call waits for its own work on `stream` to finish.
 */
moe_status_t moe_w4a16_prepack(int kind, const uint8_t *q_canon,
                               const uint16_t *scales, int E, int N, int K,
                               int group, void *dst, size_t dst_bytes,
                               moe_stream_t stream);

/* Workspace bytes needed by moe_align (256-byte aligned buffer). */
size_t moe_align_workspace_size(int M, int k, int E);

/*
 * Top-k routed token alignment (the "sorted routing" stage of
 * "perf(exl3): accelerate fat-expert prefill - #77", "Rollout"): a stable
 * counting sort of the M*k flat slot indices f = t*k + j by expert id.
 *
 *  topk_ids [M][k] int32, device.
 *  counts   [E]   int32, device, out: valid slots per expert.
 *  offsets  [E+1] int32, device, out: exclusive prefix sum of counts.
 *  perm     [M*k] int32, device, out: perm[offsets[e] + r] = the r-th
 *           smallest f with topk_ids[f] == e; entries from offsets[E] on are
 *           set to -1.
 *  inv_perm [M*k] int32, device, out (may be NULL): position of f in perm,
 *           or -1 when topk_ids[f] is outside [0, E).
 * Limits: 1 <= E <= 1024, 1 <= k <= 64, 0 <= M, M*k < 2^31.
 * Out-of-range ids are left out and reported as MOE_ERR_DEVICE_BAD_EXPERT_ID
 * through the workspace status word.  M == 0 writes zero counts and offsets.
 */
moe_status_t moe_align(const int32_t *topk_ids, int M, int k, int E,
                       int32_t *counts, int32_t *offsets, int32_t *perm,
                       int32_t *inv_perm, void *workspace, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * Router front-end fused with the alignment: from the router's logits, the
 * top-k experts of every token and their renormalised softmax weights, then
 * the alignment of those ids exactly as moe_align.  The pages do not
 * describe the router; the definition is that of the layer's benchmark
 * inputs, a softmax over all E logits, its k largest, weights renormalised
 * to sum 1:
 *   topk_ids[t][0..k-1] = experts in descending logit order, the lower
 *                         expert index first among equal logits (-0 == +0;
 *                         -inf after every number; NaN after everything);
 *   topk_w[t][j] = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0), l_j the logit
 *                  of slot j (the softmax normaliser over all E cancels).
 *
 *  logits   [M][E] fp32, device, 4-byte aligned.
 *  topk_ids [M][k] int32, topk_w [M][k] fp32, device, out.
 *  counts, offsets, perm, inv_perm, workspace: as in moe_align
 *           (workspace of moe_align_workspace_size bytes).
 * Limits: those of moe_align and k <= E.  A row holding a NaN or +inf logit
 * keeps ids in the order above, gets all-zero weights, and is reported as
 * MOE_ERR_DEVICE_BAD_LOGIT (detail = its token index); a row of only -inf
 * logits gets all-zero weights.  Batches of at most 64 tokens are routed
 * inside the alignment kernel (one launch); larger ones by a separate
 * kernel first.
 */
moe_status_t moe_route_align(const float *logits, int M, int k, int E,
                             int32_t *topk_ids, float *topk_w, int32_t *counts,
                             int32_t *offsets, int32_t *perm, int32_t *inv_perm,
                             void *workspace, size_t ws_bytes, moe_stream_t stream);

/* Workspace bytes needed by moe_w4a16_forward (256-byte aligned buffer). */
size_t moe_w4a16_workspace_size(int M, int k, int E, int H, int I);

/*
 * MoE layer forward.
 *  hidden [M][H] bf16, device, 16-byte aligned.
 *  topk_ids [M][k] int32, topk_w [M][k] fp32 (used as given), device.
 *  w13: prepacked gate+up weights (kind MOE_PACK_W13, N = 2I, K = H)
 *  w2:  prepacked down weights    (kind MOE_PACK_W2,  N = H,  K = I)
 *  out [M][H] bf16, device, 16-byte aligned: written once, rounded to
 *           nearest-even from an fp32 combine over ascending slots.
 *  workspace: moe_w4a16_workspace_size(...) bytes, 256-byte aligned.
 * Limits: H % 128 == 0, I % 128 == 0, 1 <= E <= 1024, 1 <= k <= 64,
 * 0 <= M, M*k < 2^31.  M == 0 returns MOE_OK without launching.
 * The token-tile width (rows of expert-sorted tokens per tensor-core tile) is
 * chosen from M*k/E; for testing, the environment variable
 * MOE_W4A16_TOKEN_TILE = 16, 32, 64, 128 or 160 fixes it (read once per process;
 * the workspace size follows it).  For testing the failure path only,
 * MOE_W4A16_TEST_NO_COPIES=1 (read once per process) makes the gate+up GEMM
 * issue no copies: its bounded waits give up after about a second, the call
 * reports MOE_ERR_DEVICE_TIMEOUT and its output is undefined.
 * Numerics: weights dequantised exactly to fp16, hidden converted to fp16
 * (values beyond fp16 range set MOE_ERR_DEVICE_FP16_RANGE), fp32
 * accumulation, the activation passed to the down GEMM as an fp16 hi+lo pair.
 * Kernels: five (alignment, hidden gather, gate+up GEMM, down GEMM,
 * combine), chained with programmatic dependent launch; four for batches of
 * at most 128 slots, whose first kernel aligns (in every CTA) and gathers;
 * seven above 2048 slots, aligned by three kernels over 32 CTAs.  The GEMMs
 * with 128/160-row (gate+up) and 64/80-row (down) token tiles run on
 * clusters of two CTAs (tcgen05 cta_group::2) when the matrix's 128-row
 * weight tiles come in pairs.  Opt-in:
 * MOE_W4A16_DECODE_FUSED=1 (read once per process) runs batches of at most
 * 128 slots (M*k) whose token tile is 16 rows as one cooperative kernel of
 * one CTA per SM (every CTA resident at once; the call fails with
 * MOE_ERR_CUDA where the device cannot host that) -- the same results,
 * written to `out` and to the workspace; on one GB300 it measured 7-10%
 * slower than the five kernels, hence off by default.
 */
moe_status_t moe_w4a16_forward(const uint16_t *hidden, const int32_t *topk_ids,
                               const float *topk_w, const void *w13, const void *w2,
                               uint16_t *out, int M, int k, int E, int H, int I,
                               void *workspace, size_t ws_bytes,
                               moe_stream_t stream);

/*
 * moe_w4a16_forward from router logits: the router front-end of
 * moe_route_align writes topk_ids [M][k] and topk_w [M][k] (caller-owned,
 * device, 4-byte aligned) from logits [M][E] fp32, then the layer runs on
 * them.  Other arguments, limits and the workspace are those of
 * moe_w4a16_forward (same moe_w4a16_workspace_size), plus k <= E.  Bad
 * logits are reported as in moe_route_align; their tokens' output rows are
 * zero.  Up to 64 tokens (E <= 512) are routed by the alignment kernel
 * before it aligns, larger batches by a router kernel first.
 */
moe_status_t moe_w4a16_forward_routed(const uint16_t *hidden, const float *logits,
                                      const void *w13, const void *w2, uint16_t *out,
                                      int32_t *topk_ids, float *topk_w, int M, int k,
                                      int E, int H, int I, void *workspace,
                                      size_t ws_bytes, moe_stream_t stream);

/*
 * Same as moe_w4a16_forward, and additionally records CUDA events around each
 * kernel it launches, for per-kernel timing.  `events` points to
 * n_events >= 6 cudaEvent_t handles (created by the caller, timing enabled):
 * events[i] is recorded right before kernel i and events[5] after the last;
 * kernel order: 0 align, 1 hidden gather, 2 gate+up GEMM, 3 down GEMM,
 * 4 combine.  When the call runs as the single small-batch kernel,
 * events[0] is recorded right before it and events[1..5] right after it
 * (moe_w4a16_get_diag then reports one kernel).  Recording between kernels
 * stops them from overlapping, so the sum of the intervals can exceed the
 * plain forward's time.  Returns MOE_ERR_INVALID_ARG if events is NULL or
 * n_events < 6.
 */
moe_status_t moe_w4a16_forward_profiled(const uint16_t *hidden, const int32_t *topk_ids,
                                        const float *topk_w, const void *w13, const void *w2,
                                        uint16_t *out, int M, int k, int E, int H, int I,
                                        void *workspace, size_t ws_bytes,
                                        moe_stream_t stream, void **events, int n_events);

/*
 * Size of the device array that moe_w4a16_forward_static uses as its
 * workspace: 16 MiB, reserved on every GPU that loads this library.
 */
#define MOE_W4A16_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * moe_w4a16_forward without a caller-provided workspace, for callers that
 * cannot allocate device memory: code embedded in a host framework that owns
 * every device allocation and hands out only its own tensors, or a
 * latency-bound decode loop where cudaMalloc would synchronise the device.
 * (The pages describe no such entry point; it is a convenience of this
 * library.)
 *
 *  Arguments, layouts and results are those of moe_w4a16_forward; hidden,
 *  ids, weights and out are still the caller's.  Instead of a workspace the
 *  call uses one device array of MOE_W4A16_STATIC_SCRATCH_BYTES inside the
 *  library.  It allocates nothing: no cudaMalloc, cudaFree or other
 *  allocating routine.
 *  - Sizes whose moe_w4a16_workspace_size exceeds the array are rejected
 *    with MOE_ERR_WORKSPACE_TOO_SMALL before anything is launched (at E=384,
 *    H=7168, I=2048, top-8 that admits M up to about 24 tokens).
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before
 *    any stream capture.  The address is kept for the life of the process:
 *    after cudaDeviceReset the library's device code is loaded again and
 *    the array may move, so do not call this entry point on a device that
 *    was reset after its first call.
 *  - Devices with an ordinal of 64 or more are not supported: the call
 *    returns MOE_ERR_UNSUPPORTED_DEVICE.
 *  - Every call on a device shares the one array and it keeps the last
 *    call's contents; the call itself resets what must start at zero (the
 *    status word and the split-K tickets).  Calls that overlap on the GPU
 *    (different streams, or the same array used from two threads without
 *    ordering) race and give undefined results.
 *  - Device-detected errors are recorded in the array's status word, which
 *    moe_w4a16_get_device_status cannot reach: use moe_w4a16_forward with a
 *    workspace when those errors must be observed.
 */
moe_status_t moe_w4a16_forward_static(const uint16_t *hidden, const int32_t *topk_ids,
                                      const float *topk_w, const void *w13, const void *w2,
                                      uint16_t *out, int M, int k, int E, int H, int I,
                                      moe_stream_t stream);

/*
 * Wait for `stream`, then return the status word the device recorded in
 * `workspace` during the most recent align/forward call on it (MOE_OK if
 * nothing went wrong).  `detail` (may be NULL) receives a code-specific
 * value: the offending id, or the role whose bounded wait gave up (1 a
 * producer, 2/3 an MMA issuer, 4/5 a dequantisation warp, 6 the epilogue,
 * 7 the single small-batch kernel's wait for activation rows that another
 * CTA writes).
 */
moe_status_t moe_w4a16_get_device_status(const void *workspace,
                                         moe_stream_t stream, int32_t *detail);

/*
 * Where a forward call leaves its intermediates inside the workspace (byte
 * offsets from the workspace start), for inspection after the call has
 * completed and before the next call on the same workspace:
 *   counts [E], offsets [E+1], perm [M*k], inv_perm [M*k]: int32 alignment
 *   act_hi, act_lo [M*k][I] fp16: a = silu(gate)*up in expert-sorted row
 *                  order, as the pair hi + lo (hi = fp16(a), lo = fp16(a - hi))
 *   y [M*k][H] fp32: the down projection of every sorted row.
 * Rows at and beyond offsets[E] are not written.  Returns
 * MOE_ERR_INVALID_ARG for sizes moe_w4a16_workspace_size rejects.
 */
typedef struct {
    size_t counts, offsets, perm, inv_perm, act_hi, act_lo, y;
} moe_ws_views_t;

moe_status_t moe_w4a16_workspace_views(int M, int k, int E, int H, int I,
                                       moe_ws_views_t *views);

/*
 * Diagnostics of the most recent forward call issued from the calling host
 * thread (each thread keeps its own record, so calls from other threads or
 * for other devices do not change it); `calls` counts that thread's forward
 * calls.
 */
typedef struct {
    int32_t version;          /* 2 */
    int32_t M, k, E, H, I;
    int32_t token_tile;       /* token rows per tile of the gate+up GEMM */
    int32_t grid_gemm1;       /* CTAs of the gate+up GEMM */
    int32_t grid_gemm2;       /* CTAs of the down GEMM */
    int32_t kernels_launched; /* kernels one forward call launches */
    int64_t workspace_bytes;  /* bytes of workspace the call used */
    int64_t calls;            /* forward calls since load */
    int32_t token_tile2;      /* token rows per tile of the down GEMM (version 2) */
    int32_t reserved;         /* 0 */
} moe_diag_t;

moe_status_t moe_w4a16_get_diag(moe_diag_t *diag);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */
