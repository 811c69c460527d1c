/*
 * moe_oracle.c -- plain, slow CPU oracle of the weight-only-INT4 MoE layer
 * forward (top-k alignment, gate+up GEMM with SiLU(gate)*up, down GEMM,
 * fixed-order top-k combine).
 *
 * TEST INFRASTRUCTURE ONLY.  It exists to check the CUDA library against
 * the definition of the method.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg load it; the library never does, and the
 * two share no code, header, table or helper.
 *
 * Arithmetic is IEEE double throughout (inputs are converted exactly: bf16
 * and fp32 are subsets of double).  Every sum runs over ascending index in a
 * single accumulator; there is no blocking, fusion or reordering.  OpenMP
 * only splits independent output elements across threads, so the result is
 * bit-identical for any thread count.  Build without -ffast-math.
 *
 * Sources of the definition (page title, section):
 *  - "The MoE Throughput Lever: Quantifying the INT4 Marlin GEMM on Blackwell
 *    PRO 6000", section "The Benchmark: What Was Measured": the layer is an
 *    INT4, group-size-32, 16-bit-activation MoE GEMM with E=384 experts,
 *    hidden 7168, intermediate 2048, top-8 routing.
 *  - "perf(exl3): accelerate fat-expert prefill - #77", sections "Rollout"
 *    and "Summary": tokens are grouped by expert ("sorted routing") and each
 *    expert's rows run as one batch (E1 batching); gate and up are one stacked
 *    GEMM over a shared input.
 *  - "DeepSeek-V4.1-Flash-EXL3 ... Detailed results", section "Nsight Compute
 *    on the stock kernel": the per-expert counts are prefix-scanned (the
 *    pages profile a serial scan over 384 counts).
 * The pages print no formula.  The readings used here (each one is also
 * listed in the design notes):
 *  - dequantised weight = (q - 8) * scale, q in [0, 15], one bf16 scale per
 *    group of consecutive elements along K (the reduction axis): 32 as on
 *    the pages, or 64 / 128 for the wider-group variant;
 *  - canonical packing: byte kk/2 of a row holds element kk in its low nibble
 *    when kk is even and in its high nibble when kk is odd;
 *  - w13 rows [0, I) are the gate projection, rows [I, 2I) the up projection;
 *  - activation a = silu(gate) * up with silu(v) = v / (1 + exp(-v));
 *  - the permutation is a stable counting sort of the flat slot index
 *    f = t*k + j by expert id (ascending f inside each expert segment);
 *  - out[t] = sum over j = 0..k-1 ascending of topk_w[t][j] * y(t, j), with no
 *    renormalisation of topk_w;
 *  - a slot whose expert id lies outside [0, E) is left out of the alignment
 *    (inv_perm = -1) and contributes zero;
 *  - the router (oracle_route, ahead of the layer): softmax over the E
 *    logits, top-k by descending value with ties to the lower expert index,
 *    weights renormalised to sum 1 over the k selected.
 *
 * Parity status: every function here is pinned by the CPU tests (worked
 * byte/scale fixtures, closed forms, a brute-force dense per-token path,
 * stable-sort equivalence, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double, exact: a bf16 is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Logical 4-bit code q in [0,15] of element (n, kk) of one expert's packed
 * [N][K/2] byte matrix. */
static int code_at(const uint8_t *q, int64_t K, int64_t n, int64_t kk)
{
    uint8_t byte = q[n * (K / 2) + kk / 2];
    return (kk & 1) ? (byte >> 4) : (byte & 0x0F);
}

/* Dequantised weight W[n][kk] = (q - 8) * scale[n][kk / group]. */
static double weight_at(const uint8_t *q, const uint16_t *s, int64_t K,
                        int64_t group, int64_t n, int64_t kk)
{
    int code = code_at(q, K, n, kk);
    double scale = bf16_to_double(s[n * (K / group) + kk / group]);
    return (double)(code - 8) * scale;
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Exposed for the byte-level pins: dequantised value of element (n, kk) of
 * a single [N][K/2] packed matrix with [N][K/group] bf16 scales. */
double oracle_dequant_element(const uint8_t *q, const uint16_t *s, int64_t K,
                              int64_t group, int64_t n, int64_t kk)
{
    return weight_at(q, s, K, group, n, kk);
}

/*
 * Alignment: stable counting sort of the M*k (token, slot) pairs by expert.
 *   counts[e]      = number of valid slots routed to expert e
 *   offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]   (E+1 entries)
 *   perm[offsets[e] + r] = f, the r-th flat index (ascending) with ids[f] = e
 *   inv_perm[f]    = position of f in perm, or -1 for an out-of-range id
 * Returns the number of slots with an id outside [0, E).
 */
int64_t oracle_align(const int32_t *ids, int64_t M, int64_t k, int64_t E,
                     int32_t *counts, int32_t *offsets, int32_t *perm,
                     int32_t *inv_perm)
{
    int64_t n_slots = M * k, invalid = 0;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t f = 0; f < n_slots; ++f) {
        int32_t e = ids[f];
        if (e < 0 || e >= E) { ++invalid; continue; }
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    /* second ordered pass: place f at offsets[e] + cursor[e]++ */
    for (int64_t e = 0; e < E; ++e) counts[e] = 0; /* reused as cursor */
    for (int64_t f = 0; f < n_slots; ++f) {
        int32_t e = ids[f];
        if (e < 0 || e >= E) { inv_perm[f] = -1; continue; }
        int32_t pos = offsets[e] + counts[e];
        counts[e] += 1;
        perm[pos] = (int32_t)f;
        inv_perm[f] = pos;
    }
    return invalid;
}

/*
 * Layer forward.  Shapes (row-major, canonical packing):
 *   hidden [M][H] bf16 bits        ids [M][k] int32      topk_w [M][k] fp32
 *   w13 [E][2I][H/2] uint8         s13 [E][2I][H/32] bf16 bits
 *   w2  [E][H][I/2]  uint8         s2  [E][H][I/32]  bf16 bits
 * Outputs:
 *   out [M][H] double (before any output rounding)
 *   act [M*k][I] double, optional (NULL to skip): a in sorted order
 *   yrow [M*k][H] double, required: y in sorted order (the combine reads it)
 *   counts [E], offsets [E+1], perm [M*k], inv_perm [M*k]: the alignment
 * Scratch: when act is NULL, a_scratch holds I doubles per OpenMP thread
 *          (a_scratch_len >= oracle_num_threads() * I).
 * Returns the number of out-of-range slots, or -1 if a_scratch is short.
 */
int64_t oracle_forward(const uint16_t *hidden, const int32_t *ids,
                       const float *topk_w,
                       const uint8_t *w13, const uint16_t *s13,
                       const uint8_t *w2, const uint16_t *s2,
                       int64_t M, int64_t k, int64_t E, int64_t H, int64_t I,
                       int64_t group,
                       double *out, double *act, double *yrow,
                       int32_t *counts, int32_t *offsets, int32_t *perm,
                       int32_t *inv_perm, double *a_scratch,
                       int64_t a_scratch_len)
{
    int64_t invalid = oracle_align(ids, M, k, E, counts, offsets, perm, inv_perm);
    int64_t n_valid = offsets[E];
    const int64_t w13_expert = 2 * I * (H / 2), s13_expert = 2 * I * (H / group);
    const int64_t w2_expert = H * (I / 2), s2_expert = H * (I / group);
    if (!act && a_scratch_len < (int64_t)oracle_num_threads() * I) return -1;

    /* Grouped stages: each sorted position p is one (token, slot) row of its
     * expert's batch.  Rows are independent, so threads split them. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < n_valid; ++p) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *a = act ? act + p * I : a_scratch + (int64_t)tid * I;
        int64_t f = perm[p];
        int64_t t = f / k;
        int64_t e = ids[f];
        const uint16_t *x = hidden + t * H;
        const uint8_t *q13 = w13 + e * w13_expert;
        const uint16_t *sc13 = s13 + e * s13_expert;
        const uint8_t *q2 = w2 + e * w2_expert;
        const uint16_t *sc2 = s2 + e * s2_expert;

        /* gate+up projection, then SiLU(gate) * up */
        for (int64_t n = 0; n < I; ++n) {
            double g = 0.0, u = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                double xv = bf16_to_double(x[h]);
                g += xv * weight_at(q13, sc13, H, group, n, h);
                u += xv * weight_at(q13, sc13, H, group, I + n, h);
            }
            a[n] = silu(g) * u;
        }
        /* down projection */
        double *y = yrow + p * H;
        for (int64_t hh = 0; hh < H; ++hh) {
            double acc = 0.0;
            for (int64_t n = 0; n < I; ++n)
                acc += a[n] * weight_at(q2, sc2, I, group, hh, n);
            y[hh] = acc;
        }
    }

    /* combine: ascending slot order, weights used as given */
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < M; ++t) {
        for (int64_t hh = 0; hh < H; ++hh) {
            double acc = 0.0;
            for (int64_t j = 0; j < k; ++j) {
                int32_t pos = inv_perm[t * k + j];
                if (pos < 0) continue;
                acc += (double)topk_w[t * k + j] * yrow[(int64_t)pos * H + hh];
            }
            out[t * H + hh] = acc;
        }
    }
    return invalid;
}

/*
 * Router front-end (the step that produces topk_ids and topk_w from the
 * router's logits).  The pages do not describe the router; the reading used
 * is the usual softmax top-k with renormalisation:
 *   p[e] = exp(l[e]) / sum_e' exp(l[e'])              (softmax over all E)
 *   ids[t][0..k-1] = the k experts of largest p, in descending order, the
 *                    lower expert index first among equal values
 *   w[t][j] = p[ids[t][j]] / sum_{j' < k} p[ids[t][j']]   (renormalised)
 * The softmax is monotone, so the order is taken on the logits themselves,
 * compared as numbers (-0 equals +0).  Inputs outside the ordinary range:
 *  - a logit of -inf has p = 0 and ranks after every finite logit;
 *  - NaN ranks after everything else (lower index first among NaNs);
 *  - a row holding a NaN or +inf has no softmax: its ids still follow the
 *    order above, its weights are all 0, and it is counted as a bad row;
 *  - a row whose logits are all -inf has weights all 0 (not a bad row).
 * Arithmetic in double; the weights are rounded once to fp32.
 * Returns the number of bad rows.
 */

/* 1 when logit a of expert ea comes before logit b of expert eb. */
static int ranks_before(float a, int64_t ea, float b, int64_t eb)
{
    int an = isnan(a), bn = isnan(b);
    if (an != bn) return bn;           /* the number comes first */
    if (!an && a != b) return a > b;   /* larger first; -0 == +0 */
    return ea < eb;                    /* equal (or both NaN): lower index */
}

int64_t oracle_route(const float *logits, int64_t M, int64_t E, int64_t k,
                     int32_t *ids, float *topk_w)
{
    int64_t bad_rows = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad_rows)
    for (int64_t t = 0; t < M; ++t) {
        const float *l = logits + t * E;
        int32_t *id = ids + t * k;
        float *w = topk_w + t * k;

        /* selection: k passes, each taking the first-ranked expert not yet
         * taken */
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                int taken = 0;
                for (int64_t i = 0; i < j; ++i)
                    if (id[i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
            }
            id[j] = (int32_t)best;
        }

        int bad = 0;
        double mx = -INFINITY;
        for (int64_t e = 0; e < E; ++e) {
            if (isnan(l[e]) || (isinf(l[e]) && l[e] > 0)) bad = 1;
            else if ((double)l[e] > mx) mx = (double)l[e];
        }
        if (bad || mx == -INFINITY) {
            for (int64_t j = 0; j < k; ++j) w[j] = 0.0f;
            bad_rows += bad;
            continue;
        }
        /* softmax over all E (shifted by the maximum, which leaves it
         * unchanged), then renormalised over the selected k */
        double z = 0.0;
        for (int64_t e = 0; e < E; ++e) z += exp((double)l[e] - mx);
        double sel = 0.0;
        for (int64_t j = 0; j < k; ++j) sel += exp((double)l[id[j]] - mx) / z;
        for (int64_t j = 0; j < k; ++j)
            w[j] = (float)((exp((double)l[id[j]] - mx) / z) / sel);
    }
    return bad_rows;
}
