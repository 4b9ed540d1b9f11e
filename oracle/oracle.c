/*
 * CPU oracle for the tensor-parallel row-parallel linear epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library or its Python binding may
 * include, link, load or call this file; only the tests, the smoke check and
 * the bench's CPU-baseline / reference arm do.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * It is deliberately plain and slow: straight loops in the order the method
 * states, fp32 where the method fixes fp32, fp64 for the RMSNorm statistics.
 * An OpenMP loop over independent output rows is the only parallelism; it does
 * not change the order of any per-element sum.  Built with -ffp-contract=off so
 * that no multiply-add is fused.
 *
 * Sources (web pages, cited by title and section):
 *  [RING]  DeepGEMM PR #1 "Fused ring RS: per-tile bitmask + drain-ring with
 *          owner-boundary flush", description: a fused BF16 GEMM whose fp32
 *          per-rank partials are reduce-scattered into owner row segments,
 *          readiness tracked per output tile.
 *  [LAMP]  ROCm/aiter PR #4977 "Single-kernel Lamport fused all-reduce +
 *          RMSNorm", sections "Approach" and "Correctness notes": the -0.0
 *          sentinel (0x8000 per bf16 lane, 0x80000000 per fp32 word),
 *          producer-side -0.0 -> +0.0 canonicalisation, a pack has arrived
 *          only when no word equals the sentinel; bring-up section: checked
 *          against torch's F.rms_norm.
 *  [MORI]  ROCm/mori PR #662 "Fuse DSV4-Pro wo_b's GEMM with its all-reduce",
 *          description: the all-reduce of bf16 partial outputs [M, 7168].
 * Where the pages leave a step open, the reading taken is stated at the
 * function.
 *
 * Parity pins: every function below is pinned by tests that do not re-type
 * its formula (fp64 brute force, exact integer cases, identity/one-hot
 * operands, order-sensitive sums, torch's rms_norm in fp64, closed forms);
 * the one thing not pinned here is the tensor core's internal accumulation
 * order, which the GPU comparison covers only through its tolerance.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0 /* >0 only in the pin-strength tests: plants a known mistake */
#endif

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                              */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32; widening is exact. */
static float bf16_to_f32(uint16_t b) {
    uint32_t x = (uint32_t)b << 16;
    float f;
    memcpy(&f, &x, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays NaN (quiet bit set). */
uint16_t oracle_bf16_rne(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x007FFFFFu) != 0) return (uint16_t)((x >> 16) | 0x0040u);
    uint32_t upper = x >> 16, lower = x & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* oracle_bf16_rne applied to n floats (the same function, element by element). */
void oracle_bf16_rne_n(const float *x, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(x[i]);
}

static void set_threads(int nthreads);

/*
 * fp32 -> FP8 E4M3 (OCP "e4m3fn": bias 7, no infinities, max finite 448 =
 * code 0x7E, NaN = 0x7F), round to nearest even, saturating to +-448.  Written
 * from the format's definition on the fp32 bits.
 */
uint8_t oracle_e4m3_rne_sat(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    const uint8_t sign = (uint8_t)((x >> 24) & 0x80u);
    const uint32_t E = (x >> 23) & 0xFFu, Mt = x & 0x7FFFFFu;
    if (E == 0xFFu && Mt != 0) return (uint8_t)(sign | 0x7Fu);  /* NaN */
    if (E == 0xFFu) return (uint8_t)(sign | 0x7Eu);              /* +-inf saturates */
    if (E == 0) return sign;                                     /* fp32 zero or subnormal: below 2^-10 */
    const int e = (int)E - 127;
    const uint64_t sig = (1ull << 23) | Mt;                      /* value = sig * 2^(e-23) */
    uint32_t code;
    if (e >= -6) {                                               /* e4m3 normal range */
        uint64_t q = sig >> 20, rem = sig & ((1ull << 20) - 1), half = 1ull << 19;
        if (rem > half || (rem == half && (q & 1u))) ++q;        /* q in [8, 16] */
        int ee = e;
        if (q == 16) { q = 8; ++ee; }
        const int be = ee + 7;
        if (be > 15 || (be == 15 && (q & 7u) > 6)) return (uint8_t)(sign | 0x7Eu);
        code = ((uint32_t)be << 3) | (uint32_t)(q & 7u);
    } else {                                                     /* subnormal: units of 2^-9 */
        const int shift = 14 - e;                                /* value / 2^-9 = sig / 2^shift */
        if (shift >= 63) return sign;
        uint64_t q = sig >> shift, rem = sig & ((1ull << shift) - 1), half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) ++q;        /* q in [0, 8]; 8 is 2^-6, code 0x08 */
        code = (uint32_t)q;
    }
    return (uint8_t)(sign | code);
}

/*
 * The quantising variant of the RMSNorm step, per row (dynamic, per token):
 *   y_j   = h_j / sqrt(ms + eps) * gamma_j     (as oracle_rmsnorm_rows, fp32)
 *   amax  = max_j |y_j|;  scale = amax / 448 (fp32 division; 1 if amax == 0)
 *   q_j   = e4m3(y_j / scale)                  (fp32 division, RNE, saturating)
 * x (optional) receives y_j / scale, the value each code rounds.
 */
void oracle_quant_rows(const float *y, int64_t M, int64_t N, uint8_t *q, float *scale, float *x, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        float amax = 0.0f;
        for (int64_t j = 0; j < N; ++j) {
            const float a = fabsf(y[i * N + j]);
            if (a > amax) amax = a;
        }
        const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[i] = sc;
        for (int64_t j = 0; j < N; ++j) {
            const float v = y[i * N + j] / sc;
            if (x) x[i * N + j] = v;
            q[i * N + j] = oracle_e4m3_rne_sat(v);
        }
    }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Per-rank partial GEMM  [RING], description ("fused BF16 GEMM", fp32 acc)   */
/* ------------------------------------------------------------------------ */

/*
 * One row i of P = A . B:  P[i][j] = sum_{k=0}^{K-1} f32(A[i][k]) * f32(B[k][j]).
 * A is [M,K] row-major, B is [K,N] row-major.  The product of two bf16 values is
 * exact in fp32; the sum is taken in increasing k, one fp32 add at a time,
 * starting from the k=0 product (i-k-j loop order).
 */
static void partial_row(const uint16_t *A, const uint16_t *B, int64_t N, int64_t K, int64_t i, float *prow) {
    for (int64_t j = 0; j < N; ++j) prow[j] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float a = bf16_to_f32(A[i * K + k]);
        const uint16_t *brow = B + k * N;
#if ORACLE_PLANT == 1 /* planted: transposed operand (reads B as [N,K]) */
        for (int64_t j = 0; j < N; ++j) prow[j] = prow[j] + a * bf16_to_f32(B[j * K + k]);
        (void)brow;
#else
        for (int64_t j = 0; j < N; ++j) {
            float prod = a * bf16_to_f32(brow[j]);
            prow[j] = (k == 0) ? prod : prow[j] + prod;
        }
#endif
    }
}

/* Full partial product P = A . B  ([M,N] fp32). */
void oracle_partial_gemm(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K, float *P,
                         int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) partial_row(A, B, N, K, i, P + i * N);
}

/*
 * GEMM + reduce: selected rows of the reduced result over R ranks.
 *   mode 0 (GEMM+RS):  Y = ((P_0 + P_1) + P_2) + ... + P_{R-1}, fp32 partials,
 *                      not rounded  ([RING] description: fp32 partials summed
 *                      along the ring; the fixed order r = 0..R-1 is the one the
 *                      benchmark workloads state for every segment).
 *   mode 1 (GEMM+AR):  Y = sum_r f32(bf16(P_r)) in the same order: the all-reduce
 *                      inputs are the ranks' bf16 GEMM outputs ([MORI], an
 *                      all-reduce of bf16 [M, 7168] outputs).
 * rows[0..nrows) index A's rows; Y is [nrows, N].
 */
void oracle_gemm_reduce_rows(const uint16_t *const *A, const uint16_t *const *B, int R, int64_t M, int64_t N,
                             int64_t K, const int64_t *rows, int64_t nrows, int mode, float *Y, int nthreads) {
    (void)M;
    set_threads(nthreads);
#pragma omp parallel
    {
        float *prow = (float *)malloc((size_t)N * sizeof(float));
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nrows; ++q) {
            float *y = Y + q * N;
            for (int r = 0; r < R; ++r) {
#if ORACLE_PLANT == 2 /* planted: dropped term (last rank never added) */
                if (r == R - 1 && R > 1) break;
#endif
                partial_row(A[r], B[r], N, K, rows[q], prow);
                if (mode == 1)
                    for (int64_t j = 0; j < N; ++j) prow[j] = bf16_to_f32(oracle_bf16_rne(prow[j]));
                if (r == 0) {
                    for (int64_t j = 0; j < N; ++j) y[j] = prow[j];
                } else {
#if ORACLE_PLANT == 3 /* planted: wrong sign on the ring sum */
                    for (int64_t j = 0; j < N; ++j) y[j] = y[j] - prow[j];
#else
                    for (int64_t j = 0; j < N; ++j) y[j] = y[j] + prow[j];
#endif
                }
            }
        }
        free(prow);
    }
}

/* ------------------------------------------------------------------------ */
/* Owner segments  [RING], title ("owner-boundary flush") and description     */
/* ------------------------------------------------------------------------ */

/*
 * Rank s owns the contiguous row band [s*S, (s+1)*S), S = M / R (M divisible
 * by R).  owner(row) = floor(row / S).
 */
int oracle_owner_of_row(int64_t row, int64_t M, int R) {
    int64_t S = M / R;
#if ORACLE_PLANT == 4 /* planted: off-by-one owner */
    return (int)((row + 1) / S < R ? (row + 1) / S : R - 1);
#else
    return (int)(row / S);
#endif
}

/*
 * Reading of "owner-boundary flush" (the pages give only the phrase): the rows
 * of one output tile [row0, row0+BM) ∩ [0, M) are cut at every owner-segment
 * boundary, and each piece is flushed to its owner.  Writes the pieces in
 * increasing row order as (segment, first row, one-past-last row) in absolute
 * row numbers; returns their count.
 */
int oracle_tile_pieces(int64_t row0, int64_t BM, int64_t M, int R, int64_t *seg, int64_t *begin, int64_t *end) {
    int64_t S = M / R;
    int64_t hi = row0 + BM < M ? row0 + BM : M;
    int n = 0;
    for (int64_t row = row0; row < hi;) {
        int s = oracle_owner_of_row(row, M, R);
        int64_t seg_end = (int64_t)(s + 1) * S;
        int64_t e = seg_end < hi ? seg_end : hi;
        seg[n] = s; begin[n] = row; end[n] = e;
        ++n;
        row = e;
    }
    return n;
}

/*
 * Per-tile ready bitmask ([RING], description: a per-tile bitmask replaces the
 * per-segment flag).  Bit r of tile t's word is rank r's partial of tile t.
 * Once every rank has published tile t the word is (1 << R) - 1; tiles are
 * BM x BN over the [M, N] output, T = ceil(M/BM) * ceil(N/BN).  Fills
 * words[0..nwords) with the expected state after every tile of one call has
 * been published and none has been re-armed; returns T.
 */
int64_t oracle_expected_masks(int R, int64_t M, int64_t N, int64_t BM, int64_t BN, uint32_t *words, int64_t nwords) {
    int64_t T = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    uint32_t full = (R >= 32) ? 0xFFFFFFFFu : ((1u << R) - 1u);
    for (int64_t t = 0; t < nwords; ++t) words[t] = (t < T) ? full : 0u;
    return T;
}

/*
 * Chunked owner-segment completion ([MORI], the fused GEMM -> scatter
 * follow-ups: per-(destination, chunk) completion counters; the chunk count
 * "halved until it divides the M-tiles per destination").  Reading for row
 * owners: destination s is owner segment s = rows [s*S, (s+1)*S); its M-tiles
 * are the n_s output tile rows of height BM that intersect it (a tile that
 * straddles two segments is an M-tile of both).  The requested count C is
 * halved (integer halving) until it divides n_s, giving C_s chunks; chunk c
 * of segment s is its tile rows [c*n_s/C_s, (c+1)*n_s/C_s) in increasing
 * order.  One piece is one output tile's rows stored into one segment, so a
 * chunk completes after (n_s/C_s) * ceil(N/BN) pieces.  Fills pieces[s*C + c]
 * with that count for c < C_s and 0 for the chunks a segment does not use.
 */
void oracle_chunk_pieces(int R, int64_t M, int64_t N, int64_t BM, int64_t BN, int C, int64_t *pieces) {
    int64_t S = M / R;
    int64_t tiles_n = (N + BN - 1) / BN;
    for (int s = 0; s < R; ++s) {
        for (int c = 0; c < C; ++c) pieces[(int64_t)s * C + c] = 0;
        if (S == 0 || tiles_n == 0) continue;
        int64_t t_lo = ((int64_t)s * S) / BM;
        int64_t t_hi = ((int64_t)(s + 1) * S - 1) / BM;
        int64_t n_s = t_hi - t_lo + 1;
        int64_t cs = C;
#if ORACLE_PLANT == 7 /* planted: halves only until the count is at most the M-tiles */
        while (cs > n_s) cs /= 2;
#else
        while (cs > 1 && n_s % cs != 0) cs /= 2;
#endif
        if (cs < 1) cs = 1;
        for (int64_t c = 0; c < cs; ++c) pieces[(int64_t)s * C + c] = (n_s / cs) * tiles_n;
    }
}

/* ------------------------------------------------------------------------ */
/* All-reduce + residual + RMSNorm  [LAMP]                                    */
/* ------------------------------------------------------------------------ */

/*
 * Phase A of the Lamport all-reduce, as the value it stages:
 *   s = sum_{r=0}^{R-1} f32(x_r)  in the fixed order r = 0..R-1 (fp32 adds),
 *   then the producer-side canonicalisation: an s whose bits are 0x80000000
 *   (-0.0, the fp32 sentinel) is staged as +0.0 ([LAMP], Approach:
 *   "Producers canonicalise -0.0 -> +0.0").
 * Reading: the staging words are fp32 (the fp32 sentinel 0x80000000 of the
 * page), so the reduced sum is not rounded before the residual add.
 * s is [M, N]; returns how many words were canonicalised.
 */
int64_t oracle_ar_stage(const uint16_t *const *x, int R, int64_t M, int64_t N, float *s, int nthreads) {
    int64_t count = 0;
    set_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(+ : count)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            int64_t e = i * N + j;
            float acc = bf16_to_f32(x[0][e]);
            for (int r = 1; r < R; ++r) acc = acc + bf16_to_f32(x[r][e]);
            uint32_t bits;
            memcpy(&bits, &acc, 4);
#if ORACLE_PLANT != 5 /* planted: canonicalisation skipped */
            if (bits == 0x80000000u) { acc = 0.0f; ++count; }
#endif
            s[e] = acc;
        }
    }
    return count;
}

/*
 * Phase B per row: h = s + f32(residual) (fp32 add; residual may be NULL = 0),
 * then RMSNorm as torch's F.rms_norm defines it ([LAMP], bring-up: compared
 * against F.rms_norm):
 *   ms = (1/N) sum_j h_j^2          (accumulated in fp64)
 *   y_j = h_j / sqrt(ms + eps) * gamma_j   (fp64, then one rounding to fp32)
 * y is the unrounded fp32 reference [M, N]; h_out (optional) receives h.
 */
void oracle_rmsnorm_rows(const float *s, const uint16_t *residual, const float *gamma, float eps, int64_t M,
                         int64_t N, float *y, float *h_out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel
    {
        double *h = (double *)malloc((size_t)N * sizeof(double));
#pragma omp for schedule(static)
        for (int64_t i = 0; i < M; ++i) {
            double ss = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                float hf = s[i * N + j];
                if (residual) hf = hf + bf16_to_f32(residual[i * N + j]);
                if (h_out) h_out[i * N + j] = hf;
                h[j] = (double)hf;
                ss += h[j] * h[j];
            }
#if ORACLE_PLANT == 6 /* planted: eps outside the square root */
            double inv = 1.0 / (sqrt(ss / (double)N) + (double)eps);
#else
            double inv = 1.0 / sqrt(ss / (double)N + (double)eps);
#endif
            for (int64_t j = 0; j < N; ++j) y[i * N + j] = (float)(h[j] * inv * (double)gamma[j]);
        }
        free(h);
    }
}
