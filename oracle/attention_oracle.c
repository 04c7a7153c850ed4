/*
 * Attention oracle: plain, slow, fp64 CPU attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  The GPU product path
 * never calls it and shares no code, header, table or helper with it.
 *
 * What it computes (the plain definition; the pages call the tiled method
 * mathematically identical to it, not an approximation):
 *   - "KingOfEgg: Flash Attention v1" (dandandamowang.xyz), §1.1 Scaled
 *     Dot-Product Attention:  S = Q K^T * scale,  P = softmax_row(S),  O = P V,
 *     with Q, K, V of shape [N, d] per head and heads laid out [B, H, N, D]
 *     (§1.2).
 *   - "08 · FlashAttention", §一: the three unfused steps (S, softmax(S), P V),
 *     which is the pass structure used here for each block of rows.
 *   - "第 13 课：GPU 内核与 FlashAttention", exercise `standard_attention`:
 *     subtract the row maximum before exponentiating.
 *   - "08 · FlashAttention", §四: `is_causal=True`, read as key j <= query i.
 *
 * Per (b, h) slice and query row i, with A(i) = {0..N-1} (or {0..i} causal):
 *   s_ij  = scale * sum_d q_id k_jd            (j in A(i))
 *   m_i   = max_j s_ij
 *   P_ij  = exp(s_ij - m_i) / l_i,   l_i = sum_j exp(s_ij - m_i)
 *   O_id  = sum_j P_ij v_jd
 *   LSE_i = m_i + ln l_i   (natural log of the scaled scores; the pages keep
 *                           only m and l, this is the reading that packs both)
 *
 * Everything is fp64.  Inputs arrive as fp64 copies of the stored (already
 * dtype-rounded) tensors, so bf16 inputs are represented exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ROW_BLOCK 64

/* Number of keys row i may attend to: all N, or 0..i when causal. */
static int64_t keys_for_row(int64_t i, int64_t N, int causal)
{
    if (!causal) return N;
    return i + 1 < N ? i + 1 : N;
}

/*
 * Three passes over a set of rows of ONE (b, h) slice.
 *   rows[r]  : query row index of row r (0..N-1)
 *   qh,kh,vh : the slice's Q, K, V, each [N, D] row-major
 *   S        : scratch of nr * N doubles (the materialised score rows)
 *   o        : output rows, nr x D;  lse: nr values
 * Returns the largest |sum_j P_ij - 1| seen (rows of P must sum to one).
 */
static double attend_rows(const int64_t* rows, int64_t nr,
                          const double* qh, const double* kh, const double* vh,
                          int64_t N, int64_t D, double scale, int causal,
                          double* S, double* o, double* lse)
{
    double worst = 0.0;

    /* pass 1: materialise the score rows S = scale * Q K^T over A(i) */
    for (int64_t r = 0; r < nr; r++) {
        const int64_t i = rows[r];
        const int64_t nk = keys_for_row(i, N, causal);
        const double* qi = qh + i * D;
        double* Sr = S + r * N;
        for (int64_t j = 0; j < nk; j++) {
            const double* kj = kh + j * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; d++) dot += qi[d] * kj[d];
            Sr[j] = scale * dot;
        }
    }

    /* pass 2: stable row softmax, overwriting S with P; LSE = m + ln l */
    for (int64_t r = 0; r < nr; r++) {
        const int64_t nk = keys_for_row(rows[r], N, causal);
        double* Sr = S + r * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; j++) m = Sr[j] > m ? Sr[j] : m;
        double l = 0.0;
        for (int64_t j = 0; j < nk; j++) {
            Sr[j] = exp(Sr[j] - m);
            l += Sr[j];
        }
        double psum = 0.0;
        for (int64_t j = 0; j < nk; j++) {
            Sr[j] /= l;
            psum += Sr[j];
        }
        const double err = fabs(psum - 1.0);
        worst = err > worst ? err : worst;
        lse[r] = m + log(l);
    }

    /* pass 3: O = P V */
    for (int64_t r = 0; r < nr; r++) {
        const int64_t nk = keys_for_row(rows[r], N, causal);
        const double* Pr = S + r * N;
        double* orow = o + r * D;
        for (int64_t d = 0; d < D; d++) orow[d] = 0.0;
        for (int64_t j = 0; j < nk; j++) {
            const double p = Pr[j];
            const double* vj = vh + j * D;
            for (int64_t d = 0; d < D; d++) orow[d] += p * vj[d];
        }
    }
    return worst;
}

/*
 * Full forward over [BH, N, D] inputs (BH = B*H slices, contiguous).
 * o: [BH, N, D], lse: [BH, N].  threads <= 0 means the OpenMP default.
 * *max_rowsum_err (if not NULL) receives the largest |sum_j P_ij - 1|.
 * Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 */
int oracle_attention_fwd(const double* q, const double* k, const double* v,
                         double* o, double* lse,
                         int64_t BH, int64_t N, int64_t D, double scale, int causal,
                         int threads, double* max_rowsum_err)
{
    if (!q || !k || !v || !o || !lse || BH < 1 || N < 1 || D < 1) return 1;
    const int64_t nblk = (N + ORACLE_ROW_BLOCK - 1) / ORACLE_ROW_BLOCK;
    const int64_t total = BH * nblk;
    double worst = 0.0;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads) reduction(max : worst) reduction(| : failed)
#endif
    for (int64_t t = 0; t < total; t++) {
        const int64_t bh = t / nblk;
        const int64_t r0 = (t % nblk) * ORACLE_ROW_BLOCK;
        const int64_t r1 = r0 + ORACLE_ROW_BLOCK < N ? r0 + ORACLE_ROW_BLOCK : N;
        const int64_t nr = r1 - r0;
        int64_t rows[ORACLE_ROW_BLOCK];
        for (int64_t r = 0; r < nr; r++) rows[r] = r0 + r;
        double* S = (double*)malloc((size_t)(nr * N) * sizeof(double));
        if (!S) { failed = 1; continue; }
        const double* qh = q + bh * N * D;
        const double* kh = k + bh * N * D;
        const double* vh = v + bh * N * D;
        const double e = attend_rows(rows, nr, qh, kh, vh, N, D, scale, causal, S,
                                     o + (bh * N + r0) * D, lse + bh * N + r0);
        worst = e > worst ? e : worst;
        free(S);
    }
    if (max_rowsum_err) *max_rowsum_err = worst;
    return failed ? 2 : 0;
}

/*
 * The same definition for a sample of rows: row r is query row_idx[r] of slice
 * bh_idx[r].  o_rows: [nrows, D], lse_rows: [nrows].  Rows are independent, so
 * each sampled row is exactly the row the full forward would produce.
 */
int oracle_attention_rows(const double* q, const double* k, const double* v,
                          int64_t BH, int64_t N, int64_t D, double scale, int causal,
                          const int64_t* bh_idx, const int64_t* row_idx, int64_t nrows,
                          double* o_rows, double* lse_rows, int threads)
{
    if (!q || !k || !v || !bh_idx || !row_idx || !o_rows || !lse_rows) return 1;
    if (BH < 1 || N < 1 || D < 1 || nrows < 0) return 1;
    for (int64_t r = 0; r < nrows; r++)
        if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= N) return 1;
    int failed = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads) reduction(| : failed)
#endif
    for (int64_t r = 0; r < nrows; r++) {
        double* S = (double*)malloc((size_t)N * sizeof(double));
        if (!S) { failed = 1; continue; }
        const int64_t bh = bh_idx[r];
        attend_rows(&row_idx[r], 1, q + bh * N * D, k + bh * N * D, v + bh * N * D,
                    N, D, scale, causal, S, o_rows + r * D, lse_rows + r);
        free(S);
    }
    return failed ? 2 : 0;
}

/* Number of OpenMP threads a call with threads <= 0 would use (1 without OpenMP). */
int oracle_default_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
