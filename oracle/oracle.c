/*
 * Oracle for FlashMask-style masked attention: plain, slow, fp64, CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it computes and where the definition comes from
 * ----------------------------------------------------
 * Mask (FlashMask, arXiv 2410.01359, abstract: "column-wise sparse
 * representation of attention masks"): for key column j two masked row
 * ranges, lower [lts_j, lte_j) and upper [uts_j, ute_j), half open; a range
 * with start >= end is empty; element (i, j) is masked when row i lies in
 * either range.
 *
 * Row form (blog post "FlashMask技术", §2.1 causal example, §3.3 document
 * packing, §4.1 item 3 "mask fused into the softmax"): row i attends column j
 * exactly when col_start_i <= j <= col_end_i.
 * Multi-interval row form (same blog, §6.1 item 1, several disjoint intervals
 * per row; the sink-token window of the §5 streaming example is one): row i
 * attends column j exactly when start_ik <= j <= end_ik for some slot k
 * (inclusive, as in §3.3; a slot with start > end attends nothing).
 *
 * Attention: the pages state the method is exact ("mathematically
 * equivalent", blog §2.2; "without sacrificing computational accuracy",
 * abstract), so the oracle is plain masked softmax attention:
 *     s_ij   = scale * q_i . k_j                  (on the bf16 input values)
 *     A_i    = { j : (i, j) not masked }
 *     lse_i  = ln sum_{j in A_i} exp(s_ij)        (max subtracted first, the
 *                                                  stabilisation of the
 *                                                  FlashAttention article §二.2)
 *     O_i    = sum_{j in A_i} exp(s_ij - lse_i) v_j
 * A row with A_i empty gets O_i = 0 and lse_i = -inf.
 * Backward is the exact derivative of O with upstream gradient dO:
 *     P_ij  = exp(s_ij - lse_i) on A_i, 0 elsewhere
 *     dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij,   dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i,
 *     dV_j  = sum_i P_ij dO_i
 *
 * Tile labels (blog §2.2, the three-way skip / full / masked decision per
 * (Q block, KV block)).  The printed test is garbled; the reading used is:
 * canonicalise each column's ranges (empty lower -> (N, N), empty upper ->
 * (0, 0)), take the min and max of each of the four bounds over the KV
 * block's columns, and for the Q block rows [qb, qe)
 *     SKIP    if every column's lower range covers [qb, qe) (L0max <= qb and
 *             L1min >= qe) or every column's upper range does;
 *     FULL    if not SKIP and every column's lower range misses [qb, qe)
 *             (L0min >= qe or L1max <= qb) and every upper range does too;
 *     PARTIAL otherwise.
 * oracle_tile_labels_exact gives the labels of the dense mask itself (all
 * masked / none masked / mixed) so the rule's soundness can be checked.
 *
 * Everything is row- or column-parallel with OpenMP; no cross-thread
 * reductions, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- mask rules ---------------------------------------------------------- */

static int masked_col_rule(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                           const int32_t *ute, int64_t i, int64_t j)
{
    return (lts[j] <= i && i < lte[j]) || (uts[j] <= i && i < ute[j]);
}

/* M[i*N + j] = 1 where (i, j) is masked under the column rule. */
void oracle_dense_from_cols(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                            const int32_t *ute, int64_t N, uint8_t *M)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < N; ++j)
            M[i * N + j] = (uint8_t)masked_col_rule(lts, lte, uts, ute, i, j);
}

/* M[i*N + j] = 1 where (i, j) is masked under the row rule (not attended). */
void oracle_dense_from_rows(const int32_t *cs, const int32_t *ce, int64_t N, uint8_t *M)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < N; ++j)
            M[i * N + j] = (uint8_t)!(cs[i] <= j && j <= ce[i]);
}

/* M[i*N + j] = 1 where no interval of row i contains j (starts, ends: [N, K]). */
void oracle_dense_from_row_intervals(const int32_t *starts, const int32_t *ends, int64_t N, int64_t K,
                                     uint8_t *M)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int attended = 0;
            for (int64_t k = 0; k < K; ++k)
                if (starts[i * K + k] <= j && j <= ends[i * K + k]) attended = 1;
            M[i * N + j] = (uint8_t)!attended;
        }
}

/* Number of attended (unmasked) pairs, counted element by element. */
int64_t oracle_attended_pairs(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                              const int32_t *ute, int64_t N)
{
    int64_t total = 0;
#pragma omp parallel for schedule(static) reduction(+ : total)
    for (int64_t j = 0; j < N; ++j) {
        int64_t c = 0;
        for (int64_t i = 0; i < N; ++i)
            c += !masked_col_rule(lts, lte, uts, ute, i, j);
        total += c;
    }
    return total;
}

/* ---- forward ------------------------------------------------------------- */

static double dot(const float *a, const float *b, int d)
{
    double s = 0.0;
    for (int k = 0; k < d; ++k)
        s += (double)a[k] * (double)b[k];
    return s;
}

/* Scores of row i against every attended column; returns lse_i (or -inf).
 * s[j] holds scale*q_i.k_j for attended j; att[j] = 1 for attended j. */
static double row_scores(const float *q, const float *k, const int32_t *lts, const int32_t *lte,
                         const int32_t *uts, const int32_t *ute, int64_t N, int d, double scale,
                         int64_t i, double *s, uint8_t *att)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        att[j] = (uint8_t)!masked_col_rule(lts, lte, uts, ute, i, j);
        if (att[j]) {
            s[j] = scale * dot(q + i * d, k + j * d, d);
            if (s[j] > m)
                m = s[j];
        }
    }
    if (m == -INFINITY)
        return -INFINITY;
    double sum = 0.0;
    for (int64_t j = 0; j < N; ++j)
        if (att[j])
            sum += exp(s[j] - m);
    return m + log(sum);
}

/* One head: q, k, v are [N][d] float (bf16 values).  Computes O [nrows][d]
 * and lse [nrows] for the listed rows. */
void oracle_fwd_rows(const float *q, const float *k, const float *v, const int32_t *lts,
                     const int32_t *lte, const int32_t *uts, const int32_t *ute, int64_t N, int d,
                     double scale, const int64_t *rows, int64_t nrows, double *O, double *lse)
{
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        uint8_t *att = (uint8_t *)malloc((size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t i = rows[r];
            const double L = row_scores(q, k, lts, lte, uts, ute, N, d, scale, i, s, att);
            double *o = O + r * d;
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            lse[r] = L;
            if (L == -INFINITY)
                continue;
            for (int64_t j = 0; j < N; ++j) {
                if (!att[j])
                    continue;
                const double p = exp(s[j] - L);
                for (int c = 0; c < d; ++c)
                    o[c] += p * (double)v[j * d + c];
            }
        }
        free(s);
        free(att);
    }
}

/* ---- backward ------------------------------------------------------------ */

/* Row pass for the listed rows: lse_i, D_i = sum_j P_ij dP_ij and
 * dQ_i = scale sum_j dS_ij k_j.  dQ is [nrows][d]. */
void oracle_bwd_rows(const float *q, const float *k, const float *v, const float *dO,
                     const int32_t *lts, const int32_t *lte, const int32_t *uts,
                     const int32_t *ute, int64_t N, int d, double scale, const int64_t *rows,
                     int64_t nrows, double *dQ, double *lse, double *D)
{
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double *dp = (double *)malloc(sizeof(double) * (size_t)N);
        uint8_t *att = (uint8_t *)malloc((size_t)N);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t i = rows[r];
            const double L = row_scores(q, k, lts, lte, uts, ute, N, d, scale, i, s, att);
            double *dq = dQ + r * d;
            for (int c = 0; c < d; ++c)
                dq[c] = 0.0;
            lse[r] = L;
            D[r] = 0.0;
            if (L == -INFINITY)
                continue;
            double Di = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                if (!att[j])
                    continue;
                dp[j] = dot(dO + i * d, v + j * d, d);
                Di += exp(s[j] - L) * dp[j];
            }
            D[r] = Di;
            for (int64_t j = 0; j < N; ++j) {
                if (!att[j])
                    continue;
                const double ds = exp(s[j] - L) * (dp[j] - Di);
                for (int c = 0; c < d; ++c)
                    dq[c] += scale * ds * (double)k[j * d + c];
            }
        }
        free(s);
        free(dp);
        free(att);
    }
}

/* Column pass for the listed columns: dK_j and dV_j.  lse_full and D_full
 * are length-N arrays; only the entries of rows that attend a listed column
 * are read (they come from oracle_bwd_rows).  dK, dV are [ncols][d]. */
void oracle_bwd_cols(const float *q, const float *k, const float *v, const float *dO,
                     const int32_t *lts, const int32_t *lte, const int32_t *uts,
                     const int32_t *ute, int64_t N, int d, double scale, const double *lse_full,
                     const double *D_full, const int64_t *cols, int64_t ncols, double *dK,
                     double *dV)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < ncols; ++r) {
        const int64_t j = cols[r];
        double *dk = dK + r * d;
        double *dv = dV + r * d;
        for (int c = 0; c < d; ++c) {
            dk[c] = 0.0;
            dv[c] = 0.0;
        }
        for (int64_t i = 0; i < N; ++i) {
            if (masked_col_rule(lts, lte, uts, ute, i, j))
                continue;
            const double s = scale * dot(q + i * d, k + j * d, d);
            const double p = exp(s - lse_full[i]);
            const double dp = dot(dO + i * d, v + j * d, d);
            const double ds = p * (dp - D_full[i]);
            for (int c = 0; c < d; ++c) {
                dv[c] += p * (double)dO[i * d + c];
                dk[c] += scale * ds * (double)q[i * d + c];
            }
        }
    }
}

/* ---- tile labels --------------------------------------------------------- */

enum { LBL_SKIP = 0, LBL_FULL = 1, LBL_PARTIAL = 2 };

/* labels[qt*n_k + kt] for bq x bk tiles, tile ends clipped to N. */
void oracle_tile_labels(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                        const int32_t *ute, int64_t N, int bq, int bk, uint8_t *labels)
{
    const int64_t n_q = (N + bq - 1) / bq, n_k = (N + bk - 1) / bk;
#pragma omp parallel for schedule(static)
    for (int64_t kt = 0; kt < n_k; ++kt) {
        const int64_t kb = kt * bk, ke = (kb + bk < N) ? kb + bk : N;
        int64_t L0max = INT64_MIN, L0min = INT64_MAX, L1max = INT64_MIN, L1min = INT64_MAX;
        int64_t U0max = INT64_MIN, U0min = INT64_MAX, U1max = INT64_MIN, U1min = INT64_MAX;
        for (int64_t j = kb; j < ke; ++j) {
            int64_t l0 = lts[j], l1 = lte[j], u0 = uts[j], u1 = ute[j];
            if (l0 >= l1) { l0 = N; l1 = N; }
            if (u0 >= u1) { u0 = 0; u1 = 0; }
            if (l0 > L0max) L0max = l0;
            if (l0 < L0min) L0min = l0;
            if (l1 > L1max) L1max = l1;
            if (l1 < L1min) L1min = l1;
            if (u0 > U0max) U0max = u0;
            if (u0 < U0min) U0min = u0;
            if (u1 > U1max) U1max = u1;
            if (u1 < U1min) U1min = u1;
        }
        for (int64_t qt = 0; qt < n_q; ++qt) {
            const int64_t qb = qt * bq, qe = (qb + bq < N) ? qb + bq : N;
            const int skip = (L0max <= qb && L1min >= qe) || (U0max <= qb && U1min >= qe);
            const int full = !skip && (L0min >= qe || L1max <= qb) && (U0min >= qe || U1max <= qb);
            labels[qt * n_k + kt] = (uint8_t)(skip ? LBL_SKIP : (full ? LBL_FULL : LBL_PARTIAL));
        }
    }
}

/* Labels of the dense mask: SKIP if every element of the tile is masked, FULL
 * if none is, PARTIAL otherwise. */
void oracle_tile_labels_exact(const int32_t *lts, const int32_t *lte, const int32_t *uts,
                              const int32_t *ute, int64_t N, int bq, int bk, uint8_t *labels)
{
    const int64_t n_q = (N + bq - 1) / bq, n_k = (N + bk - 1) / bk;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t qt = 0; qt < n_q; ++qt)
        for (int64_t kt = 0; kt < n_k; ++kt) {
            const int64_t qb = qt * bq, qe = (qb + bq < N) ? qb + bq : N;
            const int64_t kb = kt * bk, ke = (kb + bk < N) ? kb + bk : N;
            int64_t nm = 0;
            for (int64_t i = qb; i < qe; ++i)
                for (int64_t j = kb; j < ke; ++j)
                    nm += masked_col_rule(lts, lte, uts, ute, i, j);
            const int64_t tot = (qe - qb) * (ke - kb);
            labels[qt * n_k + kt] =
                (uint8_t)(nm == tot ? LBL_SKIP : (nm == 0 ? LBL_FULL : LBL_PARTIAL));
        }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
