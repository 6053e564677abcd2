/* TEST INFRASTRUCTURE ONLY.  A plain, slow fp64 CPU oracle for the
 * multi-head attention forward pass (and, at the end of the file, its
 * gradients).  Only the tests, the smoke check and
 * the CPU-baseline leg of the benchmark load this file; the library's
 * product path never does, and the two share no code.
 *
 * What it computes is the definition of attention, written out directly:
 *
 *   "Simple FlashAttention" (Triton-learning blog, Puzzle 9, problem
 *   statement): z_i = sum_j softmax(q_i k_1, ..., q_i k_T)_j v_j.
 *   Numerically safe softmax subtracts the row maximum first (same blog,
 *   Puzzle 8 problem statement).  FlashAttention-2 (ML-Triton paper,
 *   section 2.5, Algorithm 1) reaches exactly this result tile by tile.
 *
 * Readings of points the pages leave open (all fixed by the library's
 * interface, not by the pages):
 *   - scores are scaled: s_ij = scale * <q_i, k_j>, scale used as passed;
 *   - causal means square, top-left aligned: row i sees keys 0..i;
 *   - LSE_i = m_i + ln(l_i) in natural log on the scaled scores;
 *   - a row with an empty key set (never produced by a square mask) gets
 *     O = 0 and LSE = -inf.
 *
 * Inputs are bfloat16 bit patterns; each is widened exactly to double.
 * All arithmetic is fp64: the dot product in index order, then the row
 * maximum m, l = sum exp(s - m), P = exp(s - m) / l, O = sum_j P_j v_j.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* One query row of one head over the keys 0..nk-1 (its key set J_i).
 * q_row: [d] bf16 bits; k_bh, v_bh: [Nk, d] bf16 bits.  s: scratch of at
 * least nk doubles.  o_row: d doubles out.  p_row: optional Nk doubles out
 * (the softmax probabilities; zero for keys outside J_i). */
static void attention_row_keys(const uint16_t *q_row, const uint16_t *k_bh, const uint16_t *v_bh,
                               int64_t Nk, int64_t d, double scale, int64_t nk,
                               double *s, double *o_row, double *lse, double *p_row) {
    const int64_t N = Nk;
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    if (p_row)
        for (int64_t j = 0; j < N; ++j) p_row[j] = 0.0;
    if (nk <= 0) {
        *lse = -INFINITY;
        return;
    }
    /* scores s_ij = scale * sum_c q_ic k_jc */
    for (int64_t j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += bf16_to_f64(q_row[c]) * bf16_to_f64(k_bh[j * d + c]);
        s[j] = scale * acc;
    }
    /* row maximum and the sum of shifted exponentials */
    double m = s[0];
    for (int64_t j = 1; j < nk; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j) l += exp(s[j] - m);
    /* O_i = sum_j P_ij v_j with P_ij = exp(s_ij - m_i) / l_i */
    for (int64_t j = 0; j < nk; ++j) {
        double p = exp(s[j] - m) / l;
        if (p_row) p_row[j] = p;
        for (int64_t c = 0; c < d; ++c) o_row[c] += p * bf16_to_f64(v_bh[j * d + c]);
    }
    *lse = m + log(l);
}

/* Square case: query i of N sees keys {0..N-1}, or {0..i} under the causal
 * mask (top-left aligned). */
static void attention_row(const uint16_t *q_bh, const uint16_t *k_bh, const uint16_t *v_bh,
                          int64_t N, int64_t d, double scale, int causal, int64_t i,
                          double *s, double *o_row, double *lse, double *p_row) {
    int64_t nk = causal ? i + 1 : N;
    if (nk > N) nk = N;
    attention_row_keys(q_bh + i * d, k_bh, v_bh, N, d, scale, nk, s, o_row, lse, p_row);
}

/* Rows rows[0..nrows-1] of one head.  o_out: [nrows, d]; lse_out: [nrows].
 * nthreads <= 0 uses the OpenMP default.  Returns 0, or -1 on bad input. */
int oracle_attention_rows(const uint16_t *q_bh, const uint16_t *k_bh, const uint16_t *v_bh,
                          int64_t N, int64_t d, float scale, int causal,
                          const int64_t *rows, int64_t nrows,
                          double *o_out, double *lse_out, int nthreads) {
    if (N < 0 || d <= 0 || nrows < 0) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    int bad = 0;
#pragma omp parallel num_threads(nthreads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
        /* every thread reaches the work-sharing loop (a thread without its
         * buffer takes no rows; the call then fails as a whole) */
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r)
            if (s)
                attention_row(q_bh, k_bh, v_bh, N, d, (double)scale, causal, rows[r], s,
                              o_out + r * d, lse_out + r, NULL);
        free(s);
    }
    return bad ? -1 : 0;
}

/* Every row of every head: q, k, v are [BH, N, d]; o_out [BH, N, d];
 * lse_out [BH, N]. */
int oracle_attention_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         int64_t BH, int64_t N, int64_t d, float scale, int causal,
                         double *o_out, double *lse_out, int nthreads) {
    if (BH < 0 || N < 0 || d <= 0) return -1;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    if (!rows) return -1;
    for (int64_t i = 0; i < N; ++i) rows[i] = i;
    int rc = 0;
    for (int64_t bh = 0; bh < BH && rc == 0; ++bh) {
        const int64_t off = bh * N * d;
        rc = oracle_attention_rows(q + off, k + off, v + off, N, d, scale, causal, rows, N,
                                   o_out + off, lse_out + bh * N, nthreads);
    }
    free(rows);
    return rc;
}

/* The probability matrix P [N, N] of one head (zeros outside each row's
 * key set) together with LSE [N]; for checks of the softmax itself. */
int oracle_attention_probs(const uint16_t *q_bh, const uint16_t *k_bh, const uint16_t *v_bh,
                           int64_t N, int64_t d, float scale, int causal,
                           double *p_out, double *o_out, double *lse_out) {
    if (N < 0 || d <= 0) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!s) return -1;
    for (int64_t i = 0; i < N; ++i)
        attention_row(q_bh, k_bh, v_bh, N, d, (double)scale, causal, i, s, o_out + i * d,
                      lse_out + i, p_out + i * N);
    free(s);
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Nq queries against Nk keys of one head (q_bh [Nq, d], k_bh / v_bh
 * [Nk, d]).  Under the causal mask the queries are the last Nq positions of
 * the sequence (bottom-right aligned): query i sees keys 0 .. Nk-Nq+i, and
 * none when that bound is negative.  With Nq == Nk this is the square case. */
int oracle_attention_kv(const uint16_t *q_bh, const uint16_t *k_bh, const uint16_t *v_bh,
                        int64_t Nq, int64_t Nk, int64_t d, float scale, int causal,
                        double *o_out, double *lse_out, int nthreads) {
    if (Nq < 0 || Nk < 0 || d <= 0) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    int bad = 0;
#pragma omp parallel num_threads(nthreads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < Nq; ++i) {
            if (!s) continue;
            int64_t nk = causal ? Nk - Nq + i + 1 : Nk;
            if (nk < 0) nk = 0;
            if (nk > Nk) nk = Nk;
            attention_row_keys(q_bh + i * d, k_bh, v_bh, Nk, d, (double)scale, nk, s,
                               o_out + i * d, lse_out + i, NULL);
        }
        free(s);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ backward
 * Gradients of the loss L = sum_{i,c} dO_ic * O_ic with respect to q, k and
 * v, where O is the attention output defined above (same scale, same key
 * sets).  The pages give no attention backward; this is the derivative of
 * the forward definition written out (chain rule through the softmax):
 *
 *   P_ij  = softmax_j(s_i)          s_ij = scale <q_i, k_j>,  j in J_i
 *   D_i   = sum_c dO_ic O_ic
 *   dP_ij = sum_c dO_ic v_jc
 *   dS_ij = P_ij (dP_ij - D_i)      (softmax Jacobian applied to dP_i)
 *   dV_j  = sum_i P_ij dO_i
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j  = scale sum_i dS_ij q_i
 *
 * All in fp64 from the exact bf16 inputs; O and P are recomputed exactly
 * here (not taken from any kernel).  Query rows are split among threads;
 * each thread accumulates its own dK / dV and the partials are summed.
 * q, k, v, dout: [N, d] bf16 bits of one head; dq, dk, dv: [N, d] doubles. */
static int attention_bwd_head(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const uint16_t *dout, int64_t N, int64_t d, double scale,
                              int causal, double *dq, double *dk, double *dv, int nthreads) {
    for (int64_t x = 0; x < N * d; ++x) dq[x] = dk[x] = dv[x] = 0.0;
    if (N == 0) return 0;
    int bad = 0;
#pragma omp parallel num_threads(nthreads)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        double *dk_t = (double *)calloc((size_t)(N * d), sizeof(double));
        double *dv_t = (double *)calloc((size_t)(N * d), sizeof(double));
        const int mine = s && p && o && dk_t && dv_t;
        if (!mine) {
#pragma omp atomic write
            bad = 1;
        }
        /* every thread reaches the work-sharing loop; one without buffers
         * takes no rows (the call then fails as a whole) */
#pragma omp for schedule(dynamic, 8)
        for (int64_t i = 0; i < N; ++i) {
            if (!mine) continue;
            const uint16_t *q_row = q + i * d;
            const uint16_t *do_row = dout + i * d;
            double lse;
            int64_t nk = causal ? i + 1 : N;
            attention_row_keys(q_row, k, v, N, d, scale, nk, s, o, &lse, p);
            double D = 0.0;
            for (int64_t c = 0; c < d; ++c) D += bf16_to_f64(do_row[c]) * o[c];
            for (int64_t j = 0; j < nk; ++j) {
                double dp = 0.0;
                for (int64_t c = 0; c < d; ++c)
                    dp += bf16_to_f64(do_row[c]) * bf16_to_f64(v[j * d + c]);
                const double ds = p[j] * (dp - D);
                for (int64_t c = 0; c < d; ++c) {
                    dq[i * d + c] += scale * ds * bf16_to_f64(k[j * d + c]);
                    dk_t[j * d + c] += scale * ds * bf16_to_f64(q_row[c]);
                    dv_t[j * d + c] += p[j] * bf16_to_f64(do_row[c]);
                }
            }
        }
        if (mine) {
#pragma omp critical
            {
                for (int64_t x = 0; x < N * d; ++x) {
                    dk[x] += dk_t[x];
                    dv[x] += dv_t[x];
                }
            }
        }
        free(s);
        free(p);
        free(o);
        free(dk_t);
        free(dv_t);
    }
    return bad ? -1 : 0;
}

/* Every head: q, k, v, dout [BH, N, d]; dq, dk, dv [BH, N, d] doubles. */
int oracle_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint16_t *dout, int64_t BH, int64_t N, int64_t d, float scale,
                         int causal, double *dq, double *dk, double *dv, int nthreads) {
    if (BH < 0 || N < 0 || d <= 0) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
    nthreads = 1;
#endif
    for (int64_t bh = 0; bh < BH; ++bh) {
        const int64_t off = bh * N * d;
        if (attention_bwd_head(q + off, k + off, v + off, dout + off, N, d, (double)scale, causal,
                               dq + off, dk + off, dv + off, nthreads) != 0)
            return -1;
    }
    return 0;
}
