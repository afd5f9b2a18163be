/*
 * KDA oracle: plain fp64 token-by-token recurrence of Kimi Delta Attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle for the CUDA
 * library; it shares no code, header, table or helper with it.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may build,
 * load or call it.
 *
 * What it computes (nnterp "kimi_linear" page, the paragraph defining Kimi
 * Delta Attention; the Ascend model file, class KimiDeltaAttention, helpers
 * _l2_normalize and _torch_chunk_kda):
 *
 *   per (sequence, head), state S is K x V in fp64, starting from S0 (or 0);
 *   for every token t of the sequence, in order:
 *     qh = q_t / sqrt(sum_i q_t[i]^2 + 1e-6) * scale      (L2 norm, eps inside)
 *     kh = k_t / sqrt(sum_i k_t[i]^2 + 1e-6)
 *     S[i, :] *= exp(g_t[i])                 for every key channel i (decay first)
 *     u       = beta_t * (v_t - S^T kh)      (delta-rule residual, decayed state)
 *     S      += kh u^T
 *     o_t     = S^T qh                       (read-out from the updated state)
 *
 * Layouts (row-major, C order):
 *   q, k, g : [T_total, H, K]     v, o : [T_total, H, V]     beta : [T_total, H]
 *   cu_seqlens : [n_seqs + 1] int64, sequence n owns tokens [cu[n], cu[n+1])
 *   s0, s_final : [n_seqs, H, K, V]  (the mathematical K x V orientation)
 *
 * Sequences and heads are independent; OpenMP spreads (sequence, head) pairs
 * over host threads.  No blocking, fusion or reordering beyond the definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (sequence, head) pair run through the recurrence. */
static void kda_recurrence_one(const double *q, const double *k, const double *v,
                               const double *g, const double *beta,
                               int64_t t0, int64_t t1, int h, int H, int K, int V,
                               double scale, double *S, double *o,
                               double *qh, double *kh, double *u)
{
    for (int64_t t = t0; t < t1; ++t) {
        const double *qt = q + (t * H + h) * (int64_t)K;
        const double *kt = k + (t * H + h) * (int64_t)K;
        const double *gt = g + (t * H + h) * (int64_t)K;
        const double *vt = v + (t * H + h) * (int64_t)V;
        const double bt = beta[t * H + h];

        double sq = 0.0, sk = 0.0;
        for (int i = 0; i < K; ++i) {
            sq += qt[i] * qt[i];
            sk += kt[i] * kt[i];
        }
        const double rq = 1.0 / sqrt(sq + 1e-6);
        const double rk = 1.0 / sqrt(sk + 1e-6);
        for (int i = 0; i < K; ++i) {
            qh[i] = qt[i] * rq * scale;
            kh[i] = kt[i] * rk;
        }

        /* channel-wise decay of the state rows */
        for (int i = 0; i < K; ++i) {
            const double d = exp(gt[i]);
            double *row = S + (int64_t)i * V;
            for (int j = 0; j < V; ++j) row[j] *= d;
        }
        /* u = beta * (v - S^T kh) */
        for (int j = 0; j < V; ++j) u[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double *row = S + (int64_t)i * V;
            for (int j = 0; j < V; ++j) u[j] += row[j] * kh[i];
        }
        for (int j = 0; j < V; ++j) u[j] = bt * (vt[j] - u[j]);
        /* rank-one write */
        for (int i = 0; i < K; ++i) {
            double *row = S + (int64_t)i * V;
            for (int j = 0; j < V; ++j) row[j] += kh[i] * u[j];
        }
        /* read-out from the updated state */
        double *ot = o + (t * H + h) * (int64_t)V;
        for (int j = 0; j < V; ++j) ot[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double *row = S + (int64_t)i * V;
            for (int j = 0; j < V; ++j) ot[j] += row[j] * qh[i];
        }
    }
}

/*
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 * s0 may be NULL (zero initial state).  s_final may be NULL.
 * n_threads <= 0 leaves the OpenMP default.
 */
int kda_oracle_recurrence(const double *q, const double *k, const double *v,
                          const double *g, const double *beta,
                          const int64_t *cu_seqlens, int n_seqs, int H, int K, int V,
                          double scale, const double *s0, double *o, double *s_final,
                          int n_threads)
{
    if (!q || !k || !v || !g || !beta || !cu_seqlens || !o) return -1;
    if (n_seqs < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
    for (int n = 0; n < n_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;

    const int64_t pairs = (int64_t)n_seqs * H;
    const int64_t kv = (int64_t)K * V;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t p = 0; p < pairs; ++p) {
        const int n = (int)(p / H);
        const int h = (int)(p % H);
        double *S = (double *)malloc(sizeof(double) * (size_t)kv);
        double *work = (double *)malloc(sizeof(double) * (size_t)(2 * K + V));
        if (!S || !work) {
            free(S);
            free(work);
            failed |= 1;
            continue;
        }
        if (s0)
            memcpy(S, s0 + p * kv, sizeof(double) * (size_t)kv);
        else
            memset(S, 0, sizeof(double) * (size_t)kv);
        kda_recurrence_one(q, k, v, g, beta, cu_seqlens[n], cu_seqlens[n + 1], h, H, K, V,
                           scale, S, o, work, work + K, work + 2 * K);
        if (s_final) memcpy(s_final + p * kv, S, sizeof(double) * (size_t)kv);
        free(S);
        free(work);
    }
    return failed ? -1 : 0;
}

/* Number of threads an OpenMP parallel region would use (for reporting). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
