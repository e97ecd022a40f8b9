/*
 * Kaczmarz Linear Attention (KLA) -- sequential fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against; no product code links, loads or calls it.  It shares no
 * code, header or constant with the CUDA library.
 *
 * What it computes (one (batch, head) pair at a time, state S in R^{dk x dv},
 * row index = key dimension):
 *
 *   alpha_t = exp(log_alpha_t)                       decayed previous state
 *   S~      = alpha_t * S_{t-1}                      (scalar gate per token/head)
 *   beta_t  = eta_t / (||k_t||_2^2 + eps)            Kaczmarz step
 *   e_t     = v_t - S~^T k_t                         residual
 *   S_t     = S~ + beta_t * k_t e_t^T                delta-rule write
 *   o_t     = S_t^T q_t                              read-out after the write
 *
 * Sources (gist.science/es/paper/2605.08587, "Atencion Lineal Kaczmarz"):
 *   - the write as a constrained problem and its projection solution,
 *     section "Derivacion Teorica";
 *   - the relaxed step beta_t = eta_t/(||k_t||^2+eps), the update
 *     S_t = S~_{t-1} + beta_t k_t e_t^T and the residual e_t, section
 *     "La Regla de Actualizacion KLA" (same formulas on the German and French
 *     pages, sections "Die KLA-Aktualisierungsregel" / "La regle de mise a
 *     jour KLA").
 * The pages call S~ "the decayed previous state" without giving the decay; the
 * scalar form S~ = alpha_t S_{t-1} and the read-out o_t = S_t^T q_t are the
 * readings adopted for this library (the GDN-style scalar gate, applied before
 * the residual is formed).
 *
 * Degenerate step: when ||k_t||^2 + eps == 0 (zero key, eps = 0) the write
 * beta_t k_t e_t^T is the zero matrix in the limit, so beta_t is taken as 0.
 *
 * Layouts (all contiguous, row-major, fp64):
 *   q, k       [B, T, H, dk]
 *   v, o       [B, T, H, dv]
 *   log_alpha  [B, T, H]
 *   eta        [B, T, H]
 *   h0, hT     [B, H, dk, dv]   (h0 may be NULL: zero initial state;
 *                                 hT may be NULL: not written)
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* One token of the recurrence on one state.  S is dk x dv, updated in place;
 * o (dv) receives S_t^T q.  scratch holds dv doubles. */
static void kla_token(double* S, const double* q, const double* k,
                      const double* v, double log_alpha, double eta,
                      double eps, double* o, long dk, long dv,
                      double* e)
{
    const double alpha = exp(log_alpha);
    double nrm = 0.0;
    for (long i = 0; i < dk; ++i) nrm += k[i] * k[i];
    const double denom = nrm + eps;
    const double beta = (denom == 0.0) ? 0.0 : eta / denom;

    /* S~ = alpha S */
    for (long i = 0; i < dk * dv; ++i) S[i] *= alpha;

    /* e = v - S~^T k */
    for (long j = 0; j < dv; ++j) e[j] = v[j];
    for (long i = 0; i < dk; ++i) {
        const double ki = k[i];
        const double* row = S + i * dv;
        for (long j = 0; j < dv; ++j) e[j] -= row[j] * ki;
    }

    /* S = S~ + beta k e^T */
    for (long i = 0; i < dk; ++i) {
        const double bk = beta * k[i];
        double* row = S + i * dv;
        for (long j = 0; j < dv; ++j) row[j] += bk * e[j];
    }

    /* o = S^T q */
    if (o) {
        for (long j = 0; j < dv; ++j) o[j] = 0.0;
        for (long i = 0; i < dk; ++i) {
            const double qi = q[i];
            const double* row = S + i * dv;
            for (long j = 0; j < dv; ++j) o[j] += row[j] * qi;
        }
    }
}

/* Full forward pass over T tokens for every (b, h).  Returns 0 on success,
 * -1 on a bad argument, -2 if scratch memory could not be obtained. */
int oracle_kla_fwd(const double* q, const double* k, const double* v,
                   const double* log_alpha, const double* eta, double eps,
                   const double* h0, double* o, double* hT,
                   long B, long T, long H, long dk, long dv, int n_threads)
{
    if (!q || !k || !v || !log_alpha || !eta || !o) return -1;
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    int failed = 0;
    const long pairs = B * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (long p = 0; p < pairs; ++p) {
        const long b = p / H, h = p % H;
        double* S = (double*)malloc(sizeof(double) * (size_t)(dk * dv));
        double* e = (double*)malloc(sizeof(double) * (size_t)dv);
        if (!S || !e) { free(S); free(e); failed |= 1; continue; }
        if (h0) memcpy(S, h0 + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        for (long t = 0; t < T; ++t) {
            const long row = (b * T + t) * H + h;   /* index into [B,T,H] */
            kla_token(S, q + row * dk, k + row * dk, v + row * dv,
                      log_alpha[row], eta[row], eps, o + row * dv, dk, dv, e);
        }
        if (hT) memcpy(hT + p * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
        free(S);
        free(e);
    }
    (void)n_threads;
    return failed ? -2 : 0;
}

/* One decode step for N sequences x H heads: S [N,H,dk,dv] is updated in
 * place; q,k [N,H,dk]; v,o [N,H,dv]; log_alpha, eta [N,H]. */
int oracle_kla_decode_step(const double* q, const double* k, const double* v,
                           const double* log_alpha, const double* eta,
                           double eps, double* S, double* o,
                           long N, long H, long dk, long dv, int n_threads)
{
    if (!q || !k || !v || !log_alpha || !eta || !S || !o) return -1;
    if (N < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    int failed = 0;
    const long heads = N * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(static) reduction(| : failed)
#endif
    for (long p = 0; p < heads; ++p) {
        double* e = (double*)malloc(sizeof(double) * (size_t)dv);
        if (!e) { failed |= 1; continue; }
        kla_token(S + p * dk * dv, q + p * dk, k + p * dk, v + p * dv,
                  log_alpha[p], eta[p], eps, o + p * dv, dk, dv, e);
        free(e);
    }
    (void)n_threads;
    return failed ? -2 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
