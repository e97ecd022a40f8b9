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

/* ------------------------------------------------------------ backward
 *
 * Reverse mode of the recurrence above: given dL/do_t for every token and
 * dL/dS_T (dhT, may be NULL), the gradients with respect to q, k, v,
 * log_alpha, eta and h0.  `given` selects the step rule: 0 = Kaczmarz
 * (beta_t = eta_t/(||k_t||^2+eps), so k_t also receives the gradient that
 * flows through its norm), 1 = the learned step of gated DeltaNet
 * (beta_t = eta_t).  Each token is differentiated by hand, in the order of
 * its forward formulas, from the state before it (S_{t-1}) and after it
 * (S_t):
 *
 *   o   = S_t^T q                    dS_t += q do^T,      dq = S_t do
 *   S_t = S~ + beta k e^T            dbeta = k^T dS_t e,  dk = beta dS_t e,
 *                                    de = beta dS_t^T k,  dS~ = dS_t
 *   e   = v - S~^T k                 dv = de,  dS~ -= k de^T,  dk -= S~ de
 *   beta = eta/(n+eps), n = ||k||^2  deta = dbeta/(n+eps),
 *                                    dk += 2 k (-dbeta beta/(n+eps))
 *   S~  = alpha S_{t-1}              dalpha = <dS~, S_{t-1}>,
 *                                    dlog_alpha = alpha dalpha,
 *                                    dS_{t-1} = alpha dS~
 *
 * (beta := 0 when n + eps == 0: then deta and the norm term are 0.)  The
 * states are recomputed forward from checkpoints kept every 64 tokens.
 */

/* Forward step on S in place (either rule), without the read-out. */
static void kla_token_rule(double* S, const double* k, const double* v,
                           double log_alpha, double eta, double eps,
                           int given, long dk, long dv, double* e)
{
    const double alpha = exp(log_alpha);
    double nrm = 0.0;
    for (long i = 0; i < dk; ++i) nrm += k[i] * k[i];
    const double denom = nrm + eps;
    const double beta = given ? eta : (denom == 0.0 ? 0.0 : eta / denom);
    for (long i = 0; i < dk * dv; ++i) S[i] *= alpha;
    for (long j = 0; j < dv; ++j) e[j] = v[j];
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) e[j] -= S[i * dv + j] * k[i];
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) S[i * dv + j] += beta * k[i] * e[j];
}

/* One token backward.  Sp = S_{t-1}, St = S_t; dS holds dL/dS_t on entry
 * (including this token's later uses) and dL/dS_{t-1} on return. */
static void kla_token_bwd(const double* Sp, const double* St,
                          const double* q, const double* k, const double* v,
                          double log_alpha, double eta, double eps, int given,
                          const double* dout, double* dS, double* dq,
                          double* dk_out, double* dv_out, double* dla,
                          double* deta, long dk, long dv, double* e,
                          double* de, double* tk)
{
    const double alpha = exp(log_alpha);
    double nrm = 0.0;
    for (long i = 0; i < dk; ++i) nrm += k[i] * k[i];
    const double denom = nrm + eps;
    const double beta = given ? eta : (denom == 0.0 ? 0.0 : eta / denom);

    /* e = v - S~^T k, S~ = alpha S_{t-1} */
    for (long j = 0; j < dv; ++j) e[j] = v[j];
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) e[j] -= alpha * Sp[i * dv + j] * k[i];

    /* read-out */
    for (long i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (long j = 0; j < dv; ++j) {
            dS[i * dv + j] += q[i] * dout[j];
            acc += St[i * dv + j] * dout[j];
        }
        dq[i] = acc;
    }

    /* write */
    double dbeta = 0.0;
    for (long i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (long j = 0; j < dv; ++j) acc += dS[i * dv + j] * e[j];
        tk[i] = acc;                       /* (dS_t e)_i */
        dbeta += k[i] * acc;
        dk_out[i] = beta * acc;
    }
    for (long j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (long i = 0; i < dk; ++i) acc += dS[i * dv + j] * k[i];
        de[j] = beta * acc;
        dv_out[j] = de[j];
    }

    /* residual: dS~ = dS_t - k de^T, dk -= S~ de */
    for (long i = 0; i < dk; ++i) {
        double acc = 0.0;
        for (long j = 0; j < dv; ++j) {
            dS[i * dv + j] -= k[i] * de[j];
            acc += Sp[i * dv + j] * de[j];
        }
        dk_out[i] -= alpha * acc;
    }

    /* step size */
    if (given) {
        *deta = dbeta;
    } else if (denom != 0.0) {
        *deta = dbeta / denom;
        const double dn = -dbeta * beta / denom;
        for (long i = 0; i < dk; ++i) dk_out[i] += 2.0 * dn * k[i];
    } else {
        *deta = 0.0;
    }

    /* decay */
    double dalpha = 0.0;
    for (long i = 0; i < dk * dv; ++i) dalpha += dS[i] * Sp[i];
    *dla = dalpha * alpha;
    for (long i = 0; i < dk * dv; ++i) dS[i] *= alpha;
}

/* Backward pass for every (b, h).  dout [B,T,H,dv]; dhT [B,H,dk,dv] or NULL;
 * outputs dq, dk [B,T,H,dk], dv [B,T,H,dv], dla, deta [B,T,H],
 * dh0 [B,H,dk,dv] (may be NULL).  Returns 0, -1 (bad argument) or -2 (no
 * scratch memory). */
int oracle_kla_bwd(const double* q, const double* k, const double* v,
                   const double* log_alpha, const double* eta, double eps,
                   int given, const double* h0, const double* dout,
                   const double* dhT, double* dq, double* dk_out,
                   double* dv_out, double* dla, double* deta, double* dh0,
                   long B, long T, long H, long dk, long dv, int n_threads)
{
    if (!q || !k || !v || !log_alpha || !eta || !dout || !dq || !dk_out ||
        !dv_out || !dla || !deta)
        return -1;
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    const long seg = 64;
    const long nseg = (T + seg - 1) / seg;
    const long sz = dk * dv;
    int failed = 0;
    const long pairs = B * H;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (long p = 0; p < pairs; ++p) {
        const long b = p / H, h = p % H;
        double* ck = (double*)malloc(sizeof(double) * (size_t)((nseg + 1) * sz));
        double* sb = (double*)malloc(sizeof(double) * (size_t)((seg + 1) * sz));
        double* dS = (double*)malloc(sizeof(double) * (size_t)sz);
        double* e = (double*)malloc(sizeof(double) * (size_t)dv);
        double* de = (double*)malloc(sizeof(double) * (size_t)dv);
        double* tk = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!ck || !sb || !dS || !e || !de || !tk) {
            free(ck); free(sb); free(dS); free(e); free(de); free(tk);
            failed |= 1;
            continue;
        }
        /* forward: checkpoints at t = 0, 64, 128, ... */
        double* S = sb;
        if (h0) memcpy(S, h0 + p * sz, sizeof(double) * (size_t)sz);
        else memset(S, 0, sizeof(double) * (size_t)sz);
        for (long t = 0; t < T; ++t) {
            if (t % seg == 0)
                memcpy(ck + (t / seg) * sz, S, sizeof(double) * (size_t)sz);
            const long row = (b * T + t) * H + h;
            kla_token_rule(S, k + row * dk, v + row * dv, log_alpha[row],
                           eta[row], eps, given, dk, dv, e);
        }
        /* backward, segment by segment */
        if (dhT) memcpy(dS, dhT + p * sz, sizeof(double) * (size_t)sz);
        else memset(dS, 0, sizeof(double) * (size_t)sz);
        for (long s = nseg - 1; s >= 0; --s) {
            const long t0 = s * seg;
            const long t1 = (t0 + seg < T) ? t0 + seg : T;
            memcpy(sb, ck + s * sz, sizeof(double) * (size_t)sz);
            for (long t = t0; t < t1; ++t) {
                const long row = (b * T + t) * H + h;
                memcpy(sb + (t - t0 + 1) * sz, sb + (t - t0) * sz,
                       sizeof(double) * (size_t)sz);
                kla_token_rule(sb + (t - t0 + 1) * sz, k + row * dk,
                               v + row * dv, log_alpha[row], eta[row], eps,
                               given, dk, dv, e);
            }
            for (long t = t1 - 1; t >= t0; --t) {
                const long row = (b * T + t) * H + h;
                kla_token_bwd(sb + (t - t0) * sz, sb + (t - t0 + 1) * sz,
                              q + row * dk, k + row * dk, v + row * dv,
                              log_alpha[row], eta[row], eps, given,
                              dout + row * dv, dS, dq + row * dk,
                              dk_out + row * dk, dv_out + row * dv,
                              dla + row, deta + row, dk, dv, e, de, tk);
            }
        }
        if (dh0) memcpy(dh0 + p * sz, dS, sizeof(double) * (size_t)sz);
        free(ck); free(sb); free(dS); free(e); free(de); free(tk);
    }
    (void)n_threads;
    return failed ? -2 : 0;
}

/* ------------------------------------------------------------ preconditioned
 *
 * The diagonal-preconditioned delta rule of the adjacent page (gist.science
 * "preconditioned DeltaNet", section "Aproximacion Diagonal"): the running
 * second moments of the keys, A_t = A_{t-1} + k_t (.) k_t (per key
 * dimension), give the preconditioner P_t ~ Diag(A_t)^{-1}, squashed in log
 * space into [1/x, x] (x ~ 1.5), and applied to the write key (ATK):
 *
 *   z_i     = mean_j log(A_t,j + delta) - log(A_t,i + delta)
 *   P_t,i   = exp(log(x) tanh(z_i / log(x)))     (slope 1 at z = 0)
 *   kw_t    = P_t (.) k_t                         write key
 *   e_t     = v_t - S~^T k_t                      residual, read key k_t
 *   S_t     = S~ + beta_t kw_t e_t^T,   o_t = S_t^T q_t
 *   beta_t  = eta_t (given) or eta_t / (k_t . kw_t + eps) (Kaczmarz: at
 *             eta = 1, eps = 0 the write makes S_t^T k_t = v_t exactly)
 *
 * The page names a squash "in log space" onto [1/x, x] without the function
 * or a reference level; tanh with unit slope, centred on the mean log second
 * moment over the key dimensions, and the floor delta inside the log are
 * this library's reading.  A [B, H, dk] carries A_t (in/out, may be NULL on
 * input: zero).  Returns 0, -1 or -2 as the functions above.
 */
static void precond_key(double* A, const double* k, double* kw, long dk,
                        double x, double delta)
{
    double mean = 0.0;
    for (long i = 0; i < dk; ++i) {
        A[i] += k[i] * k[i];
        mean += log(A[i] + delta);
    }
    mean /= (double)dk;
    const double lx = log(x);
    for (long i = 0; i < dk; ++i) {
        const double z = mean - log(A[i] + delta);
        kw[i] = exp(lx * tanh(z / lx)) * k[i];
    }
}

static void pkla_token(double* S, const double* q, const double* k,
                       const double* kw, const double* v, double log_alpha,
                       double eta, double eps, int given, double* o, long dk,
                       long dv, double* e)
{
    const double alpha = exp(log_alpha);
    double kkw = 0.0;
    for (long i = 0; i < dk; ++i) kkw += k[i] * kw[i];
    const double denom = kkw + eps;
    const double beta = given ? eta : (denom == 0.0 ? 0.0 : eta / denom);
    for (long i = 0; i < dk * dv; ++i) S[i] *= alpha;
    for (long j = 0; j < dv; ++j) e[j] = v[j];
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) e[j] -= S[i * dv + j] * k[i];
    for (long i = 0; i < dk; ++i)
        for (long j = 0; j < dv; ++j) S[i * dv + j] += beta * kw[i] * e[j];
    if (o) {
        for (long j = 0; j < dv; ++j) o[j] = 0.0;
        for (long i = 0; i < dk; ++i)
            for (long j = 0; j < dv; ++j) o[j] += S[i * dv + j] * q[i];
    }
}

/* Forward pass over T tokens.  kw_out [B,T,H,dk] (may be NULL) receives the
 * write keys; A [B,H,dk] (may be NULL) holds A_0 on entry (NULL: zero) and
 * A_T on return. */
int oracle_pkla_fwd(const double* q, const double* k, const double* v,
                    const double* log_alpha, const double* eta, double eps,
                    int given, double x, double delta, const double* h0,
                    double* A, double* o, double* hT, double* kw_out,
                    long B, long T, long H, long dk, long dv, int n_threads)
{
    if (!q || !k || !v || !log_alpha || !eta || !o) return -1;
    if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0 || !(x > 1.0))
        return -1;
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
        double* Ad = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kw = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!S || !e || !Ad || !kw) {
            free(S); free(e); free(Ad); free(kw);
            failed |= 1;
            continue;
        }
        if (h0) memcpy(S, h0 + p * dk * dv, sizeof(double) * (size_t)(dk * dv));
        else memset(S, 0, sizeof(double) * (size_t)(dk * dv));
        if (A) memcpy(Ad, A + p * dk, sizeof(double) * (size_t)dk);
        else memset(Ad, 0, sizeof(double) * (size_t)dk);
        for (long t = 0; t < T; ++t) {
            const long row = (b * T + t) * H + h;
            precond_key(Ad, k + row * dk, kw, dk, x, delta);
            if (kw_out) memcpy(kw_out + row * dk, kw, sizeof(double) * (size_t)dk);
            pkla_token(S, q + row * dk, k + row * dk, kw, v + row * dv,
                       log_alpha[row], eta[row], eps, given, o + row * dv,
                       dk, dv, e);
        }
        if (hT) memcpy(hT + p * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
        if (A) memcpy(A + p * dk, Ad, sizeof(double) * (size_t)dk);
        free(S); free(e); free(Ad); free(kw);
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
