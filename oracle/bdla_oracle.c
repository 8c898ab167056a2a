/*
 * Oracle for bounded-decay gated linear attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU statement of what the hot path computes.  Only the
 * test suite, the package smoke check and the benchmark's CPU-baseline leg
 * may load this library; the CUDA library shares no code with it.
 *
 * Source of the method (web pages, cited by title and section):
 *  [P1] "Engineering Long-Context Training for Trillion-Parameter MoE Models:
 *       Three Key Breakthroughs", sec. 3.1 (chunked linear attention with a
 *       per-position cumulative decay) and sec. 3.2 (log-decay g = g_min *
 *       sigmoid(x), g_min = -5, replacing g = -softplus(x)).
 *  [P2] "Scaling Trillion-Parameter MoE and Long-Context LLMs", sec. II,
 *       first bullet (same substitution, bound -5, 16-token tiles).
 *  [P3] "Engineering Stability in Ultra-Long Context and Trillion-Parameter
 *       Sparse Models", sec. 2.1-2.2 (chunked computation, bounded decay).
 *
 * The pages fix the decay parameterisation but print no formula for the
 * attention itself.  This file takes the plainest reading that the pages
 * support: gated linear attention with one scalar decay per (token, head),
 *     lambda_t = log g_t = b * sigmoid(a_t)          (bounded, b < 0)
 *     lambda_t = -softplus(a_t)                      (unbounded ablation)
 *     S_t = exp(lambda_t) * S_{t-1} + k_t v_t^T,     S_0 = h0
 *     o_t = S_t^T q_t,                                hT = S_L
 * evaluated token by token (no chunking: the chunked algorithm on the pages
 * is an evaluation order of this recurrence, exact up to rounding).
 * The backward pass is reverse-mode differentiation of the same loop.
 *
 * Pins (tests): brute-force O(T^2) sum, b -> 0 limit (plain causal linear
 * attention), constant-decay closed form, T = 1 by hand, central finite
 * differences for every gradient, varlen == concatenation, linearity.
 *
 * The gated delta rule with the same bounded decay (fwd_delta / bwd_delta,
 * below) is the "Delta Net-style" structure the first page names beside
 * linear attention ([P1] sec. 3.1; the substitution applies to it unchanged).
 *
 * Layouts (row-major, feature innermost):
 *   q, k  [Ttot][H][dk]     v, o, dO  [Ttot][H][dv]     a, da  [Ttot][H]
 *   h0, hT, dh0, dhT  [N][H][dk][dv]    cu  [N+1] document offsets
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Log-decay [P1 sec. 3.2]: bounded b*sigmoid(a) (mode 0) or -softplus(a). */
static double log_decay(double a, double b, int mode)
{
    if (mode == 0)
        return b / (1.0 + exp(-a));
    /* softplus(a) = log(1 + e^a), written stably as max(a,0) + log1p(e^-|a|) */
    return -(fmax(a, 0.0) + log1p(exp(-fabs(a))));
}

/* d lambda / d a for the two parameterisations. */
static double log_decay_deriv(double a, double b, int mode)
{
    double s = 1.0 / (1.0 + exp(-a));
    if (mode == 0)
        return b * s * (1.0 - s);
    return -s;
}

int oracle_log_decay(int64_t n, const double *a, double b, int mode, double *lam)
{
    for (int64_t i = 0; i < n; ++i)
        lam[i] = log_decay(a[i], b, mode);
    return 0;
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Forward recurrence for N documents x H heads.  h0 may be NULL (zero
 * initial state), hT may be NULL.  Returns the number of threads used.
 */
int oracle_fwd(int N, const int64_t *cu, int H, int dk, int dv,
               const double *q, const double *k, const double *v,
               const double *a, double b, int mode, const double *h0,
               double *o, double *hT, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double g = exp(log_decay(a[t * H + h], b, mode));
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                double *ot = o + ((size_t)t * H + h) * dv;
                /* S_t = g_t S_{t-1} + k_t v_t^T */
                for (int i = 0; i < dk; ++i) {
                    double *Si = S + (size_t)i * dv;
                    const double ki = kt[i];
                    for (int j = 0; j < dv; ++j)
                        Si[j] = g * Si[j] + ki * vt[j];
                }
                /* o_t = S_t^T q_t */
                for (int j = 0; j < dv; ++j)
                    ot[j] = 0.0;
                for (int i = 0; i < dk; ++i) {
                    const double *Si = S + (size_t)i * dv;
                    const double qi = qt[i];
                    for (int j = 0; j < dv; ++j)
                        ot[j] += qi * Si[j];
                }
            }
            if (hT)
                memcpy(hT + (size_t)u * ssz, S, ssz * sizeof(double));
        }
        free(S);
    }
    return used;
}

/*
 * Reverse mode of oracle_fwd.  With D the adjoint of S_t:
 *   D += q_t dO_t^T;  dq_t = S_t dO_t;  dk_t = D v_t;  dv_t = D^T k_t;
 *   dlambda_t = g_t <D, S_{t-1}>_F;  D <- g_t D;     dh0 = D at the end.
 * S_{t-1} is recomputed from fp64 checkpoints taken every `window` tokens
 * (never by dividing by g_t).  dhT, h0 and dh0 may be NULL.
 */
int oracle_bwd(int N, const int64_t *cu, int H, int dk, int dv,
               const double *q, const double *k, const double *v,
               const double *a, double b, int mode, const double *h0,
               const double *dO, const double *dhT,
               double *dq, double *dkk, double *dvv, double *da,
               double *dh0, int window, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;
    if (window <= 0)
        window = 1024;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
        double *D = (double *)malloc(ssz * sizeof(double));
        /* states S_{t-1} for every t of one window */
        double *win = (double *)malloc((size_t)window * ssz * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            const int64_t t0 = cu[n], L = cu[n + 1] - cu[n];
            const int64_t nwin = (L + window - 1) / window;
            double *ck = (double *)malloc((size_t)(nwin > 0 ? nwin : 1) * ssz * sizeof(double));

            /* forward sweep: checkpoint S before each window */
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = 0; t < L; ++t) {
                if (t % window == 0)
                    memcpy(ck + (size_t)(t / window) * ssz, S, ssz * sizeof(double));
                const int64_t tt = t0 + t;
                const double g = exp(log_decay(a[tt * H + h], b, mode));
                const double *kt = k + ((size_t)tt * H + h) * dk;
                const double *vt = v + ((size_t)tt * H + h) * dv;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + kt[i] * vt[j];
            }

            if (dhT)
                memcpy(D, dhT + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(D, 0, ssz * sizeof(double));

            for (int64_t w = nwin - 1; w >= 0; --w) {
                const int64_t ws = w * window;
                const int64_t we = (ws + window < L) ? ws + window : L;
                /* recompute S_{t-1} for t in [ws, we) from the checkpoint */
                memcpy(S, ck + (size_t)w * ssz, ssz * sizeof(double));
                for (int64_t t = ws; t < we; ++t) {
                    memcpy(win + (size_t)(t - ws) * ssz, S, ssz * sizeof(double));
                    const int64_t tt = t0 + t;
                    const double g = exp(log_decay(a[tt * H + h], b, mode));
                    const double *kt = k + ((size_t)tt * H + h) * dk;
                    const double *vt = v + ((size_t)tt * H + h) * dv;
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + kt[i] * vt[j];
                }
                for (int64_t t = we - 1; t >= ws; --t) {
                    const int64_t tt = t0 + t;
                    const double at = a[tt * H + h];
                    const double g = exp(log_decay(at, b, mode));
                    const double *qt = q + ((size_t)tt * H + h) * dk;
                    const double *kt = k + ((size_t)tt * H + h) * dk;
                    const double *vt = v + ((size_t)tt * H + h) * dv;
                    const double *gt = dO + ((size_t)tt * H + h) * dv;
                    double *dqt = dq + ((size_t)tt * H + h) * dk;
                    double *dkt = dkk + ((size_t)tt * H + h) * dk;
                    double *dvt = dvv + ((size_t)tt * H + h) * dv;
                    const double *Sp = win + (size_t)(t - ws) * ssz; /* S_{t-1} */
                    /* D += q_t dO_t^T  (adjoint of S_t) */
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            D[(size_t)i * dv + j] += qt[i] * gt[j];
                    /* dq_t = S_t dO_t with S_t = g S_{t-1} + k v^T */
                    for (int i = 0; i < dk; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; ++j)
                            acc += (g * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];
                        dqt[i] = acc;
                    }
                    /* dk_t = D v_t */
                    for (int i = 0; i < dk; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; ++j)
                            acc += D[(size_t)i * dv + j] * vt[j];
                        dkt[i] = acc;
                    }
                    /* dv_t = D^T k_t */
                    for (int j = 0; j < dv; ++j)
                        dvt[j] = 0.0;
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            dvt[j] += D[(size_t)i * dv + j] * kt[i];
                    /* dlambda_t = g_t <D, S_{t-1}> ;  da_t = dlambda_t * dlambda/da */
                    double dot = 0.0;
                    for (size_t e = 0; e < ssz; ++e)
                        dot += D[e] * Sp[e];
                    da[tt * H + h] = g * dot * log_decay_deriv(at, b, mode);
                    /* adjoint of S_{t-1} */
                    for (size_t e = 0; e < ssz; ++e)
                        D[e] *= g;
                }
            }
            if (dh0)
                memcpy(dh0 + (size_t)u * ssz, D, ssz * sizeof(double));
            free(ck);
        }
        free(win);
        free(D);
        free(S);
    }
    return used;
}

/*
 * Per-channel (vector) decay, the variant the first page's "per-position
 * cumulative decay" ([P1] sec. 3.1) also admits: one log-decay per (token,
 * head, key channel) with the same two parameterisations ([P1] sec. 3.2),
 *     lambda_t[i] = b * sigmoid(a_t[i])   or   -softplus(a_t[i]),
 *     S_t = diag(exp(lambda_t)) S_{t-1} + k_t v_t^T,   S_0 = h0,
 *     o_t = S_t^T q_t,                                 hT = S_L,
 * i.e. row i of the dk x dv state decays by its own factor.  Layouts as
 * above except a, da: [Ttot][H][dk].
 */
int oracle_fwd_vec(int N, const int64_t *cu, int H, int dk, int dv,
                   const double *q, const double *k, const double *v,
                   const double *a, double b, int mode, const double *h0,
                   double *o, double *hT, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double *at = a + ((size_t)t * H + h) * dk;
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                double *ot = o + ((size_t)t * H + h) * dv;
                /* S_t = diag(g_t) S_{t-1} + k_t v_t^T: row i decays by g_t[i] */
                for (int i = 0; i < dk; ++i) {
                    const double gi = exp(log_decay(at[i], b, mode));
                    double *Si = S + (size_t)i * dv;
                    const double ki = kt[i];
                    for (int j = 0; j < dv; ++j)
                        Si[j] = gi * Si[j] + ki * vt[j];
                }
                /* o_t = S_t^T q_t */
                for (int j = 0; j < dv; ++j)
                    ot[j] = 0.0;
                for (int i = 0; i < dk; ++i) {
                    const double *Si = S + (size_t)i * dv;
                    const double qi = qt[i];
                    for (int j = 0; j < dv; ++j)
                        ot[j] += qi * Si[j];
                }
            }
            if (hT)
                memcpy(hT + (size_t)u * ssz, S, ssz * sizeof(double));
        }
        free(S);
    }
    return used;
}

/*
 * Reverse mode of oracle_fwd_vec.  With D the adjoint of S_t:
 *   D += q_t dO_t^T;  dq_t = S_t dO_t;  dk_t = D v_t;  dv_t = D^T k_t;
 *   dlambda_t[i] = g_t[i] sum_j D[i][j] S_{t-1}[i][j];  D <- diag(g_t) D;
 *   dh0 = D at the end.  S_{t-1} comes from fp64 checkpoints every `window`
 * tokens, recomputed forward inside each window.
 */
int oracle_bwd_vec(int N, const int64_t *cu, int H, int dk, int dv,
                   const double *q, const double *k, const double *v,
                   const double *a, double b, int mode, const double *h0,
                   const double *dO, const double *dhT,
                   double *dq, double *dkk, double *dvv, double *da,
                   double *dh0, int window, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;
    if (window <= 0)
        window = 1024;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
        double *D = (double *)malloc(ssz * sizeof(double));
        double *g = (double *)malloc((size_t)dk * sizeof(double));
        double *win = (double *)malloc((size_t)window * ssz * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            const int64_t t0 = cu[n], L = cu[n + 1] - cu[n];
            const int64_t nwin = (L + window - 1) / window;
            double *ck = (double *)malloc((size_t)(nwin > 0 ? nwin : 1) * ssz * sizeof(double));

            /* forward sweep: checkpoint S before each window */
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = 0; t < L; ++t) {
                if (t % window == 0)
                    memcpy(ck + (size_t)(t / window) * ssz, S, ssz * sizeof(double));
                const int64_t tt = t0 + t;
                const double *at = a + ((size_t)tt * H + h) * dk;
                const double *kt = k + ((size_t)tt * H + h) * dk;
                const double *vt = v + ((size_t)tt * H + h) * dv;
                for (int i = 0; i < dk; ++i) {
                    const double gi = exp(log_decay(at[i], b, mode));
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = gi * S[(size_t)i * dv + j] + kt[i] * vt[j];
                }
            }

            if (dhT)
                memcpy(D, dhT + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(D, 0, ssz * sizeof(double));

            for (int64_t w = nwin - 1; w >= 0; --w) {
                const int64_t ws = w * window;
                const int64_t we = (ws + window < L) ? ws + window : L;
                memcpy(S, ck + (size_t)w * ssz, ssz * sizeof(double));
                for (int64_t t = ws; t < we; ++t) {
                    memcpy(win + (size_t)(t - ws) * ssz, S, ssz * sizeof(double));
                    const int64_t tt = t0 + t;
                    const double *at = a + ((size_t)tt * H + h) * dk;
                    const double *kt = k + ((size_t)tt * H + h) * dk;
                    const double *vt = v + ((size_t)tt * H + h) * dv;
                    for (int i = 0; i < dk; ++i) {
                        const double gi = exp(log_decay(at[i], b, mode));
                        for (int j = 0; j < dv; ++j)
                            S[(size_t)i * dv + j] = gi * S[(size_t)i * dv + j] + kt[i] * vt[j];
                    }
                }
                for (int64_t t = we - 1; t >= ws; --t) {
                    const int64_t tt = t0 + t;
                    const double *at = a + ((size_t)tt * H + h) * dk;
                    const double *qt = q + ((size_t)tt * H + h) * dk;
                    const double *kt = k + ((size_t)tt * H + h) * dk;
                    const double *vt = v + ((size_t)tt * H + h) * dv;
                    const double *gt = dO + ((size_t)tt * H + h) * dv;
                    double *dqt = dq + ((size_t)tt * H + h) * dk;
                    double *dkt = dkk + ((size_t)tt * H + h) * dk;
                    double *dvt = dvv + ((size_t)tt * H + h) * dv;
                    double *dat = da + ((size_t)tt * H + h) * dk;
                    const double *Sp = win + (size_t)(t - ws) * ssz; /* S_{t-1} */
                    for (int i = 0; i < dk; ++i)
                        g[i] = exp(log_decay(at[i], b, mode));
                    /* D += q_t dO_t^T  (adjoint of S_t) */
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            D[(size_t)i * dv + j] += qt[i] * gt[j];
                    /* dq_t = S_t dO_t with S_t = diag(g) S_{t-1} + k v^T */
                    for (int i = 0; i < dk; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; ++j)
                            acc += (g[i] * Sp[(size_t)i * dv + j] + kt[i] * vt[j]) * gt[j];
                        dqt[i] = acc;
                    }
                    /* dk_t = D v_t */
                    for (int i = 0; i < dk; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; ++j)
                            acc += D[(size_t)i * dv + j] * vt[j];
                        dkt[i] = acc;
                    }
                    /* dv_t = D^T k_t */
                    for (int j = 0; j < dv; ++j)
                        dvt[j] = 0.0;
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            dvt[j] += D[(size_t)i * dv + j] * kt[i];
                    /* dlambda_t[i] = g_t[i] <D[i,:], S_{t-1}[i,:]>;  da = dlambda * dlambda/da */
                    for (int i = 0; i < dk; ++i) {
                        double dot = 0.0;
                        for (int j = 0; j < dv; ++j)
                            dot += D[(size_t)i * dv + j] * Sp[(size_t)i * dv + j];
                        dat[i] = g[i] * dot * log_decay_deriv(at[i], b, mode);
                    }
                    /* adjoint of S_{t-1}: row i decays by g_t[i] */
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            D[(size_t)i * dv + j] *= g[i];
                }
            }
            if (dh0)
                memcpy(dh0 + (size_t)u * ssz, D, ssz * sizeof(double));
            free(ck);
        }
        free(win);
        free(g);
        free(D);
        free(S);
    }
    return used;
}

/*
 * Gated delta rule with the bounded log-decay: the "Delta Net-style"
 * structure [P1] sec. 3.1 names beside linear attention, to which the same
 * parameterisation substitution applies.  The rule itself is the published
 * one ("Gated Delta Networks: Improving Mamba2 with Delta Rule", Yang, Kautz
 * and Hatamizadeh, 2024), written for a dk x dv state read by o = S^T q:
 *     g_t = exp(lambda_t),  lambda_t = b * sigmoid(a_t) or -softplus(a_t)
 *     S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,  S_0 = h0
 *     o_t = S_t^T q_t,                                             hT = S_L
 * with one write strength beta_t per (token, head), given as an input
 * (beta [Ttot][H]; the caller maps its own logits into (0, 1)).  Computed as
 *     r_t = S_{t-1}^T k_t,   e_t = v_t - g_t r_t,   S_t = g_t S_{t-1} + beta_t k_t e_t^T,
 * which is the same update with the projection multiplied out.
 */
int oracle_fwd_delta(int N, const int64_t *cu, int H, int dk, int dv,
                     const double *q, const double *k, const double *v,
                     const double *a, const double *beta, double b, int mode,
                     const double *h0, double *o, double *hT, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
        double *e = (double *)malloc((size_t)dv * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {
                const double g = exp(log_decay(a[t * H + h], b, mode));
                const double bt = beta[t * H + h];
                const double *qt = q + ((size_t)t * H + h) * dk;
                const double *kt = k + ((size_t)t * H + h) * dk;
                const double *vt = v + ((size_t)t * H + h) * dv;
                double *ot = o + ((size_t)t * H + h) * dv;
                /* e = v_t - g_t S_{t-1}^T k_t */
                for (int j = 0; j < dv; ++j) {
                    double r = 0.0;
                    for (int i = 0; i < dk; ++i)
                        r += S[(size_t)i * dv + j] * kt[i];
                    e[j] = vt[j] - g * r;
                }
                /* S_t = g_t S_{t-1} + beta_t k_t e^T */
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j)
                        S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + bt * kt[i] * e[j];
                /* o_t = S_t^T q_t */
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dk; ++i)
                        acc += S[(size_t)i * dv + j] * qt[i];
                    ot[j] = acc;
                }
            }
            if (hT)
                memcpy(hT + (size_t)u * ssz, S, ssz * sizeof(double));
        }
        free(e);
        free(S);
    }
    return used;
}

/*
 * Reverse mode of oracle_fwd_delta for the loss <o, dO> + <hT, dhT>.  With D
 * the adjoint of S_t and r, e as in the forward:
 *   D += q_t dO_t^T;          dq_t = S_t dO_t
 *   de = beta_t D^T k_t;      dv_t = de;            dr = -g_t de
 *   dk_t = beta_t D e + S_{t-1} dr
 *   dbeta_t = k_t^T D e
 *   dlambda_t = g_t (<D, S_{t-1}> - r . de);        da_t = dlambda_t dlambda/da
 *   D <- g_t D + k_t dr^T      (adjoint of S_{t-1})
 * and dh0 = D at the end.  S_{t-1} comes from fp64 checkpoints every
 * `window` tokens, recomputed forward inside each window.
 */
static void delta_step(int dk, int dv, double *S, const double *kt, const double *vt, double g, double bt,
                       double *e)
{
    for (int j = 0; j < dv; ++j) {
        double r = 0.0;
        for (int i = 0; i < dk; ++i)
            r += S[(size_t)i * dv + j] * kt[i];
        e[j] = vt[j] - g * r;
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + bt * kt[i] * e[j];
}

int oracle_bwd_delta(int N, const int64_t *cu, int H, int dk, int dv,
                     const double *q, const double *k, const double *v,
                     const double *a, const double *beta, double b, int mode,
                     const double *h0, const double *dO, const double *dhT,
                     double *dq, double *dkk, double *dvv, double *da, double *dbeta,
                     double *dh0, int window, int nthreads)
{
    int used = set_threads(nthreads);
    const int64_t units = (int64_t)N * H;
    const size_t ssz = (size_t)dk * dv;
    if (window <= 0)
        window = 1024;

#pragma omp parallel
    {
        double *S = (double *)malloc(ssz * sizeof(double));
        double *D = (double *)malloc(ssz * sizeof(double));
        double *e = (double *)malloc((size_t)dv * sizeof(double));
        double *r = (double *)malloc((size_t)dv * sizeof(double));
        double *de = (double *)malloc((size_t)dv * sizeof(double));
        double *dr = (double *)malloc((size_t)dv * sizeof(double));
        double *win = (double *)malloc((size_t)window * ssz * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t u = 0; u < units; ++u) {
            const int n = (int)(u / H), h = (int)(u % H);
            const int64_t t0 = cu[n], L = cu[n + 1] - cu[n];
            const int64_t nwin = (L + window - 1) / window;
            double *ck = (double *)malloc((size_t)(nwin > 0 ? nwin : 1) * ssz * sizeof(double));

            /* forward sweep: checkpoint S before each window */
            if (h0)
                memcpy(S, h0 + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(S, 0, ssz * sizeof(double));
            for (int64_t t = 0; t < L; ++t) {
                if (t % window == 0)
                    memcpy(ck + (size_t)(t / window) * ssz, S, ssz * sizeof(double));
                const int64_t tt = t0 + t;
                delta_step(dk, dv, S, k + ((size_t)tt * H + h) * dk, v + ((size_t)tt * H + h) * dv,
                           exp(log_decay(a[tt * H + h], b, mode)), beta[tt * H + h], e);
            }

            if (dhT)
                memcpy(D, dhT + (size_t)u * ssz, ssz * sizeof(double));
            else
                memset(D, 0, ssz * sizeof(double));

            for (int64_t w = nwin - 1; w >= 0; --w) {
                const int64_t ws = w * window;
                const int64_t we = (ws + window < L) ? ws + window : L;
                memcpy(S, ck + (size_t)w * ssz, ssz * sizeof(double));
                for (int64_t t = ws; t < we; ++t) {
                    memcpy(win + (size_t)(t - ws) * ssz, S, ssz * sizeof(double));
                    const int64_t tt = t0 + t;
                    delta_step(dk, dv, S, k + ((size_t)tt * H + h) * dk, v + ((size_t)tt * H + h) * dv,
                               exp(log_decay(a[tt * H + h], b, mode)), beta[tt * H + h], e);
                }
                for (int64_t t = we - 1; t >= ws; --t) {
                    const int64_t tt = t0 + t;
                    const double at = a[tt * H + h];
                    const double g = exp(log_decay(at, b, mode));
                    const double bt = beta[tt * H + h];
                    const double *qt = q + ((size_t)tt * H + h) * dk;
                    const double *kt = k + ((size_t)tt * H + h) * dk;
                    const double *vt = v + ((size_t)tt * H + h) * dv;
                    const double *gt = dO + ((size_t)tt * H + h) * dv;
                    double *dqt = dq + ((size_t)tt * H + h) * dk;
                    double *dkt = dkk + ((size_t)tt * H + h) * dk;
                    double *dvt = dvv + ((size_t)tt * H + h) * dv;
                    const double *Sp = win + (size_t)(t - ws) * ssz; /* S_{t-1} */
                    /* r = S_{t-1}^T k_t,  e = v_t - g r */
                    for (int j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (int i = 0; i < dk; ++i)
                            acc += Sp[(size_t)i * dv + j] * kt[i];
                        r[j] = acc;
                        e[j] = vt[j] - g * acc;
                    }
                    /* D += q_t dO_t^T  (adjoint of S_t) */
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            D[(size_t)i * dv + j] += qt[i] * gt[j];
                    /* dq_t = S_t dO_t with S_t = g S_{t-1} + beta k e^T */
                    for (int i = 0; i < dk; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < dv; ++j)
                            acc += (g * Sp[(size_t)i * dv + j] + bt * kt[i] * e[j]) * gt[j];
                        dqt[i] = acc;
                    }
                    /* de = beta D^T k;  dv_t = de;  dr = -g de */
                    for (int j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (int i = 0; i < dk; ++i)
                            acc += D[(size_t)i * dv + j] * kt[i];
                        de[j] = bt * acc;
                        dvt[j] = de[j];
                        dr[j] = -g * de[j];
                    }
                    /* dk_t = beta D e + S_{t-1} dr;  dbeta_t = k^T D e */
                    double db = 0.0;
                    for (int i = 0; i < dk; ++i) {
                        double De = 0.0, Sdr = 0.0;
                        for (int j = 0; j < dv; ++j) {
                            De += D[(size_t)i * dv + j] * e[j];
                            Sdr += Sp[(size_t)i * dv + j] * dr[j];
                        }
                        dkt[i] = bt * De + Sdr;
                        db += kt[i] * De;
                    }
                    dbeta[tt * H + h] = db;
                    /* dlambda_t = g (<D, S_{t-1}> - r . de) */
                    double dot = 0.0;
                    for (size_t x = 0; x < ssz; ++x)
                        dot += D[x] * Sp[x];
                    double rde = 0.0;
                    for (int j = 0; j < dv; ++j)
                        rde += r[j] * de[j];
                    da[tt * H + h] = g * (dot - rde) * log_decay_deriv(at, b, mode);
                    /* adjoint of S_{t-1}: D <- g D + k dr^T */
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j)
                            D[(size_t)i * dv + j] = g * D[(size_t)i * dv + j] + kt[i] * dr[j];
                }
            }
            if (dh0)
                memcpy(dh0 + (size_t)u * ssz, D, ssz * sizeof(double));
            free(ck);
        }
        free(win);
        free(dr);
        free(de);
        free(r);
        free(e);
        free(D);
        free(S);
    }
    return used;
}
