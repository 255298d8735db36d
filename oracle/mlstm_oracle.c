/*
 * fp64 CPU oracle for the mLSTM matrix-memory cell.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Source: "xLSTM: Extended Long Short-Term Memory".
 *   part 28/30, "Parallel mLSTM Forward Pass": eqs (71)-(78);
 *   part 28/30, "Parallel mLSTM Backward Pass", forward summary: eqs (79)-(86)
 *     and the log forget matrix, eq (101);
 *   part 28/30, recurrent mLSTM backward, eqs (59)-(70) (the recurrent
 *     forward they differentiate is what oracle_recurrent_* evaluates);
 *   part 17/30, section 2.3 tail: forget gate eq (26), output gate eq (27),
 *     multiple heads equal multiple cells (no memory mixing), and the
 *     mLSTM reuses the sLSTM stabilization.
 *
 * Readings of the pages taken here (the pages do not print them):
 *  - The recurrent forward equations themselves are not on the pages; the
 *    recurrence is the one the backward equations (59)-(70) differentiate:
 *      C_t = f_t C_{t-1} + i_t v_t k_t^T,   n_t = f_t n_{t-1} + i_t k_t,
 *      h~_t = C_t q_t / max(|n_t^T q_t|, 1),  h_t = o_t (.) h~_t,
 *    with i_t = exp(i~_t) (eq 69 has dL/di~ proportional to exp(i~)), and the
 *    forget activation f_t = sigma(f~_t), the one the parallel form fixes
 *    (eq 71 builds F from sigma(f~)).
 *  - k enters scaled by 1/sqrt(d_qk) (the 1/sqrt(d) factor is moved onto K
 *    below eq 76); q is unscaled.
 *  - Stabilizer (sLSTM eq 15 is not on the pages): a running log-space max
 *    m_t = max(log f_t + m_{t-1}, i~_t) with gates rescaled by exp(-m_t), and
 *    the normalizer floor 1 becoming exp(-m_t).  The state starts at C=0, n=0,
 *    m=-inf.  The stored (C, n) is the true state times exp(-m), so h~ does
 *    not depend on m in exact arithmetic; this m is the one that equals the
 *    parallel form's row maximum (80) at every step and keeps every rescaled
 *    gate at most 1.
 *  - The max in (75) is the row-wise max of (80).
 *
 * All arithmetic is IEEE fp64; build without -ffast-math (-inf must flow).
 * Layouts are row-major with the last index fastest:
 *   q,k [B,H,T,dqk]  v [B,H,T,dv]  igate,fgate [B,H,T]  og [B,H,T,dv]
 *   h   [B,H,T,dv]   C [B,H,dv,dqk]  n [B,H,dqk]  m [B,H]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0   /* >0 plants a known mistake (mutation tests only) */
#endif

int oracle_mutation(void) { return ORACLE_MUTATION; }

/* Team size of one call: the caller's count, or the OpenMP default when it
 * passes 0.  Given to each parallel region by a num_threads clause, so that one
 * call's choice never carries over to the next (unlike omp_set_num_threads). */
static int team_size(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* log(sigma(x)) evaluated without overflow: min(x,0) - log1p(exp(-|x|)).
 * Gives 0 at x=+inf and -inf at x=-inf. */
static double log_sigmoid(double x)
{
#if ORACLE_MUTATION == 7
    return x;                       /* mutation: exponential forget activation */
#else
    double mn = x < 0.0 ? x : 0.0;
    return mn - log1p(exp(-fabs(x)));
#endif
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* The forget-gate activation: sigma (log f = log sigma(f~), the default the
 * parallel form fixes in eqs 71 and 101) or exp (log f = f~; part 28/30 eq 70
 * allows gamma = exp).  Selected for the whole library by
 * oracle_set_forget_exp; the tests set it around a call. */
static int g_forget_exp = 0;
void oracle_set_forget_exp(int on) { g_forget_exp = on ? 1 : 0; }
static double log_forget(double x) { return g_forget_exp ? x : log_sigmoid(x); }

static double key_scale(int dqk)
{
#if ORACLE_MUTATION == 1
    (void)dqk;
    return 1.0;                     /* mutation: 1/sqrt(d) dropped */
#else
    return 1.0 / sqrt((double)dqk);
#endif
}

/* ---------------------------------------------------------------------------
 * Stabilized parallel forward for one head, one query row i (0-based).
 * part 28/30, eqs (79)-(86); eq (101) for log F; eq (78) for the output gate.
 *   D~_ij = Fbar_ij + I~_ij,  Fbar_ij = sum_{k=j+1..i} log sigma(f~_k)  (j<=i)
 *   m_i   = max_j D~_ij                                   (row-wise, eq 80)
 *   D'_ij = exp(D~_ij - m_i)                              (eq 81)
 *   C~'_ij = (q_i . k_j)/sqrt(d) * D'_ij                  (eq 82)
 *   b_i   = sum_j C~'_ij                                  (eq 83)
 *   n_i   = max(|b_i|, exp(-m_i))                         (eq 84)
 *   H~_i  = sum_j (C~'_ij / n_i) v_j                      (eqs 85-86)
 * Entries with j > i have Fbar = -inf, so D' = 0 there and they drop out of
 * every sum over j (the pages sum over j = 1..T).
 * `dt` and `cp` are scratch of length T.
 */
static void parallel_row(int T, int dqk, int dv, const double *q, const double *k,
                         const double *v, const double *ig, const double *fg,
                         const double *og, int i, double *h_row, double *m_row,
                         double *n_row, double *dt, double *cp)
{
    (void)T;
    const double s = key_scale(dqk);
    /* eq (101), evaluated for this row by walking j down from i: the sum over
     * k = j+1..i grows by one term log sigma(f~_{j+1}) per step. */
    double fbar = 0.0;              /* Fbar_ii = 0 */
    for (int j = i; j >= 0; --j) {
        if (j < i) {
#if ORACLE_MUTATION == 4
            fbar += log_forget(fg[j]);           /* mutation: sum starts at k=j */
#else
            fbar += log_forget(fg[j + 1]);
#endif
        }
        dt[j] = fbar + ig[j];       /* eq (79): D~ = Fbar + I~, I~_ij = i~_j (eq 72) */
    }
    double m = -INFINITY;           /* eq (80) */
    for (int j = 0; j <= i; ++j) if (dt[j] > m) m = dt[j];
    double b = 0.0;
    const double *qi = q + (size_t)i * dqk;
    for (int j = 0; j <= i; ++j) {
        const double *kj = k + (size_t)j * dqk;
        double qk = 0.0;
#if ORACLE_MUTATION == 8
        (void)kj;                   /* mutation: q_j . k_i instead of q_i . k_j */
        for (int c = 0; c < dqk; ++c) qk += q[(size_t)j * dqk + c] * k[(size_t)i * dqk + c];
#else
        for (int c = 0; c < dqk; ++c) qk += qi[c] * kj[c];
#endif
        double dprime = exp(dt[j] - m);                     /* eq (81) */
        cp[j] = qk * s * dprime;                            /* eq (82) */
        b += cp[j];                                         /* eq (83) */
    }
#if ORACLE_MUTATION == 3
    double nrm = fmax(fabs(b), 1.0);                        /* mutation: floor 1 */
#elif ORACLE_MUTATION == 6
    double nrm = fmax(b, exp(-m));                          /* mutation: no |.| */
#else
    double nrm = fmax(fabs(b), exp(-m));                    /* eq (84) */
#endif
    for (int c = 0; c < dv; ++c) h_row[c] = 0.0;
    for (int j = 0; j <= i; ++j) {
        double w = cp[j] / nrm;                             /* eq (85) */
        const double *vj = v + (size_t)j * dv;
        for (int c = 0; c < dv; ++c) h_row[c] += w * vj[c]; /* eq (86) */
    }
    if (og) {                                               /* eq (78) */
        const double *oi = og + (size_t)i * dv;
        for (int c = 0; c < dv; ++c) h_row[c] *= sigmoid(oi[c]);
    }
    if (m_row) *m_row = m;
    if (n_row) *n_row = nrm;
}

/* Full stabilized parallel forward over all (b,h) and all rows. */
int oracle_parallel_stabilized(int B, int H, int T, int dqk, int dv,
                               const double *q, const double *k, const double *v,
                               const double *ig, const double *fg, const double *og,
                               double *h, double *m_out, double *n_out, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
#pragma omp parallel num_threads(nteam)
    {
        double *dt = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
        double *cp = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            const double *qh = q + (size_t)bh * T * dqk, *kh = k + (size_t)bh * T * dqk;
            const double *vh = v + (size_t)bh * T * dv;
            const double *igh = ig + (size_t)bh * T, *fgh = fg + (size_t)bh * T;
            const double *ogh = og ? og + (size_t)bh * T * dv : NULL;
            for (int i = 0; i < T; ++i)
                parallel_row(T, dqk, dv, qh, kh, vh, igh, fgh, ogh, i,
                             h + ((size_t)bh * T + i) * dv,
                             m_out ? m_out + (size_t)bh * T + i : NULL,
                             n_out ? n_out + (size_t)bh * T + i : NULL, dt, cp);
        }
        free(dt);
        free(cp);
    }
    return 0;
}

/* Stabilized parallel forward for a list of sampled rows.  rows[r] holds a
 * flat (bh, i) pair as bh*T + i; row r of h_out/m_out/n_out receives it. */
int oracle_parallel_rows(int B, int H, int T, int dqk, int dv,
                         const double *q, const double *k, const double *v,
                         const double *ig, const double *fg, const double *og,
                         const long *rows, int nrows,
                         double *h_out, double *m_out, double *n_out, int nthreads)
{
    if (B < 0 || H < 0 || T <= 0 || dqk <= 0 || dv <= 0 || nrows < 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BHT = (long)B * H * T;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= BHT) return -1;
#pragma omp parallel num_threads(nteam)
    {
        double *dt = (double *)malloc(sizeof(double) * T);
        double *cp = (double *)malloc(sizeof(double) * T);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            long bh = rows[r] / T;
            int i = (int)(rows[r] % T);
            parallel_row(T, dqk, dv, q + (size_t)bh * T * dqk, k + (size_t)bh * T * dqk,
                         v + (size_t)bh * T * dv, ig + (size_t)bh * T, fg + (size_t)bh * T,
                         og ? og + (size_t)bh * T * dv : NULL, i, h_out + (size_t)r * dv,
                         m_out ? m_out + r : NULL, n_out ? n_out + r : NULL, dt, cp);
        }
        free(dt);
        free(cp);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Unstabilized parallel forward, part 28/30 eqs (71)-(73) and (76):
 *   F_ij = prod_{k=j+1..i} sigma(f~_k) (1 on the diagonal, 0 above),
 *   D = F (.) exp(I~),  C~ = (Q K^T / sqrt(d)) (.) D,
 *   H~ = C V,  C = C~ / max(|sum_j C~_ij|, 1).
 * Overflows for large |i~| or long sequences; used on small inputs only.
 */
int oracle_parallel_unstabilized(int B, int H, int T, int dqk, int dv,
                                 const double *q, const double *k, const double *v,
                                 const double *ig, const double *fg, const double *og,
                                 double *h, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
    const double s = key_scale(dqk);
#pragma omp parallel num_threads(nteam)
    {
        double *ct = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            const double *qh = q + (size_t)bh * T * dqk, *kh = k + (size_t)bh * T * dqk;
            const double *vh = v + (size_t)bh * T * dv;
            const double *igh = ig + (size_t)bh * T, *fgh = fg + (size_t)bh * T;
            for (int i = 0; i < T; ++i) {
                double rowsum = 0.0;
                for (int j = 0; j <= i; ++j) {
                    double F = 1.0;                             /* eq (71) */
                    for (int kk = j + 1; kk <= i; ++kk) F *= exp(log_forget(fgh[kk]));
                    double D = F * exp(igh[j]);                 /* eq (73) */
                    double qk = 0.0;
                    for (int c = 0; c < dqk; ++c) qk += qh[(size_t)i * dqk + c] * kh[(size_t)j * dqk + c];
                    ct[j] = qk * s * D;                         /* eq (76), C~ */
                    rowsum += ct[j];
                }
                double nrm = fmax(fabs(rowsum), 1.0);
                double *hr = h + ((size_t)bh * T + i) * dv;
                for (int c = 0; c < dv; ++c) hr[c] = 0.0;
                for (int j = 0; j <= i; ++j)
                    for (int c = 0; c < dv; ++c) hr[c] += ct[j] / nrm * vh[(size_t)j * dv + c];
                if (og) {
                    const double *oi = og + ((size_t)bh * T + i) * dv;
                    for (int c = 0; c < dv; ++c) hr[c] *= sigmoid(oi[c]);
                }
            }
        }
        free(ct);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * One stabilized recurrent step on a single head's state, in place.
 * C [dv,dqk], n [dqk], *m scalar; q,k [dqk], v [dv]; og [dv] or NULL; h [dv].
 *   m'  = max(log sigma(f~) + m, i~)
 *   f'  = exp(log sigma(f~) + m - m'),  i' = exp(i~ - m')
 *   C  <- f' C + i' v (k/sqrt(d))^T,    n <- f' n + i' k/sqrt(d)
 *   h~  = C q / max(|n . q|, exp(-m')), h = sigma(o~) (.) h~   (eqs 27, 59)
 * The stored state is the true state scaled by exp(-m).
 */
static void step_head(int dqk, int dv, double *C, double *n, double *m,
                      const double *q, const double *k, const double *v,
                      double igv, double fgv, const double *og, double *h)
{
    const double s = key_scale(dqk);
    const double lf = log_forget(fgv);
    double m_prev = *m;
#if ORACLE_MUTATION == 2
    if (isinf(m_prev) && m_prev < 0) m_prev = 0.0;   /* mutation: m_0 = 0 */
#endif
    const double m_new = fmax(lf + m_prev, igv);
    const double fp = exp(lf + m_prev - m_new);
#if ORACLE_MUTATION == 5
    const double ip = exp(igv);                      /* mutation: i' not rescaled */
#else
    const double ip = exp(igv - m_new);
#endif
    for (int r = 0; r < dv; ++r) {
        double acc = 0.0;
        for (int c = 0; c < dqk; ++c) {
            double cv = fp * C[(size_t)r * dqk + c] + ip * v[r] * (k[c] * s);
            C[(size_t)r * dqk + c] = cv;
            acc += cv * q[c];
        }
        h[r] = acc;
    }
    double nq = 0.0;
    for (int c = 0; c < dqk; ++c) {
        n[c] = fp * n[c] + ip * (k[c] * s);
        nq += n[c] * q[c];
    }
    const double nrm = fmax(fabs(nq), exp(-m_new));
    for (int r = 0; r < dv; ++r) {
        h[r] /= nrm;
        if (og) h[r] *= sigmoid(og[r]);
    }
    *m = m_new;
}

/* One stabilized step for every head, state updated in place (the generation
 * step).  q,k [B,H,dqk]; v,og,h [B,H,dv]; igate,fgate [B,H]. */
int oracle_step(int B, int H, int dqk, int dv, double *C, double *n, double *m,
                const double *q, const double *k, const double *v, const double *og,
                const double *ig, const double *fg, double *h, int nthreads)
{
    if (B < 0 || H < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
#pragma omp parallel for schedule(static) num_threads(nteam)
    for (long bh = 0; bh < BH; ++bh)
        step_head(dqk, dv, C + (size_t)bh * dv * dqk, n + (size_t)bh * dqk, m + bh,
                  q + (size_t)bh * dqk, k + (size_t)bh * dqk, v + (size_t)bh * dv,
                  ig[bh], fg[bh], og ? og + (size_t)bh * dv : NULL, h + (size_t)bh * dv);
    return 0;
}

/* Stabilized recurrent forward over whole sequences from C=0, n=0, m=-inf.
 * Writes h [B,H,T,dv] and, when non-NULL, the final state C, n, m. */
int oracle_recurrent_stabilized(int B, int H, int T, int dqk, int dv,
                                const double *q, const double *k, const double *v,
                                const double *ig, const double *fg, const double *og,
                                double *h, double *C_out, double *n_out, double *m_out,
                                int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
#pragma omp parallel num_threads(nteam)
    {
        double *C = (double *)malloc(sizeof(double) * dv * dqk);
        double *n = (double *)malloc(sizeof(double) * dqk);
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            memset(C, 0, sizeof(double) * dv * dqk);
            memset(n, 0, sizeof(double) * dqk);
            double m = -INFINITY;
            for (int t = 0; t < T; ++t) {
                size_t ti = (size_t)bh * T + t;
                step_head(dqk, dv, C, n, &m, q + ti * dqk, k + ti * dqk, v + ti * dv,
                          ig[ti], fg[ti], og ? og + ti * dv : NULL, h + ti * dv);
            }
            if (C_out) memcpy(C_out + (size_t)bh * dv * dqk, C, sizeof(double) * dv * dqk);
            if (n_out) memcpy(n_out + (size_t)bh * dqk, n, sizeof(double) * dqk);
            if (m_out) m_out[bh] = m;
        }
        free(C);
        free(n);
    }
    return 0;
}

/* Unstabilized recurrent forward, the recurrence eqs (59)-(70) differentiate:
 * f = sigma(f~), i = exp(i~), C = f C + i v (k/sqrt d)^T, n = f n + i k/sqrt d,
 * h~ = C q / max(|n.q|, 1).  Small inputs only (exp(i~) is not bounded). */
int oracle_recurrent_unstabilized(int B, int H, int T, int dqk, int dv,
                                  const double *q, const double *k, const double *v,
                                  const double *ig, const double *fg, const double *og,
                                  double *h, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
    const double s = key_scale(dqk);
#pragma omp parallel num_threads(nteam)
    {
        double *C = (double *)malloc(sizeof(double) * dv * dqk);
        double *n = (double *)malloc(sizeof(double) * dqk);
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            memset(C, 0, sizeof(double) * dv * dqk);
            memset(n, 0, sizeof(double) * dqk);
            for (int t = 0; t < T; ++t) {
                size_t ti = (size_t)bh * T + t;
                const double *qt = q + ti * dqk, *kt = k + ti * dqk, *vt = v + ti * dv;
                const double f = exp(log_forget(fg[ti])), i = exp(ig[ti]);
                double nq = 0.0;
                for (int c = 0; c < dqk; ++c) {
                    n[c] = f * n[c] + i * kt[c] * s;
                    nq += n[c] * qt[c];
                }
                const double nrm = fmax(fabs(nq), 1.0);
                for (int r = 0; r < dv; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < dqk; ++c) {
                        C[(size_t)r * dqk + c] = f * C[(size_t)r * dqk + c] + i * vt[r] * kt[c] * s;
                        acc += C[(size_t)r * dqk + c] * qt[c];
                    }
                    double hv = acc / nrm;
                    if (og) hv *= sigmoid(og[ti * dv + r]);
                    h[ti * dv + r] = hv;
                }
            }
        }
        free(C);
        free(n);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Stabilized parallel BACKWARD for one head, part 28/30 "Parallel mLSTM
 * Backward Pass", eqs (87)-(105), evaluated literally with dense T x T
 * matrices (the forward quantities of eqs (79)-(84) are recomputed first).
 * Given dH~ = dL/dH~ [T, dv], it returns dQ, dK [T, dqk], dV [T, dv] and the
 * pre-activation gradients d i~, d f~ [T].  The pages treat the stabilizer m
 * as a constant (its gradients cancel), and so does this routine.
 * Readings (the printed equations are garbled in places):
 *  - eq (90) prints sign(n); the derivative of n = max(|b|, e^-m) with
 *    respect to b is sign(b) where |b| exceeds the floor, so sign(b) is used;
 *  - eq (93): delta_{C~',B} is the delta_{C~',b} of eq (92);
 *  - eq (100): C is the normalised matrix C~' (.) (n^-1 1^T) of eq (85);
 *  - eq (105): the vector is d i~ = [d i~_1 .. d i~_T] (printed "S").
 * Matrix entries above the diagonal are zero (D' = 0 there) and are skipped.
 * Scratch: 5 T*T doubles + 4 T.
 */
static void backward_head(int T, int dqk, int dv, const double *q, const double *k,
                          const double *v, const double *ig, const double *fg, const double *dh,
                          double *dq, double *dk, double *dvv, double *dig, double *dfg,
                          double *S, double *Dp, double *Ct, double *dC, double *dDt,
                          double *m, double *b, double *n, double *rs)
{
    const double s = key_scale(dqk);
    /* forward recompute: D~ (eqs 79, 101), m (80), D' (81), C~' (82), b (83), n (84) */
    for (int i = 0; i < T; ++i) {
        double fbar = 0.0, mi = -INFINITY;
        for (int j = i; j >= 0; --j) {
            if (j < i) fbar += log_forget(fg[j + 1]);
            Dp[(size_t)i * T + j] = fbar + ig[j];                 /* D~ for now */
            if (Dp[(size_t)i * T + j] > mi) mi = Dp[(size_t)i * T + j];
        }
        m[i] = mi;
        double bi = 0.0;
        for (int j = 0; j <= i; ++j) {
            double qk = 0.0;
            for (int c = 0; c < dqk; ++c) qk += q[(size_t)i * dqk + c] * k[(size_t)j * dqk + c];
            S[(size_t)i * T + j] = qk * s;                        /* Q K^T / sqrt(d) */
            Dp[(size_t)i * T + j] = exp(Dp[(size_t)i * T + j] - mi);
            Ct[(size_t)i * T + j] = S[(size_t)i * T + j] * Dp[(size_t)i * T + j];
            bi += Ct[(size_t)i * T + j];
        }
        b[i] = bi;
        n[i] = fmax(fabs(bi), exp(-mi));
    }
    for (int i = 0; i < T; ++i) {
        /* eq (87): dC = dH~ V^T */
        for (int j = 0; j <= i; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dv; ++c) acc += dh[(size_t)i * dv + c] * v[(size_t)j * dv + c];
            dC[(size_t)i * T + j] = acc;
        }
        /* eq (89): dn = -((C~' (.) dC) 1) (.) n^-2 */
        double r = 0.0;
        for (int j = 0; j <= i; ++j) r += Ct[(size_t)i * T + j] * dC[(size_t)i * T + j];
        const double dn = -r / (n[i] * n[i]);
        /* eq (90): db = sign(b) (.) dn where |b| > exp(-m) */
#if ORACLE_MUTATION == 9
        const double db = fabs(b[i]) > exp(-m[i]) ? dn : 0.0;   /* mutation: sign(n) taken literally */
#else
        const double db = fabs(b[i]) > exp(-m[i]) ? (b[i] > 0 ? dn : (b[i] < 0 ? -dn : 0.0)) : 0.0;
#endif
        for (int j = 0; j <= i; ++j) {
            /* eqs (91)-(93): dC~' = dC / n + db, both broadcast along the row */
#if ORACLE_MUTATION == 10
            const double dct = dC[(size_t)i * T + j] / n[i];         /* mutation: eq (92) term dropped */
#else
            const double dct = dC[(size_t)i * T + j] / n[i] + db;
#endif
            const double ddp = S[(size_t)i * T + j] * dct;        /* eq (94) */
            dDt[(size_t)i * T + j] = Dp[(size_t)i * T + j] * ddp; /* eq (95) */
            dC[(size_t)i * T + j] = Dp[(size_t)i * T + j] * dct;  /* D' (.) dC~', kept for (98)-(99) */
        }
    }
    /* eq (98): dQ = (D' (.) dC~') K / sqrt(d) */
    for (int i = 0; i < T; ++i)
        for (int c = 0; c < dqk; ++c) {
            double acc = 0.0;
            for (int j = 0; j <= i; ++j) acc += dC[(size_t)i * T + j] * k[(size_t)j * dqk + c];
            dq[(size_t)i * dqk + c] = acc * s;
        }
    /* eq (99): dK = (D' (.) dC~')^T Q / sqrt(d) */
    for (int j = 0; j < T; ++j)
        for (int c = 0; c < dqk; ++c) {
            double acc = 0.0;
#if ORACLE_MUTATION == 12
            for (int i = j; i < T; ++i) acc += dC[(size_t)i * T + j] * k[(size_t)i * dqk + c];  /* mutation: K for Q */
#else
            for (int i = j; i < T; ++i) acc += dC[(size_t)i * T + j] * q[(size_t)i * dqk + c];
#endif
            dk[(size_t)j * dqk + c] = acc * s;
        }
    /* eq (100): dV = C^T dH~ with C = C~' (.) (n^-1 1^T) */
    for (int j = 0; j < T; ++j)
        for (int c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int i = j; i < T; ++i) acc += Ct[(size_t)i * T + j] / n[i] * dh[(size_t)i * dv + c];
            dvv[(size_t)j * dv + c] = acc;
        }
    /* eqs (96), (102)-(103): dFbar = dD~; d fbar_k = sum_{j<k} sum_{i>=k} dFbar_ij;
     * d f~_k = sigma(-f~_k) d fbar_k */
    for (int kk = 0; kk < T; ++kk) {
        double acc = 0.0;
        for (int i = kk; i < T; ++i)
#if ORACLE_MUTATION == 11
            for (int j = 0; j <= kk && j <= i; ++j) acc += dDt[(size_t)i * T + j];   /* mutation: j <= k */
#else
            for (int j = 0; j < kk; ++j) acc += dDt[(size_t)i * T + j];
#endif
        rs[kk] = acc;
        /* eq (103) for sigma; d f~/d fbar = 1 for the exp activation */
        dfg[kk] = (g_forget_exp ? 1.0 : sigmoid(-fg[kk])) * acc;
    }
    /* eqs (97), (105): dI = dD~; d i~_k = sum_{i>=k} dI_ik */
    for (int kk = 0; kk < T; ++kk) {
        double acc = 0.0;
        for (int i = kk; i < T; ++i) acc += dDt[(size_t)i * T + kk];
        dig[kk] = acc;
    }
}

int oracle_parallel_backward(int B, int H, int T, int dqk, int dv,
                             const double *q, const double *k, const double *v,
                             const double *ig, const double *fg, const double *dh,
                             double *dq, double *dk, double *dvv, double *dig, double *dfg, int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
    const size_t TT = (size_t)(T > 0 ? T : 1) * (size_t)(T > 0 ? T : 1);
    int fail = 0;
#pragma omp parallel num_threads(nteam)
    {
        double *buf = (double *)malloc(sizeof(double) * (5 * TT + 4 * (size_t)(T > 0 ? T : 1)));
        if (!buf) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            if (!buf) continue;
            double *S = buf, *Dp = S + TT, *Ct = Dp + TT, *dC = Ct + TT, *dDt = dC + TT;
            double *m = dDt + TT, *b = m + T, *n = b + T, *rs = n + T;
            backward_head(T, dqk, dv, q + (size_t)bh * T * dqk, k + (size_t)bh * T * dqk, v + (size_t)bh * T * dv,
                          ig + (size_t)bh * T, fg + (size_t)bh * T, dh + (size_t)bh * T * dv,
                          dq + (size_t)bh * T * dqk, dk + (size_t)bh * T * dqk, dvv + (size_t)bh * T * dv,
                          dig + (size_t)bh * T, dfg + (size_t)bh * T, S, Dp, Ct, dC, dDt, m, b, n, rs);
        }
        free(buf);
    }
    return fail ? -2 : 0;
}

/* ---------------------------------------------------------------------------
 * Recurrent BACKWARD (backpropagation through time) of the unstabilized
 * recurrence, part 28/30 eqs (59)-(70):
 *   dh~_t = o_t (.) dh_t                                              (59)
 *   dC_{t-1}^T = f_t dC_t^T + q_{t-1} dh~_{t-1}^T / N_{t-1}             (60)
 *   dn_{t-1} = f_t dn_t - (q_{t-1}^T C_{t-1}^T dh~_{t-1}) / N_{t-1}^2
 *              Omega(n_{t-1}^T q_{t-1}) q_{t-1}                         (61)
 *   dv_t^T = i_t k_t^T dC_t^T,   dk_t^T = i_t (v_t^T dC_t + dn_t^T)      (62)-(63)
 *   dq_t = C_t^T dh~_t / N_t - (q_t^T C_t^T dh~_t) / N_t^2 Omega(n_t^T q_t) n_t   (64)
 *   d f~_t = (1^T (C_{t-1} (.) dC_t) 1 + 1^T (n_{t-1} (.) dn_t)) gamma(f~_t)   (68)
 *   d i~_t = (1^T ((v_t k_t^T) (.) dC_t) 1 + 1^T (k_t (.) dn_t)) exp(i~_t)     (69)
 *   d o~_t = h~_t (.) sigma'(o~_t) (.) dh_t                               (70)
 * with N_t = max(|n_t^T q_t|, 1), Omega(z) = Theta(z-1) - Theta(-z-1), and
 * gamma = sigma' or exp for the sigma or exp forget activation.  Readings:
 *  - the key enters as s k (s = 1/sqrt(d_qk), as in the forward), so the raw
 *    key's gradient is s times the k of eq (63);
 *  - dC_t and dn_t above are the totals flowing into step t (the eq 60/61
 *    recursion evaluated one step later), i.e. each includes step t's own
 *    output term.
 * The forward states C_t, n_t of every step are kept (small cases only).
 * og may be NULL (o_t = 1, d o~ not written).
 */
int oracle_recurrent_backward(int B, int H, int T, int dqk, int dv,
                              const double *q, const double *k, const double *v,
                              const double *ig, const double *fg, const double *og, const double *dh,
                              double *dq, double *dk, double *dvv, double *dig, double *dfg, double *dog,
                              int nthreads)
{
    if (B < 0 || H < 0 || T < 0 || dqk <= 0 || dv <= 0) return -1;
    const int nteam = team_size(nthreads);
    (void)nteam;
    const long BH = (long)B * H;
    const double s = key_scale(dqk);
    const size_t CS = (size_t)dv * dqk;
    int fail = 0;
#pragma omp parallel num_threads(nteam)
    {
        /* C_t, n_t for t = -1..T-1 (index t+1), plus dC, dn, dh~, h~ */
        double *Cs = (double *)malloc(sizeof(double) * CS * (size_t)(T + 1));
        double *ns = (double *)malloc(sizeof(double) * (size_t)dqk * (T + 1));
        double *dC = (double *)malloc(sizeof(double) * CS);
        double *dn = (double *)malloc(sizeof(double) * dqk);
        double *dht = (double *)malloc(sizeof(double) * dv);
        double *ht = (double *)malloc(sizeof(double) * dv);
        if (!Cs || !ns || !dC || !dn || !dht || !ht) {
#pragma omp atomic write
            fail = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long bh = 0; bh < BH; ++bh) {
            if (fail) continue;
            memset(Cs, 0, sizeof(double) * CS);          /* C_{-1} = 0 */
            memset(ns, 0, sizeof(double) * dqk);         /* n_{-1} = 0 */
            for (int t = 0; t < T; ++t) {                /* forward, keeping every state */
                const size_t ti = (size_t)bh * T + t;
                const double f = exp(log_forget(fg[ti])), i = exp(ig[ti]);
                const double *Cp = Cs + CS * t, *np = ns + (size_t)dqk * t;
                double *Cn = Cs + CS * (t + 1), *nn = ns + (size_t)dqk * (t + 1);
                for (int c = 0; c < dqk; ++c) nn[c] = f * np[c] + i * s * k[ti * dqk + c];
                for (int r = 0; r < dv; ++r)
                    for (int c = 0; c < dqk; ++c)
                        Cn[(size_t)r * dqk + c] = f * Cp[(size_t)r * dqk + c] + i * v[ti * dv + r] * s * k[ti * dqk + c];
            }
            memset(dC, 0, sizeof(double) * CS);
            memset(dn, 0, sizeof(double) * dqk);
            for (int t = T - 1; t >= 0; --t) {
                const size_t ti = (size_t)bh * T + t;
                const double *Ct = Cs + CS * (t + 1), *nt = ns + (size_t)dqk * (t + 1);
                const double *Cp = Cs + CS * t, *np = ns + (size_t)dqk * t;
                const double i = exp(ig[ti]);
                double nq = 0.0;
                for (int c = 0; c < dqk; ++c) nq += nt[c] * q[ti * dqk + c];
                const double N = fmax(fabs(nq), 1.0);
#if ORACLE_MUTATION == 13
                const double omega = nq > 1.0 ? 1.0 : 0.0;      /* mutation: Omega's negative branch dropped */
#else
                const double omega = (nq > 1.0 ? 1.0 : 0.0) - (-nq > 1.0 ? 1.0 : 0.0);
#endif
                for (int r = 0; r < dv; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < dqk; ++c) acc += Ct[(size_t)r * dqk + c] * q[ti * dqk + c];
                    ht[r] = acc / N;                                               /* h~_t */
                    const double o = og ? sigmoid(og[ti * dv + r]) : 1.0;
                    dht[r] = o * dh[ti * dv + r];                                  /* (59) */
                    if (og) dog[ti * dv + r] = ht[r] * o * (1.0 - o) * dh[ti * dv + r];   /* (70) */
                }
                /* q^T C_t^T dh~_t = (C_t q)^T dh~_t */
                double qCdh = 0.0;
                for (int r = 0; r < dv; ++r) qCdh += ht[r] * N * dht[r];
                /* step t's own output terms join the totals (60)-(61) */
                for (int r = 0; r < dv; ++r)
                    for (int c = 0; c < dqk; ++c) dC[(size_t)r * dqk + c] += dht[r] * q[ti * dqk + c] / N;
                for (int c = 0; c < dqk; ++c) dn[c] -= qCdh / (N * N) * omega * q[ti * dqk + c];
                /* (64) */
                for (int c = 0; c < dqk; ++c) {
                    double acc = 0.0;
                    for (int r = 0; r < dv; ++r) acc += Ct[(size_t)r * dqk + c] * dht[r];
                    dq[ti * dqk + c] = acc / N - qCdh / (N * N) * omega * nt[c];
                }
                /* (62), (63) with the s of the key */
                for (int r = 0; r < dv; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < dqk; ++c) acc += dC[(size_t)r * dqk + c] * s * k[ti * dqk + c];
                    dvv[ti * dv + r] = i * acc;
                }
                for (int c = 0; c < dqk; ++c) {
                    double acc = 0.0;
                    for (int r = 0; r < dv; ++r) acc += v[ti * dv + r] * dC[(size_t)r * dqk + c];
                    dk[ti * dqk + c] = s * i * (acc + dn[c]);
                }
                /* (68), (69) */
                double sf = 0.0, si = 0.0;
                for (int r = 0; r < dv; ++r)
                    for (int c = 0; c < dqk; ++c) {
                        sf += Cp[(size_t)r * dqk + c] * dC[(size_t)r * dqk + c];
                        si += v[ti * dv + r] * s * k[ti * dqk + c] * dC[(size_t)r * dqk + c];
                    }
                for (int c = 0; c < dqk; ++c) {
                    sf += np[c] * dn[c];
                    si += s * k[ti * dqk + c] * dn[c];
                }
                const double x = fg[ti];
#if ORACLE_MUTATION == 14
                const double gamma = g_forget_exp ? exp(x) : sigmoid(x);   /* mutation: sigma for sigma' */
#else
                const double gamma = g_forget_exp ? exp(x) : sigmoid(x) * (1.0 - sigmoid(x));
#endif
                dfg[ti] = sf * gamma;
                dig[ti] = si * i;
                /* carry to step t-1: multiply by f_t (60)-(61) */
                const double f = exp(log_forget(fg[ti]));
                for (size_t e = 0; e < CS; ++e) dC[e] *= f;
                for (int c = 0; c < dqk; ++c) dn[c] *= f;
            }
        }
        free(Cs);
        free(ns);
        free(dC);
        free(dn);
        free(dht);
        free(ht);
    }
    return fail ? -2 : 0;
}
