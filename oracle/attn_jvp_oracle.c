/*
 * FP64 CPU oracle for the forward-mode JVP through softmax attention and for
 * the TrigFlow helpers.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * Sources (all on the page "带分数正则的一致性蒸馏" — consistency distillation
 * with score regularisation — a gitcode.csdn.net write-up of rCM/sCM):
 *   - section 注意力 (attention), "naive_scaled_dot_product_attention":
 *       O = softmax(s * Q K^T) V, softmax along the key axis.
 *   - section 注意力, the JVP paragraph: by the chain rule
 *       t_o = P t_v + t_p V,  t_p = P (.) t_s - (P t_s^T) P,  t_s = t_q K^T + Q t_k^T
 *     (the prose drops the scale; the kernel listing in section 前向 (forward)
 *     multiplies t_s by sm_scale, the derivative of s * Q K^T, and so do we).
 *   - section 前向 (forward): the LSE output is the natural-log log-sum-exp
 *     of the scaled scores, one float per query row.
 *   - section 时间步转换 (timestep conversion): the RectifiedFlow_TrigFlowWrapper
 *     coefficients and the TrigFlow forward process x_t = cos t x0 + sin t eps.
 *   - section 一致性模型 (consistency model), its 蒸馏代码 listing: the JVP of
 *     the wrapper coefficients and of _process_output, the tangent target g
 *     with its warm-up, NaN masks and normalisation, and the sCM loss.
 *   - section 反向 (backward): dV = P^T dO, dP = dO V^T,
 *     dS = P (.) (dP - rowsum(dP (.) P)), dQ = s dS K, dK = s dS^T Q.
 *   - section 一致性模型 (consistency model): the student keeps its QK
 *     normalisation (QK正则化), so the tangents of Q and K pass through it
 *     before the attention.  The norm itself is defined on the page
 *     "Обслуживание Ideogram v4 менее чем за секунду" (dev48.org), section on
 *     fusing RMSNorm: per head, y = x rsqrt(mean(x^2) + eps) weight.  Its
 *     tangent is the chain rule on that definition.
 *
 * Every step below is the plain definition, computed in the order written on
 * the page: two passes over the keys for the softmax (max, then exponentials),
 * then the value sums.  No blocking, no online rescaling, no fusion.
 *
 * Parity pins (tests/test_oracle.py): library SDPA and logsumexp in FP64,
 * central finite differences of O and LSE, torch.func.jvp autodiff, linearity,
 * zero tangents, constant-V rows, one-key and two-key closed forms, the
 * mu shift identity, and for TrigFlow the values printed on the page.
 * The output-side functions (tests/test_epilogue_oracle.py): finite
 * differences, torch.func.jvp of the page's _process_output, the TrigFlow
 * velocity of a perfect network, and closed forms of each term of the
 * tangent target, of its normalisation, of the loss and of the NaN masks.
 * The backward (tests/test_bwd_oracle.py): torch.autograd, a central
 * difference of <O, dO>, one key, key-shift invariance, and the rowsum
 * identity rowsum(dP (.) P) = rowsum(dO (.) O).
 * The QK normalisation (tests/test_rmsnorm_oracle.py): central differences,
 * torch.func.jvp of the torch expression, scale invariance at eps = 0, unit
 * RMS, the tangent orthogonal to x, and attention through the norm against
 * torch.func.jvp of the whole composition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Attention + JVP, one head, arbitrary query rows                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    const double *q, *qt;           /* [R, d]   query rows and their tangents  */
    const double *k, *kt;           /* [Nk, d]  keys and their tangents        */
    const double *v, *vt;           /* [Nk, dv] values and their tangents      */
    int64_t R, Nk, d, dv;
    double scale;
    double *o, *ot, *lse, *mu;      /* [R, dv], [R, dv], [R], [R]              */
    int64_t row_begin, row_end;
    int status;
} head_job;

static void one_row(const head_job *J, int64_t i, double *S, double *St, double *P)
{
    const int64_t d = J->d, dv = J->dv, Nk = J->Nk;
    const double *qi = J->q + i * d, *qti = J->qt + i * d;

    /* Step 1: scores S_ij = s * q_i . k_j and their tangents
     *         St_ij = s * (qt_i . k_j + q_i . kt_j).                         */
    for (int64_t j = 0; j < Nk; ++j) {
        const double *kj = J->k + j * d, *ktj = J->kt + j * d;
        double a = 0.0, b = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            a += qi[c] * kj[c];
            b += qti[c] * kj[c] + qi[c] * ktj[c];
        }
        S[j] = J->scale * a;
        St[j] = J->scale * b;
    }

    /* Step 2: softmax along the keys, max first for the exponentials.       */
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; ++j)
        if (S[j] > m) m = S[j];
    double l = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        P[j] = exp(S[j] - m);
        l += P[j];
    }
    for (int64_t j = 0; j < Nk; ++j) P[j] /= l;

    /* Step 3: O_i = sum_j P_ij v_j and LSE_i = ln sum_j exp(S_ij).          */
    double *oi = J->o + i * dv;
    for (int64_t c = 0; c < dv; ++c) oi[c] = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        const double *vj = J->v + j * dv;
        for (int64_t c = 0; c < dv; ++c) oi[c] += P[j] * vj[c];
    }
    J->lse[i] = m + log(l);

    /* Step 4: mu_i = sum_j P_ij St_ij (the row sum of P (.) t_s), then the
     * tangent  t_o = P t_v + t_p V  with  t_p_ij = P_ij (St_ij - mu_i).      */
    double mu = 0.0;
    for (int64_t j = 0; j < Nk; ++j) mu += P[j] * St[j];
    J->mu[i] = mu;
    double *oti = J->ot + i * dv;
    for (int64_t c = 0; c < dv; ++c) oti[c] = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        const double *vj = J->v + j * dv, *vtj = J->vt + j * dv;
        const double tp = P[j] * (St[j] - mu);
        for (int64_t c = 0; c < dv; ++c) oti[c] += P[j] * vtj[c] + tp * vj[c];
    }
}

static void *head_worker(void *arg)
{
    head_job *J = (head_job *)arg;
    double *buf = (double *)malloc(sizeof(double) * 3 * (size_t)J->Nk);
    if (!buf) { J->status = -1; return NULL; }
    for (int64_t i = J->row_begin; i < J->row_end; ++i)
        one_row(J, i, buf, buf + J->Nk, buf + 2 * J->Nk);
    free(buf);
    J->status = 0;
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments or allocation failure. */
int oracle_attn_jvp_rows(const double *q, const double *qt,
                         const double *k, const double *kt,
                         const double *v, const double *vt,
                         int64_t R, int64_t Nk, int64_t d, int64_t dv, double scale,
                         double *o, double *ot, double *lse, double *mu,
                         int nthreads)
{
    if (!q || !qt || !k || !kt || !v || !vt || !o || !ot || !lse || !mu) return -1;
    if (R < 0 || Nk < 1 || d < 1 || dv < 1) return -1;
    if (R == 0) return 0;
    if (nthreads < 1) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > R) nthreads = (int)R;

    head_job *jobs = (head_job *)calloc((size_t)nthreads, sizeof(head_job));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *started = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tid || !started) { free(jobs); free(tid); free(started); return -1; }
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        head_job *J = &jobs[t];
        J->q = q; J->qt = qt; J->k = k; J->kt = kt; J->v = v; J->vt = vt;
        J->R = R; J->Nk = Nk; J->d = d; J->dv = dv; J->scale = scale;
        J->o = o; J->ot = ot; J->lse = lse; J->mu = mu;
        J->row_begin = R * t / nthreads;
        J->row_end = R * (t + 1) / nthreads;
        J->status = -1;
        if (pthread_create(&tid[t], NULL, head_worker, J) == 0)
            started[t] = 1;
        else
            head_worker(J);   /* no thread available: run the slice here */
    }
    for (int t = 0; t < nthreads; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status != 0) rc = -1;
    }
    free(jobs);
    free(tid);
    free(started);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Exact merge of key-chunk partial results                                 */
/* ------------------------------------------------------------------------ */
/*
 * The pages do not describe a key split; this is exact algebra on the
 * definitions above.  For chunk c with partial softmax normaliser l_c:
 *   O_c = sum_{j in c} e^{S_j} v_j / l_c,   mu_c = sum_{j in c} e^{S_j} St_j / l_c,
 *   Ot_c = sum_{j in c} e^{S_j} (St_j v_j + vt_j) / l_c - mu_c O_c,
 *   LSE_c = ln l_c  (up to the common max, which cancels).
 * With l = sum_c l_c the full-row weights are w_c = l_c / l = e^{LSE_c - LSE},
 * LSE = ln sum_c e^{LSE_c}, and
 *   O = sum_c w_c O_c,  mu = sum_c w_c mu_c,  Ot = sum_c w_c (Ot_c + mu_c O_c) - mu O.
 * Layout: partials [C, rows, d] and [C, rows]; outputs [rows, d] and [rows].
 */
int oracle_merge_chunks(const double *o_c, const double *ot_c,
                        const double *lse_c, const double *mu_c,
                        int64_t C, int64_t rows, int64_t d,
                        double *o, double *ot, double *lse, double *mu)
{
    if (!o_c || !ot_c || !lse_c || !mu_c || !o || !ot || !lse || !mu) return -1;
    if (C < 1 || rows < 0 || d < 1) return -1;
    for (int64_t i = 0; i < rows; ++i) {
        double m = -INFINITY;
        for (int64_t c = 0; c < C; ++c)
            if (lse_c[c * rows + i] > m) m = lse_c[c * rows + i];
        double l = 0.0;
        for (int64_t c = 0; c < C; ++c) l += exp(lse_c[c * rows + i] - m);
        const double L = m + log(l);
        lse[i] = L;
        double mui = 0.0;
        for (int64_t c = 0; c < C; ++c)
            mui += exp(lse_c[c * rows + i] - L) * mu_c[c * rows + i];
        mu[i] = mui;
        for (int64_t e = 0; e < d; ++e) {
            double oe = 0.0, te = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                const double w = exp(lse_c[c * rows + i] - L);
                const double oce = o_c[(c * rows + i) * d + e];
                oe += w * oce;
                te += w * (ot_c[(c * rows + i) * d + e] + mu_c[c * rows + i] * oce);
            }
            o[i * d + e] = oe;
            ot[i * d + e] = te - mui * oe;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* TrigFlow helpers (section 时间步转换, timestep conversion)                */
/* ------------------------------------------------------------------------ */
/*
 * RectifiedFlow_TrigFlowWrapper, sigma_data = 1: for a TrigFlow time t,
 *   c_skip = 1 / (cos t + sin t)
 *   c_out  = -sin t / (cos t + sin t)
 *   c_in   = 1 / (cos t + sin t)
 *   c_noise = tau * sin t / (cos t + sin t)     (tau = t_scaling_factor)
 * out = {c_skip, c_out, c_in, c_noise}.  Returns -1 where cos t + sin t <= 0.
 */
int oracle_trigflow_coeffs(double t, double tau, double *out)
{
    if (!out) return -1;
    const double c = cos(t), s = sin(t);
    const double den = c + s;
    if (!(den > 0.0)) return -1;
    out[0] = 1.0 / den;
    out[1] = -s / den;
    out[2] = 1.0 / den;
    out[3] = tau * s / den;
    return 0;
}

/*
 * Time derivative of the TrigFlow forward process x_t = cos t x0 + sin t eps:
 *   dx_t/dt = -sin t x0 + cos t eps,  t given per sample b, x0/eps [B, M].
 */
int oracle_trigflow_tangent(const double *x0, const double *eps, const double *t,
                            int64_t B, int64_t M, double *out)
{
    if (!x0 || !eps || !t || !out || B < 0 || M < 0) return -1;
    for (int64_t b = 0; b < B; ++b) {
        const double s = sin(t[b]), c = cos(t[b]);
        for (int64_t i = 0; i < M; ++i)
            out[b * M + i] = -s * x0[b * M + i] + c * eps[b * M + i];
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Output side of one consistency step (section 一致性模型, consistency      */
/* model, its 蒸馏代码 listing: student_F_withT, _process_output, the tangent */
/* target g, its NaN masks and normalisation, and the sCM loss).             */
/* Tensors are [B, C, T, HW] (the page's B_C_T_H_W with H and W merged); the  */
/* time t and its tangent are given per (b, frame) as [B, T].                */
/* ------------------------------------------------------------------------ */

/*
 * The wrapper coefficients and their tangents (the page's
 * torch.func.jvp(self.scaling, (t,), (v,))):
 *   out[0..3] = c_skip, c_out, c_in, c_noise at t;
 *   out[4..7] = v * d/dt of each.
 * With D = cos t + sin t: c_skip = c_in = 1/D, c_out = -sin t / D,
 * c_noise = tau sin t / D, so d(1/D)/dt = -(cos t - sin t) / D^2,
 * d(-sin t / D)/dt = -(cos t D - sin t (cos t - sin t)) / D^2 = -1 / D^2 and
 * d(tau sin t / D)/dt = tau / D^2.
 */
int oracle_trigflow_coeffs_jvp(double t, double v, double tau, double *out)
{
    if (!out) return -1;
    const double c = cos(t), s = sin(t);
    const double den = c + s;
    if (!(den > 0.0)) return -1;
    const double den2 = den * den;
    out[0] = 1.0 / den;
    out[1] = -s / den;
    out[2] = 1.0 / den;
    out[3] = tau * s / den;
    out[4] = v * (-(c - s) / den2);
    out[5] = v * (-1.0 / den2);
    out[6] = v * (-(c - s) / den2);
    out[7] = v * (tau / den2);
    return 0;
}

/*
 * _process_output and its JVP, elementwise:
 *   x0 = c_skip x + c_out n,   F = (cos t x - x0) / sin t,
 * differentiated along (t_x, t_n, t_c_skip, t_c_out, t_t) where the
 * coefficient tangents come from oracle_trigflow_coeffs_jvp(t, t_t):
 *   t_x0 = t_c_skip x + c_skip t_x + t_c_out n + c_out t_n
 *   t_F  = ((-sin t t_t x + cos t t_x - t_x0) sin t - (cos t x - x0) cos t t_t) / sin^2 t.
 * sin t must be non-zero for every (b, frame) (t in (0, pi/2]).
 */
int oracle_process_output_jvp(const double *x, const double *n, const double *tx, const double *tn,
                              const double *t, const double *tt, int64_t B, int64_t C, int64_t T,
                              int64_t HW, double *F, double *tF)
{
    if (!x || !n || !tx || !tn || !t || !tt || !F || !tF || B < 0 || C < 0 || T < 0 || HW < 0) return -1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t f = 0; f < T; ++f) {
            const double tm = t[b * T + f], vt = tt[b * T + f];
            double k[8];
            if (oracle_trigflow_coeffs_jvp(tm, vt, 1.0, k) != 0) return -1;
            const double c = cos(tm), s = sin(tm);
            if (s == 0.0) return -1;
            for (int64_t ch = 0; ch < C; ++ch) {
                const int64_t base = ((b * C + ch) * T + f) * HW;
                for (int64_t i = 0; i < HW; ++i) {
                    const int64_t e = base + i;
                    const double x0 = k[0] * x[e] + k[1] * n[e];
                    const double tx0 = k[4] * x[e] + k[0] * tx[e] + k[5] * n[e] + k[1] * tn[e];
                    const double num = c * x[e] - x0;
                    F[e] = num / s;
                    tF[e] = ((-s * vt * x[e] + c * tx[e] - tx0) * s - num * c * vt) / (s * s);
                }
            }
        }
    return 0;
}

/*
 * Tangent target, NaN masks, normalisation and the sCM loss, in the page's order:
 *   g     = -cos t sqrt(1 - r^2 sin^2 t) (F_sg - F_teacher) - (r cos t sin t x + t_F)
 *   df_dt = -cos t (F_sg - F_teacher) - (sin t x + t_F)                (not masked)
 *   nan_g[b] = any element of g[b] is NaN;  nan_F[b] = any element of F_theta[b] is NaN
 *   for a masked sample (nan_g or nan_F) g, F_theta and F_sg are taken as 0
 *   g_n   = g / (||g[b]||_2 + 0.1)
 *   loss[b] = sum over the sample of (F_theta - F_sg - g_n)^2
 * r is the warm-up ratio min(1, iteration / tangent_warmup).
 */
int oracle_scm_tangent_loss(const double *F_theta, const double *F_sg, const double *F_teacher,
                            const double *x, const double *tF, const double *t, double r, int64_t B,
                            int64_t C, int64_t T, int64_t HW, double *g_n, double *dfdt, double *loss,
                            int *nan_g, int *nan_F)
{
    if (!F_theta || !F_sg || !F_teacher || !x || !tF || !t || !g_n || !dfdt || !loss || !nan_g || !nan_F ||
        B < 0 || C < 0 || T < 0 || HW < 0)
        return -1;
    const int64_t per = C * T * HW;
    for (int64_t b = 0; b < B; ++b) {
        int ng = 0, nf = 0;
        /* g and df_dt */
        for (int64_t ch = 0; ch < C; ++ch)
            for (int64_t f = 0; f < T; ++f) {
                const double tm = t[b * T + f];
                const double c = cos(tm), s = sin(tm);
                const double w = sqrt(1.0 - r * r * s * s);
                const int64_t base = ((b * C + ch) * T + f) * HW;
                for (int64_t i = 0; i < HW; ++i) {
                    const int64_t e = base + i;
                    const double dF = F_sg[e] - F_teacher[e];
                    g_n[e] = -c * w * dF - (r * c * s * x[e] + tF[e]);
                    dfdt[e] = -c * dF - (s * x[e] + tF[e]);
                    if (isnan(g_n[e])) ng = 1;
                    if (isnan(F_theta[e])) nf = 1;
                }
            }
        nan_g[b] = ng;
        nan_F[b] = nf;
        const int masked = ng || nf;
        /* norm over the sample */
        double ss = 0.0;
        for (int64_t e = b * per; e < (b + 1) * per; ++e) {
            if (masked) g_n[e] = 0.0;
            ss += g_n[e] * g_n[e];
        }
        const double den = sqrt(ss) + 0.1;
        double l = 0.0;
        for (int64_t e = b * per; e < (b + 1) * per; ++e) {
            g_n[e] = g_n[e] / den;
            const double a = masked ? 0.0 : F_theta[e] - F_sg[e];
            const double d = a - g_n[e];
            l += d * d;
        }
        loss[b] = l;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Primal attention backward (section 反向, backward): given the upstream     */
/* gradient dO of O = P V with P = softmax(S), S = s Q K^T,                   */
/*   dV = P^T dO,  dP = dO V^T,  dS = P (.) (dP - rowsum(dP (.) P)),          */
/*   dQ = s dS K,  dK = s dS^T Q.                                             */
/* One head; q, dO [Nq, d]; k, v [Nk, d].  P is formed from S by the plain    */
/* two-pass softmax (the page's kernel reuses the forward's LSE instead; the  */
/* probabilities are the same).                                               */
/* ------------------------------------------------------------------------ */
int oracle_attn_bwd_head(const double *q, const double *k, const double *v, const double *dO, int64_t Nq,
                         int64_t Nk, int64_t d, double scale, double *dq, double *dk, double *dv)
{
    if (!q || !k || !v || !dO || !dq || !dk || !dv || Nq < 1 || Nk < 1 || d < 1) return -1;
    double *P = (double *)malloc(sizeof(double) * (size_t)(Nq * Nk));
    double *dS = (double *)malloc(sizeof(double) * (size_t)(Nq * Nk));
    if (!P || !dS) {
        free(P);
        free(dS);
        return -2;
    }
    for (int64_t i = 0; i < Nq; ++i) {
        double m = -INFINITY;
        for (int64_t j = 0; j < Nk; ++j) {
            double s = 0.0;
            for (int64_t c = 0; c < d; ++c) s += q[i * d + c] * k[j * d + c];
            P[i * Nk + j] = s * scale;
            if (P[i * Nk + j] > m) m = P[i * Nk + j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
            P[i * Nk + j] = exp(P[i * Nk + j] - m);
            l += P[i * Nk + j];
        }
        for (int64_t j = 0; j < Nk; ++j) P[i * Nk + j] /= l;
        /* dP_ij = dO_i . v_j, then dS = P (.) (dP - rowsum(dP (.) P)) */
        double rs = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
            double dp = 0.0;
            for (int64_t c = 0; c < d; ++c) dp += dO[i * d + c] * v[j * d + c];
            dS[i * Nk + j] = dp;
            rs += dp * P[i * Nk + j];
        }
        for (int64_t j = 0; j < Nk; ++j) dS[i * Nk + j] = P[i * Nk + j] * (dS[i * Nk + j] - rs);
    }
    for (int64_t i = 0; i < Nq; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < Nk; ++j) acc += dS[i * Nk + j] * k[j * d + c];
            dq[i * d + c] = scale * acc;
        }
    for (int64_t j = 0; j < Nk; ++j)
        for (int64_t c = 0; c < d; ++c) {
            double ak = 0.0, av = 0.0;
            for (int64_t i = 0; i < Nq; ++i) {
                ak += dS[i * Nk + j] * q[i * d + c];
                av += P[i * Nk + j] * dO[i * d + c];
            }
            dk[j * d + c] = scale * ak;
            dv[j * d + c] = av;
        }
    free(P);
    free(dS);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* QK normalisation (RMSNorm over each head's d channels) and its tangent    */
/* ------------------------------------------------------------------------ */

/* For each of ``rows`` rows of d values (one token of one head):
 *   m   = (1/d) sum_c x_c^2            rho = 1 / sqrt(m + eps)
 *   y_c = x_c rho w_c
 * and along the tangent xt (chain rule: d rho = -rho^3 (1/d) sum_c x_c xt_c):
 *   a    = (1/d) sum_c x_c xt_c
 *   yt_c = w_c (xt_c rho - x_c rho^3 a)
 * x, xt, y, yt: [rows, d]; w: [d] (the norm's per-channel weight).          */
int oracle_rmsnorm_jvp(const double *x, const double *xt, const double *w, int64_t rows, int64_t d,
                       double eps, double *y, double *yt)
{
    if (rows < 0 || d < 1 || !(eps >= 0.0)) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        const double *xr = x + r * d, *xtr = xt + r * d;
        double m = 0.0, a = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            m += xr[c] * xr[c];
            a += xr[c] * xtr[c];
        }
        m /= (double)d;
        a /= (double)d;
        if (!(m + eps > 0.0)) return -2;  /* an all-zero row with eps = 0 has no norm */
        const double rho = 1.0 / sqrt(m + eps);
        const double rho3 = rho * rho * rho;
        for (int64_t c = 0; c < d; ++c) {
            y[r * d + c] = xr[c] * rho * w[c];
            yt[r * d + c] = w[c] * (xtr[c] * rho - xr[c] * rho3 * a);
        }
    }
    return 0;
}
