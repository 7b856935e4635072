/*
 * Float64 reverse mode of the gated delta-rule recurrence -- TEST INFRASTRUCTURE.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this code.  It shares nothing with the CUDA library.
 *
 * The forward is the token loop of recurrence.c (page "Diagonal Plus Low
 * Rank", section 2, opening equation):
 *
 *     Sa_t = S_{t-1} Diag(alpha_t),   y_t = Sa_t b_t,
 *     S_t  = Sa_t - y_t a_t^T + vv_t k_t^T,   o_t = S_t q_t,   alpha_t = exp(g_t).
 *
 * Its adjoint is taken step by step in reverse, for the loss
 * L = sum_t <do_t, o_t> + <dht, S_{T-1}>, with dS the gradient with respect
 * to S_t:
 *
 *     dS   += do_t q_t^T                 dq_t  = S_t^T do_t
 *     dvv_t = dS k_t                     dk_t += dS^T vv_t
 *     dy    = -dS a_t                    da_t  = -dS^T y_t
 *     dSa   = dS + dy b_t^T              db_t  = Sa_t^T dy
 *     dalpha_t[j] = sum_i dSa[i][j] S_{t-1}[i][j],   dg_t = alpha_t * dalpha_t
 *     dS_{t-1} = dSa Diag(alpha_t)
 *
 * (the per-step form of the gate gradient that page "Gated Linear Attention"
 * writes for its decayed state, dG_t = dS_t * S_{t-1} summed over the value
 * rows).  The KDA mapping a = k, b = beta k, vv = beta v is then folded back:
 * dk += da + beta db, dbeta = <db, k> + <dvv, v> (the latter only when beta
 * scales v), dv = beta dvv (or dvv).  A scalar gate sums dg over the channels.
 *
 * States are checkpointed at the start of every segment of SEG tokens and
 * recomputed forward inside the segment during the reverse sweep.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { BWD_GATE_NONE = 0, BWD_GATE_SCALAR = 1, BWD_GATE_CHANNEL = 2 };
enum { SEG = 64 };

typedef struct {
    int dk, dv, gate_kind, scale_v;
    const double *q, *k, *v, *g, *a, *b, *beta;
    long s_qk, s_v, s_g, s_ab, s_beta;
} bwd_in;

static void step_inputs(const bwd_in *in, int t, double *alpha, double *at, double *bt, double *vv)
{
    const double *kt = in->k + (long)t * in->s_qk;
    const double *vt = in->v + (long)t * in->s_v;
    const double beta_t = in->beta ? in->beta[(long)t * in->s_beta] : 0.0;
    for (int j = 0; j < in->dk; ++j) {
        double gj = 0.0;
        if (in->gate_kind == BWD_GATE_SCALAR) gj = in->g[(long)t * in->s_g];
        else if (in->gate_kind == BWD_GATE_CHANNEL) gj = in->g[(long)t * in->s_g + j];
        alpha[j] = exp(gj);
        at[j] = in->a ? in->a[(long)t * in->s_ab + j] : kt[j];
        bt[j] = in->b ? in->b[(long)t * in->s_ab + j] : beta_t * kt[j];
    }
    for (int i = 0; i < in->dv; ++i)
        vv[i] = in->scale_v ? beta_t * vt[i] : vt[i];
}

/* S_next = S Diag(alpha) - (S Diag(alpha) b) a^T + vv k^T */
static void step_forward(const bwd_in *in, int t, const double *S, double *Snext,
                         double *alpha, double *at, double *bt, double *vv)
{
    const int dk = in->dk, dv = in->dv;
    const double *kt = in->k + (long)t * in->s_qk;
    step_inputs(in, t, alpha, at, bt, vv);
    for (int i = 0; i < dv; ++i) {
        double y = 0.0;
        for (int j = 0; j < dk; ++j) y += S[(long)i * dk + j] * alpha[j] * bt[j];
        for (int j = 0; j < dk; ++j)
            Snext[(long)i * dk + j] = S[(long)i * dk + j] * alpha[j] - y * at[j] + vv[i] * kt[j];
    }
}

/*
 * One (batch, head) sequence.  Inputs as oracle_recurrence_head (a, b NULL
 * select the KDA mapping); do_ [T][dv] at stride s_o; dht [dv][dk] or NULL.
 * Outputs (each may be NULL):
 *   dq, dk_ : [T][dk] at stride s_qk
 *   dv_     : [T][dv] at stride s_v
 *   dg      : layout of g (SCALAR: one value per token; CHANNEL: [T][dk])
 *   da, db  : [T][dk] at stride s_ab (only meaningful when a, b are given)
 *   dbeta   : [T] at stride s_beta (only meaningful when beta is given)
 *   dh0     : [dv][dk]
 * Returns 0, or -1 when scratch memory cannot be allocated.
 */
int oracle_recurrence_head_bwd(int T, int dk, int dv,
                               const double *q, const double *k, long s_qk,
                               const double *v, long s_v,
                               const double *g, long s_g, int gate_kind,
                               const double *a, const double *b, long s_ab,
                               const double *beta, long s_beta, int scale_v,
                               const double *h0,
                               const double *do_, long s_o, const double *dht,
                               double *dq, double *dk_, double *dv_, double *dg,
                               double *da, double *db, double *dbeta, double *dh0)
{
    const size_t nS = (size_t)dv * dk;
    const int nseg = (T + SEG - 1) / SEG;
    bwd_in in = {dk, dv, gate_kind, scale_v, q, k, v, g, a, b, beta, s_qk, s_v, s_g, s_ab, s_beta};
    double *ck = (double *)malloc(sizeof(double) * nS * (size_t)nseg);      /* S before each segment */
    double *st = (double *)malloc(sizeof(double) * nS * (size_t)(SEG + 1)); /* states inside a segment */
    double *dS = (double *)malloc(sizeof(double) * nS);
    double *dSa = (double *)malloc(sizeof(double) * nS);
    double *alpha = (double *)malloc(sizeof(double) * dk);
    double *at = (double *)malloc(sizeof(double) * dk);
    double *bt = (double *)malloc(sizeof(double) * dk);
    double *vv = (double *)malloc(sizeof(double) * dv);
    double *y = (double *)malloc(sizeof(double) * dv);
    double *dy = (double *)malloc(sizeof(double) * dv);
    double *dvv = (double *)malloc(sizeof(double) * dv);
    double *gk = (double *)malloc(sizeof(double) * dk);    /* dS^T vv  */
    double *ga = (double *)malloc(sizeof(double) * dk);    /* da       */
    double *gb = (double *)malloc(sizeof(double) * dk);    /* db       */
    double *gal = (double *)malloc(sizeof(double) * dk);   /* dalpha   */
    int rc = 0;
    if (!ck || !st || !dS || !dSa || !alpha || !at || !bt || !vv || !y || !dy || !dvv || !gk || !ga ||
        !gb || !gal) {
        rc = -1;
        goto done;
    }

    /* forward pass: checkpoints */
    if (h0) memcpy(st, h0, sizeof(double) * nS);
    else memset(st, 0, sizeof(double) * nS);
    for (int s = 0; s < nseg; ++s) {
        memcpy(ck + nS * s, st, sizeof(double) * nS);
        const int t1 = (s + 1) * SEG < T ? (s + 1) * SEG : T;
        for (int t = s * SEG; t < t1; ++t) {
            step_forward(&in, t, st, st + nS, alpha, at, bt, vv);
            memcpy(st, st + nS, sizeof(double) * nS);
        }
    }

    /* reverse sweep */
    if (dht) memcpy(dS, dht, sizeof(double) * nS);
    else memset(dS, 0, sizeof(double) * nS);
    for (int s = nseg - 1; s >= 0; --s) {
        const int t0 = s * SEG;
        const int t1 = (s + 1) * SEG < T ? (s + 1) * SEG : T;
        memcpy(st, ck + nS * s, sizeof(double) * nS);
        for (int t = t0; t < t1; ++t)   /* st[t - t0 + 1] = S_t */
            step_forward(&in, t, st + nS * (t - t0), st + nS * (t - t0 + 1), alpha, at, bt, vv);
        for (int t = t1 - 1; t >= t0; --t) {
            const double *Sprev = st + nS * (t - t0);
            const double *St = st + nS * (t - t0 + 1);
            const double *qt = q + (long)t * s_qk;
            const double *kt = k + (long)t * s_qk;
            const double *vt = v + (long)t * s_v;
            const double *dot = do_ + (long)t * s_o;
            const double beta_t = beta ? beta[(long)t * s_beta] : 0.0;
            step_inputs(&in, t, alpha, at, bt, vv);

            /* o_t = S_t q_t */
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) dS[(long)i * dk + j] += dot[i] * qt[j];
            if (dq) {
                double *dqt = dq + (long)t * s_qk;
                for (int j = 0; j < dk; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < dv; ++i) acc += St[(long)i * dk + j] * dot[i];
                    dqt[j] = acc;
                }
            }
            /* y = Sa b with Sa = S_{t-1} Diag(alpha) */
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += Sprev[(long)i * dk + j] * alpha[j] * bt[j];
                y[i] = acc;
            }
            /* S_t = Sa - y a^T + vv k^T */
            for (int i = 0; i < dv; ++i) {
                double acc_vv = 0.0, acc_y = 0.0;
                for (int j = 0; j < dk; ++j) {
                    acc_vv += dS[(long)i * dk + j] * kt[j];
                    acc_y += dS[(long)i * dk + j] * at[j];
                }
                dvv[i] = acc_vv;
                dy[i] = -acc_y;
            }
            for (int j = 0; j < dk; ++j) {
                double acc_k = 0.0, acc_a = 0.0;
                for (int i = 0; i < dv; ++i) {
                    acc_k += dS[(long)i * dk + j] * vv[i];
                    acc_a += dS[(long)i * dk + j] * y[i];
                }
                gk[j] = acc_k;
                ga[j] = -acc_a;
            }
            /* y = Sa b */
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) dSa[(long)i * dk + j] = dS[(long)i * dk + j] + dy[i] * bt[j];
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dv; ++i) acc += Sprev[(long)i * dk + j] * alpha[j] * dy[i];
                gb[j] = acc;
            }
            /* Sa = S_{t-1} Diag(alpha) */
            for (int j = 0; j < dk; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dv; ++i) acc += dSa[(long)i * dk + j] * Sprev[(long)i * dk + j];
                gal[j] = acc;
            }
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) dS[(long)i * dk + j] = dSa[(long)i * dk + j] * alpha[j];

            /* fold the parametrisation back onto the inputs */
            if (dg) {
                if (gate_kind == BWD_GATE_CHANNEL) {
                    for (int j = 0; j < dk; ++j) dg[(long)t * s_g + j] = alpha[j] * gal[j];
                } else if (gate_kind == BWD_GATE_SCALAR) {
                    double acc = 0.0;
                    for (int j = 0; j < dk; ++j) acc += alpha[j] * gal[j];
                    dg[(long)t * s_g] = acc;
                }
            }
            if (dk_) {
                double *dkt = dk_ + (long)t * s_qk;
                for (int j = 0; j < dk; ++j) {
                    double acc = gk[j];
                    if (!a) acc += ga[j];
                    if (!b) acc += beta_t * gb[j];
                    dkt[j] = acc;
                }
            }
            if (a && da)
                for (int j = 0; j < dk; ++j) da[(long)t * s_ab + j] = ga[j];
            if (b && db)
                for (int j = 0; j < dk; ++j) db[(long)t * s_ab + j] = gb[j];
            if (dv_) {
                double *dvt = dv_ + (long)t * s_v;
                for (int i = 0; i < dv; ++i) dvt[i] = scale_v ? beta_t * dvv[i] : dvv[i];
            }
            if (beta && dbeta) {
                double acc = 0.0;
                if (!b)
                    for (int j = 0; j < dk; ++j) acc += gb[j] * kt[j];
                if (scale_v)
                    for (int i = 0; i < dv; ++i) acc += dvv[i] * vt[i];
                dbeta[(long)t * s_beta] = acc;
            }
        }
    }
    if (dh0) memcpy(dh0, dS, sizeof(double) * nS);

done:
    free(ck); free(st); free(dS); free(dSa); free(alpha); free(at); free(bt); free(vv);
    free(y); free(dy); free(dvv); free(gk); free(ga); free(gb); free(gal);
    return rc;
}
