/*
 * Float64 CPU oracle for the gated delta-rule family -- TEST INFRASTRUCTURE.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this code.  It shares nothing with the CUDA library: no header, no
 * helper, no constant.  It is deliberately the plain definition, written
 * token by token, with no chunking, blocking or reordering.
 *
 * What it computes (page "Diagonal Plus Low Rank", section 2, the opening
 * equation of the gated DPLR recurrence):
 *
 *     S_t = S_{t-1} Diag(alpha_t) (I - b_t a_t^T) + vv_t k_t^T,   S in R^{dv x dk}
 *     o_t = S_t q_t
 *
 * with alpha_t = exp(g_t) (g is the log-decay; page "Gated Linear Attention"
 * section 6.3 writes the gate in log space) and S_{-1} = h0 (zero when absent;
 * the DPLR page writes S_{[-1]} = 0 below its chunk-state equation).
 *
 * The special cases are only different inputs to the same loop:
 *   KDA      a = k, b = beta k, vv = beta v  (DPLR page, "relation to KDA";
 *            page "How to make GDN2 more stable", eq. (1) with j = k)
 *   GDN      as KDA with one scalar decay per token   (same eq. (1), D = gamma I)
 *   DeltaNet as KDA with alpha = 1                    (DeltaNet page, section 4.1)
 *   GLA      b = 0, vv = v                            (GLA page, section 5.1)
 *   DPLR     a, b given, vv = v                       (DPLR page, section 2)
 *
 * Layout: every sequence tensor is addressed as base + t * stride + j, so a
 * caller can hand over one (batch, head) slice of a [B, T, H, d] array
 * without copying.  S, h0 and ht are row-major [dv][dk].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_GATE_NONE = 0, ORACLE_GATE_SCALAR = 1, ORACLE_GATE_CHANNEL = 2 };

/*
 * One (batch, head) sequence through the recurrence.
 *
 *   q, k  : [T][dk] at row stride s_qk
 *   v     : [T][dv] at row stride s_v
 *   g     : log-decay; gate_kind NONE -> unused, SCALAR -> g[t * s_g],
 *           CHANNEL -> g[t * s_g + j]
 *   a, b  : [T][dk] at row stride s_ab, or NULL.  NULL selects the KDA
 *           mapping a = k, b = beta * k.
 *   beta  : beta[t * s_beta], or NULL (beta = 0)
 *   scale_v : nonzero -> vv = beta * v, zero -> vv = v
 *   h0    : [dv][dk] or NULL
 *   o     : [T][dv] at row stride s_o (output)
 *   ht    : [dv][dk] (output) or NULL
 * Returns 0, or -1 when scratch memory cannot be allocated.
 */
int oracle_recurrence_head(int T, int dk, int dv,
                           const double *q, const double *k, long s_qk,
                           const double *v, long s_v,
                           const double *g, long s_g, int gate_kind,
                           const double *a, const double *b, long s_ab,
                           const double *beta, long s_beta, int scale_v,
                           const double *h0, double *o, long s_o, double *ht)
{
    double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
    double *bt = (double *)malloc(sizeof(double) * (size_t)dk);
    double *y = (double *)malloc(sizeof(double) * (size_t)dv);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !alpha || !bt || !y || !vv) {
        free(S); free(alpha); free(bt); free(y); free(vv);
        return -1;
    }
    if (h0)
        memcpy(S, h0, sizeof(double) * (size_t)dv * dk);
    else
        memset(S, 0, sizeof(double) * (size_t)dv * dk);

    for (int t = 0; t < T; ++t) {
        const double *qt = q + (long)t * s_qk;
        const double *kt = k + (long)t * s_qk;
        const double *vt = v + (long)t * s_v;
        const double *at = a ? a + (long)t * s_ab : kt;
        const double beta_t = beta ? beta[(long)t * s_beta] : 0.0;

        /* alpha_t = exp(g_t): per channel, one scalar, or 1 */
        for (int j = 0; j < dk; ++j) {
            double gj = 0.0;
            if (gate_kind == ORACLE_GATE_SCALAR) gj = g[(long)t * s_g];
            else if (gate_kind == ORACLE_GATE_CHANNEL) gj = g[(long)t * s_g + j];
            alpha[j] = exp(gj);
        }
        /* b_t: given, or beta_t k_t */
        for (int j = 0; j < dk; ++j)
            bt[j] = b ? b[(long)t * s_ab + j] : beta_t * kt[j];
        /* vv_t: beta_t v_t or v_t */
        for (int i = 0; i < dv; ++i)
            vv[i] = scale_v ? beta_t * vt[i] : vt[i];

        /* S <- S Diag(alpha_t) */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(long)i * dk + j] *= alpha[j];
        /* y = (S Diag(alpha_t)) b_t */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j)
                acc += S[(long)i * dk + j] * bt[j];
            y[i] = acc;
        }
        /* S <- S Diag(alpha_t) - y a_t^T + vv_t k_t^T */
        for (int i = 0; i < dv; ++i)
            for (int j = 0; j < dk; ++j)
                S[(long)i * dk + j] += -y[i] * at[j] + vv[i] * kt[j];
        /* o_t = S_t q_t */
        double *ot = o + (long)t * s_o;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j)
                acc += S[(long)i * dk + j] * qt[j];
            ot[i] = acc;
        }
    }
    if (ht)
        memcpy(ht, S, sizeof(double) * (size_t)dv * dk);
    free(S); free(alpha); free(bt); free(y); free(vv);
    return 0;
}
