/*
 * h3ref.c -- FP64 CPU oracle of the MiniMax-H3 attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the tests, the smoke check and the bench's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (plain definitions, evaluated in double precision from the
 * exact values of the bf16 / fp32 inputs, no blocking, no fusion):
 *
 *   1. q/k RMSNorm over each 128-wide head with one 128-element weight shared by
 *      all heads ("RL-Kernel PR #539, ws1_one_h3_block", Bindings table:
 *      q_norm/k_norm bound to a plain RMSNorm on the 128-wide heads, bitwise
 *      equal to nn.RMSNorm; Status: the 128-element attn.norm_q.weight gradient):
 *          n = x / sqrt(mean_c x_c^2 + eps),   z = n * w
 *   2. partial 3-axis multimodal RoPE driven by packed (t, h, w) position ids
 *      (same page, Bindings table row rope_q/rope_k, and the Tests section:
 *      "MM-RoPE rotates" a subset of the 128 channels).  Section a in {t, h, w}
 *      owns n_a consecutive channels starting at o_a = sum_{b<a} n_b; inside it,
 *      channel o_a + j pairs with o_a + j + n_a/2 (rotate-half), j < n_a/2, and the
 *      pair is rotated by the angle p_a * theta^(-2j/n_a).  Channels at or past
 *      sum_a n_a pass through unchanged.
 *   3. non-causal attention inside each packed sample (Bindings table row
 *      attention: DeterministicAttentionOp(causal=False); packed FL2VA layouts,
 *      What section):
 *          s_ij = scale * <q^_i, k^_j>  for i, j in the same sample,
 *          p_ij = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij),
 *          o_i  = sum_j p_ij v_j,   lse_i = log sum_j exp(s_ij).
 *   4. the gradients of L = sum_i <dO_i, o_i> with respect to q, k, v and the two
 *      norm weights (Results: "gradients of the block input ... and all 12 block
 *      parameters"; Status: the 128-element norm weight gradient), written as the
 *      chain rule through (3), (2) and (1), with the weight gradient also reported
 *      per sample.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 128

/* H3REF_PLANT selects a deliberate mistake for the pin tests' sensitivity check
 * (0 = the oracle as specified; only a test build defines another value). */
#ifndef H3REF_PLANT
#define H3REF_PLANT 0
#endif
#define PLANT(n) (H3REF_PLANT == (n))

typedef struct {
    int sections[3];  /* rotary channels of the t, h and w axes (each even)     */
    double theta;     /* RoPE base                                               */
    double eps;       /* RMSNorm epsilon (inside the square root)                */
    double scale;     /* softmax scale applied to q^.k^                          */
} h3ref_params;

/* ---------------------------------------------------------------- step 1+2 */

/* RMSNorm of one 128-vector: n = x / sqrt(mean(x^2) + eps); returns 1/sqrt(...). */
static double rmsnorm_row(const float *x, double eps, double *n)
{
    double ms = 0.0;
    for (int c = 0; c < D; ++c) ms += (double)x[c] * (double)x[c];
    if (!PLANT(5)) ms /= D;
    double r = PLANT(4) ? 1.0 / (sqrt(ms) + eps) : 1.0 / sqrt(ms + eps);
    for (int c = 0; c < D; ++c) n[c] = (double)x[c] * r;
    return r;
}

/* Rotates z in place by the token's angles; sign = +1 forward, -1 inverse. */
static void rope_row(double *z, const int pos[3], const h3ref_params *p, double sign)
{
    int off = 0;
    for (int a = 0; a < 3; ++a) {
        int n = p->sections[a], half = n / 2;
        for (int j = 0; j < half; ++j) {
            double freq = pow(p->theta, (PLANT(3) ? -1.0 : -2.0) * j / (double)n);
            double ang = sign * (double)pos[a] * freq;
            if (PLANT(1) && sign > 0) ang = -ang;
            if (PLANT(10) && sign < 0) ang = -ang;
            double c = cos(ang), s = sin(ang);
            int i0 = PLANT(2) ? off + 2 * j : off + j;
            int i1 = PLANT(2) ? off + 2 * j + 1 : off + j + half;
            double u = z[i0], v = z[i1];
            z[i0] = u * c - v * s;
            z[i1] = u * s + v * c;
        }
        off += n;
    }
}

/*
 * Prologue for one [S, H, 128] tensor: y = RoPE(RMSNorm(x) * w).
 * Also returns n (normalised, before the weight) and r = 1/sqrt(mean x^2 + eps),
 * both needed by the backward.  n and r may be NULL.
 */
void h3ref_norm_rope(const float *x, int S, int H, const float *w,
                     const int32_t *pos_t, const int32_t *pos_h, const int32_t *pos_w,
                     const h3ref_params *p, double *y, double *n_out, double *r_out)
{
    #pragma omp parallel for schedule(static)
    for (long row = 0; row < (long)S * H; ++row) {
        long i = row / H;
        double n[D];
        double r = rmsnorm_row(x + row * D, p->eps, n);
        double *z = y + row * D;
        for (int c = 0; c < D; ++c) z[c] = n[c] * (double)w[c];
        int pos[3] = {pos_t[i], pos_h[i], pos_w[i]};
        rope_row(z, pos, p, +1.0);
        if (n_out) memcpy(n_out + row * D, n, sizeof n);
        if (r_out) r_out[row] = r;
    }
}

/* ------------------------------------------------------------------- step 3 */

static double dot128(const double *a, const double *b)
{
    double s = 0.0;
    for (int c = 0; c < D; ++c) s += a[c] * b[c];
    return s;
}

/* Sample index of every token from the segment offsets. */
static void token_sample(const int32_t *seg, int nseg, int *tok_sample)
{
    for (int s = 0; s < nseg; ++s)
        for (int i = seg[s]; i < seg[s + 1]; ++i) tok_sample[i] = s;
}

/*
 * Attention of pre-rotated q^, k^ (double) and v (float, exact bf16 values).
 * out [S, H, 128], lse [H, S].  Only query rows with row_mask[i] != 0 are
 * computed when row_mask is non-NULL; only heads in [h_lo, h_hi) are computed.
 */
void h3ref_attention(const double *yq, const double *yk, const float *v,
                     int S, int H, const int32_t *seg, int nseg, double scale,
                     int h_lo, int h_hi, const uint8_t *row_mask,
                     double *out, double *lse)
{
    int *ts = (int *)malloc(sizeof(int) * (S > 0 ? S : 1));
    token_sample(seg, nseg, ts);
    #pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
        #pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = h_lo; h < h_hi; ++h)
            for (int i = 0; i < S; ++i) {
                if (row_mask && !row_mask[i]) continue;
                int a = seg[ts[i]], b = seg[ts[i] + 1];
                if (PLANT(7) && b < S) b += 1;
                const double *qi = yq + ((long)i * H + h) * D;
                double m = -INFINITY;
                for (int j = a; j < b; ++j) {
                    sc[j - a] = (PLANT(6) ? 1.0 : scale) * dot128(qi, yk + ((long)j * H + h) * D);
                    if (sc[j - a] > m) m = sc[j - a];
                }
                double l = 0.0;
                for (int j = a; j < b; ++j) l += exp(sc[j - a] - m);
                double o[D] = {0};
                for (int j = a; j < b; ++j) {
                    double pij = exp(sc[j - a] - m) / l;
                    const float *vj = v + ((long)j * H + h) * D;
                    for (int c = 0; c < D; ++c) o[c] += pij * (double)vj[c];
                }
                memcpy(out + ((long)i * H + h) * D, o, sizeof o);
                if (lse) lse[(long)h * S + i] = m + log(l);
            }
        free(sc);
    }
    free(ts);
}

/* Full forward: prologue of q and k, then attention.  lse may be NULL. */
int h3ref_forward(const float *q, const float *k, const float *v,
                  const float *wq, const float *wk,
                  const int32_t *pos_t, const int32_t *pos_h, const int32_t *pos_w,
                  const int32_t *seg, int nseg, int S, int H, const h3ref_params *p,
                  int h_lo, int h_hi, const uint8_t *row_mask,
                  double *out, double *lse)
{
    size_t n = (size_t)S * H * D;
    double *yq = (double *)malloc(sizeof(double) * (n ? n : 1));
    double *yk = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (!yq || !yk) { free(yq); free(yk); return 1; }
    h3ref_norm_rope(q, S, H, wq, pos_t, pos_h, pos_w, p, yq, NULL, NULL);
    h3ref_norm_rope(k, S, H, wk, pos_t, pos_h, pos_w, p, yk, NULL, NULL);
    h3ref_attention(yq, yk, v, S, H, seg, nseg, p->scale, h_lo, h_hi, row_mask, out, lse);
    free(yq);
    free(yk);
    return 0;
}

/* ------------------------------------------------------------------- step 4 */

/*
 * Backward of the prologue for one row: given dy (gradient at the rotated
 * output), the token's positions, n = x*r and r, returns dx and adds g*n to dw
 * (g = gradient at z = n*w):
 *     g  = R(-angle) dy,   dn = g * w,
 *     dx = r * (dn - n * mean_c(dn_c n_c)),   dw += g * n.
 */
static void norm_rope_bwd_row(const double *dy, const int pos[3], const double *n, double r,
                              const float *w, const h3ref_params *p, double *dx, double *dw)
{
    double g[D];
    memcpy(g, dy, sizeof g);
    rope_row(g, pos, p, -1.0);
    double dn[D], mean_dn_n = 0.0;
    for (int c = 0; c < D; ++c) {
        dn[c] = g[c] * (double)w[c];
        mean_dn_n += dn[c] * n[c];
        dw[c] += g[c] * n[c] * (PLANT(8) ? (double)w[c] : 1.0);
    }
    mean_dn_n = PLANT(9) ? 0.0 : mean_dn_n / D;
    for (int c = 0; c < D; ++c) dx[c] = r * (dn[c] - n[c] * mean_dn_n);
}

/*
 * Full backward.  Outputs (all double): dq, dk, dv [S, H, 128]; dwq, dwk [128]
 * (sum over all tokens and heads); dwq_s, dwk_s [nseg, 128] per-sample sums
 * (may be NULL).  Heads outside [h_lo, h_hi) are skipped: their dq/dk/dv rows
 * are left untouched and they do not contribute to the weight gradients.
 *
 * Attention part, per sample and head (p from the recomputed forward):
 *     dv_j = sum_i p_ij dO_i,           dp_ij = <dO_i, v_j>,
 *     ds_ij = p_ij (dp_ij - sum_k p_ik dp_ik),
 *     dq^_i = scale sum_j ds_ij k^_j,   dk^_j = scale sum_i ds_ij q^_i.
 * Rows (i) are computed in one parallel loop, columns (j) in a second one,
 * reusing lse_i and the softmax-Jacobian row term from the first.
 */
int h3ref_backward(const float *q, const float *k, const float *v,
                   const float *wq, const float *wk,
                   const int32_t *pos_t, const int32_t *pos_h, const int32_t *pos_w,
                   const int32_t *seg, int nseg, int S, int H, const h3ref_params *p,
                   const float *dout, int h_lo, int h_hi,
                   double *dq, double *dk, double *dv, double *dwq, double *dwk,
                   double *dwq_s, double *dwk_s)
{
    size_t n = (size_t)S * H * D;
    size_t nb = sizeof(double) * (n ? n : 1);
    double *yq = malloc(nb), *yk = malloc(nb), *nq = malloc(nb), *nk = malloc(nb);
    double *dyq = malloc(nb), *dyk = malloc(nb);
    double *rq = malloc(sizeof(double) * ((size_t)S * H + 1));
    double *rk = malloc(sizeof(double) * ((size_t)S * H + 1));
    double *lse = malloc(sizeof(double) * ((size_t)S * H + 1));
    double *Dt = malloc(sizeof(double) * ((size_t)S * H + 1));
    int *ts = malloc(sizeof(int) * (S + 1));
    if (!yq || !yk || !nq || !nk || !dyq || !dyk || !rq || !rk || !lse || !Dt || !ts) return 1;
    token_sample(seg, nseg, ts);
    h3ref_norm_rope(q, S, H, wq, pos_t, pos_h, pos_w, p, yq, nq, rq);
    h3ref_norm_rope(k, S, H, wk, pos_t, pos_h, pos_w, p, yk, nk, rk);
    const double scale = p->scale;

    #pragma omp parallel
    {
        double *sc = malloc(sizeof(double) * (S + 1));
        double *dp = malloc(sizeof(double) * (S + 1));
        /* rows: lse_i, the row term sum_j p_ij dp_ij, and dq^_i */
        #pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = h_lo; h < h_hi; ++h)
            for (int i = 0; i < S; ++i) {
                int a = seg[ts[i]], b = seg[ts[i] + 1];
                const double *qi = yq + ((long)i * H + h) * D;
                const float *doi = dout + ((long)i * H + h) * D;
                double m = -INFINITY;
                for (int j = a; j < b; ++j) {
                    sc[j - a] = scale * dot128(qi, yk + ((long)j * H + h) * D);
                    if (sc[j - a] > m) m = sc[j - a];
                }
                double l = 0.0;
                for (int j = a; j < b; ++j) l += exp(sc[j - a] - m);
                double L = m + log(l), rowterm = 0.0;
                for (int j = a; j < b; ++j) {
                    const float *vj = v + ((long)j * H + h) * D;
                    double d = 0.0;
                    for (int c = 0; c < D; ++c) d += (double)doi[c] * (double)vj[c];
                    dp[j - a] = d;
                    rowterm += exp(sc[j - a] - L) * d;
                }
                double g[D] = {0};
                for (int j = a; j < b; ++j) {
                    double ds = exp(sc[j - a] - L) * (dp[j - a] - (PLANT(11) ? 0.0 : rowterm));
                    const double *kj = yk + ((long)j * H + h) * D;
                    for (int c = 0; c < D; ++c) g[c] += ds * kj[c];
                }
                for (int c = 0; c < D; ++c) dyq[((long)i * H + h) * D + c] = scale * g[c];
                lse[(long)h * S + i] = L;
                Dt[(long)h * S + i] = rowterm;
            }
        /* columns: dv_j and dk^_j */
        #pragma omp for collapse(2) schedule(dynamic, 16)
        for (int h = h_lo; h < h_hi; ++h)
            for (int j = 0; j < S; ++j) {
                int a = seg[ts[j]], b = seg[ts[j] + 1];
                const double *kj = yk + ((long)j * H + h) * D;
                const float *vj = v + ((long)j * H + h) * D;
                double gv[D] = {0}, gk[D] = {0};
                for (int i = a; i < b; ++i) {
                    const double *qi = yq + ((long)i * H + h) * D;
                    const float *doi = dout + ((long)i * H + h) * D;
                    double pij = exp(scale * dot128(qi, kj) - lse[(long)h * S + i]);
                    double d = 0.0;
                    for (int c = 0; c < D; ++c) d += (double)doi[c] * (double)vj[c];
                    double ds = pij * (d - (PLANT(11) ? 0.0 : Dt[(long)h * S + i]));
                    for (int c = 0; c < D; ++c) {
                        gv[c] += pij * (double)doi[c];
                        gk[c] += ds * qi[c];
                    }
                }
                for (int c = 0; c < D; ++c) {
                    dv[((long)j * H + h) * D + c] = gv[c];
                    dyk[((long)j * H + h) * D + c] = scale * gk[c];
                }
            }
        free(sc);
        free(dp);
    }

    /* prologue backward, weight gradients summed per sample, then over samples */
    double *dwq_loc = calloc((size_t)nseg * D + 1, sizeof(double));
    double *dwk_loc = calloc((size_t)nseg * D + 1, sizeof(double));
    for (int s = 0; s < nseg; ++s)
        for (int i = seg[s]; i < seg[s + 1]; ++i) {
            int pos[3] = {pos_t[i], pos_h[i], pos_w[i]};
            for (int h = h_lo; h < h_hi; ++h) {
                long row = (long)i * H + h;
                norm_rope_bwd_row(dyq + row * D, pos, nq + row * D, rq[row], wq, p,
                                  dq + row * D, dwq_loc + (size_t)s * D);
                norm_rope_bwd_row(dyk + row * D, pos, nk + row * D, rk[row], wk, p,
                                  dk + row * D, dwk_loc + (size_t)s * D);
            }
        }
    for (int c = 0; c < D; ++c) {
        dwq[c] = 0.0;
        dwk[c] = 0.0;
        for (int s = 0; s < nseg; ++s) {
            dwq[c] += dwq_loc[(size_t)s * D + c];
            dwk[c] += dwk_loc[(size_t)s * D + c];
        }
    }
    if (dwq_s) memcpy(dwq_s, dwq_loc, sizeof(double) * nseg * D);
    if (dwk_s) memcpy(dwk_s, dwk_loc, sizeof(double) * nseg * D);
    free(dwq_loc); free(dwk_loc);
    free(yq); free(yk); free(nq); free(nk); free(dyq); free(dyk);
    free(rq); free(rk); free(lse); free(Dt); free(ts);
    return 0;
}

/* Number of OpenMP threads the oracle runs with. */
int h3ref_num_threads(void)
{
    int n = 1;
    #pragma omp parallel
    {
        #pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
