/*
 * mhc_pre_bwd_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain double-precision CPU statement of the backward of the mHC
 * pre-mapping with Sinkhorn, used only to check the CUDA library.  Only the
 * tests and the benchmark's CPU-baseline leg may build, load or call it.  It
 * shares no code, header or constant with the CUDA path.
 *
 * Sources (page title, then the section followed):
 *  [BW]  "CANN ops-transformer 算子解析：MhcPreBackward 反向梯度算子实现与
 *        aclnn 调用指南", §一 (the outputs are the gradients of the forward),
 *        §三 3.1-3.8 (the eight stages, taken here in that order), §8.1
 *        (inputs, optional gamma and grad_x_post, hc_eps).
 *  [SK]  "CANN ops-transformer 算子详解：aclnnMhcPreSinkhorn 接口与
 *        MhcPreSinkhorn 实现剖析", §3.2 (the Sinkhorn recurrence whose saved
 *        sums and matrices sumOut / normOut are inputs here), §10 (the
 *        Sinkhorn variant's backward consumes grad_h_res of the Sinkhorn
 *        output together with sum_out and norm_out).
 *
 * Readings (each also listed in the design notes):
 *  - With sum_out / norm_out given, grad_h_res is the gradient of the
 *    Sinkhorn output and stage 0 below carries it back through the 2I
 *    normalisation steps and the softmax to the res logits; without them
 *    grad_h_res is already the gradient of the logits ([BW] §3.4 form).
 *    The pages print no formula for that stage: each step's derivative is
 *    written out from the step's definition (a division by a row or column
 *    sum, or the row softmax), using the step's saved output and sum.
 *  - Stage 3.7's RMS term uses raw x: the forward's invRms is taken over raw
 *    x, and [BW] §一 defines gradX as the gradient of that forward.
 *  - Stage 3.4's alpha_res gradient multiplies by the pre-alpha res term
 *    (hMix_res * invRms); the printed symbol is read as garbled.
 *  - Sums over tokens are formed in token order; the result is double and
 *    unrounded (the CUDA path rounds grad_x to bf16).
 * Also returned, for tolerances: the sums of absolute values of the terms
 * that make up each output.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t T, n, D, R;
    int num_iters;
    double hc_eps;
    const uint16_t *x, *grad_h_in, *grad_x_post;   /* bf16 bits */
    const double *phi, *alpha, *gamma;
    const double *grad_h_post, *grad_h_res, *inv_rms, *h_mix, *h_pre, *h_post;
    const double *sum_out, *norm_out;
    /* per-token results of the first phase */
    double *G;        /* [T][R]  H_mix_grad */
    double *coef;     /* [T]     RMS term factor -(inv_rms_grad invRms^3 / nD) */
    double *a_terms;  /* [T][3]  per-token addends of grad_alpha, then |.| */
    double *b_terms;  /* [T][R]  per-token addends of grad_bias */
    /* grad_x for the selected tokens */
    const int64_t *tok_sel;
    int64_t n_tok;
    double *grad_x, *grad_x_abs;
    /* columns for phase 2 */
    const int64_t *col_sel;
    int64_t n_col;
    double *grad_phi, *grad_phi_abs, *grad_gamma, *grad_gamma_abs;
    int64_t begin, end;
    int phase;
} bwd_job;

static double bf16_bits_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Stage 0: carry dL/d(comb) back through the Sinkhorn recurrence of [SK]
 * §3.2 to dL/d(res logits).  Step k (k >= 1) divides by a sum s: a column
 * sum for odd k, a row sum for even k; its output P'_k and sum s are saved.
 * For P' = P / s along a line, dL/dP = (dL/dP' - <dL/dP', P'>_line) / s.
 * Step 0 is the row softmax plus eps, saved as P'_0 = softmax + eps:
 * dL/dH = S (.) (dL/dP - <dL/dP, S>_row) with S = P'_0 - eps. */
static void sinkhorn_backward(const bwd_job *J, int64_t t, double *g /* [n][n] in/out */)
{
    const int64_t n = J->n, T = J->T;
    for (int k = 2 * J->num_iters - 1; k >= 1; --k) {
        const double *Pk = J->norm_out + ((int64_t)k * T + t) * n * n;
        const double *sk = J->sum_out + ((int64_t)k * T + t) * n;
        if (k & 1) {
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t i = 0; i < n; ++i) dot += g[i * n + j] * Pk[i * n + j];
                for (int64_t i = 0; i < n; ++i) g[i * n + j] = (g[i * n + j] - dot) / sk[j];
            }
        } else {
            for (int64_t i = 0; i < n; ++i) {
                double dot = 0.0;
                for (int64_t j = 0; j < n; ++j) dot += g[i * n + j] * Pk[i * n + j];
                for (int64_t j = 0; j < n; ++j) g[i * n + j] = (g[i * n + j] - dot) / sk[i];
            }
        }
    }
    const double *P0 = J->norm_out + t * n * n;
    for (int64_t i = 0; i < n; ++i) {
        double dot = 0.0;
        for (int64_t j = 0; j < n; ++j) dot += g[i * n + j] * (P0[i * n + j] - J->hc_eps);
        for (int64_t j = 0; j < n; ++j) {
            const double S = P0[i * n + j] - J->hc_eps;
            g[i * n + j] = S * (g[i * n + j] - dot);
        }
    }
}

/* Phase 1, one token: stages 3.1-3.5 (and 0), then grad_x (3.6-3.8) when
 * the token is selected (sel >= 0 is its output row). */
static void token_stages(const bwd_job *J, int64_t t, int64_t sel, double *gtmp, double *gres)
{
    const int64_t n = J->n, D = J->D, K = n * D, R = J->R;
    const uint16_t *xt = J->x + t * K;
    const uint16_t *gh = J->grad_h_in + t * D;
    const double *hmix = J->h_mix + t * R;
    const double *hpre = J->h_pre + t * n;
    const double *hpost = J->h_post + t * n;
    const double r = J->inv_rms[t];
    const double a_pre = J->alpha[0], a_post = J->alpha[1], a_res = J->alpha[2];
    double *at = J->a_terms + t * 3;
    double *bt = J->b_terms + t * R;
    at[0] = at[1] = at[2] = 0.0;

    /* 3.1  H_pre_grad[i] = sum_d grad_h_in[d] x[i][d] */
    /* 3.2  sigmoid backward of the pre gate, s = H_pre - hc_eps */
    for (int64_t i = 0; i < n; ++i) {
        double hg = 0.0;
        for (int64_t d = 0; d < D; ++d) hg += bf16_bits_value(gh[d]) * bf16_bits_value(xt[i * D + d]);
        const double s = hpre[i] - J->hc_eps;
        const double g2 = hg * s * (1.0 - s);
        gtmp[i] = g2 * a_pre;
        at[0] += g2 * (hmix[i] * r);
        bt[i] = g2;
    }
    /* 3.3  post gate: d(2 sigma)/dz = H_post (1 - H_post / 2) */
    for (int64_t i = 0; i < n; ++i) {
        const double g2 = J->grad_h_post[t * n + i] * hpost[i] * (1.0 - hpost[i] / 2.0);
        gtmp[n + i] = g2 * a_post;
        at[1] += g2 * (hmix[n + i] * r);
        bt[n + i] = g2;
    }
    /* 3.4  res affine map (after stage 0 when the Sinkhorn intermediates are given) */
    memcpy(gres, J->grad_h_res + t * n * n, (size_t)(n * n) * sizeof(double));
    if (J->norm_out) sinkhorn_backward(J, t, gres);
    for (int64_t e = 0; e < n * n; ++e) {
        gtmp[2 * n + e] = gres[e] * a_res;
        at[2] += gres[e] * (hmix[2 * n + e] * r);
        bt[2 * n + e] = gres[e];
    }
    /* 3.5  H_mix_grad = concat * invRms; inv_rms_grad = sum concat * hMix */
    double irg = 0.0;
    for (int64_t q = 0; q < R; ++q) {
        J->G[t * R + q] = gtmp[q] * r;
        irg += gtmp[q] * hmix[q];
    }
    /* d invRms / d x_k = -invRms^3 x_k / (n D) */
    J->coef[t] = -(irg * r * r * r) / (double)K;

    if (sel < 0) return;
    /* 3.6-3.8 for this token: x_rs_grad = H_mix_grad @ phi, times gamma,
     * plus the RMS term, plus H_in_grad * H_pre, plus grad_x_post. */
    const double *G = J->G + t * R;
    double *gx = J->grad_x + sel * K;
    double *gxa = J->grad_x_abs ? J->grad_x_abs + sel * K : NULL;
    for (int64_t k = 0; k < K; ++k) {
        double xrg = 0.0, xrg_abs = 0.0;
        for (int64_t q = 0; q < R; ++q) {
            xrg += G[q] * J->phi[q * K + k];
            xrg_abs += fabs(G[q] * J->phi[q * K + k]);
        }
        const double gm = J->gamma ? J->gamma[k] : 1.0;
        const int64_t i = k / D, d = k % D;
        const double xv = bf16_bits_value(xt[k]);
        const double v3 = bf16_bits_value(gh[d]) * hpre[i];
        const double mm = xrg * gm;
        const double rms = J->coef[t] * xv;
        double v = v3 + mm + rms;
        double va = fabs(v3) + xrg_abs * fabs(gm) + fabs(rms);
        if (J->grad_x_post) {
            const double p = bf16_bits_value(J->grad_x_post[t * K + k]);
            v += p;
            va += fabs(p);
        }
        gx[k] = v;
        if (gxa) gxa[k] = va;
    }
}

/* Phase 2, one column k of phi: stage 3.6's grad_phi = G^T X with
 * X = x * gamma, and stage 3.7's grad_gamma = sum_t x * x_rs_grad. */
static void column_sums(const bwd_job *J, int64_t k, int64_t out)
{
    const int64_t K = J->n * J->D, R = J->R, T = J->T;
    const double gm = J->gamma ? J->gamma[k] : 1.0;
    double gg = 0.0, gga = 0.0;
    for (int64_t q = 0; q < R; ++q) {
        double s = 0.0, sa = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double term = J->G[t * R + q] * (bf16_bits_value(J->x[t * K + k]) * gm);
            s += term;
            sa += fabs(term);
        }
        J->grad_phi[q * J->n_col + out] = s;
        if (J->grad_phi_abs) J->grad_phi_abs[q * J->n_col + out] = sa;
    }
    if (!J->grad_gamma) return;
    for (int64_t t = 0; t < T; ++t) {
        const double xv = bf16_bits_value(J->x[t * K + k]);
        double xrg = 0.0;
        for (int64_t q = 0; q < R; ++q) {
            xrg += J->G[t * R + q] * J->phi[q * K + k];
            gga += fabs(xv * J->G[t * R + q] * J->phi[q * K + k]);
        }
        gg += xv * xrg;
    }
    J->grad_gamma[out] = gg;
    if (J->grad_gamma_abs) J->grad_gamma_abs[out] = gga;
}

static void *bwd_worker(void *arg)
{
    const bwd_job *J = (const bwd_job *)arg;
    if (J->phase == 1) {
        const int64_t R = J->R, n = J->n;
        double *gtmp = (double *)malloc((size_t)R * sizeof(double));
        double *gres = (double *)malloc((size_t)(n * n) * sizeof(double));
        for (int64_t t = J->begin; t < J->end; ++t) {
            int64_t sel = -1;
            if (J->grad_x) {
                if (!J->tok_sel) {
                    sel = t;
                } else {
                    for (int64_t s = 0; s < J->n_tok; ++s)
                        if (J->tok_sel[s] == t) { sel = s; break; }
                }
            }
            token_stages(J, t, sel, gtmp, gres);
            /* a token selected twice gets its row copied */
            if (sel >= 0 && J->tok_sel)
                for (int64_t s = sel + 1; s < J->n_tok; ++s)
                    if (J->tok_sel[s] == t) {
                        const int64_t K = J->n * J->D;
                        memcpy(J->grad_x + s * K, J->grad_x + sel * K, (size_t)K * sizeof(double));
                        if (J->grad_x_abs)
                            memcpy(J->grad_x_abs + s * K, J->grad_x_abs + sel * K, (size_t)K * sizeof(double));
                    }
        }
        free(gtmp);
        free(gres);
    } else {
        for (int64_t c = J->begin; c < J->end; ++c)
            column_sums(J, J->col_sel ? J->col_sel[c] : c, c);
    }
    return NULL;
}

static void run_phase(bwd_job *base, int phase, int64_t count, int nthreads)
{
    if (nthreads > count) nthreads = count > 0 ? (int)count : 1;
    bwd_job jobs[256];
    pthread_t tid[256];
    for (int w = 0; w < nthreads; ++w) {
        jobs[w] = *base;
        jobs[w].phase = phase;
        jobs[w].begin = count * w / nthreads;
        jobs[w].end = count * (w + 1) / nthreads;
    }
    for (int w = 1; w < nthreads; ++w) pthread_create(&tid[w], NULL, bwd_worker, &jobs[w]);
    bwd_worker(&jobs[0]);
    for (int w = 1; w < nthreads; ++w) pthread_join(tid[w], NULL);
}

/* Returns 0 on success, 1 on bad arguments, 2 if out of memory.
 * grad_x: [n_tok][n][D] for the tokens in tok_sel (all T tokens, in order,
 * when tok_sel is NULL; NULL to skip).  grad_phi: [R][n_col] for the columns
 * in col_sel (all nD when col_sel is NULL), grad_gamma: [n_col] (needs
 * gamma; NULL to skip).  grad_alpha [3], grad_bias [R] and their *_abs
 * companions are always formed.  Every *_abs output is optional. */
int mhc_oracle_pre_backward(int64_t T, int64_t n, int64_t D, int num_iters, double hc_eps,
                            const uint16_t *x, const double *phi, const double *alpha, const double *gamma,
                            const uint16_t *grad_h_in, const double *grad_h_post, const double *grad_h_res,
                            const double *inv_rms, const double *h_mix, const double *h_pre,
                            const double *h_post, const double *sum_out, const double *norm_out,
                            const uint16_t *grad_x_post, int64_t n_tok, const int64_t *tok_sel,
                            int64_t n_col, const int64_t *col_sel, double *grad_x, double *grad_x_abs,
                            double *grad_phi, double *grad_phi_abs, double *grad_gamma,
                            double *grad_gamma_abs, double *grad_alpha, double *grad_alpha_abs,
                            double *grad_bias, double *grad_bias_abs, int nthreads)
{
    if (T < 0 || n < 1 || D < 1 || num_iters < 1 || !x || !phi || !alpha || !grad_h_in ||
        !grad_h_post || !grad_h_res || !inv_rms || !h_mix || !h_pre || !h_post || !grad_alpha ||
        !grad_bias || (!sum_out) != (!norm_out) || (grad_gamma && !gamma))
        return 1;
    const int64_t R = n * n + 2 * n, K = n * D;
    if (!tok_sel) n_tok = T;
    if (!col_sel) n_col = K;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;

    bwd_job J;
    memset(&J, 0, sizeof J);
    J.T = T; J.n = n; J.D = D; J.R = R;
    J.num_iters = num_iters;
    J.hc_eps = hc_eps;
    J.x = x; J.grad_h_in = grad_h_in; J.grad_x_post = grad_x_post;
    J.phi = phi; J.alpha = alpha; J.gamma = gamma;
    J.grad_h_post = grad_h_post; J.grad_h_res = grad_h_res;
    J.inv_rms = inv_rms; J.h_mix = h_mix; J.h_pre = h_pre; J.h_post = h_post;
    J.sum_out = sum_out; J.norm_out = norm_out;
    J.tok_sel = tok_sel; J.n_tok = n_tok; J.grad_x = grad_x; J.grad_x_abs = grad_x_abs;
    J.col_sel = col_sel; J.n_col = n_col;
    J.grad_phi = grad_phi; J.grad_phi_abs = grad_phi_abs;
    J.grad_gamma = grad_gamma; J.grad_gamma_abs = grad_gamma_abs;
    size_t tt = (size_t)(T > 0 ? T : 1);
    J.G = (double *)calloc(tt * (size_t)R, sizeof(double));
    J.coef = (double *)calloc(tt, sizeof(double));
    J.a_terms = (double *)calloc(tt * 3, sizeof(double));
    J.b_terms = (double *)calloc(tt * (size_t)R, sizeof(double));
    if (!J.G || !J.coef || !J.a_terms || !J.b_terms) {
        free(J.G); free(J.coef); free(J.a_terms); free(J.b_terms);
        return 2;
    }

    run_phase(&J, 1, T, nthreads);
    if (grad_phi) run_phase(&J, 2, n_col, nthreads);

    /* grad_alpha and grad_bias: sums over tokens, in token order */
    for (int c = 0; c < 3; ++c) {
        double s = 0.0, sa = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            s += J.a_terms[t * 3 + c];
            sa += fabs(J.a_terms[t * 3 + c]);
        }
        grad_alpha[c] = s;
        if (grad_alpha_abs) grad_alpha_abs[c] = sa;
    }
    for (int64_t q = 0; q < R; ++q) {
        double s = 0.0, sa = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            s += J.b_terms[t * R + q];
            sa += fabs(J.b_terms[t * R + q]);
        }
        grad_bias[q] = s;
        if (grad_bias_abs) grad_bias_abs[q] = sa;
    }
    free(J.G); free(J.coef); free(J.a_terms); free(J.b_terms);
    return 0;
}
