/*
 * mhc_pre_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, double-precision CPU statement of the mHC pre-mapping
 * forward (RMS reciprocal, projection, gates, Sinkhorn, weighted sum), used
 * only to check the CUDA library.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may build, load or call it.  It shares no
 * code, header or constant with the CUDA path.
 *
 * x arrives as bf16 bit patterns (mhc_oracle_pre) or IEEE fp16 ones
 * (mhc_oracle_pre_f16); both are exact in double.
 *
 * Sources (page title, then the section / formula followed):
 *  [V2]  "CANN ops-transformer 中 aclnnMhcPreV2 算子接口全解析：MHC 架构 H 投影
 *        矩阵与 hIn 计算实战指南", §三 (complete forward formula) and §7.3
 *        (two-gate variant: phi [2n, nD], bias [2n], hRes = 0).
 *  [SK]  "CANN ops-transformer 算子详解：aclnnMhcPreSinkhorn 接口与
 *        MhcPreSinkhorn 实现剖析", §3.1 (segment order pre/post/res of phi,
 *        alpha, bias), §3.2 (Sinkhorn recurrence and its golden description),
 *        §5.1 (shapes of sumOut / normOut, hcBeforeNorm taken before invRms).
 *  [HC]  "CANN HcPre 融合算子解析：mHC 结构前处理 custom.npu_hc_pre 与
 *        npu_hc_pre_v2 实战指南", 功能说明与计算流程 (pre_mix replaces hPre as
 *        the weights of y; hc_pre still returned) and 精度验证 (HF32
 *        simulation: clear the low 13 mantissa bits of each fp32 matmul
 *        operand, round toward zero, before multiplying).
 *
 * hf32 selects the projection's precision: 0 exact; 1 the HF32 simulation
 * on the matmul operands x (.) gamma and phi as [HC] states it; 2 the same
 * truncation applied to the folded weight gamma (.) phi (rounded to fp32
 * first) with x exact -- the reading of HF32 for a projection that carries
 * gamma on the weight side.  Without gamma, 1 and 2 are the same.
 *
 * Readings where the pages are silent or garbled (each is listed in the
 * design notes as well):
 *  - the RMS mean runs over all n*D elements of the token, from raw x;
 *  - the res logits map row-major to H[i][j] = w[2n + i*n + j];
 *  - sumOut[0] (never defined by the pages) holds the softmax row
 *    denominators sum_j exp(H[i][j] - max_j H[i][j])  -- parity unpinned;
 *  - the two-gate variant runs no Sinkhorn, hRes is 0, hPost gets + hcEps;
 *  - y is accumulated exactly (double) and handed back unrounded; rounding
 *    to bf16 is the caller's business.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t T, n, D;
    int alpha_len, num_iters, hf32, x_fp16;
    double norm_eps, hc_eps;
    const uint16_t *x;      /* bf16 bits [T][n][D] */
    const float *phi;       /* [R][n*D] */
    const float *alpha;     /* [alpha_len] */
    const float *bias;      /* [R] */
    const float *gamma;     /* [n][D] or NULL */
    const float *pre_mix;   /* [T][n] or NULL */
    double *y, *h_post, *h_res, *h_pre, *inv_rms, *h_mix, *sum_out, *norm_out;
    int64_t t_begin, t_end;
} oracle_job;

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds the subnormals 2^-14 * f / 1024, exponent 31 the
 * infinities and NaNs. */
double mhc_oracle_half_value(uint16_t bits)
{
    const int sign = bits >> 15, e = (bits >> 10) & 31, f = bits & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25);
    return sign ? -v : v;
}

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* [HC] 精度验证: HF32 keeps sign, exponent and the top 10 mantissa bits of an
 * fp32 operand, truncating the rest toward zero. */
static double hf32_value(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    u &= 0xFFFFE000u;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

static void one_token(const oracle_job *J, int64_t t, double *w, double *P)
{
    const int64_t n = J->n, D = J->D, K = n * D, T = J->T;
    const int64_t R = (J->alpha_len == 3) ? n * n + 2 * n : 2 * n;
    const uint16_t *xt = J->x + t * K;

    /* [V2] §三: invRms = (mean(xFlat^2) + normEps)^(-1/2), raw x, mean over nD. */
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double v = J->x_fp16 ? mhc_oracle_half_value(xt[k]) : bf16_value(xt[k]);
        ss += v * v;
    }
    double inv_rms = 1.0 / sqrt(ss / (double)K + J->norm_eps);

    /* [V2] §三: xGamma = xFlat (.) gammaFlat (or xFlat); hMix = xGamma phi^T. */
    for (int64_t r = 0; r < R; ++r) {
        const float *phi_r = J->phi + r * K;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double g = J->x_fp16 ? mhc_oracle_half_value(xt[k]) : bf16_value(xt[k]);
            double p = phi_r[k];
            if (J->hf32 == 2) {
                /* HF32 on the folded weight: gamma (.) phi rounded to fp32,
                 * then truncated (x is exact in the HF32 format). */
                if (J->gamma)
                    p = hf32_value((float)((double)phi_r[k] * (double)J->gamma[k]));
                else
                    p = hf32_value(phi_r[k]);
            } else {
                if (J->gamma) {
                    if (J->hf32)
                        g = hf32_value((float)(g * (double)J->gamma[k]));
                    else
                        g = g * (double)J->gamma[k];
                }
                if (J->hf32)
                    p = hf32_value(phi_r[k]);
            }
            acc += g * p;
        }
        if (J->h_mix)
            J->h_mix[t * R + r] = acc;          /* [SK] §5.1 hcBeforeNorm */
        w[r] = acc * inv_rms;                   /* [V2] §三: w = hMix (.) invRms */
    }
    if (J->inv_rms)
        J->inv_rms[t] = inv_rms;

    /* [V2] §三 gates; [SK] §3.1 segment order pre (n), post (n), res (n^2). */
    const double a0 = J->alpha[0], a1 = J->alpha[1];
    double h_pre[64];
    for (int64_t i = 0; i < n; ++i) {
        h_pre[i] = sigmoid(a0 * w[i] + (double)J->bias[i]) + J->hc_eps;
        double post = 2.0 * sigmoid(a1 * w[n + i] + (double)J->bias[n + i]);
        if (J->alpha_len == 2)
            post += J->hc_eps;                  /* [V2] §三: two-gate case only */
        J->h_post[t * n + i] = post;
        J->h_pre[t * n + i] = h_pre[i];
    }

    if (J->alpha_len == 3) {
        const double a2 = J->alpha[2];
        const double eps = J->hc_eps;
        /* H[i][j] = alpha2 * pRes + bias2, row-major reshape to [n, n]. */
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = 0; j < n; ++j)
                P[i * n + j] = a2 * w[2 * n + i * n + j] + (double)J->bias[2 * n + i * n + j];

        /* [SK] §3.2 first step: normOut[0] = softmax(H, dim=-1) + eps, the
         * softmax taken after subtracting the row maximum (golden text). */
        for (int64_t i = 0; i < n; ++i) {
            double m = P[i * n];
            for (int64_t j = 1; j < n; ++j)
                if (P[i * n + j] > m) m = P[i * n + j];
            double s = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                P[i * n + j] = exp(P[i * n + j] - m);
                s += P[i * n + j];
            }
            for (int64_t j = 0; j < n; ++j)
                P[i * n + j] = P[i * n + j] / s + eps;
            if (J->sum_out)
                J->sum_out[(0 * T + t) * n + i] = s;
        }
        if (J->norm_out)
            for (int64_t e = 0; e < n * n; ++e)
                J->norm_out[(0 * T + t) * n * n + e] = P[e];

        /* Then: column step (sum over dim -2), then (row, column) x (I - 1).
         * Step k = 1 .. 2I-1; odd k normalise columns, even k rows. */
        const int64_t steps = 2 * (int64_t)J->num_iters;
        for (int64_t k = 1; k < steps; ++k) {
            int col = (k % 2) == 1;
            for (int64_t a = 0; a < n; ++a) {
                double s = 0.0;
                for (int64_t b = 0; b < n; ++b)
                    s += col ? P[b * n + a] : P[a * n + b];
                s += eps;
                for (int64_t b = 0; b < n; ++b) {
                    if (col)
                        P[b * n + a] = P[b * n + a] / s;
                    else
                        P[a * n + b] = P[a * n + b] / s;
                }
                if (J->sum_out)
                    J->sum_out[(k * T + t) * n + a] = s;
            }
            if (J->norm_out)
                for (int64_t e = 0; e < n * n; ++e)
                    J->norm_out[(k * T + t) * n * n + e] = P[e];
        }
        if (J->h_res)
            for (int64_t e = 0; e < n * n; ++e)
                J->h_res[t * n * n + e] = P[e];
    } else if (J->h_res) {
        for (int64_t e = 0; e < n * n; ++e)
            J->h_res[t * n * n + e] = 0.0;      /* [V2] §三: hRes = 0 */
    }

    /* [V2] §三: hIn_d = sum_i hPre_i x_{i,d} from raw x; [HC]: with pre_mix
     * given, the weights are pre_mix instead. */
    for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            double m = J->pre_mix ? (double)J->pre_mix[t * n + i] : h_pre[i];
            acc += m * (J->x_fp16 ? mhc_oracle_half_value(xt[i * D + d]) : bf16_value(xt[i * D + d]));
        }
        J->y[t * D + d] = acc;
    }
}

static void *worker(void *arg)
{
    const oracle_job *J = (const oracle_job *)arg;
    const int64_t R = (J->alpha_len == 3) ? J->n * J->n + 2 * J->n : 2 * J->n;
    double *w = (double *)malloc(sizeof(double) * (size_t)R);
    double *P = (double *)malloc(sizeof(double) * (size_t)(J->n * J->n));
    for (int64_t t = J->t_begin; t < J->t_end; ++t)
        one_token(J, t, w, P);
    free(w);
    free(P);
    return NULL;
}

/* Returns 0 on success, -1 on bad arguments.  All outputs are double and
 * laid out like the operator's: y [T][D], h_post/h_pre [T][n],
 * h_res [T][n][n] (may be NULL), inv_rms [T], h_mix [T][R] (may be NULL),
 * sum_out [2I][T][n] and norm_out [2I][T][n][n] (may be NULL). */
static int run_pre(int64_t T, int64_t n, int64_t D, int alpha_len, int num_iters,
                   double norm_eps, double hc_eps, int hf32, int x_fp16,
                   const uint16_t *x, const float *phi, const float *alpha,
                   const float *bias, const float *gamma, const float *pre_mix,
                   double *y, double *h_post, double *h_res, double *h_pre,
                   double *inv_rms, double *h_mix, double *sum_out,
                   double *norm_out, int nthreads)
{
    if (T < 0 || n < 1 || n > 64 || D < 1 || (alpha_len != 2 && alpha_len != 3) ||
        num_iters < 1 || !x || !phi || !alpha || !bias || !y || !h_post || !h_pre)
        return -1;
    if (T == 0)
        return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > T) nthreads = (int)T;

    oracle_job base;
    memset(&base, 0, sizeof base);
    base.T = T; base.n = n; base.D = D;
    base.alpha_len = alpha_len; base.num_iters = num_iters; base.hf32 = hf32;
    base.x_fp16 = x_fp16;
    base.norm_eps = norm_eps; base.hc_eps = hc_eps;
    base.x = x; base.phi = phi; base.alpha = alpha; base.bias = bias;
    base.gamma = gamma; base.pre_mix = pre_mix;
    base.y = y; base.h_post = h_post; base.h_res = h_res; base.h_pre = h_pre;
    base.inv_rms = inv_rms; base.h_mix = h_mix;
    base.sum_out = sum_out; base.norm_out = norm_out;

    oracle_job *jobs = (oracle_job *)malloc(sizeof(oracle_job) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].t_begin = T * i / nthreads;
        jobs[i].t_end = T * (i + 1) / nthreads;
        pthread_create(&tid[i], NULL, worker, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(tid[i], NULL);
    free(jobs);
    free(tid);
    return 0;
}

/* The forward with x given as bf16 bit patterns (the pages' examples)... */
int mhc_oracle_pre(int64_t T, int64_t n, int64_t D, int alpha_len, int num_iters,
                   double norm_eps, double hc_eps, int hf32,
                   const uint16_t *x, const float *phi, const float *alpha,
                   const float *bias, const float *gamma, const float *pre_mix,
                   double *y, double *h_post, double *h_res, double *h_pre,
                   double *inv_rms, double *h_mix, double *sum_out,
                   double *norm_out, int nthreads)
{
    return run_pre(T, n, D, alpha_len, num_iters, norm_eps, hc_eps, hf32, 0, x, phi, alpha, bias,
                   gamma, pre_mix, y, h_post, h_res, h_pre, inv_rms, h_mix, sum_out, norm_out,
                   nthreads);
}

/* ...or as fp16 (IEEE binary16) bit patterns, the other x type the
 * Sinkhorn page lists; everything after reading x is the same. */
int mhc_oracle_pre_f16(int64_t T, int64_t n, int64_t D, int alpha_len, int num_iters,
                       double norm_eps, double hc_eps, int hf32,
                       const uint16_t *x, const float *phi, const float *alpha,
                       const float *bias, const float *gamma, const float *pre_mix,
                       double *y, double *h_post, double *h_res, double *h_pre,
                       double *inv_rms, double *h_mix, double *sum_out,
                       double *norm_out, int nthreads)
{
    return run_pre(T, n, D, alpha_len, num_iters, norm_eps, hc_eps, hf32, 1, x, phi, alpha, bias,
                   gamma, pre_mix, y, h_post, h_res, h_pre, inv_rms, h_mix, sum_out, norm_out,
                   nthreads);
}
