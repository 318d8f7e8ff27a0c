/*
 * mhc_post_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain double-precision CPU statement of the mHC post-mapping (hc_post),
 * used only to check the CUDA library.  Only the tests and the benchmark's
 * CPU-baseline leg may build, load or call it.  It shares no code, header or
 * constant with the CUDA path.
 *
 * Source: "CANN HcPre 融合算子解析：mHC 结构前处理 custom.npu_hc_pre 与
 * npu_hc_pre_v2 实战指南", mHC section (hc_pre does the pre-processing,
 * hc_post the post-processing): the output is post times the layer output
 * plus the residual streams mixed by comb.
 *
 * Reading (the printed reduction axis would scale each stream by its own row
 * sum of comb instead of mixing streams; the mixing the architecture needs
 * is taken, and listed in the design notes):
 *     out[t][j][d] = post[t][j] * x[t][d] + sum_i comb[t][i][j] * residual[t][i][d]
 * Inputs x and residual are bf16 (exact in double); the result is returned
 * unrounded.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n, D;
    const uint16_t *x;        /* bf16 bits [T][D] */
    const uint16_t *residual; /* bf16 bits [T][n][D] */
    const float *post;        /* [T][n] */
    const float *comb;        /* [T][n][n] */
    double *out;              /* [T][n][D] */
    int64_t t_begin, t_end;
} post_job;

static double bf16_bits_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static void *post_worker(void *arg)
{
    const post_job *J = (const post_job *)arg;
    const int64_t n = J->n, D = J->D;
    for (int64_t t = J->t_begin; t < J->t_end; ++t) {
        for (int64_t j = 0; j < n; ++j) {
            const double p = (double)J->post[t * n + j];
            for (int64_t d = 0; d < D; ++d) {
                double acc = p * bf16_bits_value(J->x[t * D + d]);
                for (int64_t i = 0; i < n; ++i)
                    acc += (double)J->comb[(t * n + i) * n + j] *
                           bf16_bits_value(J->residual[(t * n + i) * D + d]);
                J->out[(t * n + j) * D + d] = acc;
            }
        }
    }
    return NULL;
}

int mhc_oracle_post(int64_t T, int64_t n, int64_t D, const uint16_t *x, const uint16_t *residual,
                    const float *post, const float *comb, double *out, int nthreads)
{
    if (T < 0 || n < 1 || D < 1 || !x || !residual || !post || !comb || !out)
        return 1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > T)
        nthreads = T > 0 ? (int)T : 1;
    post_job jobs[256];
    pthread_t tid[256];
    for (int w = 0; w < nthreads; ++w) {
        post_job *J = &jobs[w];
        J->n = n;
        J->D = D;
        J->x = x;
        J->residual = residual;
        J->post = post;
        J->comb = comb;
        J->out = out;
        J->t_begin = T * w / nthreads;
        J->t_end = T * (w + 1) / nthreads;
    }
    for (int w = 1; w < nthreads; ++w)
        pthread_create(&tid[w], NULL, post_worker, &jobs[w]);
    post_worker(&jobs[0]);
    for (int w = 1; w < nthreads; ++w)
        pthread_join(tid[w], NULL);
    return 0;
}
