/*
 * kda_oracle.c - FP64 CPU oracle for the KDA (Kimi Delta Attention) mixer core.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg to check and time the CUDA library. It is not
 * part of the product path and shares no code with it.
 *
 * What it computes, step by step, for one token of one head (kimi_k3.c,
 * header comment, block "KDA per-head recurrence"):
 *   1. q,k,v = SiLU(ShortConv4(x)) per channel; the conv is depthwise and
 *      causal with 4 taps stored oldest first (kimi_k3.c, struct Kda:
 *      "depthwise taps, oldest first").
 *   2. q and k are L2-normalised over the head with eps 1e-6 inside the sqrt,
 *      then q is multiplied by d^-1/2.
 *   3. gk = gmin * sigmoid(exp(A_log[h]) * (z + dt_bias)), gmin = -5, per
 *      channel; alpha = exp(gk); beta = sigmoid(b), one scalar per head.
 *   4. S = (I - beta k k^T) Diag(alpha) S + beta k v^T with S laid out
 *      S[key][value] (kimi_k3.c, struct Model: "S[k][v]").
 *   5. o = S^T q, read after the update.
 *   6. out = sigmoid(g) * RMSNorm_head(o), the RMSNorm weight being the
 *      per-head-dim vector o_norm shared by all heads (struct Kda: o_norm[hd]).
 * The helpers follow sigmoidf_, siluf_ and rmsnorm_ of kimi_k3.c, in double.
 *
 * Readings where the pages are silent: the RMSNorm eps is a config field;
 * z and dt_bias arrive separately and are added before the multiply by
 * exp(A_log); the conv has no bias; the conv history holds the K-1 raw
 * (pre-conv) inputs; nothing crosses a sequence boundary.
 */
#include "kda_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double kdao_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

double kdao_silu(double x) { return x / (1.0 + exp(-x)); }

double kdao_conv_silu(int K, const double *taps, const double *hist, double x)
{
    /* y = sum_j taps[j] * x_{t-(K-1)+j}; the newest input meets the last tap */
    double c = 0.0;
    for (int j = 0; j < K - 1; ++j)
        c += taps[j] * hist[j];
    c += taps[K - 1] * x;
    return kdao_silu(c);
}

void kdao_l2norm(int d, const double *x, double eps, double scale, double *y)
{
    double s = 0.0;
    for (int i = 0; i < d; ++i)
        s += x[i] * x[i];
    double r = 1.0 / sqrt(s + eps);
    for (int i = 0; i < d; ++i)
        y[i] = x[i] * r * scale;
}

double kdao_gate_alpha(double A_log, double z, double dt, double gmin, double *gk_out)
{
    double gk = gmin * kdao_sigmoid(exp(A_log) * (z + dt));
    if (gk_out)
        *gk_out = gk;
    return exp(gk);
}

void kdao_delta_step(int d, double *S, const double *alpha, double beta,
                     const double *k, const double *v, const double *q, double *o)
{
    /* Diag(alpha) S: row i (key index) scaled by alpha_i */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(long)i * d + j] *= alpha[i];
    /* (I - beta k k^T) S = S - beta k (k^T S) */
    double *w = (double *)malloc(sizeof(double) * (size_t)d);
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += k[i] * S[(long)i * d + j];
        w[j] = acc;
    }
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(long)i * d + j] -= beta * k[i] * w[j];
    /* + beta k v^T */
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            S[(long)i * d + j] += beta * k[i] * v[j];
    /* o = S^T q with the updated state */
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += S[(long)i * d + j] * q[i];
        o[j] = acc;
    }
    free(w);
}

void kdao_rmsnorm_gate(int d, const double *o, const double *w, const double *g,
                       double eps, double *out)
{
    double ms = 0.0;
    for (int i = 0; i < d; ++i)
        ms += o[i] * o[i];
    double r = 1.0 / sqrt(ms / d + eps);
    for (int i = 0; i < d; ++i)
        out[i] = kdao_sigmoid(g[i]) * (o[i] * r * w[i]);
}

void kdao_unit(const kdao_cfg *cfg, int h,
               const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
               double *S, double *tail, long tail_ld, int T,
               const float *q, const float *k, const float *v, const float *z, const float *g,
               long ld, const float *b, long ldb, double *out, long ldo)
{
    const int d = cfg->d, K = cfg->K, D = cfg->H * cfg->d;
    double *xq = (double *)malloc(sizeof(double) * (size_t)d);
    double *xk = (double *)malloc(sizeof(double) * (size_t)d);
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *qh = (double *)malloc(sizeof(double) * (size_t)d);
    double *kh = (double *)malloc(sizeof(double) * (size_t)d);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)d);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    double *gg = (double *)malloc(sizeof(double) * (size_t)d);
    double *nw = (double *)malloc(sizeof(double) * (size_t)d);
    double taps[8], hist[8];
    for (int i = 0; i < d; ++i)
        nw[i] = (double)norm_w[i];

    for (int t = 0; t < T; ++t) {
        const float *src[3] = {q + (long)t * ld, k + (long)t * ld, v + (long)t * ld};
        double *dst[3] = {xq, xk, xv};
        /* 1. ShortConv + SiLU per channel, then shift the raw-input history */
        for (int x = 0; x < 3; ++x) {
            double *tx = tail + (long)x * (K - 1) * tail_ld;
            for (int i = 0; i < d; ++i) {
                const int c = h * d + i;
                for (int j = 0; j < K; ++j)
                    taps[j] = (double)conv_w[((long)x * D + c) * K + j];
                for (int j = 0; j < K - 1; ++j)
                    hist[j] = tx[(long)j * tail_ld + i];
                const double xin = (double)src[x][i];
                dst[x][i] = kdao_conv_silu(K, taps, hist, xin);
                for (int j = 0; j + 1 < K - 1; ++j)
                    tx[(long)j * tail_ld + i] = tx[(long)(j + 1) * tail_ld + i];
                if (K > 1)
                    tx[(long)(K - 2) * tail_ld + i] = xin;
            }
        }
        /* 2. L2 normalisation, q scaled after it */
        kdao_l2norm(d, xq, cfg->l2_eps, cfg->q_scale, qh);
        kdao_l2norm(d, xk, cfg->l2_eps, 1.0, kh);
        /* 3. gates */
        for (int i = 0; i < d; ++i)
            alpha[i] = kdao_gate_alpha((double)A_log[h], (double)z[(long)t * ld + i],
                                       (double)dt_bias[h * d + i], cfg->gate_lb, NULL);
        const double beta = kdao_sigmoid((double)b[(long)t * ldb]);
        /* 4-5. delta rule and readout */
        kdao_delta_step(d, S, alpha, beta, kh, xv, qh, o);
        /* 6. gated RMSNorm */
        for (int i = 0; i < d; ++i)
            gg[i] = (double)g[(long)t * ld + i];
        kdao_rmsnorm_gate(d, o, nw, gg, cfg->rms_eps, out + (long)t * ldo);
    }
    free(xq); free(xk); free(xv); free(qh); free(kh);
    free(alpha); free(o); free(gg); free(nw);
}

void kdao_sequence(const kdao_cfg *cfg,
                   const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
                   double *S, double *tail, int T,
                   const float *q, const float *k, const float *v, const float *z,
                   const float *b, const float *g, double *out, int nthreads)
{
    const int H = cfg->H, d = cfg->d;
    const long D = (long)H * d;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int h = 0; h < H; ++h) {
        const long off = (long)h * d;
        kdao_unit(cfg, h, conv_w, dt_bias, A_log, norm_w,
                  S + (long)h * d * d, tail + off, D, T,
                  q + off, k + off, v + off, z + off, g + off, D,
                  b + h, H, out + off, D);
    }
}

void kdao_decode_batch(const kdao_cfg *cfg,
                       const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
                       double *S_all, double *tail_all, const int32_t *slots, int B,
                       const float *q, const float *k, const float *v, const float *z,
                       const float *b, const float *g, double *out, int nthreads)
{
    const int H = cfg->H, d = cfg->d, K = cfg->K;
    const long D = (long)H * d;
    const long n_units = (long)B * H;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (long u = 0; u < n_units; ++u) {
        const int r = (int)(u / H), h = (int)(u % H);
        const long slot = slots[r];
        const long off = (long)h * d;
        double *S = S_all + (slot * H + h) * (long)d * d;
        double *tail = tail_all + slot * 3 * (long)(K - 1) * D + off;
        const long row = (long)r * D + off;
        kdao_unit(cfg, h, conv_w, dt_bias, A_log, norm_w, S, tail, D, 1,
                  q + row, k + row, v + row, z + row, g + row, D,
                  b + (long)r * H + h, H, out + row, D);
    }
}

int kdao_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
