/*
 * kda_oracle.h - FP64 CPU oracle for the KDA (Kimi Delta Attention) mixer core.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or
 * call this file: only tests, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Source of every formula: the header comment of kimi_k3.c, block
 * "KDA per-head recurrence", plus the Kda struct comments (conv taps oldest
 * first; dt_bias per channel, A per head, o_norm per head-dim) and the math
 * helpers sigmoidf_/siluf_/rmsnorm_ of the same file.
 *
 * Everything is double precision and strictly sequential per token.
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int H;           /* number of KDA heads */
    int d;           /* head dim (dk = dv = d) */
    int K;           /* short-conv kernel size (4) */
    double gate_lb;  /* gate lower bound gmin (-5) */
    double l2_eps;   /* eps inside the sqrt of the q/k L2 norm (1e-6) */
    double rms_eps;  /* eps of the per-head RMSNorm */
    double q_scale;  /* q multiplier after L2 (d^-1/2) */
} kdao_cfg;

/* ---- single-step helpers (exported so tests can pin each one) ---- */
double kdao_sigmoid(double x);
double kdao_silu(double x);
/* causal depthwise conv of one channel + SiLU: hist[0..K-2] oldest first, x newest */
double kdao_conv_silu(int K, const double *taps, const double *hist, double x);
/* y = x / sqrt(sum x^2 + eps) * scale */
void kdao_l2norm(int d, const double *x, double eps, double scale, double *y);
/* alpha = exp(gk), gk = gmin * sigmoid(exp(A_log) * (z + dt)); *gk_out may be NULL */
double kdao_gate_alpha(double A_log, double z, double dt, double gmin, double *gk_out);
/* S <- (I - beta k k^T) Diag(alpha) S + beta k v^T, then o = S^T q (S is [d][d], S[key][value]) */
void kdao_delta_step(int d, double *S, const double *alpha, double beta,
                     const double *k, const double *v, const double *q, double *o);
/* out = sigmoid(g) * (o / sqrt(mean(o^2) + eps) * w) */
void kdao_rmsnorm_gate(int d, const double *o, const double *w, const double *g,
                       double eps, double *out);

/* ---- one (sequence, head) unit over T tokens ----
 * conv_w  [3][D][K] float (q, k, v taps; tap 0 oldest), D = H*d
 * dt_bias [D], A_log [H], norm_w [d]
 * S       [d][d] double, this head's state, updated in place
 * tail    this head's conv history: element (x, j, i) at tail[(x*(K-1) + j)*tail_ld + i],
 *         x in {q,k,v}, j = 0 oldest, i in [0,d); updated in place
 * q,k,v,z,g: row t, channel i of this head at ptr[t*ld + i] (pointers already offset to the head)
 * b       row t at b[t*ldb]
 * out     row t, channel i at out[t*ldo + i]
 */
void kdao_unit(const kdao_cfg *cfg, int h,
               const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
               double *S, double *tail, long tail_ld, int T,
               const float *q, const float *k, const float *v, const float *z, const float *g,
               long ld, const float *b, long ldb, double *out, long ldo);

/* ---- whole sequence, all heads (heads run on up to nthreads threads) ----
 * S [H][d][d], tail [3][K-1][D], inputs [T][D], b [T][H], out [T][D]
 */
void kdao_sequence(const kdao_cfg *cfg,
                   const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
                   double *S, double *tail, int T,
                   const float *q, const float *k, const float *v, const float *z,
                   const float *b, const float *g, double *out, int nthreads);

/* ---- one decode token for a batch of B sequences (units run on up to nthreads threads) ----
 * S_all [n_slots][H][d][d], tail_all [n_slots][3][K-1][D]; row r of the inputs uses slot slots[r]
 * inputs [B][D], b [B][H], out [B][D]
 */
void kdao_decode_batch(const kdao_cfg *cfg,
                       const float *conv_w, const float *dt_bias, const float *A_log, const float *norm_w,
                       double *S_all, double *tail_all, const int32_t *slots, int B,
                       const float *q, const float *k, const float *v, const float *z,
                       const float *b, const float *g, double *out, int nthreads);

/* number of threads the OpenMP runtime would use (1 when built without OpenMP) */
int kdao_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
