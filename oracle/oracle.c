/*
 * oracle.c — plain, single-threaded C oracle of the per-layer mixed-precision
 * AdamW step (R-replica gradient mean -> optional global clip -> AdamW with
 * bias correction on the FP32 master and moments -> BF16 compute copy).
 *
 * TEST INFRASTRUCTURE ONLY: see oracle.h for who may use it and for the
 * passages it follows.  It shares no code, header, table or constant with the
 * GPU library.  Build: cc -std=c99 -O2 -ffp-contract=off -fPIC -shared -lm.
 * No fast-math, no SIMD intrinsics, no threads: each FP32 operation below is
 * one IEEE-754 single-precision operation, performed in the written order.
 *
 * The same source also builds with -fopenmp, for one purpose only: timing the
 * oracle on all host cores as a second CPU baseline.  Then the element loops
 * are split across threads (each element's operations are unchanged) and the
 * clip's double sum is taken as per-thread partials (a different summation
 * order).  Parity tests and pins use the single-threaded build, in which the
 * omp pragmas are ignored.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the element loops use: 1 in the single-threaded build. */
int32_t oracle_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- BF16 <-> FP32 ------------------------------------------------------
 * BF16 is the upper half of an IEEE binary32 (1 sign, 8 exponent, 7 fraction
 * bits).  Widening is exact.  Narrowing rounds the dropped 16 bits to the
 * nearest representable value, ties to an even last kept bit; the carry of a
 * round-up propagates into the exponent, which is exactly the next BF16 value
 * (and turns the largest finite values into infinity, as IEEE rounding does).
 * A NaN keeps its sign and gets the quiet bit so it cannot become infinity. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);           /* quiet NaN */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

void oracle_f32_to_bf16_rne_array(int64_t n, const float *x, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16_rne(x[i]);
}

void oracle_bf16_to_f32_array(int64_t n, const uint16_t *h, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_f32(h[i]);
}

/* ---- per-step scalars ---------------------------------------------------
 * The bias corrections of Adam (Kingma & Ba): bc1 = 1 - beta1^t,
 * bc2 = 1 - beta2^t, t the 1-based count of updates of this layer (the
 * SlideDP page allows exactly one aggregated update of each layer per
 * iteration, so t is the layer's own update count).  They are formed in double from the FP32
 * hyper-parameters, and each derived scalar is rounded once to FP32. */
void oracle_step_scalars_for(const oracle_hparams *hp, int64_t t, oracle_step_scalars *out)
{
    double b1 = (double)hp->beta1;
    double b2 = (double)hp->beta2;
    double bc1 = 1.0 - pow(b1, (double)t);
    double bc2 = 1.0 - pow(b2, (double)t);
    out->beta1 = hp->beta1;
    out->one_minus_beta1 = (float)(1.0 - b1);
    out->beta2 = hp->beta2;
    out->one_minus_beta2 = (float)(1.0 - b2);
    out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    out->step_size = (float)((double)hp->lr / bc1);
    out->bc2_sqrt = (float)sqrt(bc2);
    out->eps = hp->eps;
}

/* ---- a1: mean of the R gradient replicas --------------------------------
 * SlideDP, Core method / Method steps: the R ranks' gradients of layer l are
 * reduced on the GPU to one aggregated gradient G_l before the update.  The
 * aggregate is the mean: the Prerequisites section describes synchronous DP
 * as mathematically the same as one large batch on one GPU, which is what
 * averaging the ranks' gradients gives.  Summed in FP32 in replica order,
 * then divided by R. */
void oracle_grad_mean(int64_t n, int32_t R, const uint16_t *const *g, float *gm)
{
    float fr = (float)R;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float s = oracle_bf16_to_f32(g[0][i]);
        for (int32_t r = 1; r < R; ++r)
            s = s + oracle_bf16_to_f32(g[r][i]);
        gm[i] = s / fr;
    }
}

void oracle_grad_mean_f32(int64_t n, int32_t R, const float *const *g, float *gm)
{
    float fr = (float)R;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float s = g[0][i];
        for (int32_t r = 1; r < R; ++r)
            s = s + g[r][i];
        gm[i] = s / fr;
    }
}

/* ---- a2: optional global clip of the layer's mean gradient ---------------
 * Not on the pages; the benchmark workload asks for a global grad-norm clip.
 * The norm is the L2 norm of the whole layer's mean gradient (all of its
 * tensors), summed in double in index order. */
double oracle_grad_sqnorm(int64_t n, const float *gm)
{
    double s = 0.0;
#pragma omp parallel for schedule(static) reduction(+ : s)
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)gm[i];
        s = s + x * x;
    }
    return s;
}

float oracle_clip_coef(double sqnorm, float max_norm)
{
    if (!(max_norm > 0.0f))
        return 1.0f;
    double norm = sqrt(sqnorm);
    double c = (double)max_norm / (norm + 1e-6);
    if (c > 1.0)
        c = 1.0;
    return (float)c;
}

/* ---- a3..a5: AdamW on the FP32 master and moments, BF16 copy ------------
 * SlideDP Core method: host-resident FP32 master Theta_l^32 and Adam moments
 * (m_l, v_l), one update per layer per iteration (LayerAdam); the result is
 * cast FP32 -> BF16 for the next delivery (Core method: the host casts the
 * next chunk to BF16 while the current one is copied; SlideFormer section
 * 2.2: the FP32 -> BF16 type conversion is done on the host).
 * Per element, in this order, each line one FP32 operation:
 *   g  = gm*coef
 *   m  = beta1*m + (1-beta1)*g
 *   v  = beta2*v + (1-beta2)*(g*g)
 *   th = th*(1 - lr*wd)                       (decoupled decay)
 *   den = sqrt(v)/sqrt(bc2) + eps             (= sqrt(v_hat) + eps)
 *   th = th - (lr/bc1)*(m/den)                (= lr*m_hat/(sqrt(v_hat)+eps))
 *   w  = bf16_rne(th)                                                      */
void oracle_adamw_update(int64_t n, const float *gm, float coef,
                         float *theta, float *m, float *v, uint16_t *w,
                         const oracle_hparams *hp, int64_t t)
{
    oracle_step_scalars k;
    oracle_step_scalars_for(hp, t, &k);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float g = gm[i] * coef;

        float m_old = m[i] * k.beta1;
        float m_new = k.one_minus_beta1 * g;
        float mi = m_old + m_new;

        float v_old = v[i] * k.beta2;
        float g2 = g * g;
        float v_new = k.one_minus_beta2 * g2;
        float vi = v_old + v_new;

        float th = theta[i] * k.decay;
        float root = sqrtf(vi);
        float den = root / k.bc2_sqrt;
        den = den + k.eps;
        float ratio = mi / den;
        float delta = k.step_size * ratio;
        th = th - delta;

        m[i] = mi;
        v[i] = vi;
        theta[i] = th;
        if (w)
            w[i] = oracle_f32_to_bf16_rne(th);
    }
}

float oracle_layer_step(int64_t n, int32_t R, const uint16_t *const *g,
                        float *theta, float *m, float *v, uint16_t *w,
                        const oracle_hparams *hp, int64_t t)
{
    float *gm = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!gm)
        return -1.0f;
    oracle_grad_mean(n, R, g, gm);
    float coef = 1.0f;
    if (hp->max_grad_norm > 0.0f)
        coef = oracle_clip_coef(oracle_grad_sqnorm(n, gm), hp->max_grad_norm);
    oracle_adamw_update(n, gm, coef, theta, m, v, w, hp, t);
    free(gm);
    return coef;
}

float oracle_layer_step_f32g(int64_t n, int32_t R, const float *const *g,
                             float *theta, float *m, float *v, uint16_t *w,
                             const oracle_hparams *hp, int64_t t)
{
    float *gm = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!gm)
        return -1.0f;
    oracle_grad_mean_f32(n, R, g, gm);
    float coef = 1.0f;
    if (hp->max_grad_norm > 0.0f)
        coef = oracle_clip_coef(oracle_grad_sqnorm(n, gm), hp->max_grad_norm);
    oracle_adamw_update(n, gm, coef, theta, m, v, w, hp, t);
    free(gm);
    return coef;
}

/* ---- float64 brute force --------------------------------------------------
 * The same step with every quantity in double and the textbook arrangement
 * of the bias correction (corrected moments m_hat, v_hat formed explicitly). */
/* The double-precision update given the double mean gradient gm (clipped in
 * place when max_grad_norm > 0); returns the clip coefficient. */
static double f64_update(int64_t n, double *gm, double *theta, double *m, double *v,
                         const oracle_hparams *hp, int64_t t)
{
    double coef = 1.0;
    if (hp->max_grad_norm > 0.0f) {
        double sq = 0.0;
        for (int64_t i = 0; i < n; ++i)
            sq += gm[i] * gm[i];
        coef = (double)hp->max_grad_norm / (sqrt(sq) + 1e-6);
        if (coef > 1.0)
            coef = 1.0;
    }
    double b1 = hp->beta1, b2 = hp->beta2, lr = hp->lr, eps = hp->eps, wd = hp->weight_decay;
    double bc1 = 1.0 - pow(b1, (double)t), bc2 = 1.0 - pow(b2, (double)t);
    for (int64_t i = 0; i < n; ++i) {
        double gi = gm[i] * coef;
        m[i] = b1 * m[i] + (1.0 - b1) * gi;
        v[i] = b2 * v[i] + (1.0 - b2) * gi * gi;
        double mhat = m[i] / bc1;
        double vhat = v[i] / bc2;
        theta[i] = theta[i] * (1.0 - lr * wd) - lr * mhat / (sqrt(vhat) + eps);
    }
    return coef;
}

double oracle_layer_step_f64(int64_t n, int32_t R, const uint16_t *const *g,
                             double *theta, double *m, double *v,
                             const oracle_hparams *hp, int64_t t)
{
    double *gm = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!gm)
        return -1.0;
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int32_t r = 0; r < R; ++r)
            s += (double)oracle_bf16_to_f32(g[r][i]);
        gm[i] = s / (double)R;
    }
    double coef = f64_update(n, gm, theta, m, v, hp, t);
    free(gm);
    return coef;
}

double oracle_layer_step_f64_f32g(int64_t n, int32_t R, const float *const *g,
                                  double *theta, double *m, double *v,
                                  const oracle_hparams *hp, int64_t t)
{
    double *gm = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (!gm)
        return -1.0;
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int32_t r = 0; r < R; ++r)
            s += (double)g[r][i];
        gm[i] = s / (double)R;
    }
    double coef = f64_update(n, gm, theta, m, v, hp, t);
    free(gm);
    return coef;
}
