/*
 * oracle.h — the plain CPU oracle of the per-layer mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE ONLY.  This code is the independent, slow, obviously
 * correct restatement of what the GPU path computes.  Only the tests, the smoke
 * check and the CPU-baseline / reference legs of the benchmark may load it.  The
 * product library never includes this header, never links this code and never
 * falls back to it.
 *
 * What it follows (pages are cited by title and section):
 *  - "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs",
 *    Prerequisites, on the 16N-byte training state of mixed-precision Adam:
 *    BF16 compute weights and gradients (2N + 2N bytes), an FP32 master copy
 *    (4N) and FP32 first and second Adam moments (8N).
 *  - same page, Core method and Method steps: one authoritative FP32 master
 *    and (m_l, v_l) per layer, updated once per iteration from the gradient
 *    that the R ranks' layer gradients were reduced to on the GPU; the updated
 *    master is cast FP32 -> BF16 for the next delivery of the layer.
 *  - "An Efficient Heterogeneous Co-Design for Fine-Tuning on a Single GPU"
 *    (SlideFormer), section 2.2: the FP32 -> BF16 conversion of the updated
 *    weights.
 *  - "Accelerating the Training of Large Language Models using Efficient
 *    Activation Rematerialization and Optimal Hybrid Parallelism", section 3,
 *    memory footprint item 2: 12 = 4 + 4 + 4 bytes per parameter of FP32
 *    master weights and two FP32 Adam states.
 *
 * The pages name the optimizer ("Adam", "LayerAdam") but print no update
 * equation.  The reading taken here is AdamW with bias correction in its
 * common library form (Loshchilov & Hutter's decoupled weight decay applied
 * as theta *= 1 - lr*wd before the Adam term; Kingma & Ba's bias-corrected
 * moments with eps added after the square root of the corrected second
 * moment), the replicas reduced to their mean, an optional global clip of the
 * mean gradient's L2 norm (coef = min(1, c / (norm + 1e-6))), and BF16 by
 * round-to-nearest-even.
 *
 * Precision: every per-element operation is one FP32 operation in the order
 * written in oracle.c (compiled with -ffp-contract=off, no fast-math); the
 * per-step scalars and the clip norm are formed in double.  The *_f64
 * functions redo the whole step in double as a brute-force cross-check.
 */
#ifndef SLIDE_ORACLE_H
#define SLIDE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    float max_grad_norm; /* <= 0: no clip */
} oracle_hparams;

/* Per-step FP32 scalars derived in double from the FP32 hyper-parameters and
 * the 1-based step index t (bias corrections 1 - beta^t). */
typedef struct {
    float beta1, one_minus_beta1, beta2, one_minus_beta2;
    float decay;       /* 1 - lr*wd */
    float step_size;   /* lr / (1 - beta1^t) */
    float bc2_sqrt;    /* sqrt(1 - beta2^t) */
    float eps;
} oracle_step_scalars;

/* BF16 <-> FP32.  bf16 -> f32 is exact; f32 -> bf16 rounds to nearest even,
 * keeps infinities and turns NaN into a quiet NaN of the same sign. */
float    oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16_rne(float x);

/* Element-wise over arrays (for tests that round many values at once). */
void oracle_f32_to_bf16_rne_array(int64_t n, const float *x, uint16_t *out);
void oracle_bf16_to_f32_array(int64_t n, const uint16_t *h, float *out);

void oracle_step_scalars_for(const oracle_hparams *hp, int64_t t, oracle_step_scalars *out);

/* a1: gm[i] = (sum_r g[r][i], summed in FP32 in replica order) / R */
void oracle_grad_mean(int64_t n, int32_t R, const uint16_t *const *g, float *gm);

/* a1 with FP32 gradient replicas (FP32 gradient accumulation, "Accelerating
 * the Training of Large Language Models ...", section 3 and the experimental
 * setup: BF16 training with FP32 gradients): the same rule, FP32 sum in
 * replica order, divided by R. */
void oracle_grad_mean_f32(int64_t n, int32_t R, const float *const *g, float *gm);

/* a2: sum of gm[i]^2 in double, index order; coef = min(1, c/(sqrt(s)+1e-6)) */
double oracle_grad_sqnorm(int64_t n, const float *gm);
float  oracle_clip_coef(double sqnorm, float max_norm);

/* a3..a5 on n elements with a given (already decided) clip coefficient:
 * g = gm[i]*coef when coef != 1; AdamW on theta, m, v in place; w = bf16(theta). */
void oracle_adamw_update(int64_t n, const float *gm, float coef,
                         float *theta, float *m, float *v, uint16_t *w,
                         const oracle_hparams *hp, int64_t t);

/* One whole layer step: a1 + a2 (if max_grad_norm > 0) + a3..a5.
 * Returns the clip coefficient it used (1 when the clip is off); -1 on
 * allocation failure (nothing is modified then). */
float oracle_layer_step(int64_t n, int32_t R, const uint16_t *const *g,
                        float *theta, float *m, float *v, uint16_t *w,
                        const oracle_hparams *hp, int64_t t);

/* One whole layer step with FP32 gradient replicas (see oracle_grad_mean_f32). */
float oracle_layer_step_f32g(int64_t n, int32_t R, const float *const *g,
                             float *theta, float *m, float *v, uint16_t *w,
                             const oracle_hparams *hp, int64_t t);

/* Float64 brute force of the same step: theta, m, v in double, the bias
 * corrections applied to the moments (m_hat = m/(1-b1^t), v_hat = v/(1-b2^t))
 * and the update theta = theta*(1 - lr*wd) - lr*m_hat/(sqrt(v_hat)+eps).
 * Returns the clip coefficient (1 when off), -1 on allocation failure. */
/* Threads the element loops use (1 unless built with -fopenmp, which is for
 * the all-core timing only). */
int32_t oracle_threads(void);

double oracle_layer_step_f64(int64_t n, int32_t R, const uint16_t *const *g,
                             double *theta, double *m, double *v,
                             const oracle_hparams *hp, int64_t t);

/* The float64 brute force with FP32 gradient replicas. */
double oracle_layer_step_f64_f32g(int64_t n, int32_t R, const float *const *g,
                                  double *theta, double *m, double *v,
                                  const oracle_hparams *hp, int64_t t);

#ifdef __cplusplus
}
#endif
#endif
