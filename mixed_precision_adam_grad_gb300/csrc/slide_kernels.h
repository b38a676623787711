// slide_kernels.h — internal interface between the C ABI (slide_api.cu), the
// streaming engine (stream_engine.cu) and the kernels
// (grad_reduce_adamw_cast.cu).  Not installed; not part of the ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace slide {

constexpr int kMaxReplicas = 8;
constexpr int kMaxPartials = 4096;  // per-block partial sums of the clip pre-pass

// Per-step FP32 scalars of the AdamW update (formed in double on the host,
// rounded once; see adam_scalars_for in slide_api.cu).
struct AdamScalars {
    float beta1, one_minus_beta1, beta2, one_minus_beta2;
    float decay;      // 1 - lr*wd
    float step_size;  // lr / (1 - beta1^t)
    float bc2_sqrt;   // sqrt(1 - beta2^t)
    float eps;
};

struct ReplicaPtrs {
    const void *p[kMaxReplicas];
};

// Device scratch of one layer's clip reduction.
struct ClipScratch {
    double *partials;  // [kMaxPartials]
    float *coef;       // last coefficient used (written by block 0)
    unsigned *status;  // bit 0: a non-finite mean gradient was seen
};

// Replicas are BF16 (uint16_t bit patterns) unless f32_grads, then FP32.
//
// Clip pre-pass: per-block partial sums of the squared replica mean into
// scratch.partials; returns the number of partials written via *n_partials.
cudaError_t launch_grad_sqnorm(const ReplicaPtrs &g, int R, int64_t n, const ClipScratch &scratch,
                               int *n_partials, int device, cudaStream_t stream, bool f32_grads = false);

// Fused step.  When max_norm > 0 the kernel reduces the n_partials partial
// sums (in a fixed order, identically in every block) to the clip coefficient.
// status may be NULL; when check_finite is set and status is not NULL a
// non-finite mean gradient sets bit 0 of *status.  behind_prepass (clip only):
// the last operation enqueued on `stream` is this step's clip pre-pass, so the
// step is launched with programmatic serialisation and overlaps the
// pre-pass's end; it reads the partials only after the pre-pass has ended.
cudaError_t launch_grad_reduce_adamw_cast(const ReplicaPtrs &g, int R, int64_t n, float *theta,
                                          float *m, float *v, uint16_t *w, const AdamScalars &s,
                                          const ClipScratch *clip, int n_partials, float max_norm,
                                          bool check_finite, int device, cudaStream_t stream,
                                          bool test_stall = false, bool f32_grads = false,
                                          bool behind_prepass = false);

// w[i] = bf16_rne(src[i]) (used when a caller overwrites a master copy).
cudaError_t launch_cast_bf16(const float *src, uint16_t *w, int64_t n, cudaStream_t stream);

// Zero `bytes` (a multiple of 16, 16-byte aligned) of device-accessible memory
// (device memory, or pinned host memory through its device address) on
// `device`, which must be current; the grid is sized from its SM count.
cudaError_t launch_fill_zero(void *p, size_t bytes, int device, cudaStream_t stream);

// Load every kernel that a BF16-replica step without the non-finite check may
// launch on `device` (the current device), and fill the per-device launch
// caches, so that no later step of that kind loads code or queries the device.
cudaError_t preload_bf16_step_kernels(int device);

}  // namespace slide
