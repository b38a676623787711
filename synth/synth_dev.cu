/* synth_dev.cu — device side of the synthetic-input generator (see synth.h).
 * Same values as synth_host.c, bit for bit.  Also provides a gradient
 * callback for the host-streamed model step that fills the R replica
 * buffers of one unit (this stands in for the backward pass). */
#include <cuda_runtime.h>
#include <math.h>
#include "synth.h"

namespace {

constexpr int kThreads = 256;

__global__ void k_fill_master(float *out, int64_t n, int64_t offset, uint32_t seed, uint32_t unit, float scale)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        out[j] = syn_master_value(seed, unit, (uint64_t)(offset + j), scale);
}

__global__ void k_fill_grad(uint16_t *out, int64_t n, int64_t offset, syn_grad_spec sp,
                            uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        out[j] = syn_grad_bf16(&sp, unit, step, replica, (uint64_t)(offset + j), scale);
}

__global__ void k_fill_grad_f32(float *out, int64_t n, int64_t offset, syn_grad_spec sp,
                                uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        out[j] = syn_grad_value(&sp, unit, step, replica, (uint64_t)(offset + j), scale);
}

__global__ void k_normals(float *out, int64_t n, uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        out[j] = syn_normal(seed, tag, a, b, c, (uint64_t)j);
}

unsigned grid_for(int64_t n)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (n + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)sms * 16;
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    return (unsigned)want;
}

}  // namespace

extern "C" {

typedef struct {
    syn_grad_spec spec;
    int32_t n_units;
    int32_t n_replicas;
    uint32_t step;              /* set by the caller before each model step */
    uint32_t unit_id_base;      /* unit id of unit 0 in the generator's counter */
    const int64_t *unit_numel;  /* host array [n_units] */
    const int32_t *seg_begin;   /* host [n_units+1] or NULL: one segment of scale default_scale */
    const int64_t *seg_offset;  /* host, per segment: offset inside its unit */
    const int64_t *seg_len;     /* host, per segment */
    const float *seg_scale;     /* host, per segment */
    float default_scale;
    int32_t fp32_grads;         /* fill FP32 replicas (values before the BF16 rounding) */
} syn_model_grads;

int syn_dev_fill_master(float *out, int64_t n, int64_t offset, uint32_t seed, uint32_t unit, float scale,
                        cudaStream_t s)
{
    if (n <= 0) return 0;
    k_fill_master<<<grid_for(n), kThreads, 0, s>>>(out, n, offset, seed, unit, scale);
    return (int)cudaGetLastError();
}

int syn_dev_fill_grad(uint16_t *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                      uint32_t unit, uint32_t step, uint32_t replica, float scale, cudaStream_t s)
{
    if (n <= 0) return 0;
    k_fill_grad<<<grid_for(n), kThreads, 0, s>>>(out, n, offset, *sp, unit, step, replica, scale);
    return (int)cudaGetLastError();
}

int syn_dev_fill_grad_f32(float *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                          uint32_t unit, uint32_t step, uint32_t replica, float scale, cudaStream_t s)
{
    if (n <= 0) return 0;
    k_fill_grad_f32<<<grid_for(n), kThreads, 0, s>>>(out, n, offset, *sp, unit, step, replica, scale);
    return (int)cudaGetLastError();
}

int syn_dev_normals(float *out, int64_t n, uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c,
                    cudaStream_t s)
{
    if (n <= 0) return 0;
    k_normals<<<grid_for(n), kThreads, 0, s>>>(out, n, seed, tag, a, b, c);
    return (int)cudaGetLastError();
}

/* Gradient callback for the host-streamed model step: fills the R replicas
 * of unit `layer` for step `g->step`.  Returns 0 or a CUDA error code. */
int syn_dev_grad_fn(void *user, int32_t layer, void *const *replicas, cudaStream_t s)
{
    const syn_model_grads *g = (const syn_model_grads *)user;
    if (!g || layer < 0 || layer >= g->n_units) return -1;
    uint32_t unit = g->unit_id_base + (uint32_t)layer;
    for (int32_t r = 0; r < g->n_replicas; ++r) {
        const int32_t nseg = g->seg_begin ? g->seg_begin[layer + 1] - g->seg_begin[layer] : 1;
        for (int32_t q = 0; q < nseg; ++q) {
            const int32_t k = g->seg_begin ? g->seg_begin[layer] + q : 0;
            const int64_t off = g->seg_begin ? g->seg_offset[k] : 0;
            const int64_t len = g->seg_begin ? g->seg_len[k] : g->unit_numel[layer];
            const float scale = g->seg_begin ? g->seg_scale[k] : g->default_scale;
            int rc = g->fp32_grads
                         ? syn_dev_fill_grad_f32((float *)replicas[r] + off, len, off, &g->spec, unit, g->step,
                                                 (uint32_t)r, scale, s)
                         : syn_dev_fill_grad((uint16_t *)replicas[r] + off, len, off, &g->spec, unit, g->step,
                                             (uint32_t)r, scale, s);
            if (rc) return rc;
        }
    }
    return 0;
}

/* Gradient callback that copies pre-generated replicas from a device pool
 * (benchmarking the streamed step without timing the generator): unit l at
 * step t gets pool entry (l + t) % n_pool, replicas r = 0..R-1. */
typedef struct {
    int32_t n_replicas;
    int32_t n_pool;
    uint32_t step;
    int32_t fp32_grads;          /* replicas are FP32 (4 bytes per value) */
    const int64_t *unit_numel;   /* host array [n_units] */
    void *const *pool;           /* host array [n_pool * n_replicas] of device pointers */
} syn_pool_grads;

int syn_dev_pool_grad_fn(void *user, int32_t layer, void *const *replicas, cudaStream_t s)
{
    const syn_pool_grads *p = (const syn_pool_grads *)user;
    if (!p || layer < 0 || p->n_pool < 1) return -1;
    const int k = (int)(((uint32_t)layer + p->step) % (uint32_t)p->n_pool);
    const size_t bytes = (size_t)p->unit_numel[layer] * (p->fp32_grads ? 4 : 2);
    for (int32_t r = 0; r < p->n_replicas; ++r) {
        cudaError_t e = cudaMemcpyAsync(replicas[r], p->pool[k * p->n_replicas + r], bytes,
                                        cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return (int)e;
    }
    return 0;
}

}  // extern "C"
