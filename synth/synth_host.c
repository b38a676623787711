/* synth_host.c — host side of the synthetic-input generator (see synth.h).
 * Build: cc -std=c99 -O2 -ffp-contract=off -fopenmp -fPIC -shared -lm.
 * Counter-based, so the OpenMP split does not change any value. */
#include "synth.h"

void syn_host_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    syn_philox4x32_10(ctr, key, out);
}

float syn_host_uniform(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c, uint64_t i)
{
    return syn_uniform(seed, tag, a, b, c, i);
}

void syn_host_normals(float *out, int64_t n, uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = syn_normal(seed, tag, a, b, c, (uint64_t)i);
}

void syn_host_fill_master(float *out, int64_t n, int64_t offset, uint32_t seed, uint32_t unit, float scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_master_value(seed, unit, (uint64_t)(offset + j), scale);
}

void syn_host_fill_grad(uint16_t *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                        uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    syn_grad_spec s = *sp;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_grad_bf16(&s, unit, step, replica, (uint64_t)(offset + j), scale);
}

void syn_host_gather_master(float *out, const int64_t *idx, int64_t n, uint32_t seed, uint32_t unit, float scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_master_value(seed, unit, (uint64_t)idx[j], scale);
}

void syn_host_gather_grad(uint16_t *out, const int64_t *idx, int64_t n, const syn_grad_spec *sp,
                          uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    syn_grad_spec s = *sp;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_grad_bf16(&s, unit, step, replica, (uint64_t)idx[j], scale);
}

void syn_host_fill_grad_f32(float *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                            uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    syn_grad_spec s = *sp;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_grad_value(&s, unit, step, replica, (uint64_t)(offset + j), scale);
}

void syn_host_gather_grad_f32(float *out, const int64_t *idx, int64_t n, const syn_grad_spec *sp,
                              uint32_t unit, uint32_t step, uint32_t replica, float scale)
{
    syn_grad_spec s = *sp;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j)
        out[j] = syn_grad_value(&s, unit, step, replica, (uint64_t)idx[j], scale);
}
