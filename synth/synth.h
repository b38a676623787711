/*
 * synth.h — C entry points of the seeded synthetic-input generator
 * (host library libsynth_host.so: plain C + OpenMP; device library
 * libsynth_dev.so: CUDA).  Both produce the same bits for the same
 * (seed, unit, step, replica, index); see synth_rng.h for the definitions.
 *
 * Indices are positions inside a unit (a layer's flat parameter vector);
 * `offset` is the index of out[0], so a unit can be filled tensor by tensor
 * with a per-tensor scale and still match element-wise gathers.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>
#include "synth_rng.h"

#ifdef __cplusplus
extern "C" {
#endif

/* host */
void syn_host_fill_master(float *out, int64_t n, int64_t offset, uint32_t seed, uint32_t unit, float scale);
void syn_host_fill_grad(uint16_t *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                        uint32_t unit, uint32_t step, uint32_t replica, float scale);
void syn_host_gather_master(float *out, const int64_t *idx, int64_t n, uint32_t seed, uint32_t unit, float scale);
void syn_host_gather_grad(uint16_t *out, const int64_t *idx, int64_t n, const syn_grad_spec *sp,
                          uint32_t unit, uint32_t step, uint32_t replica, float scale);
void syn_host_fill_grad_f32(float *out, int64_t n, int64_t offset, const syn_grad_spec *sp,
                            uint32_t unit, uint32_t step, uint32_t replica, float scale);
void syn_host_gather_grad_f32(float *out, const int64_t *idx, int64_t n, const syn_grad_spec *sp,
                              uint32_t unit, uint32_t step, uint32_t replica, float scale);
float syn_host_uniform(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c, uint64_t i);
void syn_host_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
void syn_host_normals(float *out, int64_t n, uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c);

#ifdef __cplusplus
}
#endif
#endif
