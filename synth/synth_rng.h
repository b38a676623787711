/*
 * synth_rng.h — seeded, counter-based synthetic inputs, bit-identical on the
 * host (C) and on the GPU (CUDA).
 *
 * This is the one module that both the CUDA path's tests/benchmarks and the
 * oracle's inputs come from.  It holds none of the optimizer step's
 * arithmetic: only a random-number generator and the shaping of its output
 * into the workloads' input distributions.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3", SC'11): a 128-bit counter and a 64-bit key
 * go through 10 rounds of two 32x32->64-bit multiplies (multipliers
 * 0xD2511F53, 0xCD9E8D57) and xors, the key bumped by the Weyl constants
 * 0x9E3779B9, 0xBB67AE85 between rounds.
 *
 * Normals: Box-Muller on two 24-bit uniforms in (0, 1].  The logarithm and
 * sine/cosine are this file's own: argument reduction to a power of two
 * times f in [sqrt(1/2), sqrt(2)] with ln f = 2*atanh((f-1)/(f+1)) as an odd
 * series, and quarter-turn reduction with Taylor polynomials of sin and cos
 * on [-pi/4, pi/4].  Every floating-point step is one IEEE-754 binary32
 * operation written out explicitly (fma where an fma is meant), so the host
 * build (compiled with -ffp-contract=off) and the device build produce the
 * same bits.  They are a few ulp off the correctly rounded functions, which
 * only shapes the input distribution and is the same on both sides.
 */
#ifndef SYNTH_RNG_H
#define SYNTH_RNG_H
#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_HD static __host__ __device__ __forceinline__
#else
#include <math.h>
#define SYN_HD static inline
#endif

#if defined(__CUDA_ARCH__)
#define SYN_FMA(a, b, c) __fmaf_rn((a), (b), (c))
#define SYN_MUL(a, b) __fmul_rn((a), (b))
#define SYN_ADD(a, b) __fadd_rn((a), (b))
#define SYN_SUB(a, b) __fsub_rn((a), (b))
#define SYN_DIV(a, b) __fdiv_rn((a), (b))
#define SYN_SQRT(a) __fsqrt_rn((a))
#define SYN_FLOOR(a) floorf((a))
#else
#define SYN_FMA(a, b, c) fmaf((a), (b), (c))
#define SYN_MUL(a, b) ((a) * (b))
#define SYN_ADD(a, b) ((a) + (b))
#define SYN_SUB(a, b) ((a) - (b))
#define SYN_DIV(a, b) ((a) / (b))
#define SYN_SQRT(a) sqrtf((a))
#define SYN_FLOOR(a) floorf((a))
#endif

/* Stream tags: which input a stream of numbers feeds. */
enum {
    SYN_TAG_MASTER = 0,  /* initial FP32 master weights          */
    SYN_TAG_GRAD = 1,    /* gradient normals                     */
    SYN_TAG_CHI = 2,     /* normals of the chi-square denominator */
    SYN_TAG_ZERO = 3,    /* uniforms deciding exact-zero entries  */
    SYN_TAG_SCALE = 4,   /* uniforms of per-tensor scales         */
    SYN_TAG_MOMENT = 5   /* uniforms / normals for non-zero m, v  */
};

/* Gradient distributions. */
enum {
    SYN_GRAD_NORMAL = 0,   /* scale * N(0,1)                                  */
    SYN_GRAD_STUDENT3 = 1  /* scale * Z / sqrt(chi2_3 / 3), exact zero w.p. zero_prob */
};

typedef struct {
    uint32_t seed;
    int32_t kind;     /* SYN_GRAD_* */
    float zero_prob;  /* SYN_GRAD_STUDENT3 only */
    float pad_;
} syn_grad_spec;

SYN_HD uint32_t syn_mulhi(uint32_t a, uint32_t b)
{
#if defined(__CUDA_ARCH__)
    return __umulhi(a, b);
#else
    return (uint32_t)(((uint64_t)a * (uint64_t)b) >> 32);
#endif
}

/* Philox4x32 with 10 rounds. */
SYN_HD void syn_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint32_t hi0 = syn_mulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
        uint32_t hi1 = syn_mulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* The 4 words of block j of stream (seed, tag, a, b, c). */
SYN_HD void syn_block(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c,
                      uint64_t j, uint32_t out[4])
{
    uint32_t ctr[4], key[2];
    ctr[0] = (uint32_t)j;
    ctr[1] = a ^ ((uint32_t)(j >> 32) << 24);
    ctr[2] = b;
    ctr[3] = c;
    key[0] = seed;
    key[1] = tag;
    syn_philox4x32_10(ctr, key, out);
}

/* 24-bit uniform in (0, 1]: exact in binary32. */
SYN_HD float syn_u01(uint32_t x)
{
    return (float)((x >> 8) + 1u) * 5.9604644775390625e-08f; /* 2^-24 */
}

SYN_HD uint32_t syn_f2u(float f)
{
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    union { float f; uint32_t u; } c;
    c.f = f;
    return c.u;
#endif
}

SYN_HD float syn_u2f(uint32_t u)
{
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    union { float f; uint32_t u; } c;
    c.u = u;
    return c.f;
#endif
}

/* Natural log for x in (0, 1] (normal binary32 only, which the uniforms are). */
SYN_HD float syn_log01(float x)
{
    uint32_t u = syn_f2u(x);
    int32_t e = (int32_t)((u >> 23) & 0xffu) - 127;
    float f = syn_u2f((u & 0x007fffffu) | 0x3f800000u); /* [1, 2) */
    if (f > 1.41421356f) {
        f = SYN_MUL(f, 0.5f);
        e += 1;
    }
    float num = SYN_SUB(f, 1.0f);
    float den = SYN_ADD(f, 1.0f);
    float s = SYN_DIV(num, den);
    float s2 = SYN_MUL(s, s);
    float p = 0.111111112f;               /* 1/9 */
    p = SYN_FMA(p, s2, 0.142857149f);     /* 1/7 */
    p = SYN_FMA(p, s2, 0.2f);             /* 1/5 */
    p = SYN_FMA(p, s2, 0.333333343f);     /* 1/3 */
    p = SYN_FMA(p, s2, 1.0f);
    float two_s = SYN_MUL(s, 2.0f);
    float lnf = SYN_MUL(two_s, p);
    return SYN_FMA((float)e, 0.693147182f, lnf);
}

/* sin(2*pi*x) and cos(2*pi*x) for x in [0, 1]. */
SYN_HD void syn_sincos_2pi(float x, float *sn, float *cs)
{
    float y = SYN_MUL(x, 4.0f);                 /* quarter turns, exact */
    float kf = SYN_FLOOR(SYN_ADD(y, 0.5f));
    float r = SYN_SUB(y, kf);                   /* [-1/2, 1/2] */
    int k = (int)kf & 3;
    float a = SYN_MUL(r, 1.57079637f);          /* [-pi/4, pi/4] */
    float a2 = SYN_MUL(a, a);
    /* sin a = a(1 - a^2/6 + a^4/120 - a^6/5040 + a^8/362880) */
    float ps = 2.75573188e-06f;
    ps = SYN_FMA(ps, a2, -1.98412701e-04f);
    ps = SYN_FMA(ps, a2, 8.33333377e-03f);
    ps = SYN_FMA(ps, a2, -1.66666672e-01f);
    ps = SYN_FMA(ps, a2, 1.0f);
    float s = SYN_MUL(a, ps);
    /* cos a = 1 - a^2/2 + a^4/24 - a^6/720 + a^8/40320 - a^10/3628800 */
    float pc = -2.75573188e-07f;
    pc = SYN_FMA(pc, a2, 2.48015876e-05f);
    pc = SYN_FMA(pc, a2, -1.38888892e-03f);
    pc = SYN_FMA(pc, a2, 4.16666679e-02f);
    pc = SYN_FMA(pc, a2, -0.5f);
    float c = SYN_FMA(pc, a2, 1.0f);
    switch (k) {
    case 0: *sn = s;  *cs = c;  break;
    case 1: *sn = c;  *cs = -s; break;
    case 2: *sn = -s; *cs = -c; break;
    default: *sn = -c; *cs = s; break;
    }
}

/* Box-Muller pair from two words. */
SYN_HD void syn_box_muller(uint32_t w0, uint32_t w1, float *z0, float *z1)
{
    float u1 = syn_u01(w0), u2 = syn_u01(w1);
    float l = syn_log01(u1);
    float rad = SYN_SQRT(SYN_MUL(l, -2.0f));
    float sn, cs;
    syn_sincos_2pi(u2, &sn, &cs);
    *z0 = SYN_MUL(rad, cs);
    *z1 = SYN_MUL(rad, sn);
}

/* The 4 standard normals of block j. */
SYN_HD void syn_normal4(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c,
                        uint64_t j, float z[4])
{
    uint32_t w[4];
    syn_block(seed, tag, a, b, c, j, w);
    syn_box_muller(w[0], w[1], &z[0], &z[1]);
    syn_box_muller(w[2], w[3], &z[2], &z[3]);
}

/* Standard normal number i of stream (seed, tag, a, b, c). */
SYN_HD float syn_normal(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c, uint64_t i)
{
    float z[4];
    syn_normal4(seed, tag, a, b, c, i >> 2, z);
    return z[i & 3];
}

/* Uniform number i in (0, 1] of stream (seed, tag, a, b, c). */
SYN_HD float syn_uniform(uint32_t seed, uint32_t tag, uint32_t a, uint32_t b, uint32_t c, uint64_t i)
{
    uint32_t w[4];
    syn_block(seed, tag, a, b, c, i >> 2, w);
    return syn_u01(w[i & 3]);
}

/* binary32 -> bf16 bits, round to nearest even (inputs are finite here). */
SYN_HD uint16_t syn_to_bf16(float x)
{
    uint32_t u = syn_f2u(x);
    uint32_t keep = u >> 16, rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

/* Initial master weight i of a unit: scale * N(0,1). */
SYN_HD float syn_master_value(uint32_t seed, uint32_t unit, uint64_t i, float scale)
{
    return SYN_MUL(syn_normal(seed, SYN_TAG_MASTER, unit, 0u, 0u, i), scale);
}

/* Gradient value i of (unit, step, replica), before the BF16 rounding. */
SYN_HD float syn_grad_value(const syn_grad_spec *sp, uint32_t unit, uint32_t step,
                            uint32_t replica, uint64_t i, float scale)
{
    float z = syn_normal(sp->seed, SYN_TAG_GRAD, unit, step, replica, i);
    if (sp->kind == SYN_GRAD_STUDENT3) {
        float q[4];
        syn_normal4(sp->seed, SYN_TAG_CHI, unit, step, replica, i, q);
        float chi = SYN_MUL(q[0], q[0]);
        chi = SYN_FMA(q[1], q[1], chi);
        chi = SYN_FMA(q[2], q[2], chi);
        float den = SYN_SQRT(SYN_DIV(chi, 3.0f));
        z = SYN_DIV(z, den);
        float u = syn_uniform(sp->seed, SYN_TAG_ZERO, unit, step, replica, i);
        if (u <= sp->zero_prob)
            return 0.0f;
    }
    return SYN_MUL(z, scale);
}

SYN_HD uint16_t syn_grad_bf16(const syn_grad_spec *sp, uint32_t unit, uint32_t step,
                              uint32_t replica, uint64_t i, float scale)
{
    return syn_to_bf16(syn_grad_value(sp, unit, step, replica, i, scale));
}

#endif
