// grad_reduce_adamw_cast.cu — the fused per-layer optimizer step on sm_103a.
//
// One pass over HBM per step: read the R BF16 gradient replicas and the FP32
// master, m and v once; write master, m, v and the BF16 compute copy once.
// This is the LayerAdam step of "SlideDP: Scaling Host-Resident LLM
// Fine-Tuning Across Multiple GPUs" (Core method: GPU-side reduction of the
// R ranks' gradients, one aggregated Adam update per layer on the FP32
// master and moments, FP32 -> BF16 cast of the result), moved from host
// cores onto the GPU and fused into one kernel.
//
// The step is elementwise and bandwidth-bound ((26 + 2R) bytes and ~20 FP32
// operations per parameter), so no tensor cores: each thread moves 16-byte
// vectors (8 parameters) of every stream, the grid is persistent (SM count x
// resident blocks) with a grid-stride loop, and UNROLL vectors per thread are
// loaded before any is used to keep enough bytes in flight.
//
// Arithmetic: one IEEE FP32 operation per line of the update, explicit
// __f*_rn intrinsics so nothing is contracted into an FMA, IEEE sqrt and
// division, BF16 by round-to-nearest-even.  The replica sum is in replica
// order; the mean divides by R (a multiply by the exact inverse when R is a
// power of two).
//
// The optional global clip needs the norm of the whole layer's mean gradient
// before any element is updated, so it is a separate pre-pass (k_grad_sqnorm)
// that re-reads the replicas (2R bytes per parameter) and writes one
// double-precision partial per block; the fused kernel turns the partials
// into the coefficient in its prologue, in the same fixed order in every
// block, so every block uses the same bits.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "slide_kernels.h"

namespace slide {
namespace {

constexpr int kThreads = 256;

struct KArgs {
    ReplicaPtrs g;
    float4 *theta;
    float4 *m;
    float4 *v;
    uint4 *w;
    int64_t n;
    AdamScalars s;
    const double *partials;
    int n_partials;
    float max_norm;
    float *coef_out;
    unsigned *status;
};

__device__ __forceinline__ float bf16_lo(uint32_t word) { return __uint_as_float(word << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t word) { return __uint_as_float(word & 0xffff0000u); }

template <int R>
__device__ __forceinline__ float replica_mean(const float (&x)[R])
{
    float s = x[0];
#pragma unroll
    for (int r = 1; r < R; ++r)
        s = __fadd_rn(s, x[r]);
    if constexpr ((R & (R - 1)) == 0)
        return __fmul_rn(s, 1.0f / (float)R);  // exact: R is a power of two
    else
        return __fdiv_rn(s, (float)R);
}

// The AdamW update of one parameter (order and rounding as in slide.h).
__device__ __forceinline__ void adamw_one(float g, float &th, float &m, float &v, uint16_t &w,
                                          const AdamScalars &s)
{
    float m_old = __fmul_rn(m, s.beta1);
    float m_new = __fmul_rn(s.one_minus_beta1, g);
    float mi = __fadd_rn(m_old, m_new);

    float v_old = __fmul_rn(v, s.beta2);
    float g2 = __fmul_rn(g, g);
    float v_new = __fmul_rn(s.one_minus_beta2, g2);
    float vi = __fadd_rn(v_old, v_new);

    float t = __fmul_rn(th, s.decay);
    float root = __fsqrt_rn(vi);
    float den = __fdiv_rn(root, s.bc2_sqrt);
    den = __fadd_rn(den, s.eps);
    float ratio = __fdiv_rn(mi, den);
    float delta = __fmul_rn(s.step_size, ratio);
    t = __fsub_rn(t, delta);

    m = mi;
    v = vi;
    th = t;
    w = __bfloat16_as_ushort(__float2bfloat16_rn(t));
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint16_t lo, uint16_t hi)
{
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Deterministic clip coefficient from the per-block partials: warp 0 sums
// lane-strided in double, then a fixed shuffle-down tree; lane 0's result.
__device__ __forceinline__ float clip_coef_from_partials(const double *partials, int n_partials,
                                                          float max_norm)
{
    __shared__ float s_coef;
    if (threadIdx.x < 32) {
        double acc = 0.0;
        for (int i = threadIdx.x; i < n_partials; i += 32)
            acc += partials[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            acc += __shfl_down_sync(0xffffffffu, acc, off);
        if (threadIdx.x == 0) {
            double norm = sqrt(acc);
            double c = (double)max_norm / (norm + 1e-6);
            if (c > 1.0)
                c = 1.0;
            s_coef = (float)c;
        }
    }
    __syncthreads();
    return s_coef;
}

template <int R, bool CLIP, bool CHECK, int UNROLL>
__global__ void __launch_bounds__(kThreads) k_grad_reduce_adamw_cast(KArgs a)
{
    float coef = 1.0f;
    if constexpr (CLIP) {
        coef = clip_coef_from_partials(a.partials, a.n_partials, a.max_norm);
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.coef_out)
            *a.coef_out = coef;
    }
    const AdamScalars s = a.s;
    const int64_t nvec = a.n >> 3;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    bool bad = false;

    for (int64_t k0 = tid; k0 < nvec; k0 += stride * UNROLL) {
        uint4 gv[UNROLL][R];
        float4 th[UNROLL][2], mv[UNROLL][2], vv[UNROLL][2];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t k = k0 + (int64_t)u * stride;
            if (k < nvec) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    gv[u][r] = __ldcs(reinterpret_cast<const uint4 *>(a.g.p[r]) + k);
                th[u][0] = __ldcs(a.theta + 2 * k);
                th[u][1] = __ldcs(a.theta + 2 * k + 1);
                mv[u][0] = __ldcs(a.m + 2 * k);
                mv[u][1] = __ldcs(a.m + 2 * k + 1);
                vv[u][0] = __ldcs(a.v + 2 * k);
                vv[u][1] = __ldcs(a.v + 2 * k + 1);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t k = k0 + (int64_t)u * stride;
            if (k < nvec) {
                float tt[8] = {th[u][0].x, th[u][0].y, th[u][0].z, th[u][0].w,
                               th[u][1].x, th[u][1].y, th[u][1].z, th[u][1].w};
                float mm[8] = {mv[u][0].x, mv[u][0].y, mv[u][0].z, mv[u][0].w,
                               mv[u][1].x, mv[u][1].y, mv[u][1].z, mv[u][1].w};
                float vq[8] = {vv[u][0].x, vv[u][0].y, vv[u][0].z, vv[u][0].w,
                               vv[u][1].x, vv[u][1].y, vv[u][1].z, vv[u][1].w};
                uint16_t ww[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float x[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = (&gv[u][r].x)[e >> 1];
                        x[r] = (e & 1) ? bf16_hi(word) : bf16_lo(word);
                    }
                    float g = replica_mean<R>(x);
                    if constexpr (CHECK)
                        bad |= !isfinite(g);
                    if constexpr (CLIP)
                        g = __fmul_rn(g, coef);
                    adamw_one(g, tt[e], mm[e], vq[e], ww[e], s);
                }
                __stcs(a.theta + 2 * k, make_float4(tt[0], tt[1], tt[2], tt[3]));
                __stcs(a.theta + 2 * k + 1, make_float4(tt[4], tt[5], tt[6], tt[7]));
                __stcs(a.m + 2 * k, make_float4(mm[0], mm[1], mm[2], mm[3]));
                __stcs(a.m + 2 * k + 1, make_float4(mm[4], mm[5], mm[6], mm[7]));
                __stcs(a.v + 2 * k, make_float4(vq[0], vq[1], vq[2], vq[3]));
                __stcs(a.v + 2 * k + 1, make_float4(vq[4], vq[5], vq[6], vq[7]));
                __stcs(a.w + k, make_uint4(pack_bf16x2(ww[0], ww[1]), pack_bf16x2(ww[2], ww[3]),
                                           pack_bf16x2(ww[4], ww[5]), pack_bf16x2(ww[6], ww[7])));
            }
        }
    }

    // Ragged tail: the last n % 8 parameters, one per thread, scalar accesses.
    const int64_t tail0 = nvec << 3;
    if (tid < a.n - tail0) {
        const int64_t i = tail0 + tid;
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint16_t h = reinterpret_cast<const uint16_t *>(a.g.p[r])[i];
            x[r] = __uint_as_float((uint32_t)h << 16);
        }
        float g = replica_mean<R>(x);
        if constexpr (CHECK)
            bad |= !isfinite(g);
        if constexpr (CLIP)
            g = __fmul_rn(g, coef);
        float *thp = reinterpret_cast<float *>(a.theta);
        float *mp = reinterpret_cast<float *>(a.m);
        float *vp = reinterpret_cast<float *>(a.v);
        float t = thp[i], mm = mp[i], vq = vp[i];
        uint16_t ww;
        adamw_one(g, t, mm, vq, ww, s);
        thp[i] = t;
        mp[i] = mm;
        vp[i] = vq;
        reinterpret_cast<uint16_t *>(a.w)[i] = ww;
    }
    if constexpr (CHECK) {
        if (bad && a.status)
            atomicOr(a.status, 1u);
    }
}

// Error-free transformation of a sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    float ea = __fsub_rn(a, __fsub_rn(s, bb));
    float eb = __fsub_rn(b, bb);
    e = __fadd_rn(ea, eb);
}

// Accumulates the exact squares of FP32 values in FP32 pieces: the rounded
// square p = x*x goes into a TwoSum-compensated (hi, lo) pair and the exact
// product error fma(x, x, -p) into err, so hi + lo + err carries the sum with
// about twice FP32's precision and no FP64 work per element.
struct SqAcc {
    float hi = 0.f, lo = 0.f, err = 0.f;
    __device__ __forceinline__ void add(float x)
    {
        float p = __fmul_rn(x, x);
        float e = __fmaf_rn(x, x, -p);
        float s, c;
        two_sum(hi, p, s, c);
        hi = s;
        lo = __fadd_rn(lo, c);
        err = __fadd_rn(err, e);
    }
};

struct SqArgs {
    ReplicaPtrs g;
    int64_t n;
    double *partials;
};

template <int R, int UNROLL>
__global__ void __launch_bounds__(kThreads) k_grad_sqnorm(SqArgs a)
{
    const int64_t nvec = a.n >> 3;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    SqAcc acc;
    for (int64_t k0 = tid; k0 < nvec; k0 += stride * UNROLL) {
        uint4 gv[UNROLL][R];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t k = k0 + (int64_t)u * stride;
            if (k < nvec) {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    gv[u][r] = __ldcs(reinterpret_cast<const uint4 *>(a.g.p[r]) + k);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t k = k0 + (int64_t)u * stride;
            if (k < nvec) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float x[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = (&gv[u][r].x)[e >> 1];
                        x[r] = (e & 1) ? bf16_hi(word) : bf16_lo(word);
                    }
                    acc.add(replica_mean<R>(x));
                }
            }
        }
    }
    const int64_t tail0 = nvec << 3;
    if (tid < a.n - tail0) {
        const int64_t i = tail0 + tid;
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint16_t h = reinterpret_cast<const uint16_t *>(a.g.p[r])[i];
            x[r] = __uint_as_float((uint32_t)h << 16);
        }
        acc.add(replica_mean<R>(x));
    }

    // Block reduction in double, fixed order: shuffle-down tree per warp,
    // then warp 0 over the warps' results.
    double d = (double)acc.hi + (double)acc.lo + (double)acc.err;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        d += __shfl_down_sync(0xffffffffu, d, off);
    __shared__ double s_warp[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        s_warp[warp] = d;
    __syncthreads();
    if (warp == 0) {
        d = lane < kThreads / 32 ? s_warp[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            d += __shfl_down_sync(0xffffffffu, d, off);
        if (lane == 0)
            a.partials[blockIdx.x] = d;
    }
}

// Resident blocks per SM of a kernel, cached per (kernel, device).
template <auto Kernel>
int blocks_per_sm(int device)
{
    static int cache[64] = {0};
    if (device < 0 || device >= 64)
        return 1;
    if (cache[device] == 0) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, Kernel, kThreads, 0) != cudaSuccess || b < 1)
            b = 1;
        cache[device] = b;
    }
    return cache[device];
}

int sm_count(int device)
{
    static int cache[64] = {0};
    if (device < 0 || device >= 64)
        return 1;
    if (cache[device] == 0) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || c < 1)
            c = 1;
        cache[device] = c;
    }
    return cache[device];
}

// Persistent grid: SMs x resident blocks, fewer if there is less work.
template <auto Kernel>
unsigned grid_for(int device, int64_t n, int cap)
{
    const int64_t work = ((n >> 3) + kThreads - 1) / kThreads;  // blocks of 8-wide vectors
    int64_t g = (int64_t)sm_count(device) * blocks_per_sm<Kernel>(device);
    if (g > work)
        g = work;
    if (g > cap)
        g = cap;
    if (g < 1)
        g = 1;
    return (unsigned)g;
}

constexpr int kUnrollStep = 2;
constexpr int kUnrollSq = 2;

template <int R, bool CLIP, bool CHECK>
cudaError_t launch_step_r(const KArgs &a, int device, cudaStream_t stream)
{
    constexpr auto kern = k_grad_reduce_adamw_cast<R, CLIP, CHECK, kUnrollStep>;
    unsigned grid = grid_for<kern>(device, a.n, 1 << 30);
    kern<<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int R>
cudaError_t launch_step_flags(const KArgs &a, bool clip, bool check, int device, cudaStream_t stream)
{
    if (clip)
        return check ? launch_step_r<R, true, true>(a, device, stream)
                     : launch_step_r<R, true, false>(a, device, stream);
    return check ? launch_step_r<R, false, true>(a, device, stream)
                 : launch_step_r<R, false, false>(a, device, stream);
}

template <int R>
cudaError_t launch_sq_r(const SqArgs &a, int *n_partials, int device, cudaStream_t stream)
{
    constexpr auto kern = k_grad_sqnorm<R, kUnrollSq>;
    unsigned grid = grid_for<kern>(device, a.n, kMaxPartials);
    kern<<<grid, kThreads, 0, stream>>>(a);
    *n_partials = (int)grid;
    return cudaGetLastError();
}

__global__ void k_cast_bf16(const float *src, uint16_t *w, int64_t n)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        w[i] = __bfloat16_as_ushort(__float2bfloat16_rn(src[i]));
}

__global__ void k_fill_zero(uint4 *p, size_t n16)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_fill_zero(void *p, size_t bytes, cudaStream_t stream)
{
    const size_t n16 = bytes / 16;
    if (n16 == 0)
        return cudaSuccess;
    const int dev_blocks = sm_count(0) * 8;
    k_fill_zero<<<dev_blocks, kThreads, 0, stream>>>(reinterpret_cast<uint4 *>(p), n16);
    return cudaGetLastError();
}

cudaError_t launch_cast_bf16(const float *src, uint16_t *w, int64_t n, cudaStream_t stream)
{
    if (n <= 0)
        return cudaSuccess;
    int64_t blocks = (n + kThreads - 1) / kThreads;
    if (blocks > 4096)
        blocks = 4096;
    k_cast_bf16<<<(unsigned)blocks, kThreads, 0, stream>>>(src, w, n);
    return cudaGetLastError();
}

cudaError_t launch_grad_sqnorm(const ReplicaPtrs &g, int R, int64_t n, const ClipScratch &scratch,
                               int *n_partials, int device, cudaStream_t stream)
{
    SqArgs a{g, n, scratch.partials};
    switch (R) {
    case 1: return launch_sq_r<1>(a, n_partials, device, stream);
    case 2: return launch_sq_r<2>(a, n_partials, device, stream);
    case 3: return launch_sq_r<3>(a, n_partials, device, stream);
    case 4: return launch_sq_r<4>(a, n_partials, device, stream);
    case 5: return launch_sq_r<5>(a, n_partials, device, stream);
    case 6: return launch_sq_r<6>(a, n_partials, device, stream);
    case 7: return launch_sq_r<7>(a, n_partials, device, stream);
    case 8: return launch_sq_r<8>(a, n_partials, device, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_grad_reduce_adamw_cast(const ReplicaPtrs &g, int R, int64_t n, float *theta,
                                          float *m, float *v, uint16_t *w, const AdamScalars &s,
                                          const ClipScratch *clip, int n_partials, float max_norm,
                                          bool check_finite, int device, cudaStream_t stream)
{
    const bool do_clip = clip != nullptr && max_norm > 0.0f;
    KArgs a{};
    a.g = g;
    a.theta = reinterpret_cast<float4 *>(theta);
    a.m = reinterpret_cast<float4 *>(m);
    a.v = reinterpret_cast<float4 *>(v);
    a.w = reinterpret_cast<uint4 *>(w);
    a.n = n;
    a.s = s;
    a.partials = do_clip ? clip->partials : nullptr;
    a.n_partials = do_clip ? n_partials : 0;
    a.max_norm = max_norm;
    a.coef_out = do_clip ? clip->coef : nullptr;
    a.status = clip ? clip->status : nullptr;
    switch (R) {
    case 1: return launch_step_flags<1>(a, do_clip, check_finite, device, stream);
    case 2: return launch_step_flags<2>(a, do_clip, check_finite, device, stream);
    case 3: return launch_step_flags<3>(a, do_clip, check_finite, device, stream);
    case 4: return launch_step_flags<4>(a, do_clip, check_finite, device, stream);
    case 5: return launch_step_flags<5>(a, do_clip, check_finite, device, stream);
    case 6: return launch_step_flags<6>(a, do_clip, check_finite, device, stream);
    case 7: return launch_step_flags<7>(a, do_clip, check_finite, device, stream);
    case 8: return launch_step_flags<8>(a, do_clip, check_finite, device, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace slide
