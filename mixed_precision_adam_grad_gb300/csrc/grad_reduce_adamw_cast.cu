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
// operations per parameter with BF16 replicas, 26 + 4R with FP32 replicas),
// so no tensor cores.  The kernel is a persistent
// producer/consumer pipeline, one CTA per SM:
//  - one producer thread streams tiles of kTile parameters of every input
//    (R replicas, master, m, v) into a kStages-deep shared-memory ring with
//    1-D bulk copies (cp.async.bulk, the TMA engine's linear mode), each
//    stage guarded by a pair of mbarriers (full: bytes landed; empty: the
//    consumers are done with it);
//  - 8 consumer warps read a stage from shared memory, compute, release the
//    stage, and write master, m, v and the BF16 copy straight to global
//    memory with streaming stores.
// The copies keep the loads in flight without registers, so a handful of
// warps saturate HBM while the divisions and square roots run.  Tiles go to
// CTAs round-robin (consecutive CTAs read consecutive addresses).  The part
// of the layer after the last whole tile is done with plain vector loads by
// one CTA, and the last n % 4 parameters with scalar accesses.
//
// Arithmetic: one IEEE FP32 operation per line of the update, explicit
// __f*_rn intrinsics so nothing is contracted into an FMA, IEEE sqrt and
// division, BF16 by round-to-nearest-even.  The replica sum is in replica
// order; the mean divides by R (a multiply by the exact inverse when R is a
// power of two).
//
// The optional global clip needs the norm of the whole layer's mean gradient
// before any element is updated, so it is a separate pre-pass
// (k_grad_sqnorm_pipe, the same bulk-copy pipeline reading only the replicas:
// 2R bytes per parameter) that writes one double-precision partial per block;
// the fused kernel turns the partials into the coefficient in its prologue,
// in the same fixed order in every block, so every block uses the same bits.
// Two things make the pair cost less than two passes back to back:
//  - the clipped step is launched behind the pre-pass with programmatic
//    serialisation (where a CTA of each fits on an SM together): its CTAs
//    start while the pre-pass runs, fill their rings with gradients and
//    FP32 state, and wait for the pre-pass's end only before reading the
//    partials, so no launch gap and no pipeline ramp sit between the two;
//  - the clipped step walks its tiles from the last to the first, so it
//    begins on the gradients the pre-pass read last, which L2 still holds.
// Measured on a 101M-parameter layer with four replicas, the whole clipped
// step went from 0.973 to 0.984 of the copy peak at 42 bytes per parameter.
//
// Every wait on an mbarrier is bounded (kWaitLimitNs of wall time); a wait
// that runs out sets bit 1 of the status word, waits (bounded) for the bulk
// copies it issued to land, and the kernel returns.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "slide_kernels.h"

namespace slide {
namespace {

constexpr int kThreads = 256;            // block size of the small helper kernels
constexpr int kTile = 2048;              // parameters per pipeline tile
constexpr int kStages = 2;               // shared-memory ring depth
constexpr int kConsumerWarps = 8;        // kTile = 256 consumer threads x 8 parameters
constexpr int kPipeThreads = (kConsumerWarps + 1) * 32;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitLimitTries = 1u << 26;
static_assert(kTile == kConsumerWarps * 32 * 8, "each consumer thread owns 8 parameters of a tile");

constexpr unsigned kStatusNonFinite = 1u;
constexpr unsigned kStatusWaitLimit = 2u;

struct KArgs {
    ReplicaPtrs g;
    float *theta;
    float *m;
    float *v;
    uint16_t *w;
    int64_t n;
    AdamScalars s;
    const double *partials;
    int n_partials;
    float max_norm;
    float *coef_out;
    unsigned *status;
    int test_stall;  // test only: the producer issues nothing, so the consumers' bounded wait runs out
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

// Gradient element types: BF16 replicas (bit patterns in uint16_t) or FP32
// replicas.  V4 holds 4 consecutive values; at() widens one of them to FP32.
template <typename G>
struct GradT;

template <>
struct GradT<uint16_t> {
    using V4 = uint2;
    static __device__ __forceinline__ float at(const uint2 &v, int e)
    {
        const uint32_t word = (e < 2) ? v.x : v.y;
        return (e & 1) ? bf16_hi(word) : bf16_lo(word);
    }
    static __device__ __forceinline__ float one(const uint16_t *p, int64_t i)
    {
        return __uint_as_float((uint32_t)p[i] << 16);
    }
    // the 8 values of vector k, kept raw (16 bytes) until used
    using Raw8 = uint4;
    static __device__ __forceinline__ Raw8 load8(const void *base, int64_t k)
    {
        return __ldcs(reinterpret_cast<const uint4 *>(base) + k);
    }
    static __device__ __forceinline__ float at8(const Raw8 &q, int e)
    {
        const uint32_t word = (&q.x)[e >> 1];
        return (e & 1) ? bf16_hi(word) : bf16_lo(word);
    }
};

template <>
struct GradT<float> {
    using V4 = float4;
    static __device__ __forceinline__ float at(const float4 &v, int e)
    {
        return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    }
    static __device__ __forceinline__ float one(const float *p, int64_t i) { return p[i]; }
    struct Raw8 {
        float4 a, b;
    };
    static __device__ __forceinline__ Raw8 load8(const void *base, int64_t k)
    {
        return {__ldcs(reinterpret_cast<const float4 *>(base) + 2 * k),
                __ldcs(reinterpret_cast<const float4 *>(base) + 2 * k + 1)};
    }
    static __device__ __forceinline__ float at8(const Raw8 &q, int e)
    {
        return e < 4 ? (&q.a.x)[e] : (&q.b.x)[e - 4];
    }
};

// Mean gradient of parameter e (0..3) of a 4-wide group, from R 4-value vectors.
template <typename G, int R, bool CLIP, bool CHECK>
__device__ __forceinline__ float mean_of(const typename GradT<G>::V4 (&gw)[R], int e, float coef, bool &bad)
{
    float x[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
        x[r] = GradT<G>::at(gw[r], e);
    float g = replica_mean<R>(x);
    if constexpr (CHECK)
        bad |= !isfinite(g);
    if constexpr (CLIP)
        g = __fmul_rn(g, coef);
    return g;
}

// Update 4 consecutive parameters held in registers and store them.
template <typename G, int R, bool CLIP, bool CHECK>
__device__ __forceinline__ void update4_store(const typename GradT<G>::V4 (&gw)[R], float4 th, float4 mm,
                                              float4 vv, int64_t e0, const KArgs &a, const AdamScalars &s,
                                              float coef, bool &bad)
{
    float t[4] = {th.x, th.y, th.z, th.w};
    float m[4] = {mm.x, mm.y, mm.z, mm.w};
    float v[4] = {vv.x, vv.y, vv.z, vv.w};
    uint16_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        adamw_one(mean_of<G, R, CLIP, CHECK>(gw, e, coef, bad), t[e], m[e], v[e], w[e], s);
    __stcs(reinterpret_cast<float4 *>(a.theta + e0), make_float4(t[0], t[1], t[2], t[3]));
    __stcs(reinterpret_cast<float4 *>(a.m + e0), make_float4(m[0], m[1], m[2], m[3]));
    __stcs(reinterpret_cast<float4 *>(a.v + e0), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<uint2 *>(a.w + e0), make_uint2(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3])));
}

// Deterministic clip coefficient from the per-block partials: warp 0 sums
// lane-strided in double, then a fixed shuffle-down tree; lane 0's result.
// Called by every thread of the block.
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

// ---- mbarrier and bulk-copy helpers (inline PTX) ---------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n"
        " .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase of `bar` with the given parity has completed; false if
// kWaitLimitNs of wall time (or, as a second bound, kWaitLimitTries polls)
// passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t round = 0; round < kWaitLimitTries / 64; ++round) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (global_ns() - t0 > kWaitLimitNs)
            return false;
    }
    return false;
}

// 1-D bulk copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// The same copy with an L2 eviction-priority policy (from make_evict_first).
__device__ __forceinline__ void bulk_load_hint(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// An L2 policy that marks the lines a load brings in (or hits) as the first to
// evict: for data read once.
__device__ __forceinline__ uint64_t make_evict_first()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream, when launched with programmatic serialisation, start before this
// one ends; wait_prerequisites blocks until the kernel this one was launched
// behind has ended and its writes are visible (it returns at once for a plain
// launch).
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Shared memory of one SM on sm_103a, and what a CTA takes beyond its
// dynamic shared memory (its static shared memory and the per-CTA
// reservation), rounded up: two CTAs fit on an SM together when their
// dynamic sizes plus this margin stay within the SM's.
constexpr int64_t kSmemPerSm = 228 * 1024;
constexpr int64_t kCoResidentMargin = 4096;

template <typename G, int R>
struct Pipe {
    static constexpr uint32_t kGradBytes = kTile * sizeof(G);
    static constexpr uint32_t kF32Bytes = kTile * 4;
    static constexpr uint32_t kStageBytes = R * kGradBytes + 3 * kF32Bytes;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 2 * kStages * 8;
};

template <typename G, int R, bool CLIP, bool CHECK>
__global__ void __launch_bounds__(kPipeThreads, 1) k_grad_reduce_adamw_cast(KArgs a)
{
    using P = Pipe<G, R>;
    using V4 = typename GradT<G>::V4;
    // Loads marked evict-first in L2, for the one instance where that was
    // measured faster: one BF16 replica, no clip (0.980 against 0.976 of the
    // copy peak on a 101M-parameter layer).  With R = 8 it was slower (0.981
    // against 0.987), and with the clip it takes L2 from the gradients the
    // pre-pass left there.
    constexpr bool kHintL2 = R == 1 && !CLIP;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * P::kStageBytes);
    uint64_t *empty = full + kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = a.n / kTile;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Producer state.  The block's k-th tile is j = blockIdx.x + k * gridDim.x;
    // with the clip it is processed as tile ntiles - 1 - j, so the step starts
    // on the last tiles, whose gradients the clip pre-pass read last and L2
    // still holds.
    int p_stage = 0;
    uint32_t p_phase = 0;
    uint32_t issued = 0, issued_phase = 0;  // per stage: filled at least once, and that fill's parity
    int64_t p_j = blockIdx.x;
    const bool producer = warp == kConsumerWarps && lane == 0 && !a.test_stall;
    const uint64_t policy = kHintL2 ? make_evict_first() : 0;
    auto load = [&](void *dst, const void *src, uint32_t bytes) {
        if constexpr (kHintL2)
            bulk_load_hint(dst, src, bytes, &full[p_stage], policy);
        else
            bulk_load(dst, src, bytes, &full[p_stage]);
    };
    auto issue = [&]() {
        const int64_t tile = CLIP ? ntiles - 1 - p_j : p_j;
        unsigned char *base = smem + p_stage * P::kStageBytes;
        mbar_arrive_expect_tx(&full[p_stage], P::kStageBytes);
        const int64_t e0 = tile * kTile;
#pragma unroll
        for (int r = 0; r < R; ++r)
            load(base + r * P::kGradBytes, static_cast<const G *>(a.g.p[r]) + e0, P::kGradBytes);
        load(base + R * P::kGradBytes, a.theta + e0, P::kF32Bytes);
        load(base + R * P::kGradBytes + P::kF32Bytes, a.m + e0, P::kF32Bytes);
        load(base + R * P::kGradBytes + 2 * P::kF32Bytes, a.v + e0, P::kF32Bytes);
        issued |= 1u << p_stage;
        issued_phase = (issued_phase & ~(1u << p_stage)) | (p_phase << p_stage);
        if (++p_stage == kStages) {
            p_stage = 0;
            p_phase ^= 1u;
        }
        p_j += gridDim.x;
    };

    float coef = 1.0f;
    if constexpr (CLIP) {
        // This kernel may be launched behind the clip pre-pass with
        // programmatic serialisation, so it can start while the pre-pass
        // runs.  Nothing the pre-pass writes is read before the wait: the
        // ring's first fills read gradients and the FP32 state only (empty
        // stages need no wait), the partials come after it.
        if (producer)
            for (int k = 0; k < kStages && p_j < ntiles; ++k)
                issue();
        wait_prerequisites();
        coef = clip_coef_from_partials(a.partials, a.n_partials, a.max_norm);  // includes __syncthreads
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.coef_out)
            *a.coef_out = coef;
    }

    if (warp == kConsumerWarps) {
        // ---- producer: one thread issues the bulk copies of each tile ----
        if (!producer)
            return;
        bool ok = true;
        while (p_j < ntiles) {
            if (!mbar_wait(&empty[p_stage], p_phase ^ 1u)) {
                ok = false;
                break;
            }
            issue();
        }
        // No copy may still be landing in shared memory when the block ends:
        // wait (bounded) for the last fill of every stage.
        for (int i = 0; i < kStages; ++i)
            if (((issued >> i) & 1u) && !mbar_wait(&full[i], (issued_phase >> i) & 1u))
                ok = false;
        if (!ok && a.status)
            atomicOr(a.status, kStatusWaitLimit);
        return;
    }

    // ---- consumers: thread c owns parameters [4c, 4c+4) and [kTile/2 + 4c, +4) ----
    const AdamScalars s = a.s;
    const int c = threadIdx.x;
    bool bad = false;
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t j = blockIdx.x; j < ntiles; j += gridDim.x) {
        const int64_t tile = CLIP ? ntiles - 1 - j : j;
        if (!mbar_wait(&full[stage], phase)) {
            if (a.status)
                atomicOr(a.status, kStatusWaitLimit);
            break;
        }
        const unsigned char *base = smem + stage * P::kStageBytes;
        V4 g0[R], g1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned char *gb = base + r * P::kGradBytes;
            g0[r] = *reinterpret_cast<const V4 *>(gb + c * sizeof(V4));
            g1[r] = *reinterpret_cast<const V4 *>(gb + P::kGradBytes / 2 + c * sizeof(V4));
        }
        const unsigned char *fb = base + R * P::kGradBytes;
        const float4 t0 = *reinterpret_cast<const float4 *>(fb + c * 16);
        const float4 t1 = *reinterpret_cast<const float4 *>(fb + kTile * 2 + c * 16);
        const float4 m0 = *reinterpret_cast<const float4 *>(fb + P::kF32Bytes + c * 16);
        const float4 m1 = *reinterpret_cast<const float4 *>(fb + P::kF32Bytes + kTile * 2 + c * 16);
        const float4 v0 = *reinterpret_cast<const float4 *>(fb + 2 * P::kF32Bytes + c * 16);
        const float4 v1 = *reinterpret_cast<const float4 *>(fb + 2 * P::kF32Bytes + kTile * 2 + c * 16);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[stage]);
        const int64_t e0 = tile * kTile + 4 * c;
        update4_store<G, R, CLIP, CHECK>(g0, t0, m0, v0, e0, a, s, coef, bad);
        update4_store<G, R, CLIP, CHECK>(g1, t1, m1, v1, e0 + kTile / 2, a, s, coef, bad);
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
    }

    // ---- the part after the last whole tile, by one CTA, plain loads ----
    if (blockIdx.x == (unsigned)(ntiles % gridDim.x)) {
        const int64_t base_e = ntiles * kTile;
        const int64_t rem = a.n - base_e;           // < kTile
        const int64_t groups = rem >> 2;            // 4-wide groups, < 512
        for (int64_t q = c; q < groups; q += kConsumerWarps * 32) {
            const int64_t e0 = base_e + 4 * q;
            V4 gw[R];
#pragma unroll
            for (int r = 0; r < R; ++r)
                gw[r] = __ldcs(reinterpret_cast<const V4 *>(static_cast<const G *>(a.g.p[r]) + e0));
            const float4 t = __ldcs(reinterpret_cast<const float4 *>(a.theta + e0));
            const float4 m = __ldcs(reinterpret_cast<const float4 *>(a.m + e0));
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(a.v + e0));
            update4_store<G, R, CLIP, CHECK>(gw, t, m, v, e0, a, s, coef, bad);
        }
        const int64_t tail0 = base_e + (groups << 2);
        if (c < a.n - tail0) {
            const int64_t i = tail0 + c;
            float x[R];
#pragma unroll
            for (int r = 0; r < R; ++r)
                x[r] = GradT<G>::one(static_cast<const G *>(a.g.p[r]), i);
            float g = replica_mean<R>(x);
            if constexpr (CHECK)
                bad |= !isfinite(g);
            if constexpr (CLIP)
                g = __fmul_rn(g, coef);
            float t = a.theta[i], m = a.m[i], v = a.v[i];
            uint16_t w;
            adamw_one(g, t, m, v, w, s);
            a.theta[i] = t;
            a.m[i] = m;
            a.v[i] = v;
            a.w[i] = w;
        }
    }
    if constexpr (CHECK) {
        if (bad && a.status)
            atomicOr(a.status, kStatusNonFinite);
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
    unsigned *status;  // bit 1: a bounded wait ran out (may be NULL)
};

// Clip pre-pass as a bulk-copy pipeline, the fused kernel's structure for a
// read-only pass: one CTA per SM; a producer lane streams tiles of 4 KiB per
// replica (2048 BF16 or 1024 FP32 parameters; larger with fewer than four
// replicas, see SqPipe::kGradBytes) into a ring of up to 8 stages (at most
// 192 KiB), and 8 consumer warps read them from shared memory and
// accumulate the squared replica means.  The loads in flight sit in shared
// memory, not in registers.  Tile and ring sizes were chosen by timing the
// whole clipped step: 4 KiB tiles in 8 stages beat 8 KiB tiles, 4, 6 or 12
// stages, and the register-path kernel this replaced.  With five or more BF16
// replicas (four or more FP32), the ring is cut to what leaves room for a CTA
// of the clipped step on the SM, down to 3 stages (see SqPipe::kBeside).  The
// part after the last whole tile is read with plain vector loads by one CTA.
// Each block writes one double partial, in a fixed order.
template <typename G, int R>
struct SqPipe {
    // Bytes per replica per tile: 4 KiB from four replicas on; with fewer, a
    // tile holds more parameters (16 KiB at R = 1, 8 KiB at R = 2 and 3), so
    // that the fixed cost of a tile (a copy issued, a barrier waited on and
    // released) is spread over enough work: with 4 KiB tiles one replica's
    // pass ran at 0.41 of the copy peak and the whole clipped step at 0.906,
    // with 16 KiB at 0.57 and 0.941.
    static constexpr uint32_t kGradBytes = R >= 4 ? 4096u : (R == 1 ? 16384u : 8192u);
    static constexpr int kTile = (int)(kGradBytes / sizeof(G));  // parameters per tile
    static constexpr int kPer = (int)(16 / sizeof(G));           // parameters per 16-byte vector
    static constexpr uint32_t kStageBytes = R * kGradBytes;
    static constexpr int kFit = (int)((192u * 1024u) / kStageBytes);
    static constexpr int kAlone = kFit > 8 ? 8 : (kFit < 2 ? 2 : kFit);
    // Stages that leave room on the SM for one CTA of the clipped step beside
    // this one, so that the step can start while this pass runs.  Where at
    // least 3 fit (at least 72 KiB in flight per SM), the ring takes no more.
    static constexpr int64_t kBeside =
        (kSmemPerSm - (int64_t)Pipe<G, R>::kSmemBytes - kCoResidentMargin) / (int64_t)(kStageBytes + 16);
    static constexpr int kStages = kBeside >= 3 && kBeside < kAlone ? (int)kBeside : kAlone;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 2 * kStages * 8;
    static constexpr int kVec = (int)(kGradBytes / (16 * kConsumerWarps * 32));  // vectors per thread per replica
    static_assert(kVec >= 1 && kGradBytes == (uint32_t)kVec * 16 * kConsumerWarps * 32,
                  "a tile is a whole number of 16-byte vectors per consumer thread");
};

// Element e of a 16-byte vector of gradient values, widened to FP32.
template <typename G>
__device__ __forceinline__ float vec16_at(const uint4 &q, int e)
{
    if constexpr (sizeof(G) == 2) {
        const uint32_t word = (&q.x)[e >> 1];
        return (e & 1) ? bf16_hi(word) : bf16_lo(word);
    } else {
        return __uint_as_float((&q.x)[e]);
    }
}

template <typename G, int R>
__device__ __forceinline__ void sq_add_vec16(SqAcc &acc, const uint4 (&q)[R])
{
#pragma unroll
    for (int e = 0; e < SqPipe<G, R>::kPer; ++e) {
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            x[r] = vec16_at<G>(q[r], e);
        acc.add(replica_mean<R>(x));
    }
}

template <typename G, int R>
__global__ void __launch_bounds__(kPipeThreads, 1) k_grad_sqnorm_pipe(SqArgs a)
{
    using P = SqPipe<G, R>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + P::kStages * P::kStageBytes);
    uint64_t *empty = full + P::kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The clipped step that follows may start now: it reads these partials
    // only after this grid has ended.
    launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < P::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t ntiles = a.n / P::kTile;
    SqAcc acc;

    if (warp == kConsumerWarps) {
        // ---- producer: lane 0 issues the bulk copies; the warp then joins the reduction ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;  // per stage: filled at least once, and that fill's parity
            bool ok = true;
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    ok = false;
                    break;
                }
                unsigned char *base = smem + stage * P::kStageBytes;
                mbar_arrive_expect_tx(&full[stage], P::kStageBytes);
                const int64_t e0 = tile * P::kTile;
#pragma unroll
                for (int r = 0; r < R; ++r)
                    bulk_load(base + r * P::kGradBytes, static_cast<const G *>(a.g.p[r]) + e0, P::kGradBytes,
                              &full[stage]);
                issued |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == P::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // no copy may still be landing in shared memory when the block ends
            for (int i = 0; i < P::kStages; ++i)
                if (((issued >> i) & 1u) && !mbar_wait(&full[i], (issued_phase >> i) & 1u))
                    ok = false;
            if (!ok && a.status)
                atomicOr(a.status, kStatusWaitLimit);
        }
        __syncwarp();
    } else {
        // ---- consumers: thread c reads vectors c, c + 256, ... of every replica of a tile ----
        const int c = threadIdx.x;
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
            const bool landed = __all_sync(0xffffffffu, mbar_wait(&full[stage], phase));
            if (!landed) {  // the whole warp gives up together
                if (lane == 0 && a.status)
                    atomicOr(a.status, kStatusWaitLimit);
                break;
            }
            const unsigned char *base = smem + stage * P::kStageBytes;
            uint4 q[P::kVec][R];
#pragma unroll
            for (int j = 0; j < P::kVec; ++j)
#pragma unroll
                for (int r = 0; r < R; ++r)
                    q[j][r] = *reinterpret_cast<const uint4 *>(base + r * P::kGradBytes + j * 4096 + c * 16);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stage]);
#pragma unroll
            for (int j = 0; j < P::kVec; ++j)
                sq_add_vec16<G, R>(acc, q[j]);
            if (++stage == P::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // the part after the last whole tile, by one CTA, plain loads
        if (blockIdx.x == (unsigned)(ntiles % gridDim.x)) {
            const int64_t base_e = ntiles * P::kTile;
            const int64_t rem = a.n - base_e;  // < kTile
            const int64_t nvec = rem / P::kPer;
            for (int64_t q = c; q < nvec; q += kConsumerWarps * 32) {
                uint4 v[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    v[r] = __ldcs(reinterpret_cast<const uint4 *>(static_cast<const G *>(a.g.p[r]) + base_e) + q);
                sq_add_vec16<G, R>(acc, v);
            }
            const int64_t tail0 = base_e + nvec * P::kPer;
            if (c < a.n - tail0) {
                const int64_t i = tail0 + c;
                float x[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    x[r] = GradT<G>::one(static_cast<const G *>(a.g.p[r]), i);
                acc.add(replica_mean<R>(x));
            }
        }
    }

    // Block reduction in double, fixed order (the producer warp adds zeros).
    double d = (double)acc.hi + (double)acc.lo + (double)acc.err;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        d += __shfl_down_sync(0xffffffffu, d, off);
    __shared__ double s_warp[kConsumerWarps + 1];
    if (lane == 0)
        s_warp[warp] = d;
    __syncthreads();
    if (warp == 0) {
        d = lane < kConsumerWarps + 1 ? s_warp[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            d += __shfl_down_sync(0xffffffffu, d, off);
        if (lane == 0)
            a.partials[blockIdx.x] = d;
    }
}

// Per-device caches below are written by whichever host thread first needs
// the value; every writer computes the same value, and atomics make the
// concurrent first use by two states on two host threads well defined.
constexpr int kMaxDevices = 64;

int sm_count(int device)
{
    static std::atomic<int> cache[kMaxDevices];
    if (device < 0 || device >= kMaxDevices)
        return 1;
    int c = cache[device].load(std::memory_order_relaxed);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || c < 1)
            c = 1;
        cache[device].store(c, std::memory_order_relaxed);
    }
    return c;
}



// Whether a CTA of the clipped step fits on an SM beside a CTA of the clip
// pre-pass (dynamic shared memory of each, plus a margin for their static
// shared memory and the per-CTA reservation).  Only then is the step launched
// to overlap the pre-pass: a step whose CTAs cannot sit beside the pre-pass's
// would take the SMs the pre-pass leaves first, two CTAs to an SM, and run
// unevenly.
bool fits_beside_prepass(int device, uint32_t step_smem, uint32_t prepass_smem)
{
    static std::atomic<int> cache[kMaxDevices];
    int per_sm = 0;
    if (device >= 0 && device < kMaxDevices)
        per_sm = cache[device].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess)
            return false;
        if (device >= 0 && device < kMaxDevices)
            cache[device].store(per_sm, std::memory_order_relaxed);
    }
    return (int64_t)step_smem + prepass_smem + kCoResidentMargin <= per_sm;
}

// Raise the fused kernel's dynamic shared-memory limit on `device` (once per
// device; the device must be current).  Setting the attribute also loads the
// kernel's code on a lazily loading context.
template <typename G, int R, bool CLIP, bool CHECK>
cudaError_t prepare_pipeline_kernel(int device)
{
    constexpr auto kern = k_grad_reduce_adamw_cast<G, R, CLIP, CHECK>;
    constexpr uint32_t smem = Pipe<G, R>::kSmemBytes;
    static std::atomic<int> attr_set[kMaxDevices];
    if (device >= 0 && device < kMaxDevices && attr_set[device].load(std::memory_order_acquire))
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    // The clipped step starts while the pre-pass still runs (one CTA of each
    // per SM, 81-131 KB of shared memory each): ask for the largest shared
    // memory carve-out so that both fit on an SM at once.
    if (e == cudaSuccess && CLIP)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return e;
    if (device >= 0 && device < kMaxDevices)
        attr_set[device].store(1, std::memory_order_release);
    return cudaSuccess;
}

template <typename G, int R, bool CLIP, bool CHECK>
cudaError_t launch_step_r(const KArgs &a, int device, cudaStream_t stream, bool behind_prepass)
{
    constexpr auto kern = k_grad_reduce_adamw_cast<G, R, CLIP, CHECK>;
    constexpr uint32_t smem = Pipe<G, R>::kSmemBytes;
    static_assert(smem <= 227 * 1024, "pipeline stages exceed the shared memory of a CTA");
    cudaError_t e = prepare_pipeline_kernel<G, R, CLIP, CHECK>(device);
    if (e != cudaSuccess)
        return e;
    // one CTA per SM, never more CTAs than whole tiles (at least one, for the tail)
    int64_t grid = sm_count(device);
    const int64_t ntiles = a.n / kTile;
    if (grid > ntiles)
        grid = ntiles > 0 ? ntiles : 1;
    if (CLIP && behind_prepass && fits_beside_prepass(device, smem, SqPipe<G, R>::kSmemBytes)) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kPipeThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, a);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    kern<<<(unsigned)grid, kPipeThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <typename G, int R>
cudaError_t launch_step_flags(const KArgs &a, bool clip, bool check, int device, cudaStream_t stream,
                              bool behind_prepass)
{
    if (clip)
        return check ? launch_step_r<G, R, true, true>(a, device, stream, behind_prepass)
                     : launch_step_r<G, R, true, false>(a, device, stream, behind_prepass);
    return check ? launch_step_r<G, R, false, true>(a, device, stream, false)
                 : launch_step_r<G, R, false, false>(a, device, stream, false);
}

template <typename G>
cudaError_t launch_step_g(const KArgs &a, int R, bool clip, bool check, int device, cudaStream_t stream,
                          bool behind_prepass)
{
    switch (R) {
    case 1: return launch_step_flags<G, 1>(a, clip, check, device, stream, behind_prepass);
    case 2: return launch_step_flags<G, 2>(a, clip, check, device, stream, behind_prepass);
    case 3: return launch_step_flags<G, 3>(a, clip, check, device, stream, behind_prepass);
    case 4: return launch_step_flags<G, 4>(a, clip, check, device, stream, behind_prepass);
    case 5: return launch_step_flags<G, 5>(a, clip, check, device, stream, behind_prepass);
    case 6: return launch_step_flags<G, 6>(a, clip, check, device, stream, behind_prepass);
    case 7: return launch_step_flags<G, 7>(a, clip, check, device, stream, behind_prepass);
    case 8: return launch_step_flags<G, 8>(a, clip, check, device, stream, behind_prepass);
    default: return cudaErrorInvalidValue;
    }
}

// Raise the pipelined pre-pass's dynamic shared-memory limit on `device`
// (once per device; the device must be current; also loads its code).
template <typename G, int R>
cudaError_t prepare_sq_pipe(int device)
{
    static std::atomic<int> attr_set[kMaxDevices];
    if (device >= 0 && device < kMaxDevices && attr_set[device].load(std::memory_order_acquire))
        return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_grad_sqnorm_pipe<G, R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SqPipe<G, R>::kSmemBytes);
    if (e == cudaSuccess)  // room for the clipped step's CTA beside it (see prepare_pipeline_kernel)
        e = cudaFuncSetAttribute(k_grad_sqnorm_pipe<G, R>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return e;
    if (device >= 0 && device < kMaxDevices)
        attr_set[device].store(1, std::memory_order_release);
    return cudaSuccess;
}

template <typename G, int R>
cudaError_t launch_sq_r(const SqArgs &a, int *n_partials, int device, cudaStream_t stream)
{
    using P = SqPipe<G, R>;
    static_assert(P::kSmemBytes <= 227 * 1024, "pre-pass stages exceed the shared memory of a CTA");
    cudaError_t e = prepare_sq_pipe<G, R>(device);
    if (e != cudaSuccess)
        return e;
    // one CTA per SM, never more CTAs than whole tiles (at least one, for the tail)
    int64_t grid = sm_count(device);
    const int64_t ntiles = a.n / P::kTile;
    if (grid > ntiles)
        grid = ntiles > 0 ? ntiles : 1;
    if (grid > kMaxPartials)
        grid = kMaxPartials;
    k_grad_sqnorm_pipe<G, R><<<(unsigned)grid, kPipeThreads, P::kSmemBytes, stream>>>(a);
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

cudaError_t launch_fill_zero(void *p, size_t bytes, int device, cudaStream_t stream)
{
    const size_t n16 = bytes / 16;
    if (n16 == 0)
        return cudaSuccess;
    const int dev_blocks = sm_count(device) * 8;
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

template <typename G>
cudaError_t launch_sq_g(const SqArgs &a, int R, int *n_partials, int device, cudaStream_t stream)
{
    switch (R) {
    case 1: return launch_sq_r<G, 1>(a, n_partials, device, stream);
    case 2: return launch_sq_r<G, 2>(a, n_partials, device, stream);
    case 3: return launch_sq_r<G, 3>(a, n_partials, device, stream);
    case 4: return launch_sq_r<G, 4>(a, n_partials, device, stream);
    case 5: return launch_sq_r<G, 5>(a, n_partials, device, stream);
    case 6: return launch_sq_r<G, 6>(a, n_partials, device, stream);
    case 7: return launch_sq_r<G, 7>(a, n_partials, device, stream);
    case 8: return launch_sq_r<G, 8>(a, n_partials, device, stream);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_grad_sqnorm(const ReplicaPtrs &g, int R, int64_t n, const ClipScratch &scratch,
                               int *n_partials, int device, cudaStream_t stream, bool f32_grads)
{
    SqArgs a{g, n, scratch.partials, scratch.status};
    return f32_grads ? launch_sq_g<float>(a, R, n_partials, device, stream)
                     : launch_sq_g<uint16_t>(a, R, n_partials, device, stream);
}

namespace {

// Load (and prepare) every kernel that a BF16-replica step without the
// non-finite check can launch: the fused kernel with and without the clip and
// the clip pre-pass, for R = 1..8.
template <int R>
cudaError_t preload_bf16_r(int device)
{
    cudaError_t e = prepare_pipeline_kernel<uint16_t, R, true, false>(device);
    if (e == cudaSuccess)
        e = prepare_pipeline_kernel<uint16_t, R, false, false>(device);
    if (e == cudaSuccess)
        e = prepare_sq_pipe<uint16_t, R>(device);
    return e;
}

}  // namespace

cudaError_t preload_bf16_step_kernels(int device)
{
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = preload_bf16_r<1>(device);
    if (e == cudaSuccess) e = preload_bf16_r<2>(device);
    if (e == cudaSuccess) e = preload_bf16_r<3>(device);
    if (e == cudaSuccess) e = preload_bf16_r<4>(device);
    if (e == cudaSuccess) e = preload_bf16_r<5>(device);
    if (e == cudaSuccess) e = preload_bf16_r<6>(device);
    if (e == cudaSuccess) e = preload_bf16_r<7>(device);
    if (e == cudaSuccess) e = preload_bf16_r<8>(device);
    if (e == cudaSuccess)
        sm_count(device);
    return e;
}

cudaError_t launch_grad_reduce_adamw_cast(const ReplicaPtrs &g, int R, int64_t n, float *theta,
                                          float *m, float *v, uint16_t *w, const AdamScalars &s,
                                          const ClipScratch *clip, int n_partials, float max_norm,
                                          bool check_finite, int device, cudaStream_t stream, bool test_stall,
                                          bool f32_grads, bool behind_prepass)
{
    const bool do_clip = clip != nullptr && clip->partials != nullptr && max_norm > 0.0f;
    KArgs a{};
    a.g = g;
    a.theta = theta;
    a.m = m;
    a.v = v;
    a.w = w;
    a.n = n;
    a.s = s;
    a.partials = do_clip ? clip->partials : nullptr;
    a.n_partials = do_clip ? n_partials : 0;
    a.max_norm = max_norm;
    a.coef_out = do_clip ? clip->coef : nullptr;
    a.status = clip ? clip->status : nullptr;
    a.test_stall = test_stall ? 1 : 0;
    return f32_grads ? launch_step_g<float>(a, R, do_clip, check_finite, device, stream, behind_prepass)
                     : launch_step_g<uint16_t>(a, R, do_clip, check_finite, device, stream, behind_prepass);
}

}  // namespace slide
