// noalloc.cu — slide_adamw_step_noalloc: the fused step (clip pre-pass +
// grad_reduce_adamw_cast) for callers that cannot allocate GPU memory.
//
// Who needs it: code that runs where cudaMalloc is off limits, for example
// inside a host callback or allocator hook that must not re-enter the CUDA
// allocator, a process whose memory pool is owned and capped by a framework,
// or an embedded runtime that forbids allocation after start-up.  Such a
// caller owns every array (replicas, master, m, v, BF16 output) and cannot
// give the library the per-call scratch that the clip's partial sums need.
//
// The scratch is a file-scope __device__ array of fixed size
// (kNoAllocPartials doubles for the per-block partial sums plus one float for
// the coefficient), so this entry point never calls cudaMalloc, cudaFree or
// any allocating routine.  Every GPU that loads the library holds the array
// until the process exits.
//
// Host code cannot use the array's name as a device address: on the host that
// name is only a stand-in symbol.  The address is fetched once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device, and cached.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <string>

#include "slide.h"
#include "slide_kernels.h"
#include "slide_state.h"

namespace slide {
namespace {

// Partial sums the clip pre-pass may write: it never launches more blocks.
constexpr int kNoAllocPartials = kMaxPartials;
static_assert(kNoAllocPartials >= kMaxPartials, "the pre-pass grid is capped at kMaxPartials blocks");
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
    double partials[kNoAllocPartials];
    float coef;
    unsigned status;
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

std::mutex g_setup_mutex;
std::atomic<NoAllocScratch *> g_scratch_addr[kNoAllocMaxDevices];

// Device address of this device's copy of g_noalloc_scratch (set-up on first
// use per device; the device must be current).
slide_status scratch_for_device(int device, NoAllocScratch **out)
{
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(SLIDE_ERR_INVALID_ARG, "device ordinal beyond the no-alloc entry point's table (64)");
    NoAllocScratch *p = g_scratch_addr[device].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[device].load(std::memory_order_relaxed);
        if (!p) {
            cudaError_t e = cudaGetSymbolAddress((void **)&p, g_noalloc_scratch);
            if (e != cudaSuccess || !p)
                return fail_cuda(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                                 "cudaGetSymbolAddress of the no-alloc scratch");
            g_scratch_addr[device].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return SLIDE_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace slide

using namespace slide;

extern "C" slide_status slide_adamw_step_noalloc(int64_t n, int32_t n_replicas, const void *const *grad_replicas,
                                                 float *master, float *m, float *v, void *bf16_out,
                                                 const slide_adam_hparams *hp, int64_t step,
                                                 slide_stream_t stream)
{
    if (n < 0 || n > ((int64_t)1 << 40))
        return fail(SLIDE_ERR_INVALID_ARG, "n must lie in [0, 2^40] for slide_adamw_step_noalloc");
    if (n_replicas < 1 || n_replicas > SLIDE_MAX_REPLICAS)
        return fail(SLIDE_ERR_INVALID_ARG, "n_replicas must lie in [1, 8] for slide_adamw_step_noalloc");
    if (step < 1)
        return fail(SLIDE_ERR_INVALID_ARG, "step (the 1-based update count) must be >= 1");
    slide_status rc = check_hparams(hp);
    if (rc != SLIDE_OK)
        return rc;
    if (!grad_replicas)
        return fail(SLIDE_ERR_INVALID_ARG, "grad_replicas is NULL");
    ReplicaPtrs g{};
    for (int r = 0; r < n_replicas; ++r) {
        g.p[r] = grad_replicas[r];
        if (n > 0 && (!g.p[r] || !aligned16(g.p[r])))
            return fail(SLIDE_ERR_INVALID_ARG, "gradient replica pointer is NULL or not 16-byte aligned");
    }
    void *arrs[4] = {master, m, v, bf16_out};
    for (void *a : arrs)
        if (n > 0 && (!a || !aligned16(a)))
            return fail(SLIDE_ERR_INVALID_ARG, "master, m, v and bf16_out must be 16-byte aligned device pointers");
    if (n == 0) {
        clear_error();
        return SLIDE_OK;
    }
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    NoAllocScratch *scr = nullptr;
    if ((rc = scratch_for_device(device, &scr)) != SLIDE_OK)
        return rc;
    ClipScratch cs{scr->partials, &scr->coef, nullptr};
    cudaStream_t s = (cudaStream_t)stream;
    const AdamScalars sc = adam_scalars_for(*hp, step);
    const bool clip = hp->max_grad_norm > 0.0f;
    int n_partials = 0;
    if (clip) {
        // every partial that the update kernel reads is written by this pre-pass
        // first, so nothing has to be cleared between calls
        e = launch_grad_sqnorm(g, n_replicas, n, cs, &n_partials, device, s);
        if (e != cudaSuccess)
            return fail_cuda(e, "grad_sqnorm launch (no-alloc)");
    }
    e = launch_grad_reduce_adamw_cast(g, n_replicas, n, master, m, v, (uint16_t *)bf16_out, sc,
                                      clip ? &cs : nullptr, n_partials, clip ? hp->max_grad_norm : 0.0f,
                                      false, device, s);
    if (e != cudaSuccess)
        return fail_cuda(e, "grad_reduce_adamw_cast launch (no-alloc)");
    clear_error();
    return SLIDE_OK;
}
