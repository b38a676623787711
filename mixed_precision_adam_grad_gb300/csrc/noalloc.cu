// noalloc.cu — slide_adamw_step_noalloc: the fused step (clip pre-pass +
// grad_reduce_adamw_cast) for callers that cannot allocate GPU memory.
//
// Who needs it: code that may not call cudaMalloc or anything that allocates
// on the device, for example an allocator hook or memory-pressure handler
// that must not re-enter the CUDA allocator it is part of, a process whose
// GPU memory is a pool owned and capped by a framework (a cudaMalloc beside
// the pool can fail or break the pool's accounting), or an embedded runtime
// that forbids allocation after start-up.  Such a caller owns every array
// (replicas, master, m, v, BF16 output) and cannot hand the library the
// scratch that the clip's partial sums need, nor hold a slide_state.
//
// The scratch is a file-scope __device__ array of fixed size
// (kNoAllocPartials doubles for the per-block partial sums, one float for the
// coefficient and one status word), so this entry point never calls
// cudaMalloc, cudaFree or any allocating routine.  Every GPU that loads the
// library holds the array until the process exits.
//
// Host code cannot use the array's name as a device address: on the host that
// name is only a stand-in symbol.  The address is fetched with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on that device, and cached.  The first call on a device
// also loads every kernel this entry point can launch: on a context that
// loads code lazily (the default) that first call may load the library's
// device code and allocate its static memory, so callers make it at
// start-up, and before any stream capture.  Later calls load nothing.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
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
    unsigned status;  // bit 1: a bounded pipeline wait ran out (the step is incomplete)
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
            // load every kernel a later call may launch, so that no later call
            // loads code (which can allocate device memory)
            e = preload_bf16_step_kernels(device);
            if (e != cudaSuccess)
                return fail_cuda(e, "loading the kernels of the no-alloc entry point");
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
    ClipScratch cs{scr->partials, &scr->coef, &scr->status};
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
    // with the clip off the kernel reads no partials (max_norm 0) but still
    // reports a wait that ran out into the status word
    // SLIDE_TEST_PIPELINE_STALL (tests only): the update kernel's copy producer
    // issues nothing, so the consumers' bounded wait (2 s) runs out and the
    // status word reports it; the arrays are then undefined
    const bool stall = getenv("SLIDE_TEST_PIPELINE_STALL") != nullptr;
    e = launch_grad_reduce_adamw_cast(g, n_replicas, n, master, m, v, (uint16_t *)bf16_out, sc, &cs,
                                      n_partials, clip ? hp->max_grad_norm : 0.0f, false, device, s, stall);
    if (e != cudaSuccess)
        return fail_cuda(e, "grad_reduce_adamw_cast launch (no-alloc)");
    clear_error();
    return SLIDE_OK;
}

extern "C" slide_status slide_noalloc_status(slide_stream_t stream)
{
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDevice");
    if (device < 0 || device >= kNoAllocMaxDevices)
        return fail(SLIDE_ERR_INVALID_ARG, "device ordinal beyond the no-alloc entry point's table (64)");
    NoAllocScratch *p = g_scratch_addr[device].load(std::memory_order_acquire);
    if (!p) {  // no call on this device yet: nothing to report
        clear_error();
        return SLIDE_OK;
    }
    unsigned word = 0;
    e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(&word, &p->status, sizeof word, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && word) {
        const unsigned zero = 0;
        e = cudaMemcpy(&p->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess)
        return fail_cuda(e, "reading the no-alloc status word");
    if (word & 2u)
        return fail(SLIDE_ERR_TIMEOUT,
                    "a pipeline wait inside the kernel reached its limit; that step is incomplete");
    clear_error();
    return SLIDE_OK;
}
