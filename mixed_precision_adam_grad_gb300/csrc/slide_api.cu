// slide_api.cu — the C ABI declared in include/slide.h: argument checks,
// status codes, the thread-local last error, state allocation and the
// HBM-resident layer step.  The streamed residency's sweep is in
// stream_engine.cu.
//
// The state layout follows the 16N accounting of "SlideDP: Scaling
// Host-Resident LLM Fine-Tuning Across Multiple GPUs" (Prerequisites): per
// parameter 4 bytes of FP32 master, 4 + 4 of FP32 Adam moments and 2 of the
// BF16 compute copy owned by the state (the 2 bytes of BF16 gradient per
// replica are the caller's).  Every array starts on a 256-byte boundary of
// one arena allocation, allocated once at creation (no allocation on the
// step path).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExtCudaRt.h>

#include <sys/mman.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "slide.h"
#include "slide_kernels.h"
#include "slide_state.h"

namespace slide {

static thread_local std::string g_last_error;

slide_status fail(slide_status code, const std::string &msg)
{
    g_last_error = msg;
    return code;
}

slide_status fail_cuda(cudaError_t e, const char *what)
{
    std::string msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    g_last_error = msg;
    if (e == cudaErrorMemoryAllocation)
        return SLIDE_ERR_OOM_DEVICE;
    return SLIDE_ERR_CUDA;
}

void clear_error() { g_last_error.clear(); }

// Bias corrections of update t (1-based): bc1 = 1 - beta1^t, bc2 = 1 - beta2^t,
// formed in double from the FP32 hyper-parameters; each scalar rounded once.
AdamScalars adam_scalars_for(const slide_adam_hparams &hp, int64_t t)
{
    const double b1 = hp.beta1, b2 = hp.beta2;
    const double bc1 = 1.0 - std::pow(b1, (double)t);
    const double bc2 = 1.0 - std::pow(b2, (double)t);
    AdamScalars s;
    s.beta1 = hp.beta1;
    s.one_minus_beta1 = (float)(1.0 - b1);
    s.beta2 = hp.beta2;
    s.one_minus_beta2 = (float)(1.0 - b2);
    s.decay = (float)(1.0 - (double)hp.lr * (double)hp.weight_decay);
    s.step_size = (float)((double)hp.lr / bc1);
    s.bc2_sqrt = (float)std::sqrt(bc2);
    s.eps = hp.eps;
    return s;
}

slide_status check_hparams(const slide_adam_hparams *hp)
{
    if (!hp)
        return fail(SLIDE_ERR_INVALID_ARG, "hparams is NULL");
    const float vals[6] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm};
    for (float x : vals)
        if (!std::isfinite(x))
            return fail(SLIDE_ERR_INVALID_ARG, "hparams: non-finite value");
    if (hp->lr < 0.0f)
        return fail(SLIDE_ERR_INVALID_ARG, "hparams: lr < 0");
    if (hp->beta1 < 0.0f || hp->beta1 >= 1.0f || hp->beta2 < 0.0f || hp->beta2 >= 1.0f)
        return fail(SLIDE_ERR_INVALID_ARG, "hparams: betas must lie in [0, 1)");
    if (hp->eps < 0.0f || hp->weight_decay < 0.0f)
        return fail(SLIDE_ERR_INVALID_ARG, "hparams: eps and weight_decay must be >= 0");
    return SLIDE_OK;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static slide_status check_config(const slide_config *cfg, int64_t *max_numel)
{
    if (!cfg)
        return fail(SLIDE_ERR_INVALID_ARG, "config is NULL");
    if (cfg->n_layers < 1 || !cfg->layer_numel)
        return fail(SLIDE_ERR_INVALID_ARG, "config: n_layers must be >= 1 with a layer_numel array");
    if (cfg->n_replicas < 1 || cfg->n_replicas > SLIDE_MAX_REPLICAS)
        return fail(SLIDE_ERR_INVALID_ARG, "config: n_replicas must be in [1, 8]");
    if (cfg->residency != SLIDE_RESIDENCY_HBM && cfg->residency != SLIDE_RESIDENCY_HOST_STREAMED)
        return fail(SLIDE_ERR_INVALID_ARG, "config: unknown residency");
    if (cfg->window_layers != 0 && cfg->window_layers != 2)
        return fail(SLIDE_ERR_INVALID_ARG, "config: window_layers must be 2 (or 0 for the default 2)");
    if (cfg->chunk_bytes < 0 || (cfg->chunk_bytes % 256) != 0)
        return fail(SLIDE_ERR_INVALID_ARG, "config: chunk_bytes must be a non-negative multiple of 256");
    if (cfg->chunk_bytes_d2h < 0 || (cfg->chunk_bytes_d2h % 256) != 0)
        return fail(SLIDE_ERR_INVALID_ARG, "config: chunk_bytes_d2h must be a non-negative multiple of 256");
    if (cfg->host_arena) {
        if (cfg->residency != SLIDE_RESIDENCY_HOST_STREAMED)
            return fail(SLIDE_ERR_INVALID_ARG, "config: host_arena is for the streamed residency only");
        if (((uintptr_t)cfg->host_arena & 255u) != 0)
            return fail(SLIDE_ERR_INVALID_ARG, "config: host_arena must be 256-byte aligned");
        if (cfg->flags & SLIDE_FLAG_HOST_HUGE_PAGES)
            return fail(SLIDE_ERR_INVALID_ARG, "config: host_arena and SLIDE_FLAG_HOST_HUGE_PAGES exclude each other");
    } else if (cfg->host_arena_bytes != 0) {
        return fail(SLIDE_ERR_INVALID_ARG, "config: host_arena_bytes without a host_arena");
    }
    if (cfg->flags & ~(uint32_t)(SLIDE_FLAG_CHECK_FINITE | SLIDE_FLAG_TEST_PIPELINE_STALL | SLIDE_FLAG_FP32_GRADS |
                                 SLIDE_FLAG_BF16_COPY_IN_HBM | SLIDE_FLAG_HOST_HUGE_PAGES | SLIDE_FLAG_HOST_INPUTS))
        return fail(SLIDE_ERR_INVALID_ARG, "config: unknown flag bits");
    if ((cfg->flags & SLIDE_FLAG_HOST_INPUTS) && cfg->residency != SLIDE_RESIDENCY_HBM)
        return fail(SLIDE_ERR_INVALID_ARG, "config: SLIDE_FLAG_HOST_INPUTS is for the HBM residency");
    if (cfg->device < 0)
        return fail(SLIDE_ERR_INVALID_ARG, "config: device < 0");
    int64_t mx = 0;
    for (int32_t l = 0; l < cfg->n_layers; ++l) {
        const int64_t n = cfg->layer_numel[l];
        if (n < 0 || n > ((int64_t)1 << 40))
            return fail(SLIDE_ERR_INVALID_ARG, "config: layer_numel out of range [0, 2^40]");
        if (n > mx)
            mx = n;
    }
    if (cfg->residency == SLIDE_RESIDENCY_HOST_STREAMED) {
        // the engine keeps a few events per chunk and slot: bound the chunk count
        const int64_t in = cfg->chunk_bytes > 0 ? cfg->chunk_bytes : ((int64_t)256 << 20);
        const int64_t out = cfg->chunk_bytes_d2h > 0 ? cfg->chunk_bytes_d2h : in;
        const int64_t bytes = mx * 4;
        if ((bytes + in - 1) / in > kMaxChunksPerUnit || (bytes + out - 1) / out > kMaxChunksPerUnit)
            return fail(SLIDE_ERR_INVALID_ARG, "config: chunk_bytes / chunk_bytes_d2h too small for the largest unit "
                                               "(at most 65536 chunks per unit)");
    }
    *max_numel = mx;
    return SLIDE_OK;
}

static size_t layer_state_bytes(int64_t n)
{
    return 3 * align_up((size_t)n * 4) + align_up((size_t)n * 2);
}

// Streamed residency with the BF16 copy in HBM: FP32 state on the host, BF16 copy on the device.
static bool copy_in_hbm(const slide_config *cfg)
{
    return cfg->residency == SLIDE_RESIDENCY_HOST_STREAMED && (cfg->flags & SLIDE_FLAG_BF16_COPY_IN_HBM);
}
static size_t layer_fp32_bytes(int64_t n) { return 3 * align_up((size_t)n * 4); }
static size_t layer_bf16_bytes(int64_t n) { return align_up((size_t)n * 2); }

}  // namespace slide

using namespace slide;

extern "C" {

int32_t slide_abi_version(void) { return SLIDE_ABI_VERSION; }

const char *slide_last_error(void) { return g_last_error.c_str(); }

slide_status slide_state_bytes(const slide_config *cfg, int64_t *device_bytes, int64_t *host_pinned_bytes)
{
    int64_t mx = 0;
    slide_status rc = check_config(cfg, &mx);
    if (rc != SLIDE_OK)
        return rc;
    size_t state = 0;
    for (int32_t l = 0; l < cfg->n_layers; ++l)
        state += layer_state_bytes(cfg->layer_numel[l]);
    size_t dev = 0, host = 0;
    if (cfg->residency == SLIDE_RESIDENCY_HBM) {
        dev = state + (size_t)cfg->n_layers * scratch_bytes() + host_input_bytes(*cfg, mx);
    } else if (copy_in_hbm(cfg)) {
        for (int32_t l = 0; l < cfg->n_layers; ++l) {
            host += layer_fp32_bytes(cfg->layer_numel[l]);
            dev += layer_bf16_bytes(cfg->layer_numel[l]);
        }
        dev += engine_device_bytes(*cfg, mx);
    } else {
        host = state;
        dev = engine_device_bytes(*cfg, mx);
    }
    if (device_bytes)
        *device_bytes = (int64_t)dev;
    if (host_pinned_bytes)
        *host_pinned_bytes = (int64_t)host;
    clear_error();
    return SLIDE_OK;
}

// Size of a transparent huge page on this host (the PMD size), 2 MiB if the
// kernel does not say.
static size_t huge_page_bytes()
{
    size_t hp = 0;
    if (FILE *f = fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long v = 0;
        if (fscanf(f, "%llu", &v) == 1)
            hp = (size_t)v;
        fclose(f);
    }
    return (hp >= 4096 && (hp & (hp - 1)) == 0) ? hp : ((size_t)2 << 20);
}

// The pinned host arena.  Default: cudaHostAlloc.  With
// SLIDE_FLAG_HOST_HUGE_PAGES: an anonymous mapping aligned to the huge page
// size, advised MADV_HUGEPAGE before its pages are touched, then pinned and
// mapped for the device with cudaHostRegister (which faults the pages in), so
// the arena is backed by physically contiguous huge pages where the kernel
// can provide them.
static cudaError_t host_arena_alloc(slide_state *st, size_t bytes)
{
    if (st->cfg.host_arena) {  // the caller's pinned memory, checked by the caller of this function
        st->host_arena = st->cfg.host_arena;
        st->host_arena_owned = false;
        return cudaSuccess;
    }
    st->host_arena_owned = true;
    if (!(st->cfg.flags & SLIDE_FLAG_HOST_HUGE_PAGES))
        return cudaHostAlloc(&st->host_arena, bytes > 0 ? bytes : 1, cudaHostAllocDefault);
    const size_t hp = huge_page_bytes();
    const size_t len = (bytes + hp - 1) / hp * hp + (bytes == 0 ? hp : 0);
    void *raw = mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE, -1, 0);
    if (raw == MAP_FAILED)
        return cudaErrorMemoryAllocation;
    const uintptr_t a = ((uintptr_t)raw + hp - 1) & ~(uintptr_t)(hp - 1);
    const size_t head = a - (uintptr_t)raw;
    if (head)
        munmap(raw, head);
    if (hp - head)
        munmap((char *)a + len, hp - head);
    madvise((void *)a, len, MADV_HUGEPAGE);
    cudaError_t e = cudaHostRegister((void *)a, len, cudaHostRegisterPortable | cudaHostRegisterMapped);
    if (e != cudaSuccess) {
        munmap((void *)a, len);
        return e;
    }
    st->host_arena = (void *)a;
    st->host_map_bytes = len;
    return cudaSuccess;
}

static void host_arena_free(slide_state *st)
{
    if (!st->host_arena)
        return;
    if (!st->host_arena_owned) {
        st->host_arena = nullptr;
        return;
    }
    if (st->host_map_bytes) {
        cudaHostUnregister(st->host_arena);
        munmap(st->host_arena, st->host_map_bytes);
    } else {
        cudaFreeHost(st->host_arena);
    }
    st->host_arena = nullptr;
    st->host_map_bytes = 0;
}

static void host_inputs_destroy(slide_state *st)
{
    HostInputs *H = st->hin;
    if (!H)
        return;
    if (H->copy)
        cudaStreamSynchronize(H->copy);
    for (int b = 0; b < 2; ++b) {
        if (H->landed[b])
            cudaEventDestroy(H->landed[b]);
        if (H->consumed[b])
            cudaEventDestroy(H->consumed[b]);
    }
    if (H->copy)
        cudaStreamDestroy(H->copy);
    delete H;
    st->hin = nullptr;
}

// The staging of slide_layer_step_host in the device arena at `base` (2 sets
// x R replicas of max_numel values), its copy stream and events.
static slide_status host_inputs_create(slide_state *st, char *base, int64_t max_numel)
{
    HostInputs *H = new (std::nothrow) HostInputs();
    if (!H)
        return fail(SLIDE_ERR_OOM_HOST, "out of host memory for the host-input staging");
    st->hin = H;
    const size_t g = (st->cfg.flags & SLIDE_FLAG_FP32_GRADS) ? 4 : 2;
    const size_t per = align_up((size_t)max_numel * g);
    for (int b = 0; b < 2; ++b)
        for (int r = 0; r < st->cfg.n_replicas; ++r) {
            H->stage[b][r] = base;
            base += per;
        }
    cudaError_t e = cudaStreamCreateWithFlags(&H->copy, cudaStreamNonBlocking);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
        e = cudaEventCreateWithFlags(&H->landed[b], cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&H->consumed[b], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        slide_status rc = fail_cuda(e, "host-input staging set-up");
        host_inputs_destroy(st);
        return rc;
    }
    if (e == cudaSuccess)
        nvtxNameCudaStreamA(H->copy, "slide host-input copy");
    return SLIDE_OK;
}

slide_status slide_state_create(const slide_config *cfg, slide_state **out)
{
    if (!out)
        return fail(SLIDE_ERR_INVALID_ARG, "out is NULL");
    int64_t mx = 0;
    slide_status rc = check_config(cfg, &mx);
    if (rc != SLIDE_OK)
        return rc;
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaGetDeviceCount");
    if (cfg->device >= ndev)
        return fail(SLIDE_ERR_INVALID_ARG, "config: device ordinal out of range");
    DeviceGuard guard(cfg->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");

    slide_state *st = new (std::nothrow) slide_state();
    if (!st)
        return fail(SLIDE_ERR_OOM_HOST, "out of host memory for the state object");
    st->cfg = *cfg;
    st->cfg.layer_numel = nullptr;
    if (st->cfg.window_layers == 0)
        st->cfg.window_layers = 2;
    if (st->cfg.timeout_ms == 0)
        st->cfg.timeout_ms = 600000;
    if (st->cfg.chunk_bytes == 0)  // chosen by a sweep of both chunk sizes on the 8 x h8192 and 40 x h5120 models
        st->cfg.chunk_bytes = (int64_t)256 << 20;
    if (st->cfg.chunk_bytes_d2h == 0)
        st->cfg.chunk_bytes_d2h = st->cfg.chunk_bytes;
    st->device = cfg->device;
    st->numel.assign(cfg->layer_numel, cfg->layer_numel + cfg->n_layers);
    st->layers.resize(cfg->n_layers);

    size_t state_bytes = 0;
    for (int32_t l = 0; l < cfg->n_layers; ++l)
        state_bytes += layer_state_bytes(st->numel[l]);

    char *base = nullptr;
    if (cfg->residency == SLIDE_RESIDENCY_HBM) {
        st->dev_bytes = state_bytes + (size_t)cfg->n_layers * scratch_bytes() + host_input_bytes(*cfg, mx);
        e = cudaMalloc(&st->dev_arena, st->dev_bytes);
        if (e != cudaSuccess) {
            cudaGetLastError();
            delete st;
            return fail(SLIDE_ERR_OOM_DEVICE, std::string("cudaMalloc of the HBM state (") +
                                                  std::to_string(state_bytes) + " bytes) failed");
        }
        e = cudaMemset(st->dev_arena, 0, st->dev_bytes);
        if (e != cudaSuccess) {
            cudaFree(st->dev_arena);
            delete st;
            return fail_cuda(e, "cudaMemset of the HBM state");
        }
        base = (char *)st->dev_arena;
    } else {
        size_t mirror_bytes = 0;
        if (copy_in_hbm(cfg)) {
            state_bytes = 0;
            for (int32_t l = 0; l < cfg->n_layers; ++l) {
                state_bytes += layer_fp32_bytes(st->numel[l]);
                mirror_bytes += layer_bf16_bytes(st->numel[l]);
            }
            e = cudaMalloc(&st->dev_arena, mirror_bytes > 0 ? mirror_bytes : 256);
            if (e == cudaSuccess)
                e = cudaMemset(st->dev_arena, 0, mirror_bytes > 0 ? mirror_bytes : 256);
            if (e != cudaSuccess) {
                cudaGetLastError();
                if (st->dev_arena)
                    cudaFree(st->dev_arena);
                delete st;
                return fail(SLIDE_ERR_OOM_DEVICE, "cudaMalloc of the HBM BF16 copy (" +
                                                      std::to_string(mirror_bytes) + " bytes) failed");
            }
        }
        st->host_bytes = state_bytes;
        if (cfg->host_arena) {
            // the caller's arena must be large enough and pinned host memory
            cudaPointerAttributes pa{};
            const bool pinned = cudaPointerGetAttributes(&pa, cfg->host_arena) == cudaSuccess &&
                                pa.type == cudaMemoryTypeHost;
            cudaGetLastError();
            const char *why = cfg->host_arena_bytes < (int64_t)state_bytes
                                  ? "config: host_arena_bytes is smaller than the state's host bytes"
                                  : (!pinned ? "config: host_arena is not pinned (page-locked) host memory" : nullptr);
            if (why) {
                if (st->dev_arena)
                    cudaFree(st->dev_arena);
                delete st;
                return fail(SLIDE_ERR_INVALID_ARG, why);
            }
        }
        e = host_arena_alloc(st, st->host_bytes);
        if (e != cudaSuccess || getenv("SLIDE_FAULT_PINNED_ALLOC")) {
            // SLIDE_FAULT_PINNED_ALLOC injects this failure for tests of the
            // clean-up path (nothing stays allocated).
            if (e == cudaSuccess)
                host_arena_free(st);
            cudaGetLastError();
            if (st->dev_arena)
                cudaFree(st->dev_arena);
            delete st;
            return fail(SLIDE_ERR_OOM_HOST, std::string("cudaHostAlloc of the pinned state (") +
                                                std::to_string(state_bytes) + " bytes) failed");
        }
        // Zero the pinned state from the GPU through the memory's device
        // address (fast over the host link; a host memset of ~100 GB would
        // take many seconds).  The arena size is a multiple of 256 bytes.
        void *dptr = nullptr;
        e = cudaHostGetDevicePointer(&dptr, st->host_arena, 0);
        if (e == cudaSuccess)
            e = launch_fill_zero(dptr, st->host_bytes, st->device, 0);
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaGetLastError();
            memset(st->host_arena, 0, st->host_bytes);
        }
        base = (char *)st->host_arena;
    }

    size_t off = 0, moff = 0;
    for (int32_t l = 0; l < cfg->n_layers; ++l) {
        LayerState &L = st->layers[l];
        const size_t n = (size_t)st->numel[l];
        L.n = (int64_t)n;
        L.theta = (float *)(base + off);
        off += align_up(n * 4);
        L.m = (float *)(base + off);
        off += align_up(n * 4);
        L.v = (float *)(base + off);
        off += align_up(n * 4);
        if (copy_in_hbm(cfg)) {
            L.w = (uint16_t *)((char *)st->dev_arena + moff);
            moff += layer_bf16_bytes((int64_t)n);
        } else {
            L.w = (uint16_t *)(base + off);
            off += align_up(n * 2);
        }
    }
    if (cfg->residency == SLIDE_RESIDENCY_HBM) {
        for (int32_t l = 0; l < cfg->n_layers; ++l) {
            LayerState &L = st->layers[l];
            L.scratch.partials = (double *)(base + off);
            L.scratch.coef = (float *)(base + off + align_up(sizeof(double) * kMaxPartials));
            L.scratch.status = (unsigned *)(L.scratch.coef + 1);
            off += scratch_bytes();
        }
        if (cfg->flags & SLIDE_FLAG_HOST_INPUTS) {
            rc = host_inputs_create(st, base + off, mx);
            if (rc != SLIDE_OK) {
                cudaFree(st->dev_arena);
                delete st;
                return rc;
            }
        }
    } else {
        rc = engine_create(st);
        if (rc != SLIDE_OK) {
            host_arena_free(st);
            if (st->dev_arena)
                cudaFree(st->dev_arena);
            delete st;
            return rc;
        }
    }
    *out = st;
    clear_error();
    return SLIDE_OK;
}

void slide_state_destroy(slide_state *st)
{
    if (!st)
        return;
    DeviceGuard guard(st->device);
    if (st->engine)
        engine_destroy(st);
    host_inputs_destroy(st);
    if (st->dev_arena) {
        cudaDeviceSynchronize();
        cudaFree(st->dev_arena);
    }
    host_arena_free(st);
    delete st;
}

static slide_status check_layer(slide_state *st, int32_t layer)
{
    if (!st)
        return fail(SLIDE_ERR_INVALID_ARG, "state is NULL");
    if (layer < 0 || layer >= (int32_t)st->layers.size())
        return fail(SLIDE_ERR_INVALID_ARG, "layer index out of range");
    return SLIDE_OK;
}

// Enqueue the step of one layer (clip pre-pass if on, then the fused kernel)
// on s, reading the replicas g and writing the BF16 copy to w; the device is
// current.  `after_update`, if given, is recorded behind the fused kernel.
static slide_status enqueue_layer_step(slide_state *st, LayerState &L, const ReplicaPtrs &g,
                                       const slide_adam_hparams *hp, cudaStream_t s, uint16_t *w,
                                       cudaEvent_t after_update)
{
    const int R = st->cfg.n_replicas;
    const int64_t t = L.t + 1;
    {
        const AdamScalars sc = adam_scalars_for(*hp, t);
        const bool clip = hp->max_grad_norm > 0.0f;
        const bool check = (st->cfg.flags & SLIDE_FLAG_CHECK_FINITE) != 0;
        int n_partials = 0;
        cudaError_t e;
        if (st->trace[0])
            cudaEventRecord(st->trace[0], s);
        const bool f32g = (st->cfg.flags & SLIDE_FLAG_FP32_GRADS) != 0;
        if (clip) {
            e = launch_grad_sqnorm(g, R, L.n, L.scratch, &n_partials, st->device, s, f32g);
            if (e != cudaSuccess)
                return fail_cuda(e, "grad_sqnorm launch");
        }
        // With the clip, the update is launched right behind the pre-pass
        // and overlaps its end, unless a trace event has to separate them.
        if (st->trace[1])
            cudaEventRecord(st->trace[1], s);
        e = launch_grad_reduce_adamw_cast(g, R, L.n, L.theta, L.m, L.v, w, sc, &L.scratch, n_partials,
                                          clip ? hp->max_grad_norm : 0.0f, check, st->device, s,
                                          (st->cfg.flags & SLIDE_FLAG_TEST_PIPELINE_STALL) != 0, f32g,
                                          clip && !st->trace[1]);
        if (e != cudaSuccess)
            return fail_cuda(e, "grad_reduce_adamw_cast launch");
        if (after_update && (e = cudaEventRecord(after_update, s)) != cudaSuccess)
            return fail_cuda(e, "event record after the update");
        if (st->trace[2])
            cudaEventRecord(st->trace[2], s);
    }
    L.t = t;
    return SLIDE_OK;
}

slide_status slide_layer_step(slide_state *st, int32_t layer, const void *const *grad_replicas,
                              const slide_adam_hparams *hp, slide_stream_t stream, void *bf16_out)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    if (st->cfg.residency != SLIDE_RESIDENCY_HBM)
        return fail(SLIDE_ERR_STATE, "slide_layer_step needs the HBM residency; use slide_model_step_streamed");
    if ((rc = check_hparams(hp)) != SLIDE_OK)
        return rc;
    LayerState &L = st->layers[layer];
    const int R = st->cfg.n_replicas;
    if (!grad_replicas)
        return fail(SLIDE_ERR_INVALID_ARG, "grad_replicas is NULL");
    ReplicaPtrs g{};
    for (int r = 0; r < R; ++r) {
        g.p[r] = grad_replicas[r];
        if (L.n > 0 && (!g.p[r] || !aligned16(g.p[r])))
            return fail(SLIDE_ERR_INVALID_ARG, "gradient replica pointer is NULL or not 16-byte aligned");
    }
    uint16_t *w = bf16_out ? (uint16_t *)bf16_out : L.w;
    if (!aligned16(w))
        return fail(SLIDE_ERR_INVALID_ARG, "bf16_out is not 16-byte aligned");
    if (L.n == 0) {
        L.t += 1;
        clear_error();
        return SLIDE_OK;
    }
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    rc = enqueue_layer_step(st, L, g, hp, (cudaStream_t)stream, w, nullptr);
    if (rc == SLIDE_OK)
        clear_error();
    return rc;
}

slide_status slide_layer_step_host(slide_state *st, int32_t layer, const void *const *host_grad_replicas,
                                   const slide_adam_hparams *hp, slide_stream_t stream, void *host_bf16_out)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    if (st->cfg.residency != SLIDE_RESIDENCY_HBM || !st->hin)
        return fail(SLIDE_ERR_STATE, "slide_layer_step_host needs the HBM residency and SLIDE_FLAG_HOST_INPUTS");
    if ((rc = check_hparams(hp)) != SLIDE_OK)
        return rc;
    LayerState &L = st->layers[layer];
    const int R = st->cfg.n_replicas;
    if (!host_grad_replicas)
        return fail(SLIDE_ERR_INVALID_ARG, "host_grad_replicas is NULL");
    for (int r = 0; r < R; ++r)
        if (L.n > 0 && !host_grad_replicas[r])
            return fail(SLIDE_ERR_INVALID_ARG, "a host gradient replica pointer is NULL");
    if (L.n == 0) {
        L.t += 1;
        clear_error();
        return SLIDE_OK;
    }
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    HostInputs &H = *st->hin;
    const int b = H.next;
    const size_t gbytes = (size_t)L.n * ((st->cfg.flags & SLIDE_FLAG_FP32_GRADS) ? 4 : 2);
    cudaStream_t s = (cudaStream_t)stream;
    // copy-in on the state's copy stream, once the update that last read this
    // staging set is done; the caller's stream waits for it to land
    cudaError_t e = cudaStreamWaitEvent(H.copy, H.consumed[b], 0);
    ReplicaPtrs g{};
    for (int r = 0; r < R && e == cudaSuccess; ++r) {
        g.p[r] = H.stage[b][r];
        e = cudaMemcpyAsync(H.stage[b][r], host_grad_replicas[r], gbytes, cudaMemcpyHostToDevice, H.copy);
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(H.landed[b], H.copy);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(s, H.landed[b], 0);
    if (e != cudaSuccess)
        return fail_cuda(e, "copy-in of the host gradient replicas");
    H.next = b ^ 1;
    rc = enqueue_layer_step(st, L, g, hp, s, L.w, H.consumed[b]);
    if (rc != SLIDE_OK)
        return rc;
    if (host_bf16_out) {
        e = cudaMemcpyAsync(host_bf16_out, L.w, (size_t)L.n * 2, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess)
            return fail_cuda(e, "copy-out of the BF16 copy");
    }
    clear_error();
    return SLIDE_OK;
}

static void refresh_aborted(slide_state *st)
{
    if (!st->aborted)
        return;
    for (const LayerState &L : st->layers)
        if (L.t != st->layers[0].t)
            return;
    st->aborted = false;
}

// Copy `bytes` between caller memory and the state's arrays.  For the pinned
// host state of the streamed residency the copy goes through a device buffer
// of the window, so that only DMA touches the pinned state: on the GB300
// hosts measured, pinned pages that the CPU had read or written were read
// several times slower by the copy engines for a while afterwards, and a
// host-to-host cudaMemcpy is a CPU copy.
static cudaError_t state_copy(slide_state *st, void *dst, const void *src, size_t bytes, bool to_state)
{
    if (bytes == 0)
        return cudaSuccess;
    if (st->cfg.residency != SLIDE_RESIDENCY_HOST_STREAMED)
        return cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    cudaPointerAttributes pa{};
    const void *state_side = to_state ? dst : src;
    if (cudaPointerGetAttributes(&pa, state_side) != cudaSuccess || pa.type != cudaMemoryTypeHost) {
        cudaGetLastError();  // device-resident (the BF16 copy kept in HBM)
        return cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    }
    size_t cap = 0;
    char *stage = (char *)engine_staging(st, &cap);
    if (!stage || cap == 0)
        return cudaMemcpy(dst, src, bytes, cudaMemcpyDefault);
    cudaError_t e = cudaSuccess;
    for (size_t off = 0; off < bytes && e == cudaSuccess; off += cap) {
        const size_t len = bytes - off < cap ? bytes - off : cap;
        e = cudaMemcpy(stage, (const char *)src + off, len, cudaMemcpyDefault);
        if (e == cudaSuccess)
            e = cudaMemcpy((char *)dst + off, stage, len, cudaMemcpyDefault);
    }
    return e;
}

slide_status slide_layer_set(slide_state *st, int32_t layer, const float *master, const float *m,
                             const float *v, int64_t step)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    if (step < 0)
        return fail(SLIDE_ERR_INVALID_ARG, "step must be >= 0");
    LayerState &L = st->layers[layer];
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    if ((rc = engine_quiesce(st)) != SLIDE_OK)  // a step still in flight (slide_model_step_streamed_async)
        return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaDeviceSynchronize");
    const size_t bytes = (size_t)L.n * 4;
    const float *src[3] = {master, m, v};
    float *dst[3] = {L.theta, L.m, L.v};
    for (int k = 0; k < 3; ++k) {
        if (!src[k] || bytes == 0)
            continue;
        e = state_copy(st, dst[k], src[k], bytes, true);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaMemcpy in slide_layer_set");
    }
    if (master && L.n > 0) {
        // The pinned host arrays of the streamed residency are reached through
        // their device addresses.
        float *th_d = L.theta;
        uint16_t *w_d = L.w;
        if (st->cfg.residency == SLIDE_RESIDENCY_HOST_STREAMED) {
            e = cudaHostGetDevicePointer((void **)&th_d, L.theta, 0);
            if (e == cudaSuccess && !copy_in_hbm(&st->cfg))
                e = cudaHostGetDevicePointer((void **)&w_d, L.w, 0);
            if (e != cudaSuccess)
                return fail_cuda(e, "cudaHostGetDevicePointer in slide_layer_set");
        }
        e = launch_cast_bf16(th_d, w_d, L.n, 0);
        if (e == cudaSuccess)
            e = cudaDeviceSynchronize();
        if (e != cudaSuccess)
            return fail_cuda(e, "bf16 cast in slide_layer_set");
    }
    L.t = step;
    refresh_aborted(st);
    clear_error();
    return SLIDE_OK;
}

slide_status slide_layer_get(slide_state *st, int32_t layer, float *master, float *m, float *v,
                             uint16_t *bf16, int64_t *step)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    LayerState &L = st->layers[layer];
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    if ((rc = engine_quiesce(st)) != SLIDE_OK)  // a step still in flight (slide_model_step_streamed_async)
        return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return fail_cuda(e, "cudaDeviceSynchronize");
    const void *src[4] = {L.theta, L.m, L.v, L.w};
    void *dst[4] = {master, m, v, bf16};
    const size_t bytes[4] = {(size_t)L.n * 4, (size_t)L.n * 4, (size_t)L.n * 4, (size_t)L.n * 2};
    for (int k = 0; k < 4; ++k) {
        if (!dst[k] || bytes[k] == 0)
            continue;
        e = state_copy(st, dst[k], src[k], bytes[k], false);
        if (e != cudaSuccess)
            return fail_cuda(e, "cudaMemcpy in slide_layer_get");
    }
    if (step)
        *step = L.t;
    clear_error();
    return SLIDE_OK;
}

slide_status slide_layer_ptrs(slide_state *st, int32_t layer, float **master, float **m, float **v,
                              uint16_t **bf16)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    LayerState &L = st->layers[layer];
    if (master)
        *master = L.theta;
    if (m)
        *m = L.m;
    if (v)
        *v = L.v;
    if (bf16)
        *bf16 = L.w;
    clear_error();
    return SLIDE_OK;
}

slide_status slide_layer_last_clip_coef(slide_state *st, int32_t layer, float *coef)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    if (!coef)
        return fail(SLIDE_ERR_INVALID_ARG, "coef is NULL");
    LayerState &L = st->layers[layer];
    if (!L.scratch.coef)
        return fail(SLIDE_ERR_STATE, "no clip scratch for this residency");
    DeviceGuard guard(st->device);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(coef, L.scratch.coef, sizeof(float), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return fail_cuda(e, "reading the clip coefficient");
    if (*coef == 0.0f)  // never written: the arena starts zeroed
        *coef = 1.0f;
    clear_error();
    return SLIDE_OK;
}

slide_status slide_layer_status(slide_state *st, int32_t layer)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    LayerState &L = st->layers[layer];
    if (!L.scratch.status)
        return SLIDE_OK;
    DeviceGuard guard(st->device);
    unsigned word = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(&word, L.scratch.status, sizeof word, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && word)
        e = cudaMemset(L.scratch.status, 0, sizeof word);
    if (e != cudaSuccess)
        return fail_cuda(e, "reading the status word");
    if (word & 2u)
        return fail(SLIDE_ERR_TIMEOUT, "a pipeline wait inside the kernel reached its limit; the step is incomplete");
    if ((word & 1u) && (st->cfg.flags & SLIDE_FLAG_CHECK_FINITE))
        return fail(SLIDE_ERR_NONFINITE, "a non-finite mean gradient was seen");
    clear_error();
    return SLIDE_OK;
}

slide_status slide_trace_events(slide_state *st, void *ev_prepass_start, void *ev_update_start,
                                void *ev_update_stop)
{
    if (!st)
        return fail(SLIDE_ERR_INVALID_ARG, "state is NULL");
    st->trace[0] = (cudaEvent_t)ev_prepass_start;
    st->trace[1] = (cudaEvent_t)ev_update_start;
    st->trace[2] = (cudaEvent_t)ev_update_stop;
    clear_error();
    return SLIDE_OK;
}

slide_status slide_deliver_bf16(slide_state *st, int32_t layer, void *const *dst, int32_t n_consumers,
                                int32_t route, slide_stream_t stream)
{
    slide_status rc = check_layer(st, layer);
    if (rc != SLIDE_OK)
        return rc;
    if (n_consumers < 1 || n_consumers > SLIDE_MAX_REPLICAS || !dst)
        return fail(SLIDE_ERR_INVALID_ARG, "n_consumers must lie in [1, 8] with a dst array");
    if (route != SLIDE_DELIVER_FULL && route != SLIDE_DELIVER_SHARDED)
        return fail(SLIDE_ERR_INVALID_ARG, "unknown delivery route");
    LayerState &L = st->layers[layer];
    for (int r = 0; r < n_consumers; ++r)
        if (L.n > 0 && (!dst[r] || !aligned16(dst[r])))
            return fail(SLIDE_ERR_INVALID_ARG, "consumer pointer is NULL or not 16-byte aligned");
    if (L.n == 0) {
        clear_error();
        return SLIDE_OK;
    }
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    if ((rc = engine_quiesce(st)) != SLIDE_OK)  // the copy being delivered may still be in flight
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t n = (size_t)L.n;
    cudaError_t e = cudaSuccess;
    if (route == SLIDE_DELIVER_FULL || n_consumers == 1) {
        for (int r = 0; r < n_consumers && e == cudaSuccess; ++r)
            e = cudaMemcpyAsync(dst[r], L.w, n * 2, cudaMemcpyDefault, s);
    } else {
        // shard size: n / R rounded up to 8 elements (16 bytes) so every shard starts aligned
        const size_t shard = ((n + n_consumers - 1) / n_consumers + 7) & ~(size_t)7;
        for (int r = 0; r < n_consumers && e == cudaSuccess; ++r) {
            const size_t off = (size_t)r * shard;
            if (off >= n)
                break;
            const size_t len = n - off < shard ? n - off : shard;
            e = cudaMemcpyAsync((uint16_t *)dst[r] + off, L.w + off, len * 2, cudaMemcpyDefault, s);
        }
        // all-gather on the device: consumer q takes shard r from its owner r
        for (int r = 0; r < n_consumers && e == cudaSuccess; ++r) {
            const size_t off = (size_t)r * shard;
            if (off >= n)
                break;
            const size_t len = n - off < shard ? n - off : shard;
            for (int q = 0; q < n_consumers && e == cudaSuccess; ++q)
                if (q != r)
                    e = cudaMemcpyAsync((uint16_t *)dst[q] + off, (const uint16_t *)dst[r] + off, len * 2,
                                        cudaMemcpyDeviceToDevice, s);
        }
    }
    if (e != cudaSuccess)
        return fail_cuda(e, "slide_deliver_bf16 copies");
    clear_error();
    return SLIDE_OK;
}

slide_status slide_streamed_timeline(slide_state *st, double *out, int64_t cap)
{
    if (!st || !out)
        return fail(SLIDE_ERR_INVALID_ARG, "state or out is NULL");
    if (st->cfg.residency != SLIDE_RESIDENCY_HOST_STREAMED || !st->engine)
        return fail(SLIDE_ERR_STATE, "the timeline belongs to the host-streamed residency");
    DeviceGuard guard(st->device);
    slide_status rc = engine_timeline(st, out, cap);
    if (rc == SLIDE_OK)
        clear_error();
    return rc;
}

static slide_status model_step_streamed(slide_state *st, slide_grad_fn fn, void *user,
                                        const slide_adam_hparams *hp, bool wait_for_end)
{
    if (!st)
        return fail(SLIDE_ERR_INVALID_ARG, "state is NULL");
    if (st->cfg.residency != SLIDE_RESIDENCY_HOST_STREAMED || !st->engine)
        return fail(SLIDE_ERR_STATE, "slide_model_step_streamed needs the host-streamed residency");
    if (!fn)
        return fail(SLIDE_ERR_INVALID_ARG, "grad_fn is NULL");
    slide_status rc = check_hparams(hp);
    if (rc != SLIDE_OK)
        return rc;
    if (st->aborted)
        return fail(SLIDE_ERR_ABORTED, "an earlier sweep was aborted; restore a common version with slide_layer_set");
    for (const LayerState &L : st->layers)
        if (L.t != st->layers[0].t)
            return fail(SLIDE_ERR_VERSION, "units carry different step counts (same-version invariant)");
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    rc = engine_step(st, fn, user, *hp, wait_for_end);
    if (rc == SLIDE_OK)
        clear_error();
    return rc;
}

slide_status slide_model_step_streamed(slide_state *st, slide_grad_fn fn, void *user,
                                       const slide_adam_hparams *hp)
{
    return model_step_streamed(st, fn, user, hp, true);
}

slide_status slide_model_step_streamed_async(slide_state *st, slide_grad_fn fn, void *user,
                                             const slide_adam_hparams *hp)
{
    return model_step_streamed(st, fn, user, hp, false);
}

slide_status slide_streamed_sync(slide_state *st)
{
    if (!st)
        return fail(SLIDE_ERR_INVALID_ARG, "state is NULL");
    if (st->cfg.residency != SLIDE_RESIDENCY_HOST_STREAMED || !st->engine)
        return fail(SLIDE_ERR_STATE, "slide_streamed_sync needs the host-streamed residency");
    DeviceGuard guard(st->device);
    if (!guard.ok)
        return fail(SLIDE_ERR_CUDA, "cudaSetDevice failed");
    slide_status rc = engine_sync(st);
    if (rc == SLIDE_OK)
        clear_error();
    return rc;
}

}  // extern "C"
