// stream_engine.cu — host-resident streaming of the optimizer state through a
// bounded 2-slot HBM window (the streamed residency of slide_model_step_streamed).
//
// Design sources (page title, section):
//  - "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs",
//    Prerequisites (host-resident layer streaming: persistent state in host
//    memory, a small reusable BF16 layer window on the GPU, layers swapped in
//    forward order for the forward pass and in reverse order for the backward
//    pass) and Core method / Method steps (one authoritative host copy of the
//    FP32 master and Adam moments per layer; per-chunk pipelining of copies and
//    updates; the version gate: the next delivery of a layer waits for its
//    update; slots are reused only after their copies complete).
//  - "An Efficient Heterogeneous Co-Design for Fine-Tuning on a Single GPU"
//    (SlideFormer), sections 2.1-2.2: while layer i is processed the next one
//    is prefetched and the previous one's update proceeds; a pre-allocated,
//    fixed-size GPU window (no allocation while stepping).
//  - "Accelerating the Training of Large Language Models using Efficient
//    Activation Rematerialization and Optimal Hybrid Parallelism", section
//    5.1: copies serialised with cudaStreamWaitEvent so a buffer is reused
//    only after the copy that reads it is done; two ping-pong buffers whose
//    roles swap every step; page-locked host buffers.
//
// What differs from the pages: they run the Adam update on host cores and
// cast FP32 -> BF16 on the host; here the update and the cast run on the GPU
// (grad_reduce_adamw_cast), so per parameter and step the link moves
//   host -> device: 2 B (BF16 delivery, forward sweep) + 12 B (master, m, v)
//   device -> host: 12 B (master, m, v) + 2 B (new BF16 copy)
// and the R gradient replicas never leave HBM.
//
// Schedule of one step (all enqueued up front; the host then waits once):
//  forward sweep on the H2D stream: BF16 copy of unit l -> slot l%2;
//  reverse sweep, l = L-1 .. 0, slot s = l%2:
//    H2D stream:     master/m/v of l -> slot s, chunk by chunk; chunk k of each
//                    array first waits for the D2H of the same chunk of the
//                    unit that last used slot s (l+2), so the copy-in of l
//                    trails the copy-out of l+2 by one chunk;
//    compute stream: once the master of l has landed, grad_fn(l) fills the R
//                    replicas (while m and v still arrive); then, after the
//                    rest of l's H2D and the D2H of the BF16 copy of l+2, the
//                    clip pre-pass and the fused kernel update slot s in place;
//    D2H stream:     wait for the kernel; BF16 copy, then master/m/v of l back
//                    to the host, chunk by chunk, each chunk recording the
//                    event the next copy-in to the same bytes waits for.
//  While the kernel updates l, the H2D engine is filling the other slot with
//  l-1 and the D2H engine is draining l+1 out of it.
#include <cuda_runtime.h>

#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "slide_kernels.h"
#include "slide_state.h"

namespace slide {

namespace {

constexpr int kSlots = 2;
constexpr int kRegions = 3;  // master, m, v (the arrays the next copy-in overwrites)

struct Slot {
    float *arr[kRegions] = {nullptr, nullptr, nullptr};  // master, m, v
    uint16_t *w = nullptr;
    void *g[kMaxReplicas] = {};
    ClipScratch scratch{};
    // chunk k of region r freed by the D2H of the unit that used this slot last
    std::vector<cudaEvent_t> freed[kRegions];
    cudaEvent_t w_freed = nullptr;  // D2H of the BF16 copy done
};

size_t grad_bytes(const slide_config &cfg) { return (cfg.flags & SLIDE_FLAG_FP32_GRADS) ? 4 : 2; }

size_t slot_bytes(int64_t maxn, int R, size_t gsize)
{
    return 3 * align_up((size_t)maxn * 4) + align_up((size_t)maxn * 2) +
           align_up((size_t)maxn * gsize) * (size_t)R + scratch_bytes();
}

}  // namespace

struct StreamEngine {
    void *window = nullptr;
    size_t window_bytes = 0;
    Slot slots[kSlots];
    int64_t chunk_bytes = 0;
    int chunks_per_region = 0;
    cudaStream_t s_h2d = nullptr, s_comp = nullptr, s_d2h = nullptr;
    std::vector<cudaEvent_t> theta_done;  // per unit: the master has landed in its slot
    std::vector<cudaEvent_t> h2d_done;    // per unit: master, m and v have landed
    std::vector<cudaEvent_t> kern_done;   // per unit
    cudaEvent_t fwd_done = nullptr;
    cudaEvent_t sweep_done[3] = {nullptr, nullptr, nullptr};  // end of the H2D, compute, D2H streams
    // timeline of the last step (timing events): start, and per unit the
    // begin of its copy-in and the begin/end of its write-back
    cudaEvent_t step_start = nullptr;
    std::vector<cudaEvent_t> h2d_begin, d2h_begin, d2h_end;
    std::vector<char> recorded;  // unit reached write-back in the last step
};

size_t engine_device_bytes(const slide_config &cfg, int64_t max_numel)
{
    return kSlots * slot_bytes(max_numel, cfg.n_replicas, grad_bytes(cfg));
}

static void destroy_engine_objects(StreamEngine *E)
{
    for (Slot &s : E->slots) {
        for (auto &v : s.freed)
            for (cudaEvent_t ev : v)
                if (ev)
                    cudaEventDestroy(ev);
        if (s.w_freed)
            cudaEventDestroy(s.w_freed);
    }
    for (cudaEvent_t ev : E->h2d_done)
        if (ev)
            cudaEventDestroy(ev);
    for (cudaEvent_t ev : E->theta_done)
        if (ev)
            cudaEventDestroy(ev);
    for (cudaEvent_t ev : E->kern_done)
        if (ev)
            cudaEventDestroy(ev);
    if (E->fwd_done)
        cudaEventDestroy(E->fwd_done);
    if (E->step_start)
        cudaEventDestroy(E->step_start);
    for (auto *vec : {&E->h2d_begin, &E->d2h_begin, &E->d2h_end})
        for (cudaEvent_t ev : *vec)
            if (ev)
                cudaEventDestroy(ev);
    for (cudaEvent_t ev : E->sweep_done)
        if (ev)
            cudaEventDestroy(ev);
    for (cudaStream_t s : {E->s_h2d, E->s_comp, E->s_d2h})
        if (s)
            cudaStreamDestroy(s);
    if (E->window)
        cudaFree(E->window);
}

slide_status engine_create(slide_state *st)
{
    StreamEngine *E = new (std::nothrow) StreamEngine();
    if (!E)
        return fail(SLIDE_ERR_OOM_HOST, "out of host memory for the streaming engine");
    int64_t maxn = 0;
    for (int64_t n : st->numel)
        maxn = n > maxn ? n : maxn;
    const int R = st->cfg.n_replicas;
    E->chunk_bytes = st->cfg.chunk_bytes;
    E->chunks_per_region = (int)((maxn * 4 + E->chunk_bytes - 1) / E->chunk_bytes);
    E->window_bytes = engine_device_bytes(st->cfg, maxn);
    cudaError_t e = cudaMalloc(&E->window, E->window_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        E->window = nullptr;
        destroy_engine_objects(E);
        delete E;
        return fail(SLIDE_ERR_OOM_DEVICE, "cudaMalloc of the HBM window (" + std::to_string(E->window_bytes) +
                                              " bytes) failed");
    }
    e = cudaMemset(E->window, 0, E->window_bytes);
    char *p = (char *)E->window;
    for (Slot &s : E->slots) {
        for (int r = 0; r < kRegions; ++r) {
            s.arr[r] = (float *)p;
            p += align_up((size_t)maxn * 4);
        }
        s.w = (uint16_t *)p;
        p += align_up((size_t)maxn * 2);
        for (int r = 0; r < R; ++r) {
            s.g[r] = p;
            p += align_up((size_t)maxn * grad_bytes(st->cfg));
        }
        s.scratch.partials = (double *)p;
        s.scratch.coef = (float *)(p + align_up(sizeof(double) * kMaxPartials));
        s.scratch.status = (unsigned *)(s.scratch.coef + 1);
        p += scratch_bytes();
        for (int r = 0; r < kRegions && e == cudaSuccess; ++r) {
            s.freed[r].assign(E->chunks_per_region, nullptr);
            for (auto &ev : s.freed[r])
                if (e == cudaSuccess)
                    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        }
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&s.w_freed, cudaEventDisableTiming);
    }
    const size_t L = st->layers.size();
    E->h2d_done.assign(L, nullptr);
    E->theta_done.assign(L, nullptr);
    E->kern_done.assign(L, nullptr);
    E->h2d_begin.assign(L, nullptr);
    E->d2h_begin.assign(L, nullptr);
    E->d2h_end.assign(L, nullptr);
    E->recorded.assign(L, 0);
    // the events of the timeline keep timing; the others are sync-only
    for (size_t l = 0; l < L && e == cudaSuccess; ++l) {
        e = cudaEventCreate(&E->h2d_done[l]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&E->theta_done[l]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&E->kern_done[l]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&E->h2d_begin[l]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&E->d2h_begin[l]);
        if (e == cudaSuccess)
            e = cudaEventCreate(&E->d2h_end[l]);
    }
    if (e == cudaSuccess)
        e = cudaEventCreate(&E->fwd_done);
    if (e == cudaSuccess)
        e = cudaEventCreate(&E->step_start);
    for (int k = 0; k < 3 && e == cudaSuccess; ++k)
        e = cudaEventCreateWithFlags(&E->sweep_done[k], cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_comp, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_d2h, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        slide_status rc = fail_cuda(e, "streaming engine set-up");
        destroy_engine_objects(E);
        delete E;
        return rc;
    }
    st->engine = E;
    st->dev_bytes = E->window_bytes;
    return SLIDE_OK;
}

void engine_destroy(slide_state *st)
{
    StreamEngine *E = st->engine;
    if (!E)
        return;
    for (cudaStream_t s : {E->s_h2d, E->s_comp, E->s_d2h})
        if (s)
            cudaStreamSynchronize(s);
    destroy_engine_objects(E);
    delete E;
    st->engine = nullptr;
}

// Bounded wait for an event: polls cudaEventQuery until it completes or
// timeout_ms passes.
static slide_status wait_event(cudaEvent_t ev, uint32_t timeout_ms, const char *what)
{
    using clock = std::chrono::steady_clock;
    const auto deadline = clock::now() + std::chrono::milliseconds(timeout_ms);
    int spins = 0;
    for (;;) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess)
            return SLIDE_OK;
        if (e != cudaErrorNotReady)
            return fail_cuda(e, what);
        if (clock::now() >= deadline)
            return fail(SLIDE_ERR_TIMEOUT, std::string(what) + ": timed out");
        if (++spins > 64)
            std::this_thread::sleep_for(std::chrono::microseconds(100));
    }
}

// Copy `bytes` between host and window in chunks of the engine's chunk size.
// Copy-in (dir = H2D): chunk k of region `region` first waits for that
// chunk's freed event.  Copy-out (D2H): chunk k records the freed event.
static cudaError_t copy_region(StreamEngine *E, Slot &slot, int region, void *dst, const void *src,
                               size_t bytes, cudaMemcpyKind dir, cudaStream_t s)
{
    const size_t C = (size_t)E->chunk_bytes;
    int k = 0;
    for (size_t off = 0; off < bytes; off += C, ++k) {
        const size_t len = bytes - off < C ? bytes - off : C;
        cudaError_t e;
        if (dir == cudaMemcpyHostToDevice) {
            e = cudaStreamWaitEvent(s, slot.freed[region][k], 0);
            if (e != cudaSuccess)
                return e;
        }
        e = cudaMemcpyAsync((char *)dst + off, (const char *)src + off, len, dir, s);
        if (e != cudaSuccess)
            return e;
        if (dir == cudaMemcpyDeviceToHost) {
            e = cudaEventRecord(slot.freed[region][k], s);
            if (e != cudaSuccess)
                return e;
        }
    }
    return cudaSuccess;
}

slide_status engine_step(slide_state *st, slide_grad_fn fn, void *user, const slide_adam_hparams &hp)
{
    StreamEngine *E = st->engine;
    const int L = (int)st->layers.size();
    const int R = st->cfg.n_replicas;
    const int64_t t = st->layers[0].t + 1;
    const AdamScalars sc = adam_scalars_for(hp, t);
    const bool clip = hp.max_grad_norm > 0.0f;
    const bool check = (st->cfg.flags & SLIDE_FLAG_CHECK_FINITE) != 0;
    cudaError_t e = cudaSuccess;
    slide_status rc = SLIDE_OK;
    int done_units = 0;  // units whose update and write-back were enqueued (from L-1 down)

    for (int l = 0; l < L; ++l)
        E->recorded[l] = 0;
    e = cudaEventRecord(E->step_start, E->s_h2d);
    // forward sweep: deliver the BF16 copy of every unit, in order
    for (int l = 0; l < L && e == cudaSuccess; ++l) {
        Slot &s = E->slots[l % kSlots];
        const LayerState &U = st->layers[l];
        if (U.n > 0) {
            e = cudaStreamWaitEvent(E->s_h2d, s.w_freed, 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(s.w, U.w, (size_t)U.n * 2, cudaMemcpyHostToDevice, E->s_h2d);
        }
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(E->fwd_done, E->s_h2d);

    auto copy_in = [&](int l) -> cudaError_t {
        Slot &s = E->slots[l % kSlots];
        const LayerState &U = st->layers[l];
        const float *src[kRegions] = {U.theta, U.m, U.v};
        cudaError_t err = cudaEventRecord(E->h2d_begin[l], E->s_h2d);
        for (int r = 0; r < kRegions && err == cudaSuccess; ++r) {
            err = copy_region(E, s, r, s.arr[r], src[r], (size_t)U.n * 4, cudaMemcpyHostToDevice, E->s_h2d);
            if (r == 0 && err == cudaSuccess)
                err = cudaEventRecord(E->theta_done[l], E->s_h2d);
        }
        if (err == cudaSuccess)
            err = cudaEventRecord(E->h2d_done[l], E->s_h2d);
        return err;
    };

    // reverse sweep
    if (e == cudaSuccess && L > 0)
        e = copy_in(L - 1);
    for (int l = L - 1; l >= 0 && e == cudaSuccess && rc == SLIDE_OK; --l) {
        Slot &s = E->slots[l % kSlots];
        LayerState &U = st->layers[l];
        // prefetch the next unit of the sweep into the other slot
        if (l > 0) {
            e = copy_in(l - 1);
            if (e != cudaSuccess)
                break;
        }
        // gradients of l on the compute stream as soon as its master has landed
        // (m and v keep arriving meanwhile), then the update once all of the
        // unit is in and the slot's BF16 buffer has been written back
        e = cudaStreamWaitEvent(E->s_comp, E->theta_done[l], 0);
        if (e != cudaSuccess)
            break;
        if (U.n > 0) {
            void *reps[kMaxReplicas + 1];
            for (int r = 0; r < R; ++r)
                reps[r] = s.g[r];
            reps[R] = s.arr[0];  // the unit's FP32 master in the window (pre-update, read-only)
            int urc = fn(user, l, reps, (slide_stream_t)E->s_comp);
            if (urc != 0) {
                rc = fail(SLIDE_ERR_ABORTED, "grad_fn returned " + std::to_string(urc) + " for unit " +
                                                 std::to_string(l));
                break;
            }
        }
        e = cudaStreamWaitEvent(E->s_comp, E->h2d_done[l], 0);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(E->s_comp, s.w_freed, 0);
        if (e != cudaSuccess)
            break;
        if (U.n > 0) {
            ReplicaPtrs g{};
            for (int r = 0; r < R; ++r)
                g.p[r] = s.g[r];
            int n_partials = 0;
            const bool f32g = (st->cfg.flags & SLIDE_FLAG_FP32_GRADS) != 0;
            if (clip) {
                e = launch_grad_sqnorm(g, R, U.n, s.scratch, &n_partials, st->device, E->s_comp, f32g);
                if (e != cudaSuccess)
                    break;
            }
            e = launch_grad_reduce_adamw_cast(g, R, U.n, s.arr[0], s.arr[1], s.arr[2], s.w, sc, &s.scratch,
                                              n_partials, clip ? hp.max_grad_norm : 0.0f, check, st->device,
                                              E->s_comp, (st->cfg.flags & SLIDE_FLAG_TEST_PIPELINE_STALL) != 0,
                                              f32g);
            if (e != cudaSuccess)
                break;
        }
        e = cudaEventRecord(E->kern_done[l], E->s_comp);
        if (e != cudaSuccess)
            break;
        // write l back: the BF16 copy first (frees the slot for the next kernel), then master/m/v
        e = cudaStreamWaitEvent(E->s_d2h, E->kern_done[l], 0);
        if (e == cudaSuccess)
            e = cudaEventRecord(E->d2h_begin[l], E->s_d2h);
        if (e == cudaSuccess && U.n > 0)
            e = cudaMemcpyAsync(U.w, s.w, (size_t)U.n * 2, cudaMemcpyDeviceToHost, E->s_d2h);
        if (e == cudaSuccess)
            e = cudaEventRecord(s.w_freed, E->s_d2h);
        float *dst[kRegions] = {U.theta, U.m, U.v};
        for (int r = 0; r < kRegions && e == cudaSuccess; ++r)
            e = copy_region(E, s, r, dst[r], s.arr[r], (size_t)U.n * 4, cudaMemcpyDeviceToHost, E->s_d2h);
        if (e == cudaSuccess)
            e = cudaEventRecord(E->d2h_end[l], E->s_d2h);
        if (e == cudaSuccess) {
            E->recorded[l] = 1;
            ++done_units;
        }
    }
    if (e != cudaSuccess && rc == SLIDE_OK)
        rc = fail_cuda(e, "streamed step: enqueue");

    // bounded host waits for everything enqueued on the three streams
    slide_status wrc = SLIDE_OK;
    const cudaStream_t streams[3] = {E->s_h2d, E->s_comp, E->s_d2h};
    for (int k = 0; k < 3 && wrc == SLIDE_OK; ++k) {
        cudaError_t e2 = cudaEventRecord(E->sweep_done[k], streams[k]);
        wrc = e2 == cudaSuccess ? wait_event(E->sweep_done[k], st->cfg.timeout_ms, "streamed step")
                                : fail_cuda(e2, "streamed step: record");
    }
    if (rc == SLIDE_OK && wrc != SLIDE_OK)
        rc = wrc;

    unsigned word = 0;
    if (wrc == SLIDE_OK) {
        for (int k = 0; k < kSlots; ++k) {
            unsigned w = 0;
            if (cudaMemcpy(&w, E->slots[k].scratch.status, sizeof w, cudaMemcpyDeviceToHost) == cudaSuccess && w)
                cudaMemset(E->slots[k].scratch.status, 0, sizeof w);
            word |= w;
        }
        if ((word & 2u) && rc == SLIDE_OK)
            rc = fail(SLIDE_ERR_TIMEOUT, "a pipeline wait inside the update kernel reached its limit");
    }
    if (rc == SLIDE_OK) {
        for (LayerState &U : st->layers)
            U.t = t;
        if (check && (word & 1u))
            return fail(SLIDE_ERR_NONFINITE, "a non-finite mean gradient was seen (the step was applied)");
        return SLIDE_OK;
    }
    // Aborted part-way: units whose write-back was enqueued and has completed
    // carry t; the others keep t-1.  Mark the state until a common version is
    // restored with slide_layer_set.
    if (wrc == SLIDE_OK) {
        for (int k = 0; k < done_units; ++k)
            st->layers[L - 1 - k].t = t;
    }
    st->aborted = true;
    return rc;
}

// Timeline of the last step: per unit, milliseconds from the step's start to
// [copy-in begin, master landed, copy-in end, update end, write-back begin,
// write-back end]; then the end of the forward sweep.  NaN where a unit did
// not get that far.
slide_status engine_timeline(slide_state *st, double *out, int64_t cap)
{
    StreamEngine *E = st->engine;
    const int L = (int)st->layers.size();
    if (cap < 6 * (int64_t)L + 1)
        return fail(SLIDE_ERR_INVALID_ARG, "timeline buffer needs 6 * n_layers + 1 doubles");
    const double nan = __builtin_nan("");
    auto since = [&](cudaEvent_t ev) -> double {
        float ms = 0.0f;
        return cudaEventElapsedTime(&ms, E->step_start, ev) == cudaSuccess ? (double)ms : nan;
    };
    for (int l = 0; l < L; ++l) {
        double *o = out + 6 * l;
        if (!E->recorded[l]) {
            for (int k = 0; k < 6; ++k)
                o[k] = nan;
            continue;
        }
        o[0] = since(E->h2d_begin[l]);
        o[1] = since(E->theta_done[l]);
        o[2] = since(E->h2d_done[l]);
        o[3] = since(E->kern_done[l]);
        o[4] = since(E->d2h_begin[l]);
        o[5] = since(E->d2h_end[l]);
    }
    out[6 * L] = since(E->fwd_done);
    cudaGetLastError();  // a NaN entry leaves a sticky-free "not ready" error behind
    return SLIDE_OK;
}

}  // namespace slide
