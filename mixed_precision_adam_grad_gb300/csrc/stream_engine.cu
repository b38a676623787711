// stream_engine.cu — host-resident streaming of the optimizer state through a
// bounded 2-slot HBM window (the streamed residency of slide_model_step_streamed).
//
// Design sources (page title, section):
//  - "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs",
//    Prerequisites (host-resident layer streaming: persistent state in host
//    memory, a small reusable BF16 layer window on the GPU, layers swapped in
//    forward order for the forward pass and in reverse order for the backward
//    pass) and Core method / Method steps (one authoritative host copy of the
//    FP32 master and Adam moments per layer; per-chunk pipelining: a chunk's
//    update is released as soon as that chunk has arrived; the version gate:
//    the next delivery of a layer waits for its update; slots are reused only
//    after their copies complete).
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
// and the R gradient replicas never leave HBM.  With the BF16 copy kept in
// HBM (SLIDE_FLAG_BF16_COPY_IN_HBM) the window has no BF16 slot: the update
// writes the unit's resident copy in place, there is nothing to deliver or
// write back, and the link carries 12 B each way.
//
// A unit's arrays are split into copy-in chunks of chunk_bytes of FP32 (the
// granule of the host-to-device copies of master, m and v and of the update)
// and write-back chunks of chunk_bytes_d2h of FP32 (the granule of the
// device-to-host copies); the BF16 copy and the replicas use the same element
// ranges.  A copy into bytes of a slot waits for every write-back chunk that
// overlaps them, and a write-back chunk waits for the last update chunk that
// overlaps it (each stream runs in order, so these waits cover everything
// earlier).  Schedule of one step, all enqueued up front, then one bounded
// host wait per stream:
//  forward sweep (H2D stream): the BF16 copy of unit l -> slot l%2, in order
//                  (skipped when the copy is kept in HBM);
//  reverse sweep, l = L-1 .. 0, slot s = l%2:
//    H2D stream:     the master of l, then its m and v chunk by chunk (with
//                    the BF16 copy in HBM: master, m and v interleaved chunk by
//                    chunk); every chunk first waits for the write-back of the
//                    same bytes by the unit that used slot s before (l+2), so
//                    a slot is handed over chunk by chunk;
//    compute stream: grad_fn(l) fills the R replicas (backward's stand-in) --
//                    once the master has landed, as it reads the master; at
//                    once with the BF16 copy in HBM, where it reads that copy --
//                    and the clip pre-pass runs over the whole unit; then the
//                    fused update of chunk k is launched as soon as its pieces
//                    have landed and the BF16 chunk of l+2 has been written back;
//    D2H stream:     the write-back of chunk k (BF16 copy, master, m, v)
//                    follows its update, each piece recording the event that
//                    the next copy-in to those bytes waits for.
//  So the write-back of l starts while m and v of l are still arriving, the
//  H2D engine fills the other slot with l-1 and the D2H engine drains l+1.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <nvtx3/nvToolsExtCudaRt.h>

#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "slide_kernels.h"
#include "slide_state.h"

namespace slide {

namespace {

constexpr int kSlots = 2;
enum Region { kTheta = 0, kM = 1, kV = 2, kW = 3, kRegions = 4 };

struct Slot {
    float *arr[3] = {nullptr, nullptr, nullptr};  // master, m, v
    uint16_t *w = nullptr;
    void *g[kMaxReplicas] = {};
    ClipScratch scratch{};
    // chunk k of region r has been written back by the unit that used this slot last
    std::vector<cudaEvent_t> freed[kRegions];  // per write-back chunk
    std::vector<cudaEvent_t> mv_landed;  // copy-in chunk k of m and v has arrived
    std::vector<cudaEvent_t> upd_done;   // copy-in chunk k has been updated
};

size_t grad_bytes(const slide_config &cfg) { return (cfg.flags & SLIDE_FLAG_FP32_GRADS) ? 4 : 2; }

// The window holds the BF16 copy only when the copy lives in host memory.
bool bf16_slot(const slide_config &cfg) { return (cfg.flags & SLIDE_FLAG_BF16_COPY_IN_HBM) == 0; }

size_t slot_bytes(int64_t maxn, int R, size_t gsize, bool w_slot)
{
    return 3 * align_up((size_t)maxn * 4) + (w_slot ? align_up((size_t)maxn * 2) : 0) +
           align_up((size_t)maxn * gsize) * (size_t)R + scratch_bytes();
}

// Element range of chunk k of a unit of n parameters.
struct Chunk {
    int64_t off, len;
};

}  // namespace

struct StreamEngine {
    void *window = nullptr;
    size_t window_bytes = 0;
    Slot slots[kSlots];
    int64_t chunk_elems = 0;  // parameters per copy-in (and update) chunk
    int64_t out_elems = 0;    // parameters per write-back chunk
    int max_chunks = 0;       // copy-in chunks of the largest unit
    int max_out = 0;          // write-back chunks of the largest unit
    size_t gsize = 2;         // bytes per gradient value
    cudaStream_t s_h2d = nullptr, s_comp = nullptr, s_d2h = nullptr;
    // per unit, timing events (also the timeline of the last step)
    std::vector<cudaEvent_t> h2d_begin, theta_done, h2d_done, kern_done, d2h_begin, d2h_end;
    // per unit: its whole write-back (BF16 copy, master, m, v) has reached host
    // memory; the next step's delivery and copy-in of the unit wait for it
    std::vector<cudaEvent_t> wb_done;
    bool pending = false;          // a step was enqueued without waiting for its end
    bool nonfinite_seen = false;   // such a step saw a non-finite mean gradient (not yet reported)
    std::vector<char> recorded;  // unit reached its write-back in the last step
    // host clock (ms since the step's first event was enqueued) at which the
    // copy-in of unit l, and its update and write-back, were fully enqueued
    std::vector<double> host_copyin_enqueued, host_unit_enqueued;
    cudaEvent_t step_start = nullptr, fwd_done = nullptr;
    cudaEvent_t sweep_done[3] = {nullptr, nullptr, nullptr};  // end of the H2D, compute, D2H streams

    Chunk chunk(int64_t n, int k) const
    {
        const int64_t off = (int64_t)k * chunk_elems;
        const int64_t len = n - off < chunk_elems ? n - off : chunk_elems;
        return {off, len};
    }
    int n_chunks(int64_t n) const { return (int)((n + chunk_elems - 1) / chunk_elems); }
    Chunk out_chunk(int64_t n, int q) const
    {
        const int64_t off = (int64_t)q * out_elems;
        const int64_t len = n - off < out_elems ? n - off : out_elems;
        return {off, len};
    }
    int n_out(int64_t n) const { return (int)((n + out_elems - 1) / out_elems); }
    // make `stream` wait until every write-back chunk of `region` of slot s
    // that overlaps elements [c.off, c.off + c.len) has completed
    cudaError_t wait_freed(cudaStream_t stream, const Slot &s, int region, const Chunk &c) const
    {
        cudaError_t e = cudaSuccess;
        if (c.len <= 0)
            return e;
        const int q0 = (int)(c.off / out_elems), q1 = (int)((c.off + c.len - 1) / out_elems);
        for (int q = q0; q <= q1 && e == cudaSuccess; ++q)
            e = cudaStreamWaitEvent(stream, s.freed[region][q], 0);
        return e;
    }
};

size_t engine_device_bytes(const slide_config &cfg, int64_t max_numel)
{
    return kSlots * slot_bytes(max_numel, cfg.n_replicas, grad_bytes(cfg), bf16_slot(cfg));
}

static void destroy_engine_objects(StreamEngine *E)
{
    auto kill = [](std::vector<cudaEvent_t> &v) {
        for (cudaEvent_t ev : v)
            if (ev)
                cudaEventDestroy(ev);
        v.clear();
    };
    for (Slot &s : E->slots) {
        for (auto &v : s.freed)
            kill(v);
        kill(s.mv_landed);
        kill(s.upd_done);
    }
    for (auto *v : {&E->h2d_begin, &E->theta_done, &E->h2d_done, &E->kern_done, &E->d2h_begin, &E->d2h_end})
        kill(*v);
    kill(E->wb_done);
    for (cudaEvent_t ev : {E->step_start, E->fwd_done, E->sweep_done[0], E->sweep_done[1], E->sweep_done[2]})
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
    E->gsize = grad_bytes(st->cfg);
    E->chunk_elems = st->cfg.chunk_bytes / 4;  // chunk sizes are positive multiples of 256
    E->out_elems = st->cfg.chunk_bytes_d2h / 4;
    E->max_chunks = E->n_chunks(maxn);
    E->max_out = E->n_out(maxn);
    E->window_bytes = engine_device_bytes(st->cfg, maxn);
    cudaError_t e = cudaMalloc(&E->window, E->window_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        E->window = nullptr;
        const size_t want = E->window_bytes;
        destroy_engine_objects(E);
        delete E;
        return fail(SLIDE_ERR_OOM_DEVICE, "cudaMalloc of the HBM window (" + std::to_string(want) + " bytes) failed");
    }
    e = cudaMemset(E->window, 0, E->window_bytes);
    char *p = (char *)E->window;
    for (Slot &s : E->slots) {
        for (int r = 0; r < 3; ++r) {
            s.arr[r] = (float *)p;
            p += align_up((size_t)maxn * 4);
        }
        if (bf16_slot(st->cfg)) {
            s.w = (uint16_t *)p;
            p += align_up((size_t)maxn * 2);
        }
        for (int r = 0; r < R; ++r) {
            s.g[r] = p;
            p += align_up((size_t)maxn * E->gsize);
        }
        s.scratch.partials = (double *)p;
        s.scratch.coef = (float *)(p + align_up(sizeof(double) * kMaxPartials));
        s.scratch.status = (unsigned *)(s.scratch.coef + 1);
        p += scratch_bytes();
        auto make = [&](std::vector<cudaEvent_t> &v, int count) {
            v.assign(count, nullptr);
            for (auto &ev : v)
                if (e == cudaSuccess)
                    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        };
        for (auto &v : s.freed)
            make(v, E->max_out);
        make(s.mv_landed, E->max_chunks);
        make(s.upd_done, E->max_chunks);
    }
    const size_t L = st->layers.size();
    for (auto *v : {&E->h2d_begin, &E->theta_done, &E->h2d_done, &E->kern_done, &E->d2h_begin, &E->d2h_end}) {
        v->assign(L, nullptr);
        for (auto &ev : *v)
            if (e == cudaSuccess)
                e = cudaEventCreate(&ev);
    }
    E->wb_done.assign(L, nullptr);
    for (auto &ev : E->wb_done)
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    E->recorded.assign(L, 0);
    E->host_copyin_enqueued.assign(L, __builtin_nan(""));
    E->host_unit_enqueued.assign(L, __builtin_nan(""));
    if (e == cudaSuccess)
        e = cudaEventCreate(&E->step_start);
    if (e == cudaSuccess)
        e = cudaEventCreate(&E->fwd_done);
    for (int k = 0; k < 3 && e == cudaSuccess; ++k)
        e = cudaEventCreateWithFlags(&E->sweep_done[k], cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_comp, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&E->s_d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) {
        // names for a profiler's timeline (no effect without one attached)
        nvtxNameCudaStreamA(E->s_h2d, "slide host-to-device");
        nvtxNameCudaStreamA(E->s_comp, "slide update");
        nvtxNameCudaStreamA(E->s_d2h, "slide device-to-host");
    }
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

void *engine_staging(slide_state *st, size_t *capacity)
{
    StreamEngine *E = st->engine;
    if (!E) {
        *capacity = 0;
        return nullptr;
    }
    int64_t maxn = 0;
    for (int64_t n : st->numel)
        maxn = n > maxn ? n : maxn;
    *capacity = (size_t)maxn * 4;
    return E->slots[0].arr[0];
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

// Read and clear the slots' status words (their kernels must be done):
// bit 1, a pipeline wait in the update kernel ran out; bit 0, a non-finite
// mean gradient (with SLIDE_FLAG_CHECK_FINITE).
static unsigned take_slot_word(slide_state *st)
{
    StreamEngine *E = st->engine;
    unsigned word = 0;
    for (int k = 0; k < kSlots; ++k) {
        unsigned w = 0;
        if (cudaMemcpy(&w, E->slots[k].scratch.status, sizeof w, cudaMemcpyDeviceToHost) == cudaSuccess && w)
            cudaMemset(E->slots[k].scratch.status, 0, sizeof w);
        word |= w;
    }
    return word;
}

// Wait (bounded) for a step enqueued without waiting for its end: its
// update work only (the write-back may still drain), or everything.
static slide_status wait_pending(slide_state *st, bool everything)
{
    StreamEngine *E = st->engine;
    if (!E || !E->pending)
        return SLIDE_OK;
    const int last = everything ? 3 : 2;  // sweep_done: H2D, compute, D2H
    for (int k = 0; k < last; ++k) {
        slide_status rc = wait_event(E->sweep_done[k], st->cfg.timeout_ms, "streamed step (pipelined)");
        if (rc != SLIDE_OK) {
            st->aborted = true;
            return rc;
        }
    }
    if (everything)
        E->pending = false;
    return SLIDE_OK;
}

slide_status engine_quiesce(slide_state *st)
{
    return st->engine ? wait_pending(st, true) : SLIDE_OK;
}

slide_status engine_sync(slide_state *st)
{
    StreamEngine *E = st->engine;
    if (!E)
        return SLIDE_OK;
    slide_status rc = wait_pending(st, true);
    if (rc != SLIDE_OK)
        return rc;
    const unsigned word = take_slot_word(st);
    if (word & 2u) {
        st->aborted = true;
        return fail(SLIDE_ERR_TIMEOUT, "a pipeline wait inside the update kernel reached its limit");
    }
    const bool nonfinite = (word & 1u) || E->nonfinite_seen;
    E->nonfinite_seen = false;
    if (nonfinite && (st->cfg.flags & SLIDE_FLAG_CHECK_FINITE))
        return fail(SLIDE_ERR_NONFINITE, "a non-finite mean gradient was seen (the step was applied)");
    return SLIDE_OK;
}

slide_status engine_step(slide_state *st, slide_grad_fn fn, void *user, const slide_adam_hparams &hp,
                         bool wait_for_end)
{
    StreamEngine *E = st->engine;
    if (E->pending) {
        // the step before was enqueued without waiting: let its updates finish
        // (its write-back may keep draining behind this step's first copies)
        slide_status prc = wait_pending(st, false);
        if (prc != SLIDE_OK)
            return prc;
        const unsigned word = take_slot_word(st);
        if (word & 2u) {
            st->aborted = true;
            return fail(SLIDE_ERR_TIMEOUT, "a pipeline wait inside the update kernel reached its limit");
        }
        if (word & 1u)
            E->nonfinite_seen = true;  // reported at the next sync or synchronous step
    }
    const int L = (int)st->layers.size();
    const int R = st->cfg.n_replicas;
    const int64_t t = st->layers[0].t + 1;
    const AdamScalars sc = adam_scalars_for(hp, t);
    const bool clip = hp.max_grad_norm > 0.0f;
    const bool check = (st->cfg.flags & SLIDE_FLAG_CHECK_FINITE) != 0;
    const bool stall = (st->cfg.flags & SLIDE_FLAG_TEST_PIPELINE_STALL) != 0;
    const bool f32g = (st->cfg.flags & SLIDE_FLAG_FP32_GRADS) != 0;
    const bool w_slot = bf16_slot(st->cfg);  // false: the BF16 copy is updated in place in HBM
    cudaError_t e = cudaSuccess;
    slide_status rc = SLIDE_OK;
    int done_units = 0;  // units whose update and write-back were enqueued (from L-1 down)

    for (int l = 0; l < L; ++l) {
        E->recorded[l] = 0;
        E->host_copyin_enqueued[l] = E->host_unit_enqueued[l] = __builtin_nan("");
    }
    // Profiler ranges (host side: when each part was enqueued): the step, and
    // each unit of the reverse sweep.  No effect without a profiler attached.
    struct Range {
        explicit Range(const std::string &name) { nvtxRangePushA(name.c_str()); }
        ~Range() { nvtxRangePop(); }
    } step_range("slide streamed step t=" + std::to_string(t));
    e = cudaEventRecord(E->step_start, E->s_h2d);
    const auto host_t0 = std::chrono::steady_clock::now();
    auto host_ms = [&]() {
        return std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - host_t0).count();
    };

    // forward sweep: deliver the BF16 copy of every unit, in order (a copy
    // kept in HBM is already where the forward pass reads it)
    for (int l = 0; l < L && w_slot && e == cudaSuccess; ++l) {
        Slot &s = E->slots[l % kSlots];
        const LayerState &U = st->layers[l];
        // the host mirror of l holds the previous step's copy once its write-back is done
        e = cudaStreamWaitEvent(E->s_h2d, E->wb_done[l], 0);
        for (int k = 0; k < E->n_chunks(U.n) && e == cudaSuccess; ++k) {
            const Chunk c = E->chunk(U.n, k);
            e = E->wait_freed(E->s_h2d, s, kW, c);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(s.w + c.off, U.w + c.off, (size_t)c.len * 2, cudaMemcpyHostToDevice,
                                    E->s_h2d);
        }
    }
    if (e == cudaSuccess)
        e = cudaEventRecord(E->fwd_done, E->s_h2d);

    // copy-in of master, m, v of unit l (H2D stream).  With the BF16 copy in
    // HBM the gradient callback reads that resident copy, not the master, so
    // master, m and v arrive interleaved chunk by chunk and the update of chunk
    // k waits only for its own three pieces; otherwise the whole master comes
    // first (the callback reads it), then m and v chunk by chunk.
    auto copy_in = [&](int l) -> cudaError_t {
        Slot &s = E->slots[l % kSlots];
        const LayerState &U = st->layers[l];
        const int K = E->n_chunks(U.n);
        // the host master, m and v of l hold the previous step's values once
        // its write-back is done
        cudaError_t err = cudaStreamWaitEvent(E->s_h2d, E->wb_done[l], 0);
        if (err == cudaSuccess)
            err = cudaEventRecord(E->h2d_begin[l], E->s_h2d);
        if (!w_slot) {
            for (int k = 0; k < K && err == cudaSuccess; ++k) {
                const Chunk c = E->chunk(U.n, k);
                const float *src[3] = {U.theta, U.m, U.v};
                for (int r = 0; r < 3 && err == cudaSuccess; ++r) {
                    err = E->wait_freed(E->s_h2d, s, r, c);
                    if (err == cudaSuccess)
                        err = cudaMemcpyAsync(s.arr[r] + c.off, src[r] + c.off, (size_t)c.len * 4,
                                              cudaMemcpyHostToDevice, E->s_h2d);
                }
                if (err == cudaSuccess)
                    err = cudaEventRecord(s.mv_landed[k], E->s_h2d);
                if (err == cudaSuccess && k == 0)  // the first chunk: the update may start
                    err = cudaEventRecord(E->theta_done[l], E->s_h2d);
            }
            if (err == cudaSuccess && K == 0)
                err = cudaEventRecord(E->theta_done[l], E->s_h2d);
            if (err == cudaSuccess)
                err = cudaEventRecord(E->h2d_done[l], E->s_h2d);
            E->host_copyin_enqueued[l] = host_ms();
            return err;
        }
        for (int k = 0; k < K && err == cudaSuccess; ++k) {
            const Chunk c = E->chunk(U.n, k);
            err = E->wait_freed(E->s_h2d, s, kTheta, c);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(s.arr[0] + c.off, U.theta + c.off, (size_t)c.len * 4,
                                      cudaMemcpyHostToDevice, E->s_h2d);
        }
        if (err == cudaSuccess)
            err = cudaEventRecord(E->theta_done[l], E->s_h2d);
        for (int k = 0; k < K && err == cudaSuccess; ++k) {
            const Chunk c = E->chunk(U.n, k);
            err = E->wait_freed(E->s_h2d, s, kM, c);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(s.arr[1] + c.off, U.m + c.off, (size_t)c.len * 4, cudaMemcpyHostToDevice,
                                      E->s_h2d);
            if (err == cudaSuccess)
                err = E->wait_freed(E->s_h2d, s, kV, c);
            if (err == cudaSuccess)
                err = cudaMemcpyAsync(s.arr[2] + c.off, U.v + c.off, (size_t)c.len * 4, cudaMemcpyHostToDevice,
                                      E->s_h2d);
            if (err == cudaSuccess)
                err = cudaEventRecord(s.mv_landed[k], E->s_h2d);
        }
        if (err == cudaSuccess)
            err = cudaEventRecord(E->h2d_done[l], E->s_h2d);
        E->host_copyin_enqueued[l] = host_ms();
        return err;
    };

    // reverse sweep
    if (e == cudaSuccess && L > 0)
        e = copy_in(L - 1);
    for (int l = L - 1; l >= 0 && e == cudaSuccess && rc == SLIDE_OK; --l) {
        Slot &s = E->slots[l % kSlots];
        LayerState &U = st->layers[l];
        const int K = E->n_chunks(U.n);
        Range unit_range("slide unit " + std::to_string(l) + " (slot " + std::to_string(l % kSlots) + ")");
        // prefetch the next unit of the sweep into the other slot
        if (l > 0) {
            e = copy_in(l - 1);
            if (e != cudaSuccess)
                break;
        }
        // gradients of l (as soon as its master has landed, when the callback
        // reads the master; at once when it reads the resident BF16 copy), then
        // the clip pre-pass over the whole unit, then chunk by chunk the update
        if (w_slot) {
            e = cudaStreamWaitEvent(E->s_comp, E->theta_done[l], 0);
            if (e != cudaSuccess)
                break;
        }
        if (U.n > 0) {
            void *reps[kMaxReplicas + 1];
            for (int r = 0; r < R; ++r)
                reps[r] = s.g[r];
            // the weights a backward pass reads, pre-update and read-only: the
            // FP32 master in the window, or the unit's resident BF16 copy
            reps[R] = w_slot ? (void *)s.arr[0] : (void *)U.w;
            int urc = fn(user, l, reps, (slide_stream_t)E->s_comp);
            if (urc != 0) {
                rc = fail(SLIDE_ERR_ABORTED, "grad_fn returned " + std::to_string(urc) + " for unit " +
                                                 std::to_string(l));
                break;
            }
        }
        int n_partials = 0;
        if (clip && U.n > 0) {
            ReplicaPtrs g{};
            for (int r = 0; r < R; ++r)
                g.p[r] = s.g[r];
            e = launch_grad_sqnorm(g, R, U.n, s.scratch, &n_partials, st->device, E->s_comp, f32g);
            if (e != cudaSuccess)
                break;
        }
        for (int k = 0; k < K && e == cudaSuccess; ++k) {
            const Chunk c = E->chunk(U.n, k);
            e = cudaStreamWaitEvent(E->s_comp, s.mv_landed[k], 0);
            if (e == cudaSuccess && w_slot)
                e = E->wait_freed(E->s_comp, s, kW, c);
            if (e != cudaSuccess)
                break;
            ReplicaPtrs gk{};
            for (int r = 0; r < R; ++r)
                gk.p[r] = (const char *)s.g[r] + (size_t)c.off * E->gsize;
            e = launch_grad_reduce_adamw_cast(gk, R, c.len, s.arr[0] + c.off, s.arr[1] + c.off, s.arr[2] + c.off,
                                              (w_slot ? s.w : U.w) + c.off, sc, &s.scratch, n_partials,
                                              clip ? hp.max_grad_norm : 0.0f, check, st->device, E->s_comp, stall,
                                              f32g);
            if (e == cudaSuccess)
                e = cudaEventRecord(s.upd_done[k], E->s_comp);
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(E->kern_done[l], E->s_comp);
        if (e != cudaSuccess)
            break;
        // write-back of l, chunk by chunk behind its update: write-back chunk q
        // waits for the last update chunk that overlaps it
        float *dst[3] = {U.theta, U.m, U.v};
        const int Q = E->n_out(U.n);
        for (int q = 0; q < Q && e == cudaSuccess; ++q) {
            const Chunk c = E->out_chunk(U.n, q);
            const int k_last = (int)((c.off + c.len - 1) / E->chunk_elems);
            e = cudaStreamWaitEvent(E->s_d2h, s.upd_done[k_last], 0);
            if (e == cudaSuccess && q == 0)
                e = cudaEventRecord(E->d2h_begin[l], E->s_d2h);
            if (e == cudaSuccess && w_slot) {
                e = cudaMemcpyAsync(U.w + c.off, s.w + c.off, (size_t)c.len * 2, cudaMemcpyDeviceToHost, E->s_d2h);
                if (e == cudaSuccess)
                    e = cudaEventRecord(s.freed[kW][q], E->s_d2h);
            }
            for (int r = 0; r < 3 && e == cudaSuccess; ++r) {
                e = cudaMemcpyAsync(dst[r] + c.off, s.arr[r] + c.off, (size_t)c.len * 4, cudaMemcpyDeviceToHost,
                                    E->s_d2h);
                if (e == cudaSuccess)
                    e = cudaEventRecord(s.freed[r][q], E->s_d2h);
            }
        }
        if (e == cudaSuccess && K == 0) {
            e = cudaStreamWaitEvent(E->s_d2h, E->kern_done[l], 0);
            if (e == cudaSuccess)
                e = cudaEventRecord(E->d2h_begin[l], E->s_d2h);
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(E->d2h_end[l], E->s_d2h);
        if (e == cudaSuccess)
            e = cudaEventRecord(E->wb_done[l], E->s_d2h);
        if (e == cudaSuccess) {
            E->recorded[l] = 1;
            E->host_unit_enqueued[l] = host_ms();
            ++done_units;
        }
    }
    if (e != cudaSuccess && rc == SLIDE_OK)
        rc = fail_cuda(e, "streamed step: enqueue");

    if (!wait_for_end && rc == SLIDE_OK) {
        // return once enqueued: the next step (or a sync) waits for this one
        const cudaStream_t ss[3] = {E->s_h2d, E->s_comp, E->s_d2h};
        for (int k = 0; k < 3 && e == cudaSuccess; ++k)
            e = cudaEventRecord(E->sweep_done[k], ss[k]);
        if (e == cudaSuccess) {
            E->pending = true;
            for (LayerState &U : st->layers)
                U.t = t;
            return SLIDE_OK;
        }
        rc = fail_cuda(e, "streamed step: record");
    }

    // bounded host waits for everything enqueued on the three streams
    slide_status wrc = SLIDE_OK;
    const cudaStream_t streams[3] = {E->s_h2d, E->s_comp, E->s_d2h};
    for (int k = 0; k < 3 && wrc == SLIDE_OK; ++k) {
        cudaError_t e2 = cudaEventRecord(E->sweep_done[k], streams[k]);
        wrc = e2 == cudaSuccess ? wait_event(E->sweep_done[k], st->cfg.timeout_ms, "streamed step")
                                : fail_cuda(e2, "streamed step: record");
    }
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
    if (rc == SLIDE_OK && wrc != SLIDE_OK)
        rc = wrc;

    E->pending = false;
    if (rc == SLIDE_OK) {
        for (LayerState &U : st->layers)
            U.t = t;
        const bool nonfinite = (word & 1u) || E->nonfinite_seen;
        E->nonfinite_seen = false;
        if (check && nonfinite)
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
// [copy-in begin, master landed, copy-in end, last chunk updated, write-back
// of the first chunk may begin, write-back end] (device events), then [copy-in
// fully enqueued, update and write-back fully enqueued] (host clock); then the
// end of the forward sweep.  NaN where a unit did not get that far.
slide_status engine_timeline(slide_state *st, double *out, int64_t cap)
{
    StreamEngine *E = st->engine;
    const int L = (int)st->layers.size();
    constexpr int kPer = 8;
    if (cap < kPer * (int64_t)L + 1)
        return fail(SLIDE_ERR_INVALID_ARG, "timeline buffer needs 8 * n_layers + 1 doubles");
    if (E->pending) {
        slide_status rc = engine_quiesce(st);
        if (rc != SLIDE_OK)
            return rc;
    }
    const double nan = __builtin_nan("");
    auto since = [&](cudaEvent_t ev) -> double {
        float ms = 0.0f;
        return cudaEventElapsedTime(&ms, E->step_start, ev) == cudaSuccess ? (double)ms : nan;
    };
    for (int l = 0; l < L; ++l) {
        double *o = out + kPer * l;
        o[6] = E->host_copyin_enqueued[l];
        o[7] = E->host_unit_enqueued[l];
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
    out[kPer * L] = since(E->fwd_done);
    cudaGetLastError();
    return SLIDE_OK;
}

}  // namespace slide
