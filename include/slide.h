/*
 * slide.h — C ABI of the GB300-native per-layer mixed-precision optimizer step
 * of host-resident layer-streaming fine-tuning.
 *
 * What the step computes (the pages print no update equation; the reading is
 * stated here once and used by every entry point):
 *   for each parameter i of layer l, with R gradient replicas g_r (BF16, or
 *   FP32 with SLIDE_FLAG_FP32_GRADS) and
 *   the layer's own 1-based update count t:
 *     g   = (sum_r g_r[i], in FP32, replica order) / R       -- replica mean
 *     g  *= min(1, c / (||g||_2 + 1e-6))   if c = max_grad_norm > 0,
 *           the norm taken over the whole layer's mean gradient
 *     m   = beta1*m + (1-beta1)*g
 *     v   = beta2*v + (1-beta2)*g*g
 *     th  = th*(1 - lr*wd)                                    -- decoupled decay
 *     th  = th - (lr/(1-beta1^t)) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)
 *     w   = bf16_round_nearest_even(th)                        -- compute copy
 *   th, m, v are FP32 and updated in place; w is the BF16 compute copy.
 *   Each line is one FP32 operation (no contraction); the scalars
 *   1-beta, 1-lr*wd, lr/(1-beta1^t), sqrt(1-beta2^t) are formed in double from
 *   the FP32 hyper-parameters and rounded once to FP32.
 *
 * Sources (page title, section):
 *   - "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs":
 *     Prerequisites (mixed-precision Adam keeps 16N bytes: BF16 weights and
 *     gradients 2N + 2N, FP32 master 4N, FP32 Adam moments 8N); Core method
 *     (one authoritative FP32 master and Adam moments (m_l, v_l) per layer,
 *     updated once per iteration by LayerAdam; gradients reduced on the GPU
 *     before they leave it; a bounded, reusable BF16 layer window per GPU);
 *     Method steps (the chain backward -> reduce -> transfer -> Adam per layer,
 *     and the version gate: the next delivery of a layer waits for its update).
 *   - "An Efficient Heterogeneous Co-Design for Fine-Tuning on a Single GPU"
 *     (SlideFormer), sections 2.1-2.2: layer-granular sliding window with
 *     prefetch of the next layer and asynchronous update, a pre-allocated
 *     fixed-size GPU window, FP32 -> BF16 conversion of updated weights.
 *   - "Accelerating the Training of Large Language Models using Efficient
 *     Activation Rematerialization and Optimal Hybrid Parallelism", section 3
 *     (12 = 4 + 4 + 4 bytes of FP32 master and Adam states per parameter) and
 *     section 5.1 (event-serialised copies, ping-pong buffers, pinned memory).
 *
 * Conventions for every function:
 *   - Return a slide_status; nothing throws across the ABI.  On an error the
 *     call enqueues nothing and changes no state (except SLIDE_ERR_ABORTED,
 *     below), and slide_last_error() describes it.
 *   - "device pointer" = address in the GPU's memory (cudaMalloc or a
 *     PyTorch CUDA tensor); "host pointer" = ordinary or pinned CPU memory.
 *   - Device pointers must be 16-byte aligned; lengths are arbitrary.
 *   - A slide_state is not thread-safe: use one from one host thread at a time.
 *   - Streams are cudaStream_t values (NULL = the legacy default stream).
 */
#ifndef SLIDE_H
#define SLIDE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported entry points; everything else in the library is hidden. */
#if defined(__GNUC__)
#define SLIDE_API __attribute__((visibility("default")))
#else
#define SLIDE_API
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *slide_stream_t;

#define SLIDE_ABI_VERSION 2
#define SLIDE_MAX_REPLICAS 8

typedef enum {
    SLIDE_OK = 0,
    SLIDE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or hyper-parameter */
    SLIDE_ERR_OOM_DEVICE = 2,  /* a device allocation failed (all partial ones freed) */
    SLIDE_ERR_OOM_HOST = 3,    /* a pinned host allocation failed (all partial ones freed) */
    SLIDE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    SLIDE_ERR_VERSION = 5,     /* the same-version invariant would be broken */
    SLIDE_ERR_TIMEOUT = 6,     /* a bounded host wait ran out (timeout_ms) */
    SLIDE_ERR_NONFINITE = 7,   /* SLIDE_FLAG_CHECK_FINITE saw a NaN/Inf gradient */
    SLIDE_ERR_ABORTED = 8,     /* a streamed sweep stopped part-way; see slide_model_step_streamed */
    SLIDE_ERR_STATE = 9        /* call does not fit the state's residency */
} slide_status;

enum {
    SLIDE_RESIDENCY_HBM = 0,          /* master, m, v and the BF16 copy live in HBM */
    SLIDE_RESIDENCY_HOST_STREAMED = 1 /* they live in pinned host memory; a 2-slot HBM window */
};

enum {
    SLIDE_FLAG_CHECK_FINITE = 1u,       /* check the mean gradient for NaN/Inf each step */
    SLIDE_FLAG_TEST_PIPELINE_STALL = 2u, /* tests only: the update kernel's copy producer issues nothing,
                                            so the consumers' bounded wait (2 s) runs out and the step
                                            reports SLIDE_ERR_TIMEOUT through slide_layer_status; the
                                            layer's values are then undefined */
    SLIDE_FLAG_FP32_GRADS = 4u,          /* the R gradient replicas are FP32 (FP32 gradient
                                            accumulation), not BF16: every replica pointer then holds
                                            n floats, and the step moves 26 + 4R bytes per parameter */
    SLIDE_FLAG_BF16_COPY_IN_HBM = 8u,    /* streamed residency: keep the BF16 compute copy in HBM
                                            (2 B/param of device memory) instead of the pinned host
                                            mirror; the host holds 12 B/param and the link carries
                                            12 B/param each way per step (the update writes each
                                            unit's resident copy in place: the copy is neither
                                            delivered nor written back, and the window has no BF16
                                            buffers) */
    SLIDE_FLAG_HOST_INPUTS = 32u,        /* HBM residency: reserve device staging for
                                            slide_layer_step_host (two sets of R replica buffers for
                                            the largest layer, used in turn) and a copy stream */
    SLIDE_FLAG_HOST_HUGE_PAGES = 16u     /* streamed residency: back the pinned host state with an
                                            anonymous mapping advised for transparent huge pages and
                                            pinned with cudaHostRegister, instead of cudaHostAlloc
                                            (physically contiguous where the host kernel can provide
                                            it; the mapping is rounded up to the huge page size) */
};

/* Adam hyper-parameters (FP32).  Valid: lr >= 0, 0 <= beta1 < 1,
 * 0 <= beta2 < 1, eps >= 0, weight_decay >= 0, all finite;
 * max_grad_norm <= 0 turns the global clip off. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay, max_grad_norm;
} slide_adam_hparams;

/* State description.  layer_numel is read during slide_state_create only. */
typedef struct {
    int32_t n_layers;            /* >= 1 units (decoder layers, embedding, head ...) */
    const int64_t *layer_numel;  /* host array [n_layers]; each >= 0 parameters */
    int32_t n_replicas;          /* R, 1..SLIDE_MAX_REPLICAS */
    int32_t residency;           /* SLIDE_RESIDENCY_* */
    int32_t window_layers;       /* streamed: must be 2 (0 = 2) */
    int32_t device;              /* CUDA device ordinal */
    uint32_t timeout_ms;         /* streamed: bound of each host wait (0 = 600000) */
    uint32_t flags;              /* SLIDE_FLAG_* */
    int64_t chunk_bytes;         /* streamed: host->device chunk of master, m and v, and the
                                    update's chunk (0 = 256 MiB); bytes of FP32, multiple of 256 */
    int64_t chunk_bytes_d2h;     /* streamed: device->host write-back chunk (0 = chunk_bytes);
                                    bytes of FP32, multiple of 256; both chunk sizes must cut
                                    the largest unit into at most 65536 chunks */
    void *host_arena;            /* streamed: caller-owned pinned host memory (cudaHostAlloc, or
                                    cudaHostRegister with cudaHostRegisterMapped), 256-byte
                                    aligned, to hold the host state instead of an allocation of
                                    the state's own; NULL = the state allocates it.  The state
                                    zeroes and uses the first host_pinned_bytes (slide_state_bytes)
                                    and never frees it; it must outlive the state. */
    int64_t host_arena_bytes;    /* size of host_arena in bytes (>= the state's host bytes) */
} slide_config;

typedef struct slide_state slide_state; /* opaque; owns all of its memory */

/* Gradient callback of the streamed step (stands in for a layer's backward):
 * fill the R replica buffers replica_dev_ptrs[0..R-1] of unit `layer` (device
 * pointers into the window, each layer_numel[layer] BF16 values, or FP32 values
 * with SLIDE_FLAG_FP32_GRADS; owned by the state) with work enqueued on
 * `stream`.  replica_dev_ptrs[R] points to the unit's weights as a backward
 * pass would read them, the version being updated (read-only): the FP32 master
 * in the window (layer_numel[layer] floats; the callback runs once it has
 * landed), or, with SLIDE_FLAG_BF16_COPY_IN_HBM, the unit's resident BF16
 * compute copy (layer_numel[layer] BF16 values; the callback runs at once and
 * master, m and v arrive chunk by chunk behind it).  Return 0 on success; any
 * other value aborts the sweep. */
typedef int (*slide_grad_fn)(void *user, int32_t layer, void *const *replica_dev_ptrs,
                             slide_stream_t stream);

/* Create a state: allocates master, m, v, the BF16 copy (all zero, t = 0) and
 * the per-layer device scratch of the clip reduction; for the streamed
 * residency also the pinned host state (or uses the caller's host_arena), the
 * 2-slot HBM window and the copy and compute streams.  *out is set only on
 * SLIDE_OK.  A caller that creates streamed states one after another can pin
 * one arena once and hand it to each: on the GB300 hosts measured, pinning and
 * freeing 100+ GB repeatedly left later pinned allocations with regions that
 * the copy engines read several times slower.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Prerequisites (the 16N-byte state of mixed-precision Adam) and Core
 * method (one authoritative FP32 master and (m_l, v_l) per layer, held on the
 * host; a bounded, reusable BF16 window per GPU); "An Efficient Heterogeneous
 * Co-Design for Fine-Tuning on a Single GPU", section 2.2 (the window
 * pre-allocated once, of fixed size). */
SLIDE_API slide_status slide_state_create(const slide_config *cfg, slide_state **out);

/* Free everything the state owns after waiting for its own streams.
 * NULL-safe.  Work the caller enqueued on its own streams must be done.
 * Defined by: the same passages as slide_state_create (the state owns all of
 * its memory). */
SLIDE_API void slide_state_destroy(slide_state *st);

/* Bytes slide_state_create would allocate for cfg, computed on the host
 * without touching a GPU: device (HBM) bytes and pinned host bytes.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Prerequisites (16N bytes = 2N + 2N + 4N + 8N); "Accelerating the
 * Training of Large Language Models using Efficient Activation
 * Rematerialization and Optimal Hybrid Parallelism", section 3 (12 bytes of
 * FP32 master and Adam state per parameter). */
SLIDE_API slide_status slide_state_bytes(const slide_config *cfg, int64_t *device_bytes,
                               int64_t *host_pinned_bytes);

/* One optimizer step of one layer (HBM residency): enqueue on `stream` the
 * clip pre-pass (if max_grad_norm > 0) and the fused kernel
 * grad_reduce_adamw_cast for step t = t_layer + 1, then set t_layer = t.
 *   grad_replicas: host array of R device pointers, each to layer_numel[layer]
 *     BF16 values (FP32 values with SLIDE_FLAG_FP32_GRADS), 16-byte aligned;
 *     caller-owned, read-only, and must stay
 *     valid until the enqueued work has run.
 *   bf16_out: device pointer receiving the BF16 copy, or NULL for the state's
 *     own copy (slide_layer_ptrs).  16-byte aligned.
 * Stream-ordered: returns before the GPU finishes.  Steps of one layer must be
 * ordered with each other (same stream, or synchronised by the caller).  With
 * the clip, the fused kernel is launched to overlap the end of the pre-pass
 * (programmatic serialisation); it reads nothing the pre-pass writes before
 * the pre-pass has ended, and both start only after the stream's earlier work.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Core method (the R ranks' gradients of a layer reduced on the GPU;
 * one aggregated Adam update of the layer's FP32 master and moments per
 * iteration, LayerAdam; the result cast FP32 -> BF16 for the next delivery)
 * and Method steps (backward -> reduce -> transfer -> Adam, layer by layer).
 * The clip is the workload's; the pages describe none. */
SLIDE_API slide_status slide_layer_step(slide_state *st, int32_t layer, const void *const *grad_replicas,
                              const slide_adam_hparams *hp, slide_stream_t stream, void *bf16_out);

/* One optimizer step of one layer whose gradient replicas are in host memory
 * and whose new BF16 copy is wanted in host memory (HBM residency, state
 * created with SLIDE_FLAG_HOST_INPUTS): the R replicas are copied into the
 * next of the state's two device staging sets on the state's own copy stream,
 * the step of slide_layer_step runs on `stream` behind that copy, and the new
 * BF16 copy is copied back to host_bf16_out on `stream` (skipped if NULL).
 *   host_grad_replicas: host array of R host pointers (pinned for asynchronous
 *     copies; pageable works, synchronously), each to layer_numel[layer] BF16
 *     values (FP32 with SLIDE_FLAG_FP32_GRADS).  They must hold the gradients
 *     when the call is made (the copy does not wait for work on `stream`) and
 *     stay valid until the copy has run.
 *   host_bf16_out: host pointer receiving layer_numel[layer] BF16 values, or
 *     NULL; valid until `stream` has passed the copy.
 * The copy into a staging set waits only for the update that last read it, so
 * the copy-in of one call overlaps the update of the previous one.
 * Stream-ordered; returns before the GPU finishes.  Calls for one state must
 * come from one host thread.
 * Defined by: the passages of slide_layer_step; the copies are the transfer
 * step of "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Method steps (backward -> reduce -> transfer -> Adam), with the
 * gradients arriving from host memory. */
SLIDE_API slide_status slide_layer_step_host(slide_state *st, int32_t layer, const void *const *host_grad_replicas,
                                             const slide_adam_hparams *hp, slide_stream_t stream,
                                             void *host_bf16_out);

/* One synchronous step of every unit of a host-streamed state (residency
 * SLIDE_RESIDENCY_HOST_STREAMED).  Requires every unit's t to be equal on
 * entry (same version) else SLIDE_ERR_VERSION.
 *   forward sweep, l = 0..L-1: the BF16 copy of unit l is copied host->device
 *     into window slot l%2 (the delivery of the weights a forward would use);
 *   reverse sweep, l = L-1..0: the master of l is copied host->device into
 *     its slot and fn(user, l, replicas, compute stream) produces the R
 *     gradient replicas there; m and v follow chunk by chunk (chunk_bytes of
 *     FP32 each), and the fused step updates each chunk as soon as it has
 *     arrived; each updated chunk's master/m/v and new BF16 copy are copied
 *     device->host right behind its update.  The copy of l-1 into the other
 *     slot overlaps the update of l and the write-back of l+1, taking over the
 *     slot chunk by chunk as l+1's write-back frees it.
 * Each unit is updated exactly once; every t becomes t+1.  Returns after the
 * last write-back is complete.  If fn fails or a wait times out the sweep
 * stops: units already written back carry t+1, the rest t, the state is marked
 * aborted and every later step returns SLIDE_ERR_ABORTED until slide_layer_set
 * has restored a common version on all units.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Core method (the chunked copy pipeline with 64 MiB chunks, the update
 * of a chunk released as soon as it has landed) and Method steps (the version
 * gate: a layer's next delivery waits for its update; one update per layer
 * per iteration); "An Efficient Heterogeneous Co-Design for Fine-Tuning on a
 * Single GPU", section 2.1 (layer-granular sliding window: prefetch of the
 * next layer while the current one computes, asynchronous update);
 * "Accelerating the Training of Large Language Models using Efficient
 * Activation Rematerialization and Optimal Hybrid Parallelism", section 5.1
 * (event-serialised copies on their own streams, ping-pong buffers, pinned
 * host memory). */
SLIDE_API slide_status slide_model_step_streamed(slide_state *st, slide_grad_fn fn, void *user,
                                       const slide_adam_hparams *hp);

/* slide_model_step_streamed without the wait at its end: returns once the
 * step is enqueued, so the next step's first copies (the forward sweep's BF16
 * deliveries) run while this step's last write-backs drain.  Before enqueuing
 * it waits (bounded) for the updates of an earlier asynchronous step, whose
 * write-back may still be in flight; every unit's next delivery and copy-in
 * waits on the device for that unit's own write-back, so the same-version and
 * one-update-per-unit invariants hold as for the synchronous call.  grad_fn
 * may therefore be called while the previous step still runs on the GPU (its
 * work is ordered behind that step's on the stream it is given).  Unit
 * versions advance when the step is enqueued.  slide_streamed_sync waits for
 * the last step and reports its status; slide_layer_get, slide_layer_set,
 * slide_deliver_bf16 and slide_streamed_timeline wait for it first.  A
 * non-finite mean gradient (SLIDE_FLAG_CHECK_FINITE) seen by an asynchronous
 * step is reported by the next slide_streamed_sync or synchronous step; a
 * bounded wait that runs out is reported by the next call and marks the state
 * aborted.
 * Defined by: the passages of slide_model_step_streamed; the overlap across
 * iterations is the layer-streaming pipeline of "An Efficient Heterogeneous
 * Co-Design for Fine-Tuning on a Single GPU", section 2.1 (prefetch of the
 * next layer while the current one is processed and the previous one is
 * updated). */
SLIDE_API slide_status slide_model_step_streamed_async(slide_state *st, slide_grad_fn fn, void *user,
                                                       const slide_adam_hparams *hp);

/* Wait (bounded) for the last slide_model_step_streamed_async of a streamed
 * state and report the status of the asynchronous steps since the last
 * report: SLIDE_ERR_TIMEOUT (a bounded wait ran out; the state is aborted),
 * SLIDE_ERR_NONFINITE (with SLIDE_FLAG_CHECK_FINITE; the step was applied) or
 * SLIDE_OK.  A no-op returning SLIDE_OK when nothing is pending.
 * Defined by: the same passages as slide_model_step_streamed ("SlideDP:
 * Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs", Method steps:
 * a layer is delivered again only after its update is written back). */
SLIDE_API slide_status slide_streamed_sync(slide_state *st);

/* Copy host arrays into a layer's master / m / v (any may be NULL: left
 * unchanged) and set its step count t (>= 0).  Also rewrites the BF16 copy as
 * bf16(master) when master is given.  Synchronous.  Clears the aborted mark
 * once all units share one t.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Core method (the per-layer FP32 master and moments that this call
 * restores, for checkpoints and pre-warm hand-off) and Method steps (the
 * version gate that the common t re-establishes). */
SLIDE_API slide_status slide_layer_set(slide_state *st, int32_t layer, const float *master, const float *m,
                             const float *v, int64_t step);

/* Copy a layer's master / m / v / BF16 copy into host arrays (any may be NULL)
 * and report t.  Synchronous: waits for the state's and the device's work.
 * Defined by: the same passages as slide_layer_set (reading the state back). */
SLIDE_API slide_status slide_layer_get(slide_state *st, int32_t layer, float *master, float *m, float *v,
                             uint16_t *bf16, int64_t *step);

/* Where a layer's arrays live: device pointers for the HBM residency; for the
 * streamed one pinned host pointers (also addressable by kernels through the
 * unified address space), except the BF16 copy, which is a device pointer
 * with SLIDE_FLAG_BF16_COPY_IN_HBM.  Owned by the state, valid until destroy.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Prerequisites and Core method (where the 16N-byte state lives). */
SLIDE_API slide_status slide_layer_ptrs(slide_state *st, int32_t layer, float **master, float **m, float **v,
                              uint16_t **bf16);

/* Clip coefficient used by the last slide_layer_step of `layer` that had the
 * clip on (copied from the device; synchronous).  1.0 before any such step.
 * Defined by: the global grad-norm clip of the workload; no passage of the
 * pages describes a clip (see slide_layer_step). */
SLIDE_API slide_status slide_layer_last_clip_coef(slide_state *st, int32_t layer, float *coef);

/* Status of the steps of `layer` since the previous call (HBM residency):
 * waits for the device, reads and clears the layer's status word, and returns
 *   SLIDE_ERR_TIMEOUT   if a bounded wait inside the update kernel's copy
 *                       pipeline ran out (the step is incomplete; restore the
 *                       layer with slide_layer_set);
 *   SLIDE_ERR_NONFINITE with SLIDE_FLAG_CHECK_FINITE, if a mean gradient held
 *                       a NaN or Inf (the update was applied: the caller
 *                       decides, for example to restore with slide_layer_set);
 *   SLIDE_OK            otherwise.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Method steps (a layer is delivered again only after its update is
 * complete: this call tells the caller that an update did not complete). */
SLIDE_API slide_status slide_layer_status(slide_state *st, int32_t layer);

/* Tracing: CUDA events (cudaEvent_t values, created by the caller) that every
 * following slide_layer_step of this state records on its stream: before the
 * clip pre-pass, before the fused kernel and after it (any may be NULL; all
 * NULL turns tracing off).  The caller may pass fresh events before each step
 * to time every launch separately.  Recording adds no host synchronisation,
 * but with the clip on, an event before the fused kernel makes it wait for
 * the pre-pass's end: without one the fused kernel starts while the pre-pass
 * still runs (where a block of each fits on an SM together), so a traced
 * clipped step can take longer than an untraced one.
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Reproduction (per-phase timing of the step with GPU events). */
SLIDE_API slide_status slide_trace_events(slide_state *st, void *ev_prepass_start,
                                          void *ev_update_start, void *ev_update_stop);

/* The fused step for callers that cannot allocate GPU memory.  The paper has
 * no counterpart to this entry point.  It serves code that may not call
 * cudaMalloc or anything that allocates device memory: an allocator hook or
 * memory-pressure handler that must not re-enter the CUDA allocator it is part
 * of, a process whose GPU memory is a pool owned and capped by a framework (an
 * allocation beside the pool can fail or break its accounting), or a runtime
 * that forbids allocation after start-up.  Such code cannot hold a
 * slide_state, which owns its memory.
 *   The caller owns every array: grad_replicas (host array of n_replicas
 *   device pointers to n BF16 values each), master, m, v (n FP32 values each,
 *   updated in place) and bf16_out (n BF16 values written); all device
 *   pointers, 16-byte aligned.  step is the 1-based update count t of this
 *   update (the caller keeps it).  Same arithmetic as slide_layer_step.
 *   The clip's scratch (4096 per-block partial sums, the coefficient and a
 *   status word, about 32 KiB) is one fixed array in the library's device
 *   memory; every GPU that loads the library holds it until the process
 *   exits.  Limits: 0 <= n <= 2^40 and 1 <= n_replicas <= 8; anything else
 *   returns SLIDE_ERR_INVALID_ARG.
 *   Set-up: the first call on a device (with that device current) looks up
 *   the scratch's device address with cudaGetSymbolAddress and loads every
 *   kernel this entry point can launch.  On a context that loads device code
 *   lazily (the CUDA default) that first call may therefore load the
 *   library's code and allocate its static memory: make it at start-up, and
 *   before any stream capture.  Later calls allocate and free nothing.
 *   Sharing: every call on a device uses the one scratch, and each call
 *   overwrites what the previous one left there (the pre-pass rewrites every
 *   partial sum the update then reads, so nothing needs clearing).  Calls that
 *   may overlap on the GPU (different streams, not ordered) race with each
 *   other: order them.
 *   Errors: argument errors are returned before anything is enqueued.  A
 *   bounded wait inside the update kernel that runs out (2 s) leaves that
 *   step incomplete and marks the shared status word, which
 *   slide_noalloc_status reads (tests make that wait run out by setting the
 *   environment variable SLIDE_TEST_PIPELINE_STALL).  Stream-ordered; returns
 *   before the GPU finishes. */
SLIDE_API slide_status slide_adamw_step_noalloc(int64_t n, int32_t n_replicas, const void *const *grad_replicas,
                                                float *master, float *m, float *v, void *bf16_out,
                                                const slide_adam_hparams *hp, int64_t step,
                                                slide_stream_t stream);

/* Status of the slide_adamw_step_noalloc calls on the current device since the
 * previous slide_noalloc_status: waits for `stream`, reads and clears the
 * shared status word (no allocation), and returns SLIDE_ERR_TIMEOUT if a
 * bounded wait inside the update kernel ran out (that step is incomplete: the
 * caller restores its arrays), else SLIDE_OK.  The paper has no counterpart:
 * it completes slide_adamw_step_noalloc, whose calls have no state to hold a
 * status. */
SLIDE_API slide_status slide_noalloc_status(slide_stream_t stream);

enum {
    SLIDE_DELIVER_FULL = 0,    /* every consumer receives the whole copy from the source */
    SLIDE_DELIVER_SHARDED = 1  /* consumer r receives shard r from the source, then the shards
                                  are gathered on the device (consumer to consumer) */
};

/* Delivery of a layer's BF16 compute copy to R consumer buffers on the GPU
 * (the R ranks' copies of the next forward's weights, modelled as R device
 * buffers).  Source: the state's BF16 copy, in HBM (HBM residency) or in the
 * pinned host mirror (streamed residency).  With SLIDE_DELIVER_FULL each
 * consumer gets a full copy from the source (R x 2n bytes leave the source);
 * with SLIDE_DELIVER_SHARDED consumer r gets elements [r*s, (r+1)*s) (s = n/R
 * rounded up to a multiple of 8, the last shard shorter) from the source, and
 * then copies the other shards from their owners on the device (2n bytes leave
 * the source, (R-1) x 2n move inside HBM).  "SlideDP: Scaling Host-Resident
 * LLM Fine-Tuning Across Multiple GPUs", Core method: full delivery versus
 * sharded delivery plus GPU all-gather.
 *   dst: host array of n_consumers device pointers (16-byte aligned), each to
 *   layer_numel[layer] BF16 values; n_consumers in [1, 8].  Stream-ordered on
 *   `stream`; the source must not be updated until the delivery has run.
 * Defined by: the passage cited above. */
SLIDE_API slide_status slide_deliver_bf16(slide_state *st, int32_t layer, void *const *dst, int32_t n_consumers,
                                          int32_t route, slide_stream_t stream);

/* Timeline of the last slide_model_step_streamed, for tracing how the copies
 * and the updates overlap (host-streamed residency).  out receives, for each
 * unit l, 8 values in milliseconds from the start of that step:
 *   [8l+0] copy-in of master/m/v began   [8l+1] master landed (with the BF16
 *                                        copy in HBM: the first chunk of master,
 *                                        m and v landed)
 *   [8l+2] copy-in ended                 [8l+3] update kernel ended
 *   [8l+4] write-back began              [8l+5] write-back ended
 * (from events on the device), and, by the host clock from the moment the
 * step's first operation was enqueued,
 *   [8l+6] the copy-in of l was fully enqueued
 *   [8l+7] the update and write-back of l were fully enqueued;
 * and out[8L] = end of the forward sweep (BF16 delivery); NaN where a unit
 * did not get that far.  cap = number of doubles in out (>= 8L + 1).
 * Defined by: "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple
 * GPUs", Core method and its figure on the chunked pipeline (how the copies
 * in, the update and the copies out of a layer overlap). */
SLIDE_API slide_status slide_streamed_timeline(slide_state *st, double *out, int64_t cap);

/* Message of the last error on this host thread ("" if none).
 * Defined by: no passage; error reporting of this C ABI. */
SLIDE_API const char *slide_last_error(void);

/* SLIDE_ABI_VERSION of the loaded library.
 * Defined by: no passage; versioning of this C ABI. */
SLIDE_API int32_t slide_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif
