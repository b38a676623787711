// slide_state.h — internal definition of the opaque slide_state and helpers
// shared by slide_api.cu and stream_engine.cu.  Not part of the ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "slide.h"
#include "slide_kernels.h"

namespace slide {

struct StreamEngine;  // stream_engine.cu

// Device staging of slide_layer_step_host (SLIDE_FLAG_HOST_INPUTS): two sets
// of R replica buffers for the largest layer, used in turn, a copy stream for
// the copy-in and, per set, "landed" and "consumed" (updated) events.
struct HostInputs {
    void *stage[2][kMaxReplicas] = {};
    cudaStream_t copy = nullptr;
    cudaEvent_t landed[2] = {nullptr, nullptr};
    cudaEvent_t consumed[2] = {nullptr, nullptr};
    int next = 0;
};

struct LayerState {
    int64_t n = 0;
    float *theta = nullptr;  // HBM or pinned host (streamed)
    float *m = nullptr;
    float *v = nullptr;
    uint16_t *w = nullptr;
    ClipScratch scratch{};   // device scratch of the clip pre-pass (HBM residency)
    int64_t t = 0;           // updates applied so far
};

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess)
            prev = -1;
        ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard()
    {
        if (prev >= 0)
            cudaSetDevice(prev);
    }
};

}  // namespace slide

struct slide_state {
    slide_config cfg{};
    std::vector<int64_t> numel;
    std::vector<slide::LayerState> layers;
    int device = 0;
    void *dev_arena = nullptr;   // one cudaMalloc for all device arrays
    size_t dev_bytes = 0;
    void *host_arena = nullptr;  // pinned host state (streamed residency)
    size_t host_bytes = 0;
    size_t host_map_bytes = 0;   // > 0: host_arena is a registered mapping of this length (huge pages)
    bool host_arena_owned = true;  // false: host_arena is the caller's (never freed here)
    slide::StreamEngine *engine = nullptr;
    slide::HostInputs *hin = nullptr;  // SLIDE_FLAG_HOST_INPUTS
    bool aborted = false;
    cudaEvent_t trace[3] = {nullptr, nullptr, nullptr};  // prepass start, update start, update stop
};

namespace slide {

// Thread-local last-error message and status helpers (slide_api.cu).
slide_status fail(slide_status code, const std::string &msg);
slide_status fail_cuda(cudaError_t e, const char *what);
void clear_error();

// Per-step scalars for update t (1-based) from the FP32 hyper-parameters.
AdamScalars adam_scalars_for(const slide_adam_hparams &hp, int64_t t);
slide_status check_hparams(const slide_adam_hparams *hp);

// Most copy-in or write-back chunks a streamed unit may have.
constexpr int64_t kMaxChunksPerUnit = 65536;

// Byte layout shared by slide_state_bytes and slide_state_create.
constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
inline size_t scratch_bytes() { return align_up(sizeof(double) * kMaxPartials) + kAlign; }
// Staging of SLIDE_FLAG_HOST_INPUTS: 2 sets x R replicas of the largest layer.
inline size_t host_input_bytes(const slide_config &cfg, int64_t max_numel)
{
    if (!(cfg.flags & SLIDE_FLAG_HOST_INPUTS))
        return 0;
    const size_t g = (cfg.flags & SLIDE_FLAG_FP32_GRADS) ? 4 : 2;
    return 2 * (size_t)cfg.n_replicas * align_up((size_t)max_numel * g);
}

// Streamed residency (stream_engine.cu).
slide_status engine_create(slide_state *st);
void engine_destroy(slide_state *st);
size_t engine_device_bytes(const slide_config &cfg, int64_t max_numel);
slide_status engine_step(slide_state *st, slide_grad_fn fn, void *user, const slide_adam_hparams &hp,
                         bool wait_for_end);
// Wait for a step enqueued by slide_model_step_streamed_async (no-op otherwise)
// and report the status words of the steps since the last report.
slide_status engine_sync(slide_state *st);
// Wait for such a step without reading the status words.
slide_status engine_quiesce(slide_state *st);
slide_status engine_timeline(slide_state *st, double *out, int64_t cap);
// A device buffer of the window (idle between steps) of *capacity bytes, for
// moving data between caller memory and the pinned state by DMA only.
void *engine_staging(slide_state *st, size_t *capacity);

}  // namespace slide
