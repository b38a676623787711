// stream_engine.cu — host-resident streaming of the optimizer state through
// a 2-slot HBM window (placeholder until the engine lands).
#include "slide_state.h"

namespace slide {

size_t engine_device_bytes(const slide_config &cfg, int64_t max_numel)
{
    (void)cfg;
    (void)max_numel;
    return 0;
}

slide_status engine_create(slide_state *st)
{
    (void)st;
    return fail(SLIDE_ERR_STATE, "host-streamed residency is not available yet");
}

void engine_destroy(slide_state *st) { (void)st; }

slide_status engine_step(slide_state *st, slide_grad_fn fn, void *user, const slide_adam_hparams &hp)
{
    (void)st;
    (void)fn;
    (void)user;
    (void)hp;
    return fail(SLIDE_ERR_STATE, "host-streamed residency is not available yet");
}

}  // namespace slide
