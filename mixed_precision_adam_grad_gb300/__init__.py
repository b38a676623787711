"""GB300-native per-layer mixed-precision optimizer step of host-resident
layer-streaming fine-tuning (R-replica gradient mean -> optional global clip ->
AdamW with bias correction on FP32 master/m/v -> BF16 compute copy).

The compute lives in libslide.so (hand-written CUDA for sm_103a behind the C
ABI of include/slide.h); this package is its thin ctypes binding.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import (SlideError, SlideState, hparams, LIB_PATH,  # noqa: F401
                       slide_abi_version, slide_last_error, slide_state_bytes,
                       slide_state_create, slide_state_destroy, slide_layer_step, slide_layer_step_host,
                       slide_model_step_streamed, slide_model_step_streamed_async, slide_streamed_sync,
                       slide_layer_set, slide_layer_get,
                       slide_layer_ptrs, slide_layer_last_clip_coef, slide_layer_status,
                       slide_trace_events, slide_adamw_step_noalloc, slide_noalloc_status,
                       slide_streamed_timeline, slide_deliver_bf16)


def __getattr__(name):
    if name == "lib":
        from . import _binding
        return _binding._lib()
    raise AttributeError(name)
