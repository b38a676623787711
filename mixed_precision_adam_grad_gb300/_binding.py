"""ctypes binding of libslide.so: the entry points of include/slide.h under the
same names, with argument marshalling only (every step of the optimizer runs
in the library's CUDA kernels).

Pointers may be given as ints, torch tensors (``data_ptr()``) or numpy arrays
(host memory); streams as ints (``cudaStream_t`` values), torch streams or
None (the legacy default stream).  A non-OK status raises SlideError.  If the
library has not been built the import fails: there is no other code path.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libslide.so")

SLIDE_OK = 0
SLIDE_ERR_INVALID_ARG = 1
SLIDE_ERR_OOM_DEVICE = 2
SLIDE_ERR_OOM_HOST = 3
SLIDE_ERR_CUDA = 4
SLIDE_ERR_VERSION = 5
SLIDE_ERR_TIMEOUT = 6
SLIDE_ERR_NONFINITE = 7
SLIDE_ERR_ABORTED = 8
SLIDE_ERR_STATE = 9
STATUS_NAMES = {0: "SLIDE_OK", 1: "SLIDE_ERR_INVALID_ARG", 2: "SLIDE_ERR_OOM_DEVICE",
                3: "SLIDE_ERR_OOM_HOST", 4: "SLIDE_ERR_CUDA", 5: "SLIDE_ERR_VERSION",
                6: "SLIDE_ERR_TIMEOUT", 7: "SLIDE_ERR_NONFINITE", 8: "SLIDE_ERR_ABORTED",
                9: "SLIDE_ERR_STATE"}

SLIDE_RESIDENCY_HBM = 0
SLIDE_RESIDENCY_HOST_STREAMED = 1
SLIDE_FLAG_CHECK_FINITE = 1
SLIDE_FLAG_TEST_PIPELINE_STALL = 2
SLIDE_FLAG_FP32_GRADS = 4
SLIDE_FLAG_BF16_COPY_IN_HBM = 8
SLIDE_FLAG_HOST_HUGE_PAGES = 16
SLIDE_FLAG_HOST_INPUTS = 32
SLIDE_MAX_REPLICAS = 8
SLIDE_DELIVER_FULL = 0
SLIDE_DELIVER_SHARDED = 1


class SlideError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


class slide_adam_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("max_grad_norm", C.c_float)]


class slide_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("layer_numel", C.POINTER(C.c_int64)),
                ("n_replicas", C.c_int32), ("residency", C.c_int32),
                ("window_layers", C.c_int32), ("device", C.c_int32),
                ("timeout_ms", C.c_uint32), ("flags", C.c_uint32), ("chunk_bytes", C.c_int64),
                ("chunk_bytes_d2h", C.c_int64), ("host_arena", C.c_void_p), ("host_arena_bytes", C.c_int64)]


SLIDE_GRAD_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_int32, C.POINTER(C.c_void_p), C.c_void_p)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -m mixed_precision_adam_grad_gb300.build); there is no fallback path")
    L = C.CDLL(LIB_PATH)
    P, S = C.c_void_p, C.c_int
    L.slide_state_create.argtypes = [C.POINTER(slide_config), C.POINTER(C.c_void_p)]
    L.slide_state_create.restype = S
    L.slide_state_destroy.argtypes = [P]
    L.slide_state_destroy.restype = None
    L.slide_state_bytes.argtypes = [C.POINTER(slide_config), C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
    L.slide_state_bytes.restype = S
    L.slide_layer_step.argtypes = [P, C.c_int32, C.POINTER(C.c_void_p), C.POINTER(slide_adam_hparams), P, P]
    L.slide_layer_step.restype = S
    L.slide_layer_step_host.argtypes = [P, C.c_int32, C.POINTER(C.c_void_p), C.POINTER(slide_adam_hparams), P, P]
    L.slide_layer_step_host.restype = S
    L.slide_model_step_streamed.argtypes = [P, P, P, C.POINTER(slide_adam_hparams)]
    L.slide_model_step_streamed_async.argtypes = [P, P, P, C.POINTER(slide_adam_hparams)]
    L.slide_model_step_streamed_async.restype = S
    L.slide_streamed_sync.argtypes = [P]
    L.slide_streamed_sync.restype = S
    L.slide_model_step_streamed.restype = S
    L.slide_layer_set.argtypes = [P, C.c_int32, P, P, P, C.c_int64]
    L.slide_layer_set.restype = S
    L.slide_layer_get.argtypes = [P, C.c_int32, P, P, P, P, C.POINTER(C.c_int64)]
    L.slide_layer_get.restype = S
    L.slide_layer_ptrs.argtypes = [P, C.c_int32] + [C.POINTER(C.c_void_p)] * 4
    L.slide_layer_ptrs.restype = S
    L.slide_layer_last_clip_coef.argtypes = [P, C.c_int32, C.POINTER(C.c_float)]
    L.slide_layer_last_clip_coef.restype = S
    L.slide_layer_status.argtypes = [P, C.c_int32]
    L.slide_layer_status.restype = S
    L.slide_deliver_bf16.argtypes = [P, C.c_int32, C.POINTER(C.c_void_p), C.c_int32, C.c_int32, P]
    L.slide_deliver_bf16.restype = S
    L.slide_streamed_timeline.argtypes = [P, C.POINTER(C.c_double), C.c_int64]
    L.slide_streamed_timeline.restype = S
    L.slide_trace_events.argtypes = [P, P, P, P]
    L.slide_trace_events.restype = S
    L.slide_adamw_step_noalloc.argtypes = [C.c_int64, C.c_int32, C.POINTER(C.c_void_p), P, P, P, P,
                                           C.POINTER(slide_adam_hparams), C.c_int64, P]
    L.slide_adamw_step_noalloc.restype = S
    L.slide_noalloc_status.argtypes = [P]
    L.slide_noalloc_status.restype = S
    L.slide_last_error.argtypes = []
    L.slide_last_error.restype = C.c_char_p
    L.slide_abi_version.argtypes = []
    L.slide_abi_version.restype = C.c_int32
    return L


_LIB = None


def _lib():
    """The loaded libslide.so (loaded on first use; raises if it was not built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name):
    if name == "lib":
        return _lib()
    raise AttributeError(name)


def _check(rc: int):
    if rc != SLIDE_OK:
        raise SlideError(rc, _lib().slide_last_error().decode(errors="replace"))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):          # torch.Tensor
        return x.data_ptr()
    if hasattr(x, "ctypes"):            # numpy.ndarray (host)
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x).__name__}")


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream                 # torch.cuda.Stream / ExternalStream


def hparams(lr=1e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=0.0):
    return slide_adam_hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm)


def _config(layer_numel: Sequence[int], n_replicas: int, residency: int, device: int,
            flags: int, timeout_ms: int, chunk_bytes: int, window_layers: int, chunk_bytes_d2h: int = 0,
            host_arena=None, host_arena_bytes: int = 0):
    arr = (C.c_int64 * len(layer_numel))(*[int(n) for n in layer_numel])
    cfg = slide_config(len(layer_numel), arr, n_replicas, residency, window_layers, device,
                       timeout_ms, flags, chunk_bytes, chunk_bytes_d2h, _ptr(host_arena), host_arena_bytes)
    cfg._keep = arr
    return cfg


class SlideState:
    """Owner of a slide_state pointer (call slide_state_destroy, or use `with`)."""

    def __init__(self, handle: int, layer_numel, n_replicas, residency):
        self.handle = handle
        self.layer_numel = [int(n) for n in layer_numel]
        self.n_replicas = n_replicas
        self.residency = residency

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        slide_state_destroy(self)

    @property
    def _as_parameter_(self):
        return C.c_void_p(self.handle)


def slide_abi_version() -> int:
    return _lib().slide_abi_version()


def slide_last_error() -> str:
    return _lib().slide_last_error().decode(errors="replace")


def slide_state_bytes(layer_numel, n_replicas, residency=SLIDE_RESIDENCY_HBM, device=0, flags=0,
                      timeout_ms=0, chunk_bytes=0, window_layers=2, chunk_bytes_d2h=0, host_arena=None,
                      host_arena_bytes=0):
    cfg = _config(layer_numel, n_replicas, residency, device, flags, timeout_ms, chunk_bytes, window_layers,
                  chunk_bytes_d2h, host_arena, host_arena_bytes)
    dev, host = C.c_int64(), C.c_int64()
    _check(_lib().slide_state_bytes(C.byref(cfg), C.byref(dev), C.byref(host)))
    return dev.value, host.value


def slide_state_create(layer_numel, n_replicas, residency=SLIDE_RESIDENCY_HBM, device=0, flags=0,
                       timeout_ms=0, chunk_bytes=0, window_layers=2, chunk_bytes_d2h=0, host_arena=None,
                       host_arena_bytes=0) -> SlideState:
    """host_arena: caller-owned pinned host memory (an address, or a pinned
    tensor) of host_arena_bytes bytes for the streamed state; it must outlive
    the state."""
    cfg = _config(layer_numel, n_replicas, residency, device, flags, timeout_ms, chunk_bytes, window_layers,
                  chunk_bytes_d2h, host_arena, host_arena_bytes)
    out = C.c_void_p()
    _check(_lib().slide_state_create(C.byref(cfg), C.byref(out)))
    return SlideState(out.value, layer_numel, n_replicas, residency)


def slide_state_destroy(st: SlideState) -> None:
    if st is not None and st.handle:
        _lib().slide_state_destroy(C.c_void_p(st.handle))
        st.handle = 0


def slide_layer_step(st: SlideState, layer: int, grad_replicas, hp: slide_adam_hparams,
                     stream=None, bf16_out=None) -> None:
    ptrs = [_ptr(g) for g in grad_replicas]
    arr = (C.c_void_p * max(1, len(ptrs)))(*ptrs)
    _check(_lib().slide_layer_step(C.c_void_p(st.handle), layer, arr, C.byref(hp),
                                _stream(stream), _ptr(bf16_out)))


def slide_layer_step_host(st: SlideState, layer: int, host_grad_replicas, hp: slide_adam_hparams,
                          stream=None, host_bf16_out=None) -> None:
    """The step of a layer whose replicas are host arrays (numpy arrays, pinned
    CPU tensors or addresses); the new BF16 copy goes to host_bf16_out."""
    ptrs = [_ptr(g) for g in host_grad_replicas]
    arr = (C.c_void_p * max(1, len(ptrs)))(*ptrs)
    _check(_lib().slide_layer_step_host(C.c_void_p(st.handle), layer, arr, C.byref(hp), _stream(stream),
                                        _ptr(host_bf16_out)))


def slide_model_step_streamed(st: SlideState, fn, user, hp: slide_adam_hparams) -> None:
    """fn: address of a C slide_grad_fn (int) or a SLIDE_GRAD_FN object;
    user: an address (int), a ctypes object (passed by reference) or None."""
    if isinstance(fn, int):
        fn_ptr = C.c_void_p(fn)
    else:
        fn_ptr = C.cast(fn, C.c_void_p)
    if user is None or isinstance(user, int):
        user_ptr = C.c_void_p(user)
    else:
        user_ptr = C.cast(C.byref(user), C.c_void_p)
    _check(_lib().slide_model_step_streamed(C.c_void_p(st.handle), fn_ptr, user_ptr, C.byref(hp)))


def slide_model_step_streamed_async(st: SlideState, fn, user, hp: slide_adam_hparams) -> None:
    """slide_model_step_streamed returning once enqueued (see include/slide.h);
    fn and user must stay alive until the step has been synced."""
    fn_ptr = C.c_void_p(fn) if isinstance(fn, int) else C.cast(fn, C.c_void_p)
    if user is None or isinstance(user, int):
        user_ptr = C.c_void_p(user)
    else:
        user_ptr = C.cast(C.byref(user), C.c_void_p)
    _check(_lib().slide_model_step_streamed_async(C.c_void_p(st.handle), fn_ptr, user_ptr, C.byref(hp)))


def slide_streamed_sync(st: SlideState) -> None:
    _check(_lib().slide_streamed_sync(C.c_void_p(st.handle)))


def slide_layer_set(st: SlideState, layer: int, master=None, m=None, v=None, step: int = 0) -> None:
    _check(_lib().slide_layer_set(C.c_void_p(st.handle), layer, _ptr(master), _ptr(m), _ptr(v), step))


def slide_layer_get(st: SlideState, layer: int, master=None, m=None, v=None, bf16=None) -> int:
    """Copies into the given host arrays (any may be None); returns t."""
    t = C.c_int64()
    _check(_lib().slide_layer_get(C.c_void_p(st.handle), layer, _ptr(master), _ptr(m), _ptr(v),
                               _ptr(bf16), C.byref(t)))
    return t.value


def slide_layer_ptrs(st: SlideState, layer: int):
    ps = [C.c_void_p() for _ in range(4)]
    _check(_lib().slide_layer_ptrs(C.c_void_p(st.handle), layer, *[C.byref(p) for p in ps]))
    return tuple(p.value or 0 for p in ps)


def slide_layer_last_clip_coef(st: SlideState, layer: int) -> float:
    c = C.c_float()
    _check(_lib().slide_layer_last_clip_coef(C.c_void_p(st.handle), layer, C.byref(c)))
    return c.value


def slide_layer_status(st: SlideState, layer: int) -> int:
    """Returns the status code (SLIDE_OK, SLIDE_ERR_NONFINITE or
    SLIDE_ERR_TIMEOUT); raises on other errors."""
    rc = _lib().slide_layer_status(C.c_void_p(st.handle), layer)
    if rc not in (SLIDE_OK, SLIDE_ERR_NONFINITE, SLIDE_ERR_TIMEOUT):
        _check(rc)
    return rc


def _event(e):
    if e is None:
        return None
    if isinstance(e, int):
        return e
    return e.cuda_event                  # torch.cuda.Event (after it was created on the device)


def slide_trace_events(st: SlideState, prepass_start=None, update_start=None, update_stop=None) -> None:
    _check(_lib().slide_trace_events(C.c_void_p(st.handle), _event(prepass_start), _event(update_start),
                                  _event(update_stop)))


def slide_adamw_step_noalloc(n: int, grad_replicas, master, m, v, bf16_out, hp: slide_adam_hparams,
                             step: int, stream=None) -> None:
    """The step for callers that cannot allocate GPU memory: the caller owns
    every array and the 1-based step count; after the first call on a device
    (its one-time set-up) the library allocates nothing."""
    ptrs = [_ptr(g) for g in grad_replicas]
    arr = (C.c_void_p * max(1, len(ptrs)))(*ptrs)
    _check(_lib().slide_adamw_step_noalloc(n, len(ptrs), arr, _ptr(master), _ptr(m), _ptr(v), _ptr(bf16_out),
                                           C.byref(hp), step, _stream(stream)))


def slide_noalloc_status(stream=None) -> int:
    """Status of the no-alloc calls on the current device since the last
    query (SLIDE_OK or SLIDE_ERR_TIMEOUT); raises on other errors."""
    rc = _lib().slide_noalloc_status(_stream(stream))
    if rc not in (SLIDE_OK, SLIDE_ERR_TIMEOUT):
        _check(rc)
    return rc


def slide_streamed_timeline(st: SlideState):
    """Per-unit timeline (ms) of the last streamed step: a list of dicts and
    the end of the forward sweep."""
    L = len(st.layer_numel)
    buf = (C.c_double * (8 * L + 1))()
    _check(_lib().slide_streamed_timeline(C.c_void_p(st.handle), buf, 8 * L + 1))
    keys = ("h2d_begin", "master_landed", "h2d_end", "update_end", "d2h_begin", "d2h_end",
            "host_copyin_enqueued", "host_unit_enqueued")
    units = [dict(zip(keys, buf[8 * l:8 * l + 8])) for l in range(L)]
    return units, buf[8 * L]


def slide_deliver_bf16(st: SlideState, layer: int, dst, route=SLIDE_DELIVER_FULL, stream=None) -> None:
    """Deliver a layer's BF16 copy to len(dst) consumer device buffers."""
    ptrs = [_ptr(d) for d in dst]
    arr = (C.c_void_p * max(1, len(ptrs)))(*ptrs)
    _check(_lib().slide_deliver_bf16(C.c_void_p(st.handle), layer, arr, len(ptrs), route, _stream(stream)))
