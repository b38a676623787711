"""Seeded synthetic inputs for the tests and the benchmark (ctypes wrapper).

Both the oracle's inputs (host library, plain C + OpenMP) and the GPU runs'
inputs (device library, CUDA) come from here and are bit-identical for the
same (seed, unit, step, replica, index).  The module holds no optimizer
arithmetic: a Philox4x32-10 counter-based generator and the shaping of its
output into the workloads' distributions (synth_rng.h).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_HERE, "libsynth_host.so")
_DEV_SO = os.path.join(_HERE, "libsynth_dev.so")
_HDRS = [os.path.join(_HERE, f) for f in ("synth_rng.h", "synth.h")]
_lock = threading.Lock()
_host = None
_dev = None

GRAD_NORMAL = 0
GRAD_STUDENT3 = 1
TAG_MASTER, TAG_GRAD, TAG_CHI, TAG_ZERO, TAG_SCALE, TAG_MOMENT = range(6)


class GradSpec(C.Structure):
    _fields_ = [("seed", C.c_uint32), ("kind", C.c_int32), ("zero_prob", C.c_float),
                ("pad_", C.c_float)]


class ModelGrads(C.Structure):
    """User data of the device gradient callback for the host-streamed step."""
    _fields_ = [("spec", GradSpec), ("n_units", C.c_int32), ("n_replicas", C.c_int32),
                ("step", C.c_uint32), ("unit_id_base", C.c_uint32),
                ("unit_numel", C.c_void_p), ("seg_begin", C.c_void_p),
                ("seg_offset", C.c_void_p), ("seg_len", C.c_void_p),
                ("seg_scale", C.c_void_p), ("default_scale", C.c_float), ("fp32_grads", C.c_int32)]


class PoolGrads(C.Structure):
    """User data of the pool-copy gradient callback."""
    _fields_ = [("n_replicas", C.c_int32), ("n_pool", C.c_int32), ("step", C.c_uint32),
                ("fp32_grads", C.c_int32), ("unit_numel", C.c_void_p), ("pool", C.c_void_p)]


def _stale(so, srcs):
    return not os.path.exists(so) or any(os.path.getmtime(so) < os.path.getmtime(s) for s in srcs)


def build_host(force=False) -> str:
    src = os.path.join(_HERE, "synth_host.c")
    with _lock:
        if force or _stale(_HOST_SO, [src] + _HDRS):
            tmp = _HOST_SO + f".tmp{os.getpid()}"
            subprocess.run([os.environ.get("CC", "gcc"), "-std=c99", "-O2", "-ffp-contract=off",
                            "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                           check=True)
            os.replace(tmp, _HOST_SO)
    return _HOST_SO


def build_dev_cmd(out=_DEV_SO):
    src = os.path.join(_HERE, "synth_dev.cu")
    return ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "-o", out, src]


def build_dev(force=False) -> str:
    src = os.path.join(_HERE, "synth_dev.cu")
    with _lock:
        if force or _stale(_DEV_SO, [src] + _HDRS):
            tmp = _DEV_SO + f".tmp{os.getpid()}"
            subprocess.run(build_dev_cmd(tmp), check=True)
            os.replace(tmp, _DEV_SO)
    return _DEV_SO


def host():
    global _host
    if _host is None:
        L = C.CDLL(build_host())
        P = C.c_void_p
        u32, i64 = C.c_uint32, C.c_int64
        L.syn_host_fill_master.argtypes = [P, i64, i64, u32, u32, C.c_float]
        L.syn_host_fill_grad.argtypes = [P, i64, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float]
        L.syn_host_gather_master.argtypes = [P, P, i64, u32, u32, C.c_float]
        L.syn_host_gather_grad.argtypes = [P, P, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float]
        L.syn_host_fill_grad_f32.argtypes = [P, i64, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float]
        L.syn_host_gather_grad_f32.argtypes = [P, P, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float]
        L.syn_host_uniform.restype = C.c_float
        L.syn_host_uniform.argtypes = [u32, u32, u32, u32, u32, C.c_uint64]
        L.syn_host_philox.argtypes = [P, P, P]
        L.syn_host_normals.argtypes = [P, i64, u32, u32, u32, u32, u32]
        _host = L
    return _host


def dev():
    global _dev
    if _dev is None:
        L = C.CDLL(build_dev())
        P = C.c_void_p
        u32, i64 = C.c_uint32, C.c_int64
        L.syn_dev_fill_master.argtypes = [P, i64, i64, u32, u32, C.c_float, P]
        L.syn_dev_fill_grad.argtypes = [P, i64, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float, P]
        L.syn_dev_normals.argtypes = [P, i64, u32, u32, u32, u32, u32, P]
        L.syn_dev_fill_grad_f32.argtypes = [P, i64, i64, C.POINTER(GradSpec), u32, u32, u32, C.c_float, P]
        L.syn_dev_grad_fn.argtypes = [P, C.c_int32, P, P]
        L.syn_dev_pool_grad_fn.argtypes = [P, C.c_int32, P, P]
        _dev = L
    return _dev


def grad_fn_address() -> int:
    """Address of the C gradient callback (for the streamed model step)."""
    return C.cast(dev().syn_dev_grad_fn, C.c_void_p).value


def pool_grad_fn_address() -> int:
    """Address of the pool-copy gradient callback."""
    return C.cast(dev().syn_dev_pool_grad_fn, C.c_void_p).value


def spec(seed, kind=GRAD_NORMAL, zero_prob=0.0) -> GradSpec:
    return GradSpec(seed, kind, zero_prob, 0.0)


# ---- host ---------------------------------------------------------------

def philox(ctr, key):
    c = (C.c_uint32 * 4)(*ctr)
    k = (C.c_uint32 * 2)(*key)
    o = (C.c_uint32 * 4)()
    host().syn_host_philox(c, k, o)
    return list(o)


def normals(n, seed, tag, a=0, b=0, c=0) -> np.ndarray:
    out = np.empty(n, np.float32)
    host().syn_host_normals(out.ctypes.data, n, seed, tag, a, b, c)
    return out


def uniform(seed, tag, a, b, c, i) -> float:
    return host().syn_host_uniform(seed, tag, a, b, c, i)


def master(n, seed, unit=0, scale=0.02, offset=0) -> np.ndarray:
    out = np.empty(n, np.float32)
    host().syn_host_fill_master(out.ctypes.data, n, offset, seed, unit, scale)
    return out


def grad(n, sp: GradSpec, unit, step, replica, scale, offset=0) -> np.ndarray:
    out = np.empty(n, np.uint16)
    host().syn_host_fill_grad(out.ctypes.data, n, offset, C.byref(sp), unit, step, replica, scale)
    return out


def grad_f32(n, sp: GradSpec, unit, step, replica, scale, offset=0) -> np.ndarray:
    """FP32 gradient replica values (before any BF16 rounding)."""
    out = np.empty(n, np.float32)
    host().syn_host_fill_grad_f32(out.ctypes.data, n, offset, C.byref(sp), unit, step, replica, scale)
    return out


def gather_grad_f32(idx, sp: GradSpec, unit, step, replica, scale) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    host().syn_host_gather_grad_f32(out.ctypes.data, idx.ctypes.data, idx.size, C.byref(sp), unit, step,
                                    replica, scale)
    return out


def gather_master(idx, seed, unit=0, scale=0.02) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    host().syn_host_gather_master(out.ctypes.data, idx.ctypes.data, idx.size, seed, unit, scale)
    return out


def gather_grad(idx, sp: GradSpec, unit, step, replica, scale) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.uint16)
    host().syn_host_gather_grad(out.ctypes.data, idx.ctypes.data, idx.size, C.byref(sp), unit, step,
                                replica, scale)
    return out


# ---- device (pointers are raw device addresses; stream is a cudaStream_t) ----

def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with CUDA error {rc}")


def dev_master(ptr, n, seed, unit=0, scale=0.02, offset=0, stream=0):
    _check(dev().syn_dev_fill_master(ptr, n, offset, seed, unit, scale, stream), "syn_dev_fill_master")


def dev_grad(ptr, n, sp: GradSpec, unit, step, replica, scale, offset=0, stream=0):
    _check(dev().syn_dev_fill_grad(ptr, n, offset, C.byref(sp), unit, step, replica, scale, stream),
           "syn_dev_fill_grad")


def dev_grad_f32(ptr, n, sp: GradSpec, unit, step, replica, scale, offset=0, stream=0):
    _check(dev().syn_dev_fill_grad_f32(ptr, n, offset, C.byref(sp), unit, step, replica, scale, stream),
           "syn_dev_fill_grad_f32")


def dev_normals(ptr, n, seed, tag, a=0, b=0, c=0, stream=0):
    _check(dev().syn_dev_normals(ptr, n, seed, tag, a, b, c, stream), "syn_dev_normals")
