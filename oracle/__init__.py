"""The CPU oracle of the per-layer mixed-precision AdamW step (ctypes wrapper).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package; the
product library and its Python binding never do, and nothing in the product
falls back to it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C99, built with
``-O2 -ffp-contract=off``, no fast-math); this module only builds that file
with the host C compiler and marshals numpy arrays into it.  The passages it
follows are listed in ``oracle.h``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_SO = os.path.join(_HERE, "liboracle.so")
_SO_OMP = os.path.join(_HERE, "liboracle_omp.so")
_lock = threading.Lock()
_libs = {}


class Hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float),
                ("max_grad_norm", C.c_float)]


class StepScalars(C.Structure):
    _fields_ = [("beta1", C.c_float), ("one_minus_beta1", C.c_float),
                ("beta2", C.c_float), ("one_minus_beta2", C.c_float),
                ("decay", C.c_float), ("step_size", C.c_float),
                ("bc2_sqrt", C.c_float), ("eps", C.c_float)]


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (host C compiler).  With
    openmp=True the same source is built with -fopenmp into liboracle_omp.so,
    which is used only to time the oracle on all host cores."""
    so = _SO_OMP if openmp else _SO
    with _lock:
        fresh = os.path.exists(so) and all(
            os.path.getmtime(so) >= os.path.getmtime(p) for p in (_SRC, _HDR))
        if fresh and not force:
            return so
        cc = os.environ.get("CC", "gcc")
        tmp = so + f".tmp{os.getpid()}"
        cmd = [cc, "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        if openmp:
            cmd.insert(1, "-fopenmp")
        subprocess.run(cmd, check=True)
        os.replace(tmp, so)
        return so


def lib(openmp: bool = False):
    L = _libs.get(openmp)
    if L is None:
        # ORACLE_SO lets the mutation test load a deliberately broken copy of
        # the oracle, built from an edited oracle.c in a temporary directory.
        so = None if openmp else os.environ.get("ORACLE_SO")
        if not so:
            so = build(openmp=openmp)
        L = C.CDLL(so)
        P = C.c_void_p
        L.oracle_bf16_to_f32.restype = C.c_float
        L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
        L.oracle_f32_to_bf16_rne.restype = C.c_uint16
        L.oracle_f32_to_bf16_rne.argtypes = [C.c_float]
        L.oracle_f32_to_bf16_rne_array.argtypes = [C.c_int64, P, P]
        L.oracle_bf16_to_f32_array.argtypes = [C.c_int64, P, P]
        L.oracle_step_scalars_for.argtypes = [C.POINTER(Hparams), C.c_int64, C.POINTER(StepScalars)]
        L.oracle_grad_mean.argtypes = [C.c_int64, C.c_int32, P, P]
        L.oracle_grad_mean_f32.argtypes = [C.c_int64, C.c_int32, P, P]
        L.oracle_layer_step_f32g.restype = C.c_float
        L.oracle_layer_step_f32g.argtypes = [C.c_int64, C.c_int32, P, P, P, P, P,
                                             C.POINTER(Hparams), C.c_int64]
        L.oracle_layer_step_f64_f32g.restype = C.c_double
        L.oracle_layer_step_f64_f32g.argtypes = [C.c_int64, C.c_int32, P, P, P, P,
                                                 C.POINTER(Hparams), C.c_int64]
        L.oracle_grad_sqnorm.restype = C.c_double
        L.oracle_grad_sqnorm.argtypes = [C.c_int64, P]
        L.oracle_clip_coef.restype = C.c_float
        L.oracle_clip_coef.argtypes = [C.c_double, C.c_float]
        L.oracle_adamw_update.argtypes = [C.c_int64, P, C.c_float, P, P, P, P,
                                          C.POINTER(Hparams), C.c_int64]
        L.oracle_layer_step.restype = C.c_float
        L.oracle_layer_step.argtypes = [C.c_int64, C.c_int32, P, P, P, P, P,
                                        C.POINTER(Hparams), C.c_int64]
        L.oracle_layer_step_f64.restype = C.c_double
        L.oracle_layer_step_f64.argtypes = [C.c_int64, C.c_int32, P, P, P, P,
                                            C.POINTER(Hparams), C.c_int64]
        L.oracle_threads.restype = C.c_int32
        L.oracle_threads.argtypes = []
        _libs[openmp] = L
    return L


def threads(openmp: bool = False) -> int:
    """Threads the oracle's element loops use (1 for the default build)."""
    return lib(openmp).oracle_threads()


def hparams(lr=1e-5, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            max_grad_norm=0.0) -> Hparams:
    return Hparams(lr, beta1, beta2, eps, weight_decay, max_grad_norm)


def _as(a, dtype):
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"expected a C-contiguous {np.dtype(dtype).name} array")
    return a


def _ptr(a) -> int:
    return a.ctypes.data


def _replica_table(grads):
    """Pointer table of the replicas (all BF16 bit patterns as uint16, or all FP32)."""
    n = None
    dtype = grads[0].dtype if len(grads) else np.uint16
    if dtype not in (np.uint16, np.float32):
        raise TypeError("replicas must be uint16 (BF16 bits) or float32")
    for g in grads:
        _as(g, dtype)
        if n is None:
            n = g.size
        elif g.size != n:
            raise ValueError("all replicas must have the same length")
    tab = (C.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    return tab, (n or 0)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().oracle_bf16_to_f32_array(h.size, _ptr(h), _ptr(out))
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f32_to_bf16_rne_array(x.size, _ptr(x), _ptr(out))
    return out


def step_scalars(hp: Hparams, t: int) -> StepScalars:
    s = StepScalars()
    lib().oracle_step_scalars_for(C.byref(hp), t, C.byref(s))
    return s


def _is_f32(grads):
    return len(grads) > 0 and grads[0].dtype == np.float32


def grad_mean(grads) -> np.ndarray:
    tab, n = _replica_table(grads)
    gm = np.empty(n, np.float32)
    fn = lib().oracle_grad_mean_f32 if _is_f32(grads) else lib().oracle_grad_mean
    fn(n, len(grads), tab, _ptr(gm))
    return gm


def grad_sqnorm(gm: np.ndarray) -> float:
    _as(gm, np.float32)
    return lib().oracle_grad_sqnorm(gm.size, _ptr(gm))


def clip_coef(sqnorm: float, max_norm: float) -> float:
    return lib().oracle_clip_coef(sqnorm, max_norm)


def adamw_update(gm, coef, theta, m, v, w, hp: Hparams, t: int) -> None:
    for a in (gm, theta, m, v):
        _as(a, np.float32)
    n = gm.size
    if not (theta.size == m.size == v.size == n):
        raise ValueError("length mismatch")
    wp = None
    if w is not None:
        _as(w, np.uint16)
        if w.size != n:
            raise ValueError("length mismatch")
        wp = _ptr(w)
    lib().oracle_adamw_update(n, _ptr(gm), coef, _ptr(theta), _ptr(m), _ptr(v),
                              wp, C.byref(hp), t)


def layer_step(grads, theta, m, v, w, hp: Hparams, t: int, openmp: bool = False) -> float:
    """One step of a whole layer in place; returns the clip coefficient used.
    openmp=True runs the -fopenmp build (all-core timing only)."""
    tab, n = _replica_table(grads)
    for a in (theta, m, v):
        _as(a, np.float32)
        if a.size != n:
            raise ValueError("length mismatch")
    wp = None
    if w is not None:
        _as(w, np.uint16)
        if w.size != n:
            raise ValueError("length mismatch")
        wp = _ptr(w)
    L = lib(openmp)
    fn = L.oracle_layer_step_f32g if _is_f32(grads) else L.oracle_layer_step
    c = fn(n, len(grads), tab, _ptr(theta), _ptr(m), _ptr(v), wp, C.byref(hp), t)
    if c < 0:
        raise MemoryError("oracle_layer_step: allocation failed")
    return c


def layer_step_f64(grads, theta, m, v, hp: Hparams, t: int) -> float:
    tab, n = _replica_table(grads)
    for a in (theta, m, v):
        _as(a, np.float64)
        if a.size != n:
            raise ValueError("length mismatch")
    fn = lib().oracle_layer_step_f64_f32g if _is_f32(grads) else lib().oracle_layer_step_f64
    c = fn(n, len(grads), tab, _ptr(theta), _ptr(m), _ptr(v), C.byref(hp), t)
    if c < 0:
        raise MemoryError("oracle_layer_step_f64: allocation failed")
    return c
