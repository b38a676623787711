"""Helpers shared by the GPU parity tests, the smoke check and the benchmark's
oracle legs: drive the CUDA path through the C ABI on seeded synthetic inputs,
drive the oracle on the same inputs (generated on the host, bit-identical),
and compare with the tolerance the workloads fix:

  FP32 master, m, v:  max |gpu - oracle| <= 2e-6 * (1 + |oracle|)
  BF16 compute copy:  at most 1 BF16 ulp apart (bit patterns differ by <= 1)

and, sharper than that gate, report how many FP32 values are not bit-equal.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL_REL = 2e-6


def hp_oracle(w):
    return oracle.hparams(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, w.max_grad_norm)


def compare_fp32(name, got, want, tol=TOL_REL):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    diff = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bound = tol * (1.0 + np.abs(want.astype(np.float64)))
    bad = ~(diff <= bound)
    info = {
        "name": name,
        "n": int(got.size),
        "max_abs": float(diff.max()) if diff.size else 0.0,
        "not_bit_equal": int(np.count_nonzero(got.view(np.uint32) != want.view(np.uint32))),
        "violations": int(np.count_nonzero(bad)),
    }
    return info


def compare_bf16(name, got, want):
    a = np.asarray(got, np.uint16).astype(np.int32)
    b = np.asarray(want, np.uint16).astype(np.int32)
    # distance in units in the last place on the BF16 lattice (same sign)
    ia = np.where(a & 0x8000, -(a & 0x7FFF), a)
    ib = np.where(b & 0x8000, -(b & 0x7FFF), b)
    d = np.abs(ia - ib)
    return {"name": name, "n": int(a.size), "max_ulp": int(d.max()) if d.size else 0,
            "not_bit_equal": int(np.count_nonzero(a != b)), "violations": int(np.count_nonzero(d > 1))}


def assert_parity(reports):
    for r in reports:
        assert r["violations"] == 0, r


def unit_grad_host(w, unit_index, step, replica, idx=None):
    """BF16 gradient replica of a unit at `step` on the host (whole unit or the
    given sorted element indices)."""
    u = w.units[unit_index]
    sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
    scales = w.tensor_scales(unit_index)
    dt = np.float32 if w.fp32_grads else np.uint16
    fill = synth.grad_f32 if w.fp32_grads else synth.grad
    gather = synth.gather_grad_f32 if w.fp32_grads else synth.gather_grad
    if idx is None:
        out = np.empty(u.numel, dt)
        for (off, n), sc in zip(u.segments(), scales):
            out[off:off + n] = fill(n, sp, unit_index, step, replica, sc, offset=off)
        return out
    idx = np.asarray(idx, np.int64)
    out = np.empty(idx.size, dt)
    bounds = np.cumsum([0] + [n for _, n in u.tensors])
    for k, sc in enumerate(scales):
        sel = (idx >= bounds[k]) & (idx < bounds[k + 1])
        if sel.any():
            out[sel] = gather(idx[sel], sp, unit_index, step, replica, sc)
    return out


def unit_grad_dev(w, unit_index, step, replica, ptr, stream=0):
    u = w.units[unit_index]
    sp = synth.spec(w.seed, w.grad_kind, w.zero_prob)
    size = 4 if w.fp32_grads else 2
    fill = synth.dev_grad_f32 if w.fp32_grads else synth.dev_grad
    for (off, n), sc in zip(u.segments(), w.tensor_scales(unit_index)):
        fill(ptr + size * off, n, sp, unit_index, step, replica, sc, offset=off, stream=stream)


def sample_indices(n, k, seed=1234, extra=()):
    """Sorted unique sample: k random indices, the first and last 4096, extras."""
    rng = np.random.default_rng(seed)
    parts = [rng.integers(0, n, size=min(k, n)), np.arange(min(4096, n)),
             np.arange(max(0, n - 4096), n)]
    if len(extra):
        e = np.asarray(extra, np.int64)
        parts.append(e[(e >= 0) & (e < n)])
    return np.unique(np.concatenate(parts).astype(np.int64))


def oracle_full_coefs(w, unit_index, steps):
    """Clip coefficient of each step (by the oracle over the whole unit)."""
    hp = hp_oracle(w)
    coefs = {}
    for t in steps:
        reps = [unit_grad_host(w, unit_index, t, r) for r in range(w.R)]
        gm = oracle.grad_mean(reps)
        coefs[t] = oracle.clip_coef(oracle.grad_sqnorm(gm), hp.max_grad_norm)
        del reps, gm
    return coefs


def oracle_sampled(w, unit_index, idx, first_step, last_step, theta, m, v, coefs=None):
    """Run the oracle on the sampled elements (in place) for steps
    first_step..last_step.  With the clip on, coefs[t] must hold the oracle's
    whole-unit coefficient of step t.  Returns the BF16 copy."""
    hp = hp_oracle(w)
    wbf = np.zeros(idx.size, np.uint16)
    for t in range(first_step, last_step + 1):
        reps = [unit_grad_host(w, unit_index, t, r, idx) for r in range(w.R)]
        gm = oracle.grad_mean(reps)
        coef = coefs[t] if (w.max_grad_norm > 0) else 1.0
        oracle.adamw_update(gm, coef, theta, m, v, wbf, hp, t)
    return wbf


# ---------------------------------------------------- whole-layer runs ----
# The oracle's functions are single-threaded.  For layers of hundreds of
# millions of parameters the tests run them on disjoint slices in threads (the
# ctypes calls release the GIL): every element still goes through exactly the
# oracle's operations, and the one cross-element quantity, the clip norm, is
# the oracle's own sum over the whole mean gradient in index order.

import os  # noqa: E402
from concurrent.futures import ThreadPoolExecutor  # noqa: E402


def _workers():
    return max(1, min(32, os.cpu_count() or 1))


def slices(n, parts):
    """Disjoint [a, b) ranges covering [0, n), 64-element aligned starts."""
    if n <= 0:
        return []
    step = max(1 << 16, -(-n // max(1, parts)))
    step = (step + 63) // 64 * 64
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def oracle_step_threaded(reps, theta, m, v, w, hp, t):
    """One oracle layer step over the whole layer, in place (the same result
    as oracle.layer_step): mean of the replicas, clip coefficient over the
    whole mean, AdamW update with the BF16 copy.  Returns the coefficient."""
    n = theta.size
    nw = _workers()
    gm = np.empty(n, np.float32)
    sl = slices(n, 4 * nw)

    def mean(ab):
        a, b = ab
        gm[a:b] = oracle.grad_mean([g[a:b] for g in reps])

    def update(ab, coef):
        a, b = ab
        oracle.adamw_update(gm[a:b], coef, theta[a:b], m[a:b], v[a:b], None if w is None else w[a:b], hp, t)

    with ThreadPoolExecutor(nw) as ex:
        list(ex.map(mean, sl))
        coef = 1.0
        if hp.max_grad_norm > 0:
            coef = oracle.clip_coef(oracle.grad_sqnorm(gm), hp.max_grad_norm)
        list(ex.map(lambda ab: update(ab, coef), sl))
    return coef


def master_threaded(n, seed, unit=0):
    """The seeded initial master of a whole unit, generated on the host."""
    out = np.empty(n, np.float32)

    def fill(ab):
        a, b = ab
        out[a:b] = synth.master(b - a, seed, unit=unit, offset=a)

    with ThreadPoolExecutor(_workers()) as ex:
        list(ex.map(fill, slices(n, 4 * _workers())))
    return out


def replicas_to_host(w, unit_index, step, dev_bufs, n, check=4096, seed=0):
    """Host copies of the R replicas that the seeded generator wrote into the
    device buffers `dev_bufs` (torch tensors) for (unit, step); a random
    sample of each is checked against the host generator first, so the
    oracle's inputs are the generator's values whichever twin produced them."""
    import torch
    torch.cuda.synchronize()
    out = []
    rng = np.random.default_rng(seed + 7919 * step + unit_index)
    idx = np.unique(np.concatenate([rng.integers(0, n, size=min(check, n)), [0, n - 1]])).astype(np.int64)
    for r, buf in enumerate(dev_bufs):
        h = buf[:n].cpu().numpy()
        h = h.view(np.float32) if w.fp32_grads else h.view(np.uint16)
        want = unit_grad_host(w, unit_index, step, r, idx)
        assert np.array_equal(h[idx].view(np.uint8), want.view(np.uint8)), "device generator disagrees with host"
        out.append(h)
    return out


def _merge(reports):
    out = dict(reports[0])
    for r in reports[1:]:
        out["n"] += r["n"]
        out["not_bit_equal"] += r["not_bit_equal"]
        out["violations"] += r["violations"]
        for k in ("max_abs", "max_ulp"):
            if k in out:
                out[k] = max(out[k], r[k])
    return out


def compare_fp32_all(name, got, want, chunk=1 << 25):
    """compare_fp32 over every element, in chunks (bounded temporaries)."""
    n = got.size
    return _merge([compare_fp32(name, got[a:a + chunk], want[a:a + chunk]) for a in range(0, max(n, 1), chunk)])


def compare_bf16_all(name, got, want, chunk=1 << 25):
    n = got.size
    return _merge([compare_bf16(name, got[a:a + chunk], want[a:a + chunk]) for a in range(0, max(n, 1), chunk)])
