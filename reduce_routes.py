"""Measurement of the two gradient-reduction routes that "SlideDP: Scaling
Host-Resident LLM Fine-Tuning Across Multiple GPUs" compares (Prerequisites
and Core method): the CPU-reduce route, where every rank's gradient of a layer
leaves the GPU and the host reduces them (R x the gradient bytes cross the
host link), against the GPU route, where the R gradients are reduced on the
GPU before anything leaves it.

This is measurement code beside bench.py, not part of the product package:
the product's only route is the GPU one (the replicas are averaged inside the
fused update kernel as it reads them).  Here the CPU route is modelled on one
GPU: the R replica buffers are copied to pinned host memory, averaged on the
host (FP32 sum in replica order, divided by R), and the mean goes back to the
GPU as a single FP32 replica for the same fused update.  Both routes must end
in the same state; the tests also hold the CPU route against the oracle.
"""
from __future__ import annotations

import time

import numpy as np


def host_replica_mean(reps_bf16):
    """Mean of R BF16 replicas (uint16 bit patterns) on the host: widen to
    FP32, sum in replica order in FP32, divide by R."""
    acc = (reps_bf16[0].astype(np.uint32) << 16).view(np.float32).copy()
    for g in reps_bf16[1:]:
        acc += (g.astype(np.uint32) << 16).view(np.float32)
    acc /= np.float32(len(reps_bf16))
    return acc


def measure_cpu_reduce_route(S, torch, synth, n, R, seed=1, hp=None, scale=1e-3, return_states=False,
                             host_alloc=None):
    """Run one optimizer step of an n-parameter layer by both routes from the
    same master (seeded, m = v = 0, t = 1) on the same R seeded BF16 replicas
    (synth.dev_grad with spec(seed), unit 0, step 1, replica r, `scale`).

    Returns timings, the host-link bytes each route moved (counted from the
    buffers actually copied) and whether the two final states are
    bit-identical; with return_states=True also both final states as host
    arrays (master, m, v, BF16 copy).  host_alloc(shape, dtype) supplies the
    pinned host buffers (default: torch's pinned allocator)."""
    hp = hp or S.hparams(max_grad_norm=1.0)
    sp = synth.spec(seed)
    reps = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
    for r in range(R):
        synth.dev_grad(reps[r].data_ptr(), n, sp, 0, 1, r, scale)
    th0 = synth.master(n, seed)
    gpu = S.slide_state_create([n], R)
    cpu = S.slide_state_create([n], 1, flags=S.SLIDE_FLAG_FP32_GRADS)
    alloc = host_alloc or (lambda shape, dtype: torch.empty(shape, dtype=dtype, pin_memory=True))
    host_reps = [alloc(n, torch.int16) for _ in range(R)]
    mean_host = alloc(n, torch.float32)
    mean_dev = torch.empty(n + 64, dtype=torch.float32, device="cuda")
    try:
        S.slide_layer_set(gpu, 0, master=th0, step=0)
        S.slide_layer_set(cpu, 0, master=th0, step=0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        S.slide_layer_step(gpu, 0, reps, hp)
        torch.cuda.synchronize()
        t_gpu = time.perf_counter() - t0

        t0 = time.perf_counter()
        d2h_bytes = 0
        for r in range(R):
            host_reps[r].copy_(reps[r][:n], non_blocking=True)
            d2h_bytes += host_reps[r].numel() * host_reps[r].element_size()
        torch.cuda.synchronize()
        t_d2h = time.perf_counter() - t0
        t0 = time.perf_counter()
        mean = host_replica_mean([h.numpy().view(np.uint16) for h in host_reps])
        t_reduce = time.perf_counter() - t0
        t0 = time.perf_counter()
        mean_host.numpy()[:] = mean
        mean_dev[:n].copy_(mean_host, non_blocking=True)
        h2d_bytes = mean_host.numel() * mean_host.element_size()
        S.slide_layer_step(cpu, 0, [mean_dev], hp)
        torch.cuda.synchronize()
        t_back = time.perf_counter() - t0

        a = [np.empty(n, np.float32) for _ in range(3)] + [np.empty(n, np.uint16)]
        b = [np.empty(n, np.float32) for _ in range(3)] + [np.empty(n, np.uint16)]
        S.slide_layer_get(gpu, 0, *a)
        S.slide_layer_get(cpu, 0, *b)
        same = all(np.array_equal(x.view(np.uint8), y.view(np.uint8)) for x, y in zip(a, b))
    finally:
        S.slide_state_destroy(gpu)
        S.slide_state_destroy(cpu)
    out = {"params": n, "replicas": R, "identical_results": bool(same),
           "gpu_route": {"s": t_gpu, "link_bytes": 0},
           "cpu_route": {"s": t_d2h + t_reduce + t_back, "d2h_s": t_d2h, "host_reduce_s": t_reduce,
                         "h2d_and_update_s": t_back, "d2h_bytes": d2h_bytes, "h2d_bytes": h2d_bytes,
                         "link_bytes": d2h_bytes + h2d_bytes,
                         "host_reduce": "numpy FP32 in replica order, one host thread"},
           "amplification_d2h_bytes": f"{R} x 2n (every replica) instead of none"}
    if return_states:
        out["states"] = {"gpu": a, "cpu": b}
    return out
