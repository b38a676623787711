"""A layer longer than 2^31 elements: every index of the fused kernel, the clip
pre-pass and the generator must be 64-bit.

One layer of 2^31 + 2^20 + 13 parameters (ragged against the 2048-parameter
tiles and the 8-wide vectors), R = 2 BF16 replicas: about 40 GB of HBM.

  step 1, clip off: sampled elements (random, both ends, and a window around
          element 2^31) against the oracle, which computes them one by one;
  step 2, clip on:  the threshold is set to half the layer's gradient norm,
          which torch computes in float64 over the same device gradients
          (a library routine, independent of the kernels); the kernel's
          coefficient must match min(1, c / (norm + 1e-6)) within 2 FP32 ulp,
          and the sampled elements are replayed by the oracle with that
          coefficient.

Gate as elsewhere: |gpu - oracle| <= 2e-6*(1+|oracle|) on the FP32 master,
m and v, <= 1 BF16 ulp on the copy; step 1 must also be bit-equal.
"""
import math
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from synth import workloads as W  # noqa: E402
import parity_util as pu  # noqa: E402

N = (1 << 31) + (1 << 20) + 13
R = 2


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


class _DevArray:
    """A raw device pointer seen by torch (no copy, no ownership)."""

    def __init__(self, ptr, n, typestr):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 2}


def _gather(ptr, n, typestr, idx_dev):
    t = torch.as_tensor(_DevArray(ptr, n, typestr), device="cuda")
    return t[idx_dev].cpu().numpy()


def _device_sqnorm_of_mean(grads, n, chunk=1 << 28):
    """sum_i mean_i^2 in float64, mean_i = (g0_i + g1_i) * 0.5 in FP32 (exact:
    the sum of two BF16 values rounded once, then halved)."""
    acc = torch.zeros((), dtype=torch.float64, device="cuda")
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        g = grads[0][a:b].view(torch.bfloat16).float() + grads[1][a:b].view(torch.bfloat16).float()
        g = g * 0.5
        acc += (g.double() ** 2).sum()
    return float(acc.item())


def _compare(S, st, idx, idx_dev, th_s, m_s, v_s, w_s, t, bit_equal):
    pt, pm, pv, pw = S.slide_layer_ptrs(st, 0)
    th = _gather(pt, N, "<f4", idx_dev)
    m = _gather(pm, N, "<f4", idx_dev)
    v = _gather(pv, N, "<f4", idx_dev)
    wb = _gather(pw, N, "<i2", idx_dev).view(np.uint16)
    rep = [pu.compare_fp32(f"theta t{t}", th, th_s), pu.compare_fp32(f"m t{t}", m, m_s),
           pu.compare_fp32(f"v t{t}", v, v_s), pu.compare_bf16(f"w t{t}", wb, w_s)]
    pu.assert_parity(rep)
    assert np.array_equal(wb, oracle.f32_to_bf16(th))
    if bit_equal:
        assert all(r["not_bit_equal"] == 0 for r in rep), rep
    return rep


def test_layer_longer_than_2_pow_31(S):
    torch.cuda.empty_cache()  # blocks cached by earlier tests in this process
    free, _ = torch.cuda.mem_get_info()
    need = 14 * N + 2 * R * (N + 64) + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB of free device memory, {free / 2**30:.0f} GiB free")
    w = W.Workload("max_size", [W.Unit("flat", [("flat", N)])], R=R, steps=2, seed=21, lr=1e-3)
    boundary = np.arange((1 << 31) - 2048, (1 << 31) + 2048, dtype=np.int64)
    idx = pu.sample_indices(N, 40_000, seed=77, extra=boundary)
    assert idx[-1] == N - 1 and (idx == (1 << 31)).any()
    idx_dev = torch.from_numpy(idx).cuda()

    st = S.slide_state_create([N], R)
    grads = None
    try:
        synth.dev_master(S.slide_layer_ptrs(st, 0)[0], N, w.seed)
        grads = [torch.empty(N + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
        th_s = synth.gather_master(idx, w.seed)
        m_s, v_s = np.zeros(idx.size, np.float32), np.zeros(idx.size, np.float32)

        # step 1: clip off
        for r in range(R):
            pu.unit_grad_dev(w, 0, 1, r, grads[r].data_ptr())
        S.slide_layer_step(st, 0, grads, S.hparams(*w.hparams_tuple()))
        w_s = pu.oracle_sampled(w, 0, idx, 1, 1, th_s, m_s, v_s)
        _compare(S, st, idx, idx_dev, th_s, m_s, v_s, w_s, 1, bit_equal=True)

        # step 2: clip on, threshold at half the norm of the mean gradient
        for r in range(R):
            pu.unit_grad_dev(w, 0, 2, r, grads[r].data_ptr())
        torch.cuda.synchronize()
        sq = _device_sqnorm_of_mean(grads, N)
        c = float(np.float32(0.5 * math.sqrt(sq)))
        w2 = replace(w, max_grad_norm=c)
        coef = oracle.clip_coef(sq, c)
        assert 0.4 < coef < 0.6
        S.slide_layer_step(st, 0, grads, S.hparams(*w2.hparams_tuple()))
        gc = S.slide_layer_last_clip_coef(st, 0)
        assert abs(gc - coef) <= 2 * np.spacing(np.float32(coef)), (gc, coef)
        w_s = pu.oracle_sampled(w2, 0, idx, 2, 2, th_s, m_s, v_s, coefs={2: coef})
        _compare(S, st, idx, idx_dev, th_s, m_s, v_s, w_s, 2, bit_equal=False)
        assert S.slide_layer_get(st, 0) == 2
    finally:
        del grads
        S.slide_state_destroy(st)
        torch.cuda.empty_cache()
