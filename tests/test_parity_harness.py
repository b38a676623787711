"""The harness that runs the oracle over whole full-size layers (no GPU):
running the oracle's functions on disjoint slices in threads must give the
same bits as the oracle's own whole-layer step, with and without the clip,
and the chunked comparisons must report what the one-shot ones report."""
import numpy as np
import pytest

import oracle
import synth
import parity_util as pu


@pytest.mark.parametrize("n,R,clip,fp32", [(1_000_003, 4, 1.0, False), (300_001, 3, 1e-3, False),
                                           (262_144 + 17, 8, 0.0, False), (200_003, 4, 1.0, True)])
def test_threaded_oracle_step_equals_oracle_layer_step(n, R, clip, fp32):
    sp = synth.spec(3)
    hp = oracle.hparams(lr=1e-3, max_grad_norm=clip)
    mk = synth.grad_f32 if fp32 else synth.grad
    a = [synth.master(n, 3), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    b = [x.copy() for x in a]
    for t in (1, 2, 3):
        reps = [mk(n, sp, 0, t, r, 1e-3) for r in range(R)]
        c1 = oracle.layer_step(reps, *a, hp, t)
        c2 = pu.oracle_step_threaded(reps, *b, hp, t)
        assert np.float32(c1) == np.float32(c2)
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_threaded_master_equals_one_call():
    n = 3_000_017
    assert np.array_equal(pu.master_threaded(n, 9, unit=2).view(np.uint32),
                          synth.master(n, 9, unit=2).view(np.uint32))


def test_chunked_compare_equals_one_shot():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100_003).astype(np.float32)
    y = x.copy()
    y[::97] = np.nextafter(y[::97], np.float32(np.inf))
    y[5] += 1.0
    one = pu.compare_fp32("x", x, y)
    many = pu.compare_fp32_all("x", x, y, chunk=4096)
    assert one == many
    wx = oracle.f32_to_bf16(x)
    wy = oracle.f32_to_bf16(y)
    assert pu.compare_bf16("w", wx, wy) == pu.compare_bf16_all("w", wx, wy, chunk=1000)
