"""The seeded input generator (host side; its device twin is compared bit for
bit in the GPU tests).  Philox4x32-10 is pinned to the published known-answer
vectors of Salmon et al. (SC'11, the Random123 distribution); the shaped
outputs are checked for the distributions the workloads name."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def test_philox_known_answers():
    kat = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, want in kat:
        assert synth.philox(ctr, key) == want


def test_normals_are_standard_normal():
    scipy_stats = pytest.importorskip("scipy.stats")
    z = synth.normals(2_000_000, seed=3, tag=synth.TAG_GRAD).astype(np.float64)
    assert abs(z.mean()) < 3e-3
    assert abs(z.std() - 1) < 3e-3
    assert abs((z ** 3).mean()) < 1e-2
    assert abs((z ** 4).mean() - 3) < 3e-2
    assert scipy_stats.kstest(z[:300_000], "norm").pvalue > 1e-3


def test_own_log_and_sincos_close_to_libm():
    """Box-Muller's log and sin/cos are this generator's own (bit-identical on
    host and GPU); the normals they give must still be close to the ones the
    true functions give for the same Philox words (computed here in double)."""
    n = 4096
    zs = synth.normals(4 * n, seed=11, tag=7, a=1, b=2, c=3).astype(np.float64)
    ref = []
    for j in range(n):
        w = synth.philox([j, 1, 2, 3], [11, 7])
        for a, b in ((w[0], w[1]), (w[2], w[3])):
            u1 = ((a >> 8) + 1) * 2.0 ** -24
            u2 = ((b >> 8) + 1) * 2.0 ** -24
            r = np.sqrt(-2 * np.log(u1))
            ref += [r * np.cos(2 * np.pi * u2), r * np.sin(2 * np.pi * u2)]
    assert np.max(np.abs(zs - np.array(ref))) < 1.2e-5


def test_fill_and_gather_agree_with_offsets():
    sp = synth.spec(9)
    full = synth.grad(10_000, sp, unit=2, step=3, replica=1, scale=1e-3)
    part = synth.grad(3_000, sp, unit=2, step=3, replica=1, scale=1e-3, offset=4_001)
    assert np.array_equal(full[4_001:7_001], part)
    idx = np.array([0, 1, 4_000, 9_999, 5_555])
    assert np.array_equal(synth.gather_grad(idx, sp, 2, 3, 1, 1e-3), full[idx])
    m = synth.master(5_000, seed=4, unit=1)
    assert np.array_equal(synth.gather_master(idx[idx < 5000], 4, 1), m[idx[idx < 5000]])
    # different replica / step / unit streams differ
    assert not np.array_equal(full, synth.grad(10_000, sp, unit=2, step=3, replica=0, scale=1e-3))
    assert not np.array_equal(full, synth.grad(10_000, sp, unit=2, step=4, replica=1, scale=1e-3))


def test_student_t3_with_exact_zeros():
    sp = synth.spec(4, synth.GRAD_STUDENT3, 0.001)
    g = synth.grad(2_000_000, sp, unit=0, step=1, replica=0, scale=1e-3)
    x = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64) / 1e-3
    zero_frac = np.mean(g == 0)
    assert 0.0008 < zero_frac < 0.0012
    nz = x[g != 0]
    # Student-t with 3 degrees of freedom: median |t| = 0.7649, P(|t| > 3) = 0.0577
    assert abs(np.median(np.abs(nz)) - 0.7649) < 0.01
    assert abs(np.mean(np.abs(nz) > 3) - 0.0577) < 0.002


def test_workload_sizes():
    assert W.h2560_r1().numel == 100_930_560
    assert W.h5120_r8_logscale().numel == 330_311_680
    assert W.h5120x40_streamed().numel == 14_769_602_560
    assert W.h8192x8_streamed().numel == 7_021_395_968
    s = W.h5120_r8_logscale().tensor_scales(0)
    assert len(s) == 9 and all(1e-5 <= x <= 1e-2 for x in s) and len(set(s)) == 9
