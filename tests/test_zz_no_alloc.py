"""The entry point for callers that cannot allocate GPU memory.

slide_adamw_step_noalloc serves code that may not call cudaMalloc: an
allocator hook or memory-pressure handler that must not re-enter the CUDA
allocator it belongs to, a process whose GPU memory is a pool owned and capped
by a framework, a runtime that forbids allocation after start-up.  The caller
owns every array, and the clip's scratch is one fixed array inside the
library.

Here it is called through the C ABI, two calls in a row (the second reuses the
scratch the first left behind), and compared on the same seeded inputs with
  - the oracle, within the tolerance of the other GPU tests (2e-6*(1+|x|) on
    the FP32 master, m and v; 1 BF16 ulp on the copy), bit for bit where the
    clip is off;
  - the allocating entry point, slide_layer_step, bit for bit (same kernels).
After its one-time set-up on the device, further calls must leave the
device's free memory unchanged, whatever R and clip setting they use.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
import parity_util as pu  # noqa: E402


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


@pytest.mark.parametrize("n,R,clip", [((1 << 20) + 5, 4, 1.0), (70001, 3, 1e-3), (4099, 1, 0.0),
                                      (300_007, 8, 0.0)])
def test_noalloc_matches_oracle_and_slide_layer_step(S, n, R, clip):
    seed, lr, scale = 31, 1e-3, 1e-3
    sp = synth.spec(seed)
    hp = S.hparams(lr=lr, max_grad_norm=clip)
    hp_or = oracle.hparams(lr=lr, max_grad_norm=clip)
    grads = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
    th0 = synth.master(n, seed)

    # caller-owned arrays for the no-alloc entry point
    th = torch.from_numpy(th0.copy()).cuda()
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    w = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    # the oracle's state
    o_th, o_m, o_v = th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    o_w = np.zeros(n, np.uint16)

    st = S.slide_state_create([n], R)
    try:
        S.slide_layer_set(st, 0, master=th0, step=0)
        for t in (1, 2):
            for r in range(R):
                synth.dev_grad(grads[r].data_ptr(), n, sp, 0, t, r, scale)
            free0 = free_bytes()
            S.slide_adamw_step_noalloc(n, grads, th, m, v, w, hp, t)
            free1 = free_bytes()
            if t == 2:    # the device's set-up is behind us: nothing may be allocated
                assert free1 == free0, (free0, free1)
            S.slide_layer_step(st, 0, grads, hp)
            oracle.layer_step([synth.grad(n, sp, 0, t, r, scale) for r in range(R)],
                              o_th, o_m, o_v, o_w, hp_or, t)
            a, b, c = (np.empty(n, np.float32) for _ in range(3))
            wb = np.empty(n, np.uint16)
            assert S.slide_layer_get(st, 0, a, b, c, wb) == t
            got = [th.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy(), w[:n].cpu().numpy().view(np.uint16)]
            # against the oracle
            rep = [pu.compare_fp32(f"theta t{t}", got[0], o_th), pu.compare_fp32(f"m t{t}", got[1], o_m),
                   pu.compare_fp32(f"v t{t}", got[2], o_v), pu.compare_bf16(f"w t{t}", got[3], o_w)]
            pu.assert_parity(rep)
            if clip == 0.0:
                assert all(r["not_bit_equal"] == 0 for r in rep), rep
            # against the allocating entry point
            rep = [pu.compare_fp32("theta", got[0], a), pu.compare_fp32("m", got[1], b),
                   pu.compare_fp32("v", got[2], c), pu.compare_bf16("w", got[3], wb)]
            pu.assert_parity(rep)
            assert all(r["not_bit_equal"] == 0 for r in rep), rep
        assert S.slide_noalloc_status() == S.SLIDE_OK
    finally:
        S.slide_state_destroy(st)


def test_noalloc_allocates_nothing_after_setup(S):
    """One call sets the device up; calls with every replica count and the
    clip on and off then leave the free device memory unchanged."""
    n = 65_543
    sp = synth.spec(5)
    grads = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(8)]
    for r in range(8):
        synth.dev_grad(grads[r].data_ptr(), n, sp, 0, 1, r, 1e-3)
    th = torch.from_numpy(synth.master(n, 5)).cuda()
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    w = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    S.slide_adamw_step_noalloc(n, grads[:2], th, m, v, w, S.hparams(max_grad_norm=1.0), 1)
    assert S.slide_noalloc_status() == S.SLIDE_OK
    free0 = free_bytes()
    t = 2
    for R in range(1, 9):
        for clip in (0.0, 1.0):
            S.slide_adamw_step_noalloc(n, grads[:R], th, m, v, w, S.hparams(max_grad_norm=clip), t)
            t += 1
    assert free_bytes() == free0
    assert S.slide_noalloc_status() == S.SLIDE_OK
    assert np.isfinite(th.cpu().numpy()).all()


def test_noalloc_status_reports_a_wait_that_ran_out(S, monkeypatch):
    """A bounded wait inside the update kernel that runs out is reported once
    by slide_noalloc_status, which clears it; the next call is correct again.
    The wait is made to run out on purpose (test-only switch: the kernel's copy
    producer issues nothing), with no fault and no unbounded wait."""
    n, R, seed = 70_001, 2, 13
    sp = synth.spec(seed)
    grads = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
    for r in range(R):
        synth.dev_grad(grads[r].data_ptr(), n, sp, 0, 1, r, 1e-3)
    th = torch.from_numpy(synth.master(n, seed)).cuda()
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    w = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    hp = S.hparams(max_grad_norm=1.0)
    assert S.slide_noalloc_status() == S.SLIDE_OK
    monkeypatch.setenv("SLIDE_TEST_PIPELINE_STALL", "1")
    S.slide_adamw_step_noalloc(n, grads, th, m, v, w, hp, 1)
    monkeypatch.delenv("SLIDE_TEST_PIPELINE_STALL")
    assert S.slide_noalloc_status() == S.SLIDE_ERR_TIMEOUT
    assert S.slide_noalloc_status() == S.SLIDE_OK      # read and cleared
    # the caller restores its arrays and steps again: as the oracle
    th.copy_(torch.from_numpy(synth.master(n, seed)))
    m.zero_()
    v.zero_()
    S.slide_adamw_step_noalloc(n, grads, th, m, v, w, hp, 1)
    assert S.slide_noalloc_status() == S.SLIDE_OK
    o_th, o_m, o_v = synth.master(n, seed), np.zeros(n, np.float32), np.zeros(n, np.float32)
    o_w = np.zeros(n, np.uint16)
    oracle.layer_step([synth.grad(n, sp, 0, 1, r, 1e-3) for r in range(R)], o_th, o_m, o_v, o_w,
                      oracle.hparams(max_grad_norm=1.0), 1)
    pu.assert_parity([pu.compare_fp32("theta", th.cpu().numpy(), o_th), pu.compare_fp32("m", m.cpu().numpy(), o_m),
                      pu.compare_fp32("v", v.cpu().numpy(), o_v),
                      pu.compare_bf16("w", w[:n].cpu().numpy().view(np.uint16), o_w)])


def test_noalloc_rejects_out_of_range(S):
    g = [torch.zeros(64, dtype=torch.int16, device="cuda")]
    x = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(S.SlideError) as e:
        S.slide_adamw_step_noalloc((1 << 40) + 1, g, x, x, x, g[0], S.hparams(), 1)
    assert e.value.status == S.SLIDE_ERR_INVALID_ARG
    with pytest.raises(S.SlideError) as e:
        S.slide_adamw_step_noalloc(16, g * 9, x, x, x, g[0], S.hparams(), 1)
    assert e.value.status == S.SLIDE_ERR_INVALID_ARG
    with pytest.raises(S.SlideError) as e:
        S.slide_adamw_step_noalloc(16, g, x, x, x, g[0], S.hparams(), 0)
    assert e.value.status == S.SLIDE_ERR_INVALID_ARG
