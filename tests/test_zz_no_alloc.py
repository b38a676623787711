"""The entry point for callers that cannot allocate GPU memory.

slide_adamw_step_noalloc serves code that may not call cudaMalloc (an
allocator hook or host callback that must not re-enter the CUDA allocator, a
framework-owned and capped memory pool, a runtime that forbids allocation
after start-up): the caller owns every array and the clip's scratch is a
fixed array inside the library.  Here it is called through the C ABI and
compared with the allocating entry point, slide_layer_step, on the same
inputs, for two calls in a row (the second call reuses the scratch the first
one left behind), with the clip on, within the tolerance the other GPU tests
use (2e-6*(1+|x|) on FP32 master/m/v, 1 BF16 ulp on the copy); the two run
the same kernels, so the results must also be bit-identical.

This file is named to be collected last, so a run that stops at the first
failure has run every other test before it.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
import parity_util as pu  # noqa: E402


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


@pytest.mark.parametrize("n,R,clip", [((1 << 20) + 5, 4, 1.0), (70001, 3, 1e-3), (4099, 1, 0.0)])
def test_noalloc_matches_slide_layer_step(S, n, R, clip):
    seed = 31
    sp = synth.spec(seed)
    hp = S.hparams(lr=1e-3, max_grad_norm=clip)
    grads = [torch.empty(n + 64, dtype=torch.int16, device="cuda") for _ in range(R)]
    th0 = synth.master(n, seed)

    # caller-owned arrays for the no-alloc entry point
    th = torch.from_numpy(th0.copy()).cuda()
    m = torch.zeros(n, dtype=torch.float32, device="cuda")
    v = torch.zeros(n, dtype=torch.float32, device="cuda")
    w = torch.zeros(n + 8, dtype=torch.int16, device="cuda")

    st = S.slide_state_create([n], R)
    try:
        S.slide_layer_set(st, 0, master=th0, step=0)
        for t in (1, 2):
            for r in range(R):
                synth.dev_grad(grads[r].data_ptr(), n, sp, 0, t, r, 1e-3)
            S.slide_adamw_step_noalloc(n, grads, th, m, v, w, hp, t)
            S.slide_layer_step(st, 0, grads, hp)
            torch.cuda.synchronize()
            a, b, c = (np.empty(n, np.float32) for _ in range(3))
            wb = np.empty(n, np.uint16)
            assert S.slide_layer_get(st, 0, a, b, c, wb) == t
            got = [th.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy(), w[:n].cpu().numpy().view(np.uint16)]
            rep = [pu.compare_fp32("theta", got[0], a), pu.compare_fp32("m", got[1], b),
                   pu.compare_fp32("v", got[2], c), pu.compare_bf16("w", got[3], wb)]
            pu.assert_parity(rep)
            assert all(r["not_bit_equal"] == 0 for r in rep), rep
    finally:
        S.slide_state_destroy(st)


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
