"""Delivery of the emitted BF16 copy to R consumer buffers (full delivery
versus sharded delivery plus an on-device all-gather, the two parameter routes
of "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across Multiple GPUs",
Core method), from HBM and from the pinned host mirror: every consumer ends
with the layer's BF16 copy, bit for bit, and nothing past n is touched."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


@pytest.mark.parametrize("residency", [0, 1])
@pytest.mark.parametrize("route", [0, 1])
@pytest.mark.parametrize("R", [1, 3, 8])
def test_delivery_routes_bit_exact(S, residency, route, R):
    sizes = [5, 1_000_003, 0]
    st = S.slide_state_create(sizes, 2, residency=residency)
    try:
        for li, n in enumerate(sizes):
            S.slide_layer_set(st, li, master=synth.master(n, 17, unit=li), step=0)
        for li, n in enumerate(sizes):
            want = np.empty(n, np.uint16)
            S.slide_layer_get(st, li, bf16=want)
            dst = [torch.full((n + 64,), 0x5A5A, dtype=torch.int16, device="cuda") for _ in range(R)]
            S.slide_deliver_bf16(st, li, dst, route=route)
            torch.cuda.synchronize()
            for d in dst:
                got = d.cpu().numpy().view(np.uint16)
                assert np.array_equal(got[:n], want)
                assert np.all(got[n:] == 0x5A5A)
    finally:
        S.slide_state_destroy(st)


def test_delivery_argument_errors(S):
    st = S.slide_state_create([100], 1)
    try:
        d = torch.zeros(128, dtype=torch.int16, device="cuda")
        for kw in (dict(dst=[d] * 9, route=0), dict(dst=[d], route=7), dict(dst=[d.data_ptr() + 2], route=0)):
            with pytest.raises(S.SlideError) as e:
                S.slide_deliver_bf16(st, 0, kw["dst"], route=kw["route"])
            assert e.value.status == S.SLIDE_ERR_INVALID_ARG
    finally:
        S.slide_state_destroy(st)
