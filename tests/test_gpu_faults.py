"""Failure paths made on the host or by a bounded wait that runs out, never by
a GPU fault, trap or hang:

- the update kernel's copy pipeline: with SLIDE_FLAG_TEST_PIPELINE_STALL the
  producer issues no copy, so every consumer's bounded wait (2 s) runs out;
  the kernel records that in the layer's status word and returns; the host
  reads SLIDE_ERR_TIMEOUT and the context stays usable;
- a pinned host allocation that fails (injected with SLIDE_FAULT_PINNED_ALLOC)
  returns SLIDE_ERR_OOM_HOST and leaves nothing allocated.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    return S


def test_pipeline_wait_limit_reports_timeout(S):
    n, R = 3 * 2048 + 77, 2
    st = S.slide_state_create([n], R, flags=S.SLIDE_FLAG_TEST_PIPELINE_STALL)
    try:
        g = [torch.zeros(n + 64, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        S.slide_layer_step(st, 0, g, S.hparams())
        assert S.slide_layer_status(st, 0) == S.SLIDE_ERR_TIMEOUT
        assert "limit" in S.slide_last_error()
        assert S.slide_layer_status(st, 0) == S.SLIDE_OK       # the mark was cleared
    finally:
        S.slide_state_destroy(st)
    # the context is intact: a normal state steps and reads back
    st = S.slide_state_create([n], R)
    try:
        g = [torch.zeros(n + 64, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        th = np.full(n, 0.25, np.float32)
        S.slide_layer_set(st, 0, master=th, step=0)
        S.slide_layer_step(st, 0, g, S.hparams(weight_decay=0.0))
        out = np.empty(n, np.float32)
        assert S.slide_layer_get(st, 0, out) == 1
        assert np.all(out == np.float32(0.25))                   # g = 0, wd = 0: unchanged
        assert S.slide_layer_status(st, 0) == S.SLIDE_OK
    finally:
        S.slide_state_destroy(st)


def test_pinned_allocation_failure_frees_everything(S):
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    os.environ["SLIDE_FAULT_PINNED_ALLOC"] = "1"
    try:
        with pytest.raises(S.SlideError) as e:
            S.slide_state_create([1 << 20, 1 << 20], 2, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
        assert e.value.status == S.SLIDE_ERR_OOM_HOST
    finally:
        del os.environ["SLIDE_FAULT_PINNED_ALLOC"]
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (8 << 20)
    st = S.slide_state_create([1 << 20, 1 << 20], 2, residency=S.SLIDE_RESIDENCY_HOST_STREAMED)
    S.slide_state_destroy(st)
