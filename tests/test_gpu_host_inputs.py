"""The step of a layer whose gradient replicas are in host memory
(slide_layer_step_host): the replicas are copied into the state's device
staging on its copy stream, the step runs behind the copy, and the new BF16
copy comes back to host memory.  Compared on every element with the oracle
(2e-6*(1+|x|) on master, m and v, 1 BF16 ulp on the copy; bit for bit without
the clip), with the inputs taken straight from the host generator.
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


@pytest.mark.parametrize("R,clip,fp32,pinned", [(3, 0.0, False, False), (4, 1.0, False, True),
                                                (2, 1e-3, True, True), (8, 0.0, False, True)])
def test_host_input_step_matches_oracle(S, R, clip, fp32, pinned):
    sizes = [70001, 4099, (1 << 20) + 5]
    seed, lr, steps = 17, 1e-3, 3
    sp = synth.spec(seed)
    mk = synth.grad_f32 if fp32 else synth.grad
    flags = S.SLIDE_FLAG_HOST_INPUTS | (S.SLIDE_FLAG_FP32_GRADS if fp32 else 0)
    hp = S.hparams(lr=lr, max_grad_norm=clip)
    hp_or = oracle.hparams(lr=lr, max_grad_norm=clip)
    st = S.slide_state_create(sizes, R, flags=flags)
    stream = torch.cuda.Stream()
    try:
        ref = []
        for li, n in enumerate(sizes):
            th0 = synth.master(n, seed, unit=li)
            S.slide_layer_set(st, li, master=th0, step=0)
            ref.append([th0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)])
        outs = {}
        keep = []
        # every step of every layer is enqueued before anything is synchronised,
        # so calls run with the copy-in of one overlapping the update of the last
        for t in range(1, steps + 1):
            for li, n in enumerate(sizes):
                reps = [mk(n, sp, li, t, r, 1e-3) for r in range(R)]
                if pinned:
                    reps = [torch.from_numpy(x if fp32 else x.view(np.int16)).pin_memory() for x in reps]
                    out = torch.empty(n, dtype=torch.int16, pin_memory=True)
                else:
                    out = np.empty(n, np.uint16)
                keep.append((reps, out))
                S.slide_layer_step_host(st, li, reps, hp, stream, out)
                outs[(li, t)] = out
        stream.synchronize()
        for t in range(1, steps + 1):
            for li, n in enumerate(sizes):
                host = [mk(n, sp, li, t, r, 1e-3) for r in range(R)]
                oracle.layer_step(host, *ref[li], hp_or, t)
                out = outs[(li, t)]
                got_w = out.numpy().view(np.uint16) if hasattr(out, "numpy") else out
                rep = pu.compare_bf16(f"w l{li} t{t}", got_w, ref[li][3])
                pu.assert_parity([rep])
        for li, n in enumerate(sizes):
            a, b, c = (np.empty(n, np.float32) for _ in range(3))
            assert S.slide_layer_get(st, li, a, b, c) == steps
            rep = [pu.compare_fp32("theta", a, ref[li][0]), pu.compare_fp32("m", b, ref[li][1]),
                   pu.compare_fp32("v", c, ref[li][2])]
            pu.assert_parity(rep)
            if clip == 0.0:
                assert all(r["not_bit_equal"] == 0 for r in rep), rep
    finally:
        S.slide_state_destroy(st)


def test_host_input_step_needs_the_flag(S):
    st = S.slide_state_create([100], 1)
    try:
        with pytest.raises(S.SlideError) as e:
            S.slide_layer_step_host(st, 0, [np.zeros(100, np.uint16)], S.hparams())
        assert e.value.status == S.SLIDE_ERR_STATE
    finally:
        S.slide_state_destroy(st)
