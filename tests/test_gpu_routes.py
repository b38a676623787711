"""The CPU-reduce route (every replica copied to the host and averaged there)
against the oracle, and against the GPU route (replicas averaged inside the
update kernel).  "SlideDP: Scaling Host-Resident LLM Fine-Tuning Across
Multiple GPUs", Prerequisites and Core method: both routes compute the same
update from the same aggregated gradient; the CPU route moves every rank's
gradient (R x 2n bytes of BF16) over the host link, the GPU route none.

Gate: |x - oracle| <= 2e-6*(1+|oracle|) on FP32 master, m, v and <= 1 BF16 ulp
on the copy; the two routes must also agree bit for bit with each other.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
import parity_util as pu  # noqa: E402
import reduce_routes  # noqa: E402


@pytest.mark.parametrize("n,R,clip", [(1_000_003, 4, 1.0), (4099, 3, 1e-3), (77, 8, 0.0)])
def test_cpu_reduce_route_matches_oracle(n, R, clip):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixed_precision_adam_grad_gb300 as S
    seed, scale = 1, 1e-3
    hp = S.hparams(max_grad_norm=clip)
    out = reduce_routes.measure_cpu_reduce_route(S, torch, synth, n, R, seed=seed, hp=hp, scale=scale,
                                                 return_states=True)
    # the CPU route moved every replica device -> host and one FP32 mean back
    assert out["cpu_route"]["d2h_bytes"] == R * 2 * n
    assert out["cpu_route"]["h2d_bytes"] == 4 * n
    assert out["gpu_route"]["link_bytes"] == 0
    assert out["identical_results"], "the two routes disagree"

    # the oracle on the same replicas (generated on the host), one step from the same master
    sp = synth.spec(seed)
    reps = [synth.grad(n, sp, 0, 1, r, scale) for r in range(R)]
    th = synth.master(n, seed)
    m, v, w = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)
    oracle.layer_step(reps, th, m, v, w, oracle.hparams(max_grad_norm=clip), 1)
    got = out["states"]["cpu"]
    rep = [pu.compare_fp32("theta", got[0], th), pu.compare_fp32("m", got[1], m),
           pu.compare_fp32("v", got[2], v), pu.compare_bf16("w", got[3], w)]
    pu.assert_parity(rep)
    if clip == 0.0:   # same FP32 operations on both sides without the clip
        assert all(r["not_bit_equal"] == 0 for r in rep), rep
