"""The CPU-reduce route (every replica copied to the host and averaged there)
and the GPU route (replicas averaged inside the update kernel) give the same
update bit for bit ("SlideDP: Scaling Host-Resident LLM Fine-Tuning Across
Multiple GPUs", Prerequisites and Core method: both routes leave the
semantics unchanged; the GPU route saves the R x gradient copies)."""
import os
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.mark.parametrize("n,R", [(1_000_003, 4), (4099, 3), (77, 8)])
def test_cpu_and_gpu_reduce_routes_agree(n, R):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    import mixed_precision_adam_grad_gb300 as S
    import synth
    out = bench.measure_cpu_reduce_route(S, torch, synth, n, R)
    assert out["identical_results"], out
    assert out["cpu_route"]["link_bytes"] == R * 2 * n + 4 * n
