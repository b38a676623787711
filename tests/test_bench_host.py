"""Host logic of bench.py (no GPU): the max-over-ranks timing on a 2-rank gloo
process group, the clock-sample parsing, and the reference arm's rank rule."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank
    out[rank] = bench.max_over_ranks(ms, dist)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single():
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_clock_parse():
    lines = ["0, 1965, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n",
             "0, 2070, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
             "0, 2070, 2070, 951.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n",
             "garbage\n"]
    c = bench.ClockSampler.parse(lines)
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_minimum():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_unit_spread_and_overlap():
    """Per-step spread of the unit copy-in times and the busy/overlap summary
    of a streamed timeline, on a hand-made timeline with one slow unit."""
    nan = float("nan")
    units = []
    t = 10.0
    for i, dur in enumerate([30.0, 20.0, 20.0, 60.0, 20.0, 25.0]):
        units.append({"h2d_begin": t, "master_landed": t + 5, "h2d_end": t + dur, "update_end": t + dur,
                      "d2h_begin": t + 6, "d2h_end": t + dur + 4})
        t += dur
    sp = bench.unit_spread(units)
    assert sp["slowest_unit"] == 3
    assert sp["median_unit_copy_in_ms"] == 20.0
    assert sp["unit_max_over_median"] == 3.0
    assert bench.unit_spread(units[:2])["slowest_unit"] is None
    units[2] = {k: nan for k in units[2]}
    assert bench.unit_spread(units)["slowest_unit"] == 3
    ov = bench.timeline_overlap([u for u in units if u["h2d_begin"] == u["h2d_begin"]], 10.0)
    assert ov["step_ms"] == t + 4


def test_slice_unit_keeps_leading_tensors():
    from synth import workloads as W
    u = W.h5120_r8_logscale().units[0]
    full = u.numel
    s = bench.slice_unit(u, 100_000_000)
    assert s.numel == 100_000_000
    assert [t for t, _ in s.tensors] == [t for t, _ in u.tensors[:len(s.tensors)]]
    assert all(a == b for a, b in zip(s.tensors[:-1], u.tensors))
    assert bench.slice_unit(u, full + 5).numel == full


def test_streamed_leg_rejects_unknown_layout_suffix():
    class A:
        streamed_bf16_in_hbm = False
    with pytest.raises(ValueError):
        bench.run_streamed(A(), None, None, None, "h8192x8_streamed+bogus")
