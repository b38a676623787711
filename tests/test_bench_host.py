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
    assert sp["median_unit_copy_in_ms_per_gparam"] == 22.5e9
    assert sp["unit_max_over_median"] == 60.0 / 22.5
    # per parameter: unit 0 with twice the parameters is not slow
    sp = bench.unit_spread(units, sizes=[2, 1, 1, 1, 1, 1])
    assert sp["slowest_unit"] == 3 and sp["unit_max_over_median"] == 3.0
    assert bench.unit_spread(units[:1])["slowest_unit"] is None
    # the last unit of the sweep counts too
    assert bench.unit_spread(units[:3] + [dict(units[4], h2d_end=units[4]["h2d_begin"] + 200.0)])["slowest_unit"] == 3
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


def _full_record():
    """A record shaped like run_ours' (values made up, timelines long)."""
    n, R = 330_311_680, 8
    units = [{"h2d_begin": 1.0 * i, "master_landed": 1.0 * i + 0.2, "h2d_end": 1.0 * i + 0.9,
              "update_end": 1.0 * i + 1.0, "d2h_begin": 1.0 * i + 0.3, "d2h_end": 1.0 * i + 1.2} for i in range(42)]
    streamed = {"workload": "h8192x8_streamed", "description": "x" * 300, "params": 7_021_395_968, "replicas": 8,
                "steps": 5, "s_per_step": 0.66, "s_per_step_each": [0.66, 0.67, 0.65, 0.7, 0.66],
                "s_per_step_min": 0.65, "s_per_step_mean": 0.668, "gparam_s": 10.6, "roofline_s": 0.644,
                "frac": 0.97, "frac_fastest_step": 0.99,
                "per_step": [{"s": 0.66, "unit_max_over_median": 1.1, "slowest_unit": 3,
                              "median_unit_copy_in_ms": 80.0}] * 5,
                "link_bytes_per_step": {"h2d": 14 * 7_021_395_968, "d2h": 14 * 7_021_395_968},
                "bf16_copy_in_hbm": False, "achieved_link_gbs_each_way": 148.0,
                "link": {"h2d_gbs": 211.0, "d2h_gbs": 193.0, "h2d_concurrent_gbs": 171.0,
                         "d2h_concurrent_gbs": 170.0, "bidir_gbs": 340.0, "probe": "p"},
                "link_monitor_before": {"h2d": {"median_gbs": 168.0}}, "link_monitor_after": {},
                "host_pinned_gb": 98.3, "window_gb": 52.7, "create_s": 10.0, "chunk_mib": 64,
                "grad_callback": "g" * 200, "s_per_step_with_generator_callback": 1.23,
                "cpu_baseline": {"value": 0.05, "unit": "Gparam/s", "cores": 1, "kind": "oracle",
                                 "s_per_step_extrapolated": 140.0, "sample": "s" * 300},
                "timeline_fastest_step": {"units_ms": units}, "timeline_slowest_step": {"units_ms": units},
                "bf16_delivery": {"full": {"ms": 66.4}}, "timing": "t",
                "pipelined": {"s_per_step": 0.59, "roofline_s": 0.578, "frac": 0.98,
                              "s_per_step_each": [0.59] * 5, "s_per_step_incl_last_drain": 0.6}}
    hbm = {"workload": "h2560_R4_clip", "description": "d", "params": 100_930_560, "replicas": 4, "steps": 20,
           "value": 155.0, "unit": "Gparam/s", "ms_per_step": 0.65, "hbm_gbs": 6500.0,
           "roofline": {"bound": "hbm", "kernel": "grad_reduce_adamw_cast", "achieved": 6700.0, "peak": 6779.0,
                        "unit": "GB/s", "frac": 0.988, "traffic": None, "traffic_note": "n",
                        "bytes_per_launch": 34 * 100_930_560, "bytes_per_param": 34, "avg_launch_ms": 0.51,
                        "launches": 20},
           "prepass": {"achieved": 5900.0, "frac": 0.87, "avg_launch_ms": 0.137, "bytes_per_param": 8},
           "step_roofline_frac": 0.96}
    bytes_upd = 42 * n
    avg = 2.07
    ach = bytes_upd / (avg * 1e-3) / 1e9
    return {
        "metric": bench.METRIC, "value": 159.3, "unit": "Gparam/s", "n_gpus": 1, "steps": 20, "warmup": 5,
        "ms_per_step": 2.074, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "h5120_R8_logscale", "description": "one h=5120 decoder layer", "params": n,
                   "replicas": R, "max_grad_norm": 0.0, "parallelism": "replicas-only x1", "l2": "larger",
                   "clock_samples": "c"},
        "hbm_gbs": 6690.0,
        "roofline": {"bound": "hbm", "kernel": "grad_reduce_adamw_cast", "achieved": ach, "peak": 6779.0,
                     "unit": "GB/s", "frac": ach / 6779.0, "traffic": 13.6e9, "traffic_note": "ncu",
                     "peak_kind": "measured (MEASURED_PEAKS.json hbm_gbs)", "bytes_per_launch": bytes_upd,
                     "avg_launch_ms": avg, "bytes_per_param": 42, "launches": 20},
        "prepass": None, "step_roofline_frac": 0.98, "gpu_launches": 20,
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9},
        "e2e": {"value": 12.0, "unit": "Gparam/s", "h2d_bytes_per_step": 2 * R * n, "d2h_bytes_per_step": 2 * n,
                "steps": 20, "pipelining": "p" * 100},
        "cpu_baseline": {"value": 0.05, "unit": "Gparam/s", "cores": 1, "kind": "oracle", "gbs": 2.1,
                         "gbs_bytes_per_param": 42, "cpu_model": "Neoverse-V2", "sample": "s" * 400},
        "cpu_baseline_all_cores": {"value": 0.8, "unit": "Gparam/s", "cores": 16, "kind": "oracle_openmp",
                                   "gbs": 33.0, "gbs_bytes_per_param": 42, "cpu_model": "Neoverse-V2",
                                   "sample": "s"},
        "fp32_grad_variant": dict(hbm, workload="h2560_R4_clip_fp32grads"),
        "other_hbm_workloads": {"h2560_R1": dict(hbm, workload="h2560_R1", prepass=None),
                                "h2560_R4_clip": hbm},
        "cpu_reduce_route": {"params": n, "replicas": R, "identical_results": True,
                             "gpu_route": {"s": 0.002, "link_bytes": 0},
                             "cpu_route": {"s": 3.0, "d2h_bytes": 2 * R * n, "h2d_bytes": 4 * n,
                                           "link_bytes": 2 * R * n + 4 * n}},
        "chunk_sweep": {k: {"workload": k, "chosen": [64, 64],
                            "points": [{"h2d_mib": a, "d2h_mib": b, "frac": 0.9, "s_per_step": 0.7}
                                       for a in (32, 64, 128, 256) for b in (64, 256)]}
                        for k in ("h8192x8_streamed", "h5120x40_streamed")},
        "streamed": streamed,
        "streamed_also": {"h5120x40_streamed": dict(streamed, workload="h5120x40_streamed",
                                                    bf16_copy_in_hbm=True),
                          "h8192x8_streamed+bf16hbm": dict(streamed, bf16_copy_in_hbm=True),
                          "h8192x8_streamed+x": {"workload": "h8192x8_streamed", "skipped": "host memory " * 40}},
    }


def test_compact_headline_is_last_and_small(capsys, tmp_path):
    import json
    full = _full_record()
    out = tmp_path / "detail.json"
    bench.report(full, str(out))
    lines = capsys.readouterr().out.strip().splitlines()
    last = lines[-1]
    assert len(last.encode()) < 4096, len(last.encode())
    assert all(x.startswith("detail ") for x in lines[:-1])
    h = json.loads(last)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
              "gpu_launches"):
        assert k in h, k
    assert h["config"]["workload"] == "h5120_R8_logscale"
    rf = h["roofline"]
    # frac recomputes from the line's own fields (to the rounding of 4 digits)
    ach = rf["bytes_per_launch"] / (rf["avg_launch_ms"] * 1e-3) / 1e9
    assert abs(ach / rf["achieved"] - 1) < 1e-3
    assert abs(rf["achieved"] / rf["peak"] / rf["frac"] - 1) < 1e-3
    assert rf["launches"] == 20
    assert h["e2e"]["h2d_bytes_per_step"] == 16 * 330_311_680
    st = h["streamed"]
    assert st["h8192x8_streamed"]["frac"] == 0.97 and st["h8192x8_streamed"]["unit_max_over_median"] == 1.1
    assert st["h8192x8_streamed"]["async_s_per_step"] == 0.59
    assert "skipped" in st["h8192x8_streamed+x"]
    assert st["h5120x40_streamed"]["bf16_in_hbm"] is True
    assert len(h["chunk_sweep"]["h5120x40_streamed"]["points"]) == 8
    assert json.load(open(out))["streamed"]["timeline_fastest_step"]["units_ms"][0]["h2d_begin"] == 0.0


def test_pinned_arena_carving():
    """The run's arena hands out 256-byte aligned, non-overlapping pieces,
    and a reset makes its space reusable by the next leg."""
    import numpy as np
    import torch
    backing = np.zeros(1 << 20, np.uint8)
    a = object.__new__(bench.PinnedArena)
    a.addr, a.nbytes, a.top = (backing.ctypes.data + 255) // 256 * 256, (1 << 20) - 256, 0
    t1 = a.tensor(1000, torch.int16)
    t2 = a.tensor((3, 5), torch.float32)
    assert t1.data_ptr() % 256 == 0 and t2.data_ptr() % 256 == 0
    assert t2.data_ptr() >= t1.data_ptr() + 2000
    t1.fill_(7)
    t2.fill_(1.5)
    assert int(t1.sum()) == 7000 and float(t2.sum()) == 22.5
    m = a.mark()
    p = a.carve(4096)
    a.reset(m)
    assert a.carve(4096) == p
    with pytest.raises(MemoryError):
        a.carve(1 << 21)
    a.reset()
    assert a.tensor(10, torch.uint8).data_ptr() == a.addr


def test_e2e_link_roofline():
    """The device-to-host bytes run beside part of the host-to-device bytes at
    the concurrent rates; the rest of the host-to-device bytes run alone."""
    link = {"h2d_gbs": 10.0, "d2h_gbs": 8.0, "h2d_concurrent_gbs": 5.0, "d2h_concurrent_gbs": 4.0}
    e2e = {"h2d_bytes_per_step": 1000e9, "d2h_bytes_per_step": 100e9, "value": 1.0}
    # 25 s with both busy (100 GB down at 4, 125 GB up at 5), then 875 GB up at 10
    r = bench.e2e_link_roofline(e2e, link, n=112.5e9)
    assert abs(r["s"] - 112.5) < 1e-9
    assert abs(r["frac"] - 1.0) < 1e-12
    # the smaller direction is host-to-device: it ends first and the rest goes down alone
    e2e2 = {"h2d_bytes_per_step": 50e9, "d2h_bytes_per_step": 200e9, "value": 1.0}
    r2 = bench.e2e_link_roofline(e2e2, link, n=30e9)
    assert abs(r2["s"] - (10 + 160e9 / 8e9)) < 1e-9


def test_streamed_legs_use_the_runs_best_link_probe():
    """A leg whose own probe caught the link in a slow moment is measured
    against the best probe of the run, never against a lowered roofline."""
    fast = {"h2d_gbs": 210.0, "d2h_gbs": 190.0, "h2d_concurrent_gbs": 170.0, "d2h_concurrent_gbs": 170.0,
            "bidir_gbs": 340.0}
    slow = {k: v * 0.8 for k, v in fast.items()}
    best = bench.best_link([slow, fast])
    assert all(best[k] == fast[k] for k in bench.LINK_KEYS)
    N = 1_000_000_000
    t_slow = bench.link_roofline_s(slow, N, True)
    leg = {"params": N, "bf16_copy_in_hbm": True, "s_per_step": t_slow, "s_per_step_min": t_slow,
           "roofline_s": t_slow, "frac": 1.0, "link_bytes_per_step": {"h2d": 12 * N, "d2h": 12 * N},
           "pipelined": {"s_per_step": t_slow}}
    bench.rebase_streamed(leg, best)
    assert leg["own_probe"]["frac"] == 1.0
    assert abs(leg["frac"] - 0.8) < 1e-12          # every rate 1.25x faster: the bound is 0.8x the time
    assert abs(leg["pipelined"]["frac"] - 0.8) < 1e-12
    assert leg["roofline_link"] is best
