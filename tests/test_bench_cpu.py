"""bench.py host logic without a GPU: argument defaults, the roofline
arithmetic, the reference arm on the small workload, and the multi-process
reduction (max over ranks, barrier) on two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_defaults(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert (a.gpus, a.steps, a.warmup, a.impl, a.workload, a.mode) == (1, 5, 3, "ours", 4, "fast")
    assert a.warmup >= 3


def test_roofline_counts():
    # pair by pair: the 16-lane pipe binds; 6 of 8 targets take sin and cos
    # on it, so 16 / (2 * 6/8) = 10.7 pairs per SM per clock.  Per target:
    # the phase with the weight's phase (3) and the two real FMAs of a polar
    # weight (2); a hardware-sin/cos target adds its reduction and 2 pi t (4),
    # a polynomial target 12 FP32 operations; targets go in packed pairs (61
    # instructions per group of 8)
    lanes, xu, issue = bench.per_pair_counts("direct")
    assert (lanes, xu, issue) == (5 + (4 * 6 + 12 * 2) / 8, 2 * 6 / 8, 61 / 8)
    assert abs(bench.peak_pairs_per_s(152, 2070.0, "direct") - 152 * (16 / xu) * 2070e6) < 1
    assert 16 / xu < min(128 / lanes, 128 / issue)
    # the recurrence with step records: per target 4 lanes in 2 instructions
    # (the first two targets take no step), per (thread, sample) 11 lanes
    # (the anchor's phase 3, reduction 1, 2 pi t 1, g_0 2, g_1 4), 3
    # operations on the 16-lane pipe (sin, cos, rintf) and 14 instructions
    lanes, xu, issue = bench.per_pair_counts("recurrence")
    V = bench.TARGETS_PER_THREAD
    assert abs(lanes - (4 - 4 / V + 11 / V)) < 1e-12 and abs(xu - 3 / V) < 1e-12
    assert abs(issue - (2 + 12 / V)) < 1e-12
    # a warp evaluating its own step phasor: 19 lanes, 6 on the 16-lane pipe
    # (4 sin/cos, 2 rintf) and 21 instructions per (thread, sample)
    lanes_t, xu_t, issue_t = bench.per_pair_counts("recurrence-per-thread")
    assert abs(lanes_t - (4 - 4 / V + 19 / V)) < 1e-12 and abs(xu_t - 6 / V) < 1e-12
    assert abs(issue_t - (2 + 19 / V)) < 1e-12
    # with V = 32 the FP32 lanes bind
    assert abs(bench.peak_pairs_per_s(152, 2070.0, "recurrence") - 152 * (128 / lanes) * 2070e6) < 1
    # accurate pair by pair: 26 FP32 lane operations per pair bind
    lanes, xu, issue = bench.per_pair_counts("direct-accurate")
    assert abs(bench.peak_pairs_per_s(152, 2070.0, "direct-accurate") - 152 * (128 / lanes) * 2070e6) < 1
    for path in ("source", "source-horner", "recurrence-accurate", "recurrence-accurate-shared"):
        assert all(v > 0 for v in bench.per_pair_counts(path))
    # the step records take work off the accurate recurrence too
    assert bench.per_pair_counts("recurrence-accurate")[0] < bench.per_pair_counts("recurrence-accurate-shared")[0]


def test_profiled_traffic_is_guarded():
    assert bench.profiled_traffic(2, "fast") is None
    assert bench.profiled_traffic(4, "accurate") is None
    v = bench.profiled_traffic(4, "fast")
    assert v is None or v > 0


def test_reference_arm_runs(tmp_path):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "pairs/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench as b

    w, r, _ = b.dist_init()
    b.barrier(w)
    m = b.max_over_ranks(10.0 + r, w)
    with open(os.path.join(out, f"r{r}.txt"), "w") as f:
        f.write(repr(m))
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    vals = [float(open(tmp_path / f"r{i}.txt").read()) for i in range(2)]
    assert vals == [11.0, 11.0]
