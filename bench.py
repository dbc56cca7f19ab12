"""Benchmark of the F^H D gather on one GB300 (or N replicas under torchrun).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5] [--mode fast|accurate]

Prints ONE JSON line.  The default workload is the 256^3-voxel, 100000-sample
kooshball F^H D ("Case study - iterative MRI reconstruction", section 17.3:
the 256^3 x 100k example), in fast mode.

value      voxel-sample pairs per second over the K timed steps, inputs resident
           in device memory; a step is one fhd_compute call (sample pack, gather,
           fix-up).  GFLOP/s = 13 flop/pair x pairs/s / 1e9 (k.x: 3 mul + 2 add;
           complex multiply-accumulate: 4 mul + 4 add; sin/cos not counted).
e2e        the same metric through the public API with pinned HOST buffers:
           every step copies the inputs host->device, runs fhd_compute and
           copies rho back device->host, all inside the timed region; as a
           pipelined client would, step k+1's inputs and step k's result
           cross the host link on two copy streams while step k computes.
roofline   the gather kernel against its plain-ALU bound
           SMs x clock x min(128 / n_fma, 16 / n_xu, 128 / n_issue) pairs/s:
           128 FP32 lanes, a 16-lane pipe for the hardware sin/cos and the
           rounding rintf, and 4 schedulers issuing one warp instruction (32
           lanes) per clock, per SM; n_fma, n_xu and n_issue are the
           algorithm's FP32 lane operations, 16-lane-pipe operations and
           instructions per pair (per_pair_counts: every phase range-reduced
           before its sin/cos, polar weights in the adjoint gather).  On the
           benchmark's grid voxels the fast gather runs the equal-spacing
           recurrence, V = 32 targets per thread, packed f32x2 arithmetic, two
           chains: n_fma = 4 - 4/V + 19/V, n_xu = 6/V, n_issue = 2 + 19/V.
           Maximum SM clock.  The kernel's duration comes from CUDA events
           recorded on its stream around the gather and fix-up launches of
           every timed step.
secondary  the accurate mode evaluated pair by pair (the path of non-grid
           voxels) on the same workload, two steps after the timed region,
           with its own roofline (default line only; --no-secondary skips it).
cpu_baseline  the fp64 CPU oracle on a bounded voxel sample of the same
           workload (test infrastructure; never used by the GPU path).

--impl reference times that oracle alone, as the reference arm, on the same
workload and metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FLOP_PER_PAIR = 13
FMA_LANES_PER_SM = 128   # fp32 FMA-pipe results per SM per clock
MUFU_LANES_PER_SM = 16   # sin/cos results per SM per clock (measured on GB300)
ISSUE_PER_SM = 128       # 4 schedulers x 1 warp instruction (32 lanes) per clock
L2_BYTES = 129 * 1024 * 1024
TARGETS_PER_THREAD = 32


def per_pair_counts(path: str):
    """(FP32 lane operations, 16-lane-pipe operations, issued instructions) per
    pair of the algorithm on `path` (all three count what the algorithm needs,
    not what the compiler emits; the 16-lane pipe runs the hardware sin/cos and
    the rounding rintf).  Every phase is in cycles and range-reduced before
    its sin/cos; the adjoint gathers' weights are polar {|w|, arg(w) / 2 pi},
    so the weight's phase joins the pair's phase and the multiply-accumulate
    is two real FMAs."""
    V = TARGETS_PER_THREAD
    if path == "direct":
        # per target: k.x + arg(w) (3 FMA-pipe operations) and |w| (cos, sin)
        # into the sums (2 FFMA); 6 of 8 targets of a group: t = p - rint(p)
        # with the FMA-pipe rounding (3) and 2 pi t (1), sin and cos on the
        # 16-lane pipe; the other 2 (one packed pair): the fast polynomial
        # (half-period reduction 3, u^2 1, sin 4, cos 4) with the sign flips
        # on the weight.  Targets go in packed f32x2 pairs: 13 instructions per
        # hardware-sin/cos pair of targets (3 + 4 + 4 sin/cos + 2), 22 for the
        # polynomial pair (3 + 12 + 5 + 2)
        g = 8.0
        return 5.0 + (4.0 * 6 + 12.0 * 2) / g, 2.0 * 6 / g, (3 * 13.0 + 22.0) / g
    if path == "direct-accurate":
        # per target: the compensated phase (3 FMUL, 3 rintf, 3 FFMA, 3 FADD
        # with arg(w)), the accurate polynomial (half-period reduction 3, u^2
        # 1, sin 6, cos 5), |w| (cos, sin) into the sums (2): 26 FP32 lane
        # operations and 3 rintf; targets in packed pairs: per two targets 12
        # (the three fractions) + 3 (sums) + 3 (reduction) + 4 (sign flips,
        # on the weight) + 1 + 6 + 5 (polynomials) + 2 (sums) = 36
        # instructions
        return 26.0, 3.0, 18.0
    if path == "source":
        # the fast forward gather's source side (segments of S = 32 equally
        # spaced voxel sources, Cartesian weights) by Clenshaw's recurrence,
        # groups of G = 8 targets, each target's (re, im) in one packed pair:
        # per pair one packed add or subtract and one packed FMA (4 lane
        # operations, 2 instructions); per (target, segment) the phase of e_0
        # (3), its reduction and 2 pi t (4), 2 sin/cos, P = y_0 - y_1 / z and
        # e_0 P into the tile sums (2 packed FMAs each: 8 lanes; with the
        # swaps and sign pairs about 23 instructions); per (source, group)
        # one shared-memory load; the step phasor z once per run of segments
        # with the same step (once per tile on an image grid, not counted).
        S, G = 32.0, 8.0
        return 4.0 + 15.0 / S, 2.0 / S, 2.0 + 23.0 / S + 1.0 / G
    if path == "source-horner":
        # accurate mode's forward gather: the same segments by Horner's rule,
        # two targets per packed pair: per pair the complex multiply-add
        # acc = acc z + w as two packed FMAs for the real parts and two for
        # the imaginary parts of two targets (4 lane operations, 2
        # instructions); per (target, segment) the phase of e_0 (3), its
        # reduction and 2 pi t (4), 2 sin/cos, and e_0 times the segment's sum
        # into the tile sums (4 lanes; about 13 instructions); per (source,
        # group) one shared-memory load and the two weight pairs (3).
        S, G = 32.0, 8.0
        return 4.0 + 11.0 / S, 2.0 / S, 2.0 + 13.0 / S + 3.0 / G
    if path == "recurrence-accurate":
        # the two-chain recurrence of accurate mode on an image grid: the step
        # phasor u and the chain coefficients come from the tile's step
        # records (evaluated once per sample by the pack kernel); per (thread,
        # sample) the compensated phase of the anchor with the weight's phase
        # (9 FMA-pipe operations, 3 rintf), the accurate polynomial (15, 2
        # sign flips), g_0 = |w| (cos, sin) (2), g_1 = g_0 u (4); per target
        # the packed add and step (4 lanes, 2 instructions; no step for the
        # first two targets)
        lanes = 4.0 - 4.0 / V + (9 + 15 + 2 + 4) / V
        xu = 3.0 / V
        issue = 2.0 + (-2 + 12 + 17 + 2 + 4) / V
        return lanes, xu, issue
    if path == "recurrence-accurate-shared":
        # the same where a warp's voxels share a spacing other than the step
        # records' one: the step phasor and the chain coefficient shared by
        # the warp, 2 cos(theta_d) (1), 3 shuffles, and 1/32 of the owner
        # lane's work (the step's compensated phase and sincospif, the
        # coefficient: about 52 operations)
        lanes = 4.0 - 4.0 / V + (9 + 15 + 2 + 4 + 1 + 52.0 / 32) / V
        xu = (3.0 + 3.0 / 32) / V
        issue = 2.0 + (-2 + 12 + 17 + 2 + 4 + 1 + 3 + 55.0 / 32) / V
        return lanes, xu, issue
    if path == "recurrence-per-thread":
        # fast mode where the warp's voxels do not share the step records'
        # spacing: per (thread, sample) the two phases as 3 packed
        # instructions (6 lane operations), + arg(w) (1), the two reductions
        # (2 rintf, 2 FADD) and 2 pi t as one packed multiply (2 lanes),
        # g_0 = |w| (cos, sin) (2), g_1 = g_0 u (4), 2 cos(theta_d) (1),
        # 2 cos(2 theta_d) (1), 4 sin/cos; per target as below
        lanes = 4.0 - 4.0 / V + 19.0 / V
        xu = 6.0 / V
        issue = (2.0 * V - 2.0 + 3.0 + 1.0 + 2.0 + 2.0 + 1.0 + 4.0 + 2.0 + 4.0 + 1.0 + 1.0) / V
        return lanes, xu, issue
    # recurrence (fast mode) on an image grid, V targets per thread, as two
    # chains (even and odd targets), the step phasor u and the chain
    # coefficients from the tile's step records.  Per (thread, sample): the
    # anchor's phase with arg(w) (3 FFMA), its reduction (1 rintf, 1 FADD)
    # and 2 pi t (1), sin and cos, g_0 = |w| (cos, sin) (2), g_1 = g_0 u (4).
    # Per target: one packed add into its accumulator (2 lane operations),
    # and from the third target on one packed three-term step (2 lane
    # operations; the steps to targets 2 and 3 use 2 cos(theta_d), the rest
    # 2 cos(2 theta_d)).
    lanes = 4.0 - 4.0 / V + 11.0 / V
    xu = 3.0 / V
    issue = (2.0 * V - 2.0 + 3.0 + 1.0 + 1.0 + 1.0 + 2.0 + 2.0 + 4.0) / V
    return lanes, xu, issue


WORKLOAD_NAMES = {
    1: "2D 32x32 voxels x 2048 spiral samples, F^H D",
    2: "64^3 voxels x 16384 uniform-random samples, F^H D",
    3: "128^3 voxels x 262144 stack-of-spirals samples, F^H D",
    4: "256^3 voxels x 100000 kooshball samples, F^H D",
    5: "128^3 voxels x 262144 stack-of-spirals samples, F^H F rho",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--mode", choices=["fast", "accurate", "fast-direct", "accurate-direct"], default="fast")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--replicas", action="store_true",
                    help="with N > 1 GPUs: every rank runs the whole workload as an independent problem (weak "
                         "scaling) instead of one problem sharded over the ranks (strong scaling, the default)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary accurate pair-by-pair measurement of the default line")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--ladder", action="store_true",
                    help="time the case study's optimisation ladder (include/fhd_ladder.h) next to the library "
                         "on workloads 1 and 2 instead of the benchmark line (one JSON line per variant)")
    ap.add_argument("--cg", type=int, default=0, metavar="ITERS",
                    help="time ITERS conjugate-gradient iterations (fhd_cg_solve, tolerance 0) on the workload's "
                         "geometry instead of the benchmark line (one JSON line)")
    ap.add_argument("--lam", type=float, default=0.0, help="Tikhonov weight lambda of --cg")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            # one rank per GPU: bind the rank to its device before NCCL starts
            torch.cuda.set_device(local)
            try:
                dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
            except TypeError:  # a PyTorch without the device_id argument
                dist.init_process_group(backend="nccl")
        else:
            dist.init_process_group(backend="gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- workload
def load_workload(i: int):
    from inputs import make_workload

    return make_workload(i)


def peak_pairs_per_s(sms: int, mhz: float, path: str = "direct") -> float:
    if path == "fhf":
        # F^H F rho: half the pairs in the forward gather (source side,
        # Clenshaw's recurrence), half in the adjoint gather (target
        # recurrence); the bound of the whole is the pair-weighted harmonic
        # mean of the two.
        a = peak_pairs_per_s(sms, mhz, "source")
        b = peak_pairs_per_s(sms, mhz, "recurrence")
        return 2.0 / (1.0 / a + 1.0 / b)
    n_fma, n_mufu, n_issue = per_pair_counts(path)
    per_clk = min(FMA_LANES_PER_SM / n_fma, MUFU_LANES_PER_SM / n_mufu, ISSUE_PER_SM / n_issue)
    return sms * per_clk * mhz * 1e6


def fp32_probe(fhd, device: int):
    """FP32 lane operations per second of the library's packed-FMA probe
    kernel on `device` (fhd_test_fma2_rate), or None if it failed."""
    import ctypes

    rate = ctypes.c_double(0.0)
    if fhd.load().fhd_test_fma2_rate(device, ctypes.byref(rate)) != 0 or rate.value <= 0:
        return None
    return rate.value


KERNEL_SOURCES = ("non_cartesian_mri_gather_gb300/csrc/fhd_kernels.cuh",
                  "non_cartesian_mri_gather_gb300/csrc/sincos_poly.cuh",
                  "non_cartesian_mri_gather_gb300/csrc/fhd_api.cu")
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "gather_kernel_fast_256cube_100k_dram.md")


def profiled_traffic(workload: int, mode: str):
    """DRAM bytes per gather launch from the committed ncu summary, or None when
    the summary is for another workload/mode or the kernel sources changed since."""
    import hashlib

    if workload != 4 or mode != "fast":
        return None  # the committed capture is of the default workload and mode
    try:
        fields = {}
        with open(TRAFFIC_PROFILE) as f:
            for line in f:
                if ":" in line and not line.startswith(("|", " ", "#")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        h = hashlib.sha256()
        for rel in KERNEL_SOURCES:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != fields.get("kernel_sources_sha256"):
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(p, seconds: float):
    """Time the fp64 oracle on a strided voxel sample sized for about `seconds`."""
    import oracle

    orc = oracle.get()
    D = None if p.op == "fhf" else (p.Dr, p.Di)
    # calibrate on a small sample
    n_cal = max(1, min(p.N, int(2e7 // max(p.M, 1))))
    idx = np.linspace(0, p.N - 1, n_cal).astype(np.int64)
    t0 = time.perf_counter()
    if D is not None:
        orc.adjoint(p.kx, p.ky, p.kz, D, p.x[idx], p.y[idx], p.z[idx])
    else:
        orc.adjoint(p.kx, p.ky, p.kz, (p.rho_r[: p.M], p.rho_i[: p.M]), p.x[idx], p.y[idx], p.z[idx])
    dt = max(time.perf_counter() - t0, 1e-6)
    rate = n_cal * p.M / dt
    n = int(min(p.N, max(n_cal, seconds * rate / p.M)))
    idx = np.linspace(0, p.N - 1, n).astype(np.int64)
    t0 = time.perf_counter()
    if D is not None:
        orc.adjoint(p.kx, p.ky, p.kz, D, p.x[idx], p.y[idx], p.z[idx])
    else:
        orc.adjoint(p.kx, p.ky, p.kz, (p.rho_r[: p.M], p.rho_i[: p.M]), p.x[idx], p.y[idx], p.z[idx])
    dt = time.perf_counter() - t0
    cores = orc.threads()
    # the per-core rate: one thread on a sample of about a tenth of the time
    n1 = max(1, min(n, int(0.1 * seconds * rate / cores / p.M)))
    idx1 = np.linspace(0, p.N - 1, n1).astype(np.int64)
    prev = orc.set_threads(1)
    try:
        t1 = time.perf_counter()
        if D is not None:
            orc.adjoint(p.kx, p.ky, p.kz, D, p.x[idx1], p.y[idx1], p.z[idx1])
        else:
            orc.adjoint(p.kx, p.ky, p.kz, (p.rho_r[: p.M], p.rho_i[: p.M]), p.x[idx1], p.y[idx1], p.z[idx1])
        dt1 = time.perf_counter() - t1
    finally:
        orc.set_threads(prev)
    return {"value": n * p.M / dt, "unit": "pairs/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {p.N} voxels (evenly spaced) x all {p.M} samples, adjoint sum, fp64, "
                      f"{dt:.1f} s", "seconds": dt, "pairs": n * p.M,
            "per_core_value": n1 * p.M / dt1,
            "per_core_sample": f"{n1} voxels x all {p.M} samples on 1 thread, {dt1:.1f} s"}


def run_reference(args, world, rank):
    """Reference arm: the fp64 CPU oracle, bounded sample per step, rank 0 only."""
    if rank != 0:
        return
    p = load_workload(args.workload)
    per_step = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        oracle_sample(p, min(per_step, 2.0))
    vals, secs, last = [], [], None
    for _ in range(args.steps):
        last = oracle_sample(p, per_step)
        vals.append(last["pairs"])
        secs.append(last["seconds"])
    value = sum(vals) / sum(secs)
    line = {
        "impl": "reference", "metric": "F^H D voxel-sample pairs/s", "value": value, "unit": "pairs/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(secs) / len(secs), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "gflops": FLOP_PER_PAIR * value / 1e9,
        "config": {"workload": WORKLOAD_NAMES[args.workload], "N": p.N, "M": p.M},
        "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": last["cores"], "kind": "oracle",
                         "sample": f"per step: {last['sample']}", "per_core_value": last["per_core_value"],
                         "per_core_sample": last["per_core_sample"]},
        "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
def gather_launches(fhd, shape, sms, n_targets, n_sources):
    """Kernels one gather of the library launches: pack, describe, gather and
    fix-up on the persistent path (no fix-up with a single CTA); the split
    gather and (with more than one slice) the slice reduction on the split
    path, which the library takes by the rule fhd_test_split_shape reports."""
    import ctypes

    per_block = shape["threads"] * shape["targets_per_thread"]
    partial_bytes = 2 * shape["ctas"] * 2 * per_block * 4
    k = ctypes.c_int(0)
    split = fhd.load().fhd_test_split_shape(n_targets, n_sources, sms, shape["ctas"], partial_bytes,
                                            ctypes.byref(k), None)
    if split == 1:
        return 1 + (1 if k.value > 1 else 0)
    work = -(-n_targets // per_block) * -(-n_sources // shape["tile_sources"])
    return 3 + (1 if min(work, shape["ctas"]) > 1 else 0)


def run_ours(args, world, rank, local):
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fhd.load()
    mode = {"fast": fhd.MODE_FAST, "accurate": fhd.MODE_ACCURATE, "fast-direct": fhd.MODE_FAST_DIRECT,
            "accurate-direct": fhd.MODE_ACCURATE_DIRECT}[args.mode]
    # The benchmark voxels are power-of-two grids: every thread's 32
    # consecutive voxels are exactly equally spaced, so the recurrence runs
    # unless disabled.
    path = {"fast": "recurrence", "accurate": "recurrence-accurate", "fast-direct": "direct",
            "accurate-direct": "direct-accurate"}[args.mode]
    p = load_workload(args.workload)
    fhf = p.op == "fhf"
    if fhf:  # F^H F rho: the forward gather (voxel sources) then the adjoint gather
        path = "direct" if args.mode.endswith("direct") else "fhf"
    job_pairs = p.pairs  # one problem; with replicas every rank runs its own
    job_N = p.N
    # One problem sharded over the ranks (non_cartesian_mri_gather_gb300.sharded):
    # F^H D by voxel ranges, no exchange; F^H F rho with the image sharded by
    # voxel ranges and two all-gathers (rho, then F rho) between the passes.
    shard = world > 1 and not args.replicas
    n0, n1 = 0, p.N
    if shard:
        from non_cartesian_mri_gather_gb300 import sharded

        n0, n1 = sharded.partition(p.N, world, rank)
        if not fhf:
            p.x, p.y, p.z = (np.ascontiguousarray(a[n0:n1]) for a in (p.x, p.y, p.z))
        else:
            p.rho_r, p.rho_i = (np.ascontiguousarray(a[n0:n1]) for a in (p.rho_r, p.rho_i))
    n_out = n1 - n0
    names = ("x", "y", "z", "rho_r", "rho_i", "kx", "ky", "kz") if fhf else ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")
    host = {k: torch.from_numpy(getattr(p, k)) for k in names}
    d = {k: v.to(dev) for k, v in host.items()}
    rho_r = torch.empty(n_out, dtype=torch.float32, device=dev)
    rho_i = torch.empty(n_out, dtype=torch.float32, device=dev)
    ws = fhd.Workspace(fhd.OP_FHF if fhf else fhd.OP_FHD, p.N, p.M, local)
    stream = torch.cuda.current_stream(dev)
    shape = fhd.fhd_launch_shape(local, mode)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    input_bytes = sum(v.numel() * 4 for v in d.values())

    def step(e0=None, e1=None, dd=None, out=None, mode=mode):
        dd = d if dd is None else dd
        rr, ri = (rho_r, rho_i) if out is None else out
        if fhf:
            if e0 is not None:
                e0.record(stream)
            if shard:
                o_r, o_i = sharded.fhfrho_apply_sharded(dd["x"], dd["y"], dd["z"], dd["rho_r"], dd["rho_i"], dd["kx"],
                                                        dd["ky"], dd["kz"], mode=mode)
                rr.copy_(o_r)
                ri.copy_(o_i)
            else:
                fhd.fhfrho_apply(dd["x"], dd["y"], dd["z"], dd["rho_r"], dd["rho_i"], dd["kx"], dd["ky"], dd["kz"],
                                 rr, ri, mode=mode, workspace=ws)
            if e1 is not None:
                e1.record(stream)
        elif e0 is None:
            fhd.fhd_compute(dd["kx"], dd["ky"], dd["kz"], dd["Dr"], dd["Di"], dd["x"], dd["y"], dd["z"], rr, ri,
                            mode=mode, workspace=ws)
        else:
            fhd.fhd_compute_profiled(dd["kx"], dd["ky"], dd["kz"], dd["Dr"], dd["Di"], dd["x"], dd["y"], dd["z"], rr,
                                     ri, mode, ws, e0, e1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fhd.fhd_workspace_status(ws) != 0:
        raise SystemExit("kernel reported a pipeline timeout during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for pair in ev + step_ev:  # create the CUDA events before the timed region
        for e in pair:
            e.record(stream)
    # Inputs that fit in L2 are evicted before every timed step by writing a
    # buffer of twice the L2 size; the write lies outside the step's events.
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if input_bytes <= L2_BYTES else None
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    for (e0, e1), (s0, s1) in zip(ev, step_ev):
        if flush is not None:
            flush.fill_(1.0)
        s0.record(stream)
        step(e0, e1)
        s1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    status = fhd.fhd_workspace_status(ws)
    if status != 0:
        raise SystemExit(f"kernel status {status} in the timed region")
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ms_local = sum(step_ms) / args.steps
    ms = max_over_ranks(ms_local, world)
    gather_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    pairs = p.pairs if not (shard and fhf) else 2 * n_out * p.M  # this rank's pairs
    job = job_pairs if shard else world * job_pairs  # pairs all ranks process per step
    value = job / (ms * 1e-3)

    # ---- end to end through the public API with pinned host buffers.  A
    # pipelined client: step k+1's inputs cross host -> device on one stream
    # and step k's result device -> host on another while step k computes
    # (inputs and outputs double-buffered on the device); every step's copies
    # lie inside the timed region, which runs from before the first input
    # copy to the end of the last result copy.
    e2e = None
    if not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in host.items()}
        out_r = torch.empty(n_out, dtype=torch.float32).pin_memory()
        out_i = torch.empty(n_out, dtype=torch.float32).pin_memory()
        bufs = [d, {k: torch.empty_like(v) for k, v in d.items()}]
        outs = [(rho_r, rho_i), (torch.empty_like(rho_r), torch.empty_like(rho_i))]
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]

        def h2d(slot):
            with torch.cuda.stream(h2d_s):
                if used[slot]:
                    h2d_s.wait_event(comp_done[slot])  # the step that read this buffer is done
                for k in names:
                    bufs[slot][k].copy_(pin[k], non_blocking=True)
                h2d_done[slot].record(h2d_s)

        def compute(slot):
            stream.wait_event(h2d_done[slot])
            if used[slot]:
                stream.wait_event(d2h_done[slot])  # this output buffer has been read back
            step(dd=bufs[slot], out=outs[slot])
            comp_done[slot].record(stream)
            used[slot] = True

        def d2h(slot):
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(comp_done[slot])
                out_r.copy_(outs[slot][0], non_blocking=True)
                out_i.copy_(outs[slot][1], non_blocking=True)
                d2h_done[slot].record(d2h_s)

        def run_e2e(k_steps, s_ev=None, t_ev=None):
            if s_ev is not None:
                s_ev.record(stream)
                h2d_s.wait_event(s_ev)
            h2d(0)
            for i in range(k_steps):
                if i + 1 < k_steps:
                    h2d((i + 1) % 2)
                compute(i % 2)
                d2h(i % 2)
            if t_ev is not None:
                stream.wait_stream(d2h_s)
                t_ev.record(stream)

        run_e2e(2)
        torch.cuda.synchronize()
        k2 = max(3, min(args.steps, 5))
        barrier(world)
        torch.cuda.synchronize()
        s2, t2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        run_e2e(k2, s2, t2)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(s2.elapsed_time(t2) / k2, world)

        # the same steps with the copies in line (one stream, no overlap)
        def serial_step():
            for k in names:
                d[k].copy_(pin[k], non_blocking=True)
            step()
            out_r.copy_(rho_r, non_blocking=True)
            out_i.copy_(rho_i, non_blocking=True)

        serial_step()
        barrier(world)
        torch.cuda.synchronize()
        s3, t3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record(stream)
        for _ in range(k2):
            serial_step()
        t3.record(stream)
        torch.cuda.synchronize()
        ms_serial = max_over_ranks(s3.elapsed_time(t3) / k2, world)
        e2e = {"value": job / (ms_e2e * 1e-3), "unit": "pairs/s", "h2d_bytes_per_step": input_bytes,
               "d2h_bytes_per_step": 2 * n_out * 4, "ms_per_step": ms_e2e, "steps": k2,
               "pipeline": "inputs of step k+1 copied in and the result of step k copied out while step k "
                           "computes (two copy streams, double-buffered device arrays)",
               "serial": {"value": job / (ms_serial * 1e-3), "ms_per_step": ms_serial,
                          "note": "copy in, compute, copy out on one stream, no overlap"}}

    if rank != 0:
        return
    if fhf:
        m0, m1 = sharded.partition(p.M, world, rank) if shard else (0, p.M)
        gathers = [(m1 - m0, p.N), (n_out, p.M)]
    else:
        gathers = [(p.N, p.M)]
    launches = sum(gather_launches(fhd, shape, sms, nt, ns) for nt, ns in gathers)

    # ---- roofline of the gather kernel (plain-ALU bound)
    peaks = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz") or clk.get("sm_max_mhz") or 2070.0)
    peak = peak_pairs_per_s(sms, max_mhz, path)
    achieved = pairs / (gather_ms * 1e-3)
    n_fma, n_mufu, n_issue = per_pair_counts("recurrence" if path == "fhf" else path)
    roof = {
        "bound": "alu",
        "achieved": FLOP_PER_PAIR * achieved / 1e12,
        "peak": FLOP_PER_PAIR * peak / 1e12,
        "unit": "TFLOP/s",
        "frac": achieved / peak,
        "traffic": profiled_traffic(args.workload, args.mode),
        "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
        "kernel": "gather_kernel" if not fhf else "gather_kernel x2 (whole fhfrho_apply call)",
        "kernel_ms": gather_ms,
        "path": path,
        "peak_basis": (f"{sms} SMs x {max_mhz:.0f} MHz x min({FMA_LANES_PER_SM}/{n_fma:g}, "
                       f"{MUFU_LANES_PER_SM}/{n_mufu:g}, {ISSUE_PER_SM}/{n_issue:g}) pairs/clk x "
                       f"{FLOP_PER_PAIR} flop/pair ({path} path)") if path != "fhf" else (
            f"{sms} SMs x {max_mhz:.0f} MHz, pair-weighted harmonic mean of the forward gather's "
            f"source-side (Clenshaw) bound and the adjoint gather's target-recurrence bound x {FLOP_PER_PAIR} "
            f"flop/pair"),
        "direct_path_peak": FLOP_PER_PAIR * peak_pairs_per_s(sms, max_mhz, "direct") / 1e12,
        # the plain pair-by-pair bound (a sin and a cos per pair), which the
        # recurrences exceed: achieved / that bound
        "frac_of_direct_path_peak": achieved / peak_pairs_per_s(sms, max_mhz, "direct"),
    }
    if clk.get("sm_mhz"):
        roof["frac_at_sampled_clock"] = achieved / peak_pairs_per_s(sms, clk["sm_mhz"], path)
    if fhf and not args.mode.startswith("fast"):
        roof["peak_basis"] += " (the fast mode's operation counts: an upper bound for accurate mode)"
    # ---- the packed FP32 rate this GPU reaches in practice (a register-only
    # probe kernel, after the timed region): the gather's FP32 lane operations
    # per second, from the same per-pair count as the bound, as a share of it
    probe = fp32_probe(fhd, torch.cuda.current_device())
    if probe:
        lanes_per_pair = ((per_pair_counts("source")[0] + per_pair_counts("recurrence")[0]) / 2 if fhf
                          else n_fma)
        lanes = achieved * lanes_per_pair
        roof["fp32_probe"] = {"lane_ops_per_s": probe, "frac_of_nominal": probe / (sms * FMA_LANES_PER_SM *
                                                                                   max_mhz * 1e6),
                              "gather_lane_ops_per_s": lanes, "gather_frac_of_probe": lanes / probe}

    # ---- secondary: the accurate pair-by-pair path on the same workload (the
    # path a caller with non-grid voxels takes in accurate mode), a few steps
    secondary = None
    if not fhf and args.mode == "fast" and not args.no_secondary:
        acc_mode = fhd.MODE_ACCURATE_DIRECT
        step(mode=acc_mode)
        torch.cuda.synchronize()
        sec = []
        for _ in range(2):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for e in (a0, a1, g0, g1):
                e.record(stream)
            torch.cuda.synchronize()
            a0.record(stream)
            step(g0, g1, mode=acc_mode)
            a1.record(stream)
            torch.cuda.synchronize()
            sec.append((a0.elapsed_time(a1), g0.elapsed_time(g1)))
        s_ms = sum(x[0] for x in sec) / len(sec)
        s_gather = sum(x[1] for x in sec) / len(sec)
        s_peak = peak_pairs_per_s(sms, max_mhz, "direct-accurate")
        s_ach = pairs / (s_gather * 1e-3)
        nf, nx, ni = per_pair_counts("direct-accurate")
        secondary = {
            "mode": "accurate-direct", "value": pairs / (s_ms * 1e-3), "unit": "pairs/s", "ms_per_step": s_ms,
            "steps": len(sec), "warmup": 1,
            "roofline": {"bound": "alu", "achieved": FLOP_PER_PAIR * s_ach / 1e12,
                         "peak": FLOP_PER_PAIR * s_peak / 1e12, "unit": "TFLOP/s", "frac": s_ach / s_peak,
                         "kernel_ms": s_gather, "path": "direct-accurate",
                         "peak_basis": f"{sms} SMs x {max_mhz:.0f} MHz x min({FMA_LANES_PER_SM}/{nf:g}, "
                                       f"{MUFU_LANES_PER_SM}/{nx:g}, {ISSUE_PER_SM}/{ni:g}) pairs/clk x "
                                       f"{FLOP_PER_PAIR} flop/pair"},
            "note": "accurate mode evaluated pair by pair (FHD_MODE_ACCURATE_DIRECT): the path of non-grid voxels",
        }

    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = oracle_sample(p, args.cpu_seconds)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "per_core_value", "per_core_sample")}

    line = {
        "metric": "F^H F rho voxel-sample pairs/s (both passes)" if fhf else "F^H D voxel-sample pairs/s",
        "value": value,
        "unit": "pairs/s",
        "gflops": FLOP_PER_PAIR * value / 1e9,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_median": float(np.median(step_ms)),
        "ms_per_step_best": min(step_ms),
        "higher_is_better": True,
        "scaling": "strong" if shard else "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "mode": args.mode,
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD_NAMES[args.workload],
            "N": job_N,
            "M": p.M,
            "pairs_per_step": job,
            "flop_per_pair": FLOP_PER_PAIR,
            "l2": f"inputs exceed L2 ({input_bytes / 2**20:.0f} MiB of inputs vs {L2_BYTES / 2**20:.0f} MiB L2)"
                  if input_bytes > L2_BYTES else
                  f"L2 flushed before every timed step ({2 * L2_BYTES / 2**20:.0f} MiB write outside the step's events)",
            "launch": shape,
            "parallelism": (f"one problem sharded over {world} ranks (voxel ranges"
                            + (", two all-gathers per step)" if fhf else ", no exchange)")) if shard else
                           (f"replicas x{world}" if world > 1 else "single GPU"),
        },
        "roofline": roof,
        "secondary": secondary,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_ladder(args):
    """One JSON line per (workload, variant): the ladder steps L0-L5, the scatter
    form (workload 1 only: its atomics serialise on every voxel) and the
    library's accurate and fast paths, timed with CUDA events after warm-up."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    fhd.load()
    for wl in (1, 2):
        p = load_workload(wl)
        d = {k: torch.from_numpy(getattr(p, k)).cuda() for k in ("kx", "ky", "kz", "Dr", "Di", "x", "y", "z")}
        args_t = (d["kx"], d["ky"], d["kz"], d["Dr"], d["Di"], d["x"], d["y"], d["z"])
        runs = [(v, lambda v=v: fhd.fhd_compute_variant(v, *args_t)) for v in fhd.VARIANTS
                if not (v == "scatter" and wl != 1)]
        ws = fhd.Workspace(fhd.OP_FHD, p.N, p.M)
        for name, mode in (("library accurate", fhd.MODE_ACCURATE), ("library fast", fhd.MODE_FAST)):
            runs.append((name, lambda mode=mode: fhd.fhd_compute(*args_t, mode=mode, workspace=ws)))
        ref = None
        for name, fn in runs:
            for _ in range(max(1, args.warmup)):
                out = fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(1, args.steps)
            a.record()
            for _ in range(reps):
                out = fn()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b) / reps
            val = torch.complex(out[0].double(), out[1].double()).cpu().numpy()
            if ref is None:
                ref = val
            rel = float(np.linalg.norm(val - ref) / np.linalg.norm(ref))
            pairs = p.N * p.M
            print(json.dumps({"ladder": name, "workload": WORKLOAD_NAMES[wl], "ms": ms, "pairs_per_s": pairs / (ms * 1e-3),
                              "gflops_13": FLOP_PER_PAIR * pairs / (ms * 1e-3) / 1e9,
                              "rel_l2_vs_naive": rel}), flush=True)


def run_cg(args):
    """One JSON line: args.cg iterations of fhd_cg_solve on the workload's
    voxels and samples, timed with CUDA events around the whole solve (b =
    F^H D, then per iteration one F^H F p and the vector updates) after
    args.warmup untimed solves, median of args.steps solves.  The data D are
    the workload's k-space data; for workload 5 (an image workload) D = F rho
    of its phantom (accurate mode), so the solve should approach that image.
    Pairs per solve: N M for b plus 2 N M per iteration."""
    import torch

    import non_cartesian_mri_gather_gb300 as fhd

    fhd.load()
    mode = {"fast": fhd.MODE_FAST, "accurate": fhd.MODE_ACCURATE, "fast-direct": fhd.MODE_FAST_DIRECT,
            "accurate-direct": fhd.MODE_ACCURATE_DIRECT}[args.mode]
    p = load_workload(args.workload)
    dev = torch.device("cuda", 0)
    names = ("x", "y", "z", "kx", "ky", "kz") + (("rho_r", "rho_i") if p.op == "fhf" else ("Dr", "Di"))
    d = {k: torch.from_numpy(getattr(p, k)).to(dev) for k in names}
    if p.op == "fhf":
        Dr, Di = fhd.fwd_compute(d["x"], d["y"], d["z"], d["rho_r"], d["rho_i"], d["kx"], d["ky"], d["kz"],
                                 mode=fhd.MODE_ACCURATE)
    else:
        Dr, Di = d["Dr"], d["Di"]
    ws = fhd.CgWorkspace(p.N, p.M)

    def solve(info=False):
        return fhd.fhd_cg_solve(d["kx"], d["ky"], d["kz"], Dr, Di, d["x"], d["y"], d["z"], lam=args.lam,
                                max_iter=args.cg, tol=0.0, mode=mode, workspace=ws, info=info)

    for _ in range(args.warmup):
        solve()
    torch.cuda.synchronize()
    times = []
    for _ in range(max(1, args.steps)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        solve()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    rr, ri, (iters, rs, stopped) = solve(info=True)
    pairs = p.N * p.M * (1 + 2 * iters)
    line = {"metric": "CG solve voxel-sample pairs/s", "value": pairs / (ms * 1e-3), "unit": "pairs/s",
            "ms_per_solve": ms, "iterations": iters, "ms_per_iteration": ms / max(iters, 1), "rs_final": rs,
            "stopped": stopped, "lambda": args.lam, "mode": args.mode, "steps": len(times), "warmup": args.warmup,
            "config": {"workload": WORKLOAD_NAMES[args.workload], "N": p.N, "M": p.M,
                       "data": "F rho of the phantom" if p.op == "fhf" else "the workload's k-space data"}}
    if p.op == "fhf":
        got = torch.complex(rr.double(), ri.double()).cpu().numpy()
        truth = p.rho_r.astype(np.float64) + 1j * p.rho_i
        line["rel_to_phantom"] = float(np.linalg.norm(got - truth) / np.linalg.norm(truth))
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.ladder:
        run_ladder(args)
        return
    if args.cg:
        run_cg(args)
        return
    world, rank, local = dist_init()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
