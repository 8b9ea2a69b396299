#!/usr/bin/env python
"""Benchmark of the differentiable projection step at box 256 (cubic).

One step is the whole hot path over one batch: forward 3D->2D projection of a
256^3 spectrum for 512 poses with shifts (cubic, radius 128), the L2-loss
gradient g = 2 (y - target) against seeded noisy targets (SNR 0.1), and the
backward pass producing dL/dR, dL/dshift and dL/dvolume.  The forward carries
the L2 data term (tp_project_3d_2d_l2): it writes y and g and reduces the
rotation and shift gradients from its own gather of the stencil derivatives;
the volume gradient is the brick scatter of g.  The metric is
Fourier samples per second (one sample = one stored output RFFT pixel) over
forward + backward, in Gsamples/s.

  python bench.py [--gpus N --steps K --warmup W]   # this library, one JSON line
  python bench.py --impl reference                   # the float64 CPU oracle arm

With N > 1 (torchrun, one process per GPU) every rank runs an independent
512-pose problem against its own volume (weak scaling, no collective on the
data path); rank 0 prints the aggregate.  The L2 is flushed (a 256 MB write)
between timed steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = 5
METRIC = "Fourier samples/sec (Gsamples/s) fwd+bwd at box 256 cubic; % of mem roofline"
UNIT = "Gsamples/s"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample-poses", type=int, default=512,
                    help="poses of the workload one CPU-baseline oracle step processes")
    ap.add_argument("--cpu-min-seconds", type=float, default=10.0,
                    help="the CPU-baseline leg repeats oracle steps until this much time has passed")
    ap.add_argument("--ref-poses", type=int, default=8,
                    help="poses per step of the reference (oracle) arm (each step also pays for "
                         "the float64 volume gradient of the whole 256^3 spectrum)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--eager", action="store_true",
                    help="time the step's launches one by one instead of replaying a CUDA graph")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary figures of the headline line (2D step, box-256 "
                         "backprojection)")
    ap.add_argument("--poses", type=int, default=None,
                    help="pose count (default: the workload's 512); smaller runs are for profiling")
    ap.add_argument("--workload", default="fwdbwd",
                    choices=["fwdbwd", "project", "rot2d", "backproject", "backproject-backward",
                             "oversampling", "hostlink"],
                    help="fwdbwd: the differentiable step (the headline, default); project: box-128 "
                         "cubic forward of 4096 poses (--oversampling 1 or 2); rot2d: 2D rotate + "
                         "shift of 1024 images at 128, forward and backward; backproject: "
                         "2048 images into a 256^3 data + weight spectrum; backproject-backward: "
                         "the gradients of that backprojection; oversampling: cubic at s = 1 "
                         "against linear at s = 2 with the padding FFT, box 128, 4096 poses; "
                         "hostlink: pinned host <-> device copy bandwidth, the bound of the "
                         "end-to-end figure")
    ap.add_argument("--interp", default="cubic", choices=["linear", "cubic"],
                    help="interpolation of the project and backproject workloads")
    ap.add_argument("--oversampling", type=int, default=1, choices=[1, 2],
                    help="oversampling of the project workload (2: the 256^3 padded spectrum)")
    ap.add_argument("--ncu-summary", metavar="RAW_CSV", nargs="+", default=None,
                    help="write profiles/ncu_traffic.json from `ncu -i REP --page raw --csv` "
                         "exports (one capture per kernel; the first launch of each kernel in "
                         "the order given is kept)")
    return ap.parse_args()


def config_dict(w, P):
    c = synth.CONFIGS[WORKLOAD]
    return {"workload": c["name"], "box": c["box"], "poses": P, "interp": c["interp"],
            "oversampling": 1.0, "radius": c["radius"], "shift_px": c["shift_lim"],
            "loss": "L2 vs noisy targets, SNR 0.1", "l2_cache": "flushed between steps (256 MB write)",
            "samples_per_step": P * c["box"] * (c["box"] // 2 + 1)}


def in_radius_count(N, r):
    kx = np.arange(N // 2 + 1)[None, :]
    ky = np.fft.fftfreq(N, 1.0 / N)[:, None]
    return int((kx * kx + ky * ky <= r * r).sum())


# ---------------------------------------------------------------------------
# CPU oracle (reference arm and cpu_baseline leg).
def oracle_step(w, P):
    import oracle
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    vol, R, t = w["vol"], w["rot"][:, :P], w["shift"][:, :P]
    y = oracle.project(3, vol, R, shift=t, **kw)
    g = 2.0 * (y - w["target"][:, :P])
    oracle.project_backward(3, g, vol, R, shift=t, **kw)


def oracle_sample_workload(P):
    w = synth.workload(WORKLOAD, poses=P)
    rng = synth.streams(7000 + WORKLOAD, 1)[0]
    w["target"] = synth.complex_normal(w["grad"].shape, rng)   # any target: the cost is the same
    return w


def cpu_baseline(P, min_seconds):
    """The oracle, as it stands, on this host's cores: whole steps over the
    first P poses, repeated (at most 10 times) until min_seconds passed."""
    import oracle
    w = oracle_sample_workload(P)
    reps, dt = 0, 0.0
    while reps < 10 and (reps == 0 or dt < min_seconds):
        t0 = time.perf_counter()
        oracle_step(w, P)
        dt += time.perf_counter() - t0
        reps += 1
    samples = reps * P * w["box"] * (w["box"] // 2 + 1)
    cores = oracle.num_threads()
    # The same step on one thread, over a smaller leading subset of poses.
    P1 = max(1, P // 32)
    w1 = oracle_sample_workload(P1)
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle_step(w1, P1)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(cores)
    return {"value": samples / dt / 1e9, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} x {P} of the 512 poses of the box-256 step (fwd + L2 grad + bwd), "
                      f"float64, {dt:.1f} s",
            "single_thread": {"value": P1 * w1["box"] * (w1["box"] // 2 + 1) / dt1 / 1e9,
                              "sample": f"{P1} poses, {dt1:.1f} s"},
            "cpu_model": cpu_model()}


def cpu_model():
    """The host CPU's model name, from /proc/cpuinfo when there is one."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    P = args.ref_poses
    w = oracle_sample_workload(P)
    samples = P * w["box"] * (w["box"] // 2 + 1)
    for _ in range(args.warmup):
        oracle_step(w, P)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, P)
        times.append(time.perf_counter() - t0)
    value = samples * len(times) / sum(times) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, 512),
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "value": value,
                             "unit": UNIT,
                             "sample": f"each step: {P} of the 512 poses (fwd + L2 grad + bwd)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# Clock sampling during the timed region (nvidia-smi query loop, read-only).
class ClockSampler:
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        import torch
        self.bus = None
        try:
            p = torch.cuda.get_device_properties(index)
            self.bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:  # noqa: BLE001
            pass
        self.proc, self.error = None, None

    def __enter__(self):
        import subprocess
        import tempfile
        self.out = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception as e:  # noqa: BLE001
            self.error = str(e)
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait()

    def record(self):
        if self.proc is None:
            return {"error": self.error or "nvidia-smi unavailable"}
        self.out.seek(0)
        rows = [r.split(", ") for r in self.out.read().strip().splitlines() if r.strip()]
        if self.bus:
            mine = [r for r in rows if r[0].upper().endswith(self.bus[-7:])]
            rows = mine or rows
        sm, mx, reasons = [], None, set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for name, flag in zip(self.REASONS, r[3:7]):
                    if flag.strip() == "Active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"error": "no clock samples"}
        return {"sm_mhz": float(statistics.median(sm)), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "n_samples": len(sm)}


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6400.0, "fallback"


# The sources of the step's kernels (k_brick_project, k_brick_scatter_cubic
# and the binning passes): a committed ncu summary is reported only while
# these files are unchanged.
KERNEL_SOURCES = ("tp_brick.cu", "tp_device.cuh")


def kernel_source_sha():
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        f = os.path.join(ROOT, "backprojection_tp_project_gather_b300", "csrc", name)
        with open(f, "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


# The two kernels that do the work of a step, by the bench's segment names.
NCU_KERNELS = {"project_3d_2d": "k_brick_project", "volume_grad_scatter": "k_brick_scatter_cubic"}
NCU_METRICS = {"dram__bytes_read.sum": "dram_read_bytes", "dram__bytes_write.sum": "dram_write_bytes",
               "gpu__time_duration.sum": "duration_ns",
               "gpu__compute_memory_throughput.avg.pct_of_peak_sustained_elapsed": "mem_sol_pct",
               "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed": "dram_pct",
               "lts__throughput.avg.pct_of_peak_sustained_elapsed": "l2_pct",
               "l1tex__throughput.avg.pct_of_peak_sustained_elapsed": "l1_pct",
               "sm__warps_active.avg.pct_of_peak_sustained_active": "warps_active_pct",
               "launch__registers_per_thread": "registers"}
UNIT_SCALE = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9,
              "ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6, "nsecond": 1,
              "%": 1, "register/thread": 1, "": 1}


def ncu_summary(csv_paths, out_path):
    """Write profiles/ncu_traffic.json from `ncu -i <rep> --page raw --csv` exports.

    One entry per bench segment with the captured launch's DRAM bytes, duration
    and throughput percentages, tagged with the hash of the kernel sources so
    that a stale summary is never reported against changed kernels.  Each
    export may hold one kernel (one capture per kernel) or several; the first
    launch of each kernel is kept."""
    import csv
    if isinstance(csv_paths, str):
        csv_paths = [csv_paths]
    kernels = {}
    for csv_path in csv_paths:
        rows = list(csv.reader(open(csv_path)))
        hdr = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
        names, units = rows[hdr], rows[hdr + 1]
        col = {n: i for i, n in enumerate(names)}
        for r in rows[hdr + 2:]:
            if len(r) != len(names):
                continue
            kname = r[col["Kernel Name"]]
            seg = next((s for s, k in NCU_KERNELS.items() if k + "<" in kname or k + "(" in kname),
                       None)
            if seg is None or seg in kernels:
                continue
            d = {"kernel": kname.split("(")[0]}
            for m, key in NCU_METRICS.items():
                if m in col and r[col[m]] not in ("", "n/a"):
                    d[key] = float(r[col[m]].replace(",", "")) * UNIT_SCALE.get(units[col[m]], 1)
            if "dram_read_bytes" in d and "dram_write_bytes" in d:
                d["dram_bytes_per_launch"] = d["dram_read_bytes"] + d["dram_write_bytes"]
            kernels[seg] = d
    out = {"source_sha": kernel_source_sha(),
           "from": [os.path.basename(p) for p in csv_paths], "kernels": kernels}
    with open(out_path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    return out


def ncu_profile():
    """The committed ncu summary, if the kernel sources still match it."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("source_sha") != kernel_source_sha():
            return None
        return d["kernels"]
    except Exception:  # noqa: BLE001
        return None


# ---------------------------------------------------------------------------
# Multi-rank aggregation: every rank times its own steps; the job's time is
# the slowest rank's and its throughput counts the samples of all ranks.
def max_over_ranks(value, dist=None, device=None):
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, samples_per_rank_step, steps, job_ms):
    """Gsamples/s of the whole job: all ranks' samples over the slowest rank's time."""
    return world * samples_per_rank_step * steps / (job_ms * 1e-3) / 1e9


def run_ours(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    cpu_line = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu_line = cpu_baseline(args.cpu_sample_poses, args.cpu_min_seconds)

    import backprojection_tp_project_gather_b300 as tp

    seed = 1000 + WORKLOAD + 100 * rank           # rank 0 = the single-GPU workload
    w = synth.workload(WORKLOAD, seed=seed, poses=args.poses)
    P, N = w["P"], w["box"]
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])
    dev = torch.device("cuda", local)
    vol = torch.from_numpy(w["vol"]).to(dev)
    # Current estimates = the true poses perturbed (small rotation, ~1 px shift).
    rng = synth.streams(seed + 50, 3)
    R_true = torch.from_numpy(w["rot"]).to(dev)
    t_true = torch.from_numpy(w["shift"]).to(dev)
    axis = rng[0].standard_normal((P, 3))
    axis /= np.linalg.norm(axis, axis=1, keepdims=True)
    ang = np.deg2rad(2.0) * rng[0].standard_normal(P)
    K = np.zeros((P, 3, 3))
    K[:, 0, 1], K[:, 0, 2], K[:, 1, 2] = -axis[:, 2], axis[:, 1], -axis[:, 0]
    K = K - K.transpose(0, 2, 1)
    dR = (np.eye(3) + np.sin(ang)[:, None, None] * K
          + (1 - np.cos(ang))[:, None, None] * (K @ K))
    rot_a = torch.from_numpy((w["rot"][0].astype(np.float64) @ dR).astype(np.float32)[None]).to(dev)
    shift_a = (t_true + torch.from_numpy(rng[1].normal(0, 1, (1, P, 2)).astype(np.float32)).to(dev))
    # A second set of estimates (the first nudged by ~0.1 degree, ~0.05 px):
    # steps alternate between the two, so that every step brings new poses
    # (as the updated estimates of a refinement would) and the forward bins
    # them; the backward of the same step reuses that binning.
    eps = torch.from_numpy(0.002 * rng[1].standard_normal((1, P, 3, 3)).astype(np.float32)).to(dev)
    rot_b = rot_a + eps
    shift_b = shift_a + 0.05
    pose_sets = [(rot_a, shift_a), (rot_b, shift_b)]
    rot, shift = rot_a.clone(), shift_a.clone()
    # Targets: clean projections at the true poses plus noise of 10x the signal power.
    clean = tp.tp_project_3d_2d(vol, R_true, t_true, **kw)  # (workspace allocated per call here)
    noise = torch.from_numpy(synth.complex_normal((1, P, N, N // 2 + 1), rng[2])).to(dev)
    mask = torch.from_numpy(np.fft.fftfreq(N, 1.0 / N)[:, None] ** 2
                            + np.arange(N // 2 + 1)[None, :] ** 2 <= w["radius"] ** 2).to(dev)
    n_in = float(mask.sum())
    sig_pow = (clean.abs() ** 2 * mask).sum((2, 3), keepdim=True) / n_in
    target = (clean + noise * torch.sqrt(10.0 * sig_pow) * mask).contiguous()
    del clean, noise

    y = torch.empty_like(target)
    g = torch.empty_like(target)
    grad_vol = torch.zeros_like(vol)
    grad_rot = torch.zeros_like(rot)
    grad_shift = torch.zeros_like(shift)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ws = torch.zeros(tp.tp_workspace_bytes(1, 1, P, N, w["interp"]), dtype=torch.uint8, device=dev)
    kw["workspace"] = ws
    stream = torch.cuda.current_stream()


    # A step's inputs (volume, targets, poses) and results (gradients); the
    # device-resident timing uses set 0, the end-to-end pipeline both.
    bufs = [dict(vol=vol, target=target, rot=rot, shift=shift, grad_vol=grad_vol,
                 grad_rot=grad_rot, grad_shift=grad_shift)]

    def step(ev=None, i=0, b=None):
        if b is None:
            b = bufs[0]
            # This step's pose estimates (an 18 KB device copy, untimed).
            b["rot"].copy_(pose_sets[i & 1][0])
            b["shift"].copy_(pose_sets[i & 1][1])
        V, R, T = b["vol"], b["rot"], b["shift"]
        if ev:
            ev[0].record(stream)
        b["grad_vol"].zero_()
        b["grad_rot"].zero_()
        b["grad_shift"].zero_()
        if ev:
            ev[1].record(stream)
        # Forward with the L2 data term: y, g = 2 (y - target) and the rotation
        # and shift gradients from the forward's own derivative gather.
        tp.tp_project_3d_2d_l2(V, R, T, b["target"], out=y, grad_out=g, grad_rot=b["grad_rot"],
                               grad_shift=b["grad_shift"], **kw)
        if ev:
            ev[2].record(stream)
        # Volume gradient: the scatter of g (the binning of this step's poses kept).
        tp.tp_project_3d_2d_backward(g, V, R, T, grad_vol=b["grad_vol"], want_rot=False,
                                     want_shift=False, **kw)
        if ev:
            ev[3].record(stream)

    for i in range(args.warmup):
        flush.zero_()
        step(i=i)
    torch.cuda.synchronize()

    # The step's launches (zeroing, forward, volume gradient: all on the
    # device, the binning decisions included) are captured once as a CUDA
    # graph and replayed every timed step; the pose estimates are copied in
    # before each replay, untimed.  --eager times the launches one by one.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(b=bufs[0])
        torch.cuda.synchronize()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.zero_()                                            # L2 flush, untimed
            if graph is None:
                step(events[i], i=args.warmup + i)
            else:
                bufs[0]["rot"].copy_(pose_sets[(args.warmup + i) & 1][0])
                bufs[0]["shift"].copy_(pose_sets[(args.warmup + i) & 1][1])
                events[i][0].record(stream)
                graph.replay()
                events[i][3].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = np.array([events[i][0].elapsed_time(events[i][3]) for i in range(args.steps)])

    # Per step: zeroing of the gradients, the forward with the L2 term (output,
    # residual gradient, rotation and shift gradients), the volume gradient:
    # from launches one by one (a replayed graph has no events inside).
    nb = min(args.steps, 20)
    bevents = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb)]
    for i in range(nb):
        flush.zero_()
        step(bevents[i], i=args.warmup + args.steps + i)
    torch.cuda.synchronize()
    seg = np.array([[bevents[i][0].elapsed_time(bevents[i][1]),
                     bevents[i][1].elapsed_time(bevents[i][2]),
                     bevents[i][2].elapsed_time(bevents[i][3])] for i in range(nb)])
    total_ms = max_over_ranks(step_ms.sum(), dist, dev)
    samples = P * N * (N // 2 + 1)
    value = whole_job_rate(world, samples, args.steps, total_ms)

    # End to end through the public API with host buffers: every step copies
    # its inputs (volume, targets, poses) in from pinned host memory and its
    # gradients out.  The copies run on two copy streams, pipelined with the
    # compute of the neighbouring steps over two device buffer sets: step i's
    # inputs go up while step i-1 computes, its gradients come down while
    # step i+1 computes.
    h_vol = vol.cpu().pin_memory()
    h_poses = [(r.cpu().pin_memory(), t.cpu().pin_memory()) for r, t in pose_sets]
    h_target = target.cpu().pin_memory()
    bufs.append({k: torch.empty_like(t) for k, t in bufs[0].items()})
    outs = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory()
                  for t in (vol, rot, shift)) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_vol, h_poses[0][0], h_poses[0][1], h_target))
    d2h = sum(t.numel() * t.element_size() for t in outs[0])
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        b = bufs[i & 1]
        up.wait_event(comp_done[i & 1])        # step i-2 is done with these buffers
        with torch.cuda.stream(up):
            b["vol"].copy_(h_vol, non_blocking=True)
            b["rot"].copy_(h_poses[i & 1][0], non_blocking=True)
            b["shift"].copy_(h_poses[i & 1][1], non_blocking=True)
            b["target"].copy_(h_target, non_blocking=True)
        h2d_done[i & 1].record(up)

    def download(i):
        b, o = bufs[i & 1], outs[i & 1]
        down.wait_event(comp_done[i & 1])
        with torch.cuda.stream(down):
            o[0].copy_(b["grad_vol"], non_blocking=True)
            o[1].copy_(b["grad_rot"], non_blocking=True)
            o[2].copy_(b["grad_shift"], non_blocking=True)
        d2h_done[i & 1].record(down)

    def e2e_run(n, start):
        up.wait_event(start)
        upload(0)
        for i in range(n):
            stream.wait_event(h2d_done[i & 1])
            stream.wait_event(d2h_done[i & 1])   # step i-2's gradients have left
            step(b=bufs[i & 1])
            comp_done[i & 1].record(stream)
            if i + 1 < n:
                upload(i + 1)
            download(i)
        for k in range(min(n, 2)):
            stream.wait_event(d2h_done[k])

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(2, e0)                                # warm-up of the pipeline
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0.record(stream)
    e2e_run(args.e2e_steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = whole_job_rate(world, samples, args.e2e_steps, e2e_ms)

    # Secondary figures, timed the same way in the same run (rank 0, one GPU):
    # the 2D rotate + shift step and the 2048-image box-256 backprojection.
    secondary = None
    if rank == 0 and not args.no_secondary:
        secondary = {}
        r = rot2d_setup(tp, dev, stream, 20, 3)
        ms, _ = _timed(r["step"], 20, 3, stream, flush)
        secondary["rot2d_fwdbwd"] = {"workload": r["config"]["workload"],
                                     "ms": float(ms.mean()), "forward_ms": r["forward_ms"](),
                                     "gsamples_s": r["samples"] / (float(ms.mean()) * 1e-3) / 1e9}
        del r
        for interp in ("cubic", "linear"):
            r = backproject_setup(tp, dev, interp)
            ms, _ = _timed(r["step"], 5, 2, stream, flush)
            secondary[f"backproject_{interp}"] = {
                "workload": r["config"]["workload"], "ms": float(ms.mean()),
                "gsamples_s": r["samples"] / (float(ms.mean()) * 1e-3) / 1e9,
                "timed": "whole call (binning + kernels), data + weight spectra"}
            del r
        torch.cuda.empty_cache()

    if rank == 0:
        names = ["zero_gradients", "project_3d_2d_l2", "volume_grad_scatter"]
        mean_seg = seg.mean(0)
        n_in = P * in_radius_count(N, w["radius"])
        # Algorithmic HBM bytes per launch: the forward reads the volume once
        # and, per stored pixel, the target (8 B) and writes y and g (16 B);
        # the scatter reads g (8 B per stored pixel) and reads and writes the
        # volume gradient once.
        kern = {"project_3d_2d": (mean_seg[1], samples * 24 + vol.numel() * 8),
                "volume_grad_scatter": (mean_seg[2], samples * 8 + 2 * vol.numel() * 8)}
        dom = max(kern, key=lambda k: kern[k][0])
        t_ms, nbytes = kern[dom]
        peak, peak_src = measured_peak_hbm()
        achieved = nbytes / (t_ms * 1e-3) / 1e9
        prof = ncu_profile()
        traffic, sol = None, None
        if prof:
            traffic = prof.get(dom, {}).get("dram_bytes_per_launch")
            # Memory SOL % (max of DRAM, L2, L1 throughput) of the three
            # kernels, weighted by their share of the step.
            wsum = sum(kern[k][0] for k in kern if "mem_sol_pct" in prof.get(k, {}))
            if wsum > 0:
                sol = {"mem_sol_pct_time_weighted": sum(
                    kern[k][0] * prof[k]["mem_sol_pct"] for k in kern
                    if "mem_sol_pct" in prof.get(k, {})) / wsum,
                       "per_kernel": {k: {m: prof[k].get(m) for m in
                                          ("mem_sol_pct", "l1_pct", "l2_pct", "dram_pct")}
                                      for k in kern if k in prof},
                       "source": "profiles/ncu_traffic.json (ncu --set full, same sources)"}
        # The scatter's own bound is the shared-memory pipe: every in-radius
        # sample reads and writes its 64 tile words (8 B each) once; the pipe
        # moves 128 B per clock per SM.
        clk = clocks.record()
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        smem_bytes = n_in * 64 * 8 * 2
        smem_peak = sms * 128 * clk.get("sm_mhz", 2032.0) * 1e6 / 1e9
        smem_achieved = smem_bytes / (mean_seg[2] * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Gaussian-blob volume, uniform SO(3) poses, noisy targets)",
            "config": {**config_dict(w, P),
                       "launch": ("step launches one by one" if args.eager else
                                  "step captured once as a CUDA graph, replayed every step "
                                  "(breakdown_ms from launches one by one)")},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic,
                         "algorithmic_bytes_per_launch": nbytes},
            "roofline_shared": {"bound": "shared", "kernel": "volume_grad_scatter",
                                "achieved": smem_achieved, "peak": smem_peak, "unit": "GB/s",
                                "frac": smem_achieved / smem_peak,
                                "peak_source": f"{sms} SMs x 128 B/clk x median sampled SM clock "
                                               f"({clk.get('sm_mhz')} MHz)",
                                "algorithmic_bytes_per_launch": smem_bytes,
                                "per_unit": "64 taps x (8 B read + 8 B written) per in-radius "
                                            "sample"},
            "ncu_memory_sol": sol,
            "secondary": secondary,
            "breakdown_ms": {n: float(mean_seg[i]) for i, n in enumerate(names)},
            "fwd_gsamples_s": samples / (mean_seg[1] * 1e-3) / 1e9,
            "bwd_gsamples_s": samples / (mean_seg[2] * 1e-3) / 1e9,
            "in_radius_samples_per_step": n_in,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                    "copies": "every step: volume, targets, poses up; volume, rotation and shift "
                              "gradients down; pipelined with the neighbouring steps' compute "
                              "on two copy streams"},
            # per step: the forward with the L2 term (pose geometry, brick masks,
            # unit plan, gather with the zero fill as its prologue: 4) and the
            # volume-gradient call (geometry, masks, plan: 3; the sample lists
            # of this step's poses: begin, count, sums, items, fill: 5; the
            # scatter: 1), as the step's ncu launch list shows
            "gpu_launches": 13 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu_line,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Further workloads (one GPU; not the headline line): each prints one JSON
# line with CUDA-event timing of its step, inputs resident, L2 flushed.  The
# 2D step and the box-256 backprojection are also timed in the headline run,
# as its "secondary" figures.
def rot2d_setup(tp, dev, stream, steps, warmup):
    """The 2D rotate + shift step of 1024 images at box 128 (forward, then the image,
    rotation and shift gradients); forward_ms() gives the forward's mean time.  The
    forward and the backward (gradient zeroing and the backward call) are each
    captured once as a CUDA graph and replayed every step, so that the host's
    launch time does not stretch the step."""
    import torch
    w = synth.workload(2)
    N, n = w["box"], w["img"].shape[0]
    img = torch.from_numpy(w["img"]).to(dev)
    rot = torch.from_numpy(w["rot"]).to(dev)
    shift = torch.from_numpy(w["shift"]).to(dev)
    g = torch.from_numpy(w["grad"]).to(dev)
    out = torch.empty((n, 1, N, N // 2 + 1), dtype=torch.complex64, device=dev)
    gi, gr, gs = torch.zeros_like(img), torch.zeros_like(rot), torch.zeros_like(shift)
    kw = dict(interp=w["interp"], oversampling=1.0, radius=w["radius"])

    def forward():
        tp.tp_project_2d_2d(img, rot, shift, out=out, **kw)

    def backward():
        gi.zero_()
        gr.zero_()
        gs.zero_()
        tp.tp_project_2d_2d_backward(g, img, rot, shift, grad_img=gi, grad_rot=gr,
                                     grad_shift=gs, **kw)

    forward()
    backward()
    torch.cuda.synchronize()
    graphs = []
    for body in (forward, backward):
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            body()
        graphs.append(gph)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]

    def step(i):
        k = i - warmup
        if 0 <= k < steps:
            ev[k][0].record(stream)
        graphs[0].replay()
        if 0 <= k < steps:
            ev[k][1].record(stream)
        graphs[1].replay()

    samples = n * N * (N // 2 + 1)
    img_bytes = samples * 8
    return {"step": step, "samples": samples,
            "forward_ms": lambda: float(np.mean([a.elapsed_time(b) for a, b in ev])),
            # forward: image read, output written; backward: g and the image read,
            # the image gradient read and written
            "bytes": 2 * img_bytes + 2 * img_bytes + 2 * img_bytes,
            "config": {"workload": f"rot2d-{n}img-box{N}-{w['interp']}", "images": n, "box": N,
                       "interp": w["interp"], "radius": w["radius"], "shift_px": 5.0,
                       "l2_cache": "flushed between steps (256 MB write)",
                       "launch": "forward and backward each replayed as a CUDA graph"}}


def backproject_setup(tp, dev, interp, backward=False, images=None):
    """2048 noise images (box 256) backprojected into a data and a weight spectrum, or
    (backward) the gradients of that backprojection."""
    import torch
    w = synth.workload(4, poses=images)
    n, N = w["P"], w["box"]
    samples = n * N * (N // 2 + 1)
    proj = torch.from_numpy(w["proj"]).to(dev)
    # Two pose sets used in turn, so that every call bins its poses and sorts
    # its samples anew (a workspace keeps them only for unchanged poses).
    rots = [torch.from_numpy(w["rot"]).to(dev),
            torch.from_numpy(synth.random_rotations(n, synth.streams(7005, 1)[0])
                             .reshape(w["rot"].shape).astype(np.float32)).to(dev)]
    rot = rots[0]
    kw = dict(interp=interp, oversampling=1.0, radius=w["radius"])
    shape = (1, N, N, N // 2 + 1)
    ws = torch.zeros(tp.tp_workspace_bytes(1, 1, n, N, interp), dtype=torch.uint8, device=dev)
    vol_bytes = 8 * N * N * (N // 2 + 1)
    cfg = {"workload": f"backproject-box{N}-{n}img-{interp}", "box": N, "images": n,
           "interp": interp, "radius": w["radius"], "weights": "1 (default)",
           "poses": "two seeded pose sets in turn: every call bins its poses and sorts its "
                    "samples",
           "l2_cache": "flushed between steps (256 MB write)"}
    if not backward:
        data = torch.zeros(shape, dtype=torch.complex64, device=dev)
        wvol = torch.zeros(shape, dtype=torch.float32, device=dev)

        def step(i):
            tp.tp_backproject_2d_3d(proj, rots[i & 1], data_vol=data, weight_vol=wvol, workspace=ws,
                                    **kw)
        nbytes = samples * 8 + 2 * vol_bytes + 2 * vol_bytes // 2
        metric = "backprojected Fourier samples/sec (Gsamples/s), data + weight spectra"
    else:
        rng = synth.streams(7004, 1)[0]
        G = torch.from_numpy(synth.complex_normal(shape, rng)).to(dev)
        GW = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dev)
        gp = torch.empty_like(proj)
        gw = torch.empty(proj.shape, dtype=torch.float32, device=dev)
        gr = torch.zeros_like(rot)
        sc = torch.empty(tp.tp_backproject_backward_scratch_bytes(1, 1, n, N, N, True),
                         dtype=torch.uint8, device=dev)

        def step(i):
            gr.zero_()
            tp.tp_backproject_2d_3d_backward(G, proj, rots[i & 1], grad_weight_vol=GW, grad_proj=gp,
                                             grad_weights=gw, grad_rot=gr, scratch=sc,
                                             workspace=ws, **kw)
        # data: spectrum read, y and D written (32 B), images read with y and
        # D (40 B); weights: spectrum read and converted, y_W and D_W written,
        # read back with grad_weights written (4 B).
        nbytes = (vol_bytes + samples * 32 + samples * 40
                  + vol_bytes // 2 + vol_bytes + samples * 32 + samples * 36)
        metric = ("Fourier samples/sec (Gsamples/s) of the backprojection's gradients "
                  "(images, image weights, rotations)")
        cfg["upstream"] = "random data (complex) and weight (real) spectrum gradients"
    return {"step": step, "samples": samples, "bytes": nbytes, "metric": metric, "config": cfg}


def _timed(step, steps, warmup, stream, flush):
    import torch
    for i in range(warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clocks:
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(stream)
            step(warmup + i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    ms = np.array([a.elapsed_time(b) for a, b in ev])
    return ms, clocks.record()


def run_workload(args):
    import torch
    import backprojection_tp_project_gather_b300 as tp

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    peak, peak_src = measured_peak_hbm()
    line = {"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "ours", "workload": args.workload}

    if args.workload == "project":
        s = args.oversampling
        w = synth.workload(3, oversampling=s)
        N, P = w["box"], w["P"]
        samples = P * N * (N // 2 + 1)
        vol = torch.from_numpy(w["vol"]).to(dev)
        rot = torch.from_numpy(w["rot"]).to(dev)
        out = torch.empty((1, P, N, N // 2 + 1), dtype=torch.complex64, device=dev)
        kw = dict(N=N, interp=args.interp, oversampling=float(s), radius=w["radius"])
        ws = torch.zeros(tp.tp_workspace_bytes(1, 1, P, vol.shape[1], args.interp),
                         dtype=torch.uint8, device=dev)
        rots = [rot, rot + 1e-4]          # new poses every step: the binning re-runs

        def step(i):
            tp.tp_project_3d_2d(vol, rots[i & 1], out=out, workspace=ws, **kw)
        ms, clocks = _timed(step, args.steps, args.warmup, stream, flush)
        t = float(ms.mean())
        nbytes = samples * 8 + vol.numel() * 8
        line.update(metric="projected Fourier samples/sec (Gsamples/s)", unit="Gsamples/s",
                    value=samples / (t * 1e-3) / 1e9, ms_per_step=t, clocks=clocks,
                    config={"workload": f"project-box{N}-{P}poses-{args.interp}-s{s}", "box": N,
                            "volume_box": int(vol.shape[1]), "poses": P, "interp": args.interp,
                            "oversampling": s, "radius": w["radius"],
                            "l2_cache": "flushed between steps (256 MB write)"},
                    roofline={"bound": "hbm", "achieved": nbytes / (t * 1e-3) / 1e9, "peak": peak,
                              "peak_source": peak_src, "unit": "GB/s",
                              "frac": nbytes / (t * 1e-3) / 1e9 / peak, "traffic": None,
                              "algorithmic_bytes_per_step": nbytes,
                              "timed": "whole call (binning + kernels)"})
    elif args.workload == "rot2d":
        r = rot2d_setup(tp, dev, stream, args.steps, args.warmup)
        ms, clocks = _timed(r["step"], args.steps, args.warmup, stream, flush)
        fwd = r["forward_ms"]()
        t = float(ms.mean())
        nbytes = r["bytes"]
        line.update(metric="Fourier samples/sec (Gsamples/s) of the 2D rotate + shift, fwd + bwd",
                    unit="Gsamples/s", value=r["samples"] / (t * 1e-3) / 1e9, ms_per_step=t,
                    clocks=clocks, breakdown_ms={"forward": fwd, "backward": t - fwd},
                    config=r["config"],
                    roofline={"bound": "hbm", "achieved": nbytes / (t * 1e-3) / 1e9, "peak": peak,
                              "peak_source": peak_src, "unit": "GB/s",
                              "frac": nbytes / (t * 1e-3) / 1e9 / peak, "traffic": None,
                              "algorithmic_bytes_per_step": nbytes,
                              "timed": "forward + backward calls"})
    elif args.workload in ("backproject", "backproject-backward"):
        r = backproject_setup(tp, dev, args.interp, args.workload == "backproject-backward",
                              args.poses)
        ms, clocks = _timed(r["step"], args.steps, args.warmup, stream, flush)
        t = float(ms.mean())
        nbytes = r["bytes"]
        line.update(metric=r["metric"], unit="Gsamples/s", value=r["samples"] / (t * 1e-3) / 1e9,
                    ms_per_step=t, config=r["config"], clocks=clocks,
                    roofline={"bound": "hbm", "achieved": nbytes / (t * 1e-3) / 1e9, "peak": peak,
                              "peak_source": peak_src, "unit": "GB/s",
                              "frac": nbytes / (t * 1e-3) / 1e9 / peak, "traffic": None,
                              "algorithmic_bytes_per_step": nbytes,
                              "timed": "whole call (binning + kernels)"})
    elif args.workload == "hostlink":
        # The copies of the end-to-end step (203 MB up, 68 MB down) at the
        # link's own rates: one direction at a time, then both at once on two
        # streams, as the pipelined step issues them.
        up_b, down_b = 202921984, 67655680
        h_up = torch.empty(up_b, dtype=torch.uint8).pin_memory()
        d_up = torch.empty(up_b, dtype=torch.uint8, device=dev)
        h_dn = torch.empty(down_b, dtype=torch.uint8).pin_memory()
        d_dn = torch.empty(down_b, dtype=torch.uint8, device=dev)
        s_up, s_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def h2d(i):
            d_up.copy_(h_up, non_blocking=True)

        def d2h(i):
            h_dn.copy_(d_dn, non_blocking=True)

        def both(i):
            cur = torch.cuda.current_stream()
            s_up.wait_stream(cur)
            s_dn.wait_stream(cur)
            with torch.cuda.stream(s_up):
                d_up.copy_(h_up, non_blocking=True)
            with torch.cuda.stream(s_dn):
                h_dn.copy_(d_dn, non_blocking=True)
            cur.wait_stream(s_up)
            cur.wait_stream(s_dn)
        res = {}
        for name, fn, nbytes in (("h2d", h2d, up_b), ("d2h", d2h, down_b),
                                 ("both", both, up_b + down_b)):
            ms, clocks = _timed(fn, args.steps, args.warmup, stream, flush)
            t = float(ms.mean())
            res[name] = {"ms": t, "GB_s": nbytes / (t * 1e-3) / 1e9}
        fwd_bwd_samples = 512 * 256 * 129
        line.update(metric="pinned host <-> device copy time of one end-to-end step's bytes",
                    unit="ms", value=res["both"]["ms"], higher_is_better=False,
                    ms_per_step=res["both"]["ms"], results=res, clocks=clocks,
                    config={"workload": "hostlink-203MB-up-68MB-down",
                            "e2e_bound_gsamples_s": fwd_bwd_samples / (res["both"]["ms"] * 1e-3)
                            / 1e9})
    elif args.workload == "oversampling":
        c = synth.CONFIGS[3]
        M, P = c["box"], c["poses"]
        r_vol, r_rot = synth.streams(1003, 5)[:2]
        cen, sig, amp = synth.blob_params(M, c["blobs"], r_vol, 3)
        dens = torch.from_numpy(synth.blob_density(M, cen, sig, amp, 3).astype(np.float32)).to(dev)
        rot = torch.from_numpy(synth.random_rotations(P, r_rot)[None]).to(dev)
        radius = c["radius"]
        out = torch.empty((1, P, M, M // 2 + 1), dtype=torch.complex64, device=dev)
        ws1 = torch.zeros(tp.tp_workspace_bytes(1, 1, P, M, "cubic"), dtype=torch.uint8, device=dev)
        ws2 = torch.zeros(tp.tp_workspace_bytes(1, 1, P, 2 * M, "linear"), dtype=torch.uint8,
                          device=dev)
        big = torch.zeros((2 * M,) * 3, dtype=torch.float32, device=dev)
        o = M // 2

        def spec(d):
            return torch.fft.rfftn(torch.fft.ifftshift(d)).unsqueeze(0).contiguous()

        def cubic1(i):
            tp.tp_project_3d_2d(spec(dens), rot, out=out, interp="cubic", radius=radius,
                                workspace=ws1)

        def linear2(i):
            big[o:o + M, o:o + M, o:o + M] = dens
            tp.tp_project_3d_2d(spec(big), rot, N=M, out=out, interp="linear", oversampling=2.0,
                                radius=radius, workspace=ws2)

        def cubic2(i):
            big[o:o + M, o:o + M, o:o + M] = dens
            tp.tp_project_3d_2d(spec(big), rot, N=M, out=out, interp="cubic", oversampling=2.0,
                                radius=radius, workspace=ws2)
        res = {}
        for name, fn in (("cubic_s1", cubic1), ("linear_s2", linear2), ("cubic_s2", cubic2)):
            ms, clocks = _timed(fn, args.steps, args.warmup, stream, flush)
            res[name] = {"ms": float(ms.mean())}
        # Accuracy against the exact transform of the density at the sample
        # positions p = R^T k (box-M units), on the first Q poses: separable
        # sums over x, y, z as batched complex products in float64.
        Q = 16
        ky = torch.fft.fftfreq(M, 1.0 / M, device=dev, dtype=torch.float64)
        kx = torch.arange(M // 2 + 1, device=dev, dtype=torch.float64)
        KY, KX = torch.meshgrid(ky, kx, indexing="ij")
        inside = (KX * KX + KY * KY <= radius * radius)
        x = torch.arange(M, device=dev, dtype=torch.float64) - M // 2
        d64 = dens.double().to(torch.complex128)
        exact = torch.zeros((Q, M, M // 2 + 1), dtype=torch.complex128, device=dev)
        R64 = rot[0, :Q].double()
        for q in range(Q):
            p = (R64[q, 0][:, None, None] * KX + R64[q, 1][:, None, None] * KY)   # (3, M, X)
            pk = p.reshape(3, -1)                                                 # (3, S)
            ex = torch.exp(-2j * np.pi * pk[0][:, None] * x[None, :] / M)        # (S, M)
            ey = torch.exp(-2j * np.pi * pk[1][:, None] * x[None, :] / M)
            ez = torch.exp(-2j * np.pi * pk[2][:, None] * x[None, :] / M)
            vals = torch.empty(pk.shape[1], dtype=torch.complex128, device=dev)
            for a in range(0, pk.shape[1], 1024):
                sl = slice(a, a + 1024)
                t1 = torch.einsum("zyx,sx->szy", d64, ex[sl])
                t2 = torch.einsum("szy,sy->sz", t1, ey[sl])
                vals[sl] = torch.einsum("sz,sz->s", t2, ez[sl])
            exact[q] = vals.reshape(M, M // 2 + 1) * inside
        # Fourier shells of 1 pixel (|k| rounded) and real-space rings of 2 pixels
        # about the image centre.
        shell = torch.round(torch.sqrt(KX * KX + KY * KY)).long()
        nshell = int(radius) + 1
        cc = torch.arange(M, device=dev, dtype=torch.float64) - M // 2
        ring = (torch.sqrt(cc[:, None] ** 2 + cc[None, :] ** 2) / 2).long()
        nring = M // 4 + 1                                  # out to half the box
        ex_img = torch.fft.fftshift(torch.fft.irfft2(exact, s=(M, M)), dim=(-2, -1))
        ex_pow = torch.zeros(nring, dtype=torch.float64, device=dev).index_add_(
            0, ring.flatten().clamp(max=nring - 1).repeat(Q), (ex_img ** 2).flatten())
        for name, fn in (("cubic_s1", cubic1), ("linear_s2", linear2), ("cubic_s2", cubic2)):
            fn(0)
            torch.cuda.synchronize()
            got = out[0, :Q].to(torch.complex128) * inside
            res[name]["rel_l2_vs_exact"] = float(torch.linalg.vector_norm(got - exact)
                                                 / torch.linalg.vector_norm(exact))
            # Relative error per shell, over the Q poses.
            e2 = torch.zeros(nshell, dtype=torch.float64, device=dev).index_add_(
                0, shell[inside].repeat(Q), (torch.abs(got - exact)[:, inside] ** 2).flatten())
            n2 = torch.zeros(nshell, dtype=torch.float64, device=dev).index_add_(
                0, shell[inside].repeat(Q), (torch.abs(exact)[:, inside] ** 2).flatten())
            curve = torch.sqrt(e2 / n2.clamp(min=1e-300)).cpu().numpy()
            res[name]["shell_rel_error"] = [round(float(c), 6) for c in curve]
            over = np.nonzero(curve > 0.1)[0]
            res[name]["first_shell_over_10pct"] = int(over[0]) if len(over) else None
            # Real-space intensity relative to the exact projection, ring by ring:
            # sum(img * exact) / sum(exact^2) (1 = no falloff).
            img = torch.fft.fftshift(torch.fft.irfft2(got, s=(M, M)), dim=(-2, -1))
            cross = torch.zeros(nring, dtype=torch.float64, device=dev).index_add_(
                0, ring.flatten().clamp(max=nring - 1).repeat(Q), (img * ex_img).flatten())
            res[name]["realspace_gain_per_2px_ring"] = [
                round(float(a / b), 5) if b > 1e-6 * float(ex_pow.max()) else None
                for a, b in zip(cross.cpu().numpy(), ex_pow.cpu().numpy())]
        samples = P * M * (M // 2 + 1)
        line.update(metric="box-128 forward incl. rfftn (and the 2x padding for s = 2): ms per "
                           "4096 poses and rel. L2 error vs the exact transform",
                    unit="ms", value=res["cubic_s1"]["ms"], higher_is_better=False,
                    ms_per_step=res["cubic_s1"]["ms"], results=res, clocks=clocks,
                    config={"workload": "oversampling-study-box128-4096poses",
                            "radius": radius, "exact_subset": f"first {Q} poses, in-radius pixels",
                            "shells": "1-pixel |k| shells (rounded), rel. error over the subset",
                            "realspace": "irfft2 of each projection vs the exact one, fftshifted, "
                                         "2-pixel rings about the centre out to half the box",
                            "samples_per_step": samples,
                            "fft": "torch.fft.rfftn (cuFFT) inside the timed region"})
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.ncu_summary:
        out = ncu_summary(args.ncu_summary, os.path.join(ROOT, "profiles", "ncu_traffic.json"))
        print(json.dumps(out, indent=1))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "fwdbwd":
        return run_workload(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
