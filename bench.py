#!/usr/bin/env python3
"""Throughput of the fused SSIM loss: fp32 forward + backward, megapixels/s.

Workload: the 1080p splatting-render pair, 1 x 3 x 1080 x 1920 float32,
padding "valid", gradient for img1 only (TriSSIM README, "Performance": 1080p,
fp32, valid, forward + backward).  A step is one ssim_fwd (training mode, the
gradient fields saved) plus one ssim_bwd, back to back on one stream, through
the C ABI.  MP = N*H*W / 1e6 input pixels per step (channels not counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  With N > 1 (torchrun, one process per GPU) every rank
processes its own image -- the batch is sharded, there is no data exchange --
and the time is the maximum over ranks ("scaling": "weak").

--impl reference times the CPU oracle (test infrastructure: the plain
double-precision statement of the loss) on the host cores, each step a bounded
band of rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "splat1080_valid"
METRIC = "fp32 SSIM fwd+bwd megapixels/s at 1080p valid; % of HBM roofline"
UNIT = "MP/s"
NOMINAL_HBM_GBS = 8000.0
FLUSH_BYTES = 256 << 20
KERNEL_NAME = "ssim2d_stream_kernel<true,false>"
PROFILE = os.path.join(ROOT, "profiles", "ssim2d_grad_splat1080_valid.md")
PROFILE3D = os.path.join(ROOT, "profiles", "ssim3d_volume128_valid.md")

# Algorithmic float32 operations of the gradient-mode kernel per input pixel
# (fused forward statistics, SSIM derivatives, adjoint and chain rule), counting
# an FMA as 2 flops: an 11-tap row pass and column pass of the four shifted
# statistics (44 + 44 FMA) and of the three adjoint maps (33 + 33 FMA), plus
# the shifted products (5), SSIM and its derivatives (30) and the chain rule (3).
GRAD_FMA_PER_PIXEL = 44 + 44 + 33 + 33  # row + column passes of 4 statistics, of 3 adjoint maps
GRAD_OTHER_PER_PIXEL = 5 + 30 + 3       # shifted products, SSIM and derivatives, chain rule
GRAD_FLOPS_PER_PIXEL = 2 * GRAD_FMA_PER_PIXEL + GRAD_OTHER_PER_PIXEL
# 3D (the three kernels of the training forward together): three 11-tap passes of four
# statistics and of three adjoint maps, plus the same per-voxel work.
GRAD3D_FLOPS_PER_VOXEL = 2 * (3 * 44 + 3 * 33) + GRAD_OTHER_PER_PIXEL
KERNEL3D_NAME = "ssim3d_xy_kernel + ssim3d_z_kernel<true,false> + ssim3d_adjoint_kernel<false>"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the extra timed variants")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name from workloads.WORKLOADS (default: the 1080p valid pair)")
    ap.add_argument("--path", choices=["train", "infer", "pyramid"], default="train",
                    help="the call a step times: train (training forward + stored backward, the "
                         "metric), infer (forward only) or pyramid (the six-octave per-octave "
                         "stage, 2D only); the last two print a short line (for profiling)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0}, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms meanwhile."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # "under load": samples drawing more than 200 W; if none did (a short
        # run between samples), the figures are over all samples, and say so
        loaded = [r for r in rows if r[2] > 200.0]
        basis = loaded or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in basis for i, v in enumerate(r[3][1:])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in basis),
                "sm_max_mhz": max(r[1] for r in basis),
                "power_w_max": max(r[2] for r in rows),
                "samples": len(rows), "samples_under_load": len(loaded),
                "sm_mhz_basis": "samples above 200 W" if loaded else
                                "all samples (none above 200 W)",
                "reasons": reasons}


# ------------------------------------------------------------------ oracle (CPU)

def oracle_band(name: str, n_rows: int):
    """(x, y, dl) for the first n_rows rows (2D) or slices (3D) of the workload
    pair: a bounded sample of it."""
    from workloads import dl_vector, make_inputs

    x, y = make_inputs(name)
    n_rows = max(11, min(n_rows, x.shape[2]))
    return (x[:, :, :n_rows].copy(), y[:, :, :n_rows].copy(), dl_vector(name))


def time_oracle_step(oracle, x, y, dl, padding="valid", want_grad2=False):
    t0 = time.perf_counter()
    if x.ndim == 5:
        oracle.ssim3d(x, y, padding)
        oracle.ssim3d_grad(x, y, dl, padding, want_grad2=want_grad2)
    else:
        oracle.ssim2d(x, y, padding)
        oracle.ssim2d_grad(x, y, dl, padding, want_grad2=want_grad2)
    return time.perf_counter() - t0


def size_oracle_band(oracle, name, target_s: float):
    """Rows (slices) of the workload whose oracle step takes about target_s seconds."""
    from workloads import WORKLOADS

    wl = WORKLOADS[name]
    full = wl.shape[2]
    rows = 32 if wl.ndim == 2 else 12
    x, y, dl = oracle_band(name, rows)
    t = time_oracle_step(oracle, x, y, dl, wl.padding, wl.want_grad2)
    while t < target_s / 2 and rows < full:
        rows = min(full, int(rows * min(8.0, max(2.0, target_s / max(t, 1e-3)))))
        x, y, dl = oracle_band(name, rows)
        t = time_oracle_step(oracle, x, y, dl, wl.padding, wl.want_grad2)
    return rows, (x, y, dl), t


def units(shape):
    """Megapixels (megavoxels) per step: N times the spatial extent, channels not counted."""
    n = shape[0]
    for s in shape[2:]:
        n *= s
    return n / 1e6


def cpu_baseline(name: str, unit: str, target_s: float = 4.0):
    import oracle
    from workloads import WORKLOADS

    wl = WORKLOADS[name]
    oracle.build()
    rows, (x, y, dl), _ = size_oracle_band(oracle, name, target_s)
    times = [time_oracle_step(oracle, x, y, dl, wl.padding, wl.want_grad2) for _ in range(3)]
    t = statistics.median(times)
    cores = oracle.num_threads()
    # the same on one thread, on a band of about a second
    rows1 = max(11, int(rows * min(1.0, 1.0 / max(t * cores, 1e-6))))
    x1, y1, dl1 = oracle_band(name, rows1)
    oracle.set_num_threads(1)
    try:
        t1 = time_oracle_step(oracle, x1, y1, dl1, wl.padding, wl.want_grad2)
    finally:
        oracle.set_num_threads(cores)
    what = "rows" if wl.ndim == 2 else "slices"
    return {"value": units(x.shape) / t, "unit": unit, "cores": cores,
            "kind": "oracle",
            "sample": f"{what} 0..{rows} of the {'x'.join(map(str, wl.shape))} pair ({wl.padding}), "
                      f"mean + gradients, median of 3 ({t:.2f} s each)",
            "value_1_thread": units(x1.shape) / t1,
            "sample_1_thread": f"{what} 0..{x1.shape[2]}, one run ({t1:.2f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from workloads import WORKLOADS

    wl = WORKLOADS[args.workload]
    unit = UNIT if wl.ndim == 2 else "Mvoxel/s"
    oracle.build()
    budget = 150.0  # seconds for the whole run
    per_step = max(0.5, min(5.0, budget / max(1, args.steps + args.warmup)))
    rows, (x, y, dl), _ = size_oracle_band(oracle, args.workload, per_step)
    for _ in range(args.warmup):
        time_oracle_step(oracle, x, y, dl, wl.padding, wl.want_grad2)
    times = [time_oracle_step(oracle, x, y, dl, wl.padding, wl.want_grad2)
             for _ in range(args.steps)]
    mp = units(x.shape)
    total = sum(times)
    value = mp * len(times) / total
    what = "rows" if wl.ndim == 2 else "slices"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "shape": list(wl.shape), "padding": wl.padding,
                   "grads": "img1, img2" if wl.want_grad2 else "img1", "sample_" + what: rows},
        "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{what} 0..{rows} of the {'x'.join(map(str, wl.shape))} "
                                   f"pair per step"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, steps: int, max_ms: float) -> float:
    """Units processed by all ranks per second, over the slowest rank's time."""
    return world * units_per_rank * steps / (max_ms / 1e3)


# The sources that build the kernels a profile summary covers: its traffic
# figure stands while these are unchanged.
PROFILE_SOURCES = {
    PROFILE: ("common.cuh", "ssim2d.cuh", "ssim2d.cu"),
    PROFILE3D: ("common.cuh", "ssim2d.cuh", "ssim3d.cuh", "ssim3d.cu"),
}


def kernel_source_digest(names):
    """Digest of the named sources with their comments and blank lines taken
    out (a comment cannot change a kernel's traffic)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "differentiable_image_quality_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        code = [ln.split("//", 1)[0].rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


def profiled_traffic(path=PROFILE):
    """DRAM bytes per launch of the profiled kernel(s) from a committed ncu
    summary, if it was taken from the current sources of those kernels; else
    None."""
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_digest(PROFILE_SOURCES[path]):
        return None
    return float(m.group(1))


def workload_setup(pkg, torch, dev, name):
    """Device inputs and outputs of one workload, and its per-step call closures."""
    from workloads import WORKLOADS, dl_vector, make_inputs

    wl = WORKLOADS[name]
    is3d = wl.ndim == 3
    x, y = make_inputs(name)
    dl = dl_vector(name)
    N = x.shape[0]
    g2wanted = wl.want_grad2
    fwd_call = pkg.ssim3d_fwd if is3d else pkg.ssim_fwd
    bwd_call = pkg.ssim3d_bwd if is3d else pkg.ssim_bwd
    fused_call = pkg.ssim3d_fwd_bwd if is3d else pkg.ssim_fwd_bwd
    tx, ty = torch.from_numpy(x).to(dev), torch.from_numpy(y).to(dev)
    tdl = torch.from_numpy(dl).to(dev)
    mean = torch.empty(N, device=dev)
    saved = torch.empty(pkg.saved_bytes(x.shape, g2wanted) // 4, device=dev)
    g1 = torch.empty_like(tx)
    g2 = torch.empty_like(ty) if g2wanted else None
    w = {"wl": wl, "x": x, "y": y, "tx": tx, "ty": ty, "tdl": tdl, "mean": mean, "saved": saved,
         "g1": g1, "g2": g2, "fwd": fwd_call, "bwd": bwd_call, "is3d": is3d,
         "mp": units(x.shape), "elems": x.size}
    w["fwd_train"] = lambda: fwd_call(tx, ty, wl.padding, mean, saved=saved, want_grad2=g2wanted)
    w["bwd_saved"] = lambda: bwd_call(tdl, tx, ty, wl.padding, g1, g2, saved=saved)
    w["fwd_infer"] = lambda: fwd_call(tx, ty, wl.padding, mean)
    w["bwd_recompute"] = lambda: bwd_call(tdl, tx, ty, wl.padding, g1, g2)
    w["single_call"] = lambda: fused_call(tx, ty, wl.padding, tdl, mean, g1, g2)
    return w


def make_timer(torch, dev, world, flush):
    import torch.distributed as dist

    stream = torch.cuda.current_stream(dev)

    def timed(fn_a, fn_b, steps, warmup):
        """Per-step device times of fn_a then fn_b, L2 flushed before each step."""
        for _ in range(warmup):
            flush.zero_()
            fn_a()
            if fn_b:
                fn_b()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for e in ev:
            flush.zero_()
            e[0].record(stream)
            fn_a()
            e[1].record(stream)
            if fn_b:
                fn_b()
            e[2].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        ta = [e[0].elapsed_time(e[1]) for e in ev]
        tb = [e[1].elapsed_time(e[2]) for e in ev]
        return ta, tb

    return timed


def roofline_figures(w, step_ms, fwd_ms, peaks, alu_peak_tflops):
    """Minimal HBM bytes of a forward + backward step and its fraction of the
    measured copy peak; the training forward's flops and its fraction of the
    fp32 ALU peak."""
    elems = w["elems"]
    grads = 2 if w["wl"].want_grad2 else 1
    min_bytes = (2 * elems + 2 * elems + grads * elems) * 4  # fwd: read 2; bwd: read 2, write grads
    flops_px = GRAD3D_FLOPS_PER_VOXEL if w["is3d"] else GRAD_FLOPS_PER_PIXEL
    achieved_tflops = flops_px * elems / (fwd_ms / 1e3) / 1e12
    hbm_gbs = min_bytes / (step_ms / 1e3) / 1e9
    return {"min_bytes": min_bytes, "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peaks["hbm_gbs"],
            "flops_px": flops_px, "tflops": achieved_tflops,
            "alu_frac": achieved_tflops / alu_peak_tflops}


def workload_summary(w, timed, steps, peaks, alu_peak_tflops):
    """The step and its parts on one workload (fewer steps than the headline)."""
    step_ms, _ = timed(lambda: (w["fwd_train"](), w["bwd_saved"]()), None, steps, 3)
    ta, tb = timed(w["fwd_train"], w["bwd_saved"], steps, 3)
    ra, rb = timed(w["fwd_infer"], w["bwd_recompute"], steps, 3)
    sa, _ = timed(w["single_call"], None, steps, 3)
    mp = w["mp"]
    st, fw = statistics.mean(step_ms), statistics.mean(ta)
    rf = roofline_figures(w, st, fw, peaks, alu_peak_tflops)
    return {"shape": list(w["x"].shape), "padding": w["wl"].padding,
            "grads": "img1, img2" if w["wl"].want_grad2 else "img1",
            "fwd_bwd_mps": mp / (st / 1e3), "us_per_step": 1e3 * st,
            "fwd_mps": mp / (fw / 1e3), "bwd_mps": mp / (statistics.mean(tb) / 1e3),
            "fwd_infer_mps": mp / (statistics.mean(ra) / 1e3),
            "bwd_recompute_mps": mp / (statistics.mean(rb) / 1e3),
            "single_call_fwd_bwd_mps": mp / (statistics.mean(sa) / 1e3),
            "hbm_frac": rf["hbm_frac"], "alu_frac": rf["alu_frac"], "steps": steps}


def run_path(args, pkg, torch, dev, w, timed, world, rank):
    """One call timed on its own (forward only, or the per-octave stage)."""
    x, wl, mp = w["x"], w["wl"], w["mp"]
    if args.path == "infer":
        fn, what = w["fwd_infer"], "forward only (inference), mean of each image"
    else:
        if w["is3d"]:
            raise SystemExit("--path pyramid needs a 2D workload")
        octs = 6
        means = torch.empty((octs, 3, x.shape[0]), device=dev)
        tx, ty = w["tx"], w["ty"]

        def fn():
            pkg.ssim_pyramid(tx, ty, wl.padding, octs, out_means=means)

        what = f"per-octave stage, {octs} octaves (l, cs, S means)"
    ts, _ = timed(fn, None, args.steps, max(3, args.warmup))
    total_ms = max_over_ranks(sum(ts), world, dev)
    if rank == 0:
        unit = UNIT if not w["is3d"] else "Mvoxel/s"
        print(json.dumps({"metric": f"fp32 SSIM {what}, {unit}", "path": args.path,
                          "value": whole_job_rate(mp, world, args.steps, total_ms), "unit": unit,
                          "n_gpus": world, "steps": args.steps, "ms_per_step": total_ms / args.steps,
                          "higher_is_better": True,
                          "config": {"workload": args.workload, "shape": list(x.shape),
                                     "padding": wl.padding}}), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_ours(args):
    import torch
    import torch.distributed as dist

    import differentiable_image_quality_gb300 as pkg
    from workloads import WORKLOADS

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkg._abi.load()
    name = args.workload
    w = workload_setup(pkg, torch, dev, name)
    wl, x, is3d, mp, elems = w["wl"], w["x"], w["is3d"], w["mp"], w["elems"]
    unit = UNIT if not is3d else "Mvoxel/s"
    N = x.shape[0]
    g2wanted = wl.want_grad2
    fwd_call, bwd_call = w["fwd"], w["bwd"]
    mean, saved, g1, g2, tdl = w["mean"], w["saved"], w["g1"], w["g2"], w["tdl"]
    flush = torch.empty(FLUSH_BYTES // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    timed = make_timer(torch, dev, world, flush)

    def train_step():
        w["fwd_train"]()
        w["bwd_saved"]()

    if args.path != "train":
        return run_path(args, pkg, torch, dev, w, timed, world, rank)

    # the step as a whole (no event between forward and backward, so the
    # backward's launch may overlap the forward's tail), then the two halves
    with ClockSampler(local) as clocks:
        step_ms, _ = timed(train_step, None, args.steps, max(3, args.warmup))
    clk = clocks.summary()
    ta, tb = timed(w["fwd_train"], w["bwd_saved"], args.steps, 3)

    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = whole_job_rate(mp, world, args.steps, total_ms)
    fwd_ms = statistics.mean(ta)
    bwd_ms = statistics.mean(tb)

    # ---- end to end through the public API with host buffers (pinned).  Every
    # step copies its two input images host -> device and reads its loss (the
    # per-image means) back; two input buffers let the copy of step k + 1 run
    # on a copy stream while step k computes.  The serial form, which also
    # reads the gradients back, is reported beside it.
    # the pair as one pinned host buffer and one device buffer per slot: one
    # copy per step (img1 and img2 are its two halves)
    hxy = torch.empty((2,) + tuple(x.shape), dtype=torch.float32).pin_memory()
    hxy[0].copy_(torch.from_numpy(x))
    hxy[1].copy_(torch.from_numpy(w["y"]))
    hg1 = torch.empty(x.shape, dtype=torch.float32).pin_memory()
    hg2 = torch.empty(x.shape, dtype=torch.float32).pin_memory() if g2wanted else None
    hm = torch.empty(N, dtype=torch.float32).pin_memory()
    dxy = [torch.empty((2,) + tuple(x.shape), dtype=torch.float32, device=dev) for _ in range(2)]
    dbuf = [(d[0], d[1]) for d in dxy]
    copy_stream = torch.cuda.Stream(dev)
    hloss = torch.empty((args.steps + max(3, args.warmup), N), dtype=torch.float32).pin_memory()

    def e2e_pipelined(steps, warmup):
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        losses = [hloss[k] for k in range(warmup + steps)]
        on_copy = torch.cuda.stream(copy_stream)
        for k in range(warmup + steps):
            b = k % 2
            dx, dy = dbuf[b]
            if k == warmup:
                t0.record(copy_stream)
            with on_copy:
                if used[b]:
                    copy_stream.wait_event(freed[b])
                dxy[b].copy_(hxy, non_blocking=True)
                copied[b].record(copy_stream)
            stream.wait_event(copied[b])
            fwd_call(dx, dy, wl.padding, mean, saved=saved, want_grad2=g2wanted)
            bwd_call(tdl, dx, dy, wl.padding, g1, g2, saved=saved)
            losses[k].copy_(mean, non_blocking=True)
            freed[b].record(stream)
            used[b] = True
        t1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        return t0.elapsed_time(t1)

    e2e_ms = max_over_ranks(e2e_pipelined(args.steps, max(3, args.warmup)), world, dev)
    e2e_value = whole_job_rate(mp, world, args.steps, e2e_ms)

    def e2e_serial_step():
        dx, dy = dbuf[0]
        dxy[0].copy_(hxy, non_blocking=True)
        fwd_call(dx, dy, wl.padding, mean, saved=saved, want_grad2=g2wanted)
        bwd_call(tdl, dx, dy, wl.padding, g1, g2, saved=saved)
        hg1.copy_(g1, non_blocking=True)
        if g2wanted:
            hg2.copy_(g2, non_blocking=True)
        hm.copy_(mean, non_blocking=True)

    ts_, _ = timed(e2e_serial_step, None, args.steps, max(3, args.warmup))
    e2e_serial_value = whole_job_rate(mp, world, args.steps, max_over_ranks(sum(ts_), world, dev))

    peaks, peak_kind = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sm_count = props.multi_processor_count
    sm_max = float(clk.get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0))
    alu_peak_tflops = sm_count * 128 * 2 * sm_max * 1e6 / 1e12

    extras = {}
    workloads = {}
    if not args.no_extras:
        ra, rb = timed(w["fwd_infer"], w["bwd_recompute"], args.steps, 3)
        sa, _ = timed(w["single_call"], None, args.steps, 3)
        pyr = {}
        if not is3d:
            # the per-octave stage: l, cs and S means of every octave (maps not written)
            H, W = x.shape[2], x.shape[3]
            octs = 0
            while octs < 6 and min(pkg.pyramid_extents(H, W, octs + 1)[-1]) >= (
                    11 if wl.padding == "valid" else 1):
                octs += 1
            pyr_means = torch.empty((octs, 3, N), device=dev)
            tx, ty = w["tx"], w["ty"]

            def pyramid():
                pkg.ssim_pyramid(tx, ty, wl.padding, octs, out_means=pyr_means)

            pa, _ = timed(pyramid, None, args.steps, 3)
            pyr = {"pyramid_octaves": octs, "pyramid_mps": mp / (statistics.mean(pa) / 1e3),
                   "pyramid_us": 1e3 * statistics.mean(pa)}
        extras = {
            "fwd_train_mps": mp / (fwd_ms / 1e3),
            "bwd_saved_mps": mp / (bwd_ms / 1e3),
            "fwd_infer_mps": mp / (statistics.mean(ra) / 1e3),
            "bwd_recompute_mps": mp / (statistics.mean(rb) / 1e3),
            "recompute_path_fwd_bwd_mps": mp / ((statistics.mean(ra) + statistics.mean(rb)) / 1e3),
            "single_call_fwd_bwd_mps": mp / (statistics.mean(sa) / 1e3),
            **pyr,
        }
        # every other workload of the suite, fewer steps each (rank 0's GPU only
        # matters for the line; every rank runs them so that collectives stay matched)
        for other in WORKLOADS:
            if other == name:
                continue
            wo = workload_setup(pkg, torch, dev, other)
            workloads[other] = workload_summary(wo, timed, max(10, min(args.steps, 50)), peaks,
                                                alu_peak_tflops)
            del wo
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    step_mean = statistics.mean(step_ms)
    rf = roofline_figures(w, step_mean, fwd_ms, peaks, alu_peak_tflops)
    workloads[name] = {
        "shape": list(x.shape), "padding": wl.padding,
        "grads": "img1, img2" if g2wanted else "img1",
        "fwd_bwd_mps": mp / (step_mean / 1e3), "us_per_step": 1e3 * step_mean,
        "fwd_mps": mp / (fwd_ms / 1e3), "bwd_mps": mp / (bwd_ms / 1e3),
        **({"fwd_infer_mps": extras["fwd_infer_mps"],
            "bwd_recompute_mps": extras["bwd_recompute_mps"],
            "single_call_fwd_bwd_mps": extras["single_call_fwd_bwd_mps"]} if extras else {}),
        "hbm_frac": rf["hbm_frac"], "alu_frac": rf["alu_frac"], "steps": args.steps}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, unit)

    traffic = (profiled_traffic() if name == WORKLOAD else
               profiled_traffic(PROFILE3D) if name == "volume128_valid" else None)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": step_mean, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "shape": list(x.shape), "padding": wl.padding,
                   "grads": "img1, img2" if g2wanted else "img1",
                   "path": "saved gradient fields (training forward) + scaling backward",
                   "l2": "flushed before every step (256 MiB write outside the timed events)",
                   "timing": "CUDA events around each step (forward + backward) on the launching "
                             "stream; value = K steps / sum; fwd_ms, bwd_ms from a second pass "
                             "with an event between them"},
        # per step: the forward kernel(s) (2D: one; 3D: xy, z, adjoint) and the scaling backward
        "gpu_launches": (2 if not is3d else 4) * args.steps,
        "roofline": {"kernel": KERNEL_NAME if not is3d else KERNEL3D_NAME, "bound": "alu",
                     "achieved": rf["tflops"], "peak": alu_peak_tflops, "unit": "TFLOP/s",
                     "frac": rf["alu_frac"],
                     "traffic": traffic,
                     "traffic_source": ("ncu capture of the same kernel sources, per launch, from "
                                        "the committed profile summary (not measured in this run)"
                                        if traffic is not None else
                                        "no ncu capture of the current kernel sources"),
                     "peak_basis": f"{sm_count} SMs x 128 fp32 lanes x 2 flops x {sm_max:.0f} MHz",
                     "flops_per_pixel": rf["flops_px"]},
        "hbm_roofline": {"min_bytes_per_step": rf["min_bytes"], "achieved_gbs": rf["hbm_gbs"],
                         "frac_of_8tbs": rf["hbm_gbs"] / NOMINAL_HBM_GBS,
                         "frac_of_measured": rf["hbm_frac"],
                         "measured_peak_gbs": peaks["hbm_gbs"], "peak_kind": peak_kind},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "e2e": {"value": e2e_value, "unit": unit,
                "h2d_bytes_per_step": 2 * elems * 4,
                "d2h_bytes_per_step": N * 4,
                "how": "public API, pinned host images copied in and the loss (per-image means) "
                       "read back every step; two input buffers, the copy of step k+1 on a "
                       "copy stream overlapping step k; value = K steps / their elapsed time",
                "serial_with_gradient_readback": {
                    "value": e2e_serial_value, "unit": unit,
                    "h2d_bytes_per_step": 2 * elems * 4,
                    "d2h_bytes_per_step": (2 if g2wanted else 1) * elems * 4 + N * 4}},
        "clocks": clk,
        "cpu_baseline": cpu,
        **extras,
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
