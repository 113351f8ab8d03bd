"""Benchmark: giga pixel-pulse backprojections per second on GB300.

One step is one full backprojection of the page-sized airborne spotlight
scene (Na = 4096 pulses, Nr = 4096 range bins, 1024 x 1024 image at 0.15 m;
SARBP-GPU §1.2 and §3.3 of the page "基于GPU的SAR后向投影成像优化与CUDA加速实践"):
the echo table build, the main backprojection kernel and the partial-sum
reduction, all through the C-ABI call sarbp_backproject.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) each rank backprojects its
own, independently seeded frame on its own GPU; there is no data exchange.
The reported value is all ranks' updates divided by the slowest rank's time.
``--impl reference`` times the FP64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "giga pixel-pulse backprojections/sec on 1 GB300; % of SFU/FP32 roofline"
UNIT = "Gupd/s"
WORKLOAD = ("page-sized airborne spotlight: Na=4096 pulses, Nr=4096 complex64 bins, "
            "1024x1024 image at 0.15 m, 64 point targets + clutter sigma=0.1")
# SARBP-GPU §3.3: about 0.8 s per frame on an RTX 3080 for Na = 4096 and a
# 1024 x 1024 image (4096 * 1024 * 1024 updates, §1.2) -> 5.37 Gupd/s.
PAGE_GUPD = 4096 * 1024 * 1024 / 0.8 / 1e9
MUFU_PER_SM_CLK = 16          # sine/cosine lanes per SM per clock
FMA_PER_SM_CLK = 128          # FP32 lanes per SM per clock
# FP32-pipe operations per update of the page's loop for each interpolation
# (SARBP-GPU §2.2 and the §3.3 pseudo-code): p - a (3), |p - a|^2 (3), the
# range index (1) and its fraction or rounding (1), the interpolation (linear:
# 2 complex lerps = 4; 8-tap sinc: 8 real weights on complex samples = 16;
# nearest: none) and the phase multiply-accumulate (4). The height map adds
# no operation: the pixel's z enters p - a like x and y.
FMA_OPS_PER_UPDATE = {"linear": 16, "sinc8": 28, "nearest": 12, "heights": 16,
                      "heights_sinc8": 28, "heights_nearest": 12}
LARGE_SCENES = ("large_scene", "nonideal_track")
MUFU_PER_UPDATE = 2           # sin and cos of the phase; the range needs no sqrt here
PAGE_SFU_PER_UPDATE = 3       # the page's loop: sqrt, sin, cos
SM_MAX_MHZ_FALLBACK = 2070.0
HBM_GBS_FALLBACK = 6796.9   # measured copy bandwidth of these GB300s, used when no peaks file is present


def measured_hbm_gbs() -> tuple[float, str]:
    """HBM copy bandwidth from the measured-peaks file beside this script, else the constant."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        if v > 0:
            return v, "measured"
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return HBM_GBS_FALLBACK, "fallback"


HBM_GBS, HBM_BASIS = measured_hbm_gbs()
L2_FLUSH_BYTES = 256 << 20
# ncu dram__bytes_read.sum + dram__bytes_write.sum of one bp_kernel<0> launch on
# the page-sized scene (profiles/bp_kernel_page_spotlight.md), and the SHA-256
# of the kernel sources that capture ran: the bench reports the figure only
# while the sources are unchanged, and null (no counters for this kernel) after
MAIN_KERNEL_TRAFFIC = 10_690_560
MAIN_KERNEL_TRAFFIC_SOURCES = ("domain_backprojection_sarbp_gb300/csrc/sarbp_kernels.cu",
                               "domain_backprojection_sarbp_gb300/csrc/sarbp_internal.h",
                               "domain_backprojection_sarbp_gb300/csrc/sarbp_device.cuh")
MAIN_KERNEL_TRAFFIC_SHA256 = "5e2a4afd84899884890f512c53a24fab41bc125e5b82117a234d540c11fa188d"


def kernel_sources_sha256(paths=None) -> str:
    """SHA-256 over the kernel sources, in order."""
    h = hashlib.sha256()
    for rel in paths or MAIN_KERNEL_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def main_kernel_traffic():
    """The captured traffic while the kernel sources match the capture, else None."""
    try:
        same = kernel_sources_sha256() == MAIN_KERNEL_TRAFFIC_SHA256
    except OSError:
        same = False
    return MAIN_KERNEL_TRAFFIC if same else None


# ------------------------------------------------------------------ ranks
def rank_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(updates_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job throughput in Gupd/s: every rank's updates over the slowest rank's time."""
    return updates_per_step * steps * world / max_seconds / 1e9


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, stamped in wall time."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.samples = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm = float(parts[1])
                smax = float(parts[2])
            except ValueError:
                continue
            active = [n for n, v in zip(self.NAMES, parts[4:]) if v.lower() == "active"]
            self.samples.append((ts, sm, smax, active))

    def wait_first(self, timeout: float = 5.0):
        """Block until the first sample arrives (nvidia-smi takes a moment to
        start; a short timed region would otherwise see none), at most timeout s."""
        end = time.time() + timeout
        while self.proc is not None and not self.samples and time.time() < end:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:
            inside = self.samples
            window = "whole run (timed region shorter than the sampling interval)"
        reasons = sorted({r for s in inside for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ CPU oracle leg
def oracle_rate(scene, seconds: float = 8.0, threads: int = 0, seed: int = 0):
    """Oracle Gupd/s on a random pixel sample sized for about ``seconds`` of wall time."""
    import oracle
    rng = np.random.default_rng(seed)
    npx = scene.params["nx"] * scene.params["ny"]
    # two calibration runs: the first (64 pixels) is dominated by thread start-up
    # and overestimates the cost per pixel; the second takes about a tenth of
    # the requested time
    per_pixel = None
    size = 64
    for _ in range(2):
        probe = rng.choice(npx, size=min(npx, size), replace=False)
        _, secs, used = oracle.backproject(scene.params, scene.echoes, scene.antenna_pos, probe,
                                           threads=threads, return_info=True)
        per_pixel = max(secs, 1e-6) / probe.size
        size = int(max(64, 0.1 * seconds / per_pixel))
    count = int(min(npx, max(256, seconds / per_pixel)))
    pix = rng.choice(npx, size=count, replace=False)
    _, secs, used = oracle.backproject(scene.params, scene.echoes, scene.antenna_pos, pix,
                                       threads=threads, return_info=True)
    updates = count * scene.params["na"]
    return dict(value=updates / secs / 1e9, unit=UNIT, cores=int(used), kind="oracle",
                sample=f"{count} random pixels x all {scene.params['na']} pulses "
                       f"({updates:.3e} updates) of the same scene, {secs:.2f} s wall")


def cpu_model() -> str:
    """The host CPU's model name as the OS reports it."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def cpu_baseline(scene, seconds: float):
    """The oracle on all host cores (the reported baseline) and on one thread,
    with the full-image times both rates extrapolate to, beside the page's own
    single-thread figure for this scene size."""
    allc = oracle_rate(scene, seconds=seconds)
    one = oracle_rate(scene, seconds=max(1.0, seconds / 4), threads=1, seed=1)
    updates = scene.params["na"] * scene.params["nx"] * scene.params["ny"]
    allc.update(
        cpu_model=cpu_model(), hardware_threads=os.cpu_count(),
        one_thread={"value": one["value"], "unit": UNIT, "sample": one["sample"]},
        extrapolated_full_image_s={"all_cores": updates / (allc["value"] * 1e9),
                                   "one_thread": updates / (one["value"] * 1e9)},
        page_figure={"one_thread_cpu_s": 56.0, "gpu_s_per_frame": 0.8,
                     "scene": "Na=4096 pulses, 1024x1024 image",
                     "hardware": "RTX 3080 GPU; CPU not stated",
                     "speedup_over_one_thread": "more than 70x",
                     "serial_cpu_vs_gpu": "about 50 min against under 1 min (scene not stated)"})
    return allc


def run_reference(args, scene):
    """The oracle as it stands, timed on the host cores, one bounded sample per step."""
    import oracle
    rng = np.random.default_rng(7)
    npx = scene.params["nx"] * scene.params["ny"]
    calib = oracle_rate(scene, seconds=1.0)
    per_step_pixels = int(max(64, min(npx, calib["value"] * 1e9 * args.ref_step_seconds
                                      / scene.params["na"])))
    pix = rng.choice(npx, size=per_step_pixels, replace=False)
    for _ in range(args.warmup):
        oracle.backproject(scene.params, scene.echoes, scene.antenna_pos, pix[:64])
    total, used = 0.0, 0
    for _ in range(args.steps):
        _, secs, used = oracle.backproject(scene.params, scene.echoes, scene.antenna_pos, pix,
                                           return_info=True)
        total += secs
    updates = per_step_pixels * scene.params["na"]
    value = updates * args.steps / total / 1e9
    sample = (f"{per_step_pixels} random pixels x all {scene.params['na']} pulses per step "
              f"({updates:.3e} updates)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": value / PAGE_GUPD,
        "dtype": "f64", "data": "synthetic", "config": config_block(scene, "n/a (CPU)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": int(used), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_block(scene, l2):
    p = scene.params
    return {"workload": WORKLOAD, "na": p["na"], "nr": p["nr"], "nx": p["nx"], "ny": p["ny"],
            "pixel_m": p["dx"], "updates_per_step": p["na"] * p["nx"] * p["ny"], "l2": l2,
            "seed": scene.cfg.seed}


# ------------------------------------------------------------------ GPU leg
def time_calls(call, steps, flush, stream):
    """Summed CUDA-event milliseconds of ``steps`` calls, L2 flushed before each."""
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    total = 0.0
    for i in range(steps):
        flush.fill_(float(i))
        start.record(stream)
        call()
        end.record(stream)
        end.synchronize()
        total += start.elapsed_time(end)
    return total


def large_scene_lines(name, steps, flush, stream, dev, roofs):
    """Per-call rates of the linear and windowed-sinc backprojection of one of
    the large scenes (device-resident inputs, L2 flushed before each call)."""
    import torch

    from domain_backprojection_sarbp_gb300 import Plan
    from synth import scenes

    cfg = scenes.config_by_name(name)
    t0 = time.perf_counter()
    sc = scenes.make_scene(cfg)
    gen_s = time.perf_counter() - t0
    p = sc.params
    updates = p["na"] * p["nx"] * p["ny"]
    echoes = torch.from_numpy(sc.echoes).to(dev)
    pos = torch.from_numpy(sc.antenna_pos).to(dev)
    del sc
    image = torch.empty((p["ny"], p["nx"]), dtype=torch.complex64, device=dev)
    out = {"workload": f"{name}: Na={p['na']} pulses, Nr={p['nr']} complex64 bins, "
                       f"{p['nx']}x{p['ny']} image at {p['dx']} m",
           "updates_per_call": updates, "scene_generation_s": gen_s}
    with Plan(p, interp="sinc8") as plan:
        plan.set_timing(True)
        for interp in ("linear", "sinc8"):
            def call():
                plan.backproject(image, echoes, pos, interp=interp)
            for _ in range(3):
                call()
            torch.cuda.synchronize(dev)
            plan.kernel_times()
            ms = time_calls(call, steps, flush, stream)
            main_ms, launches = plan.kernel_times()
            main = updates / (main_ms / max(launches, 1) / 1e3) / 1e9
            out[interp] = {"steps": steps, "value": updates * steps / (ms / 1e3) / 1e9,
                           "unit": UNIT, "ms_per_step": ms / steps, "main_kernel_gupd": main,
                           "mufu_roof_frac": main / roofs["mufu"],
                           "fma_roof_frac": main / roofs["fma"][interp]}
    del echoes, pos, image
    torch.cuda.empty_cache()
    return out


def run_ours(args, scene, rank, world, local, dist):
    import torch

    from domain_backprojection_sarbp_gb300 import Plan
    from domain_backprojection_sarbp_gb300 import build as native_build

    native_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    p = scene.params
    updates = p["na"] * p["nx"] * p["ny"]
    echoes = torch.from_numpy(scene.echoes).to(dev)
    pos = torch.from_numpy(scene.antenna_pos).to(dev)
    image = torch.empty((p["ny"], p["nx"]), dtype=torch.complex64, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = Plan(p)
    info = plan.describe()
    plan.set_timing(True)

    # the clock sampler runs from before the warm-up, so that the timed region
    # has samples however short it is
    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.wait_first()
    for _ in range(args.warmup):
        plan.backproject(image, echoes, pos)
    torch.cuda.synchronize(dev)
    plan.kernel_times()                                  # drop warm-up launches

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(float(i))                            # evict L2 between steps (untimed)
        starts[i].record(stream)
        plan.backproject(image, echoes, pos)
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t1 = time.time()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    main_ms, launches = plan.kernel_times()
    total_s = sum(step_ms) / 1e3
    max_s = max_over_ranks(dist, total_s, device=dev)
    value = aggregate_value(updates, args.steps, world, max_s)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()

    # end to end through the host-buffer entry point: pinned inputs in, image out
    h_echo = torch.from_numpy(scene.echoes).pin_memory()
    h_pos = torch.from_numpy(scene.antenna_pos).pin_memory()
    h_img = torch.empty((p["ny"], p["nx"]), dtype=torch.complex64).pin_memory()
    for _ in range(max(1, min(args.warmup, 3))):
        plan.backproject_host(h_img, h_echo, h_pos, stream=stream)
    e2e_steps = max(3, min(args.steps, 20))
    barrier(dist)
    te0 = time.perf_counter()
    for _ in range(e2e_steps):
        plan.backproject_host(h_img, h_echo, h_pos, stream=stream)
    te = time.perf_counter() - te0
    e2e_max = max_over_ranks(dist, te, device=dev)
    h2d_bytes, d2h_bytes = plan.host_transfer_bytes()

    # the windowed-sinc variant on the same scene (device-resident, L2 flushed)
    variants = {}
    if not args.no_variants:
        def time_interp(interp, label):
            steps_v = max(3, min(args.steps, 20))
            for _ in range(3):
                plan.backproject(image, echoes, pos, interp=interp)
            torch.cuda.synchronize(dev)
            plan.kernel_times()
            total = 0.0
            for i in range(steps_v):
                flush.fill_(float(i))
                starts[0].record(stream)
                plan.backproject(image, echoes, pos, interp=interp)
                ends[0].record(stream)
                ends[0].synchronize()
                total += starts[0].elapsed_time(ends[0])
            main_ms_v, launches_v = plan.kernel_times()
            variants[interp] = {
                "interp": label, "steps": steps_v,
                "value": updates * steps_v / (total / 1e3) / 1e9, "unit": UNIT,
                "ms_per_step": total / steps_v,
                "main_kernel_gupd": updates / (main_ms_v / max(launches_v, 1) / 1e3) / 1e9,
            }

        # end to end again, pulses in chunks of 1024 with copies overlapped
        for _ in range(2):
            plan.backproject_streamed(h_img, h_echo, h_pos, chunk_pulses=1024, stream=stream)
        ts0 = time.perf_counter()
        for _ in range(e2e_steps):
            plan.backproject_streamed(h_img, h_echo, h_pos, chunk_pulses=1024, stream=stream)
        ts = time.perf_counter() - ts0
        s_h2d, s_d2h = plan.host_transfer_bytes()
        variants["e2e_streamed"] = {
            "api": "sarbp_backproject_streamed (pinned host buffers, chunks of 1024 pulses, "
                   "band copies overlapped with the compute)",
            "steps": e2e_steps, "value": updates * e2e_steps / ts / 1e9, "unit": UNIT,
            "ms_per_step": ts / e2e_steps * 1e3,
            "h2d_bytes_per_step": int(s_h2d), "d2h_bytes_per_step": int(s_d2h),
        }
        time_interp("sinc8", "8-tap windowed sinc (SARBP_SINC8)")
        time_interp("nearest", "nearest neighbour (SARBP_NEAREST)")
        # the same pulses onto a voxel grid of 8 planes 0.5 m apart
        nzv = 8
        vol = torch.empty((nzv, p["ny"], p["nx"]), dtype=torch.complex64, device=dev)
        for _ in range(2):
            plan.backproject_volume(vol, echoes, pos, 0.5)
        torch.cuda.synchronize(dev)
        plan.kernel_times()
        steps_v = max(3, min(args.steps, 10))
        total = 0.0
        for i in range(steps_v):
            flush.fill_(float(i))
            starts[0].record(stream)
            plan.backproject_volume(vol, echoes, pos, 0.5)
            ends[0].record(stream)
            ends[0].synchronize()
            total += starts[0].elapsed_time(ends[0])
        main_ms_v, launches_v = plan.kernel_times()
        variants["volume"] = {
            "interp": f"linear, voxel grid of {nzv} planes (sarbp_backproject_volume)",
            "steps": steps_v, "value": nzv * updates * steps_v / (total / 1e3) / 1e9, "unit": UNIT,
            "ms_per_step": total / steps_v,
            "main_kernel_gupd": updates / (main_ms_v / max(launches_v, 1) / 1e3) / 1e9,
        }
        del vol
        # the same pulses onto pixels raised by 40 m of seeded terrain
        from synth import scenes as scenes_mod
        hmap = scenes_mod.terrain(p["nx"], p["ny"], p["dx"], 20337, relief=40.0)
        heights = torch.from_numpy(hmap).to(dev)
        with Plan(p, height_range=(float(hmap.min()), float(hmap.max()))) as hplan:
            hplan.set_timing(True)
            for hinterp, key in (("linear", "heights"), ("sinc8", "heights_sinc8"),
                                 ("nearest", "heights_nearest")):
                for _ in range(3):
                    hplan.backproject_heights(image, echoes, pos, heights, interp=hinterp)
                torch.cuda.synchronize(dev)
                hplan.kernel_times()
                steps_v = max(3, min(args.steps, 20 if hinterp != "sinc8" else 10))
                total = 0.0
                for i in range(steps_v):
                    flush.fill_(float(i))
                    starts[0].record(stream)
                    hplan.backproject_heights(image, echoes, pos, heights, interp=hinterp)
                    ends[0].record(stream)
                    ends[0].synchronize()
                    total += starts[0].elapsed_time(ends[0])
                main_ms_v, launches_v = hplan.kernel_times()
                variants[key] = {
                    "interp": f"{hinterp}, pixels on a 40 m terrain height map "
                              "(sarbp_backproject_heights)",
                    "steps": steps_v, "value": updates * steps_v / (total / 1e3) / 1e9, "unit": UNIT,
                    "ms_per_step": total / steps_v,
                    "main_kernel_gupd": updates / (main_ms_v / max(launches_v, 1) / 1e3) / 1e9,
                }
        # range compression of this scene's shape (SARBP-GPU §3.1): raw chirps -> echoes
        from domain_backprojection_sarbp_gb300 import RangeCompressor
        from synth import chirp as chirp_mod
        ref = torch.from_numpy(chirp_mod.chirp().astype(np.complex64)).to(dev)
        raw = torch.empty_like(echoes).normal_()
        rc_out = torch.empty_like(echoes)
        band = chirp_mod.BANDWIDTH / (chirp_mod.C_LIGHT / (2 * chirp_mod.DR))
        rc_steps = max(3, min(args.steps, 20))
        with RangeCompressor(ref, p["na"], p["nr"], "hamming", band) as rcomp:
            for _ in range(3):
                rcomp(rc_out, raw)
            torch.cuda.synchronize(dev)
            r_ms = 0.0
            for i in range(rc_steps):
                flush.fill_(float(i))
                starts[0].record(stream)
                rcomp(rc_out, raw)
                ends[0].record(stream)
                ends[0].synchronize()
                r_ms += starts[0].elapsed_time(ends[0])
            # raw frame to image in one call: the compression fused with the
            # echo table (the compressed frame never reaches HBM), then the
            # backprojection
            def raw_call():
                plan.backproject_raw(image, raw, pos, rcomp)
            for _ in range(3):
                raw_call()
            torch.cuda.synchronize(dev)
            raw_ms = time_calls(raw_call, rc_steps, flush, stream)
        rc_bytes = 2 * p["na"] * p["nr"] * 8
        rc_gbs = rc_bytes * rc_steps / (r_ms / 1e3) / 1e9
        # FFT size and the conventional 5 N log2 N flops per complex transform
        # (two transforms per pulse) plus 6 N for the filter product
        n_fft = 1 << int(np.ceil(np.log2(p["nr"] + ref.shape[0] - 1)))
        rc_flops = p["na"] * (2 * 5 * n_fft * np.log2(n_fft) + 6 * n_fft)
        rc_tflops = rc_flops * rc_steps / (r_ms / 1e3) / 1e12
        fp32_peak = info["sms"] * 128 * 2 * SM_MAX_MHZ_FALLBACK * 1e6 / 1e12
        variants["range_compression"] = {
            "what": f"matched filter, {p['na']} pulses x {p['nr']} samples, 359-sample chirp, "
                    f"Hamming, FFT size {n_fft}", "steps": rc_steps, "ms_per_step": r_ms / rc_steps,
            "achieved_gbs": rc_gbs,
            "roofline": {"bound": "alu", "achieved": rc_tflops, "peak": fp32_peak,
                         "unit": "TFLOP/s", "frac": rc_tflops / fp32_peak,
                         "flops_per_launch": rc_flops,
                         "peak_basis": "SMs x 128 FP32 lanes x 2 (FMA) x 2070 MHz",
                         "hbm_frac": rc_gbs / HBM_GBS, "hbm_peak_gbs": HBM_GBS,
                         "hbm_peak_basis": HBM_BASIS, "algorithmic_bytes": rc_bytes},
        }
        step_mean_ms = statistics.mean(step_ms)
        variants["raw_to_image"] = {
            "api": "sarbp_backproject_raw (raw 4096 x 4096 frame, 359-sample chirp, Hamming: "
                   "range compression fused with the echo table, then the backprojection)",
            "steps": rc_steps, "ms_per_step": raw_ms / rc_steps,
            "value": updates * rc_steps / (raw_ms / 1e3) / 1e9, "unit": UNIT,
            "separate_calls_ms": r_ms / rc_steps + step_mean_ms,
            "separate_calls": "sarbp_range_compress then sarbp_backproject, each timed above",
        }
        del raw, rc_out
    plan.close()

    sms = info["sms"]
    clock_mhz = SM_MAX_MHZ_FALLBACK
    if clocks and clocks.get("sm_max_mhz"):
        clock_mhz = clocks["sm_max_mhz"]
    peak = sms * clock_mhz * 1e6 * MUFU_PER_SM_CLK / MUFU_PER_UPDATE / 1e9
    page_peak = sms * clock_mhz * 1e6 * MUFU_PER_SM_CLK / PAGE_SFU_PER_UPDATE / 1e9
    fma_peaks = {k: sms * clock_mhz * 1e6 * FMA_PER_SM_CLK / v / 1e9
                 for k, v in FMA_OPS_PER_UPDATE.items()}
    achieved = updates / (main_ms / max(launches, 1) / 1e3) / 1e9 if launches else None
    # every interpolation variant issues one sine and one cosine per update on its
    # common path, so it shares the main kernel's MUFU roof; the FP32-pipe roof
    # counts the page loop's own FP32 operations of that variant
    for key, var in variants.items():
        if "main_kernel_gupd" in var:
            var["mufu_roof_frac"] = var["main_kernel_gupd"] / peak
            if key in fma_peaks:
                var["fma_roof_frac"] = var["main_kernel_gupd"] / fma_peaks[key]
    if not args.no_variants and not args.no_large:
        roofs = {"mufu": peak, "fma": fma_peaks}
        for name in LARGE_SCENES:
            variants[name] = large_scene_lines(name, max(3, min(args.steps, 5)), flush, stream,
                                               dev, roofs)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": value / PAGE_GUPD,
        "dtype": "f32", "data": "synthetic",
        "config": config_block(scene, f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB write)"),
        "roofline": {
            "bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT,
            "frac": (achieved / peak) if achieved else None, "traffic": main_kernel_traffic(),
            "kernel": "bp_kernel",
            "peak_basis": f"{sms} SMs x {clock_mhz:.0f} MHz x {MUFU_PER_SM_CLK} MUFU/clk / "
                          f"{MUFU_PER_UPDATE} MUFU per update",
            "frac_of_page_loop_roof": (achieved / page_peak) if achieved else None,
            "fma_roof_frac": (achieved / fma_peaks["linear"]) if achieved else None,
            "fma_peak_basis": f"{sms} SMs x {clock_mhz:.0f} MHz x {FMA_PER_SM_CLK} FP32 lanes/clk / "
                              "the page loop's FP32 operations per update "
                              f"({FMA_OPS_PER_UPDATE})",
        },
        "e2e": {"value": aggregate_value(updates, e2e_steps, world, e2e_max), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
                "api": "sarbp_backproject_host (pinned, device-mapped host buffers: the kernels read "
                       "the band of range bins the image reaches and write the image in place)"},
        "gpu_launches": args.steps * info["kernels_per_call"],
        "clocks": clocks,
        "plan": info,
        "variants": variants,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(scene, args.cpu_seconds)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="page_spotlight")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the interpolation-variant and large-scene measurements")
    ap.add_argument("--no-large", action="store_true",
                    help="skip the large-scene (16384 x 2048^2, 8192 x 4096^2) lines")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from synth import scenes
    rank, world, local = rank_env()
    cfg = scenes.config_by_name(args.config)

    if args.impl == "reference":
        if rank != 0:
            return 0
        import oracle
        oracle.build()
        scene = scenes.make_scene(cfg)
        print(json.dumps(run_reference(args, scene)), flush=True)
        return 0

    import torch
    dist = init_dist(world, "nccl" if torch.cuda.is_available() else "gloo")
    # each rank backprojects its own frame: same geometry, its own seed
    scene = scenes.make_scene(cfg, seed=cfg.seed + 1000 * rank)
    if rank == 0:
        import oracle
        oracle.build()
    out = run_ours(args, scene, rank, world, local, dist)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
