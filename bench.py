"""Throughput benchmark: 4K -> 1080p RGB uint8 bilinear resize on one GB300.

One step = one bilinear resize of a 3840x2160 RGB u8 frame to 1920x1080
through the C ABI (resize_u8), the whole hot path (tables come from the plan,
built once per geometry, outside the timed region).  The frames are the
smooth synthetic content (sum of sinusoids + noise) in a ring of distinct
device input/output sets (14 for this workload, 435 MB, over 3x the 129 MB
L2), so every step reads its input from HBM.  The K timed steps are one CUDA
graph of K launches (back to back on one stream; graphs of at most 4096
launches when K is larger), replayed once between two CUDA events, after W
warm-up steps, with a barrier and device synchronise on both sides.  A short
device-side hold queued before the start event keeps host submission latency
out of the timed region.

Printed (one JSON line): output Gpix/s (`value`), the dominant kernel's
roofline (algorithmic bytes per launch / average launch duration, against the
measured HBM copy peak), a trimmed mean over further timed replays, the
library's 1:1 copy baseline moving the same bytes, the end-to-end figure
through resize_u8_host from page-locked host buffers, the oracle timed on the
host cores (median of three samples, with the host's core count and CPU
model), and the SM clocks sampled during the timed region and during the
busy period just before it.

`--impl reference` times the CPU oracle (the only other implementation of the
method) on the same workload instead, each step a bounded band of output rows.
`--workload` selects one of the other resize workloads for local studies; the
default is the headline one.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MB = 1e6
L2_BYTES = 129 * 1024 * 1024
GRAPH_MAX = 4096        # launches per captured graph
SETTLE_S = 0.5          # seconds of graph replays right before the timed region
TRIM_REPLAYS = 11       # extra timed graph replays for the trimmed mean
HOLD_CYCLES = 2_000_000  # device hold before a start event (about 1 ms at 2 GHz)
CSRC = os.path.join(ROOT, "bilinear_image_resize_gb300", "csrc")

# name -> (description, kind, H, W, OH, OW, C, mode, batch)
WORKLOADS = {
    "4k_to_1080p": ("4K->1080p RGB u8 bilinear (3840x2160 -> 1920x1080, smooth synthetic)",
                    "u8", 2160, 3840, 1080, 1920, 3, "linear", 1),
    "1080p_to_4k": ("1080p->4K RGB u8 bilinear upscale (1920x1080 -> 3840x2160)", "u8", 1080, 1920, 2160, 3840, 3,
                    "linear", 1),
    "4k_to_1080p_nearest": ("4K->1080p RGB u8 nearest", "u8", 2160, 3840, 1080, 1920, 3, "nearest", 1),
    "1080p_to_540p": ("1080p->960x540 RGB u8 bilinear", "u8", 1080, 1920, 540, 960, 3, "linear", 1),
    "1080p_to_720p": ("1080p->1280x720 RGB u8 bilinear", "u8", 1080, 1920, 720, 1280, 3, "linear", 1),
    "batch64_720p_to_224_norm": ("64x 1280x720 RGB u8 -> 224x224 bilinear + normalise, f32 NCHW", "norm", 720, 1280,
                                 224, 224, 3, "linear", 64),
    "f32_8192_to_5980_filter3x3": ("f32 8192x8192 -> 5980x5980 bilinear + 3x3 filter", "filt", 8192, 8192, 5980,
                                   5980, 1, "linear", 1),
    "tiny_64x48_to_128x96": ("u8 64x48 -> 128x96 bilinear", "u8", 48, 64, 96, 128, 1, "linear", 1),
    "4k_to_1080p_gray": ("4K RGB u8 -> gray (BT.601) -> 1080p bilinear, fused (3840x2160x3 -> 1920x1080x1)",
                         "gray", 2160, 3840, 1080, 1920, 3, "linear", 1),
    "1080p_to_4k_mirror": ("1080p->4K RGB u8 bilinear upscale, mirror border", "u8", 1080, 1920, 2160, 3840, 3,
                           "linear", 1),
    "1080p_to_4k_wrap": ("1080p->4K RGB u8 bilinear upscale, wrap border", "u8", 1080, 1920, 2160, 3840, 3,
                         "linear", 1),
}
for _k in (5, 7):
    WORKLOADS[f"f32_8192_to_5980_filter{_k}x{_k}"] = (
        f"f32 8192x8192 -> 5980x5980 bilinear + {_k}x{_k} filter", "filt", 8192, 8192, 5980, 5980, 1, "linear", 1)
for _k in (8, 16, 32, 64):
    WORKLOADS[f"f32_4096_valid_filter{_k}"] = (
        f"f32 4096x4096 {_k}x{_k} correlation over the valid region (standalone)", "valid", 4096, 4096,
        4097 - _k, 4097 - _k, 1, "none", 1)
# border rule of a workload's plan (RZ_BORDER_*; clamp when absent)
WORKLOADS["f32_8192_to_5980"] = ("f32 8192x8192 -> 5980x5980 bilinear (plain resize_f32)", "f32", 8192, 8192, 5980,
                                  5980, 1, "linear", 1)
WORKLOADS["4k_to_1080p_rgba"] = ("4K->1080p RGBA u8 bilinear (exact kernel)", "u8", 2160, 3840, 1080, 1920, 4,
                                  "linear", 1)
WORKLOADS["4k_to_1080p_rgba_texture"] = ("4K->1080p RGBA u8 bilinear through the texture unit (hardware filtering, "
                                          "not bit-exact)", "tex", 2160, 3840, 1080, 1920, 4, "linear", 1)
WORKLOADS["4k_to_1366x768"] = ("4K->1366x768 RGB u8 bilinear (no exact ratio: the any-ratio direct kernel)", "u8",
                                2160, 3840, 768, 1366, 3, "linear", 1)
WORKLOADS["720p_to_1080p"] = ("1280x720->1920x1080 RGB u8 bilinear upscale (1.5x: the row-separable streaming kernel)",
                              "u8", 720, 1280, 1080, 1920, 3, "linear", 1)
WORKLOADS["multi_256_mixed"] = ("256 RGB u8 bilinear resizes of 4 mixed small geometries (640x480->320x240, "
                                 "1280x720->224x224, 320x240->640x480, 800x600->300x300) in one launch",
                                 "multi", 0, 0, 0, 0, 3, "linear", 256)
MULTI_GEOMS = [(480, 640, 240, 320), (720, 1280, 224, 224), (240, 320, 480, 640), (600, 800, 300, 300)]
WORKLOADS["1080p_to_540p_and_720p"] = ("1080p RGB u8 -> 960x540 and -> 1280x720 bilinear, both resizes of each frame "
                                       "in one CUDA graph (two resize_u8 launches per step)", "pair", 1080, 1920,
                                       0, 0, 3, "linear", 1)
PAIR_GEOMS = [(540, 960), (720, 1280)]
WORKLOAD_BORDER = {"1080p_to_4k_mirror": 1, "1080p_to_4k_wrap": 2}
# filter width of the filter workloads (3 when absent)
WORKLOAD_FILTER_K = {f"f32_8192_to_5980_filter{k}x{k}": k for k in (5, 7)}
WORKLOAD_FILTER_K.update({f"f32_4096_valid_filter{k}": k for k in (8, 16, 32, 64)})


def fp32_fma_peak_tflops(sm_mhz=2070.0, sms=152):
    """FP32 peak from unit counts and clocks: sms x 128 FMA lanes x 2 FLOP x clock."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


FILTER_TC_MIN_K = 48           # the library's automatic choice: tensor cores from this width
TF32_OVER_BF16 = 1.1 / 2.25    # nominal dense TF32 / BF16 tensor rates


def filter_tc_flops(K, OH, OW):
    """FLOPs the tensor-core correlation executes per launch: 128 x 32 output
    tiles, per filter row 3 MMAs (hi*hi, hi*lo, lo*hi) per 8-wide K step over
    K_T = 32 ceil((32 + K - 1) / 32) Toeplitz columns, 2 x 128 x 32 x 8 each."""
    tiles = ((OW + 31) // 32) * ((OH + 127) // 128)
    chunks = (32 + K - 1 + 31) // 32
    return tiles * K * 3 * (4 * chunks) * 2 * 128 * 32 * 8


def trimmed_mean(xs, frac=0.1):
    """Mean after sorting and dropping `frac` of the samples at each end (the
    Volcanic page's *Measure performance carefully*: discard outliers, then
    average); at least one sample is kept."""
    v = sorted(float(x) for x in xs)
    if not v:
        raise ValueError("no samples")
    k = int(len(v) * frac)
    if 2 * k >= len(v):
        k = (len(v) - 1) // 2
    v = v[k:len(v) - k]
    return sum(v) / len(v)


def host_cpu():
    """Core count and CPU model of this host (lscpu, else /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    key = line.split(":", 1)[0].strip().lower()
                    if key in ("model name", "cpu part") and ":" in line:
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_count": os.cpu_count(), "model": model or "unknown", "machine": platform.machine()}


DEFAULT_WORKLOAD = "4k_to_1080p"
METRIC = "output Gpix/s and achieved HBM GB/s (% of GB300 peak), 4K->1080p RGB u8 bilinear"


# ------------------------------------------------------------------ helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(x, dist, device):
    """The largest of every rank's x (the slowest rank's time), via an
    all-reduce on `device` (a CUDA device under NCCL, the CPU under gloo)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gpix(px_per_step, steps, world, ms_max):
    """Whole-job output Gpix/s: every rank's steps over the slowest rank's time."""
    return px_per_step * steps * world / (ms_max / 1e3) / 1e9


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def algorithmic_bytes(kind, H, W, OH, OW, C, mode, batch):
    """Bytes the method must move per launch: every source row a tap reads
    (whole rows: every 32-byte sector of a tapped row holds a tap at these
    ratios) plus the output."""
    import bilinear_image_resize_gb300 as rz
    m = rz.RZ_LINEAR if mode == "linear" else rz.RZ_NEAREST
    yofs, _, _ = rz.resize_axis_table(H, OH, m)
    rows = set(int(r) for r in yofs)
    if m == rz.RZ_LINEAR:
        rows |= set(min(int(r) + 1, H - 1) for r in yofs)
    in_es = 4 if kind in ("filt", "f32") else 1
    out_es = 1 if kind in ("u8", "gray", "tex") else 4
    read = len(rows) * W * C * in_es
    write = OH * OW * (1 if kind == "gray" else C) * out_es
    return batch * read, batch * write


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms in a thread."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for (t, line) in self.samples:
            if not (t0 <= t <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_sources_hash(cu: str) -> str:
    """sha256[:16] over a kernel's .cu file and the two headers it includes:
    the key that ties a committed ncu summary to the code it measured."""
    h = hashlib.sha256()
    for name in (cu, "rz_device.h", "rz_internal.h"):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(workload: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the summary is missing or the kernel's sources have
    changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"ncu_{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
        m_hash = re.search(r"kernel sources \((\w+\.cu) \+ headers\) sha256\[:16\]:\s*`([0-9a-f]{16})`", text)
        m_bytes = re.search(r"dram bytes per launch:\s*`?([0-9]+)", text)
        if not m_hash or not m_bytes or kernel_sources_hash(m_hash.group(1)) != m_hash.group(2):
            return None
    except OSError:
        return None
    return int(m_bytes.group(1))


# ------------------------------------------------------------------ the GPU arm

def make_frames(kind, H, W, C, batch, count, dev):
    import numpy as np
    import torch

    from bilinear_image_resize_gb300 import synth
    if kind in ("u8", "gray", "tex"):
        base = synth.smooth_rgb(W, H, 3) if (C == 3 and W >= 1920) else synth.random_u8((H, W, C), seed=3)
        if base.shape != (H, W, C):
            base = synth.random_u8((H, W, C), seed=3)
        t = torch.from_numpy(np.ascontiguousarray(base)).to(dev)
        frames = [t.clone() for _ in range(count)]
        for i, f in enumerate(frames):        # distinct content per frame, same statistics
            if i:
                f.copy_(torch.roll(t, shifts=7 * i, dims=1))
        return frames
    if kind == "norm":
        base = torch.from_numpy(synth.frames_rgb(batch, W, H, 4)).to(dev)
        return [base.clone() if i else base for i in range(count)]
    base = torch.from_numpy(synth.float_gray(W, H, 5)).to(dev)
    return [base.clone() if i else base for i in range(count)]


def make_outputs(kind, OH, OW, C, batch, count, dev):
    import torch
    if kind in ("u8", "tex"):
        shape, dt = (OH, OW, C), torch.uint8
    elif kind == "gray":
        shape, dt = (OH, OW), torch.uint8
    elif kind == "f32":
        shape, dt = (OH, OW), torch.float32
    elif kind == "norm":
        shape, dt = (batch, C, OH, OW), torch.float32
    else:
        shape, dt = (OH, OW), torch.float32
    return [torch.empty(shape, dtype=dt, device=dev) for _ in range(count)]


def make_epi(rz, synth, kind, workload=""):
    """The fused epilogue of a workload kind (None for the plain uint8 resize)."""
    if kind == "norm":
        return rz.make_epilogue(rz.RZ_EPI_NORMALIZE_NCHW, mean=synth.NORM_MEAN, std=synth.NORM_STD)
    if kind == "filt":
        K = WORKLOAD_FILTER_K.get(workload, 3)
        if K != 3:
            return rz.make_epilogue(rz.RZ_EPI_FILTER, wk=synth.filter_weights_k(K))
        return rz.make_epilogue(rz.RZ_EPI_FILTER3X3, w3x3=synth.filter_weights())
    if kind == "gray":
        return rz.make_epilogue(rz.RZ_EPI_GRAY_RGB)
    return None


def gpu_arm(args, rank, local_rank, world):
    import numpy as np
    import torch

    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import synth

    desc, kind, H, W, OH, OW, C, mode_s, batch = WORKLOADS[args.workload]
    mode = rz.RZ_LINEAR if mode_s == "linear" else rz.RZ_NEAREST
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)

    rd, wr = algorithmic_bytes(kind, H, W, OH, OW, C, mode_s, batch)
    step_bytes = rd + wr
    in_bytes = batch * H * W * C * (4 if kind in ("filt", "f32") else 1)
    out_bytes = wr
    ring = max(2, min(64, int(3 * L2_BYTES // (in_bytes + out_bytes)) + 1))
    frames = make_frames(kind, H, W, C, batch, ring, dev)
    outs = make_outputs(kind, OH, OW, C, batch, ring, dev)
    plan = rz.resize_plan_create(H, W, OH, OW, mode, border=WORKLOAD_BORDER.get(args.workload, 0))
    if args.tile:
        tr, tw = (int(v) for v in args.tile.split("x"))
        fam = {"u8": rz.KIND_U8, "norm": rz.KIND_NORMALIZE, "filt": rz.KIND_FILTER3X3}[kind]
        rz.resize_plan_set_tile(plan, fam, tr, tw)
    if args.stages:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_STAGES, args.stages)
    if args.generic:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_GENERIC_ONLY, 1)
    if args.ctas_per_sm:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_CTAS_PER_SM, args.ctas_per_sm)
    if args.grid_per_tile:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_GRID_MODE, 1)
    if args.no_pdl:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_PDL, 0)
    if args.u8_kernel:
        rz.resize_plan_set_option(plan, rz.RZ_OPT_U8_KERNEL, args.u8_kernel)
    epi = make_epi(rz, synth, kind, args.workload)
    textures = [rz.Texture(f) for f in frames] if kind == "tex" else None

    def step(i):
        s, d = frames[i % ring], outs[i % ring]
        if kind == "u8":
            rz.resize_u8(plan, s, d, stream=stream)
        elif kind == "tex":
            textures[i % ring].resize(d, stream=stream)
        elif kind == "f32":
            rz.resize_f32(plan, s, d, stream=stream)
        else:
            rz.resize_fused(plan, s, d, epi, stream=stream)

    torch.cuda.synchronize()
    # warm-up, eager (also sets kernel attributes before any capture)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()

    # the K timed steps as graphs of at most GRAPH_MAX launches: one graph
    # for any K up to GRAPH_MAX, so the timed region has no gap between graphs
    G = max(1, min(args.steps, GRAPH_MAX))

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        return g

    g_full = capture(G)
    # the graph must do the work: its output for frame 0 equals an eager call's
    ref0 = torch.empty_like(outs[0])
    with torch.cuda.stream(stream):
        if kind == "u8":
            rz.resize_u8(plan, frames[0], ref0, stream=stream)
        elif kind == "tex":
            textures[0].resize(ref0, stream=stream)
        elif kind == "f32":
            rz.resize_f32(plan, frames[0], ref0, stream=stream)
        else:
            rz.resize_fused(plan, frames[0], ref0, epi, stream=stream)
        outs[0].zero_()
        g_full.replay()
    torch.cuda.synchronize()
    if not torch.equal(outs[0], ref0):
        raise RuntimeError("captured graph did not reproduce the eager result")
    del ref0
    rem = args.steps % G
    g_rem = capture(rem) if rem else None
    reps = args.steps // G
    # graph warm-up replays; replay() launches on torch's current stream, so
    # every replay below runs with `stream` current
    with torch.cuda.stream(stream):
        g_full.replay()
    torch.cuda.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(visible[local_rank] if local_rank < len(visible) else local_rank)
    sampler.start()
    time.sleep(0.3)
    # a busy period right before the timed region (clocks settle; the sampler
    # records them: the timed region itself is often shorter than its period)
    t_settle0 = time.time()
    while time.time() - t_settle0 < SETTLE_S:
        with torch.cuda.stream(stream):
            for _ in range(8):
                g_full.replay()
        torch.cuda.synchronize()
    t_settle1 = time.time()

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        hold_stream(stream)
        ev0.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    if dist:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)

    # further timed replays of the first graph, one event pair each, for the
    # trimmed mean (not part of the contract's timed region)
    per_launch_us = []
    for _ in range(TRIM_REPLAYS):
        with torch.cuda.stream(stream):
            hold_stream(stream)
            ev0.record(stream)
            g_full.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        per_launch_us.append(ev0.elapsed_time(ev1) * 1e3 / G)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t_host0 - 0.02, t_host1 + 0.02)
    clocks["settle"] = sampler.summary(t_settle0, t_settle1)
    replays = {"launches_per_replay": G, "replays": len(per_launch_us),
               "per_launch_us": [round(x, 4) for x in per_launch_us],
               "trimmed_mean_us": trimmed_mean(per_launch_us), "median_us": statistics.median(per_launch_us),
               "trim": "10% of the sorted samples dropped at each end"}

    ms_max = max_over_ranks(ms, dist, dev) if dist else ms

    # eager (per-call launch) rate, for reference
    with torch.cuda.stream(stream):
        ev0.record(stream)
        n_eager = min(args.steps, 2000)
        for i in range(n_eager):
            step(i)
        ev1.record(stream)
    torch.cuda.synchronize()
    eager_ms = ev0.elapsed_time(ev1) / n_eager

    # end to end through resize_u8_host (u8 workloads): pinned host frames,
    # H2D + kernel + D2H every step, three streams in rotation
    e2e = None
    if kind == "u8":
        e2e = e2e_u8(rz, plan, frames[0], H, W, OH, OW, C, dev, n=max(10, min(args.steps, 200)))

    # the 1:1 copy baseline moving this step's bytes (half read, half
    # written), timed the same way
    ceiling = copy_baseline(rz, step_bytes, ring, stream, dev, G)

    # several frames per launch (resize_u8_batch), u8 workloads
    batched = None
    if kind == "u8" and args.batch_frames > 0:
        batched = batched_u8(rz, plan, frames, H, W, OH, OW, C, args.batch_frames, stream, dev, step_bytes)

    px = OH * OW * batch
    value = aggregate_gpix(px, args.steps, world, ms_max)
    launch_ms = ms / args.steps
    achieved = step_bytes / (launch_ms / 1e3) / 1e9
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    res = {
        "value": value, "ms": ms_max, "launch_ms": launch_ms, "eager_ms_per_step": eager_ms,
        "achieved_gbs": achieved, "peak_gbs": peak, "peak_src": src, "step_bytes": step_bytes,
        "read_bytes": rd, "write_bytes": wr, "ring": ring, "graph_steps": G, "clocks": clocks, "e2e": e2e,
        "desc": desc, "px": px, "batched": batched, "copy_ceiling": ceiling, "replays": replays,
    }
    for t in textures or ():
        t.destroy()
    plan.destroy()
    return res


def valid_arm(args, local_rank):
    """The standalone K x K correlation (filter2d_valid_f32): graph-replayed
    launches over a ring of inputs larger than L2, event-timed on the
    launching stream, FLOPs = 2 K^2 per output."""
    import torch

    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import synth
    desc, kind, H, W, OH, OW, C, _m, batch = WORKLOADS[args.workload]
    K = WORKLOAD_FILTER_K[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    ring = max(2, int(3 * L2_BYTES // (4 * (H * W + OH * OW))) + 1)
    base = torch.from_numpy(synth.float_gray(W, H, 5)).to(dev)
    srcs = [base if i == 0 else torch.roll(base, 3 * i, 1) for i in range(ring)]
    dsts = [torch.empty((OH, OW), dtype=torch.float32, device=dev) for _ in range(ring)]
    wt = torch.from_numpy(synth.filter_weights_k(K)).to(dev)

    def step(i):
        rz.filter2d_valid_f32(srcs[i % ring], wt, dsts[i % ring], stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    G = max(1, min(ring * max(1, 24 // ring), args.steps))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):
            step(i)
    ref0 = dsts[0].clone()
    with torch.cuda.stream(stream):
        dsts[0].zero_()
        g.replay()
    torch.cuda.synchronize()
    if not torch.equal(dsts[0], ref0):
        raise RuntimeError("captured graph did not reproduce the eager result")
    reps = max(1, args.steps // G)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        hold_stream(stream)
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = ev0.elapsed_time(ev1)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t0 - 0.02, t1 + 0.02)
    n = reps * G
    launch_s = ms / 1e3 / n
    tflops = 2.0 * K * K * OH * OW / launch_s / 1e12
    peak = fp32_fma_peak_tflops(clocks["sm_max_mhz"] or 2070.0)
    tensor = K >= FILTER_TC_MIN_K
    peaks, src = measured_peaks()
    return {"steps": n, "ms": ms, "launch_ms": launch_s * 1e3, "tflops": tflops, "peak": peak, "clocks": clocks,
            "value": OH * OW / launch_s / 1e9, "desc": desc, "K": K, "ring": ring, "graph_steps": G,
            "tensor": tensor, "tc_tflops": filter_tc_flops(K, OH, OW) / launch_s / 1e12 if tensor else None,
            "tf32_peak": float(peaks.get("bf16_tflops", 1900.0)) * TF32_OVER_BF16, "peak_src": src}


def multi_arm(args, local_rank):
    """resize_u8_multi: N jobs of mixed geometries per launch, two sets of
    distinct frames in rotation (together larger than L2), graph-replayed and
    event-timed; beside it the same jobs as N separate resize_u8 launches
    (one plan per geometry), also graph-replayed."""
    import torch

    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import synth
    desc, kind, _H, _W, _OH, _OW, C, _m, N = WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    geoms = [MULTI_GEOMS[k % len(MULTI_GEOMS)] for k in range(N)]
    bases = {g: torch.from_numpy(synth.random_u8((g[0], g[1], C), seed=11 + i)).to(dev)
             for i, g in enumerate(MULTI_GEOMS)}
    sets = []
    for sidx in range(2):
        srcs = [torch.roll(bases[g], 5 * k + sidx, 1) for k, g in enumerate(geoms)]
        dsts = [torch.empty((g[2], g[3], C), dtype=torch.uint8, device=dev) for g in geoms]
        jobs, _ = rz.make_jobs(srcs, dsts)
        sets.append((srcs, dsts, jobs))
    plans = {g: rz.resize_plan_create(*g, rz.RZ_LINEAR) for g in MULTI_GEOMS}
    rd = wr = 0
    for g in geoms:
        r_, w_ = algorithmic_bytes("u8", g[0], g[1], g[2], g[3], C, "linear", 1)
        rd, wr = rd + r_, wr + w_
    px = sum(g[2] * g[3] for g in geoms)

    def multi(i):
        srcs, dsts, jobs = sets[i % 2]
        rz.resize_u8_multi(jobs, N, C, rz.RZ_LINEAR, stream=stream)

    def separate(i):
        srcs, dsts, _ = sets[i % 2]
        for g, s_, d_ in zip(geoms, srcs, dsts):
            rz.resize_u8(plans[g], s_, d_, stream=stream)

    def timed(fn, reps):
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(4):
                fn(i)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            hold_stream(stream)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (4 * reps)

    # the one-launch result equals the separate launches' result
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        separate(0)
    torch.cuda.synchronize()
    ref = [d.clone() for d in sets[0][1]]
    with torch.cuda.stream(stream):
        for d in sets[0][1]:
            d.zero_()
        multi(0)
    torch.cuda.synchronize()
    if not all(torch.equal(a, b) for a, b in zip(ref, sets[0][1])):
        raise RuntimeError("resize_u8_multi differs from the per-geometry launches")
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    reps = max(1, args.steps // 4)
    ms = timed(multi, reps)
    t1 = time.time()
    ms_sep = timed(separate, max(1, reps // 8))
    time.sleep(0.1)
    sampler.stop()
    peaks, src = measured_peaks()
    gbs = (rd + wr) / (ms / 1e3) / 1e9
    return {"ms": ms, "ms_separate": ms_sep, "value": px / (ms / 1e3) / 1e9, "gbs": gbs,
            "peak": float(peaks.get("hbm_gbs", 6800.0)), "peak_src": src, "bytes": rd + wr, "px": px,
            "steps": reps * 4, "clocks": sampler.summary(t0 - 0.02, t1 + 0.02), "desc": desc, "jobs": N}


def pair_arm(args, local_rank):
    """The two 1080p downscales (to 960x540, exact 2x; to 1280x720, exact
    3:2) of each frame as one step, K steps captured in one CUDA graph on one
    stream (2K launches), over a ring of frames larger than L2, timed between
    events after a device hold."""
    import numpy as np
    import torch

    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import synth
    desc, kind, H, W, _OH, _OW, C, _m, _b = WORKLOADS[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    rd = wr = 0
    for oh, ow in PAIR_GEOMS:
        r_, w_ = algorithmic_bytes("u8", H, W, oh, ow, C, "linear", 1)
        rd, wr = rd + r_, wr + w_
    per_set = H * W * C + sum(oh * ow * C for oh, ow in PAIR_GEOMS)
    ring = max(2, int(3 * L2_BYTES // per_set) + 1)
    base = torch.from_numpy(np.ascontiguousarray(synth.smooth_rgb(W, H, 2))).to(dev)
    frames = [torch.roll(base, 7 * i, 1).contiguous() for i in range(ring)]
    outs = [[torch.empty((oh, ow, C), dtype=torch.uint8, device=dev) for oh, ow in PAIR_GEOMS] for _ in range(ring)]
    plans = [rz.resize_plan_create(H, W, oh, ow, rz.RZ_LINEAR) for oh, ow in PAIR_GEOMS]
    px = sum(oh * ow for oh, ow in PAIR_GEOMS)

    def step(i):
        for p_, d_ in zip(plans, outs[i % ring]):
            rz.resize_u8(p_, frames[i % ring], d_, stream=stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    ref = [d.clone() for d in outs[0]]
    G = max(1, min(args.steps, GRAPH_MAX))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):
            step(i)
    with torch.cuda.stream(stream):
        for d in outs[0]:
            d.zero_()
        g.replay()
    torch.cuda.synchronize()
    if not all(torch.equal(a, b) for a, b in zip(ref, outs[0])):
        raise RuntimeError("captured graph did not reproduce the eager result")
    reps = max(1, args.steps // G)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    t_settle0 = time.time()
    while time.time() - t_settle0 < SETTLE_S:
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
    t_settle1 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        hold_stream(stream)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = e0.elapsed_time(e1) / (reps * G)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(t0 - 0.02, t1 + 0.02)
    clocks["settle"] = sampler.summary(t_settle0, t_settle1)
    peaks, src = measured_peaks()
    for p_ in plans:
        p_.destroy()
    gbs = (rd + wr) / (ms / 1e3) / 1e9
    return {"ms": ms, "value": px / (ms / 1e3) / 1e9, "gbs": gbs, "peak": float(peaks.get("hbm_gbs", 6800.0)),
            "peak_src": src, "bytes": rd + wr, "px": px, "steps": reps * G, "clocks": clocks, "desc": desc,
            "ring": ring, "graph_steps": G}


def hold_stream(stream):
    """Queue a short device-side wait (torch's spin kernel, about 1 ms) on
    `stream`, so that the host has queued the events and graphs that follow
    before the device reaches them: host submission latency stays out of the
    timed region.  A no-op where torch lacks the helper."""
    import torch
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(HOLD_CYCLES)


def copy_baseline(rz, step_bytes, ring, stream, dev, launches):
    """The library's 1:1 copy baseline (resize_copy_baseline: 256-thread
    CTAs, 16-byte loads and stores, PDL, pre-wait L2 prefetch) moving the
    step's byte count (half read, half written) over a ring of buffers, timed
    like the resize (one graph of `launches` launches between events after a
    device hold); also without the prefetch, and without PDL."""
    import torch
    n = max(16, step_bytes // 2 // 16 * 16)
    srcs = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(ring)]
    dsts = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(ring)]
    srcs[0].copy_(torch.randint(0, 256, (n,), dtype=torch.uint8, device=dev))
    with torch.cuda.stream(stream):
        rz.resize_copy_baseline(srcs[0], dsts[0], stream=stream)
    torch.cuda.synchronize()
    if not torch.equal(srcs[0], dsts[0]):
        raise RuntimeError("resize_copy_baseline did not copy its source")
    k = max(launches, ring)

    def timed(flags):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(k):
                rz.resize_copy_baseline(srcs[i % ring], dsts[i % ring], flags, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        us = []
        for _ in range(5):
            with torch.cuda.stream(stream):
                hold_stream(stream)
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            us.append(e0.elapsed_time(e1) * 1e3 / k)
        return statistics.median(us)

    us = timed(rz.RZ_COPY_PDL | rz.RZ_COPY_L2_PREFETCH)
    us_np = timed(rz.RZ_COPY_PDL)
    us_plain = timed(0)
    return {"what": "resize_copy_baseline (1:1 copy kernel: 256-thread CTAs, 16-byte loads and stores, PDL, "
                    "pre-wait L2 prefetch)", "bytes_moved": 2 * n, "us_per_copy": us,
            "gbs": 2 * n / (us * 1e-6) / 1e9, "us_per_copy_no_prefetch": us_np, "us_per_copy_no_pdl": us_plain,
            "launches_per_replay": k, "statistic": "median of 5 graph replays"}


def batched_u8(rz, plan, frames, H, W, OH, OW, C, nf, stream, dev, frame_bytes, launches=48):
    """Frames per second when `nf` frames go through one resize_u8_batch
    launch: distinct batches in rotation, as many as make together more than
    three times L2 (two at least), graph-replayed launches timed with events
    on the launching stream after a device hold, after a check that frame 0
    of a batched launch equals the single-frame call's output."""
    import torch
    nsets = max(2, -(-3 * L2_BYTES // (nf * frame_bytes)))
    sets = []
    for b in range(nsets):
        src = torch.stack([frames[(b * nf + i) % len(frames)] for i in range(nf)])
        sets.append((src, torch.empty((nf, OH, OW, C), dtype=torch.uint8, device=dev)))
    one = torch.empty((OH, OW, C), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        rz.resize_u8(plan, sets[0][0][0], one, stream=stream)
        for src, dst in sets:
            rz.resize_u8_batch(plan, src, dst, stream=stream)
    torch.cuda.synchronize()
    if not torch.equal(sets[0][1][0], one):
        raise RuntimeError("batched launch did not reproduce the single-frame result")
    n = max(8, nsets)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            src, dst = sets[i % nsets]
            rz.resize_u8_batch(plan, src, dst, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    reps = max(1, launches // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        hold_stream(stream)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * n)
    peaks, _src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    gbs = nf * frame_bytes / (ms / 1e3) / 1e9
    return {"frames_per_launch": nf, "value": nf * OH * OW / (ms / 1e3) / 1e9, "unit": "Gpix/s",
            "ms_per_launch": ms, "launches": reps * n, "entry": "resize_u8_batch",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak},
            "l2": f"{nsets} batches of {nf} frames in rotation, {nf * frame_bytes / MB:.0f} MB each"}


def e2e_u8(rz, plan, dev_frame, H, W, OH, OW, C, dev, n):
    import torch
    host_src = [dev_frame.cpu().pin_memory() for _ in range(2)]
    host_dst = [torch.empty((OH, OW, C), dtype=torch.uint8).pin_memory() for _ in range(3)]
    streams = [torch.cuda.Stream(device=dev) for _ in range(3)]
    dsrc = [torch.empty((H, W, C), dtype=torch.uint8, device=dev) for _ in range(3)]
    ddst = [torch.empty((OH, OW, C), dtype=torch.uint8, device=dev) for _ in range(3)]
    for i in range(3):     # warm-up
        rz.resize_u8_host(plan, host_src[i % 2], host_dst[i], dsrc[i], ddst[i], stream=streams[i])
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    main = torch.cuda.current_stream(dev)
    start.record(main)
    for s in streams:
        s.wait_event(start)
    for i in range(n):
        k = i % 3
        rz.resize_u8_host(plan, host_src[i % 2], host_dst[k], dsrc[k], ddst[k], stream=streams[k])
    for k in range(3):
        ends[k].record(streams[k])
    torch.cuda.synchronize()
    ms = max(start.elapsed_time(e) for e in ends)
    return {"value": OH * OW * n / (ms / 1e3) / 1e9, "unit": "Gpix/s",
            "h2d_bytes_per_step": H * W * C, "d2h_bytes_per_step": OH * OW * C,
            "ms_per_step": ms / n, "streams": 3, "steps": n}


# ------------------------------------------------------------------ the oracle on the host

def oracle_rate(workload, budget_s):
    """Gpix/s of the oracle over a bounded sample: whole output bands of the
    workload, repeated until `budget_s` of single-threaded CPU time."""
    import numpy as np

    import oracle
    from bilinear_image_resize_gb300 import synth
    desc, kind, H, W, OH, OW, C, mode, batch = WORKLOADS[workload]
    border = WORKLOAD_BORDER.get(workload, 0)
    if kind == "gray":
        img = synth.smooth_rgb(W, H, 3)

        def run(rows):
            return oracle.gray_resize_u8(img, OH, OW)
    elif kind in ("u8", "tex"):
        img = synth.smooth_rgb(W, H, 3) if (C == 3 and W >= 1920) else synth.random_u8((H, W, C), seed=3)
        if mode == "linear":
            def run(rows):
                return oracle.linear_u8_rows(img, OH, OW, 0, rows, border)
        else:
            def run(rows):
                return oracle.nearest_u8(img, OH, OW)
    elif kind == "norm":
        frames = synth.frames_rgb(batch, W, H, 4)

        def run(rows):
            return oracle.linear_u8_normalize(frames[0], OH, OW, synth.NORM_MEAN, synth.NORM_STD)
    elif kind == "pair":
        img = synth.smooth_rgb(W, H, 2)
        OH, OW = 1, sum(oh * ow for oh, ow in PAIR_GEOMS)   # pixels of one step (both outputs)

        def run(rows):
            return [oracle.linear_u8(img, oh, ow) for oh, ow in PAIR_GEOMS]
    elif kind == "multi":
        imgs = [synth.random_u8((g[0], g[1], C), seed=11 + i) for i, g in enumerate(MULTI_GEOMS)]
        OH, OW = 1, sum(g[2] * g[3] for g in MULTI_GEOMS)   # pixels of one pass over the geometries

        def run(rows):
            return [oracle.linear_u8(im, g[2], g[3]) for im, g in zip(imgs, MULTI_GEOMS)]
    elif kind == "valid":
        img = synth.float_gray(W, H, 5)
        wk = synth.filter_weights_k(WORKLOAD_FILTER_K[workload])
        K = wk.shape[0]

        def run(rows):
            # output rows [0, rows) need input rows [0, rows + K - 1)
            return oracle.filter_valid(img[:rows + K - 1], wk)
    elif kind == "f32":
        img = synth.float_gray(W, H, 5)

        def run(rows):
            return oracle.linear_f32(img, OH, OW)
    else:
        img = synth.float_gray(W, H, 5)
        K = WORKLOAD_FILTER_K.get(workload, 3)
        w = synth.filter_weights() if K == 3 else synth.filter_weights_k(K)

        def run(rows):
            if K == 3:
                return oracle.linear_f32_filter3x3(img, OH, OW, w)
            return oracle.linear_f32_filter(img, OH, OW, w)
    t0 = time.perf_counter()
    run(min(OH, 8))
    probe = time.perf_counter() - t0
    rows_full = OH if (kind in ("u8", "tex") and mode == "linear") else None
    if kind == "valid":
        # a band of output rows sized by the probe so the sample fits the budget
        per_row = max(probe / 8, 1e-6)
        rows_full = int(max(1, min(OH, budget_s / 3 / per_row)))
    n_px = 0
    calls = 0
    t0 = time.perf_counter()
    while True:
        if rows_full:
            run(rows_full)
            n_px += rows_full * OW
        else:
            run(None)
            n_px += OH * OW
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return n_px / dt / 1e9, calls, dt, probe


def oracle_sample(workload, budget_s, unit="Gpix/s"):
    """The oracle's rate as the median of three samples of budget_s / 3 each
    (single-threaded), with the host's core count and CPU model."""
    runs = [oracle_rate(workload, budget_s / 3.0) for _ in range(3)]
    vals = [r[0] for r in runs]
    return {"value": statistics.median(vals), "unit": unit, "cores": 1, "kind": "oracle",
            "samples": [round(v, 6) for v in vals], "statistic": "median of 3",
            "calls": sum(r[1] for r in runs), "seconds": sum(r[2] for r in runs), "host": host_cpu()}


def reference_arm(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    desc, kind, H, W, OH, OW, C, mode, batch = WORKLOADS[args.workload]
    import oracle
    from bilinear_image_resize_gb300 import synth
    import numpy as np
    img = synth.smooth_rgb(W, H, 3) if (kind == "u8" and C == 3 and W >= 1920) else None
    if kind != "u8" or mode != "linear" or img is None:
        value, calls, dt, _ = oracle_rate(args.workload, 10.0)
        total_s = dt
        steps_px = None
    else:
        # each step: a band of output rows sized so that W + K steps take about a minute
        border = WORKLOAD_BORDER.get(args.workload, 0)
        t0 = time.perf_counter()
        oracle.linear_u8_rows(img, OH, OW, 0, OH, border)
        per_frame = time.perf_counter() - t0
        budget = 60.0 / max(1, args.steps + args.warmup)
        rows = int(max(1, min(OH, OH * budget / max(per_frame, 1e-6))))
        for _ in range(args.warmup):
            oracle.linear_u8_rows(img, OH, OW, 0, rows, border)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.linear_u8_rows(img, OH, OW, 0, rows, border)
        total_s = time.perf_counter() - t0
        value = rows * OW * args.steps / total_s / 1e9
        steps_px = rows * OW
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "Gpix/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": desc, "sample": f"{steps_px} output pixels (a band of rows) per step"
                   if steps_px else "whole outputs, 10 s", "threads": 1},
        "cpu_baseline": {"value": value, "unit": "Gpix/s", "cores": 1, "kind": "oracle",
                         "sample": f"bands of {steps_px} output pixels per step, single-threaded C oracle",
                         "host": host_cpu()},
        "e2e": {"value": value, "unit": "Gpix/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ short run for profilers

def profile_run(args):
    """A few eager launches of the workload and nothing else (no graphs, no
    clock sampling, no CPU baseline): the command the ncu captures run."""
    import __graft_entry__
    __graft_entry__.build()
    import torch

    import bilinear_image_resize_gb300 as rz
    from bilinear_image_resize_gb300 import synth
    desc, kind, H, W, OH, OW, C, mode_s, batch = WORKLOADS[args.workload]
    mode = rz.RZ_LINEAR if mode_s == "linear" else rz.RZ_NEAREST
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if kind == "multi":
        geoms = [MULTI_GEOMS[k % len(MULTI_GEOMS)] for k in range(batch)]
        srcs = [torch.from_numpy(synth.random_u8((g[0], g[1], C), seed=11 + k)).to(dev) for k, g in enumerate(geoms)]
        dsts = [torch.empty((g[2], g[3], C), dtype=torch.uint8, device=dev) for g in geoms]
        jobs, _ = rz.make_jobs(srcs, dsts)
        for i in range(args.warmup + args.profile):
            rz.resize_u8_multi(jobs, batch, C, rz.RZ_LINEAR)
        torch.cuda.synchronize()
        print(f"profile run: {args.warmup} + {args.profile} launches of {desc}")
        return
    if kind == "valid":
        K = WORKLOAD_FILTER_K[args.workload]
        srcs = [torch.from_numpy(synth.float_gray(W, H, 5)).to(dev) for _ in range(2)]
        dsts = [torch.empty((OH, OW), dtype=torch.float32, device=dev) for _ in range(2)]
        wt = torch.from_numpy(synth.filter_weights_k(K)).to(dev)
        for i in range(args.warmup + args.profile):
            rz.filter2d_valid_f32(srcs[i % 2], wt, dsts[i % 2])
        torch.cuda.synchronize()
        print(f"profile run: {args.warmup} + {args.profile} launches of {desc}")
        return
    in_bytes = batch * H * W * C * (4 if kind in ("filt", "f32") else 1)
    ring = max(2, min(64, int(3 * L2_BYTES // max(1, in_bytes)) + 1))
    frames = make_frames(kind, H, W, C, batch, ring, dev)
    outs = make_outputs(kind, OH, OW, C, batch, ring, dev)
    plan = rz.resize_plan_create(H, W, OH, OW, mode, border=WORKLOAD_BORDER.get(args.workload, 0))
    epi = make_epi(rz, synth, kind, args.workload)
    nf = args.batch_frames if (kind == "u8" and args.profile_batched) else 0
    if nf:
        # two batches of nf frames in rotation, one resize_u8_batch launch each
        sets = [(torch.stack([frames[(b * nf + i) % ring] for i in range(nf)]),
                 torch.empty((nf, OH, OW, C), dtype=torch.uint8, device=dev)) for b in range(2)]
    textures = [rz.Texture(f) for f in frames] if kind == "tex" else None
    for i in range(args.warmup + args.profile):
        if nf:
            rz.resize_u8_batch(plan, *sets[i % 2])
        elif kind == "tex":
            textures[i % ring].resize(outs[i % ring])
        elif kind == "f32":
            rz.resize_f32(plan, frames[i % ring], outs[i % ring])
        elif kind == "u8":
            rz.resize_u8(plan, frames[i % ring], outs[i % ring])
        else:
            rz.resize_fused(plan, frames[i % ring], outs[i % ring], epi)
    torch.cuda.synchronize()
    assert rz.resize_plan_status(plan) == rz.RZ_OK
    plan.destroy()
    what = f"batches of {nf} frames of " if nf else ""
    print(f"profile run: {args.warmup} + {args.profile} launches of {what}{desc}")


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--tile", default="", help="override tile as ROWSxCOLS (tuning only)")
    ap.add_argument("--stages", type=int, default=0, help="staged-tile ring depth (tuning only)")
    ap.add_argument("--generic", action="store_true", help="disable the exact 2x path (tuning only)")
    ap.add_argument("--ctas-per-sm", type=int, default=0, help="cap resident CTAs per SM (tuning only)")
    ap.add_argument("--grid-per-tile", action="store_true", help="one CTA per tile (tuning only)")
    ap.add_argument("--no-pdl", action="store_true", help="plain stream-ordered launches (tuning only)")
    ap.add_argument("--u8-kernel", type=int, default=0,
                    help="RZ_OPT_U8_KERNEL: 1 staged tiles, 2 streaming, 3 direct loads (tuning only)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--batch-frames", type=int, default=8,
                    help="uint8 workloads: also time this many frames per resize_u8_batch launch (0: skip)")
    ap.add_argument("--profile", type=int, default=0,
                    help="only run W + N eager launches (for ncu captures); prints no JSON line")
    ap.add_argument("--profile-batched", action="store_true",
                    help="with --profile on a uint8 workload: launches of --batch-frames frames each")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        reference_arm(args)
        return
    if args.profile:
        profile_run(args)
        return

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")

    import __graft_entry__
    __graft_entry__.build()

    if WORKLOADS[args.workload][1] == "multi":
        r = multi_arm(args, local_rank)
        if rank == 0:
            cpu = oracle_sample(args.workload, args.cpu_budget)
            cpu["sample"] = f"{cpu['calls']} passes over the 4 geometries in {cpu['seconds']:.1f} s, single-threaded"
            line = {
                "metric": f"output Gpix/s and achieved HBM GB/s, {r['desc']}", "value": r["value"],
                "unit": "Gpix/s", "n_gpus": world, "steps": r["steps"], "warmup": args.warmup,
                "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "u8", "data": "synthetic",
                "config": {"workload": r["desc"], "jobs_per_launch": r["jobs"],
                           "l2": "two sets of distinct frames in rotation, together larger than L2",
                           "launch": "CUDA graphs of 4 resize_u8_multi launches, one stream",
                           "algorithmic_bytes_per_step": r["bytes"]},
                "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": r["peak"], "unit": "GB/s",
                             "frac": r["gbs"] / r["peak"],
                             "peak_source": f"{r['peak_src']} HBM copy (MEASURED_PEAKS.json hbm_gbs)",
                             "traffic": profile_traffic(args.workload)},
                "separate_launches": {"ms_per_step": r["ms_separate"],
                                      "value": r["px"] / (r["ms_separate"] / 1e3) / 1e9, "unit": "Gpix/s",
                                      "what": f"the same {r['jobs']} jobs as {r['jobs']} resize_u8 launches "
                                              "(one plan per geometry), graph-replayed"},
                "cpu_baseline": cpu,
                "e2e": None, "gpu_launches": r["steps"], "clocks": r["clocks"],
            }
            print(json.dumps(line), flush=True)
        return

    if WORKLOADS[args.workload][1] == "pair":
        r = pair_arm(args, local_rank)
        if rank == 0:
            cpu = oracle_sample(args.workload, args.cpu_budget)
            cpu["sample"] = (f"{cpu['calls']} steps (both outputs of a frame) in {cpu['seconds']:.1f} s, "
                             "single-threaded C oracle")
            line = {
                "metric": f"output Gpix/s and achieved HBM GB/s, {r['desc']}", "value": r["value"],
                "unit": "Gpix/s", "n_gpus": world, "steps": r["steps"], "warmup": args.warmup,
                "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "u8", "data": "synthetic",
                "config": {"workload": r["desc"], "l2": f"ring of {r['ring']} frames and outputs > 3x L2",
                           "launch": f"one CUDA graph of {r['graph_steps']} steps (two resize_u8 launches each), "
                                     "one stream, after a device hold",
                           "algorithmic_bytes_per_step": r["bytes"]},
                "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": r["peak"], "unit": "GB/s",
                             "frac": r["gbs"] / r["peak"],
                             "peak_source": f"{r['peak_src']} HBM copy (MEASURED_PEAKS.json hbm_gbs)",
                             "traffic": None},
                "cpu_baseline": cpu, "e2e": None, "gpu_launches": 2 * r["steps"], "clocks": r["clocks"],
            }
            print(json.dumps(line), flush=True)
        return

    if WORKLOADS[args.workload][1] == "valid":
        r = valid_arm(args, local_rank)
        if rank == 0:
            cpu = oracle_sample(args.workload, args.cpu_budget)
            cpu["sample"] = (f"{cpu['calls']} bands of output rows in {cpu['seconds']:.1f} s, "
                             "single-threaded C oracle")
            line = {
                "metric": f"output Gpix/s and FP32 TFLOP/s, {r['desc']}", "value": r["value"], "unit": "Gpix/s",
                "n_gpus": world, "steps": r["steps"], "warmup": args.warmup, "ms_per_step": r["launch_ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": {"workload": r["desc"], "l2": f"ring of {r['ring']} input/output sets > 3x L2",
                           "launch": f"CUDA graphs of {r['graph_steps']} filter2d_valid_f32 launches, one stream",
                           "flops_per_step": 2 * r["K"] ** 2 * WORKLOADS[args.workload][4] ** 2},
                "roofline": ({"bound": "tensor", "achieved": r["tc_tflops"], "peak": r["tf32_peak"],
                              "unit": "TFLOP/s", "frac": r["tc_tflops"] / r["tf32_peak"],
                              "peak_source": f"{r['peak_src']} bf16 (MEASURED_PEAKS.json bf16_tflops) x nominal "
                                             "TF32/BF16 ratio 1.1/2.25",
                              "flops": "executed by the tensor-core kernel (3 TF32 products per tap pair over "
                                       "Toeplitz tiles)",
                              "traffic": profile_traffic(args.workload)} if r["tensor"] else
                             {"bound": "alu", "achieved": r["tflops"], "peak": r["peak"], "unit": "TFLOP/s",
                              "frac": r["tflops"] / r["peak"],
                              "peak_source": "derived: 152 SMs x 128 FP32 FMA lanes x 2 FLOP x max SM clock",
                              "traffic": profile_traffic(args.workload)}),
                "useful": {"tflops": r["tflops"], "fp32_fma_peak": r["peak"], "frac_of_fp32_fma_peak":
                           r["tflops"] / r["peak"], "flops": "2 K^2 per output",
                           "kernel": "tensor cores (k_filter_tc)" if r["tensor"] else "FP32 FMA (k_filter_valid)"},
                "cpu_baseline": cpu,
                "e2e": None, "gpu_launches": r["steps"], "clocks": r["clocks"],
            }
            print(json.dumps(line), flush=True)
        return

    r = gpu_arm(args, rank, local_rank, world)

    if rank == 0:
        cpu = None
        if world == 1:
            cpu = oracle_sample(args.workload, args.cpu_budget)
            cpu["sample"] = (f"{cpu['calls']} whole outputs of this workload in {cpu['seconds']:.1f} s, "
                             "single-threaded C oracle")
        traffic = profile_traffic(args.workload)
        desc = r["desc"]
        line = {
            "metric": METRIC,
            "value": r["value"],
            "unit": "Gpix/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": r["ms"] / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "u8" if WORKLOADS[args.workload][1] in ("u8", "gray", "tex") else "f32",
            "data": "synthetic",
            "config": {
                "workload": desc,
                "l2": f"ring of {r['ring']} distinct input/output sets "
                      f"({r['ring'] * (r['read_bytes'] + r['write_bytes']) / MB:.0f} MB) > 3x L2; every step L2-cold",
                "launch": f"the {args.steps} timed steps as CUDA graphs of {r['graph_steps']} "
                          f"{'resize_u8' if WORKLOADS[args.workload][1] == 'u8' else 'resize_fused'} launches "
                          f"(one frame or batch each) on one stream, after a device hold",
                "algorithmic_bytes_per_step": r["step_bytes"],
                "parallelism": f"{world} independent replica(s)",
                "tuning": {k: v for k, v in (("tile", args.tile), ("stages", args.stages),
                                             ("generic_only", args.generic), ("ctas_per_sm", args.ctas_per_sm),
                                             ("grid_per_tile", args.grid_per_tile), ("no_pdl", args.no_pdl),
                                             ("u8_kernel", args.u8_kernel))
                           if v} or "automatic",
            },
            "hbm_gbs": r["achieved_gbs"],
            "roofline": {
                "bound": "hbm",
                "achieved": r["achieved_gbs"],
                "peak": r["peak_gbs"],
                "unit": "GB/s",
                "frac": r["achieved_gbs"] / r["peak_gbs"],
                "peak_source": f"{r['peak_src']} HBM copy (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": traffic,
            },
            "cpu_baseline": cpu,
            "e2e": r["e2e"],
            "gpu_launches": args.steps,
            "eager_ms_per_step": r["eager_ms_per_step"],
            "clocks": r["clocks"],
            "batched": r["batched"],
            "copy_ceiling": dict(r["copy_ceiling"],
                                 resize_over_copy_time=(r["launch_ms"] * 1e3) / r["copy_ceiling"]["us_per_copy"]),
            "replays": r["replays"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
