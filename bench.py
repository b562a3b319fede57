"""Throughput of the tile-binned Gaussian-splat raster path on one GB300.

One step = one pass of the whole path over the 4-camera x 1M-splat 1920x1080
workload (workload 3): size query + intersection/sort (gs_isect_tiles),
tile ranges (gs_tile_offsets), forward (gs_rasterize_fwd) and backward
(gs_rasterize_bwd, upstream gradients N(0,1)).  All calls go through the
C ABI; inputs are resident in HBM; L2 is flushed between steps outside the
step's CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle, one camera of the same workload per
step, on the host cores (there is no other implementation of this path).
N > 1 runs N independent replicas (one per rank, launched by torchrun);
the path has no exchange step.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# the OpenMP oracle's threads sleep between its calls instead of spinning
os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")

METRIC = "Msplat-isect/s + Mpixel/s fwd(+bwd) at 1 GB300; % HBM / FP32-SFU roofline"
WORKLOADS = {
    2: "w2: 1 camera x 100,000 splats, 1024x1024, tile 16, elliptical radii",
    3: "w3: 4 cameras x 1,000,000 splats, 1920x1080, tile 16, elliptical radii",
    4: "w4: 1 camera x 6,000,000 splats, 3840x2160, tile 16, elliptical radii",
    5: "w5: backward on the w2 scene, upstream gradients N(0,1) seed 1",
}
WORKLOAD = WORKLOADS[3]
L2_FLUSH_BYTES = 256 << 20

# Algorithmic work per pair, counted from the per-pixel formulas (FMA = one
# operation):
#   forward, per evaluated pair: dx, dy, the quadratic form, the exponent's
#     scale, o * exp, the clamp and the two tests (13 FP32) + one ex2 (SFU);
#     per composited pair: T alpha, three colour FMAs, the T update and the
#     threshold test (6 FP32)
#   backward, per valid pair: alpha re-evaluation, T_before recovery,
#     colour / opacity / mean / conic terms and the recurrences (45 FP32) +
#     one ex2 and one reciprocal (SFU)
FWD_OPS_EVAL = 13
FWD_OPS_COMP = 6
FWD_SFU_EVAL = 1
BWD_OPS_VALID = 45
BWD_SFU_VALID = 2


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._proc = None
        self._thread = None
        self.active = False

    def start(self):
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self._proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.monotonic(), self.active, parts))

    def stop(self):
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        rows = [p for (_, act, p) in self.samples if act] or [p for (_, _, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------ GPU arm


class Path:
    """Buffers and the C-ABI call sequence of one step."""

    def __init__(self, scene, dev):
        import torch

        from tile_gaussian_splat_gb300 import binding as gs, scenes

        self.gs, self.torch, self.s, self.dev = gs, torch, scene, dev
        s = scene
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.host = {k: v for k, v in s.arrays().items() if v is not None}
        g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=1)
        self.host["grad_render_colors"] = g_rgb
        self.host["grad_render_alphas"] = g_a
        self.d = {k: t(v) for k, v in self.host.items()}
        self.d["backgrounds"] = None
        self.status = gs.new_status(dev)
        self.tpg = torch.empty((s.C, s.N), dtype=torch.int32, device=dev)
        self.q_ws = torch.empty(gs.gs_isect_workspace_size(s.C, s.N, s.tile_width,
                                                           s.tile_height, 0, True),
                                dtype=torch.uint8, device=dev)
        I = self.query()
        self.I = I
        self.ws = torch.empty(gs.gs_isect_workspace_size(s.C, s.N, s.tile_width, s.tile_height,
                                                         I, True), dtype=torch.uint8, device=dev)
        self.keys = torch.empty(I, dtype=torch.int64, device=dev)
        self.ids = torch.empty(I, dtype=torch.int32, device=dev)
        self.offsets = torch.empty((s.C, s.tile_height, s.tile_width), dtype=torch.int32,
                                   device=dev)
        self.rgb = torch.empty((s.C, s.height, s.width, 3), dtype=torch.float32, device=dev)
        self.alpha = torch.empty((s.C, s.height, s.width, 1), dtype=torch.float32, device=dev)
        self.last = torch.empty((s.C, s.height, s.width), dtype=torch.int32, device=dev)
        self.trace = torch.empty((I, 8), dtype=torch.int32, device=dev)
        self.grads = dict(
            grad_means2d=torch.empty((s.C, s.N, 2), dtype=torch.float32, device=dev),
            grad_conics=torch.empty((s.C, s.N, 3), dtype=torch.float32, device=dev),
            grad_colors=torch.empty((s.C, s.N, 3), dtype=torch.float32, device=dev),
            grad_opacities=torch.empty((s.C, s.N), dtype=torch.float32, device=dev),
            grad_backgrounds=None, grad_means2d_abs=None)
        self.pinned = None

    def query(self):
        gs, s, d = self.gs, self.s, self.d
        import ctypes as ct
        total = ct.c_int64(0)
        gs._check(gs.lib().gs_isect_tiles(
            gs._ptr(d["means2d"]), gs._ptr(d["radii"]), 1, gs._ptr(d["depths"]), s.C, s.N,
            s.tile_size, s.tile_width, s.tile_height, 1, gs._ptr(self.tpg), ct.byref(total),
            None, None, 0, gs._ptr(self.q_ws), self.q_ws.numel(), gs._ptr(self.status),
            gs._stream()), "query")
        return int(total.value)

    def emit(self, I):
        gs, s, d = self.gs, self.s, self.d
        gs._check(gs.lib().gs_isect_tiles(
            gs._ptr(d["means2d"]), gs._ptr(d["radii"]), 1, gs._ptr(d["depths"]), s.C, s.N,
            s.tile_size, s.tile_width, s.tile_height, 1, None, None, gs._ptr(self.keys),
            gs._ptr(self.ids), I, gs._ptr(self.ws), self.ws.numel(), gs._ptr(self.status),
            gs._stream()), "emit")

    def ranges(self):
        self.gs.gs_tile_offsets(self.keys, self.s.C, self.s.tile_width, self.s.tile_height,
                                d_status=self.status, out=self.offsets)

    def forward(self, pair_counts=None):
        s, d = self.s, self.d
        self.gs.gs_rasterize_fwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None,
                                 None, s.width, s.height, s.tile_size, self.offsets, self.ids,
                                 s.alpha_cutoff, s.transmittance_threshold, d_status=self.status,
                                 out=(self.rgb, self.alpha, self.last), pair_counts=pair_counts,
                                 trace=self.trace)

    def backward(self):
        s, d = self.s, self.d
        self.gs.gs_rasterize_bwd(d["means2d"], d["conics"], d["colors"], d["opacities"], None,
                                 None, s.width, s.height, s.tile_size, self.offsets, self.ids,
                                 s.alpha_cutoff, self.alpha, self.last, d["grad_render_colors"],
                                 d["grad_render_alphas"], d_status=self.status, out=self.grads,
                                 trace=self.trace)

    def step(self, ev=None):
        """ev: 6 CUDA events recorded between the stages, or None."""
        rec = (lambda i: ev[i].record()) if ev else (lambda i: None)
        rec(0)
        I = self.query()
        if I != self.I:
            raise RuntimeError("intersection count changed between steps")
        rec(1)
        self.emit(I)
        rec(2)
        self.ranges()
        rec(3)
        self.forward()
        rec(4)
        self.backward()
        rec(5)

    # end to end: host inputs in pinned memory, copies inside the timed region.
    # Two buffer sets and two copy streams: step k+1's upload and step k-1's
    # download overlap step k's kernels.
    def _outputs(self):
        return [self.rgb, self.alpha, self.grads["grad_means2d"], self.grads["grad_conics"],
                self.grads["grad_colors"], self.grads["grad_opacities"]]

    def use_set(self, b):
        st = self.sets[b]
        self.d, self.rgb, self.alpha, self.grads = st["d"], st["rgb"], st["alpha"], st["grads"]

    def setup_e2e(self):
        torch = self.torch
        like = lambda t: None if t is None else torch.empty_like(t)
        base = {"d": self.d, "rgb": self.rgb, "alpha": self.alpha, "grads": self.grads}
        other = {"d": {k: like(v) for k, v in self.d.items()}, "rgb": like(self.rgb),
                 "alpha": like(self.alpha), "grads": {k: like(v) for k, v in self.grads.items()}}
        self.sets = [base, other]
        self.pinned_in = [{k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory()
                           for k, v in self.host.items()} for _ in range(2)]
        self.pinned_out = []
        for b in range(2):
            self.use_set(b)
            self.pinned_out.append([torch.empty(o.shape, dtype=o.dtype).pin_memory()
                                    for o in self._outputs()])
        self.use_set(0)
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        h2d = sum(v.numel() * v.element_size() for v in self.pinned_in[0].values())
        d2h = sum(o.numel() * o.element_size() for o in self._outputs())
        return h2d, d2h

    def run_e2e(self, steps):
        """`steps` pipelined end-to-end steps; returns wall ms per step."""
        torch = self.torch
        comp = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def upload(k):
            b = k % 2
            with torch.cuda.stream(self.s_in):
                if k >= 2:
                    self.s_in.wait_event(ev_comp[b])  # step k-2 is done reading set b
                for key, h in self.pinned_in[b].items():
                    self.sets[b]["d"][key].copy_(h, non_blocking=True)
                ev_in[b].record(self.s_in)

        torch.cuda.synchronize()
        t0 = time.perf_counter()
        upload(0)
        for k in range(steps):
            b = k % 2
            if k + 1 < steps:
                upload(k + 1)
            comp.wait_event(ev_in[b])
            if k >= 2:
                comp.wait_event(ev_out[b])  # step k-2's results are on the host
            self.use_set(b)
            self.step()
            ev_comp[b].record(comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_comp[b])
                for o, h in zip(self._outputs(), self.pinned_out[b]):
                    h.copy_(o, non_blocking=True)
                ev_out[b].record(self.s_out)
        torch.cuda.synchronize()
        ms = (time.perf_counter() - t0) * 1e3 / steps
        self.use_set(0)
        return ms


def _src_sha(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _traffic_for(kernel, launches_per_step):
    """Per-launch DRAM bytes from a committed ncu summary, or None if absent or
    taken on a different source of the kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != _src_sha(e["source"]):
        return None
    return e.get("dram_bytes_per_launch")


def max_over_ranks(x, world, dev):
    """The largest x over the replicas (each rank passes its own); x itself
    when there is one rank.  dev: where the reduction tensor lives (the GPU
    with NCCL, the CPU with gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms, world):
    """Units per second of all replicas together over the slowest rank's time
    (weak scaling: every rank processes units_per_rank)."""
    return units_per_rank * world / (ms * 1e-3)


def run_ours(args, rank, world, scene):
    import torch
    import torch.distributed as dist

    local = int(os.environ.get("LOCAL_RANK", 0))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    path = Path(scene, dev)
    s = scene
    pixels = s.C * s.width * s.height

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        path.step()
        flush.zero_()
    stream.synchronize()
    path.gs.check_status(path.status, "warmup")

    # work measures for the roofline (outside the timed region)
    work = work_counts(path)
    max_list = work.pop("max_tile_list")

    if world > 1:
        dist.barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    clocks.active = True
    t_wall = time.perf_counter()
    for k in range(args.steps):
        path.step(ev[k])
        flush.zero_()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks.active = False
    time.sleep(0.25)
    clocks.stop()
    if world > 1:
        dist.barrier()
    path.gs.check_status(path.status, "timed steps")

    stage_ms = np.array([[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(5)]
                         for k in range(args.steps)])
    step_ms = stage_ms.sum(axis=1)
    ms = max_over_ranks(float(step_ms.mean()), world, dev)

    # end to end through host buffers (pipelined: see Path.run_e2e)
    h2d, d2h = path.setup_e2e()
    path.run_e2e(3)
    # the median of three runs: host-side copies see other traffic on the
    # host's memory now and then, which a single run can catch
    e2e_runs = sorted(path.run_e2e(max(5, min(args.steps, 20))) for _ in range(3))
    e2e = max_over_ranks(e2e_runs[1], world, dev)

    proj = bins = steps_trace = None
    if not args.main_only:
        proj = time_projection(dev, flush, max(args.warmup, 3), max(5, min(args.steps, 20)))
        bins = time_bins(path, max_list, flush, max(args.warmup, 3),
                         max(5, min(args.steps, 20)))
        steps_trace = time_steps_trace(path, flush, max(args.warmup, 3),
                                       max(5, min(args.steps, 10)))
    I = path.I
    del path
    torch.cuda.empty_cache()

    hbm_peak, peak_kind = _peaks()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks = measure_peaks(dev, sm_count)
    others = {} if args.main_only else time_other_workloads(
        dev, flush, peaks, hbm_peak, max(5, min(args.steps, 10)), max(args.warmup, 3))

    if rank != 0:
        return None
    for side in (proj, bins):
        if side is not None:
            side["achieved_gbs"] = round(side["bytes"] / (side["ms"] * 1e-3) / 1e9, 1)
            side["frac"] = round(side["achieved_gbs"] / hbm_peak, 4)
    st = stage_ms.mean(axis=0)
    clk = clocks.summary()
    stages = stage_report(s, I, st, work, peaks, hbm_peak)
    dom = STAGES[int(np.argmax(st))]
    traffic = _traffic_for({"raster_fwd": "k_raster_fwd", "raster_bwd": "k_raster_bwd"}.get(
        dom, dom), 1)
    if dom in ("raster_fwd", "raster_bwd"):
        roof = {"bound": "alu", "kernel": "k_" + dom, "achieved": stages[dom]["achieved_tops"],
                "peak": round(peaks["fp32_ops"] / 1e12, 2),
                "unit": "Tops/s (FP32 pipe, FMA = 1 op)", "frac": stages[dom]["frac"],
                "sfu_frac": stages[dom]["sfu_frac"], "traffic": traffic,
                "peak_source": peaks["source"], "ops_per_pair": stages[dom]["ops_model"]}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": stages[dom]["achieved_gbs"],
                "peak": hbm_peak, "unit": "GB/s", "frac": stages[dom]["frac"],
                "traffic": traffic, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}
    isect_ms = float(st[0] + st[1] + st[2])
    value = whole_job_rate(pixels, ms, world) / 1e6
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "Mpixel/s (whole step: isect+sort+ranges+fwd+bwd)",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": f"synthetic (seeded workload {args.workload} generator)",
        "config": workload_config(s, I, max_list, world),
        "msplat_isect_per_s": round(I / (isect_ms * 1e-3) / 1e6, 1),
        "msplat_per_s": round(s.C * s.N / (ms * 1e-3) / 1e6, 1),
        "mpixel_per_s_fwd": stages["raster_fwd"]["mpix_s"],
        "mpixel_per_s_bwd": stages["raster_bwd"]["mpix_s"],
        "stages": stages,
        "isect_sort_ranges": isect_summary(s, I, st, hbm_peak),
        "work": work,
        "roofline": roof,
        "peaks": peaks,
        "project": proj,
        "bins": bins,
        "step_trace": steps_trace,
        "workloads": others,
        "e2e": {"value": round(whole_job_rate(pixels, e2e, world) / 1e6, 2),
                "unit": "Mpixel/s",
                "note": "pinned host inputs -> image + gradients on the host; uploads and "
                        "downloads overlapped with the previous/next step; median of 3 runs",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e, 3),
                "runs_ms_per_step": [round(x, 3) for x in e2e_runs]},
        "gpu_launches": args.steps * launches_per_step(s),
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
    }
    return line


STAGES = ["isect_query", "isect_emit_sort", "tile_ranges", "raster_fwd", "raster_bwd"]


def launches_per_step(s):
    """Kernels of one step: count, count word, rects + depth histograms, 4
    depth passes, emit, the camera/tile passes, ranges, forward, backward."""
    return 1 + 1 + 1 + 4 + 1 + up_passes(s) + 1 + 1 + 1


def up_passes(s):
    from tile_gaussian_splat_gb300 import binding as gsb
    key_bits = gsb.gs_tile_bits(s.tile_width, s.tile_height) + max(0, (s.C - 1).bit_length())
    return (key_bits + 7) // 8


def impl_bytes(s, I):
    """Bytes each intersection stage of this implementation must move:
    query: mean 8 + radii 8 + count 4 per splat; emit+sort: rects + depth
    histograms (read mean, radii, depth; write a 16-byte rect) 36 B/splat,
    depth sort 12 + 3 x 16 B/splat, emission (order + rect gather) 20 B/splat
    and an 8-byte key+id per intersection, camera|tile passes 16 B per
    intersection each, the last one 24 B (read 8, write the 12-byte output,
    gather 4 bytes of depth); ranges: 8 B per intersection + 4 B per tile."""
    CN = s.C * s.N
    up = up_passes(s)
    tile_pass_bytes = (16 * (up - 1) + 24) if up else 24
    return {"isect_query": CN * (8 + 8 + 4),
            "isect_emit_sort": CN * (36 + 60 + 20) + I * (8 + tile_pass_bytes),
            "tile_ranges": I * 8 + s.C * s.tile_width * s.tile_height * 4}


def method_bytes(s, I):
    """The method's own traffic as the pages' pipeline moves it (count + scan
    24 B per splat; emission 24 B per splat + 12 B per intersection; an LSD
    sort over the significant key bits: an 8-byte histogram read plus 24 B
    per intersection per 8-bit pass; ranges 8 B per intersection + 4 B per
    tile)."""
    CN = s.C * s.N
    from tile_gaussian_splat_gb300 import binding as gsb
    key_bits = 32 + gsb.gs_tile_bits(s.tile_width, s.tile_height) + \
        max(0, (s.C - 1).bit_length())
    passes = (key_bits + 7) // 8
    return {"isect_query": CN * 24,
            "isect_emit_sort": CN * 24 + I * 12 + I * (8 + 24 * passes),
            "tile_ranges": I * 8 + s.C * s.tile_width * s.tile_height * 4}


def isect_summary(s, I, st, hbm_peak):
    """Intersect + sort + ranges as one stage, under both byte models."""
    ms = float(st[0] + st[1] + st[2])
    out = {"ms": round(ms, 4), "msplat_isect_per_s": round(I / (ms * 1e-3) / 1e6, 1),
           "msplat_per_s": round(s.C * s.N / (ms * 1e-3) / 1e6, 1)}
    for name, model in (("impl", impl_bytes(s, I)), ("method", method_bytes(s, I))):
        b = sum(model.values())
        gbs = b / (ms * 1e-3) / 1e9
        out[f"bytes_{name}"] = int(b)
        out[f"achieved_gbs_{name}"] = round(gbs, 1)
        out[f"frac_{name}"] = round(gbs / hbm_peak, 4)
    return out


def stage_report(s, I, st, work, peaks, hbm_peak):
    pixels = s.C * s.width * s.height
    ib, mb = impl_bytes(s, I), method_bytes(s, I)
    stages = {}
    for i, n in enumerate(STAGES):
        sec = float(st[i]) * 1e-3
        e = {"ms": round(float(st[i]), 4)}
        if n in ib:
            gbs = ib[n] / sec / 1e9
            e.update(bound="hbm", achieved_gbs=round(gbs, 1), frac=round(gbs / hbm_peak, 4),
                     achieved_gbs_method=round(mb[n] / sec / 1e9, 1),
                     frac_method=round(mb[n] / sec / 1e9 / hbm_peak, 4))
        else:
            if n == "raster_fwd":
                ops = FWD_OPS_EVAL * work["pairs_evaluated_fwd"] + \
                    FWD_OPS_COMP * work["pairs_composited"]
                sfu = FWD_SFU_EVAL * work["pairs_evaluated_fwd"]
                model = f"{FWD_OPS_EVAL} FP32 + {FWD_SFU_EVAL} SFU per evaluated pair, " \
                        f"{FWD_OPS_COMP} FP32 per composited pair"
                # the same count over every list entry up to each pixel's stop
                # (entries the kernel skips as unreachable included)
                ops_all = FWD_OPS_EVAL * work["pairs_to_termination"] + \
                    FWD_OPS_COMP * work["pairs_composited"]
                e["frac_all_entries"] = round(ops_all / sec / peaks["fp32_ops"], 4)
            else:
                ops = BWD_OPS_VALID * work["pairs_composited"]
                sfu = BWD_SFU_VALID * work["pairs_composited"]
                model = f"{BWD_OPS_VALID} FP32 + {BWD_SFU_VALID} SFU per valid pair"
            e.update(bound="alu", achieved_tops=round(ops / sec / 1e12, 3),
                     frac=round(ops / sec / peaks["fp32_ops"], 4),
                     sfu_frac=round(sfu / sec / peaks["sfu_ops"], 4), ops_model=model,
                     mpix_s=round(pixels / sec / 1e6, 1))
        stages[n] = e
    return stages


def workload_config(s, I, max_list, world):
    return {"workload": WORKLOADS[3] if s.C == 4 else s.name, "C": s.C, "N": s.N,
            "width": s.width, "height": s.height, "tile_size": 16, "n_isects": int(I),
            "max_tile_list": int(max_list), "pixels_per_step": s.C * s.width * s.height,
            "l2": "flushed between steps (256 MB write outside the step events)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def measure_peaks(dev, sm_count):
    """FP32 and ex2 throughput from the library's probes (gs_peak_probe),
    timed with CUDA events on the launching stream, best of 5 after 2
    warm-ups; 8 blocks of 256 threads per SM (64 warps)."""
    import torch

    from tile_gaussian_splat_gb300 import binding as gsb

    blocks = sm_count * 8
    out = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    res = {}
    for kind, name, iters in ((0, "ffma", 20000), (1, "ffma2", 10000), (2, "ex2", 2500)):
        best = None
        for k in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ops = gsb.gs_peak_probe(kind, iters, blocks, out)
            b.record()
            b.synchronize()
            if k >= 2:
                r = ops / (a.elapsed_time(b) * 1e-3)
                best = r if best is None else max(best, r)
        res[name] = best
    fp32 = max(res["ffma"], res["ffma2"])
    return {"fp32_ops": fp32, "sfu_ops": res["ex2"],
            "ffma_tops": round(res["ffma"] / 1e12, 2), "ffma2_tops": round(res["ffma2"] / 1e12, 2),
            "ex2_tops": round(res["ex2"] / 1e12, 3), "sm_count": sm_count,
            "source": "measured: gs_peak_probe FFMA / packed FFMA2 / ex2.approx loops, "
                      f"{sm_count} SMs x 64 warps, best of 5 (FP32 peak = the faster FMA form)"}


def work_counts(path):
    """Pairs of the step's forward and backward (one extra forward with the
    pair counters, outside the timed region)."""
    import torch

    s, dev = path.s, path.dev
    counts = torch.zeros((s.C, s.height, s.width, 3), dtype=torch.int32, device=dev)
    path.forward(pair_counts=counts)
    n_eval = int(counts[..., 0].sum(dtype=torch.int64))
    n_comp = int(counts[..., 1].sum(dtype=torch.int64))
    # entries up to each pixel's stop: the whole list, or up to its last id
    # when T fell below the threshold
    offs = path.offsets.reshape(-1).to(torch.int64)
    ends = torch.cat([offs[1:], torch.tensor([path.I], device=dev)])
    TW, TH = s.tile_width, s.tile_height
    ys = torch.arange(s.height, device=dev) // 16
    xs = torch.arange(s.width, device=dev) // 16
    cs = torch.arange(s.C, device=dev)
    t = (cs[:, None, None] * TH + ys[None, :, None]) * TW + xs[None, None, :]
    start, end = offs[t], ends[t]
    T = 1.0 - path.alpha[..., 0].to(torch.float64)
    stopped = T < float(s.transmittance_threshold)
    upto = torch.where(stopped, path.last.to(torch.int64) + 1 - start, end - start)
    lens = ends - offs
    return {"pairs_evaluated_fwd": n_eval, "pairs_composited": n_comp,
            "pairs_to_termination": int(upto.clamp(min=0).sum()),
            "max_tile_list": int(lens.max())}


def time_steps(path, flush, steps, warmup):
    """Per-stage CUDA-event times (ms) of `steps` steps, L2 flushed between."""
    import torch

    for _ in range(warmup):
        path.step()
        flush.zero_()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
    for k in range(steps):
        path.step(ev[k])
        flush.zero_()
    torch.cuda.synchronize()
    return np.array([[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(5)]
                     for k in range(steps)])


def time_other_workloads(dev, flush, peaks, hbm_peak, steps, warmup):
    """Workload 2 and workload 4 (the heavy-list scene) as whole steps, and
    workload 5 (the backward on workload 2's scene) from workload 2's step."""
    import torch

    from tile_gaussian_splat_gb300 import scenes

    out = {}
    for k in (2, 4):
        sc = scenes.workload(k)
        path = Path(sc, dev)
        st = time_steps(path, flush, steps, warmup)
        path.gs.check_status(path.status, f"workload {k}")
        work = work_counts(path)
        m = st.mean(axis=0)
        stages = stage_report(sc, path.I, m, work, peaks, hbm_peak)
        px = sc.C * sc.width * sc.height
        out[f"w{k}"] = {"workload": WORKLOADS[k], "ms_per_step": round(float(m.sum()), 4),
                        "mpixel_per_s": round(px / (m.sum() * 1e-3) / 1e6, 1),
                        "n_isects": path.I, "max_tile_list": work["max_tile_list"],
                        "isect_sort_ranges": isect_summary(sc, path.I, m, hbm_peak),
                        "stages": stages, "work": work}
        if k == 2:
            b = stages["raster_bwd"]
            out["w5"] = {"workload": WORKLOADS[5], "ms": b["ms"], "mpixel_per_s": b["mpix_s"],
                         "achieved_tops": b["achieved_tops"], "frac": b["frac"],
                         "sfu_frac": b["sfu_frac"], "valid_pairs": work["pairs_composited"],
                         "note": "the backward stage of the w2 step (trace-driven, upstream "
                                 "gradients N(0,1) seed 1)"}
        del path
        torch.cuda.empty_cache()
    return out


def time_projection(dev, flush, warmup, steps):
    """gs_project on 4 cameras x 1M Gaussians at 1920x1080 (the 3D scene of
    the same size as workload 3), timed alone: it makes the raster path's
    inputs and is not part of the raster step.  Outputs include the
    compensations and the float radii gs_isect_tiles takes."""
    import torch

    from tile_gaussian_splat_gb300 import binding as gsb
    from tile_gaussian_splat_gb300 import scenes

    s = scenes.scene3d()
    t = lambda a: torch.from_numpy(a).to(dev)
    m, cv, V, K = t(s.means), t(s.covars), t(s.viewmats), t(s.intrinsics)
    out = gsb.gs_project(m, cv, V, K, s.width, s.height, compensation=True, radii_float=True)
    for _ in range(warmup):
        gsb.gs_project(m, cv, V, K, s.width, s.height, out=out)
        flush.zero_()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        gsb.gs_project(m, cv, V, K, s.width, s.height, out=out)
        b.record()
        flush.zero_()
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    CN = s.C * s.N
    visible = int((out["radii"][..., 0] > 0).sum())
    return {"kernel": "k_project", "ms": round(ms, 4), "bound": "hbm",
            "bytes": s.N * 48 + CN * 44,
            "msplat_per_s": round(CN / (ms * 1e-3) / 1e6, 1),
            "config": {"scene": s.name, "C": s.C, "N": s.N, "width": s.width,
                       "height": s.height, "visible_pairs": visible,
                       "outputs": "radii, means2d, depths, conics, compensations, radii_float",
                       "l2": "flushed between launches"}}


def time_steps_trace(path, flush, warmup, steps, max_steps=64):
    """The per-pixel step trace (gs_rasterize_fwd_steps, gs_rasterize_bwd_steps)
    on the step's scene, timed apart: the alternative to the mask trace that
    the step uses.  max_steps records per pixel; pixels with more composites
    fall back to the list walk in the backward."""
    import torch

    s, d, gsb = path.s, path.d, path.gs
    K = max_steps

    def fwd():
        return gsb.gs_rasterize_fwd_steps(d["means2d"], d["conics"], d["colors"],
                                          d["opacities"], None, None, s.width, s.height, 16,
                                          path.offsets, path.ids, s.alpha_cutoff,
                                          s.transmittance_threshold, K, d_status=path.status)

    _, alpha, last, st = fwd()

    def bwd():
        return gsb.gs_rasterize_bwd_steps(d["means2d"], d["conics"], d["colors"],
                                          d["opacities"], None, None, s.width, s.height, 16,
                                          path.offsets, path.ids, s.alpha_cutoff, alpha, last,
                                          st, d["grad_render_colors"], d["grad_render_alphas"],
                                          d_status=path.status)

    res = {}
    for name, fn in (("fwd", fwd), ("bwd", bwd)):
        for _ in range(warmup):
            fn()
            flush.zero_()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
            flush.zero_()
        torch.cuda.synchronize()
        res[name] = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    gsb.check_status(path.status, "steps")
    cnt = st[2]
    over = int((cnt > K).sum())
    rec = int(torch.clamp(cnt, max=K).sum(dtype=torch.int64))
    out = {"kernels": "k_raster_fwd<.., steps>, k_raster_bwd_steps", "max_steps": K,
           "fwd_ms": round(res["fwd"], 4), "bwd_ms": round(res["bwd"], 4),
           "fallback_pixels": over, "records": rec,
           "record_bytes": rec * 8,
           "note": "per-pixel step trace, the alternative to the step's mask trace; "
                   "timed apart, not part of the step"}
    del st
    return out


def time_bins(path, max_list, flush, warmup, steps):
    """gs_bin_splats on the step's scene: the fixed-capacity bin lists that
    can replace emit + sort + ranges (capacity = the longest tile list
    rounded up to 32), timed alone."""
    import torch

    s, d, gsb = path.s, path.d, path.gs
    M = (max_list + 31) // 32 * 32
    out = (torch.empty((s.C, s.tile_height, s.tile_width, M), dtype=torch.int32, device=path.dev),
           torch.empty((s.C, s.tile_height, s.tile_width), dtype=torch.int32, device=path.dev))
    call = lambda: gsb.gs_bin_splats(d["means2d"], d["radii"], d["depths"], s.tile_size,
                                     s.tile_width, s.tile_height, M, d_status=path.status,
                                     out=out)
    for _ in range(warmup):
        call()
        flush.zero_()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        call()
        b.record()
        flush.zero_()
    torch.cuda.synchronize()
    gsb.check_status(path.status, "bins")
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    nb = s.C * s.tile_width * s.tile_height
    # fill: mean + radii per splat, one 4-byte id per intersection; sort: read
    # the id, gather 4 bytes of depth, write every slot (ids and -1s)
    return {"kernels": "k_bin_fill, k_bin_merge (+ k_bin_merge_large above 2048 per bin)",
            "ms": round(ms, 4), "capacity": M,
            "bytes": s.C * s.N * 16 + path.I * (4 + 4 + 4) + nb * M * 4,
            "note": "alternative to emit + sort + ranges; not part of the step"}


# -------------------------------------------------------- oracle arm


def oracle_camera_step(scene, c, g_rgb, g_a):
    """One step of the oracle on camera c of the workload: intersect + sort +
    offsets of its N splats (single-threaded C++), then the forward and the
    backward over every pixel of that camera (the OpenMP build of the same
    oracle, pixels handed out dynamically to every host core).  Returns
    (seconds, intersections, isect seconds)."""
    import oracle

    s = scene
    sl = slice(c, c + 1)
    t0 = time.perf_counter()
    tpg, keys, ids = oracle.isect_tiles(s.means2d[sl], s.radii[sl], s.depths[sl], 16,
                                        s.tile_width, s.tile_height)
    offsets = oracle.tile_offsets(keys, 1, s.tile_width, s.tile_height)
    t_isect = time.perf_counter() - t0
    fwd = oracle.rasterize_fwd(s.means2d[sl], s.conics[sl], s.colors[sl], s.opacities[sl], None,
                               None, s.width, s.height, 16, offsets, ids, s.alpha_cutoff,
                               s.transmittance_threshold, omp=True)
    oracle.rasterize_bwd(s.means2d[sl], s.conics[sl], s.colors[sl], s.opacities[sl], None, None,
                         s.width, s.height, 16, offsets, ids, s.alpha_cutoff,
                         fwd["render_alphas"], fwd["last_ids"], g_rgb[sl], g_a[sl], omp=True)
    return time.perf_counter() - t0, int(keys.size), t_isect


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(scene):
    """The oracle timed on the host cores: one camera of the workload through
    the whole path (see oracle_camera_step), about 2-10 s."""
    import oracle
    from tile_gaussian_splat_gb300 import scenes

    g_rgb, g_a = scenes.upstream_grads(scene.C, scene.height, scene.width, seed=1)
    sec, keys, t_isect = oracle_camera_step(scene, 0, g_rgb, g_a)
    px = scene.width * scene.height
    return {"value": round(px / sec / 1e6, 6), "unit": "Mpixel/s", "cores": oracle.threads_omp(),
            "kind": "oracle",
            "sample": f"oracle on camera 0 of {scene.C}: isect+sort+offsets of {scene.N} splats "
                      f"({keys} keys, 1 thread, {t_isect:.2f} s), forward + backward of all "
                      f"{px} pixels (OpenMP build, {oracle.threads_omp()} threads, dynamic "
                      f"schedule over pixels); {sec:.2f} s",
            "cpu": cpu_model(), "nproc": os.cpu_count()}


def run_reference(args, rank, world):
    """The oracle arm: each step runs the whole path on one camera of the
    workload (cameras in turn), isect single-threaded and the raster on every
    host core; the value is that camera's pixels over the step's own time."""
    if rank != 0:
        return None
    import oracle
    from tile_gaussian_splat_gb300 import scenes

    scene = scenes.workload3()
    s = scene
    # the workload's intersection count and longest list (set-up, not timed)
    _, keys, _ = oracle.isect_tiles(s.means2d, s.radii, s.depths, 16, s.tile_width,
                                    s.tile_height)
    offs = oracle.tile_offsets(keys, s.C, s.tile_width, s.tile_height).reshape(-1)
    I = int(keys.size)
    max_list = int(np.diff(np.append(offs.astype(np.int64), I)).max())
    del keys
    g_rgb, g_a = scenes.upstream_grads(s.C, s.height, s.width, seed=1)
    for k in range(args.warmup):
        oracle_camera_step(s, k % s.C, g_rgb, g_a)
    per_step = []
    for k in range(args.steps):
        sec, _, _ = oracle_camera_step(s, k % s.C, g_rgb, g_a)
        per_step.append(sec)
    sec = float(np.mean(per_step))
    px = s.width * s.height
    value = px / sec / 1e6
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "Mpixel/s (whole step: isect+sort+ranges+fwd+bwd)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded workload 3 generator)",
        "config": workload_config(s, I, max_list, 1),
        "cpu_baseline": {"value": round(value, 6), "unit": "Mpixel/s",
                         "cores": oracle.threads_omp(), "kind": "oracle",
                         "sample": f"each step: one camera of {s.C} in turn ({s.N} splats, "
                                   f"{px} pixels): isect+sort+offsets single-threaded, "
                                   f"forward + backward on {oracle.threads_omp()} threads "
                                   "(OpenMP, dynamic schedule over pixels)",
                         "cpu": cpu_model(), "nproc": os.cpu_count()},
        "e2e": {"value": round(value, 6), "unit": "Mpixel/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--main-only", action="store_true",
                    help="time the step alone: no projection, bin-list, step-trace or "
                         "workload 2/4/5 lines (profiling runs)")
    ap.add_argument("--workload", type=int, default=3, choices=[2, 3, 4],
                    help="3 is the measured workload; 2 and 4 serve profiling")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        from tile_gaussian_splat_gb300 import scenes
        sc = scenes.workload(args.workload)
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline and args.workload == 3:
            # before any CUDA work: the oracle runs in this process
            cpu = cpu_baseline(sc)
        line = run_ours(args, rank, world, sc)
        if line is not None:
            line["cpu_baseline"] = cpu
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
