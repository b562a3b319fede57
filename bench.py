"""Throughput of the tile-binned Gaussian-splat raster path on one GB300.

One step = one pass of the whole path over the 4-camera x 1M-splat 1920x1080
workload (workload 3): size query + intersection/sort (gs_isect_tiles),
tile ranges (gs_tile_offsets), forward (gs_rasterize_fwd) and backward
(gs_rasterize_bwd, upstream gradients N(0,1)).  All calls go through the
C ABI; inputs are resident in HBM; L2 is flushed between steps outside the
step's CUDA events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle on bounded samples of the same
workload (host cores; there is no other implementation of this path).
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

METRIC = "Msplat-isect/s + Mpixel/s fwd(+bwd) at 1 GB300; % HBM / FP32-SFU roofline"
WORKLOADS = {
    2: "w2: 1 camera x 100,000 splats, 1024x1024, tile 16, elliptical radii",
    3: "w3: 4 cameras x 1,000,000 splats, 1920x1080, tile 16, elliptical radii",
    4: "w4: 1 camera x 6,000,000 splats, 3840x2160, tile 16, elliptical radii",
}
WORKLOAD = WORKLOADS[3]
SM_COUNT = 152
FP32_LANES = 128
SM_MAX_MHZ = 2070.0
L2_FLUSH_BYTES = 256 << 20

# algorithmic FP32-pipe operations (FMA = 1) per pair, counted from the
# per-pixel formulas of the compositing and its adjoint
FWD_OPS_EVAL = 15     # dx, dy, quadratic form (9), o*exp, clamp, two tests
FWD_OPS_COMP = 7      # T*alpha, 3 colour FMAs, 1-alpha, T update, threshold test
BWD_OPS_EVAL = 15     # re-evaluation of alpha for every entry up to last_id
BWD_OPS_VALID = 40    # recovery, colour/opacity/mean/conic terms, recurrences


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
    counts = torch.zeros((s.C, s.height, s.width, 3), dtype=torch.int32, device=dev)
    path.forward(pair_counts=counts)
    n_eval = int(counts[..., 0].sum(dtype=torch.int64))
    n_comp = int(counts[..., 1].sum(dtype=torch.int64))
    bwd_eval = int(counts[..., 2].sum(dtype=torch.int64))
    offs = path.offsets.reshape(-1).to(torch.int64)
    ends = torch.cat([offs[1:], torch.tensor([path.I], device=dev)])
    list_len = (ends - offs)
    max_list = int(list_len.max())

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
    e2e = max_over_ranks(path.run_e2e(max(5, min(args.steps, 20))), world, dev)

    proj = time_projection(dev, flush, max(args.warmup, 3), max(5, min(args.steps, 20)))
    bins = time_bins(path, max_list, flush, max(args.warmup, 3), max(5, min(args.steps, 20)))

    if rank != 0:
        return None

    hbm_peak, peak_kind = _peaks()
    proj.update(achieved_gbs=round(proj["bytes"] / (proj["ms"] * 1e-3) / 1e9, 1))
    proj["frac"] = round(proj["achieved_gbs"] / hbm_peak, 4)
    bins.update(achieved_gbs=round(bins["bytes"] / (bins["ms"] * 1e-3) / 1e9, 1))
    bins["frac"] = round(bins["achieved_gbs"] / hbm_peak, 4)
    st = stage_ms.mean(axis=0)
    names = ["isect_query", "isect_emit_sort", "tile_ranges", "raster_fwd", "raster_bwd"]
    CN, I = s.C * s.N, path.I
    tiles = s.C * s.tile_width * s.tile_height
    from tile_gaussian_splat_gb300 import binding as gsb
    key_bits = gsb.gs_tile_bits(s.tile_width, s.tile_height) + max(0, (s.C - 1).bit_length())
    up_passes = (key_bits + 7) // 8
    # algorithmic bytes: what each stage must read and write
    # emit+sort: rects + depth histograms (read mean, radii, depth; write a
    # 16-byte rect) 36 B/splat; depth sort 12 + 3 x 16 B/splat; emission
    # (order + rect gather) 20 B/splat and an 8-byte key+id per intersection;
    # camera|tile passes 16 B per intersection each, the last one 24 B (read
    # 8, write the 12-byte output, gather 4 bytes of depth)
    tile_pass_bytes = (16 * (up_passes - 1) + 24) if up_passes else 24
    bytes_ = {
        "isect_query": CN * (8 + 8 + 4),
        "isect_emit_sort": CN * (36 + 60 + 20) + I * (8 + tile_pass_bytes),
        "tile_ranges": I * 8 + tiles * 4,
    }
    clk = clocks.summary()
    mhz = SM_MAX_MHZ
    alu_peak = SM_COUNT * FP32_LANES * mhz * 1e6
    fwd_ops = FWD_OPS_EVAL * n_eval + FWD_OPS_COMP * n_comp
    bwd_ops = BWD_OPS_EVAL * bwd_eval + BWD_OPS_VALID * n_comp
    stages = {}
    for i, n in enumerate(names):
        e = {"ms": round(float(st[i]), 4)}
        if n in bytes_:
            gbs = bytes_[n] / (st[i] * 1e-3) / 1e9
            e.update(bound="hbm", achieved_gbs=round(gbs, 1), frac=round(gbs / hbm_peak, 4))
        elif n == "raster_fwd":
            a = fwd_ops / (st[i] * 1e-3)
            e.update(bound="alu", achieved_tops=round(a / 1e12, 3), frac=round(a / alu_peak, 4),
                     mpix_s=round(pixels / (st[i] * 1e-3) / 1e6, 1))
        else:
            a = bwd_ops / (st[i] * 1e-3)
            e.update(bound="alu", achieved_tops=round(a / 1e12, 3), frac=round(a / alu_peak, 4),
                     mpix_s=round(pixels / (st[i] * 1e-3) / 1e6, 1))
        stages[n] = e
    isect_ms = float(st[0] + st[1] + st[2])
    dom = names[int(np.argmax(st))]
    src = {"raster_fwd": "tile_gaussian_splat_gb300/csrc/raster.cu",
           "raster_bwd": "tile_gaussian_splat_gb300/csrc/raster.cu"}.get(
        dom, "tile_gaussian_splat_gb300/csrc/sort.cu")
    traffic = _traffic_for({"raster_fwd": "k_raster_fwd", "raster_bwd": "k_raster_bwd"}.get(
        dom, dom), 1)
    if dom in ("raster_fwd", "raster_bwd"):
        roof = {"bound": "alu", "kernel": "k_" + dom, "achieved": stages[dom]["achieved_tops"],
                "peak": round(alu_peak / 1e12, 2), "unit": "Tops/s (FP32 pipe, FMA=1)",
                "frac": stages[dom]["frac"], "traffic": traffic,
                "peak_source": "152 SMs x 128 FP32 lanes x 2070 MHz"}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": stages[dom]["achieved_gbs"],
                "peak": hbm_peak, "unit": "GB/s", "frac": stages[dom]["frac"],
                "traffic": traffic, "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})"}
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
        "data": "synthetic (seeded workload 3 generator)",
        "config": {"workload": WORKLOADS[args.workload], "C": s.C, "N": s.N, "width": s.width,
                   "height": s.height, "tile_size": 16, "n_isects": I,
                   "max_tile_list": max_list, "pixels_per_step": pixels,
                   "l2": "flushed between steps (256 MB write outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "msplat_isect_per_s": round(I / (isect_ms * 1e-3) / 1e6, 1),
        "mpixel_per_s_fwd": stages["raster_fwd"]["mpix_s"],
        "mpixel_per_s_bwd": stages["raster_bwd"]["mpix_s"],
        "stages": stages,
        "work": {"pairs_evaluated_fwd": n_eval, "pairs_composited": n_comp,
                 "pairs_evaluated_bwd": bwd_eval},
        "roofline": roof,
        "project": proj,
        "bins": bins,
        "e2e": {"value": round(whole_job_rate(pixels, e2e, world) / 1e6, 2),
                "unit": "Mpixel/s (pinned host inputs -> image + gradients on host, "
                        "uploads/downloads overlapped with the previous/next step)",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e, 3)},
        # per step: count, count word, rects + depth histograms, 4 depth
        # passes, emit, the camera/tile passes, ranges, forward, backward
        "gpu_launches": args.steps * (1 + 1 + 1 + 4 + 1 + up_passes + 1 + 1 + 1),
        "clocks": clk,
        "wall_s_timed": round(t_wall, 3),
    }
    return line


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
    return {"kernels": "k_bin_fill, k_bin_sort", "ms": round(ms, 4), "capacity": M,
            "bytes": s.C * s.N * 16 + path.I * (4 + 4 + 4) + nb * M * 4,
            "note": "alternative to emit + sort + ranges; not part of the step"}


# -------------------------------------------------------- oracle arm


def cpu_sample(scene, budget_tiles=1000, seed=0):
    """Times the oracle on a bounded sample of the workload: intersect + sort +
    offsets of camera 0 (all its splats), forward + backward on budget_tiles
    tiles spread over that camera.  Returns (seconds per full step estimate,
    description)."""
    import oracle
    from tile_gaussian_splat_gb300 import scenes

    s = scene
    c = 0
    m, r, dpt = s.means2d[c:c + 1], s.radii[c:c + 1], s.depths[c:c + 1]
    t0 = time.perf_counter()
    tpg, keys, ids = oracle.isect_tiles(m, r, dpt, 16, s.tile_width, s.tile_height)
    offsets = oracle.tile_offsets(keys, 1, s.tile_width, s.tile_height)
    t_isect = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    ntiles = s.tile_width * s.tile_height
    tiles = rng.choice(ntiles, min(budget_tiles, ntiles), replace=False)
    pix = []
    for t in tiles:
        ty, tx = divmod(int(t), s.tile_width)
        for y in range(ty * 16, min(s.height, ty * 16 + 16)):
            for x in range(tx * 16, min(s.width, tx * 16 + 16)):
                pix.append(y * s.width + x)
    pix = np.array(pix, np.int64)
    g_rgb, g_a = scenes.upstream_grads(1, s.height, s.width, seed=1)
    arrs = dict(means2d=m, conics=s.conics[c:c + 1], colors=s.colors[c:c + 1],
                opacities=s.opacities[c:c + 1])
    t0 = time.perf_counter()
    fwd = oracle.rasterize_fwd(arrs["means2d"], arrs["conics"], arrs["colors"],
                               arrs["opacities"], None, None, s.width, s.height, 16, offsets, ids,
                               s.alpha_cutoff, s.transmittance_threshold, pixels=pix)
    oracle.rasterize_bwd(arrs["means2d"], arrs["conics"], arrs["colors"], arrs["opacities"],
                         None, None, s.width, s.height, 16, offsets, ids, s.alpha_cutoff,
                         fwd["render_alphas"], fwd["last_ids"], g_rgb, g_a, pixels=pix)
    t_raster = time.perf_counter() - t0
    pixels = s.C * s.width * s.height
    est = t_isect * s.C + t_raster / pix.size * pixels
    desc = (f"oracle, 1 thread: isect+sort+offsets of camera 0 ({s.N} splats, {keys.size} "
            f"keys) in {t_isect:.2f} s, x{s.C} cameras; fwd+bwd of {pix.size} pixels "
            f"({tiles.size} random tiles) in {t_raster:.2f} s, scaled to {pixels} pixels")
    return est, desc


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from tile_gaussian_splat_gb300 import scenes

    scene = scenes.workload3()
    pixels = scene.C * scene.width * scene.height
    for _ in range(max(args.warmup, 3) if args.warmup else 0):
        cpu_sample(scene, budget_tiles=8)
    per_step = []
    desc = ""
    for k in range(args.steps):
        est, desc = cpu_sample(scene, budget_tiles=24, seed=k)
        per_step.append(est)
    sec = float(np.mean(per_step))
    value = pixels / sec / 1e6
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "Mpixel/s (whole step: isect+sort+ranges+fwd+bwd)",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded workload 3 generator)",
        "config": {"workload": WORKLOAD, "C": scene.C, "N": scene.N, "width": scene.width,
                   "height": scene.height, "tile_size": 16},
        "cpu_baseline": {"value": round(value, 6), "unit": "Mpixel/s", "cores": 1,
                         "kind": "oracle", "sample": desc},
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
            # before any CUDA work: the oracle runs in this process, single thread
            est, desc = cpu_sample(sc)
            cpu = {"value": round(sc.C * sc.width * sc.height / est / 1e6, 6),
                   "unit": "Mpixel/s", "cores": 1, "kind": "oracle", "sample": desc}
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
