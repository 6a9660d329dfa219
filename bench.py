#!/usr/bin/env python3
"""Benchmark of the implicit-GEMM convolution path on GB300.

One step = one pass of the workload's hot path over one batch of synthetic
input.  The default workload, ``baseline``, is every convolution the
benchmark configurations name, at full size, one after the other:

  tiny_bf16         bf16 16x16x16 -> 16, 3x3 s1 p1
  resnet_bf16       bf16 32x56x56x64 -> 64, 3x3 s1 p1, + 1.0*source
  resnet_down_bf16  bf16 32x56x56x64 -> 32x28x28x128, 3x3 s2 p1
  fp8_res           e4m3 16x64x64x320 -> 320 (bf16 out), 3x3 FCRS s1 p1, + 0.5*source
  vae_silu_bf16     bf16 1x256x256x512 -> 512, 3x3 s1 p1, SiLU
  vae_head_bf16     bf16 1x512x512x128 -> 3, 3x3 s1 p1
  convT_f16         f16 transposed 8x32x32x256 -> 8x64x64x128, 4x4 RSFC s2 p1, ReLU
  fwd5x5_f16        f16 8x128x128x128 -> 8x64x64x128, 5x5 s2 p2

Each conv runs as a stream of back-to-back launches over rotating copies of
all its tensors (input, packed filter, source, output) that together exceed
3 x L2, so that every launch reads its operands from HBM (inputs larger than
L2 in place of a flush); the stream is bracketed by CUDA events on the launch
stream and the per-launch time is its event time over the launches.  The
tiny conv, too small for that within 64 copies, streams over 64 copies right
after an L2 flush (a write of max(2 x L2, 256 MiB), outside its events): no
launch's operands have been touched since the flush.  Each conv's events
follow one untimed launch of the same conv (of its stream's last copy,
before the flush for the tiny conv), so its code is warm while its operands
come from HBM.  The step time is the sum of the convs' per-launch times; ``per_kernel``
also reports each conv alone after a flush, right after a different conv
(``us_isolated``: that includes the launch latency a stream hides and the
kernel's code fetched cold).
``value`` is the step's algorithmic FLOPs over the step time (whole job: all
ranks' FLOPs over the slowest rank's time); ``per_kernel`` gives each conv's
time, TFLOP/s, GB/s and fraction of its own roofline; ``roofline`` is the
dominant conv's (the one with the largest share of the step).  Filters are
packed once before timing (pack_us).  Other workloads: ``resnet_block`` (the
3x3 residual conv then the stride-2 downsample, back to back after one flush
per step) or any single workload name.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload baseline|resnet_block|<one of synthetic.WORKLOADS>]

--impl reference times the CPU oracle (single-threaded fp64 direct loops) on
a bounded sample of the same workload per step, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "conv TFLOP/s per dtype/shape and % of GB300 dense tensor peak (GB/s if mem-bound)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["transposed_conv_implicit_gb300/csrc/conv_kernel.cuh",
                  "transposed_conv_implicit_gb300/csrc/ptx.cuh",
                  "transposed_conv_implicit_gb300/csrc/conv_params.h",
                  "transposed_conv_implicit_gb300/csrc/conv_api.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_kernels.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_kernels_gather.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_launch.cuh",
                  "transposed_conv_implicit_gb300/csrc/conv_direct.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_rowtap.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_kernels_pair.cu",
                  "transposed_conv_implicit_gb300/csrc/conv_kernels_sk.cu",
                  "transposed_conv_implicit_gb300/csrc/segment_copy.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                data = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = data.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if isinstance(v, (int, float)):
                    out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def workload_cases(name):
    from transposed_conv_implicit_gb300 import synthetic
    if name == "baseline":
        return [synthetic.WORKLOADS[n] for n in synthetic.BASELINE_SET]
    if name == "resnet_block":
        return [synthetic.WORKLOADS[n] for n in synthetic.RESNET_BLOCK]
    return [synthetic.WORKLOADS[name]]


def workload_dtype(cases) -> str:
    dtypes = sorted(set(c.dtype for c in cases))
    return dtypes[0] if len(dtypes) == 1 else "/".join(dtypes) + " (per conv, fp32 accumulate)"


def flush_each_conv(name) -> bool:
    """The baseline set times every conv on its own, after its own flush."""
    return name == "baseline"


def describe(cases):
    parts = []
    for c in cases:
        kind = "convT" if c.kind == "transposed" else "conv"
        s = "%s %s %dx%dx%dx%d -> %dx%dx%dx%d %dx%d s%d p%d" % (
            c.dtype, kind, c.N, c.H, c.W, c.C_in, c.N, c.Ho, c.Wo, c.C_out, c.R, c.S, c.stride, c.pad)
        if c.groups > 1:
            s += " groups=%d" % c.groups
        if c.has_residual:
            s += " +%.2g*src" % c.beta
        if c.epilogue != "none":
            s += " " + c.epilogue
        parts.append(s)
    return "; ".join(parts)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self._reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._reader.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle timing
def decode_inputs(cases, inputs):
    """The oracle's fp64 view of each case's input, filter and source."""
    import oracle
    dec = []
    for case, inp in zip(cases, inputs):
        dec.append((oracle.decode(_bits(inp["x"]), case.dtype),
                    oracle.decode(_bits(inp["w"]), case.dtype),
                    oracle.decode(_bits(inp["src"]), case.out_dtype) if inp["src"] is not None
                    else None))
    return dec


def oracle_sample_seconds(cases, inputs, budget_s):
    """Time the oracle (as it stands) on seeded output pixels (all channels)
    of every conv of the workload, repeated while `budget_s` lasts.
    Returns (flops, seconds, pixels per conv)."""
    import numpy as np
    dec = decode_inputs(cases, inputs)
    rng = np.random.default_rng(4321)
    t0 = time.perf_counter()
    oracle_points_step(cases, dec, 4, rng)
    per_pix = max((time.perf_counter() - t0) / 4, 1e-9)
    npix = max(1, int(budget_s / 4 / per_pix))
    flops = 0
    pixels = 0
    t0 = time.perf_counter()
    while True:
        flops += oracle_points_step(cases, dec, npix, rng)
        pixels += npix
        if time.perf_counter() - t0 >= budget_s:
            break
    return flops, time.perf_counter() - t0, pixels


def oracle_points_step(cases, dec, npix, rng):
    """One reference-arm step: the oracle evaluates `npix` output pixels (all
    channels) of each case, at seeded random positions."""
    import numpy as np
    import oracle
    flops = 0
    for case, (x, w, src) in zip(cases, dec):
        total_pix = case.N * case.Ho * case.Wo
        pix = rng.integers(0, total_pix, size=npix)
        pts = (pix[:, None] * case.C_out + np.arange(case.C_out)[None, :]).reshape(-1)
        _oracle_points(case, x, w, src, pts)
        flops += 2 * npix * case.C_out * case.R * case.S * case.C_in
    return flops


def _bits(t):
    from transposed_conv_implicit_gb300 import synthetic
    return synthetic.raw_bits(t)


def _oracle_points(case, x, w, src, pts):
    import oracle
    st, pd = (case.stride,) * 2, case.pads
    if case.kind == "transposed":
        return oracle.conv_transposed_points(x, w, pts, out_hw=(case.Ho, case.Wo), stride=st,
                                             padding=pd, source=src, beta=case.beta,
                                             act=case.epilogue)
    return oracle.conv2d_fwd_points(x, w, pts, filter_is_fcrs=case.filter_layout == "FCRS",
                                    stride=st, padding=pd, dilation=case.dilations, source=src,
                                    beta=case.beta, act=case.epilogue, groups=case.groups)


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = os.environ.get("BENCH_DIST_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_max(value: float, world: int, device) -> float:
    """Max of a host float over all ranks (host-side timing reduction only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(step_ms, flops_per_step: float, world: int, device):
    """(ms per step, whole-job TFLOP/s) from this rank's timed steps.

    Every rank runs the same steps on its own replica, so the job processed
    world x steps x flops_per_step; the time is the slowest rank's."""
    total_ms = dist_max(float(sum(step_ms)), world, device)
    steps = len(step_ms)
    return total_ms / steps, flops_per_step * world * steps / (total_ms * 1e-3) / 1e12


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from transposed_conv_implicit_gb300 import synthetic
    cases = workload_cases(args.workload)
    inputs = [synthetic.make_inputs(c) for c in cases]
    dec = decode_inputs(cases, inputs)
    rng = np.random.default_rng(1234)
    # Size the per-step sample so the whole run stays within about two minutes.
    t0 = time.perf_counter()
    oracle_points_step(cases, dec, 8, rng)
    per_pix = (time.perf_counter() - t0) / 8
    budget = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    npix = max(1, int(budget / max(per_pix, 1e-9)))
    for _ in range(args.warmup):
        oracle_points_step(cases, dec, npix, rng)
    flops = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += oracle_points_step(cases, dec, npix, rng)
    secs = time.perf_counter() - t0
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": workload_dtype(cases), "data": "synthetic",
        "config": {"workload": args.workload + ": " + describe(cases),
                   "sample": "%d output pixels x all channels per conv per step" % npix},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": "%d seeded output pixels (all channels) of each conv per step, "
                                   "fp64 single-threaded direct loops" % npix},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm
def conv_bound(case, peaks):
    """(bound, tensor peak TFLOP/s) of one conv: HBM when its arithmetic
    intensity is below the ridge of its dtype's tensor peak, else tensor.
    fp8 takes twice the measured bf16 peak (the nominal dense ratio)."""
    tensor_peak = peaks["bf16_tflops"] * (2.0 if case.dtype == "f8e4m3" else 1.0)
    ridge = tensor_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return ("hbm" if case.flops / case.bytes < ridge else "tensor"), tensor_peak


def run_ours(args, world, rank, local):
    import torch
    import transposed_conv_implicit_gb300 as cg
    from transposed_conv_implicit_gb300 import synthetic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cases = workload_cases(args.workload)
    inputs = [synthetic.make_inputs(c) for c in cases]
    stream = torch.cuda.current_stream(dev)
    per_conv_flush = flush_each_conv(args.workload)

    # Device-resident tensors, packed filters, bound launches.
    calls, outs, packed = [], [], []
    pack_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    dev_inputs = []
    for case, inp in zip(cases, inputs):
        x = inp["x"].to(dev)
        w = inp["w"].to(dev)
        src = inp["src"].to(dev) if inp["src"] is not None else None
        dev_inputs.append((x, w, src))
    pack_ev[0].record(stream)
    for case, (x, w, src) in zip(cases, dev_inputs):
        st, pd = (case.stride,) * 2, case.pads
        if case.kind == "transposed":
            packed.append(cg.conv_transposed_pack_filter(w, stride=st, padding=pd))
        else:
            packed.append(cg.conv2d_pack_filter(w, filter_is_fcrs=case.filter_layout == "FCRS"))
    pack_ev[1].record(stream)
    # A workspace with room for stream-K partials (the planner then uses that
    # schedule where it expects a gain).
    workspace = cg.new_workspace(cg.CONV_STATUS_BYTES + cg.conv_streamk_workspace_size(), dev)

    def bind(case, x, pk, src, out):
        st, pd = (case.stride,) * 2, case.pads
        kw = dict(r=case.R, s=case.S, stride=st, has_residual=case.has_residual, source=src,
                  beta=case.beta, epilogue=case.epilogue, workspace=workspace, stream=stream)
        if case.kind == "transposed":
            return cg.bind_conv_transposed_packed(x, pk, out, padding=pd, **kw)
        return cg.bind_conv2d_fwd_packed(x, pk, out, symmetric_padding=pd, dilation=case.dilations,
                                         num_groups=case.groups, **kw)

    for case, (x, w, src), pk in zip(cases, dev_inputs, packed):
        out = torch.empty(case.out_shape, dtype=synthetic.TORCH_DTYPES[case.out_dtype], device=dev)
        outs.append(out)
        calls.append(bind(case, x, pk, src, out))
    torch.cuda.synchronize(dev)
    pack_us = pack_ev[0].elapsed_time(pack_ev[1]) * 1e3

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    # Baseline set: each conv runs as a stream of back-to-back launches over
    # rotating copies of all its tensors (input, packed filter, source,
    # output) that together exceed 3 x L2, so every launch reads its operands
    # from HBM; the per-launch time is the stream's event time over the
    # launches.  A conv too small for that within 64 copies streams over 64
    # copies right after an L2 flush: each launch still reads operands that
    # nothing has touched since the flush.
    rotate_sets, flush_first = [], []
    if per_conv_flush:
        for i, case in enumerate(cases):
            x, w, src = dev_inputs[i]
            per_copy = case.bytes
            ncopy = max(1, math.ceil(3 * l2 / per_copy))
            flush_first.append(ncopy > 64)
            ncopy = min(ncopy, 64)
            group = [calls[i]]
            for _ in range(ncopy - 1):
                o = torch.empty_like(outs[i])
                group.append(bind(case, x.clone(), packed[i].clone(),
                                  src.clone() if src is not None else None, o))
            rotate_sets.append(group)
        torch.cuda.synchronize(dev)

    def new_events():
        n = len(calls) if per_conv_flush else 1
        return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n)]

    def step(evs):
        """One step.  Baseline set: each conv's stream of launches (or its one
        launch after a flush) inside its own events.  Otherwise: one flush,
        then the convs back to back inside one pair of events (a conv may set
        up while the previous one drains: programmatic dependent launch)."""
        if per_conv_flush:
            # Each conv's events follow one untimed launch of the same conv,
            # so its kernel's code is warm (after another kernel, and with L2
            # flushed, that code would be fetched from HBM: up to ~8 us on
            # the tiny conv); its operands still come from HBM.
            for i, (e0, e1) in enumerate(evs):
                group = rotate_sets[i]
                group[-1]()
                if flush_first[i]:
                    flush.fill_(1)
                e0.record(stream)
                for call in group:
                    call()
                e1.record(stream)
        else:
            flush.fill_(1)
            evs[0][0].record(stream)
            for call in calls:
                call()
            evs[0][1].record(stream)

    def launches_of(i):
        return len(rotate_sets[i]) if per_conv_flush else 1

    warm_ev = new_events()
    for _ in range(args.warmup):
        step(warm_ev)
    torch.cuda.synchronize(dev)
    status, bits = cg.conv_check_device_status(workspace)
    if status != 0:
        raise RuntimeError("device status after warm-up: %s (bits %d)" % (cg.conv_status_string(status), bits))

    # Timed region: K steps, flushes outside the events.
    ev = [new_events() for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 or world > 1 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for k in range(args.steps):
        step(ev[k])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    dist_barrier(world)
    clocks = sampler.stop() if sampler else None
    status, bits = cg.conv_check_device_status(workspace)
    if status != 0:
        raise RuntimeError("device status after timing: %s (bits %d)" % (cg.conv_status_string(status), bits))

    isolated_ms = None
    if per_conv_flush:
        # Per-launch time of conv i in step k; a step's time is their sum.
        per_kernel_ms = [[ev[k][i][0].elapsed_time(ev[k][i][1]) / launches_of(i)
                          for k in range(args.steps)] for i in range(len(calls))]
        step_ms = [sum(per_kernel_ms[i][k] for i in range(len(calls))) for k in range(args.steps)]
        # For reference: every conv alone between events right after a flush
        # (this includes the launch latency a stream of launches hides).
        reps = 20
        iev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in calls] for _ in range(reps)]
        for k in range(reps):
            for i, call in enumerate(calls):
                flush.fill_(1)
                iev[k][i][0].record(stream)
                call()
                iev[k][i][1].record(stream)
        torch.cuda.synchronize(dev)
        isolated_ms = [statistics.median(iev[k][i][0].elapsed_time(iev[k][i][1]) for k in range(reps))
                       for i in range(len(calls))]
    else:
        step_ms = [sum(a.elapsed_time(b) for a, b in ev[k]) for k in range(args.steps)]
        # Per-kernel durations (for the roofline): every launch bracketed by
        # its own events on the launch stream, each step after an L2 flush.
        kreps = max(10, min(args.steps, 100))
        kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
               for _ in range(kreps)]
        for k in range(kreps):
            flush.fill_(1)
            for i, call in enumerate(calls):
                kev[k][i].record(stream)
                call()
            kev[k][len(calls)].record(stream)
        torch.cuda.synchronize(dev)
        per_kernel_ms = [[kev[k][i].elapsed_time(kev[k][i + 1]) for k in range(kreps)]
                         for i in range(len(calls))]
    ms_per_step, value = whole_job_value(step_ms, sum(c.flops for c in cases), world, dev)

    # Host cost of one bound C-ABI call (ctypes with pre-marshalled arguments,
    # the library's prepared-call cache lookup and the launch), and the wall
    # time from the call to a completed synchronize.
    host_us, sync_us = [], []
    for call in calls:
        ts = []
        for rep in range(60):
            t0 = time.perf_counter()
            call()
            ts.append(time.perf_counter() - t0)
            if rep % 10 == 9:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        host_us.append(statistics.median(ts[10:]) * 1e6)
        ts = []
        for rep in range(20):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            call()
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - t0)
        sync_us.append(statistics.median(ts[5:]) * 1e6)

    # Roofline of the dominant kernel (largest share of the step) and every
    # conv's fraction of its own bound.
    mean_k = [statistics.fmean(v) for v in per_kernel_ms]
    dom = max(range(len(cases)), key=lambda i: mean_k[i])
    peaks, peak_src = load_peaks()
    per_kernel = {}
    for i, c in enumerate(cases):
        us = mean_k[i] * 1e3
        bound, tpeak = conv_bound(c, peaks)
        tf = c.flops / (us * 1e-6) / 1e12
        gbs = c.bytes / (us * 1e-6) / 1e9
        floor_us = max(c.bytes / (peaks["hbm_gbs"] * 1e9), c.flops / (tpeak * 1e12)) * 1e6
        per_kernel[c.name] = {
            "us": round(us, 3), "tflops": round(tf, 2), "gbs": round(gbs, 1),
            "bound": bound if floor_us >= 1.0 else "launch",
            "frac": round(gbs / peaks["hbm_gbs"] if bound == "hbm" else tf / tpeak, 4),
            "frac_hbm": round(gbs / peaks["hbm_gbs"], 4), "frac_tensor": round(tf / tpeak, 4),
            "tensor_peak_tflops": tpeak,
            "p10_us": round(_pct(per_kernel_ms[i], 10) * 1e3, 3),
            "p90_us": round(_pct(per_kernel_ms[i], 90) * 1e3, 3),
            "host_us_per_call": round(host_us[i], 2), "call_to_sync_us": round(sync_us[i], 2),
            "traffic": lookup_traffic(c.name)}
        if per_conv_flush:
            n = launches_of(i)
            per_kernel[c.name]["timing"] = (
                "stream of %d back-to-back launches over rotating copies (%d MB in all%s)"
                % (n, n * c.bytes >> 20, ", after an L2 flush" if flush_first[i] else ""))
            per_kernel[c.name]["us_isolated"] = round(isolated_ms[i] * 1e3, 3)
    dcase = cases[dom]
    dbound, dpeak = conv_bound(dcase, peaks)
    if dbound == "hbm":
        roof = {"bound": "hbm", "achieved": dcase.bytes / (mean_k[dom] * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": dcase.flops / (mean_k[dom] * 1e-3) / 1e12,
                "peak": dpeak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = peak_src
    roof["peak_kind"] = "burst (each conv timed on its own)" if dbound == "tensor" else "copy"
    roof["kernel"] = dcase.name
    roof["traffic"] = lookup_traffic(dcase.name)

    e2e = run_e2e(args, cases, inputs, dev, stream) if not args.no_e2e else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        flops, secs, pixels = oracle_sample_seconds(cases, inputs, args.cpu_budget)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
               "sample": "%d seeded output pixels (all channels) of each of the %d convs, fp64 "
                         "single-threaded direct loops, %.1f s" % (pixels, len(cases), secs)}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": workload_dtype(cases),
        "data": "synthetic",
        "config": {"workload": args.workload + ": " + describe(cases),
                   "l2": ("inputs larger than L2: each conv streams over rotating copies of "
                          "its tensors totalling >= 3 x L2 (%d MiB); a conv too small for that "
                          "within 64 copies streams over 64 copies after a flush (write of %d "
                          "MiB) outside its events; each "
                          "conv's events follow one untimed launch of the same conv (its code "
                          "warm, its operands not)"
                          % (3 * l2 >> 20, flush.numel() >> 20)) if per_conv_flush else
                         "flushed before every step (write of %d MiB), flush outside the events"
                         % (flush.numel() >> 20),
                   "step_time": "sum over the convs of their per-launch event time" if per_conv_flush
                                else "events around the whole step",
                   "filters": "packed once before timing",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "gpu": props.name, "sms": props.multi_processor_count},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(launches_of(i) + (1 if per_conv_flush else 0)
                            for i in range(len(calls))) * args.steps,
        "step_us_p10_p90": [round(_pct(step_ms, 10) * 1e3, 2), round(_pct(step_ms, 90) * 1e3, 2)],
        "clocks": clocks,
        "pack_us": round(pack_us, 2),
        "per_kernel": per_kernel,
        "wall_s": round(wall, 3),
        "kernel_hash": kernel_source_hash(),
    }
    print(json.dumps(line))
    return 0


def _pct(vals, p):
    s = sorted(vals)
    return s[min(len(s) - 1, max(0, int(round(p / 100.0 * (len(s) - 1)))))]


def lookup_traffic(kernel_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    if data.get("kernel_hash") != kernel_source_hash():
        return None
    entry = data.get("kernels", {}).get(kernel_name)
    return entry.get("dram_bytes_per_launch") if entry else None


def run_e2e(args, cases, inputs, dev, stream):
    """End to end through the public API: every step copies its inputs from
    pinned host memory to the device, runs the convolutions and copies the
    outputs back to pinned host memory.  Steps are pipelined as a serving loop
    would run them: a copy-in stream, the compute stream and a copy-out stream
    with two sets of device tensors, so step k+1's inputs and step k-1's
    outputs cross the host link while step k computes.  (One stream per
    tensor copy measured the same: ~174 GB/s host to device is the link.)"""
    import torch
    import transposed_conv_implicit_gb300 as cg
    from transposed_conv_implicit_gb300 import synthetic
    nbuf = 2
    host_in, host_out, packed = [], [], []
    dev_in = [[] for _ in range(nbuf)]
    dev_out = [[] for _ in range(nbuf)]
    h2d = d2h = 0
    for case, inp in zip(cases, inputs):
        hx = inp["x"].pin_memory()
        hs = inp["src"].pin_memory() if inp["src"] is not None else None
        host_in.append((hx, hs))
        for b in range(nbuf):
            dev_in[b].append((torch.empty_like(hx, device=dev),
                              torch.empty_like(hs, device=dev) if hs is not None else None))
            dev_out[b].append(torch.empty(case.out_shape, dtype=synthetic.TORCH_DTYPES[case.out_dtype],
                                          device=dev))
        h2d += hx.numel() * hx.element_size() + (hs.numel() * hs.element_size() if hs is not None else 0)
        o = dev_out[0][-1]
        host_out.append(torch.empty(o.shape, dtype=o.dtype, pin_memory=True))
        d2h += o.numel() * o.element_size()
        w = inp["w"].to(dev)
        st, pd = (case.stride,) * 2, case.pads
        if case.kind == "transposed":
            packed.append(cg.conv_transposed_pack_filter(w, stride=st, padding=pd))
        else:
            packed.append(cg.conv2d_pack_filter(w, filter_is_fcrs=case.filter_layout == "FCRS"))
    ws = cg.new_workspace(cg.CONV_STATUS_BYTES + cg.conv_streamk_workspace_size(), dev)
    n_in = n_out = 1
    s_ins = [torch.cuda.Stream(dev) for _ in range(n_in)]
    s_outs = [torch.cuda.Stream(dev) for _ in range(n_out)]
    s_in, s_out = s_ins[0], s_outs[0]
    s_comp = stream
    in_done = [torch.cuda.Event() for _ in range(nbuf)]
    comp_done = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def one_step(k):
        b = k % nbuf
        pairs = []
        for (hx, hs), (dx, ds) in zip(host_in, dev_in[b]):
            pairs.append((dx, hx))
            if hs is not None:
                pairs.append((ds, hs))
        for i, (d, h) in enumerate(pairs):
            si = s_ins[i % n_in]
            with torch.cuda.stream(si):
                if used[b]:
                    si.wait_event(comp_done[b])  # the buffer's previous convs have read it
                d.copy_(h, non_blocking=True)
        for si in s_ins[1:]:
            ev = torch.cuda.Event()
            ev.record(si)
            s_in.wait_event(ev)
        in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        if used[b]:
            s_comp.wait_event(out_done[b])  # the buffer's previous outputs are on the host
        for case, (dx, ds), pk, o in zip(cases, dev_in[b], packed, dev_out[b]):
            st, pd = (case.stride,) * 2, case.pads
            kw = dict(r=case.R, s=case.S, stride=st, has_residual=case.has_residual, source=ds,
                      beta=case.beta, epilogue=case.epilogue, workspace=ws, stream=s_comp)
            if case.kind != "transposed":
                kw["dilation"] = case.dilations
                kw["num_groups"] = case.groups
            if case.kind == "transposed":
                cg.conv_transposed_packed(dx, pk, o, padding=pd, **kw)
            else:
                cg.conv2d_fwd_packed(dx, pk, o, symmetric_padding=pd, **kw)
        comp_done[b].record(s_comp)
        for i, (o, ho) in enumerate(zip(dev_out[b], host_out)):
            so = s_outs[i % n_out]
            with torch.cuda.stream(so):
                so.wait_event(comp_done[b])
                ho.copy_(o, non_blocking=True)
        for so in s_outs[1:]:
            ev = torch.cuda.Event()
            ev.record(so)
            s_out.wait_event(ev)
        out_done[b].record(s_out)
        used[b] = True

    for k in range(max(1, args.warmup)):
        one_step(k)
    torch.cuda.synchronize(dev)
    steps = max(1, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_comp)
    for sx in s_ins + s_outs:
        sx.wait_event(e0)
    for k in range(steps):
        one_step(k)
    for b in range(nbuf):  # the timed region ends when every output is on the host
        s_comp.wait_event(out_done[b])
    e1.record(s_comp)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    status, bits = cg.conv_check_device_status(ws)
    if status != 0:
        raise RuntimeError("device status after e2e: %s" % cg.conv_status_string(status))
    flops = sum(c.flops for c in cases)
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipeline": "copy-in, compute and copy-out streams, two sets of device tensors"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="baseline")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
