"""Benchmark of the packed RoPE attention forward (libpk) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config NAME]

One step = one pk_attend call (tile scheduler + attention kernel) over the whole workload.
The default workload is the largest of the five configurations that fits one GPU, the long
packed batch (H=16, bf16, log-normal lengths of median 256 clipped to [1, 8192], packed to
T = 131072 tokens, RoPE base 160000, every key); --config picks another of tiny / global /
local / long / short.

Reported (one JSON line on rank 0):
  value       useful TFLOP/s: 256 x (query, key) pairs the window lets through x heads,
              divided by the device time of the K timed steps (CUDA events on the launch
              stream, inputs resident in HBM);
  e2e         the same metric through the C ABI with host buffers: each step copies qkv,
              tables and cu from pinned host memory, runs, and copies out and lse back;
  roofline    the attention kernel alone (events the library records around it) against
              the measured HBM copy bandwidth (or the bf16 tensor peak when FLOPs bind);
  cpu_baseline the fp64 oracle on the host cores over a bounded sample of the workload.
Between timed steps the L2 (129 MB) cannot serve the inputs: steps rotate over several
copies of the input and output buffers whose total is well above the L2 size.

--impl reference times the oracle (the slow CPU statement of the method) as the reference
arm, on the same workload and metric.

--op rope and --op backward time the standalone rotation (pk_rope: GB/s against the measured
HBM copy rate) and the backward pass (pk_attend_backward: useful TFLOP/s at 640 flop per
visible pair) on the same workloads; the default --op attend is the forward above.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed RoPE attention fwd: useful TFLOP/s & tokens/s on 1 GB300; % of roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of the attention kernel per launch from an ncu capture, valid only while the
# kernel's sources have the recorded hash (kernel_source_hash; otherwise reported as null).
NCU_TRAFFIC = {  # {config_name: (kernel_source_hash() of the captured kernel, bytes per launch)}
    # pk_attend_tc_kernel on the long batch (profiles/pk_attend_tc_kernel_long.md)
    "long": ("2e6a5db189da945cdacae7f6da011250fa218392", 1067494144),
    # pk_attend_band_kernel on the short-sequence workload (profiles/pk_attend_band_kernel_short.md)
    "short": ("7e911277ba6985bdc10e830c5b59631600b83deb", 382067200),
}


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's); x itself at one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


KERNEL_NAMES = {0: "pk_attend_band_kernel", 1: "pk_attend_f32_kernel", 2: "pk_attend_tc_kernel",
                3: "pk_attend_q4_kernel", 4: "pk_attend_tc_kernel (single-record items)",
                5: "pk_attend_split_kernel"}
# the source file of each forward kernel (enum pk_kernel)
KERNEL_SOURCES = {0: "pk_attend_band.cu", 1: "pk_attend_f32.cu", 2: "pk_attend_tc.cu", 3: "pk_attend_q4.cu",
                  4: "pk_attend_tc.cu", 5: "pk_attend_split.cu"}


def kernel_source_hash(kernel: int = 2) -> str:
    """sha1 over what a forward kernel is built from: its source, the device headers and the
    build flags."""
    h = hashlib.sha1()
    for rel in (("csrc", KERNEL_SOURCES[kernel]), ("csrc", "pk_dev.cuh"), ("csrc", "pk_attn_common.cuh"),
                ("build.py",)):
        with open(os.path.join(ROOT, "rope_cu_tile_gb300", *rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def input_sets(wl) -> int:
    """How many copies of the input and output buffers the timed steps rotate through, so
    that no step finds its inputs in the 129 MB L2 (1 when one set is already larger than
    twice the L2)."""
    e = synth.elem_size(wl.dtype)
    set_bytes = wl.T * 3 * wl.H * 64 * e + wl.T * wl.H * 64 * e + 4 * wl.H * wl.T
    return max(1, min(8, int(np.ceil(3 * L2_BYTES / set_bytes)))) if set_bytes < 2 * L2_BYTES else 1


def l2_note(wl) -> str:
    n = input_sets(wl)
    if n == 1:
        return "inputs larger than L2"
    return (f"rotating {n} input/output sets ({n} x {(wl.T * 3 * wl.H * 64 * synth.elem_size(wl.dtype)) / 1e6:.0f} "
            f"MB qkv) so no step finds its inputs in the 129 MB L2")


def work(wl):
    pairs = synth.visible_pairs(wl.lens, wl.window) * wl.H
    return 256.0 * pairs, synth.algorithmic_bytes(wl)


# ------------------------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        loaded = [x for x in sm if x >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# the oracle on the host cores


def _oracle_first(orc, wl, n):
    """Run the oracle on the first n sequences (all heads); (seconds, useful flops, tokens)."""
    lens = wl.lens[:n]
    T = int(lens.sum())
    cu = synth.cu_from_lens(lens)
    P = max(1, int(lens.max()))
    t0 = time.perf_counter()
    orc.attend(wl.qkv[:T], wl.cos[:P], wl.sin[:P], cu, wl.H, wl.window, wl.scale, wl.dtype)
    return time.perf_counter() - t0, 256.0 * synth.visible_pairs(lens, wl.window) * wl.H, T


def oracle_sample(orc, wl, budget_s):
    """How many leading sequences the oracle finishes in about budget_s seconds (estimated
    from a small calibration run)."""
    n = min(wl.S, max(1, orc.threads() // max(1, wl.H) + 1))
    dt, flops, _ = _oracle_first(orc, wl, n)
    rate = flops / max(dt, 1e-9)
    cum = np.cumsum([256.0 * synth.visible_pairs([L], wl.window) * wl.H for L in wl.lens])
    return int(min(wl.S, max(n, np.searchsorted(cum, rate * budget_s) + 1)))


def cpu_baseline(wl, budget_s=12.0, n=None):
    """The fp64 oracle, as it stands, over the first sequences of the workload (all heads),
    as many as fit in about budget_s seconds of host time."""
    import oracle

    orc = oracle.get()
    if n is None:
        n = oracle_sample(orc, wl, budget_s)
    dt, flops, T = _oracle_first(orc, wl, n)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": orc.threads(), "kind": "oracle",
            "sample": f"first {n} of {wl.S} sequences ({T} tokens, all {wl.H} heads), fp64, "
                      f"{dt:.2f} s wall", "seconds": dt, "tokens_per_s": T / dt}


# ------------------------------------------------------------------------------------------
# the CUDA path


def device_tensors(wl, torch, dev):
    def t(a):
        if wl.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        if wl.dtype == "f16":
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)

    return t(wl.qkv), t(wl.cos), t(wl.sin), torch.from_numpy(wl.cu.astype(np.int64).astype(np.int32)).to(dev)


def run_gpu(wl, steps, warmup, rank, world, dev_index, tuned=True):
    import torch

    import rope_cu_tile_gb300 as pk

    pk.load()
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flops, abytes = work(wl)
    e = synth.elem_size(wl.dtype)
    nsets = input_sets(wl)
    max_len = int(wl.lens.max())
    qkv0, cos, sin, cu = device_tensors(wl, torch, dev)
    td = qkv0.dtype
    sets = []
    for k in range(nsets):
        q = qkv0 if k == 0 else qkv0.clone()
        sets.append((q, torch.empty((wl.T, wl.H * 64), dtype=td, device=dev),
                     torch.empty((wl.H, wl.T), dtype=torch.float32, device=dev)))
    torch.cuda.synchronize()

    def step(i):
        q, o, l = sets[i % nsets]
        pk.attend(q, cos, sin, cu, wl.H, wl.window, wl.scale, out=o, lse=l, stream=stream, max_len=max_len,
                  tuned=tuned)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    if pk.last_status(stream) != 0:
        raise RuntimeError("device error during warm-up")
    kernel = (pk.pk_tune_pick(pk.dtype_code(qkv0), wl.H, wl.window, wl.T, max_len) if tuned
              else pk.pk_forward_kernel(pk.dtype_code(qkv0), wl.window))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev_index) as clk:
        # the step time: K steps with nothing between the calls (per-kernel events would break
        # the overlap of the scheduler with the attention kernel's set-up)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(steps):
                step(warmup + i)
            ev1.record(stream)
        torch.cuda.synchronize()
        # the kernels' own durations: the same K steps again with CUDA events around each
        # kernel on the launch stream (the library records them)
        pk.profile_start(steps)
        with torch.cuda.stream(stream):
            for i in range(steps):
                step(warmup + steps + i)
        torch.cuda.synchronize()
        sched_ms, attend_ms, calls = pk.profile_stop()
    ms = ev0.elapsed_time(ev1)
    if pk.last_status(stream) != 0:
        raise RuntimeError("device error during timed steps")
    ms = max_over_ranks(ms, world)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    h_qkv = torch.from_numpy(np.ascontiguousarray(wl.qkv).view(np.int16 if e == 2 else np.float32)).pin_memory()
    h_cos = torch.from_numpy(np.ascontiguousarray(wl.cos).view(np.int16 if e == 2 else np.float32)).pin_memory()
    h_sin = torch.from_numpy(np.ascontiguousarray(wl.sin).view(np.int16 if e == 2 else np.float32)).pin_memory()
    h_cu = torch.from_numpy(wl.cu.astype(np.int64).astype(np.int32)).pin_memory()
    h_out = torch.empty((wl.T, wl.H * 64), dtype=torch.int16 if e == 2 else torch.float32).pin_memory()
    h_lse = torch.empty((wl.H, wl.T), dtype=torch.float32).pin_memory()
    # two device buffer sets so that step i + 1's inputs travel in while step i computes and
    # step i - 1's results travel out: copy-in, compute and copy-out streams ordered by events
    sets2 = []
    for _ in range(2):
        sets2.append(dict(
            qkv=torch.empty(h_qkv.shape, dtype=h_qkv.dtype, device=dev),
            cos=torch.empty(h_cos.shape, dtype=h_cos.dtype, device=dev),
            sin=torch.empty(h_sin.shape, dtype=h_sin.dtype, device=dev),
            cu=torch.empty(h_cu.shape, dtype=torch.int32, device=dev),
            out=torch.empty(h_out.shape, dtype=h_out.dtype, device=dev),
            lse=torch.empty(h_lse.shape, dtype=torch.float32, device=dev),
            copied=torch.cuda.Event(), computed=torch.cuda.Event(), read=torch.cuda.Event()))
    h2d = h_qkv.numel() * h_qkv.element_size() + 2 * h_cos.numel() * h_cos.element_size() + 4 * h_cu.numel()
    d2h = h_out.numel() * h_out.element_size() + 4 * h_lse.numel()
    code = pk.dtype_code(qkv0)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sh = pk._stream_handle(stream)

    def e2e_step(i):
        b = sets2[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(b["computed"])  # the step that used these buffers two steps ago
            b["qkv"].copy_(h_qkv, non_blocking=True)
            b["cos"].copy_(h_cos, non_blocking=True)
            b["sin"].copy_(h_sin, non_blocking=True)
            b["cu"].copy_(h_cu, non_blocking=True)
            b["copied"].record(s_in)
        stream.wait_event(b["copied"])
        stream.wait_event(b["read"])  # its results of two steps ago have been read out
        if tuned:
            rc = pk.pk_attend_tuned(code, b["qkv"].data_ptr(), b["cos"].data_ptr(), b["sin"].data_ptr(),
                                    b["cu"].data_ptr(), wl.S, wl.T, wl.H, wl.window, float(wl.scale), max_len,
                                    b["out"].data_ptr(), b["lse"].data_ptr(), sh)
        else:
            rc = pk.pk_attend_dt(code, b["qkv"].data_ptr(), b["cos"].data_ptr(), b["sin"].data_ptr(),
                                 b["cu"].data_ptr(), wl.S, wl.T, wl.H, wl.window, float(wl.scale),
                                 b["out"].data_ptr(), b["lse"].data_ptr(), sh)
        if rc:
            raise RuntimeError(f"forward call -> {rc}")
        b["computed"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["computed"])
            h_out.copy_(b["out"], non_blocking=True)
            h_lse.copy_(b["lse"], non_blocking=True)
            b["read"].record(s_out)

    e_steps = max(3, min(steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s_in)
    stream.wait_event(f0)
    for i in range(e_steps):
        e2e_step(2 + i)
    f1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = f0.elapsed_time(f1) / e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)

    return {"ms_per_step": ms / steps, "attend_ms": attend_ms / max(calls, 1),
            "schedule_ms": sched_ms / max(calls, 1), "calls": calls, "flops": flops, "bytes": abytes,
            "nsets": nsets, "clocks": clk.summary(), "e2e_ms": e2e_ms, "h2d": int(h2d), "d2h": int(d2h),
            "kernel": kernel}


def run_rope(wl, steps, warmup, dev_index, dims=64):
    """The standalone rotation (pk_rope) over the workload's packed qkv, out of place: q and k
    rotated, v copied. Algorithmic bytes: qkv read once and written once, plus the tables."""
    import torch

    import rope_cu_tile_gb300 as pk

    pk.load()
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    e = synth.elem_size(wl.dtype)
    qkv0, _, _, cu = device_tensors(wl, torch, dev)
    P = max(1, int(wl.lens.max()))
    c, s = synth.rope_tables_dims(P, dims, wl.base)
    cos = device_tensors(dataclasses.replace(wl, cos=synth.to_storage(c, wl.dtype)), torch, dev)[1]
    sin = device_tensors(dataclasses.replace(wl, cos=synth.to_storage(s, wl.dtype)), torch, dev)[1]
    qkv_bytes = wl.T * 3 * wl.H * 64 * e
    abytes = 2 * qkv_bytes + 2 * P * (dims // 2) * e + 4 * (wl.S + 1)
    nsets = max(1, min(8, int(np.ceil(3 * L2_BYTES / (2 * qkv_bytes))))) if 2 * qkv_bytes < 2 * L2_BYTES else 1
    sets = [(qkv0 if k == 0 else qkv0.clone(), torch.empty_like(qkv0)) for k in range(nsets)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    def step(i):
        x, y = sets[i % nsets]
        pk.rope(x, cos, sin, cu, wl.H, dims, False, False, out=y, status=status, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev_index) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for i in range(steps):
                step(warmup + i)
            ev1.record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device error in pk_rope")
    ms = ev0.elapsed_time(ev1) / steps
    return {"ms": ms, "bytes": abytes, "nsets": nsets, "clocks": clk.summary(), "dims": dims}


def run_backward(wl, steps, warmup, dev_index):
    """pk_attend_backward on the workload (the forward's out and lse computed once, outside the
    timed region; a fixed random dout). Useful FLOP: 640 per visible pair (S, dP, dV, dQ, dK)."""
    import torch

    import rope_cu_tile_gb300 as pk

    pk.load()
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    qkv, cos, sin, cu = device_tensors(wl, torch, dev)
    with torch.cuda.stream(stream):
        out, lse = pk.attend(qkv, cos, sin, cu, wl.H, wl.window, wl.scale, stream=stream)
        g = torch.Generator(device=dev).manual_seed(5)
        dout = torch.randn(out.shape, generator=g, device=dev).to(out.dtype)
        dqkv = torch.empty_like(qkv)
    torch.cuda.synchronize()

    def step():
        pk.attend_backward(qkv, cos, sin, cu, wl.H, wl.window, wl.scale, out, lse, dout, dqkv=dqkv, stream=stream,
                           max_len=int(wl.lens.max()))

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev_index) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(steps):
                step()
            ev1.record(stream)
        torch.cuda.synchronize()
    if pk.last_status(stream) != 0:
        raise RuntimeError("device error in pk_attend_backward")
    return {"ms": ev0.elapsed_time(ev1) / steps, "clocks": clk.summary()}


def roofline(wl, attend_ms, peaks, peak_src, kernel=2):
    flops, abytes = work(wl)
    t_bw = abytes / (peaks["hbm_gbs"] * 1e9)
    t_fl = flops / (peaks["bf16_tflops"] * 1e12)
    if t_fl > t_bw:
        achieved = flops / (attend_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s"}
    else:
        achieved = abytes / (attend_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s"}
    r["frac"] = achieved / peak
    r["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    h, tr = NCU_TRAFFIC.get(wl.name, (None, None))
    r["traffic"] = tr if (h is not None and h == kernel_source_hash(kernel)) else None
    r["t_roof_us"] = max(t_bw, t_fl) * 1e6
    r["kernel"] = KERNEL_NAMES.get(kernel, str(kernel))
    return r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="long", choices=list(synth.CONFIG_NAMES))
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--kernel", default="auto", choices=["auto", "tc", "tc_single", "q4", "f32", "split"],
                    help="auto: pk_attend_tuned picks (default); otherwise pk_attend with that kernel "
                         "(tc, tc_single, q4: 16-bit inputs; f32, split: fp32 inputs; windows of 1..16 "
                         "always run the band kernel)")
    ap.add_argument("--storage", default=None, choices=["bf16", "f16", "f32"],
                    help="store the workload's qkv and tables in this type instead of its own (same lengths, "
                         "heads, window, tables and seed)")
    ap.add_argument("--op", default="attend", choices=["attend", "rope", "backward"],
                    help="attend: the attention path (default); rope: the standalone rotation; "
                         "backward: pk_attend_backward")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and "RANK" not in os.environ:
        world = 1
    wl = synth.make_config(args.config)
    workload = f"{args.config}: {synth.CONFIG_TEXT[args.config]}"
    if args.storage is not None and args.storage != wl.dtype:
        wl = synth.make_lens_workload(f"{args.config}_{args.storage}", wl.lens, args.storage, H=wl.H, window=wl.window,
                                      base=wl.base, seed=synth.CONFIG_NAMES.index(args.config))
        workload += f" (stored as {args.storage})"
    flops, abytes = work(wl)
    cfg = {"workload": workload, "T": wl.T, "S": wl.S, "H": wl.H,
           "D": 64, "window": wl.window, "scale": wl.scale, "seed": synth.CONFIG_NAMES.index(args.config),
           "useful_gflop": flops / 1e9, "algorithmic_mb": abytes / 1e6,
           "l2": l2_note(wl), "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        # each step: the same bounded sample, sized so that the whole run takes ~2 minutes
        n = oracle_sample(oracle.get(), wl, 120.0 / (args.warmup + args.steps))
        vals = []
        cb = None
        for i in range(args.warmup + args.steps):
            cb = cpu_baseline(wl, n=n)
            if i >= args.warmup:
                vals.append(cb["value"])
        v = statistics.median(vals)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["seconds"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cb["cores"], "kind": "oracle",
                                 "sample": cb["sample"]},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if args.op == "rope":
        if rank != 0:
            return
        r = run_rope(wl, args.steps, args.warmup, local)
        peaks, psrc = load_peaks()
        gbs = r["bytes"] / (r["ms"] * 1e-3) / 1e9
        cfg.update({"op": "pk_rope (q and k rotated, v copied, out of place)", "dims": r["dims"],
                    "algorithmic_mb": r["bytes"] / 1e6,
                    "l2": f"rotating {r['nsets']} input/output sets" if r["nsets"] > 1 else "inputs larger than L2"})
        cfg.pop("useful_gflop", None)
        line = {"metric": "pk_rope: GB/s on 1 GB300; % of HBM roofline", "value": gbs, "unit": "GB/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
                "data": "synthetic", "config": cfg,
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / peaks["hbm_gbs"], "peak_source": psrc, "traffic": None,
                             "kernel": "pk_rope_kernel"},
                "gpu_launches": args.steps, "clocks": r["clocks"]}
        print(json.dumps(line))
        return
    if args.op == "backward":
        if rank != 0:
            return
        r = run_backward(wl, args.steps, args.warmup, local)
        peaks, psrc = load_peaks()
        bflops = 2.5 * flops  # 640 against the forward's 256 per visible pair
        tfs = bflops / (r["ms"] * 1e-3) / 1e12
        cfg.update({"op": "pk_attend_backward (dqkv from dout; forward's out and lse precomputed)",
                    "useful_gflop": bflops / 1e9})
        line = {"metric": "pk_attend_backward: useful TFLOP/s on 1 GB300; % of roofline", "value": tfs,
                "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
                "data": "synthetic", "config": cfg,
                "roofline": {"bound": "tensor", "achieved": tfs, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": tfs / peaks["bf16_tflops"], "peak_source": psrc, "traffic": None,
                             "kernel": "pk_bwd_mma_kernel" if wl.dtype != "f32" else "pk_bwd_main_kernel"},
                "gpu_launches": 4 * args.steps, "clocks": r["clocks"]}
        print(json.dumps(line))
        return
    if world > 1:
        import torch.distributed as dist
        import torch
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.kernel != "auto":
        os.environ["PK_ATTN"] = args.kernel
    r = run_gpu(wl, args.steps, args.warmup, rank, world, local, tuned=args.kernel == "auto")
    peaks, psrc = load_peaks()
    value = world * flops / (r["ms_per_step"] * 1e-3) / 1e12
    tokens_s = world * wl.T / (r["ms_per_step"] * 1e-3)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic", "config": cfg,
            "tokens_per_s": tokens_s,
            "roofline": roofline(wl, r["attend_ms"], peaks, psrc, r["kernel"]),
            "kernel": {"picked": KERNEL_NAMES.get(r["kernel"], str(r["kernel"])),
                       "by": ("pk_attend_tuned (timed once per shape key during warm-up)" if args.kernel == "auto"
                              else f"--kernel {args.kernel}")},
            "step_roofline_frac": (max(abytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
                                   / (r["ms_per_step"] * 1e-3)),
            "kernel_ms": {"preparation (tile scheduler or cu check)": r["schedule_ms"], "attention": r["attend_ms"],
                          "timing": "a second pass of the same steps with CUDA events around each kernel"},
            "e2e": {"value": world * flops / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"]},
            "gpu_launches": 2 * args.steps, "clocks": r["clocks"]}
    if rank == 0:
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
