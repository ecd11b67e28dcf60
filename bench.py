#!/usr/bin/env python3
"""Throughput of the multi-adapter LoRA delta on GB300, as one JSON line.

A step is one pass of the whole hot path over one batch: build the routing
metadata, the packed forward (shrink + expand, H saved) and the packed
backward (dH, dB, dA, dX), all through the C ABI.  The workload is the packed
training batch 4096->4096, N=8 adapters of ranks {8,16,16,32,32,64,64,128},
4 x 1024 tokens each (T = 32768), bf16 with fp32 accumulation; its inputs
(x and dY 268 MB each, y 268 MB) are larger than L2, so no flush is needed
between steps.  The decode batch (256 tokens over 8 adapters of rank 32,
three projections) is timed beside it for the SGMV-decode GB/s figure.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica of the workload (the path
shards by batch with no exchange); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "packed multi-LoRA fwd+bwd tokens/s"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20


# ---------------------------------------------------------------------------- accounting
def step_bytes(spec: wl.Spec) -> dict:
    """Algorithmic HBM bytes per call: each activation read once per pass, y / dX
    read and written, adapter weights read once per pass, dA / dB written once,
    H written by the forward and read by the backward."""
    T, di, do = spec.n_tokens, spec.d_in, spec.d_out
    counts = np.bincount(spec.ids, minlength=spec.n_adapters)
    th = int((counts * spec.ranks).sum())           # sum_i T_i r_i
    w = int(spec.sum_r) * (di + do)                 # adapter weight elements
    fwd = 2 * T * di + 4 * T * do + 2 * w + 4 * th
    bwd = 2 * T * do + 2 * T * di + 4 * T * di + 4 * th + 2 * w + 4 * w
    return {"fwd": fwd, "bwd": bwd}


# kernels of a step in launch order (forward, then backward with H saved), and
# the kernel template each one runs
STEP_KERNELS = (("shrink", "tc_rowproj"), ("expand", "tc_colproj"), ("hconv", "h_to_bf16"), ("dB", "tc_tokred"),
                ("dh", "tc_rowproj"), ("dA", "tc_tokred"), ("dX", "tc_colproj"))


def kernel_bytes(spec: wl.Spec) -> dict:
    """Algorithmic HBM bytes of each kernel launch of a step: its activations
    read once, y / dX read and written, its adapter weights read once, H / dH
    (r_i columns) written or read once, dA / dB written once."""
    T, di, do = spec.n_tokens, spec.d_in, spec.d_out
    counts = np.bincount(spec.ids, minlength=spec.n_adapters)
    th = int((counts * spec.ranks).sum())           # sum_i T_i r_i
    r = int(spec.sum_r)
    rw = 64 if spec.r_max <= 64 else 128
    return {"shrink": 2 * T * di + 2 * r * di + 4 * th, "expand": 4 * T * do + 2 * r * do + 4 * th,
            "hconv": 4 * T * int(spec.r_max) + 2 * T * rw,
            "dh": 2 * T * do + 2 * r * do + 4 * th, "dB": 2 * T * do + 4 * th + 4 * r * do,
            "dA": 2 * T * di + 4 * th + 4 * r * di, "dX": 4 * T * di + 2 * r * di + 4 * th}


def step_flops(spec: wl.Spec) -> int:
    counts = np.bincount(spec.ids, minlength=spec.n_adapters)
    th = int((counts * spec.ranks).sum())
    return 6 * th * (spec.d_in + spec.d_out)


def decode_bytes(spec: wl.Spec) -> int:
    """x read, y read + written, weights of the adapters present read once."""
    present = np.unique(spec.ids)
    r = int(spec.ranks[present].sum())
    return 2 * spec.n_tokens * spec.d_in + 4 * spec.n_tokens * spec.d_out + 2 * r * (spec.d_in + spec.d_out)


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e datasheet figure, for context beside the measured copy bandwidth


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def traffic_record(kernel: str, n_tokens: int):
    """DRAM bytes per launch from a committed ncu summary of the same kernel on
    the same workload size, when it still matches the kernel's source (else
    None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("tokens") != n_tokens:
        return None
    import hashlib

    src = os.path.join(ROOT, rec["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return rec["bytes_per_launch"] if h == rec.get("source_sha") else None


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, mem, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                if len(f) > 9:
                    mem.append(float(f[9]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "mem_mhz": statistics.median(mem) if mem else None, "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm
class Workload:
    def __init__(self, spec: wl.Spec, dev):
        import torch

        import adapter_sgmv_gb300 as lora

        self.spec, self.dev = spec, dev
        self.inp = wl.device_inputs(spec, dev, y0="randn", dX0="zero")
        self.table = lora.AdapterTable(self.inp["A"], self.inp["B"], spec.ranks.tolist(),
                                       torch.from_numpy(spec.scales), spec.d_in, spec.d_out)
        self.offsets = torch.from_numpy(spec.seg_offsets).to(dev) if spec.sorted else None
        self.ids = None if spec.sorted else torch.from_numpy(spec.ids).to(dev)
        nb = lora.lora_segments_bytes(spec.n_tokens, spec.n_adapters)
        self.seg_storage = torch.empty(nb, dtype=torch.uint8, device=dev)
        self.ws = lora.workspace(self.table, spec.n_tokens, dev)
        T = spec.n_tokens
        self.y = self.inp["y0"]
        self.H = torch.empty((T, spec.r_max), dtype=torch.float32, device=dev)
        self.dX = self.inp["dX0"]
        self.dA = torch.empty((spec.sum_r, spec.d_in), dtype=torch.float32, device=dev)
        self.dB = torch.empty((spec.sum_r, spec.d_out), dtype=torch.float32, device=dev)
        self.side = lora.SideStreams(dev)  # the backward's dB / dA run on these beside dh / dX
        self.deterministic = False  # dA / dB summed in a fixed span order (lora_packed_bwd_ex)
        self.segs = None

    def build(self, stream=None):
        import adapter_sgmv_gb300 as lora

        self.segs = lora.lora_build_segments(ids=self.ids, seg_offsets=self.offsets, n_tokens=self.spec.n_tokens,
                                             n_adapters=self.spec.n_adapters, storage=self.seg_storage,
                                             stream=stream)

    def fwd(self, stream=None, x=None, events=None):
        """Packed forward; with ``events`` the marked call records them around
        its kernels (events[2k], events[2k + 1] bracket kernel k)."""
        import adapter_sgmv_gb300 as lora

        x = self.inp["x"] if x is None else x
        if events is None:
            lora.lora_packed_fwd(self.y, self.H, x, self.table, self.segs, self.ws, stream=stream)
        else:
            lora.lora_packed_fwd_marked(self.y, self.H, x, self.table, self.segs, self.ws, events, stream=stream)

    def bwd(self, stream=None, x=None, dY=None, events=None):
        import adapter_sgmv_gb300 as lora

        x = self.inp["x"] if x is None else x
        dY = self.inp["dY"] if dY is None else dY
        if events is None and self.deterministic:
            lora.lora_packed_bwd_ex(self.dX, self.dA, self.dB, dY, x, self.H, self.table, self.segs, self.ws,
                                    side=self.side, deterministic=True, stream=stream)
        elif events is None:
            lora.lora_packed_bwd_concurrent(self.dX, self.dA, self.dB, dY, x, self.H, self.table, self.segs, self.ws,
                                            self.side, stream=stream)
        else:
            lora.lora_packed_bwd_marked(self.dX, self.dA, self.dB, dY, x, self.H, self.table, self.segs, self.ws,
                                        events, stream=stream)


def kernels_per_step(spec: wl.Spec) -> int:
    """Kernels the library launches per step (builder + forward + backward)."""
    T, N = spec.n_tokens, spec.n_adapters
    one_block = 2 * T + 32 * N + 2 * (N + 1) <= 200 * 1024 // 4  # ids, perm and counts in shared memory
    build = 1 if (spec.sorted and N <= 4095) or (not spec.sorted and one_block) else 6
    return build + 2 + 5  # forward: shrink, expand; backward: H to bf16, dB, dh, dA, dX


def time_steps(work: Workload, steps: int, warmup: int, stream, per_kernel: bool = False):
    """Warm-up, then `steps` timed steps between two events on `stream`.
    Returns (start, end, call events per step, kernel event pairs per step);
    with per_kernel the library records an event pair around every kernel
    of the packed calls (same kernels, same stream)."""
    import torch

    for _ in range(warmup):
        work.build(stream)
        work.fwd(stream)
        work.bwd(stream)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(STEP_KERNELS))] for _ in range(steps)]
    if per_kernel:  # create the events outside the timed region
        for row in kev:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        ev[k][0].record(stream)
        work.build(stream)
        ev[k][1].record(stream)
        work.fwd(stream, events=kev[k][:4] if per_kernel else None)
        ev[k][2].record(stream)
        work.bwd(stream, events=kev[k][4:] if per_kernel else None)
        ev[k][3].record(stream)
    end.record(stream)
    return start, end, ev, (kev if per_kernel else None)


def kernel_times(work: Workload, steps: int, stream, hbm: float) -> dict:
    """Each kernel's mean duration over `steps` steps in which the library
    records an event pair around every kernel of the packed calls (the
    backward's kernels then run one after another on `stream`), with its
    algorithmic bytes and the fraction of the HBM peak they reach."""
    import torch

    _, _, _, kev = time_steps(work, steps, 1, stream, per_kernel=True)
    torch.cuda.synchronize()
    kb = kernel_bytes(work.spec)
    out = {}
    for j, (use, tmpl) in enumerate(STEP_KERNELS):
        ms = statistics.mean(row[2 * j].elapsed_time(row[2 * j + 1]) for row in kev)
        gbs = kb[use] / (ms * 1e-3) / 1e9
        out[use] = {"kernel": tmpl, "ms": round(ms, 4), "bytes": kb[use], "GB/s": round(gbs, 1),
                    "frac_of_hbm": round(gbs / hbm, 4)}
    return out


def time_config(spec: wl.Spec, dev, stream, steps: int = 10, warmup: int = 3, sequential: bool = False) -> dict:
    """One full step (build + fwd + bwd) of another workload: ms and tokens/s.
    With `sequential`, the same step is also timed as one single-adapter step
    per adapter (N builds, N forwards, N backwards) for the packing speed-up."""
    import torch

    work = Workload(spec, dev)
    start, end, _, _ = time_steps(work, steps, warmup, stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    by = step_bytes(spec)
    hbm, _, _ = measured_peaks()
    out = {"tokens": spec.n_tokens, "ms_per_step": round(ms, 4), "tokens/s": round(spec.n_tokens / (ms * 1e-3), 1),
           "GB/s": round((by["fwd"] + by["bwd"]) / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm": round((by["fwd"] + by["bwd"]) / (ms * 1e-3) / 1e9 / hbm, 4),
           "kernels_ms": kernel_times(work, steps, stream, hbm)}
    del work
    torch.cuda.empty_cache()
    if sequential:
        subs = []
        for i in range(spec.n_adapters):
            n = int((spec.ids == i).sum())
            if n:
                subs.append(Workload(wl.custom(f"{spec.name}_a{i}", spec.d_in, spec.d_out, [spec.ranks[i]],
                                               [spec.alphas[i]], np.zeros(n, np.int32), seed=i), dev))
        for _ in range(warmup):
            for w in subs:
                w.build(stream), w.fwd(stream), w.bwd(stream)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(steps):
            for w in subs:
                w.build(stream), w.fwd(stream), w.bwd(stream)
        s1.record(stream)
        torch.cuda.synchronize()
        seq = s0.elapsed_time(s1) / steps
        out["sequential_ms_per_step"] = round(seq, 4)
        out["packing_speedup"] = round(seq / ms, 3)
        del subs
        torch.cuda.empty_cache()
    return out


def time_e2e(work: Workload, steps: int, warmup: int, stream):
    """Same step with the activations coming from pinned host memory and the
    adapter gradients going back to it, every copy inside the timed region.
    As a training loop would, the next step's inputs are copied (two copy
    streams, 4 chunks per tensor) into a second device buffer set while the
    current step computes; each step's gradients are read back after its
    backward."""
    import torch

    hx = work.inp["x"].cpu().pin_memory()
    hdy = work.inp["dY"].cpu().pin_memory()
    hdA = torch.empty(work.dA.shape, dtype=work.dA.dtype).pin_memory()
    hdB = torch.empty(work.dB.shape, dtype=work.dB.dtype).pin_memory()
    dxs = [torch.empty_like(work.inp["x"]) for _ in range(2)]
    ddys = [torch.empty_like(work.inp["dY"]) for _ in range(2)]
    copy_streams = [torch.cuda.Stream(stream.device) for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]   # set i holds the next step's inputs
    consumed = [torch.cuda.Event() for _ in range(2)]  # set i is no longer read by a backward
    n_chunks = 4

    def h2d(i):
        """host -> set i on the copy streams, after the step that last read set i"""
        for cs in copy_streams:
            cs.wait_event(consumed[i])
        for src, dst in ((hx, dxs[i]), (hdy, ddys[i])):
            rows = src.shape[0]
            for c in range(n_chunks):
                r0, r1 = rows * c // n_chunks, rows * (c + 1) // n_chunks
                with torch.cuda.stream(copy_streams[c % 2]):
                    dst[r0:r1].copy_(src[r0:r1], non_blocking=True)
        # the compute stream starts the step once both copy streams are done
        e2 = torch.cuda.Event()
        copy_streams[1].record_event(e2)
        copy_streams[0].wait_event(e2)
        copy_streams[0].record_event(copied[i])

    def run(n):
        for i in range(2):
            consumed[i].record(stream)
        h2d(0)
        for k in range(n):
            i = k % 2
            stream.wait_event(copied[i])
            if k + 1 < n:
                h2d(1 - i)  # next step's inputs, overlapping this step's compute
            work.build(stream)
            work.fwd(stream, x=dxs[i])
            work.bwd(stream, x=dxs[i], dY=ddys[i])
            consumed[i].record(stream)
            with torch.cuda.stream(stream):
                hdA.copy_(work.dA, non_blocking=True)
                hdB.copy_(work.dB, non_blocking=True)

    run(warmup)
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for cs in copy_streams:
        cs.wait_event(s)
    run(steps)
    for cs in copy_streams:
        stream.wait_stream(cs)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    h2d_bytes = hx.numel() * hx.element_size() + hdy.numel() * hdy.element_size()
    d2h = hdA.numel() * hdA.element_size() + hdB.numel() * hdB.element_size()
    return ms, h2d_bytes, d2h


def time_decode(dev, stream, reps: int = 50):
    """SGMV decode (packed_fwd on the decode batch) per projection, L2-cold:
    a CUDA graph replays `reps` calls that rotate over enough independent
    buffer sets to exceed 3x L2."""
    import torch

    import adapter_sgmv_gb300 as lora

    hbm, _, _ = measured_peaks()
    out = {}
    for p in range(3):
        spec = wl.decode(p)
        nbytes = decode_bytes(spec)
        n_sets = max(2, int(3 * L2_BYTES / nbytes) + 1)
        ids = torch.from_numpy(spec.ids).to(dev)
        segs = lora.lora_build_segments(ids=ids, n_adapters=spec.n_adapters)
        sets = []
        for q in range(n_sets):
            s_q = wl.Spec(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids, False, seed=q,
                          with_bwd=False)
            inp = wl.device_inputs(s_q, dev, y0="randn", need=("A", "B", "x", "y0"))
            tab = lora.AdapterTable(inp["A"], inp["B"], spec.ranks.tolist(), torch.from_numpy(spec.scales),
                                    spec.d_in, spec.d_out)
            ws = lora.workspace(tab, spec.n_tokens, dev)
            sets.append((tab, inp["x"], inp["y0"], ws))
        for tab, x, y, ws in sets:  # warm-up, also outside capture
            lora.lora_packed_fwd(y, None, x, tab, segs, ws, stream=stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(reps):
                tab, x, y, ws = sets[k % n_sets]
                lora.lora_packed_fwd(y, None, x, tab, segs, ws, stream=stream)
        times = []
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            for _ in range(20):
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record(stream)
                g.replay()
                e.record(stream)
                e.synchronize()
                times.append(s.elapsed_time(e) / reps)
        ms = statistics.median(times)
        # single call, not graphed: launch latency included, one call at a time
        eager = []
        with torch.cuda.stream(stream):
            for k in range(20):
                tab, x, y, ws = sets[k % n_sets]
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record(stream)
                lora.lora_packed_fwd(y, None, x, tab, segs, ws, stream=stream)
                e.record(stream)
                e.synchronize()
                eager.append(s.elapsed_time(e))
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[f"{spec.d_in}x{spec.d_out}"] = {"us_per_call": round(ms * 1e3, 3), "bytes": nbytes,
                                            "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4),
                                            "us_per_call_eager": round(statistics.median(eager) * 1e3, 3)}
        del sets, g
        torch.cuda.empty_cache()
    return out


QWEN3_4B_SHARED_X = {"qkv": ((4096, 1024, 1024), 32), "gate_up": ((9728, 9728), 32)}


def time_decode_multi(dev, stream, reps: int = 50) -> dict:
    """A decode layer's projections that read the same x (Qwen3-4B: hidden
    2560 -> q 4096 / k 1024 / v 1024, and -> gate / up 9728), 256 one-token
    requests over 8 adapters of rank 32: one lora_multi_fwd call against one
    lora_packed_fwd call per projection, each replayed from a CUDA graph over
    rotating buffer sets larger than 3x L2 (as in time_decode)."""
    import torch

    import adapter_sgmv_gb300 as lora

    hbm, _, _ = measured_peaks()
    out = {}
    base = wl.decode(0)  # ids: one token per request, adapter uniform over 8
    ids = torch.from_numpy(base.ids).to(dev)
    segs = lora.lora_build_segments(ids=ids, n_adapters=base.n_adapters)
    for name, (d_outs, r) in QWEN3_4B_SHARED_X.items():
        specs = [wl.Spec(f"{name}{p}", 2560, d, np.full(8, r, np.int32), np.full(8, 2.0 * r), base.ids, False,
                         seed=p, with_bwd=False) for p, d in enumerate(d_outs)]
        nbytes = sum(decode_bytes(s) for s in specs) - (len(specs) - 1) * 2 * base.n_tokens * 2560
        n_sets = max(2, int(3 * L2_BYTES / nbytes) + 1)
        sets = []
        for q in range(n_sets):
            x = None
            tabs, ys, wss = [], [], []
            for p, s in enumerate(specs):
                s_q = wl.Spec(s.name, s.d_in, s.d_out, s.ranks, s.alphas, s.ids, False, seed=100 * q + p,
                              with_bwd=False)
                inp = wl.device_inputs(s_q, dev, y0="randn", need=("A", "B", "x", "y0"))
                x = inp["x"] if x is None else x
                tabs.append(lora.AdapterTable(inp["A"], inp["B"], s.ranks.tolist(), torch.from_numpy(s.scales),
                                              s.d_in, s.d_out))
                ys.append(inp["y0"])
                wss.append(lora.workspace(tabs[-1], s.n_tokens, dev))
            ws_m = torch.empty(lora.lora_multi_workspace_bytes(tabs, base.n_tokens), dtype=torch.uint8, device=dev)
            sets.append((x, tabs, ys, wss, ws_m))

        def multi(k):
            x, tabs, ys, _, ws_m = sets[k % n_sets]
            lora.lora_multi_fwd(ys, None, x, tabs, segs, ws_m, stream=stream)

        def separate(k):
            x, tabs, ys, wss, _ = sets[k % n_sets]
            for tab, y, ws in zip(tabs, ys, wss):
                lora.lora_packed_fwd(y, None, x, tab, segs, ws, stream=stream)

        res = {}
        for label, fn in (("multi", multi), ("separate", separate)):
            with torch.cuda.stream(stream):
                for k in range(n_sets):
                    fn(k)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(reps):
                    fn(k)
            times = []
            with torch.cuda.stream(stream):
                for _ in range(3):
                    g.replay()
                torch.cuda.synchronize()
                for _ in range(20):
                    s0 = torch.cuda.Event(enable_timing=True)
                    s1 = torch.cuda.Event(enable_timing=True)
                    s0.record(stream)
                    g.replay()
                    s1.record(stream)
                    s1.synchronize()
                    times.append(s0.elapsed_time(s1) / reps)
            res[label] = statistics.median(times)
            del g
        gbs = nbytes / (res["multi"] * 1e-3) / 1e9
        out[name] = {"projections": [f"2560x{d}" for d in d_outs], "us_per_call": round(res["multi"] * 1e3, 3),
                     "us_separate_calls": round(res["separate"] * 1e3, 3),
                     "speedup": round(res["separate"] / res["multi"], 3), "bytes": nbytes, "GB/s": round(gbs, 1),
                     "frac_of_hbm": round(gbs / hbm, 4)}
        del sets
        torch.cuda.empty_cache()
    return out


def time_adamw(spec: wl.Spec, dev, stream, reps: int = 20) -> dict:
    """The fused per-adapter AdamW step (masters, moments, bf16 refresh) on
    the workload's adapter table, rotating over enough buffer sets to exceed
    L2; algorithmic bytes 30 per weight (w, g, m, v read, w, m, v written in
    fp32, the bf16 copy written)."""
    import torch

    import adapter_sgmv_gb300 as lora

    hbm, _, _ = measured_peaks()
    sr = int(spec.sum_r)
    elems = sr * (spec.d_in + spec.d_out)
    nbytes = 30 * elems
    n_sets = max(2, int(3 * L2_BYTES / nbytes) + 1)
    sets = []
    for q in range(n_sets):
        z = lambda d: torch.zeros((sr, d), dtype=torch.float32, device=dev)
        r = lambda d: torch.randn((sr, d), dtype=torch.float32, device=dev) * 0.01
        A_bf = torch.zeros((sr, spec.d_in), dtype=torch.bfloat16, device=dev)
        B_bf = torch.zeros((sr, spec.d_out), dtype=torch.bfloat16, device=dev)
        tab = lora.AdapterTable(A_bf, B_bf, spec.ranks.tolist(), torch.from_numpy(spec.scales), spec.d_in, spec.d_out)
        sets.append((tab, r(spec.d_in), r(spec.d_out), r(spec.d_in), r(spec.d_out), z(spec.d_in), z(spec.d_in),
                     z(spec.d_out), z(spec.d_out)))
    lr = torch.full((spec.n_adapters,), 1e-4, device=dev)
    step = torch.ones(spec.n_adapters, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        for k in range(n_sets + 3):
            lora.lora_adamw_step(*sets[k % n_sets][:1], *sets[k % n_sets][1:], lr, step, stream=stream)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for k in range(reps):
            lora.lora_adamw_step(*sets[k % n_sets][:1], *sets[k % n_sets][1:], lr, step, stream=stream)
        s1.record(stream)
        torch.cuda.synchronize()
    us = s0.elapsed_time(s1) / reps * 1e3
    gbs = nbytes / (us * 1e-6) / 1e9
    del sets
    torch.cuda.empty_cache()
    return {"us_per_step": round(us, 2), "weights": elems, "bytes": nbytes, "GB/s": round(gbs, 1),
            "frac_of_hbm": round(gbs / hbm, 4)}


def time_fused_base(spec: wl.Spec, dev, stream, reps: int = 10) -> dict:
    """A LoRA layer's forward, y = x W^T + the packed delta, in the library's
    single persistent launch (lora_fused_base_fwd), against the same layer
    done unfused: the base GEMM by cuBLAS (torch.matmul) then lora_packed_fwd
    accumulating the delta into its output.  Inputs (x 268 MB) exceed L2.
    Algorithmic flops: 2 T d_in d_out (base) + 2 sum_t r_i (d_in + d_out)."""
    import torch

    import adapter_sgmv_gb300 as lora

    _, bf16_peak, src = measured_peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            sustained = float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        sustained = None
    inp = wl.device_inputs(spec, dev, need={"A", "B", "x", "W"})
    T, d_in, d_out = spec.n_tokens, spec.d_in, spec.d_out
    tab = lora.AdapterTable(inp["A"], inp["B"], spec.ranks.tolist(), torch.from_numpy(spec.scales), d_in, d_out)
    segs = lora.lora_build_segments(seg_offsets=torch.from_numpy(spec.seg_offsets).to(dev), n_tokens=T,
                                    n_adapters=spec.n_adapters, device=dev)
    ws_f = torch.empty(lora.lora_fused_base_workspace_bytes(tab, T), dtype=torch.uint8, device=dev)
    ws_p = lora.workspace(tab, T, dev)
    y = torch.empty((T, d_out), dtype=torch.bfloat16, device=dev)
    H = torch.empty((T, spec.r_max), dtype=torch.float32, device=dev)
    x, W = inp["x"], inp["W"]
    rank_tok = np.repeat(spec.ranks.astype(np.int64), np.diff(spec.seg_offsets))
    flops = 2 * T * d_in * d_out + 2 * int(rank_tok.sum()) * (d_in + d_out)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(reps):
                fn()
            s1.record(stream)
            torch.cuda.synchronize()
        return s0.elapsed_time(s1) / reps

    fused = lambda: lora.lora_fused_base_fwd(y, H, x, W, tab, segs, ws_f, stream=stream)
    ms = timed(fused)
    assert lora.lora_query_status(segs) == 0
    ms_cublas = timed(lambda: torch.matmul(x, W.t(), out=y))

    def unfused():
        torch.matmul(x, W.t(), out=y)
        lora.lora_packed_fwd(y, H, x, tab, segs, ws_p, stream=stream)

    ms_unfused = timed(unfused)
    tf = flops / (ms * 1e-3) / 1e12
    out = {"workload": f"packed4096 layer forward: T={T}, {d_in}->{d_out}, ranks "
                       f"{{{','.join(str(int(r)) for r in spec.ranks)}}}, y = x W^T + s_i (x A_i^T) B_i^T",
           "ms": round(ms, 4), "flops": flops,
           "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                        "frac": round(tf / bf16_peak, 4), "peak_source": f"{src} (burst, cuBLAS bf16)",
                        "frac_of_sustained": round(tf / sustained, 4) if sustained else None},
           "cublas_base_ms": round(ms_cublas, 4),
           "cublas_base_TFLOP/s": round(2 * T * d_in * d_out / (ms_cublas * 1e-3) / 1e12, 1),
           "unfused_ms": round(ms_unfused, 4),
           "speedup_vs_unfused": round(ms_unfused / ms, 3)}
    del inp, y, H, ws_f, ws_p, segs, tab
    torch.cuda.empty_cache()
    return out


def packing_plan(spec: wl.Spec, ms_step: float, fused: dict | None, dev, stream) -> dict | None:
    """The packing planner (lora_plan_pack) on a PLoRA-sized search space, its
    cost model taken from this run's measurements of one 4096 -> 4096
    projection: the LoRA path's time per token from the packed step above
    (its rank term from the step's algorithmic bytes, 8 B per token and unit
    of rank, at the measured bandwidth), the fixed time of a step from the
    intercept against a 1024-token step of the same workload, and the frozen
    base's time per token from cuBLAS (forward GEMM + input-gradient GEMM,
    2x the base GEMM measured beside the fused layer).  The model: 32 layers
    x 7 such projections (a 7B-class dense model, 4096 wide), frozen bf16
    weights 14 GB + 4 GB of workspace per job; 120 configurations = ranks
    {8..128} x tokens per step {1024..8192} x 6 learning rates (the rate does
    not change the cost), each trained on 20 M tokens; 8 GPUs of 280 GB."""
    import torch

    import adapter_sgmv_gb300 as lora

    if fused is None:
        return None
    T = spec.n_tokens
    small = Workload(wl.packed4096(tokens_per_adapter=128), dev)  # T = 1024
    start, end, _, _ = time_steps(small, 10, 3, stream)
    torch.cuda.synchronize()
    ms_small = start.elapsed_time(end) / 10
    del small
    per_tok = ms_step * 1e-3 / T
    sb = step_bytes(spec)
    gbs = (sb["fwd"] + sb["bwd"]) / (ms_step * 1e-3)
    rank_coef = 8.0 / gbs
    counts = np.bincount(spec.ids, minlength=spec.n_adapters)
    mean_rank = float((counts * spec.ranks).sum()) / T
    proj = 32 * 7  # projections per model step
    cost = {"step_overhead_s": proj * max(0.0, ms_small * 1e-3 - 1024 * per_tok),
            "base_s_per_token": proj * 2 * fused["cublas_base_ms"] * 1e-3 / T,
            "lora_s_per_token": proj * (per_tok - mean_rank * rank_coef),
            "lora_s_per_token_rank": proj * rank_coef,
            "gpu_mem_bytes": 280 << 30, "job_mem_bytes": 18 << 30, "mem_unit_bytes": 64 << 20, "n_gpus": 8}
    configs = []
    for r in (8, 16, 32, 64, 128):
        for tok in (1024, 2048, 4096, 8192):
            for _ in range(6):
                mem = proj * r * 8192 * 18 + tok * 4096 * 2 * 32 * 12  # adapter state (bf16, fp32 master,
                configs.append({"rank": r, "tokens_per_step": tok, "steps": 20_000_000 // tok,  # moments, grad)
                                "mem_bytes": mem})                                                # + activations
    t0 = time.perf_counter()
    plan = lora.lora_plan_pack(configs, cost)
    plan_ms = (time.perf_counter() - t0) * 1e3
    w = lambda c: cost["base_s_per_token"] + cost["lora_s_per_token"] + cost["lora_s_per_token_rank"] * c["rank"]
    alone = sorted((c["steps"] * (cost["step_overhead_s"] + c["tokens_per_step"] * w(c)) for c in configs),
                   reverse=True)
    free = [0.0] * cost["n_gpus"]
    for d in alone:  # one configuration per job, longest first on the GPU that frees first
        g = min(range(len(free)), key=lambda q: (free[q], q))
        free[g] += d
    sizes = [j["n_configs"] for j in plan["jobs"]]
    return {"configs": len(configs), "gpus": cost["n_gpus"], "jobs": len(plan["jobs"]),
            "configs_per_job": [min(sizes), max(sizes)], "makespan_h": round(plan["makespan_s"] / 3600, 3),
            "one_config_per_job_makespan_h": round(max(free) / 3600, 3),
            "speedup_vs_one_config_per_job": round(max(free) / plan["makespan_s"], 3),
            "planner_ms": round(plan_ms, 1),
            "cost_model": {k: (float(f"{v:.4g}") if isinstance(v, float) else v) for k, v in cost.items()},
            "small_step_ms": round(ms_small, 4)}


def cpu_baseline(spec: wl.Spec, target_s: float = 10.0):
    """The fp64 oracle on a bounded sample of the same workload (first tokens of
    every adapter), on this host's cores; tokens/s."""
    import oracle

    oracle.build()
    cores = oracle.threads()
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))

    def run(per_adapter):
        rows = []
        for i in range(spec.n_adapters):
            idx = np.flatnonzero(spec.ids == i)[:per_adapter]
            rows.append(idx)
        rows = np.concatenate(rows)
        sub = wl.custom(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids[rows], seed=spec.seed)
        host = wl.host_inputs(sub)
        f = lambda k: wl.bf16_bits_to_f64(host[k])
        A, B, x, dY, y0, dX0 = (f(k) for k in ("A", "B", "x", "dY", "y0", "dX0"))
        t0 = time.perf_counter()
        y, H = oracle.fwd(tab, sub.ids, A, B, x, y0)
        oracle.bwd(tab, sub.ids, A, B, x, H, dY, dX0)
        return len(rows), time.perf_counter() - t0

    per = 2
    n, dt = run(per)
    for _ in range(3):  # grow the sample until it takes about target_s (the fixed cost makes one guess short)
        if dt >= 0.5 * target_s or per >= 4096:
            break
        per = int(max(per + 1, min(4096, per * target_s / max(dt, 1e-3))))
        n, dt = run(per)
    # one host thread on a smaller sample, beside the all-core figure
    oracle.set_threads(1)
    try:
        per1 = max(2, per // max(1, cores))
        n1, dt1 = run(per1)
    finally:
        oracle.set_threads(cores)
    return {"value": round(n / dt, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} tokens ({per} per adapter) of the same workload, fwd+bwd in fp64, {dt:.1f} s",
            "one_thread": {"value": round(n1 / dt1, 2), "sample": f"{n1} tokens, {dt1:.1f} s"}}


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (every rank gets it): the job's clock when the
    replicas run side by side."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, rank, world, dev):
    import torch
    import torch.distributed as dist

    import adapter_sgmv_gb300 as lora

    lora.build_library()
    lora.lib()
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    if args.decode_only:  # the decode measurement alone (profiling runs)
        return ({"decode_sgmv": time_decode(dev, stream), "decode_multi_projection": time_decode_multi(dev, stream)}
                if rank == 0 else None)
    if args.only is not None:  # one workload's steps alone (profiling runs)
        return {"workload": args.only, **time_config(named_workload(args.only), dev, stream, steps=args.steps,
                                                       warmup=args.warmup)} if rank == 0 else None
    spec = wl.packed4096(tokens_per_adapter=args.tokens_per_adapter)
    work = Workload(spec, dev)
    torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        start, end, ev, _ = time_steps(work, args.steps, args.warmup, stream)
        torch.cuda.synchronize()
    # per-kernel durations: the same number of steps again, with the library
    # recording an event pair around every kernel (the pairs cost ~20 us per
    # step, so the headline pass above runs without them)
    mstart, mend, _, kev = time_steps(work, args.steps, 1, stream, per_kernel=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    st = lora.lora_query_status(work.segs, stream)
    if st != 0:
        raise RuntimeError(f"device status {lora.STATUS.get(st, st)}")
    total_ms = start.elapsed_time(end)
    t_build = [e[0].elapsed_time(e[1]) for e in ev]
    t_fwd = [e[1].elapsed_time(e[2]) for e in ev]
    t_bwd = [e[2].elapsed_time(e[3]) for e in ev]
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    ms_step = total_ms / args.steps
    T = spec.n_tokens
    value = world * T * args.steps / (total_ms * 1e-3)

    hbm, tflops, peak_src = measured_peaks()
    by = step_bytes(spec)
    # each kernel's mean duration over the timed steps, from the event pairs the
    # library recorded around it on the launching stream
    kb = kernel_bytes(spec)
    per_kernel = {}
    for j, (use, tmpl) in enumerate(STEP_KERNELS):
        ms = statistics.mean(row[2 * j].elapsed_time(row[2 * j + 1]) for row in kev)
        per_kernel[use] = {"kernel": tmpl, "ms": round(ms, 4), "bytes": kb[use],
                           "GB/s": round(kb[use] / (ms * 1e-3) / 1e9, 1)}
    templates = {}
    for use, tmpl in STEP_KERNELS:
        t = templates.setdefault(tmpl, {"ms": 0.0, "bytes": 0, "launches": 0})
        t["ms"] += per_kernel[use]["ms"]
        t["bytes"] += kb[use]
        t["launches"] += 1
    dom = max(templates, key=lambda k: templates[k]["ms"])  # the most time per step
    dom_ms = templates[dom]["ms"] / templates[dom]["launches"]
    dom_bytes = templates[dom]["bytes"] / templates[dom]["launches"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9

    # the same steps with the ordered (bit-reproducible) dA / dB sums
    work.deterministic = True
    dstart, dend, _, _ = time_steps(work, args.steps, 2, stream)
    torch.cuda.synchronize()
    work.deterministic = False
    det_ms = dstart.elapsed_time(dend) / args.steps
    e2e_ms, h2d, d2h = time_e2e(work, max(3, args.steps // 2), 2, stream) if not args.no_e2e else (None, 0, 0)
    decode = time_decode(dev, stream) if rank == 0 and not args.no_decode else None
    decode_multi = time_decode_multi(dev, stream) if rank == 0 and not args.no_decode else None
    others = None
    if rank == 0 and not args.no_sweep:
        del work
        torch.cuda.empty_cache()
        others = {f"sweep3584x18944_N{n}": time_config(wl.sweep(n), dev, stream, sequential=True)
                  for n in (2, 4, 8, 16, 32)}
        base = others["sweep3584x18944_N2"]["tokens/s"]
        for n in (2, 4, 8, 16, 32):  # tokens/s(N) / tokens/s(2): flat means linear in N
            others[f"sweep3584x18944_N{n}"]["efficiency_vs_N2"] = round(
                others[f"sweep3584x18944_N{n}"]["tokens/s"] / base, 3)
        others["skewed4096x14336_N32"] = time_config(wl.skewed(), dev, stream)
    adamw = time_adamw(spec, dev, stream) if rank == 0 else None
    fused = time_fused_base(spec, dev, stream) if rank == 0 and not args.no_fused else None
    plan = packing_plan(spec, ms_step, fused, dev, stream) if rank == 0 and not args.no_plan else None
    cpu = cpu_baseline(spec, args.cpu_seconds) if rank == 0 and not args.no_cpu else None

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shapes of the packed training batch)",
        "config": dict(workload_config(spec, args.tokens_per_adapter),
                       l2="inputs larger than L2 (x, dY, y 268 MB each); no flush",
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "breakdown_ms": {"lora_build_segments": round(statistics.mean(t_build), 4),
                         "lora_packed_fwd": round(statistics.mean(t_fwd), 4),
                         "lora_packed_bwd": round(statistics.mean(t_bwd), 4)},
        "step_bytes": by["fwd"] + by["bwd"], "step_flops": step_flops(spec),
        "step_GB/s": round((by["fwd"] + by["bwd"]) / (ms_step * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                     "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic_record(dom, spec.n_tokens),
                     "bytes_per_launch": int(dom_bytes), "ms_per_launch": round(dom_ms, 4),
                     "launches_per_step": templates[dom]["launches"],
                     "tensor_frac_at_this_time": round(step_flops(spec) / (ms_step * 1e-3) / 1e12 / tflops, 4)},
        "deterministic_bwd": {"ms_per_step": round(det_ms, 4), "extra_ms": round(det_ms - ms_step, 4),
                              "note": "lora_packed_bwd_ex with LORA_BWD_DETERMINISTIC: dA / dB bit-identical "
                                      "run to run (every adapter here has four spans of 1024 tokens)"},
        "kernels_ms": per_kernel,
        "kernels_note": ("from a second pass of the same steps with an event pair around every kernel "
                         f"({round(mstart.elapsed_time(mend) / args.steps, 4)} ms per step with the pairs, "
                         "where the backward's kernels run one after another instead of dB next to dh and dA next to dX)"),
        "e2e": ({"value": round(world * T / (e2e_ms * 1e-3), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h} if e2e_ms is not None else None),
        "gpu_launches": kernels_per_step(spec) * args.steps,
        "clocks": clk.summary(),
        "decode_sgmv": decode,
        "decode_multi_projection": decode_multi,
        "adamw_step": adamw,
        "fused_base_lora": fused,
        "packing_plan": plan,
        "other_workloads": others,
        "cpu_baseline": cpu,
    }
    return line


# ---------------------------------------------------------------------------- reference arm
def named_workload(name: str) -> wl.Spec:
    if name == "packed4096":
        return wl.packed4096()
    if name == "skewed":
        return wl.skewed()
    if name.startswith("sweep") and name[5:].isdigit():
        return wl.sweep(int(name[5:]))
    raise SystemExit(f"unknown workload {name!r}")


def workload_config(spec: wl.Spec, tokens_per_adapter: int) -> dict:
    """The benchmarked workload, named the same way by both arms."""
    return {"workload": "packed4096: 4096->4096, N=8 ranks {8,16,16,32,32,64,64,128}, alpha 16/32, "
                        f"8 sorted segments x {tokens_per_adapter} tokens (T={spec.n_tokens}), fwd+bwd",
            "tokens_per_step": spec.n_tokens, "d_in": spec.d_in, "d_out": spec.d_out, "adapters": spec.n_adapters}


def run_reference(args):
    """The fp64 oracle (the only reference this method has) on the host cores:
    each step is a bounded sample of the same workload; tokens/s."""
    import oracle

    spec = wl.packed4096(tokens_per_adapter=args.tokens_per_adapter)
    oracle.build()
    per = args.ref_tokens_per_adapter
    rows = np.concatenate([np.flatnonzero(spec.ids == i)[:per] for i in range(spec.n_adapters)])
    sub = wl.custom(spec.name, spec.d_in, spec.d_out, spec.ranks, spec.alphas, spec.ids[rows], seed=spec.seed)
    host = wl.host_inputs(sub)
    f = lambda k: wl.bf16_bits_to_f64(host[k])
    A, B, x, dY, y0, dX0 = (f(k) for k in ("A", "B", "x", "dY", "y0", "dX0"))
    tab = oracle.Table(spec.ranks, spec.scales.astype(np.float64))

    def step():
        y, H = oracle.fwd(tab, sub.ids, A, B, x, y0)
        oracle.bwd(tab, sub.ids, A, B, x, H, dY, dX0)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    n = len(rows)
    value = n * args.steps / dt
    cores = oracle.threads()
    sample = f"{n} tokens per step ({per} per adapter) of the packed4096 workload, fwd+bwd in fp64"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": dict(workload_config(spec, args.tokens_per_adapter), sample_tokens_per_step=n,
                       parallelism="host cores"),
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens-per-adapter", type=int, default=16)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the adapter-count sweep and the skewed batch")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused base + delta layer forward")
    ap.add_argument("--no-plan", action="store_true", help="skip the packing planner run")
    ap.add_argument("--decode-only", action="store_true", help="time only the decode batch (profiling runs)")
    ap.add_argument("--only", default=None, metavar="WORKLOAD",
                    help="time only this workload's steps and print its figures (profiling runs): packed4096, "
                         "skewed, sweep2 .. sweep32")
    ap.add_argument("--tokens-per-adapter", type=int, default=4096,
                    help="tokens per adapter of the packed batch (4096 is the benchmarked workload; "
                         "smaller values give the small profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch

    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(dev)
        dist.init_process_group("nccl", device_id=dev)
    line = run_ours(args, rank, world, dev)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
