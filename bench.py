#!/usr/bin/env python
"""Benchmark of MoE expert-parallel dispatch + combine on GB300.

One step = layout + dispatch (one fused call) -> combine over one batch of the
DeepSeek-shape decode workload (8 logical EP ranks x 128 tokens, hidden 7168
fp8 e4m3 with 128-element fp32 scales, 256 experts, top-8, max_m 128), inputs
resident in HBM (--unfused: layout and dispatch as two calls). The synthetic
experts run once before timing (their outputs stay resident; layout is
deterministic, so every step gathers valid rows). Before every timed step,
outside the timed events, L2 is flushed: a buffer of twice its size is written
and another one read, so each step starts from a cold L2 with no dirty lines.

Arms:
  --impl native (default): the CUDA library through its C ABI; prints one JSON
    line with the device-timed value, the end-to-end value (host buffers,
    copies inside the timed region), the roofline of the dominant kernel
    (combine), the CPU oracle baseline, clocks and launch counts.
  --impl reference: the CPU oracle on the host cores, each step a bounded
    sample of the same workload.

Multi-GPU (torchrun): every rank runs an independent replica (no collective
on the data path); rank 0 prints the whole-job value = all ranks' tokens /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import contextlib
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s vs 8 TB/s, H=7168 top-8/256"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "ds_decode"


# --- process group ------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_over_ranks(value: float, world: int, op: str, device=None) -> float:
    """max or sum of a per-rank float over all ranks (identity on one rank)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def whole_job(tokens_per_rank_step: int, local_ms_total: float, steps: int, world: int, device=None) -> dict:
    """Whole-job throughput: tokens of all ranks over the slowest rank's time."""
    slow_ms = reduce_over_ranks(local_ms_total, world, "max", device)
    tokens = reduce_over_ranks(tokens_per_rank_step * steps, world, "sum", device)
    return {"value": tokens / (slow_ms / 1e3), "ms_per_step": slow_ms / steps, "tokens": tokens}


# --- clocks ------------------------------------------------------------------

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "utilization.gpu", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples (every 20 ms) from before the warm-up steps to after the
    last measurement (the per-config steps and the end-to-end pass included)."""

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.gpu = vis.split(",")[local_rank] if vis else str(local_rank)
        self.samples = []
        self.proc = None
        self.thread = None
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={','.join(CLOCK_FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(CLOCK_FIELDS):
                self.samples.append(parts)

    def stop(self) -> dict:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        busy_only = [s for s in self.samples if (num(s[3]) or 0) > 0]
        busy = busy_only or self.samples
        sm = [num(s[0]) for s in busy if num(s[0]) is not None]
        mx = [num(s[1]) for s in self.samples if num(s[1]) is not None]
        reasons = sorted({REASON_NAMES[i] for s in busy for i in range(4) if s[4 + i].lower() == "active"})
        power = [num(s[2]) for s in busy if num(s[2]) is not None]
        window = round(time.time() - self.t0, 2) if self.t0 is not None else None
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "window_s": window, "interval_ms": 20,
                "reasons": reasons, "samples": len(self.samples), "busy_samples": len(busy_only),
                "power_w_max": max(power) if power else None}


# --- roofline inputs ------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError, TypeError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(name: str) -> str:
    with open(os.path.join(ROOT, "combine_moe_layout_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel_file.replace('.cu', '')}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(kernel_file):
        return None
    return float(m_bytes.group(1))


def profiled_dispatch_traffic(workload: str):
    """DRAM bytes of one layout+dispatch call from the committed per-workload ncu summary, if it was
    taken on the current layout and dispatch sources."""
    path = os.path.join(ROOT, "profiles", f"moe_combine_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_bytes = re.search(r"dispatch_dram_bytes_per_step:\s*([0-9.eE+]+)", text)
    if not m_bytes:
        return None
    for name in ("moe_dispatch.cu", "moe_layout.cu", "moe_layout_dispatch.cu"):
        m = re.search(r"`" + re.escape(name) + r"` ([0-9a-f]+)", text)
        if not m or m.group(1) != kernel_source_hash(name):
            return None
    return float(m_bytes.group(1))


# --- native arm -------------------------------------------------------------------

# Throughput configs reported beside the headline workload (the DeepSeek-shape
# prefill batch and the other large shapes).
PER_CONFIG = ("ds_prefill", "mixtral", "skewed")


def time_config(name, K, W, num_sms, dev, flush, world):
    """K steps (fused layout+dispatch call -> combine) of one more workload on its
    own buffers, timed like the headline step: L2 flushed before each step
    outside the events, CUDA events on the launching stream, max over ranks."""
    import torch

    from combine_moe_layout_gb300 import _binding as B
    from combine_moe_layout_gb300 import pipeline as P
    from combine_moe_layout_gb300 import workloads as wl

    w = wl.WORKLOADS[name]
    desc = B.MoeDesc.of(w, num_sms)
    need = sum(B.moe_buffer_sizes(desc).values()) + 3 * w.num_tokens * w.in_row_bytes + (2 << 30)
    free = torch.cuda.mem_get_info(dev)[0]
    if free < need:
        return {"unavailable": f"needs {need / 2**30:.1f} GiB of device memory, {free / 2**30:.1f} GiB free"}
    inp = wl.make_inputs(w)
    step = P.MoeStep(w, dev, num_sms)
    d = P.to_device(inp, dev)
    stream = torch.cuda.current_stream()
    step.reset()
    step.run(d, fused=True)  # the synthetic experts once; their outputs stay resident
    if step.error() != B.MOE_OK:
        raise RuntimeError(f"{name}: first step failed")
    for _ in range(W):
        flush()
        step.layout_dispatch(d)
        step.combine(d)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    torch.cuda.synchronize()
    barrier(world)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step.layout_dispatch(d)
        step.combine(d)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    for i in range(K):  # per kernel: events between the two calls
        flush()
        ev[i][0].record(stream)
        step.layout_dispatch(d)
        ev[i][1].record(stream)
        step.combine(d)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if step.error() != B.MOE_OK:
        raise RuntimeError(f"{name}: timed steps latched an error")
    kern = {"layout_dispatch": statistics.mean(a.elapsed_time(b) for a, b, _ in ev),
            "combine": statistics.mean(b.elapsed_time(c) for _, b, c in ev)}
    job = whole_job(w.num_tokens, sum(step_ms), K, world, dev)
    ab = dict(w.algorithmic_bytes())
    ab["layout_dispatch"] = ab["layout"] + ab["dispatch"]
    peak, peak_kind = measured_hbm_peak()
    step_s = job["ms_per_step"] / 1e3
    kernels = {}
    for kname, ms in kern.items():
        gbs = ab[kname] / (ms / 1e3) / 1e9
        kernels[kname] = {"us": round(ms * 1e3, 2), "algorithmic_bytes": ab[kname], "GBps": round(gbs, 1),
                          "frac_of_measured_hbm": round(gbs / peak, 4)}
    dom = max(kernels, key=lambda kk: kernels[kk]["us"])
    nk = B.moe_layout_dispatch_kernels(step.desc)
    out = {
        "description": wl.DESCRIPTIONS[name],
        "tokens_per_step": w.num_tokens,
        "us_per_step": round(job["ms_per_step"] * 1e3, 2),
        "tokens_per_s": round(job["value"], 1),
        "algorithmic_bytes_per_step": ab["total"],
        "step_GBps": round(ab["total"] / step_s / 1e9, 1),
        "frac_of_measured": round(ab["total"] / step_s / 1e9 / peak, 4),
        "frac_of_8TBps": round(ab["total"] / step_s / 1e9 / NOMINAL_HBM_GBS, 4),
        "step_kernels": ("fused layout+dispatch kernel, combine" if nk == 1 else
                         "layout+dispatch call (a layout kernel, then the dispatch kernel), combine"),
        "kernels": kernels,
        "roofline": {"kernel": "combine_kernel" if dom == "combine" else "layout+dispatch", "bound": "hbm",
                     "achieved": kernels[dom]["GBps"], "peak": peak, "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "unit": "GB/s", "frac": kernels[dom]["frac_of_measured_hbm"],
                     "traffic": (profiled_traffic("moe_combine.cu", name) if dom == "combine"
                                 else profiled_dispatch_traffic(name)),
                     "algorithmic_bytes_per_launch": ab[dom]},
        "gpu_launches": (nk + 1) * K,
        "steps": K,
    }
    del step, d
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_native(args, rank, local_rank, world):
    import numpy as np
    import torch

    from combine_moe_layout_gb300 import _binding as B
    from combine_moe_layout_gb300 import pipeline as P
    from combine_moe_layout_gb300 import workloads as wl

    assert torch.cuda.is_available(), "the native arm needs a CUDA device"
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    step = P.MoeStep(w, dev, args.num_sms)
    d = P.to_device(inp, dev)
    stream = torch.cuda.current_stream()
    step.reset()
    step.run(d)  # also runs the synthetic experts once; their outputs stay resident
    status = step.error()
    if status != B.MOE_OK:
        raise RuntimeError(f"first step failed: {B.moe_status_string(status)}")

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_n = max(2 * l2, 256 << 20)
    flush_w = torch.empty(flush_n, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(flush_n // 4, dtype=torch.float32, device=dev)

    def flush():
        # write a buffer twice the L2 size, then read another one: the timed step
        # starts from a cold L2 that holds no dirty lines of the flush
        flush_w.fill_(1)
        flush_r.sum()

    fused = not args.unfused
    kernels = B.moe_layout_dispatch_kernels(step.desc) + 1 if fused else 3
    packed = packed_y = None
    if args.packed:
        # receive hook + packed combine: expert outputs resident in packed order
        packed = B.allocate_packed(step.desc, dev)
        step.layout_dispatch(d)
        step.recv(packed)
        ts = step.buf.tok_slot.view(-1).long()
        m = packed.packed_meta[:w.num_tokens * w.topk].long()
        slot_of_packed = ts[(m[:, 0] * w.tokens_per_rank + m[:, 1]) * w.topk + m[:, 3]]
        packed_y = step.y.index_select(0, slot_of_packed).contiguous()
        step.combine_packed(d, packed_y, packed)
        if step.error() != B.MOE_OK:
            raise RuntimeError("packed step failed")
        kernels += 2

    def path(dd, out=None):
        if fused:
            step.layout_dispatch(dd)
        else:
            step.layout(dd)
            step.dispatch(dd)
        if packed is not None:
            step.recv(packed)
            step.combine_packed(dd, packed_y, packed, out=out)
        else:
            step.combine(dd, out=out)

    K, W = args.steps, args.warmup
    sampler = ClockSampler(local_rank).start()
    for _ in range(W):
        flush()
        path(d)
    torch.cuda.synchronize()
    barrier(world)

    timed = lambda: path(d)  # noqa: E731
    if args.graph:
        # the step's launches captured once into a CUDA graph and replayed
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            path(d)
        torch.cuda.synchronize()
        timed = graph.replay
        for _ in range(W):
            flush()
            timed()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    barrier(world)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        timed()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # per-kernel durations, CUDA events on the launching stream (a second pass of K steps)
    stages = [("layout_dispatch", step.layout_dispatch)] if fused else \
        [("layout", step.layout), ("dispatch", step.dispatch)]
    if packed is not None:
        stages.append(("recv", lambda dd: step.recv(packed)))
        stages.append(("combine_packed", lambda dd: step.combine_packed(dd, packed_y, packed)))
    else:
        stages.append(("combine", step.combine))
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    for i in range(K):
        flush()
        kev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn(d)
            kev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    kern_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in kev) for j, (name, _) in enumerate(stages)}

    # the other throughput configs, each timed the same way on its own buffers (freed after)
    per_config = {}
    if not (args.no_per_config or args.packed or args.graph or args.unfused):
        for name in PER_CONFIG:
            if name != w.name:
                per_config[name] = time_config(name, K, W, args.num_sms, dev, flush, world)

    # end to end: the step's inputs packed in one pinned host buffer, copied in
    # with one H2D copy, and the output read back, all inside the timed region
    e2e = None
    if not args.no_e2e:
        parts = [np.ascontiguousarray(inp.x).view(np.uint8).ravel(), inp.topk_idx.view(np.uint8).ravel(),
                 inp.topk_weights.view(np.uint8).ravel()]
        if inp.x_scales is not None:
            parts.append(inp.x_scales.view(np.uint8).ravel())
        offs, o = [], 0
        for a_ in parts:
            offs.append(o)
            o += (a_.size + 255) // 256 * 256
        hpack = torch.empty(o, dtype=torch.uint8).pin_memory()
        for a_, off in zip(parts, offs):
            hpack[off:off + a_.size].copy_(torch.from_numpy(a_))
        dpack = torch.empty(o, dtype=torch.uint8, device=dev)

        def view(pack, i_, dtype, shape):
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            return pack[offs[i_]:offs[i_] + n].view(dtype).view(shape)

        def inputs_in(pack):
            R_, T_, H_, k_ = w.num_ranks, w.tokens_per_rank, w.hidden, w.topk
            xx = view(pack, 0, torch.uint8 if w.dtype == "fp8" else torch.bfloat16, (R_, T_, H_))
            return P.DeviceInputs(view(pack, 1, torch.int32, (R_, T_, k_)), view(pack, 2, torch.float32, (R_, T_, k_)),
                                  xx, view(pack, 3, torch.float32, (R_, T_, H_ // 128))
                                  if inp.x_scales is not None else None)

        hout = torch.empty((w.num_tokens, w.hidden), dtype=torch.bfloat16).pin_memory()
        out_view = step.buf.out.view(w.num_tokens, w.hidden)
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        mode = args.e2e_mode
        if mode == "auto":
            # small batches: the copy engine brings the inputs in faster than the kernels pull them, and the
            # next step's copy overlaps this step; large ones: the kernels read the inputs straight from host memory
            mode = "pipelined" if w.num_tokens <= 2048 else "zero-copy"
        if mode.startswith("pipelined") and (packed is not None or
                                    2 * sum(B.moe_buffer_sizes(step.desc).values()) > torch.cuda.mem_get_info(dev)[0] // 2):
            mode = "hybrid"   # the packed path, or no room for two more sets of step buffers
        e2e_ms = None
        if mode in ("pipelined", "pipelined-copy"):
            # consecutive steps overlap on several streams: step i + 1's inputs are copied in by a copy engine
            # while step i + 1 dispatches (a high-priority stream, so its blocks take SM slots as step i's
            # combine blocks retire) beside step i's combine. "pipelined": combine writes the bf16 output into
            # pinned host memory over NVLink-C2C. "pipelined-copy": combine writes it to device memory and a
            # second copy engine, on a fourth stream, moves it to pinned host memory while the SMs go on with
            # the next step. Three sets of step buffers, input packs and host outputs rotate: set i % 3 is
            # reused by step i + 3 once step i's combine (the last reader of its pack, slot ids and flags) and
            # its output copy are done. The expert outputs a step reads were last touched two steps (about
            # twice a step's traffic, several times L2) earlier, so no L2 flush sits between the steps.
            ce_out = mode == "pipelined-copy"
            ring = [step] + [P.MoeStep(w, dev, args.num_sms) for _ in range(2)]
            for r_ in ring[1:]:
                r_.reset()
                r_.run(d)  # the synthetic experts once, as for the first set
            dpacks = [dpack] + [torch.empty_like(dpack) for _ in range(2)]
            d2s = [inputs_in(p_) for p_ in dpacks]
            houts = [hout] + [torch.empty_like(hout).pin_memory() for _ in range(2)]
            hout_steps = [h_.view(w.num_ranks, w.tokens_per_rank, w.hidden) for h_ in houts]
            copy_stream = torch.cuda.Stream(dev)
            disp_stream = torch.cuda.Stream(dev, priority=-1)  # a lower number is a higher priority
            comb_stream = torch.cuda.Stream(dev, priority=0)
            out_stream = torch.cuda.Stream(dev)
            side = (copy_stream, disp_stream, comb_stream, out_stream)

            def pipelined(n):
                for s_ in side:
                    s_.wait_stream(stream)
                copied = [torch.cuda.Event() for _ in range(n)]
                dispatched = [torch.cuda.Event() for _ in range(n)]
                done = [torch.cuda.Event() for _ in range(n)]  # combine, and the output copy if any, finished
                for i in range(n):
                    j = i % 3
                    if i >= 3:
                        copy_stream.wait_event(done[i - 3])  # step i - 3 no longer uses set j
                    with torch.cuda.stream(copy_stream):
                        dpacks[j].copy_(hpack, non_blocking=True)
                        copied[i].record(copy_stream)
                    disp_stream.wait_event(copied[i])
                    with torch.cuda.stream(disp_stream):
                        if fused:
                            ring[j].layout_dispatch(d2s[j])
                        else:
                            ring[j].layout(d2s[j])
                            ring[j].dispatch(d2s[j])
                        dispatched[i].record(disp_stream)
                    comb_stream.wait_event(dispatched[i])
                    with torch.cuda.stream(comb_stream):
                        if ce_out:
                            ring[j].combine(d2s[j])
                            combined = torch.cuda.Event()
                            combined.record(comb_stream)
                        else:
                            ring[j].combine(d2s[j], out=hout_steps[j])
                            done[i].record(comb_stream)
                    if ce_out:
                        out_stream.wait_event(combined)
                        with torch.cuda.stream(out_stream):
                            houts[j].copy_(ring[j].buf.out.view(w.num_tokens, w.hidden), non_blocking=True)
                            done[i].record(out_stream)
                for s_ in side:
                    stream.wait_stream(s_)

            pipelined(W)
            torch.cuda.synchronize()
            t0_, t1_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0_.record(stream)
            pipelined(K)
            t1_.record(stream)
            torch.cuda.synchronize()
            e2e_ms = t0_.elapsed_time(t1_)
            for r_ in ring:
                if r_.error() != B.MOE_OK:
                    raise RuntimeError("pipelined end-to-end steps latched an error")
            how = ("pipelined: each step's packed inputs copied in by a copy engine on its own stream; the step "
                   "dispatches on a high-priority stream beside the previous step's combine, "
                   + ("which writes the bf16 output to device memory, and a second copy engine moves it to pinned "
                      "host memory on a fourth stream; " if ce_out else
                      "which writes the bf16 output straight into pinned host memory; ")
                   + "three sets of step buffers, input packs and host outputs rotate instead of an L2 flush "
                   "between steps")
        elif mode == "copy":
            d2 = inputs_in(dpack)
            for i in range(K):
                flush()
                eev[i][0].record(stream)
                dpack.copy_(hpack, non_blocking=True)
                path(d2)
                hout.copy_(out_view, non_blocking=True)
                eev[i][1].record(stream)
            how = "one pinned H2D copy of the packed inputs, one D2H copy of the bf16 output"
        elif mode == "hybrid":
            d2 = inputs_in(dpack)
            hout_steps = hout.view(w.num_ranks, w.tokens_per_rank, w.hidden)
            for i in range(K):
                flush()
                eev[i][0].record(stream)
                dpack.copy_(hpack, non_blocking=True)
                path(d2, out=hout_steps)
                eev[i][1].record(stream)
            how = ("one pinned H2D copy of the packed inputs (copy engine), then combine writes the bf16 output "
                   "straight into pinned host memory over NVLink-C2C")
        else:
            h2 = inputs_in(hpack)
            hout_steps = hout.view(w.num_ranks, w.tokens_per_rank, w.hidden)
            for i in range(K):
                flush()
                eev[i][0].record(stream)
                path(h2, out=hout_steps)
                eev[i][1].record(stream)
            how = ("zero-copy: the kernels read the packed inputs from pinned host memory and write the bf16 "
                   "output into pinned host memory over NVLink-C2C, no separate copies")
        torch.cuda.synchronize()
        if e2e_ms is None:
            e2e_ms = sum(a.elapsed_time(b) for a, b in eev)
        e2e = {"value": None, "unit": "tokens/s", "h2d_bytes_per_step": int(sum(a_.size for a_ in parts)),
               "d2h_bytes_per_step": hout.numel() * 2, "local_ms_total": e2e_ms, "mode": mode, "copies": how}
        if mode != "copy":
            path(d)  # the same step on device buffers, to compare
            torch.cuda.synchronize()
        want = out_view.cpu().view(torch.int16)
        for h_ in (houts if mode.startswith("pipelined") else [hout]):
            if not torch.equal(h_.view(torch.int16), want):
                raise RuntimeError("end-to-end output differs from the device output")

    clocks = sampler.stop()
    status = step.error()
    if status != B.MOE_OK:
        raise RuntimeError(f"timed steps latched an error: {B.moe_status_string(status)}")

    red_dev = dev
    job = whole_job(w.num_tokens, sum(step_ms), K, world, red_dev)
    if e2e is not None:
        ej = whole_job(w.num_tokens, e2e.pop("local_ms_total"), K, world, red_dev)
        e2e["value"] = ej["value"]
        e2e["ms_per_step"] = ej["ms_per_step"]

    if rank != 0:
        return None

    ab = dict(w.algorithmic_bytes())
    ab["layout_dispatch"] = ab["layout"] + ab["dispatch"]
    comb = "combine_packed" if packed is not None else "combine"
    if packed is not None:
        ab["total"] = ab["total_packed"]
    peak, peak_kind = measured_hbm_peak()
    comb_s = kern_ms[comb] / 1e3
    achieved = ab[comb] / comb_s / 1e9
    traffic = profiled_traffic("moe_combine.cu", w.name) if packed is None else None
    kernel_stats = {}
    for name in kern_ms:
        gbs = ab[name] / (kern_ms[name] / 1e3) / 1e9
        kernel_stats[name] = {"us": round(kern_ms[name] * 1e3, 3), "algorithmic_bytes": ab[name],
                              "GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 4)}
    step_s = job["ms_per_step"] / 1e3
    line = {
        "metric": METRIC,
        "value": round(job["value"], 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(job["ms_per_step"], 6),
        "ms_per_step_median_rank0": round(statistics.median(step_ms), 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32",
        "data": "synthetic",
        "impl": "native",
        "config": {
            "workload": w.name,
            "description": wl.DESCRIPTIONS[w.name],
            "tokens_per_step_per_gpu": w.num_tokens,
            "algorithmic_bytes_per_step": ab["total"],
            "path": "layout (int32) -> dispatch (e4m3 rows + fp32 scales, byte copy) -> combine (bf16 in, fp32 "
                    "accumulate, bf16 out); synthetic experts outside the timed region",
            "l2": "flushed before every timed step, outside the timed events: a write of a buffer of 2x L2 "
                  "then a read of another (cold, clean L2)",
            "step_kernels": (("fused layout+dispatch kernel, combine" if B.moe_layout_dispatch_kernels(step.desc) == 1
                              else "layout+dispatch call (a layout kernel, then the dispatch kernel: the fused "
                                   "kernel's staging does not fit this batch), combine")
                             if fused else "layout, dispatch, combine"),
            "launch": "one CUDA graph replay per step" if args.graph else "direct launches through the C ABI",
            "receive": "receive hook packs the slots expert-major, packed combine" if packed is not None
                       else "combine reads the fixed slots",
            "parallelism": "replicas only: one independent EP group of 8 logical ranks per GPU",
            "num_sms": args.num_sms,
        },
        "step_hbm": {"GBps": round(ab["total"] / step_s / 1e9, 1),
                     "frac_of_8TBps": round(ab["total"] / step_s / 1e9 / NOMINAL_HBM_GBS, 4),
                     "frac_of_measured": round(ab["total"] / step_s / 1e9 / peak, 4)},
        "roofline": {"kernel": "combine_kernel", "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (copy bandwidth)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": ab[comb]},
        "kernels": kernel_stats,
        "kernel_timing": "CUDA events between the launches, a second pass of the same K steps",
        "per_config": per_config,
        "e2e": e2e,
        "gpu_launches": kernels * K + sum(c.get("gpu_launches", 0) for c in per_config.values()),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world >= 1:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    return line


def measured_tensor_peak():
    """Dense bf16 TFLOP/s from MEASURED_PEAKS.json: (burst, sustained, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["bf16_tflops"]), float(m["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


def run_expert(args, rank, local_rank, world):
    """One step = fused layout+dispatch -> receive hook -> expert stage (linear 1 +
    SwiGLU, linear 2 on the tensor cores) -> packed combine, on a bf16 workload
    with synthetic expert weights resident in HBM."""
    import numpy as np
    import torch

    from combine_moe_layout_gb300 import _binding as B
    from combine_moe_layout_gb300 import pipeline as P
    from combine_moe_layout_gb300 import workloads as wl

    assert torch.cuda.is_available(), "the native arm needs a CUDA device"
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    init_dist(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.tokens_per_rank or args.intermediate:
        from dataclasses import replace
        T_ = args.tokens_per_rank or w.tokens_per_rank
        I_ = args.intermediate or w.intermediate
        w = replace(w, name=f"{w.name}_T{T_}_I{I_}", tokens_per_rank=T_, max_m=T_, intermediate=I_)
        wl.DESCRIPTIONS.setdefault(w.name, f"{wl.DESCRIPTIONS[args.workload]}; {T_} tokens per rank, I {I_}")
    fp8 = w.dtype != "bf16"   # e4m3 rows: the fp8 expert stage with fp8 weights
    inp = wl.make_inputs(w)
    step = P.MoeStep(w, dev, args.num_sms)
    d = P.to_device(inp, dev)
    wts = wl.expert_weights_fp8(w, dev) if fp8 else wl.expert_weights(w, dev)
    packed = B.allocate_packed(step.desc, dev)
    rows, H, I = w.num_tokens * w.topk, w.hidden, w.intermediate
    h = torch.empty((rows, I), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    hs = torch.empty((rows, I // 128), dtype=torch.float32, device=dev) if fp8 else None
    y = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    step.reset()

    if fp8:
        gate_up = lambda dd, out=None: B.moe_expert_gate_up_fp8(  # noqa: E731
            step.desc, I, packed.region_offsets, packed.packed_x, packed.packed_scales, wts.w_gate,
            wts.w_gate_scales, wts.w_up, wts.w_up_scales, h, hs, step.buf.err)
        down = lambda dd, out=None: B.moe_expert_down_fp8(  # noqa: E731
            step.desc, I, packed.region_offsets, h, hs, wts.w_down, wts.w_down_scales, y, step.buf.err)
    else:
        gate_up = lambda dd, out=None: B.moe_expert_gate_up(  # noqa: E731
            step.desc, I, packed.region_offsets, packed.packed_x, wts.w_gate, wts.w_up, h, step.buf.err)
        down = lambda dd, out=None: B.moe_expert_down(  # noqa: E731
            step.desc, I, packed.region_offsets, h, wts.w_down, y, step.buf.err)
    stages = [("layout_dispatch", lambda dd, out=None: step.layout_dispatch(dd)),
              ("recv", lambda dd, out=None: step.recv(packed)),
              ("expert_gate_up", gate_up),
              ("expert_down", down),
              ("combine_packed", lambda dd, out=None: step.combine_packed(dd, y, packed, out=out))]

    def path(dd, out=None):
        for _, fn in stages:
            fn(dd, out)

    path(d)
    if step.error() != B.MOE_OK:
        raise RuntimeError("first expert step failed")

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(flush_w.numel() // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_w.fill_(1)
        flush_r.sum()

    K, W = args.steps, args.warmup
    sampler = ClockSampler(local_rank).start()
    for _ in range(W):
        flush()
        path(d)
    torch.cuda.synchronize()
    barrier(world)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        path(d)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    for i in range(K):
        flush()
        kev[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn(d)
            kev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    kern_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in kev) for j, (name, _) in enumerate(stages)}

    # end to end: routing, rows and weights read from pinned host memory and the
    # bf16 output written there by the kernels themselves (zero-copy over NVLink-C2C)
    e2e = None
    if not args.no_e2e:
        hd = P.to_pinned_host(inp)
        hout = torch.empty((w.num_ranks, w.tokens_per_rank, H), dtype=torch.bfloat16).pin_memory()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush()
            eev[i][0].record(stream)
            path(hd, out=hout)
            eev[i][1].record(stream)
        torch.cuda.synchronize()
        nbytes = inp.x.nbytes + inp.topk_idx.nbytes + inp.topk_weights.nbytes + \
            (inp.x_scales.nbytes if inp.x_scales is not None else 0)
        e2e = {"value": None, "unit": "tokens/s", "h2d_bytes_per_step": int(nbytes),
               "d2h_bytes_per_step": hout.numel() * 2,
               "local_ms_total": sum(a.elapsed_time(b) for a, b in eev),
               "copies": "zero-copy: the kernels read routing and rows from pinned host memory and write the "
                         "bf16 output into pinned host memory over NVLink-C2C"}
        path(d)
        torch.cuda.synchronize()
        if not torch.equal(hout.view(torch.int16), step.buf.out.cpu().view(torch.int16)):
            raise RuntimeError("end-to-end output differs from the device output")
    clocks = sampler.stop()
    if step.error() != B.MOE_OK:
        raise RuntimeError("timed expert steps latched an error")
    job = whole_job(w.num_tokens, sum(step_ms), K, world, dev)
    if e2e is not None:
        ej = whole_job(w.num_tokens, e2e.pop("local_ms_total"), K, world, dev)
        e2e["value"], e2e["ms_per_step"] = ej["value"], ej["ms_per_step"]
    if rank != 0:
        return None

    flops = {"expert_gate_up": 2 * rows * H * 2 * I, "expert_down": 2 * rows * I * H}
    # bytes each linear map must move at least once: the weights of the experts
    # that received rows, the packed input rows, the output rows
    used = int((packed.region_offsets[w.num_ranks::w.num_ranks].cpu() -
                packed.region_offsets[:-1:w.num_ranks].cpu() > 0).sum())
    if fp8:   # e4m3 weights, rows and h, with their fp32 block scales; bf16 y
        gbytes = {"expert_gate_up": used * 2 * (I * H + I * H // 128 // 128 * 4) + rows * (H + H // 128 * 4) +
                  rows * (I + I // 128 * 4),
                  "expert_down": used * (H * I + H * I // 128 // 128 * 4) + rows * (I + I // 128 * 4) + rows * H * 2}
        weight_bytes = 3 * w.num_experts * I * H
    else:
        gbytes = {"expert_gate_up": used * 2 * I * H * 2 + rows * H * 2 + rows * I * 2,
                  "expert_down": used * H * I * 2 + rows * I * 2 + rows * H * 2}
        weight_bytes = 3 * w.num_experts * I * H * 2
    burst, sustained, kind = measured_tensor_peak()
    if fp8:   # the fp8 tensor rate: the measured bf16 rate times the nominal fp8 / bf16 ratio (4.5 / 2.25)
        burst, sustained, kind = 2 * burst, 2 * sustained, kind + " bf16 x 2 (nominal fp8/bf16 ratio)"
    hbm, hbm_kind = measured_hbm_peak()
    top = max(flops, key=lambda n: kern_ms[n])
    # the kernel's bound: whichever of its flops and its bytes takes longer at the measured peaks
    tensor_bound = flops[top] / (sustained * 1e12) >= gbytes[top] / (hbm * 1e9)
    # the fp8 kernel's form follows the expected rows per expert: below one 128-row tile the weight stream
    # bounds it (4 stages, direct stores), above it the tensor cores do (3 stages, staged stores)
    rows_per_expert = w.num_tokens * w.topk // w.num_experts
    kname = (("grouped_gemm_fp8_kernel<4, 0>" if rows_per_expert < 128 else "grouped_gemm_fp8_kernel<3, 1>")
             if fp8 else "grouped_gemm_kernel")
    ab = dict(w.algorithmic_bytes())
    kernel_stats = {}
    for name, ms in kern_ms.items():
        st = {"us": round(ms * 1e3, 3)}
        if name in flops:
            tf = flops[name] / (ms / 1e3) / 1e12
            gbs = gbytes[name] / (ms / 1e3) / 1e9
            st.update({"flops": flops[name], "TFLOPs": round(tf, 1), "frac_of_sustained_tensor": round(tf / sustained, 4),
                       "frac_of_burst_tensor": round(tf / burst, 4), "algorithmic_bytes": gbytes[name],
                       "GBps": round(gbs, 1), "frac_of_measured_hbm": round(gbs / hbm, 4)})
        else:
            key = {"layout_dispatch": None, "recv": "recv", "combine_packed": "combine_packed"}[name]
            nbytes = ab["layout"] + ab["dispatch"] if key is None else ab[key]
            st.update({"algorithmic_bytes": nbytes, "GBps": round(nbytes / (ms / 1e3) / 1e9, 1)})
        kernel_stats[name] = st
    line = {
        "metric": METRIC, "value": round(job["value"], 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(job["ms_per_step"], 6),
        "ms_per_step_median_rank0": round(statistics.median(step_ms), 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16", "data": "synthetic", "impl": "native",
        "config": {
            "workload": w.name + "+experts", "description": wl.DESCRIPTIONS[w.name],
            "expert_mlp": f"{w.num_experts} experts, linear 1 {H}->2x{I} with SwiGLU, linear 2 {I}->{H}, "
                          + ("e4m3 weights with 128x128 fp32 block scales, h e4m3 with 128-element scales, "
                             if fp8 else "bf16 ") +
                          f"weights N(0,1/K) ({weight_bytes / 1e9:.2f} GB resident)",
            "tokens_per_step_per_gpu": w.num_tokens, "flops_per_step": sum(flops.values()),
            "path": "fused layout+dispatch -> receive hook (expert-major packing) -> linear 1 + SwiGLU -> linear 2 "
                    + ("(tcgen05 kind::f8f6f4 grouped GEMMs, fp32 block-scale promotion) " if fp8 else
                       "(tcgen05 grouped GEMMs, fp32 accumulate) ") + "-> packed combine",
            "l2": "flushed before every timed step, outside the timed events",
            "launch": "direct launches through the C ABI",
            "parallelism": "replicas only: one independent EP group per GPU",
        },
        "roofline": ({"kernel": kname + " (" + top + ")", "bound": "tensor",
                      "achieved": kernel_stats[top]["TFLOPs"], "peak": sustained,
                      "peak_kind": f"{kind} {'fp8' if fp8 else 'bf16'} dense, sustained (the kernel runs inside a "
                                   "multi-ms step)",
                      "unit": "TFLOP/s", "frac": kernel_stats[top]["frac_of_sustained_tensor"],
                      "frac_of_burst": kernel_stats[top]["frac_of_burst_tensor"],
                      "traffic": profiled_traffic("moe_expert_fp8.cu" if fp8 else "moe_expert.cu", w.name),
                      "algorithmic_flops_per_launch": flops[top]} if tensor_bound else
                     {"kernel": kname + " (" + top + ")", "bound": "hbm",
                      "achieved": kernel_stats[top]["GBps"], "peak": hbm, "peak_kind": f"{hbm_kind} (copy bandwidth)",
                      "unit": "GB/s", "frac": kernel_stats[top]["frac_of_measured_hbm"],
                      "traffic": profiled_traffic("moe_expert_fp8.cu" if fp8 else "moe_expert.cu", w.name),
                      "algorithmic_bytes_per_launch": gbytes[top]}),
        "kernels": kernel_stats,
        "kernel_timing": "CUDA events between the launches, a second pass of the same K steps",
        "e2e": e2e, "gpu_launches": (B.moe_layout_dispatch_kernels(step.desc) + 5) * K,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_expert(w, inp, args.cpu_seconds)
    return line


def cpu_baseline_expert(w, inp, seconds: float) -> dict:
    """The oracle's layout over all tokens plus the expert MLP of the k choices of
    sampled tokens (about `seconds` of CPU work), as tokens/s."""
    import numpy as np
    import torch

    import oracle
    from combine_moe_layout_gb300 import workloads as wl
    t0 = time.perf_counter()
    oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    t_layout = time.perf_counter() - t0
    x = inp.x.reshape(w.num_tokens, w.hidden)
    idx = inp.topk_idx.reshape(w.num_tokens, w.topk)
    H, I = w.hidden, w.intermediate
    if w.dtype == "bf16":
        wts = wl.expert_weights(w, "cpu")
        bits = [t.view(torch.int16).numpy().view(np.uint16) for t in (wts.w_gate, wts.w_up, wts.w_down)]

        def row(tok, e):
            oracle.expert_mlp_row(x[tok], bits[0][e], bits[1][e], bits[2][e])
        weights = "the workload's synthetic bf16 weights"
    else:
        # the oracle's cost does not depend on the weight values: random e4m3 codes and unit block scales
        # for the experts the sampled tokens reach (generating all of the fp8 weights on the host would
        # take longer than the sample)
        xs = inp.x_scales.reshape(w.num_tokens, H // 128)
        rng = np.random.default_rng(0)
        cache = {}

        def weights_of(e):
            if e not in cache:
                q = [rng.integers(0, 0x7E, shape, dtype=np.uint8) for shape in ((I, H), (I, H), (H, I))]
                sc = [np.ones((a.shape[0] // 128, a.shape[1] // 128), np.float32) for a in q]
                cache[e] = (q, sc)
            return cache[e]

        def row(tok, e):
            (wg, wu, wd), (sg, su, sd) = weights_of(int(e))
            hv, hq, hs = oracle.gate_up_row_fp8(x[tok], xs[tok], wg, sg, wu, su)
            oracle.linear_row_fp8(hq, hs, wd, sd)
        weights = "random e4m3 weight codes (the oracle's cost does not depend on them)"
    spent, n = 0.0, 0
    with _one_core() as core:
        while n < 1 or spent < seconds:
            tok = (n * 7919) % w.num_tokens
            t0 = time.perf_counter()
            for e in idx[tok]:
                row(tok, e)
            spent += time.perf_counter() - t0
            n += 1
    per_tok = spent / n + t_layout / w.num_tokens
    return {"value": round(1.0 / per_tok, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"layout of all {w.num_tokens} tokens + the {w.topk} expert MLP rows of {n} tokens, "
                      f"single-threaded C oracle (fp64), {weights}", "seconds": round(spent + t_layout, 2),
            "cpu": _cpu_model(), "pinned_core": core}


# --- the CPU oracle (baseline leg and reference arm) ---------------------------------

def _oracle_sample_step(w, inp, sel):
    """One oracle step over the selected tokens: layout (all tokens), dispatch and
    combine of the selection; the synthetic experts run outside the timed part.
    Returns seconds spent in layout + dispatch + combine."""
    import oracle
    dt = w.dtype_code
    t0 = time.perf_counter()
    counts, flags, tok_slot = oracle.layout(inp.topk_idx, w.num_experts, w.max_m)
    slots = oracle.dispatch(inp.x, inp.x_scales, tok_slot, w.num_experts, w.max_m, dt, sel)
    t1 = time.perf_counter()
    y = oracle.expert_stub(slots, w.num_ranks, w.hidden, w.num_experts, w.max_m, dt)
    t2 = time.perf_counter()
    oracle.combine(tok_slot, inp.topk_weights, slots.slot_id, y, w.num_experts, w.max_m, sel)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2)


@contextlib.contextmanager
def _one_core():
    """Pin the calling thread (the one that runs the single-threaded oracle) to one
    core while the oracle is timed, and restore its affinity afterwards; yields the
    core, or None where affinity cannot be set."""
    try:
        old = os.sched_getaffinity(0)
        core = min(old)
        os.sched_setaffinity(0, {core})
    except (AttributeError, OSError, ValueError):
        yield None
        return
    try:
        yield core
    finally:
        os.sched_setaffinity(0, old)


def _cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_baseline(w, inp, seconds: float) -> dict:
    """The oracle on the whole batch, repeated until about `seconds` of CPU work."""
    import numpy as np
    sel = np.arange(w.num_tokens, dtype=np.int64)
    spent, reps = 0.0, 0
    with _one_core() as core:
        while reps < 1 or spent < seconds:
            spent += _oracle_sample_step(w, inp, sel)
            reps += 1
            if reps >= 50:
                break
    return {"value": round(reps * w.num_tokens / spent, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} full {w.name} steps ({w.num_tokens} tokens each), single-threaded C oracle "
                      f"(gcc -O2), synthetic experts excluded", "seconds": round(spent, 2),
            "cpu": _cpu_model(), "host_cores_available": os.cpu_count(), "pinned_core": core}


def run_reference(args, rank, local_rank, world):
    import numpy as np

    from combine_moe_layout_gb300 import workloads as wl
    if rank != 0:
        return None
    w = wl.WORKLOADS[args.workload]
    inp = wl.make_inputs(w)
    K, W = args.steps, args.warmup
    # size each step's token sample so the whole run stays within ~2 minutes
    pilot = np.arange(min(16, w.num_tokens), dtype=np.int64)
    per_tok = _oracle_sample_step(w, inp, pilot) / pilot.size
    budget = min(1.0, 120.0 / max(1, K + W))
    n = int(max(1, min(w.num_tokens, budget / max(per_tok, 1e-9))))
    cursor = 0

    def next_sel():
        nonlocal cursor
        s = (np.arange(n, dtype=np.int64) + cursor) % w.num_tokens
        cursor = (cursor + n) % w.num_tokens
        return s

    with _one_core() as core:
        for _ in range(W):
            _oracle_sample_step(w, inp, next_sel())
        spent = sum(_oracle_sample_step(w, inp, next_sel()) for _ in range(K))
    value = K * n / spent
    return {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(spent / K * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "description": wl.DESCRIPTIONS[w.name],
                   "sample": f"{n} of {w.num_tokens} tokens per step (layout over all tokens)"},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} tokens per step, {K} steps", "cpu": _cpu_model(), "pinned_core": core},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def calibrate(local_rank: int) -> dict:
    """Bandwidth of plain device writes (torch's float32 fill: 16-byte stores), reads
    (a float32 matrix-vector product, which reads its matrix once) and copies (read + write) over a range of sizes around the
    step's, each timed like the step (L2 flushed before each, CUDA events, median
    of 100), the time of an empty launch, and a floor for the decode step built
    from these rates: a launch, then dispatch's bytes at the write and read rates,
    then combine's at the read and write rates."""
    import torch

    from combine_moe_layout_gb300 import workloads as wl

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_r = torch.ones(flush_w.numel() // 4, dtype=torch.float32, device=dev)
    tiny = torch.empty(4, dtype=torch.float32, device=dev)

    def timeit(fn, n=100):
        for _ in range(5):
            flush_w.fill_(1)
            flush_r.sum()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            flush_w.fill_(1)
            flush_r.sum()
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3

    launch_us = timeit(lambda: tiny.fill_(1.0))
    rows = []
    for mb in (15, 30, 60, 120, 240, 480, 960):
        n = mb << 20
        a = torch.empty(n // 4, dtype=torch.float32, device=dev)
        b = torch.empty_like(a)
        a.fill_(1.0)
        mat = a.view(-1, 4096)
        vec = torch.ones(4096, dtype=torch.float32, device=dev)
        fill_us = timeit(lambda: a.fill_(7.0))
        read_us = timeit(lambda: torch.mv(mat, vec))  # reads the matrix once (cuBLAS GEMV)
        copy_us = timeit(lambda: b.copy_(a))
        rows.append({"MiB": mb, "fill_us": round(fill_us, 2), "fill_GBps": round(n / fill_us / 1e3, 1),
                     "read_us": round(read_us, 2), "read_GBps": round(n / read_us / 1e3, 1),
                     "copy_us": round(copy_us, 2), "copy_GBps_read_plus_write": round(2 * n / copy_us / 1e3, 1)})
        del a, b

    def rate(kind, mib):  # GB/s of the launch-free part, at the nearest measured size
        r = min(rows, key=lambda r_: abs(r_["MiB"] - mib))
        return (r["MiB"] << 20) / max(r[kind + "_us"] - launch_us, 1e-3) / 1e3

    w = wl.WORKLOADS["ds_decode"]
    N, k, H, sc = w.num_tokens, w.topk, w.hidden, w.scales_per_row * 4
    disp_w = N * k * (w.row_bytes + sc + 16) + N * k * 4
    disp_r = N * (w.in_row_bytes + sc)
    comb_r = N * k * 2 * H + N * k * 8
    comb_w = N * 2 * H
    wr, rd = rate("fill", disp_w / 2**20), rate("read", comb_r / 2**20)
    floor_us = launch_us + (disp_w / wr + disp_r / rd + comb_r / rd + comb_w / wr) / 1e3
    host = []
    for mb in (7.5, 15, 60, 240):
        n = int(mb * (1 << 20))
        h = torch.empty(n, dtype=torch.uint8).pin_memory()
        dd = torch.empty(n, dtype=torch.uint8, device=dev)
        h2d_us = timeit(lambda: dd.copy_(h, non_blocking=True), 50)
        d2h_us = timeit(lambda: h.copy_(dd, non_blocking=True), 50)
        host.append({"MiB": mb, "h2d_us": round(h2d_us, 2), "h2d_GBps": round(n / h2d_us / 1e3, 1),
                     "d2h_us": round(d2h_us, 2), "d2h_GBps": round(n / d2h_us / 1e3, 1)})
        del h, dd
    return {"calibration": "torch float32 fill (16-byte stores: write only), a float32 matrix-vector product "
                           "(cuBLAS GEMV: reads the matrix once) and copy (read + write), L2 flushed before each, "
                           "median of 100; pinned host <-> device copies, median of 50",
            "gpu": torch.cuda.get_device_name(dev), "empty_launch_us": round(launch_us, 2), "rows": rows,
            "host_copies": host,
            "ds_decode_floor": {"us": round(floor_us, 2), "write_GBps": round(wr, 1), "read_GBps": round(rd, 1),
                                "bytes": {"dispatch_write": disp_w, "dispatch_read": disp_r,
                                          "combine_read": comb_r, "combine_write": comb_w},
                                "model": "one launch + dispatch writes and combine's output at the plain-write "
                                         "rate + dispatch and combine reads at the plain-read rate, each rate "
                                         "taken without its launch time at the nearest measured size; layout "
                                         "latency and the second kernel's launch are not counted"}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default=None, help=f"default {DEFAULT_WORKLOAD} (mixtral with --expert)")
    ap.add_argument("--num-sms", type=int, default=0)
    ap.add_argument("--unfused", action="store_true", help="time layout and dispatch as two calls")
    ap.add_argument("--graph", action="store_true", help="replay the step's launches from a CUDA graph")
    ap.add_argument("--packed", action="store_true",
                    help="step = layout+dispatch, the receive hook (expert-major packing), the packed combine")
    ap.add_argument("--expert", action="store_true",
                    help="step = layout+dispatch, receive hook, expert stage (linear 1 + SwiGLU, linear 2 on the "
                         "tensor cores), packed combine; bf16 workload (default mixtral)")
    ap.add_argument("--tokens-per-rank", type=int, default=0, help="--expert: override T (a smaller profiling case)")
    ap.add_argument("--intermediate", type=int, default=0, help="--expert: override the expert MLP width I")
    ap.add_argument("--calibrate", action="store_true",
                    help="print the bandwidth of plain device writes and copies at the step's sizes and exit")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-mode", choices=("auto", "hybrid", "zero-copy", "copy", "pipelined", "pipelined-copy"), default="auto",
                    help="end to end: auto = pipelined up to 2048 tokens, zero-copy above; "
                         "hybrid = a copy engine moves the inputs in and combine writes the output "
                         "straight to pinned host memory; zero-copy = the kernels also read the inputs from host "
                         "memory; copy = copy engines move both; pipelined = hybrid with each step's input copy and "
                         "dispatch overlapping the previous step's combine; pipelined-copy = pipelined with "
                         "combine writing to device memory and a copy engine moving the output out")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other throughput configs (ds_prefill, mixtral, skewed)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.workload is None:
        args.workload = "mixtral" if args.expert else DEFAULT_WORKLOAD
    if args.steps is None:
        args.steps = (50 if args.expert else 2000) if args.impl == "native" else 20
    if args.warmup is None:
        args.warmup = (5 if args.expert else 20) if args.impl == "native" else 3
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    rank, local_rank, world = dist_env()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if args.calibrate:
        print(json.dumps(calibrate(local_rank)), flush=True)
        return
    native = run_expert if args.expert else run_native
    line = (native if args.impl == "native" else run_reference)(args, rank, local_rank, world)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
