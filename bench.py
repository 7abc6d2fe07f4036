#!/usr/bin/env python
"""Throughput of the MoE layer forward on one GB300 (or N replicas).

Default workload: the Qwen3-30B-A3B-shaped decode layer (E=128, top_k=8,
H=2048, I=768, bf16) at M=64 tokens, seeded synthetic weights and inputs
already resident in HBM.  A step is one moe_forward call -- the whole layer
(router logits, softmax/top-k/renormalize, align, grouped GEMM 1 +
SiLU-and-mul, grouped GEMM 2 + weighted combine) over one batch -- timed with
CUDA events around the call on the launching stream; the L2 is flushed (a
512 MB write) between steps, outside the events, and each step routes a
different x.

Printed (rank 0, one JSON line): tokens/s, the roofline of the dominant
kernel (grouped GEMM 1: HBM-bound in decode, tensor-bound in large prefill),
its duration taken with CUDA events in a breakdown pass through the step
entry points right after the timed steps, its DRAM traffic from the committed
ncu summary while the kernel code is unchanged, the end-to-end figure through
moe_forward with host buffers (every step's copy of x in and y out inside the
timed region; the better of a serial loop and one that overlaps the copies of
neighbouring steps with the layer on three streams, both reported), the CPU
oracle timed on a bounded sample, SM clocks sampled during the timed region,
the GPU and driver, and the workload's other batch sizes.

`--impl reference` times the CPU oracle instead (the slow reference arm).
Under torchrun every rank runs its own replica (no collective on the data
path); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
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

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s; % HBM roofline (decode), % bf16 TC peak (prefill)"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_CFG = {"toy": 1, "decode": 2, "prefill": 3, "stack": 4, "tail": 5}


# ----------------------------------------------------------------------------- accounting

def layer_bytes(w, M, D):
    """Algorithmic bytes of one layer: the D touched experts' W13 and W2, the
    router (or the given logits), x and y (and the residual), ids and weights."""
    b = D * 3 * w.H * w.I * 2 + 2 * M * w.H * 2 + M * w.top_k * 8
    b += M * w.E * 2 if w.logits_given else w.E * w.H * 2
    if w.residual:
        b += M * w.H * 2
    return b


def gemm1_bytes(w, M, D):
    """Algorithmic bytes of grouped GEMM 1: each touched expert's W13 [2I, H]
    once, the M input rows once, the M*top_k activation rows written once."""
    return D * 2 * w.I * w.H * 2 + M * w.H * 2 + M * w.top_k * w.I * 2


def layer_bytes_fp8(w, M, D):
    """layer_bytes with E4M3 expert weights: one byte per weight plus one fp32
    scale per weight row (2I rows of W13, H rows of W2 per expert)."""
    return layer_bytes(w, M, D) - D * 3 * w.H * w.I * 2 + D * (3 * w.H * w.I + (2 * w.I + w.H) * 4)


def gemm1_bytes_fp8(w, M, D):
    """Grouped GEMM 1 on E4M3 codes: W13 codes and row scales of the touched
    experts, the M quantized rows of x and their scales, a written in bf16."""
    return D * 2 * w.I * (w.H + 4) + M * (w.H + 4) + M * w.top_k * w.I * 2


def layer_flops(w, M):
    return M * w.top_k * 6 * w.H * w.I + (0 if w.logits_given else 2 * M * w.H * w.E)


def gemm1_flops(w, M):
    """GEMM 1 multiply-adds (2 flops each): every pair against the 2I rows of W13."""
    return M * w.top_k * 2 * (2 * w.I) * w.H


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ----------------------------------------------------------------------------- run metadata

def gpu_info(device):
    """Name and driver of the GPU the bench ran on."""
    info = {"name": torch.cuda.get_device_name(device), "driver": None}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.split()
        info["driver"] = out[0] if out else None
    except (OSError, subprocess.SubprocessError):
        pass
    return info


# ----------------------------------------------------------------------------- profiled traffic

PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "mixture_experts_layer_renorm_gb300", "csrc")


def code_digest(path):
    """sha256 of a C/CUDA source with its comments removed and whitespace
    collapsed: it changes when the code changes, not when a comment does."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def profiled_traffic(summary_name, block_size):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
    dominant kernel, from the committed ncu summary `profiles/<summary_name>`,
    or None when there is none for this block size or when the code of a
    kernel source it lists has changed since the counters were taken
    (code_digest per file)."""
    path = os.path.join(PROFILES, summary_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"^\s*traffic_bytes_per_launch\s*=\s*(\d+)\s*$", text, re.M)
    b = re.search(r"^\s*block_size_m\s*=\s*(\d+)\s*$", text, re.M)
    srcs = re.findall(r"^\s*source\s+(\S+)\s+code\s+sha256\s*=\s*([0-9a-f]{64})\s*$", text, re.M)
    if m is None or b is None or not srcs or int(b.group(1)) != block_size:
        return None
    for name, digest in srcs:
        f = os.path.join(CSRC, name)
        if not os.path.exists(f) or code_digest(f) != digest:
            return None
    return int(m.group(1))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.gpu = str(device.index or 0)
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except (AttributeError, RuntimeError):
            pass
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- our arm

class Layer:
    """Device-resident weights, inputs and buffers of one workload point."""

    def __init__(self, moe, w, M, n_inputs, device, layer=0, fp8=False):
        self.w, self.M, self.fp8 = w, M, fp8
        wt = (synth.layer_weights_fp8 if fp8 else synth.layer_weights)(w, layer=layer, device=device)
        self.wr, self.bias, self.w13, self.w2 = wt["w_router"], wt["router_bias"], wt["w13"], wt["w2"]
        self.s13, self.s2 = wt.get("w13_scale"), wt.get("w2_scale")
        self.inputs = [synth.layer_input(w, M, rep=r, device=device) for r in range(n_inputs)]
        self.B = w.block_size_m or moe.moe_pick_block_size(M, w.E, w.top_k, w.H, w.I)
        P = M * w.top_k
        cap = moe.moe_align_capacity(M, w.top_k, w.E, self.B)
        i32 = dict(dtype=torch.int32, device=device)
        self.logits = torch.empty((M, w.E), dtype=torch.bfloat16, device=device)
        self.ids = torch.empty((M, w.top_k), **i32)
        self.wts = torch.empty((M, w.top_k), dtype=torch.float32, device=device)
        self.sorted = torch.empty((cap,), **i32)
        self.eids = torch.empty((cap // self.B,), **i32)
        self.offs = torch.empty((w.E + 1,), **i32)
        self.npost = torch.empty((1,), **i32)
        self.a = torch.empty((P, w.I), dtype=torch.bfloat16, device=device)
        self.y = torch.empty((M, w.H), dtype=torch.bfloat16, device=device)
        self.ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, 0, device=device, fp8=fp8)
        if fp8:
            self.qx = torch.empty((M, w.H), dtype=torch.uint8, device=device)
            self.sx = torch.empty((M,), dtype=torch.float32, device=device)
            self.qa = torch.empty((P, w.I), dtype=torch.uint8, device=device)
            self.sa = torch.empty((P,), dtype=torch.float32, device=device)
        self.phases = (["route", "quant_x", "gemm1_act", "quant_a", "gemm2_combine"] if fp8
                       else ["route", "gemm1_act", "gemm2_combine"])

    def kernels_per_step(self):
        """Our kernels per step: routing (one fused launch up to 256 tokens, else
        router + top-k + align), GEMM 1, GEMM 2 and the output pass."""
        if self.M <= 256 and self.M * self.w.top_k <= 16384:
            route = 1
        else:
            route = (0 if self.w.logits_given else 1) + 1 + (1 if self.M * self.w.top_k <= 2048 else 2)
        # E4M3 weights: two more launches, the per-row quantizations of x and a
        return route + 1 + 2 + (2 if self.fp8 else 0)

    def step(self, moe, i, stream, ev):
        """One pass of the layer through the step entry points; ev[0..len(phases)]
        bracket the phases (routing S0-S2, GEMM 1 + activation, GEMM 2 +
        combine, and with E4M3 weights the quantizations of x and a)."""
        w, inp = self.w, self.inputs[i]
        x = inp["x"]
        res = x if w.residual else None
        ev[0].record(stream)
        moe.moe_route(w.top_k, self.B, self.ids, self.wts, self.sorted, self.eids, self.offs,
                      self.npost, self.ws, x=None if w.logits_given else x,
                      w_router=self.wr, router_logits=inp["router_logits"], router_bias=self.bias,
                      renormalize=w.renormalize, stream=stream)
        ev[1].record(stream)
        if self.fp8:
            moe.moe_quantize_rows_fp8(x, self.qx, self.sx, stream=stream)
            ev[2].record(stream)
            moe.moe_grouped_gemm_w13_act_fp8(self.qx, self.sx, self.w13, self.s13, self.sorted,
                                             self.eids, self.npost, w.top_k, self.B, self.a,
                                             stream=stream)
            ev[3].record(stream)
            moe.moe_quantize_rows_fp8(self.a, self.qa, self.sa, stream=stream)
            ev[4].record(stream)
            moe.moe_grouped_gemm_w2_combine_fp8(self.qa, self.sa, self.w2, self.s2, self.sorted,
                                                self.eids, self.npost, self.wts, w.top_k, self.B,
                                                self.y, self.ws, residual=res, stream=stream)
            ev[5].record(stream)
            return
        moe.moe_grouped_gemm_w13_act(x, self.w13, self.sorted, self.eids, self.npost, w.top_k,
                                     self.B, self.a, stream=stream)
        ev[2].record(stream)
        moe.moe_grouped_gemm_w2_combine(self.a, self.w2, self.sorted, self.eids, self.npost,
                                        self.wts, w.top_k, self.B, self.y, self.ws,
                                        residual=res, stream=stream)
        ev[3].record(stream)

    def forward(self, moe, i, stream):
        """One pass of the layer through the whole-layer entry point moe_forward
        (moe_forward_fp8 for E4M3 weights; what the timed steps run: its
        kernels may overlap each other's launch)."""
        w, inp = self.w, self.inputs[i]
        x = inp["x"]
        if self.fp8:
            moe.moe_forward_fp8(x, self.w13, self.s13, self.w2, self.s2, w.top_k, self.y, self.ws,
                                w_router=None if w.logits_given else self.wr,
                                router_logits=inp["router_logits"], router_bias=self.bias,
                                residual=x if w.residual else None, renormalize=w.renormalize,
                                block_size_m=self.B, stream=stream)
            return
        moe.moe_forward(x, self.w13, self.w2, w.top_k, self.y, self.ws,
                        w_router=None if w.logits_given else self.wr,
                        router_logits=inp["router_logits"], router_bias=self.bias,
                        residual=x if w.residual else None, renormalize=w.renormalize,
                        block_size_m=self.B, stream=stream)

    def distinct_experts(self, moe, i, stream):
        inp = self.inputs[i]
        logits = inp["router_logits"]
        if logits is None:
            moe.moe_router_logits(inp["x"], self.wr, self.logits, router_bias=self.bias, stream=stream)
            logits = self.logits
        moe.moe_topk_softmax(logits, self.w.top_k, self.ids, self.wts,
                             renormalize=self.w.renormalize, stream=stream)
        stream.synchronize()
        return int(torch.unique(self.ids).numel())

    def pairs_per_expert(self):
        """Pairs per expert of the last routing this layer computed."""
        n = torch.bincount(self.ids.reshape(-1).long(), minlength=self.w.E).cpu()
        active = n[n > 0]
        return {"max": int(n.max()), "mean_active": round(float(active.float().mean()), 2),
                "experts_without_pairs": int((n == 0).sum())}


def run_point(moe, w, M, steps, warmup, device, stream, flush, L=None, fp8=False):
    """Timed steps: moe_forward with CUDA events around each step only.  Then a
    breakdown pass through the step entry points with events between routing,
    GEMM 1 and GEMM 2 (events between kernels keep them from overlapping, so
    the breakdown is not the timed number)."""
    if L is None:
        L = Layer(moe, w, M, warmup + steps, device, fp8=fp8)
    # inputs are drawn on the default stream; the steps run on `stream`
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(warmup + steps)]
    with torch.cuda.stream(stream):
        torch.cuda.nvtx.range_push(f"warm-up M={M}")
        for i in range(warmup):
            flush.zero_()
            L.forward(moe, i, stream)
        stream.synchronize()
        torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_push(f"timed steps M={M}")
        for i in range(warmup, warmup + steps):
            flush.zero_()
            evs[i][0].record(stream)
            L.forward(moe, i, stream)
            evs[i][1].record(stream)
        stream.synchronize()
        torch.cuda.nvtx.range_pop()
    step_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(warmup, warmup + steps)]
    nb = min(steps, 10)
    ne = len(L.phases) + 1
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(ne)] for _ in range(nb)]
    with torch.cuda.stream(stream):
        # one untimed pass first: the first call of a step entry point pays
        # one-time host work (symbol lookups) inside its events
        L.step(moe, warmup, stream, [torch.cuda.Event(enable_timing=True) for _ in range(ne)])
        torch.cuda.nvtx.range_push(f"breakdown M={M}")
        for i in range(nb):
            flush.zero_()
            L.step(moe, warmup + i, stream, bev[i])
        stream.synchronize()
        torch.cuda.nvtx.range_pop()
    per = [[bev[i][j].elapsed_time(bev[i][j + 1]) for j in range(ne - 1)] for i in range(nb)]
    D = [L.distinct_experts(moe, i, stream) for i in range(warmup, warmup + steps)]
    return L, per, step_ms, D


def e2e_point(moe, L, steps, warmup, device, stream, flush):
    """Through moe_forward with pinned host buffers: every step copies its x
    (and logits) in and its y out.  Two passes over the same steps:

    serial     H2D, the layer and D2H of one step, then the next step (events
               around each step; the host waits after each);
    pipelined  how a serving loop streams batches: H2D on one stream, the
               layers on `stream`, D2H on a third, with two device buffers
               each for x and y, so that the copies of steps i+1 and i-1 run
               while step i computes; one pair of events around all steps.

    Both time every step's copies in and out; the pipelined total is the
    reported end-to-end number."""
    w, M = L.w, L.M
    n = warmup + steps
    hx = [inp["x"].cpu().pin_memory() for inp in L.inputs[:n]]
    hl = [inp["router_logits"].cpu().pin_memory() if inp["router_logits"] is not None else None
          for inp in L.inputs[:n]]
    hy = [torch.empty((M, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx = [torch.empty((M, w.H), dtype=torch.bfloat16, device=device) for _ in range(2)]
    dl = ([torch.empty((M, w.E), dtype=torch.bfloat16, device=device) for _ in range(2)]
          if w.logits_given else [None, None])
    dy = [L.y, torch.empty_like(L.y)]

    def forward(b):
        moe.moe_forward(dx[b], L.w13, L.w2, w.top_k, dy[b], L.ws, w_router=L.wr,
                        router_logits=dl[b], router_bias=L.bias,
                        residual=dx[b] if w.residual else None, renormalize=w.renormalize,
                        block_size_m=L.B, stream=stream)

    serial = []
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(n):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dx[0].copy_(hx[i], non_blocking=True)
            if dl[0] is not None:
                dl[0].copy_(hl[i], non_blocking=True)
            forward(0)
            hy[0].copy_(dy[0], non_blocking=True)
            e1.record(stream)
            stream.synchronize()
            if i >= warmup:
                serial.append(e0.elapsed_time(e1))

    h2d_s = torch.cuda.Stream(device)
    d2h_s = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def pipelined(first, count, timed):
        torch.cuda.synchronize()
        x_free = [None, None]    # the layer that last read dx[b]
        y_free = [None, None]    # the D2H that last read dy[b]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d_s.wait_event(start)
        for j in range(count):
            i, b = first + j, j % 2
            with torch.cuda.stream(h2d_s):
                if x_free[b] is not None:
                    h2d_s.wait_event(x_free[b])
                dx[b].copy_(hx[i], non_blocking=True)
                if dl[b] is not None:
                    dl[b].copy_(hl[i], non_blocking=True)
                x_in = ev()
                x_in.record(h2d_s)
            with torch.cuda.stream(stream):
                stream.wait_event(x_in)
                if y_free[b] is not None:
                    stream.wait_event(y_free[b])
                flush.zero_()
                forward(b)
                done = ev()
                done.record(stream)
                x_free[b] = done
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done)
                hy[b].copy_(dy[b], non_blocking=True)
                y_out = ev()
                y_out.record(d2h_s)
                y_free[b] = y_out
        for e in y_free:
            if e is not None:
                stream.wait_event(e)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    pipelined(0, warmup, False)
    total = pipelined(warmup, steps, True)
    h2d = M * w.H * 2 + (M * w.E * 2 if w.logits_given else 0)
    return total, serial, h2d, M * w.H * 2


def cpu_baseline(w, L, budget_s=12.0):
    """The oracle, as it stands, on the host cores: repeated whole-batch layers
    of this workload until about budget_s seconds have passed."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    inp = L.inputs[0]
    M = L.M
    sample_tokens = min(M, 64)
    x = synth.bf16_bits(inp["x"])[:sample_tokens]
    lg = None if inp["router_logits"] is None else synth.bf16_bits(inp["router_logits"])[:sample_tokens]
    w13, w2 = synth.bf16_bits(L.w13), synth.bf16_bits(L.w2)
    wr = None if L.wr is None else synth.bf16_bits(L.wr)
    bias = None if L.bias is None else L.bias.cpu().numpy()
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.moe_forward(x, w13, w2, w.top_k, w_router=wr, router_logits=lg, router_bias=bias,
                           residual=x if w.residual else None, renormalize=w.renormalize)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 50:
            break
    dt = time.perf_counter() - t0
    return {"value": round(n * sample_tokens / dt, 3), "unit": UNIT, "cores": oracle.get_threads(),
            "kind": "oracle",
            "sample": f"{n} x {w.name} layer on {sample_tokens} tokens (full expert weights), {dt:.1f} s"}


# ----------------------------------------------------------------------------- the 64-layer stack

class Stack:
    """The 64-layer decode stack: independent seeded weights per layer, layer
    l+1 reads y_l (computed with residual x_l), one workspace for every layer."""

    def __init__(self, moe, w, M, n_inputs, device):
        self.w, self.M = w, M
        self.layers = [synth.layer_weights(w, layer=l, device=device) for l in range(w.layers)]
        self.inputs = [synth.layer_input(w, M, rep=r, device=device)["x"] for r in range(n_inputs)]
        self.B = w.block_size_m or moe.moe_pick_block_size(M, w.E, w.top_k, w.H, w.I)
        self.ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, 0, device=device)
        self.buf = [torch.empty((M, w.H), dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.ids = [torch.empty((M, w.top_k), dtype=torch.int32, device=device)
                    for _ in range(w.layers)]

    @staticmethod
    def kernels_for(w, M):
        """moe_forward per layer: routing (one fused launch up to 256 tokens, else
        router + top-k + align), GEMM 1, GEMM 2 and the output pass."""
        if M <= 256 and M * w.top_k <= 16384:
            route = 1
        else:
            route = 2 + (1 if M * w.top_k <= 2048 else 2)
        return w.layers * (route + 3)

    def step(self, moe, x, stream, keep_ids=False):
        """x (held in buf[0]) through every layer; returns the output buffer."""
        w = self.w
        cur, nxt = self.buf[0], self.buf[1]
        if x is not cur:
            cur.copy_(x, non_blocking=True)
        for l, wt in enumerate(self.layers):
            moe.moe_forward(cur, wt["w13"], wt["w2"], w.top_k, nxt, self.ws, w_router=wt["w_router"],
                            router_bias=wt["router_bias"], residual=cur, renormalize=w.renormalize,
                            block_size_m=self.B, topk_ids_out=self.ids[l] if keep_ids else None,
                            stream=stream)
            cur, nxt = nxt, cur  # ping-pong: a layer's input is dead once its output exists
        return cur


def stack_bytes(w, M, distinct_per_layer):
    return sum(layer_bytes(w, M, d) for d in distinct_per_layer)


def run_stack(moe, args, w, M, device, stream, flush, world):
    S = Stack(moe, w, M, args.warmup + args.steps, device)
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        # capture one step (64 layers) reading buf[0]; replay it per step
        with torch.cuda.stream(stream):
            S.step(moe, S.buf[0], stream)  # first calls do per-device set-up outside the capture
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            out_buf = S.step(moe, S.buf[0], stream)
    times = []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if graph is not None:
                    S.buf[0].copy_(S.inputs[i], non_blocking=True)
                    graph.replay()
                else:
                    S.step(moe, S.inputs[i], stream)
                e1.record(stream)
                if i >= args.warmup:
                    times.append((e0, e1))
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in times]
    # distinct experts per layer of the last step's routing, for the byte count
    with torch.cuda.stream(stream):
        S.step(moe, S.inputs[-1], stream, keep_ids=True)
    stream.synchronize()
    D = [int(torch.unique(ids).numel()) for ids in S.ids]
    return S, step_ms, D, clk


def ours_stack(args, moe, w, M, device, stream, flush, world, rank, peaks):
    S, step_ms, D, clk = run_stack(moe, args, w, M, device, stream, flush, world)
    block_size = S.B
    one_kernel = None
    if M <= 16 and not args.no_points:
        # the same step with the one-kernel decode layer (opt-in), for comparison
        del S
        os.environ["MOE_DECODE_LAYER"] = "on"
        try:
            _, k_ms, _, _ = run_stack(moe, args, w, M, device, stream, flush, world)
        finally:
            os.environ.pop("MOE_DECODE_LAYER", None)
        k_total = max_over_ranks(sum(k_ms), world, device)
        one_kernel = {"ms_per_step": round(k_total / args.steps, 5),
                      "tokens_per_s": round(world * M * args.steps / (k_total / 1e3), 2)}
        S = None
    total_ms = max_over_ranks(sum(step_ms), world, device)
    ms_per_step = total_ms / args.steps
    value = world * M * args.steps / (total_ms / 1e3)
    sb = stack_bytes(w, M, D)
    gbs = sb / (ms_per_step / 1e3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded x ~ N(0,1), 64 layers of weights ~ N(0,0.02), bf16; new x every step",
        "config": {"workload": f"{w.name}_m{M}", "M": M, "E": w.E, "top_k": w.top_k, "H": w.H,
                   "I": w.I, "layers": w.layers, "block_size_m": block_size, "residual": True,
                   "cuda_graph": bool(args.graph),
                   "l2": f"flushed between steps ({args.flush_mb} MB write, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "whole 64-layer step", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "traffic": None, "peak_source": peaks["source"], "algorithmic_bytes": int(sb)},
        "distinct_experts_per_layer": round(statistics.mean(D), 2),
        "gpu": gpu_info(device),
        "e2e": None, "cpu_baseline": None,
        "gpu_launches": Stack.kernels_for(w, M) * args.steps,
        "clocks": clk.summary(),
        "one_kernel_layer": one_kernel,
    }
    print(json.dumps(line), flush=True)



def prefill_point(moe, args, device, stream, flush, peaks, world):
    """The prefill layer (Qwen3-30B-A3B shape, Zipf(1.1) router skew) at
    M = 16384: tokens/s, the layer's fraction of the bf16 tensor-core peak and
    the roofline of its dominant kernel, grouped GEMM 1 (tensor-bound there),
    from the breakdown pass after the timed steps."""
    w = synth.WORKLOADS[WORKLOAD_CFG["prefill"]]
    M = max(w.Ms)
    steps = max(5, args.steps // 2)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        L, per, step_ms, D = run_point(moe, w, M, steps, args.warmup, device, stream, flush)
    total = max_over_ranks(sum(step_ms), world, device)
    ms = total / steps
    gemm1_ms = statistics.mean(p[1] for p in per)
    g1_tflops = gemm1_flops(w, M) / (gemm1_ms / 1e3) / 1e12
    lay_tflops = layer_flops(w, M) / (ms / 1e3) / 1e12
    lay_bytes = statistics.mean(layer_bytes(w, M, d) for d in D)
    out = {
        "workload": f"{w.name}_m{M}", "M": M, "block_size_m": L.B,
        "value": round(world * M / (ms / 1e3), 1), "unit": UNIT, "ms_per_layer": round(ms, 5),
        "layer_tc_frac": round(lay_tflops / peaks["bf16_tflops"], 4),
        "layer_hbm_frac": round(lay_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
        "roofline": {"kernel": "grouped GEMM 1 + SiLU-and-mul", "bound": "tensor",
                     "achieved": round(g1_tflops, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(g1_tflops / peaks["bf16_tflops"], 4),
                     "algorithmic_flops": int(gemm1_flops(w, M)), "ms": round(gemm1_ms, 5),
                     "traffic": profiled_traffic(f"k_gemm_tc_gemm1_{w.name}_m{M}.md", L.B),
                     "peak_source": peaks["source"]},
        "step_breakdown_ms": {k: round(statistics.mean(p[j] for p in per), 5) for j, k in
                              enumerate(["route", "gemm1_act", "gemm2_combine"])},
        "distinct_experts": round(statistics.mean(D), 2),
        "steps": steps, "warmup": args.warmup,
        "gpu_launches": L.kernels_per_step() * steps,
        "clocks": clk.summary(),
    }
    del L
    return out


def fp8_point(moe, args, device, stream, flush, peaks, world, cfg_name, M):
    """The layer with E4M3 expert weights (moe_forward_fp8) on one workload
    point: tokens/s and the roofline of grouped GEMM 1 against HBM (decode) or
    the FP8 tensor peak (prefill), taken as the measured bf16 peak times the
    nominal FP8/bf16 ratio 2 (4.5 / 2.25 PFLOP/s dense)."""
    w = synth.WORKLOADS[WORKLOAD_CFG[cfg_name]]
    steps = max(5, args.steps // 2)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        L, per, step_ms, D = run_point(moe, w, M, steps, args.warmup, device, stream, flush, fp8=True)
    total = max_over_ranks(sum(step_ms), world, device)
    ms = total / steps
    g1 = L.phases.index("gemm1_act")
    gemm1_ms = statistics.mean(p[g1] for p in per)
    f8_tflops = 2.0 * peaks["bf16_tflops"]
    g1_flops = gemm1_flops(w, M)
    g1_bytes = statistics.mean(gemm1_bytes_fp8(w, M, d) for d in D)
    ridge = f8_tflops * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if g1_flops / g1_bytes > ridge:
        roof = {"bound": "tensor", "achieved": round(g1_flops / (gemm1_ms / 1e3) / 1e12, 1),
                "peak": f8_tflops, "unit": "TFLOP/s", "algorithmic_flops": int(g1_flops),
                "peak_source": f"{peaks['source']} bf16 x 2 (nominal FP8/bf16 ratio)"}
    else:
        roof = {"bound": "hbm", "achieved": round(g1_bytes / (gemm1_ms / 1e3) / 1e9, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "algorithmic_bytes": int(g1_bytes),
                "peak_source": peaks["source"]}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    lay_bytes = statistics.mean(layer_bytes_fp8(w, M, d) for d in D)
    out = {
        "workload": f"{w.name}_fp8_m{M}", "M": M, "block_size_m": L.B, "dtype": "e4m3 x e4m3 -> f32",
        "value": round(world * M / (ms / 1e3), 1), "unit": UNIT, "ms_per_layer": round(ms, 5),
        "layer_hbm_frac": round(lay_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
        "layer_tc_frac_fp8": round(layer_flops(w, M) / (ms / 1e3) / 1e12 / f8_tflops, 4),
        "roofline": dict({"kernel": "grouped GEMM 1 (E4M3) + SiLU-and-mul"}, **roof,
                         ms=round(gemm1_ms, 5),
                         traffic=profiled_traffic(f"k_gemm_tc_gemm1_{w.name}_fp8_m{M}.md", L.B)),
        "step_breakdown_ms": {k: round(statistics.mean(p[j] for p in per), 5)
                              for j, k in enumerate(L.phases)},
        "distinct_experts": round(statistics.mean(D), 2),
        "steps": steps, "warmup": args.warmup,
        "gpu_launches": L.kernels_per_step() * steps,
        "clocks": clk.summary(),
    }
    del L
    return out


def ours(args):
    import mixture_experts_layer_renorm_gb300 as moe
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    moe.load_library(build_if_missing=True)
    w = synth.WORKLOADS[WORKLOAD_CFG[args.workload]]
    if args.block_size:
        w = dataclasses.replace(w, block_size_m=args.block_size)
    M = args.M or max(w.Ms)
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=device)
    flush = torch.empty(args.flush_mb << 20, dtype=torch.uint8, device=device)
    if w.layers > 1:
        ours_stack(args, moe, w, M, device, stream, flush, world, rank, peaks)
        return
    if args.fp8:
        # one point with E4M3 expert weights (the fp8 entry of the default
        # decode line, for any single-layer workload and M)
        out = fp8_point(moe, args, device, stream, flush, peaks, world, args.workload, M)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return

    L = Layer(moe, w, M, args.warmup + args.steps, device)
    # the timed region: K steps, barrier + synchronize on both sides
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        L, per, step_ms, D = run_point(moe, w, M, args.steps, args.warmup, device, stream, flush, L)
    torch.cuda.synchronize()
    barrier(world)
    local_total_ms = sum(step_ms)
    total_ms = max_over_ranks(local_total_ms, world, device)
    ms_per_step = total_ms / args.steps
    value = world * M * args.steps / (total_ms / 1e3)

    gemm1_ms = statistics.mean(p[1] for p in per)
    D_mean = statistics.mean(D)
    g1_bytes = statistics.mean(gemm1_bytes(w, M, d) for d in D)
    g1_flops = gemm1_flops(w, M)
    lay_bytes = statistics.mean(layer_bytes(w, M, d) for d in D)
    lay_gbs = lay_bytes / (ms_per_step / 1e3) / 1e9
    flops = layer_flops(w, M)
    lay_tflops = flops / (ms_per_step / 1e3) / 1e12
    # which roof binds GEMM 1: its arithmetic intensity against the ridge of the measured peaks
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if g1_flops / g1_bytes > ridge:
        roof = {"bound": "tensor", "achieved": round(g1_flops / (gemm1_ms / 1e3) / 1e12, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "algorithmic_flops": int(g1_flops)}
    else:
        roof = {"bound": "hbm", "achieved": round(g1_bytes / (gemm1_ms / 1e3) / 1e9, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "algorithmic_bytes": int(g1_bytes)}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)

    e2e_pipe, e2e_serial, h2d, d2h = e2e_point(moe, L, args.steps, args.warmup, device, stream, flush)
    pipe_total = max_over_ranks(e2e_pipe, world, device)
    serial_total = max_over_ranks(sum(e2e_serial), world, device)
    # the better of the two loops a user would run: small batches are latency
    # bound (the serial loop), large ones hide the copies behind the layer
    pipelined_better = pipe_total < serial_total
    e2e_total = pipe_total if pipelined_better else serial_total
    e2e_value = world * M * args.steps / (e2e_total / 1e3)

    points = []
    if not args.no_points:
        for m in w.Ms:
            if m == M:
                continue
            _, p_per, p_ms, p_D = run_point(moe, w, m, max(5, args.steps // 2), args.warmup, device,
                                            stream, flush)
            ms = statistics.mean(p_ms)
            bpl = statistics.mean(layer_bytes(w, m, d) for d in p_D)
            points.append({"M": m, "tokens_per_s": round(m / (ms / 1e3), 1), "ms_per_layer": round(ms, 5),
                           "hbm_frac_layer": round(bpl / (ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                           "tc_frac_layer": round(layer_flops(w, m) / (ms / 1e3) / 1e12
                                                  / peaks["bf16_tflops"], 4),
                           "route_ms": round(statistics.mean(p[0] for p in p_per), 5),
                           "gemm1_ms": round(statistics.mean(p[1] for p in p_per), 5),
                           "gemm2_ms": round(statistics.mean(p[2] for p in p_per), 5),
                           "distinct_experts": round(statistics.mean(p_D), 2)})

    # the one-kernel decode layer (opt-in) beside the default path, at the
    # decode sizes it serves
    one_kernel = []
    if not args.no_points:
        for m in sorted(set(w.Ms) | {M}):
            if m > 16:
                continue
            os.environ["MOE_DECODE_LAYER"] = "on"
            try:
                _, _, k_ms, _ = run_point(moe, w, m, max(5, args.steps // 2), args.warmup, device,
                                          stream, flush)
            finally:
                os.environ.pop("MOE_DECODE_LAYER", None)
            ms = statistics.mean(k_ms)
            one_kernel.append({"M": m, "ms_per_layer": round(ms, 5),
                               "tokens_per_s": round(m / (ms / 1e3), 1)})

    # the prefill half of the metric (% of bf16 tensor-core peak), timed in the
    # same run: the Zipf-skewed prefill layer at its largest batch
    prefill = None
    if args.workload == "decode" and not args.no_prefill:
        prefill = prefill_point(moe, args, device, stream, flush, peaks, world)

    # the same two points with E4M3 expert weights (moe_forward_fp8)
    fp8 = None
    if args.workload == "decode" and not args.no_fp8:
        fp8 = {"decode": fp8_point(moe, args, device, stream, flush, peaks, world, "decode", M)}
        if not args.no_prefill:
            fp8["prefill"] = fp8_point(moe, args, device, stream, flush, peaks, world, "prefill",
                                       max(synth.WORKLOADS[WORKLOAD_CFG["prefill"]].Ms))

    if rank != 0:
        return
    cpu = None if (world > 1 or args.no_cpu_baseline) else cpu_baseline(w, L)
    kernels = L.kernels_per_step()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded x ~ N(0,1), weights ~ N(0,0.02), bf16; new x every step",
        "config": {"workload": f"{w.name}_m{M}", "M": M, "E": w.E, "top_k": w.top_k, "H": w.H,
                   "I": w.I, "block_size_m": L.B, "renormalize": w.renormalize,
                   "l2": f"flushed between steps ({args.flush_mb} MB write, outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": dict({"kernel": "grouped GEMM 1 + SiLU-and-mul"}, **roof,
                         traffic=profiled_traffic(f"k_gemm_tc_gemm1_{w.name}_m{M}.md", L.B),
                         peak_source=peaks["source"], ms=round(gemm1_ms, 5),
                         timing="GEMM 1 between CUDA events on its stream, in the breakdown pass "
                                "that follows the timed steps"),
        "layer_roofline": {"achieved_gbs": round(lay_gbs, 1),
                           "hbm_frac": round(lay_gbs / peaks["hbm_gbs"], 4),
                           "achieved_tflops": round(lay_tflops, 3),
                           "tc_frac": round(lay_tflops / peaks["bf16_tflops"], 5),
                           "algorithmic_bytes": int(lay_bytes), "flops": int(flops),
                           "distinct_experts": round(D_mean, 2)},
        "pairs_per_expert": L.pairs_per_expert(),
        "gpu": gpu_info(device),
        "step_breakdown_ms": {k: round(statistics.mean(p[j] for p in per), 5) for j, k in
                              enumerate(["route", "gemm1_act", "gemm2_combine"])},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_total / args.steps, 5),
                "mode": ("pipelined: H2D, layer and D2H of consecutive steps on three streams"
                         if pipelined_better else "serial: H2D, layer, D2H, then the next step"),
                "serial_ms_per_step": round(serial_total / args.steps, 5),
                "pipelined_ms_per_step": round(pipe_total / args.steps, 5)},
        "cpu_baseline": cpu,
        "gpu_launches": kernels * args.steps,
        "clocks": clk.summary(),
        "points": points,
        "one_kernel_layer": one_kernel,
        "prefill": prefill,
        "fp8": fp8,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- reference arm

def reference(args):
    """The CPU oracle as the reference arm: each step is the layer on a bounded
    sample of the workload's tokens, on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    w = synth.WORKLOADS[WORKLOAD_CFG[args.workload]]
    M = args.M or max(w.Ms)
    sample = min(M, args.ref_tokens)
    wt = synth.layer_weights(w, device="cuda" if torch.cuda.is_available() else "cpu")
    w13, w2 = synth.bf16_bits(wt["w13"]), synth.bf16_bits(wt["w2"])
    wr = None if wt["w_router"] is None else synth.bf16_bits(wt["w_router"])
    bias = None if wt["router_bias"] is None else wt["router_bias"].cpu().numpy()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    times = []
    for i in range(args.warmup + args.steps):
        inp = synth.layer_input(w, M, rep=i, device=dev)
        x = synth.bf16_bits(inp["x"])[:sample]
        lg = None if inp["router_logits"] is None else synth.bf16_bits(inp["router_logits"])[:sample]
        t0 = time.perf_counter()
        oracle.moe_forward(np.ascontiguousarray(x), w13, w2, w.top_k, w_router=wr,
                           router_logits=lg, router_bias=bias,
                           residual=x if w.residual else None, renormalize=w.renormalize)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = sample * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded x ~ N(0,1), weights ~ N(0,0.02), bf16",
        "config": {"workload": f"{w.name}_m{M}", "M": M, "E": w.E, "top_k": w.top_k, "H": w.H,
                   "I": w.I, "sampled_tokens_per_step": sample},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": oracle.get_threads(),
                         "kind": "oracle",
                         "sample": f"{sample} of {M} tokens per step, full expert weights"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_CFG), default="decode")
    ap.add_argument("--M", type=int, default=0, help="tokens per step (default: the largest of the workload)")
    ap.add_argument("--flush-mb", type=int, default=512)
    ap.add_argument("--no-points", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="time only the workload's layer with E4M3 expert weights (moe_forward_fp8)")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the E4M3-weight points of the decode run")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workload: skip the prefill point (M = 16384) in the same run")
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--block-size", type=int, default=0,
                    help="block_size_m of the align and the grouped GEMMs (default: the library's pick)")
    ap.add_argument("--graph", action="store_true",
                    help="stack workload: replay each 64-layer step from a CUDA graph")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
