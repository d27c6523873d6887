#!/usr/bin/env python
"""Benchmark of the w8a8 scaled quantiser + scaled matmul on GB300.

Headline workload (one "step"): Llama-3-8B decode, fp8 e4m3 w8a8.  For every
token count M in {1, 16, 64, 256} and every projection -- QKV [6144 x 4096]
(merged layer, one shared per-tensor weight scale), O [4096 x 4096],
gate-up [28672 x 4096], down [4096 x 14336] -- the step quantises the bf16
activations (dynamic, per token) and runs the scaled matmul with per-channel
weight scales to a bf16 output.  Weights are quantised once at set-up and
stay resident; the 218 MB of weights are larger than the 129 MB L2, so every
step streams them from HBM.  The step is captured once in a CUDA graph and
replayed.

Timing: W warm-up steps, then samples of exactly K steps, each bracketed by
a device synchronisation (and a barrier over ranks) with CUDA events on the
launching stream, repeated until at least half a second has been timed so
that the clock sampler sees the load; the median sample is reported.

The JSON line also carries the other configurations under "configs", each
with its roofline and the oracle timed on the host cores on a bounded
sample: fp8 prefill at M = 4096 with static per-tensor scales, int8 w8a8 at
Llama-3-70B shapes and M = 8192, the scaled FP8 KV-cache round trip, decode
attention over the e4m3 KV cache and the activation quantiser at prefill
sizes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica (the path has
no exchange step); value is the aggregate over ranks and time is the max
over ranks.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "w8a8 scaled-GEMM TFLOP/s (% dense FP8/INT8 peak); quant GB/s (% HBM) on 1 GB300"
UNIT = "TFLOP/s"

DECODE_MS = (1, 16, 64, 256)
LLAMA8B = (("qkv", 6144, 4096, True), ("o", 4096, 4096, False),
           ("gate_up", 28672, 4096, False), ("down", 4096, 14336, False))
LLAMA70B = (("qkv", 10240, 8192), ("gate_up", 57344, 8192), ("down", 8192, 28672))

QUANT_PREFILL = ((4096, 4096), (4096, 14336), (8192, 8192), (8192, 28672))
ATTN_SHAPE = (16, 4096, 8, 32, 128)   # sequences, tokens, KV heads, query heads, head dim
MIN_TIMED_S = 0.5
DECODE_WORKLOAD = ("Llama-3-8B decode fp8 e4m3: M in {1,16,64,256} x QKV/O/gate-up/down, dynamic per-token act, "
                   "per-channel weights (QKV shared)")

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks and throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_ratio_for(kernel_key: str):
    """DRAM bytes / algorithmic bytes of a kernel from the committed ncu
    capture (profiles/traffic.json), if it was taken on the current kernel
    source (the source hash must match); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get(kernel_key)
    if not ent:
        return None
    src = os.path.join(ROOT, ent.get("source", ""))
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except Exception:
        return None
    if h != ent.get("source_sha256_16"):
        return None
    return ent.get("dram_over_algorithmic")


def max_over_ranks(t_local: float, device=None) -> float:
    """Max of a per-rank time over all ranks (identity without a process
    group).  The replicas share no data; this is the timing reduction only."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t_local
    tt = torch.tensor([t_local], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def aggregate_tflops(flops_per_step_per_rank: float, steps: int, t_max: float, world: int) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (weak scaling: per-rank work is fixed)."""
    return world * flops_per_step_per_rank * steps / t_max / 1e12


# ---------------------------------------------------------------- workloads (GPU)

class DecodeWorkload:
    """Llama-3-8B decode fp8: 4 token counts x 4 projections."""

    def __init__(self, dev, seed=1000):
        import torch
        import int8_w8a8_scaled_gb300 as w8
        import synthetic_inputs as si
        self.torch, self.w8 = torch, w8
        self.weights = {}
        for i, (name, N, K, shared) in enumerate(LLAMA8B):
            wt = si.normal((N, K), seed=seed + i, std=0.02, device=dev)
            wq = torch.empty(N, K, dtype=torch.float8_e4m3fn, device=dev)
            sw = torch.empty(1 if shared else N, dtype=torch.float32, device=dev)
            # merged QKV: one per-tensor scale over the concatenated weight
            w8.scaled_quant(wt, wq, sw, per_token=not shared, dynamic=True)
            self.weights[name] = (wq, sw, N, K)
            del wt
        self.items = []
        ws_need = 0
        for M in DECODE_MS:
            for j, (name, N, K, _) in enumerate(LLAMA8B):
                x = si.normal_with_outliers((M, K), seed=seed + 100 + M * 10 + j, device=dev)
                aq = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=dev)
                sa = torch.empty(M, dtype=torch.float32, device=dev)
                out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
                cfg = None
                # quantiser + matmul (the automatic route of quant_scaled_mm;
                # `fused` items would run its one-kernel route)
                fused = False
                self.items.append({"M": M, "name": name, "x": x, "aq": aq, "sa": sa, "out": out, "cfg": cfg,
                                   "fused": fused})
                ws_need = max(ws_need, w8.mm_workspace_size(M, N, K, w8.E4M3, cfg),
                              w8._lib.load().w8a8_quant_scaled_mm_workspace_size(M, N, K, w8.E4M3))
        self.ws = w8.Workspace(ws_need, dev)
        torch.cuda.synchronize()

    def flops(self, items=None):
        return sum(2.0 * it["M"] * self.weights[it["name"]][2] * self.weights[it["name"]][3]
                   for it in (items if items is not None else self.items))

    def gemm_bytes(self, items=None):
        # algorithmic bytes of the matmul kernels: 1-byte weights once, the
        # activations once (16-bit x where the kernel quantises them itself,
        # 1-byte codes otherwise), 16-bit output, fp32 scales
        tot = 0
        for it in (items if items is not None else self.items):
            _, sw, N, K = self.weights[it["name"]]
            M = it["M"]
            tot += N * K + (2 if it["fused"] else 1) * M * K + 2 * M * N + 4 * (M + sw.numel())
        return tot

    def quant_bytes(self):
        # the separate quantiser kernels: 2 B read + 1 B write per element, 4 B scale per row
        return sum(it["M"] * it["x"].shape[1] * 3 + 4 * it["M"] for it in self.items if not it["fused"])

    def run_quant(self):
        for it in self.items:
            if not it["fused"]:
                self.w8.scaled_quant(it["x"], it["aq"], it["sa"], per_token=True, dynamic=True)

    def _fused(self, it):
        wq, sw, _, _ = self.weights[it["name"]]
        self.w8.quant_scaled_mm(it["x"], wq, sw, it["out"], scale_a_out=it["sa"], workspace=self.ws)

    def run_gemm(self, items=None):
        # the matmul kernels of a step (those that quantise their own
        # activations included); the others read codes quantised beforehand
        for it in (items if items is not None else self.items):
            wq, sw, _, _ = self.weights[it["name"]]
            if it["fused"]:
                self._fused(it)
            else:
                self.w8.scaled_mm(it["aq"], wq, it["sa"], sw, it["out"], workspace=self.ws, config=it["cfg"])

    def second_set(self):
        """The step's activations, codes, scales and outputs once more (the
        weights and workspace are shared), for double-buffered host copies."""
        return [dict(it, x=it["x"].clone(), aq=it["aq"].clone(), sa=it["sa"].clone(), out=it["out"].clone())
                for it in self.items]

    def run_step(self, items=None):
        for it in (items if items is not None else self.items):
            wq, sw, _, _ = self.weights[it["name"]]
            if it["fused"]:
                self._fused(it)
            else:
                self.w8.scaled_quant(it["x"], it["aq"], it["sa"], per_token=True, dynamic=True)
                self.w8.scaled_mm(it["aq"], wq, it["sa"], sw, it["out"], workspace=self.ws, config=it["cfg"])

    def launches_per_step(self):
        return sum(1 if it["fused"] else 2 for it in self.items)

    def gemms_per_step(self):
        return len(self.items)


def graph_of(fn, stream):
    import torch
    with torch.cuda.stream(stream):
        fn()  # warm: one-time host set-up happens outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def _time_once(run, stream, steps, barrier=None):
    """Seconds for exactly `steps` calls of run() (CUDA events on `stream`,
    device synchronised and ranks at a barrier on both sides)."""
    import torch
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            run()
        end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end) / 1e3


def timed(run, stream, steps, warmup, min_s=MIN_TIMED_S, barrier=None, device=None):
    """W warm-up calls, then timed samples of exactly `steps` calls each,
    repeated until at least `min_s` seconds of timed work (so that the clock
    sampler sees the load).  Every rank runs the same number of samples.
    Returns (median seconds per sample, number of samples)."""
    import math
    with_stream(stream, lambda: [run() for _ in range(warmup)])
    probe = _time_once(run, stream, steps, barrier)
    n = max(1, min(10_000, math.ceil(min_s / max(probe, 1e-9))))
    n = int(max_over_ranks(float(n), device))
    ts = [_time_once(run, stream, steps, barrier) for _ in range(n)]
    return statistics.median(ts), n


def with_stream(stream, fn):
    import torch
    with torch.cuda.stream(stream):
        return fn()


def time_graph(g, stream, steps, warmup, barrier=None, device=None):
    """Median seconds per step of graph replays (see timed())."""
    t, n = timed(g.replay, stream, steps, warmup, barrier=barrier, device=device)
    return t / steps, n


def r4(x):
    """Four significant digits (keeps the JSON line short)."""
    if x is None:
        return None
    return float(f"{x:.4g}")


def measure_prefill_fp8(dev, steps, warmup, stream, pk):
    """Llama-3-8B prefill, M = 4096, static per-tensor activation and weight
    scales (absmax / 448 of a seeded calibration tensor), heavy-tailed
    activation columns (Student-t, nu = 4)."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    M = 4096
    items = []
    for j, (name, N, K, _) in enumerate(LLAMA8B):
        wt = si.normal((N, K), seed=2000 + j, std=0.02, device=dev)
        wq = torch.empty(N, K, dtype=torch.float8_e4m3fn, device=dev)
        sw = torch.empty(1, dtype=torch.float32, device=dev)
        w8.scaled_quant(wt, wq, sw, per_token=False, dynamic=True)
        del wt
        calib = si.student_t_columns((M, K), seed=2100 + j, device=dev)
        cq = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=dev)
        sa = torch.empty(1, dtype=torch.float32, device=dev)
        w8.scaled_quant(calib, cq, sa, per_token=False, dynamic=True)  # calibration -> static scale
        del calib, cq
        x = si.student_t_columns((M, K), seed=2200 + j, device=dev)
        aq = torch.empty(M, K, dtype=torch.float8_e4m3fn, device=dev)
        out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        items.append((x, aq, sa, wq, sw, out, N, K))
    ws = w8.Workspace(max(w8.mm_workspace_size(M, N, K, w8.E4M3) for *_, N, K in items), dev)

    def step():
        for x, aq, sa, wq, sw, out, N, K in items:
            w8.scaled_quant(x, aq, sa, per_token=False, dynamic=False)
            w8.scaled_mm(aq, wq, sa, sw, out, workspace=ws)

    def gemm_only():
        for x, aq, sa, wq, sw, out, N, K in items:
            w8.scaled_mm(aq, wq, sa, sw, out, workspace=ws)

    flops = sum(2.0 * M * N * K for *_, N, K in items)
    t_step, n1 = time_graph(graph_of(step, stream), stream, steps, warmup)
    t_gemm, n2 = time_graph(graph_of(gemm_only, stream), stream, steps, warmup)
    fp8_peak = pk["bf16_tflops"] * 2.0  # nominal fp8 / bf16 ratio 4.5 / 2.25
    ach = flops / t_gemm / 1e12
    del items
    torch.cuda.empty_cache()
    return {"value": r4(flops / t_step / 1e12), "unit": "TFLOP/s", "ms_per_step": r4(t_step * 1e3),
            "samples": n1 + n2,
            "roofline": {"bound": "tensor", "achieved": r4(ach), "peak": r4(fp8_peak), "frac": r4(ach / fp8_peak),
                         "kernel": "4 GEMMs"}}


def measure_int8_70b(dev, steps, warmup, stream, pk):
    """int8 w8a8 at Llama-3-70B shapes, M = 8192: dynamic per-token /127
    activations, per-channel int8 weights, int32 accumulation, fp16 out."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    M = 8192
    items = []
    for j, (name, N, K) in enumerate(LLAMA70B):
        wt = si.normal((N, K), seed=3000 + j, std=0.02, device=dev)
        wq = torch.empty(N, K, dtype=torch.int8, device=dev)
        sw = torch.empty(N, dtype=torch.float32, device=dev)
        w8.scaled_quant(wt, wq, sw, per_token=True, dynamic=True)
        del wt
        x = si.normal_with_outliers((M, K), seed=3100 + j, device=dev)
        aq = torch.empty(M, K, dtype=torch.int8, device=dev)
        sa = torch.empty(M, dtype=torch.float32, device=dev)
        out = torch.empty(M, N, dtype=torch.float16, device=dev)
        items.append((x, aq, sa, wq, sw, out, N, K))
    ws = w8.Workspace(max(w8.mm_workspace_size(M, N, K, w8.INT8) for *_, N, K in items), dev)

    def step():
        for x, aq, sa, wq, sw, out, N, K in items:
            w8.scaled_quant(x, aq, sa, per_token=True, dynamic=True)
            w8.scaled_mm(aq, wq, sa, sw, out, workspace=ws)

    flops = sum(2.0 * M * N * K for *_, N, K in items)
    # a step is ~13 ms: one step per sample
    t_step, n = time_graph(graph_of(step, stream), stream, 1, warmup)
    ach = flops / t_step / 1e12
    del items
    torch.cuda.empty_cache()
    return {"value": r4(ach), "unit": "TFLOP/s", "ms_per_step": r4(t_step * 1e3), "samples": n,
            "roofline": {"bound": "tensor", "achieved": r4(ach), "peak": r4(pk["bf16_tflops"]),
                         "frac": r4(ach / pk["bf16_tflops"]), "frac_fp8": r4(ach / (2.0 * pk["bf16_tflops"])),
                         "kernel": "quant+GEMM, f16 route"}}


def measure_kv(dev, steps, warmup, stream, pk):
    """Scaled FP8 KV cache: K and V bf16 [65536, 8, 128] with rare spikes,
    per-tensor dynamic absmax/448 quantisation to e4m3 then dequantisation."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    T, H, D = 65536, 8, 128
    bufs = []
    for j in range(2):
        x = si.kv_with_spikes(T, H, D, seed=4000 + j, device=dev).reshape(T * H, D)
        q = torch.empty(T * H, D, dtype=torch.float8_e4m3fn, device=dev)
        s = torch.empty(1, dtype=torch.float32, device=dev)
        y = torch.empty(T * H, D, dtype=torch.bfloat16, device=dev)
        wsq = torch.zeros(16, dtype=torch.uint8, device=dev)
        bufs.append((x, q, s, y, wsq))
    n = T * H * D

    def quant():
        for x, q, s, y, wsq in bufs:
            w8.scaled_quant(x, q, s, per_token=False, dynamic=True, workspace=wsq)

    def dequant():
        for x, q, s, y, wsq in bufs:
            w8.scaled_dequant(q, s, y)

    tq, n1 = time_graph(graph_of(quant, stream), stream, steps, warmup)
    td, n2 = time_graph(graph_of(dequant, stream), stream, steps, warmup)
    qb, db = 2 * n * 5, 2 * n * 3
    hbm = pk["hbm_gbs"]
    return {"value": r4(qb / tq / 1e9), "unit": "GB/s", "dequant_gbs": r4(db / td / 1e9),
            "us": [r4(tq * 1e6), r4(td * 1e6)], "samples": n1 + n2,
            "roofline": {"bound": "hbm", "frac": r4(qb / tq / 1e9 / hbm), "dequant_frac": r4(db / td / 1e9 / hbm),
                         "peak": r4(hbm), "kernel": "5 B/elt, dequant 3"}}


def measure_quant_prefill(dev, steps, warmup, stream, pk):
    """The activation quantiser at prefill sizes: [4096, 4096], [4096,
    14336], [8192, 8192], [8192, 28672] bf16, dynamic per token, e4m3."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    bufs = []
    for j, (R, C) in enumerate(QUANT_PREFILL):
        x = si.normal_with_outliers((R, C), seed=6000 + j, device=dev)
        q = torch.empty(R, C, dtype=torch.float8_e4m3fn, device=dev)
        s = torch.empty(R, dtype=torch.float32, device=dev)
        bufs.append((x, q, s))

    def run():
        for x, q, s in bufs:
            w8.scaled_quant(x, q, s, per_token=True, dynamic=True)

    t, n = time_graph(graph_of(run, stream), stream, steps, warmup)
    byts = sum(R * C * 3 + 4 * R for R, C in QUANT_PREFILL)
    gbs = byts / t / 1e9
    del bufs
    torch.cuda.empty_cache()
    return {"value": r4(gbs), "unit": "GB/s", "us": r4(t * 1e6), "samples": n,
            "roofline": {"bound": "hbm", "achieved": r4(gbs), "peak": r4(pk["hbm_gbs"]),
                         "frac": r4(gbs / pk["hbm_gbs"]), "kernel": "3 B/elt + 4 B/row"}}


def measure_kv_attention(dev, steps, warmup, stream, pk):
    """Decode attention reading an e4m3 KV cache with per-tensor K / V scales:
    16 sequences x 4096 tokens, 32 query heads over 8 KV heads of 128
    (Llama-3-8B), one query token per sequence.  Two cache sets alternate
    (268 MB, larger than L2), so every call streams its cache from HBM."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    B, T, Hkv, Hq, D = ATTN_SHAPE

    def finite_codes(seed):
        c = si.random_codes((B, T, Hkv, D), seed=seed, device=dev)
        return torch.where((c & 0x7F) == 0x7F, c - 1, c)     # NaN codes -> +-448

    sets = []
    for j in range(2):
        kc = finite_codes(5000 + 2 * j)
        vc = finite_codes(5001 + 2 * j)
        q = si.normal((B, Hq, D), seed=5100 + j, device=dev)
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        sets.append((q, kc, vc, out))
    lens = torch.full((B,), T, dtype=torch.int32, device=dev)
    ks = torch.full((1,), 0.02, dtype=torch.float32, device=dev)
    vs = torch.full((1,), 0.01, dtype=torch.float32, device=dev)
    ws = w8.Workspace(w8.attention_workspace_size(B, Hq, T), dev)

    def step():
        for q, kc, vc, out in sets:
            w8.fp8_kv_decode_attention(q, kc, vc, lens, ks, vs, out, workspace=ws, stream=stream)

    t, n = time_graph(graph_of(step, stream), stream, steps, warmup)
    t /= len(sets)
    byts = attention_bytes()
    hbm = pk["hbm_gbs"]
    gbs = byts / t / 1e9
    del sets
    torch.cuda.empty_cache()
    return {"value": r4(gbs), "unit": "GB/s", "us": r4(t * 1e6), "samples": n,
            "roofline": {"bound": "hbm", "achieved": r4(gbs), "peak": r4(hbm), "frac": r4(gbs / hbm),
                         "kernel": "codes+q+out"}}


def attention_bytes():
    B, T, Hkv, Hq, D = ATTN_SHAPE
    return 2 * B * T * Hkv * D + 2 * 2 * B * Hq * D   # codes of K and V, q and out (bf16)


# ---------------------------------------------------------------- CPU baselines (oracle)
# The oracle as it stands, timed on the host cores on a bounded sample of
# each workload.  Inputs are made on the CPU by synthetic_inputs (same laws
# and shapes as the GPU workloads) and quantised by the oracle; the sample
# is what the timer covers.

_ORACLE_WEIGHTS = {}


def _oracle_weights(seed):
    """The four projections' weights quantised by the oracle, made once per
    process (setup, outside every timed sample)."""
    if seed not in _ORACLE_WEIGHTS:
        import oracle
        import synthetic_inputs as si
        wq = {}
        for i, (name, N, K, shared) in enumerate(LLAMA8B):
            wt = si.bits16(si.normal((N, K), seed=seed + i, std=0.02))
            wq[name] = oracle.quant(wt, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR if shared else oracle.PER_ROW)
        _ORACLE_WEIGHTS[seed] = wq
    return _ORACLE_WEIGHTS[seed]


def oracle_decode_sample(budget_s: float, seed=5000):
    """Time the oracle on a bounded sample of the decode step: full rows of
    the four projections (activation quantisation + scaled matmul), rows
    added until the time budget is used.  Returns (flops, seconds, rows, cores)."""
    import oracle
    import synthetic_inputs as si
    wq = _oracle_weights(seed)
    flops = 0.0
    rows = 0
    t0 = time.perf_counter()
    elapsed = 0.0
    r = 0
    while elapsed < budget_s:
        for j, (name, N, K, _) in enumerate(LLAMA8B):
            x = si.bits16(si.normal_with_outliers((1, K), seed=seed + 100 + r * 7 + j))
            aq, sa = oracle.quant(x, oracle.BF16, oracle.E4M3, oracle.PER_ROW)
            q, s = wq[name]
            oracle.scaled_mm(aq, q, sa, s, oracle.E4M3, oracle.BF16)
            flops += 2.0 * N * K
        rows += 1
        r += 1
        elapsed = time.perf_counter() - t0
    return flops, elapsed, rows, oracle.num_threads()


def _sample_pairs(M, N, rows=64, cols=64, tile_m=128, tile_n=128, seed=0):
    """(m, n) pairs of the large-M oracle sample: `rows` full rows, `cols`
    full columns and every (tile_m x tile_n) tile's four corners."""
    import numpy as np
    rng = np.random.default_rng(seed)
    rm = rng.choice(M, size=min(rows, M), replace=False)
    cn = rng.choice(N, size=min(cols, N), replace=False)
    mm = [np.repeat(rm, N), np.tile(np.arange(M), len(cn))]
    nn = [np.tile(np.arange(N), len(rm)), np.repeat(cn, M)]
    tm = np.arange(0, M, tile_m)
    tn = np.arange(0, N, tile_n)
    for dm in (0, tile_m - 1):
        for dn in (0, tile_n - 1):
            gm, gn = np.meshgrid(np.minimum(tm + dm, M - 1), np.minimum(tn + dn, N - 1), indexing="ij")
            mm.append(gm.ravel())
            nn.append(gn.ravel())
    return np.concatenate(mm).astype(np.int64), np.concatenate(nn).astype(np.int64)


def cpu_prefill_sample():
    """Config 3 sample: the QKV projection at M = 4096 (static per-tensor
    scales): quantise the activations with the calibration scale, then the
    scaled matmul on 64 rows, 64 columns and the tile corners."""
    import oracle
    import synthetic_inputs as si
    M, (name, N, K, _) = 4096, LLAMA8B[0]
    wq, sw = oracle.quant(si.bits16(si.normal((N, K), seed=2000, std=0.02)), oracle.BF16, oracle.E4M3,
                          oracle.PER_TENSOR)
    _, sa = oracle.quant(si.bits16(si.student_t_columns((M, K), seed=2100)), oracle.BF16, oracle.E4M3,
                         oracle.PER_TENSOR)
    x = si.bits16(si.student_t_columns((M, K), seed=2200))
    im, inn = _sample_pairs(M, N, seed=3)
    t0 = time.perf_counter()
    aq, _ = oracle.quant(x, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR, scale=sa)
    oracle.scaled_mm_sample(aq, wq, sa, sw, oracle.E4M3, oracle.BF16, im, inn)
    t = time.perf_counter() - t0
    return {"value": r4(2.0 * im.size * K / t / 1e12), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"QKV: quant, 64 rows+64 cols+corners, {t:.1f} s"}


def cpu_int8_sample():
    """Config 4 sample: the QKV-70B projection at M = 8192: per-token int8
    activation quantisation of every row, then the exact scaled matmul on
    64 rows, 64 columns and the tile corners."""
    import oracle
    import synthetic_inputs as si
    M, (name, N, K) = 8192, LLAMA70B[0]
    wq, sw = oracle.quant(si.bits16(si.normal((N, K), seed=3000, std=0.02)), oracle.BF16, oracle.INT8,
                          oracle.PER_ROW)
    x = si.bits16(si.normal_with_outliers((M, K), seed=3100))
    im, inn = _sample_pairs(M, N, seed=4)
    t0 = time.perf_counter()
    aq, sa = oracle.quant(x, oracle.BF16, oracle.INT8, oracle.PER_ROW)
    oracle.scaled_mm_sample(aq, wq, sa, sw, oracle.INT8, oracle.FP16, im, inn)
    t = time.perf_counter() - t0
    return {"value": r4(2.0 * im.size * K / t / 1e12), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "sample": f"QKV: quant, 64 rows+64 cols+corners, {t:.1f} s"}


def cpu_kv_full():
    """Config 5 in full: per-tensor dynamic quantisation of K and V
    [65536, 8, 128] and their dequantisation, by the oracle."""
    import oracle
    import synthetic_inputs as si
    T, H, D = 65536, 8, 128
    xs = [si.bits16(si.kv_with_spikes(T, H, D, seed=4000 + j).reshape(T * H, D)) for j in range(2)]
    t0 = time.perf_counter()
    for x in xs:
        q, s = oracle.quant(x, oracle.BF16, oracle.E4M3, oracle.PER_TENSOR)
        oracle.dequant(q, oracle.E4M3, s, oracle.PER_TENSOR, oracle.BF16)
    t = time.perf_counter() - t0
    n = T * H * D
    return {"value": r4(2 * n * 8 / t / 1e9), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"full K,V quant+dequant, {t:.1f} s"}


def cpu_quant_prefill_sample(rows=1024):
    """Prefill quantiser sample: the first `rows` rows of each of the four
    sizes, dynamic per token."""
    import oracle
    import synthetic_inputs as si
    xs = [si.bits16(si.normal_with_outliers((rows, C), seed=6000 + j)) for j, (_, C) in enumerate(QUANT_PREFILL)]
    t0 = time.perf_counter()
    for x in xs:
        oracle.quant(x, oracle.BF16, oracle.E4M3, oracle.PER_ROW)
    t = time.perf_counter() - t0
    byts = sum(rows * C * 3 + 4 * rows for _, C in QUANT_PREFILL)
    return {"value": r4(byts / t / 1e9), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} rows/size, {t:.2f} s"}


def cpu_attention_sample():
    """Attention sample: one sequence of 4096 tokens, all 32 query heads."""
    import numpy as np
    import oracle
    import synthetic_inputs as si
    from oracle import attention as oa
    B, T, Hkv, Hq, D = ATTN_SHAPE
    b = 4
    kc = si.random_codes((b, T, Hkv, D), seed=5000).numpy()
    vc = si.random_codes((b, T, Hkv, D), seed=5001).numpy()
    kc = np.where((kc & 0x7F) == 0x7F, kc - 1, kc).astype(np.uint8)
    vc = np.where((vc & 0x7F) == 0x7F, vc - 1, vc).astype(np.uint8)
    q = si.bits16(si.normal((b, Hq, D), seed=5100))
    t0 = time.perf_counter()
    oa.fp8_kv_decode_attention(q, oracle.BF16, kc, vc, np.full(b, T, np.int32), 0.02, 0.01, 1.0 / np.sqrt(D))
    t = time.perf_counter() - t0
    byts = b * (2 * T * Hkv * D + 2 * 2 * Hq * D)
    return {"value": r4(byts / t / 1e9), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{b}/{B} seqs, numpy, {t:.2f} s"}


# ---------------------------------------------------------------- ncu cases

PROFILE_CASES = {
    # name: (description, builder) -- small enough for an ncu capture, inputs
    # larger than L2 where DRAM figures matter
    "decode_gemm": "fp8 decode GEMM, M=16 x gate-up [28672 x 4096] (117 MB of weights)",
    "m256_gemm": "fp8 decode GEMM, M=256 x down [4096 x 14336] (59 MB of weights)",
    "prefill_gemm": "fp8 prefill GEMM, M=4096 x gate-up [28672 x 4096]",
    "prefill_down": "fp8 prefill GEMM, M=4096 x down [4096 x 14336] (CTA pairs, last round in K halves)",
    "int8_gemm": "int8 GEMM, M=8192 x QKV-70B [10240 x 8192]",
    "quant_tokens": "per-token dynamic e4m3 quantiser, [4096 x 14336] bf16",
    "quant_kv": "per-tensor dynamic e4m3 quantiser (absmax + convert), KV [524288 x 128] bf16",
    "dequant_kv": "e4m3 -> bf16 dequantiser, KV [524288 x 128]",
    "decode_step": "the decode step (16 quantisers + 16 GEMMs), eager launches",
    "quant_decode": "per-token dynamic e4m3 quantiser of one decode token, [1 x 4096] bf16",
    "attention": "decode attention over an e4m3 KV cache, 16 seqs x 4096 tokens, 32 q / 8 kv heads x 128",
}


def run_profile_case(name: str, launches: int):
    """Run `launches` calls of one kernel family on a fixed small case (for
    ncu: capture with -k/-s/-c).  Prints the kernel configuration."""
    import torch
    import int8_w8a8_scaled_gb300 as w8
    import synthetic_inputs as si
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    def quantised(shape, seed, qdtype, per_row, weight):
        x = (si.normal(shape, seed=seed, std=0.02, device=dev) if weight
             else si.normal_with_outliers(shape, seed=seed, device=dev))
        q = torch.empty(*shape, dtype=qdtype, device=dev)
        s = torch.empty(shape[0] if per_row else 1, dtype=torch.float32, device=dev)
        w8.scaled_quant(x, q, s, per_token=per_row, dynamic=True)
        return q, s

    if name == "decode_step":
        wl = DecodeWorkload(dev)
        for _ in range(launches):
            wl.run_step()
        torch.cuda.synchronize()
        print(json.dumps({"case": name, "configs": {f"M{it['M']}_{it['name']}": w8.pick_config(
            it["M"], wl.weights[it["name"]][2], wl.weights[it["name"]][3], w8.E4M3) for it in wl.items}}))
        return
    if name.endswith("_gemm") or name == "prefill_down":
        M, N, K, qd = {"decode_gemm": (16, 28672, 4096, w8.E4M3), "prefill_gemm": (4096, 28672, 4096, w8.E4M3),
                       "prefill_down": (4096, 4096, 14336, w8.E4M3), "int8_gemm": (8192, 10240, 8192, w8.INT8),
                       "m256_gemm": (256, 4096, 14336, w8.E4M3)}[name]
        qt = torch.float8_e4m3fn if qd == w8.E4M3 else torch.int8
        a, sa = quantised((M, K), 1, qt, True, False)
        b, sb = quantised((N, K), 2, qt, True, True)
        out = torch.empty(M, N, dtype=torch.bfloat16 if qd == w8.E4M3 else torch.float16, device=dev)
        cfg = None
        ws = w8.Workspace(w8.mm_workspace_size(M, N, K, qd, cfg), dev)
        print(json.dumps({"case": name, "config": cfg or w8.pick_config(M, N, K, qd)}), flush=True)
        for _ in range(launches):
            w8.scaled_mm(a, b, sa, sb, out, workspace=ws, config=cfg)
    elif name == "quant_decode":
        x = si.normal_with_outliers((1, 4096), seed=3, device=dev)
        q = torch.empty(1, 4096, dtype=torch.float8_e4m3fn, device=dev)
        s = torch.empty(1, dtype=torch.float32, device=dev)
        for _ in range(launches):
            w8.scaled_quant(x, q, s, per_token=True, dynamic=True)
    elif name == "quant_tokens":
        x = si.normal_with_outliers((4096, 14336), seed=3, device=dev)
        q = torch.empty(4096, 14336, dtype=torch.float8_e4m3fn, device=dev)
        s = torch.empty(4096, dtype=torch.float32, device=dev)
        for _ in range(launches):
            w8.scaled_quant(x, q, s, per_token=True, dynamic=True)
    elif name == "attention":
        B, T, Hkv, Hq, D = 16, 4096, 8, 32, 128
        kc = si.random_codes((B, T, Hkv, D), seed=5000, device=dev)
        vc = si.random_codes((B, T, Hkv, D), seed=5001, device=dev)
        q = si.normal((B, Hq, D), seed=5100, device=dev)
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        lens = torch.full((B,), T, dtype=torch.int32, device=dev)
        ks = torch.full((1,), 0.02, dtype=torch.float32, device=dev)
        for _ in range(launches):
            w8.fp8_kv_decode_attention(q, kc, vc, lens, ks, ks, out)
    elif name in ("quant_kv", "dequant_kv"):
        x = si.kv_with_spikes(65536, 8, 128, seed=4, device=dev).reshape(-1, 128)
        q = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=dev)
        s = torch.empty(1, dtype=torch.float32, device=dev)
        w8.scaled_quant(x, q, s, per_token=False, dynamic=True)
        y = torch.empty_like(x)
        for _ in range(launches):
            if name == "quant_kv":
                w8.scaled_quant(x, q, s, per_token=False, dynamic=True)
            else:
                w8.scaled_dequant(q, s, y)
    else:
        raise SystemExit(f"unknown profile case {name}; known: {sorted(PROFILE_CASES)}")
    torch.cuda.synchronize()
    if w8.device_status() != 0:
        raise SystemExit("a kernel reported a pipeline timeout")


def run_int8_routes():
    """Compile and run probes/int8_routes.cu: mma.sync s8 and f16 throughput
    with register operands (the int8 matmul's route choice; the tcgen05
    kind::f16 route is the library's own int8 matmul, measured by the int8
    configuration of this benchmark)."""
    from int8_w8a8_scaled_gb300 import _build
    src = os.path.join(ROOT, "int8_w8a8_scaled_gb300", "probes", "int8_routes.cu")
    os.makedirs(_build.BUILD, exist_ok=True)
    exe = os.path.join(_build.BUILD, "int8_routes")
    subprocess.run([_build.nvcc(), *_build.ARCH, "-O3", src, "-o", exe], check=True)
    return subprocess.run([exe]).returncode


# ---------------------------------------------------------------- main paths

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    per_step_budget = max(0.02, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_decode_sample(per_step_budget)
    tot_f, tot_t, tot_rows = 0.0, 0.0, 0
    cores = oracle.num_threads()
    for _ in range(args.steps):
        f, t, rows, cores = oracle_decode_sample(per_step_budget)
        tot_f += f
        tot_t += t
        tot_rows += rows
    val = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "parallelism": "replicas"},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{tot_rows} activation rows (M=1) through all four projections: "
                                   "oracle quantisation + exact scaled matmul"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(wl, stream, dev, steps, warmup, barrier):
    """The decode step end to end through the public API with host buffers:
    every step uploads its activations from pinned host memory and reads its
    outputs back, pipelined over two device buffer sets (step k+1's upload
    and step k-1's download run on copy streams while step k computes; the
    computes stay in order on one stream, so they share the workspace)."""
    import torch
    sets = [wl.items, wl.second_set()]
    graphs = [graph_of(lambda: wl.run_step(sets[0]), stream), graph_of(lambda: wl.run_step(sets[1]), stream)]
    host_x = [it["x"].cpu().pin_memory() for it in wl.items]
    host_o = [[torch.empty(it["out"].shape, dtype=it["out"].dtype).pin_memory() for it in wl.items]
              for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_x)
    d2h = sum(h.numel() * h.element_size() for h in host_o[0])
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    k = [0]

    def e2e_step():
        b = k[0] % 2
        k[0] += 1
        up.wait_event(ev_comp[b])          # set b's activations are free again
        with torch.cuda.stream(up):
            for it, hx in zip(sets[b], host_x):
                it["x"].copy_(hx, non_blocking=True)
            ev_up[b].record(up)
        stream.wait_event(ev_up[b])
        stream.wait_event(ev_down[b])      # set b's outputs have been read back
        with torch.cuda.stream(stream):
            graphs[b].replay()
            ev_comp[b].record(stream)
        down.wait_event(ev_comp[b])
        with torch.cuda.stream(down):
            for it, ho in zip(sets[b], host_o[b]):
                ho.copy_(it["out"], non_blocking=True)
            ev_down[b].record(down)

    def sample():
        torch.cuda.synchronize()
        if barrier:
            barrier()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(up)                    # the first upload is inside the timed region
        for _ in range(steps):
            e2e_step()
        for b in range(2):
            stream.wait_event(ev_down[b])  # ... and so is the last download
        e_ev.record(stream)
        torch.cuda.synchronize()
        if barrier:
            barrier()
        return s_ev.elapsed_time(e_ev) / 1e3

    import math
    for _ in range(warmup):
        e2e_step()
    probe = sample()
    n = int(max_over_ranks(float(max(1, math.ceil(MIN_TIMED_S / max(probe, 1e-9)))), dev))
    t = statistics.median([sample() for _ in range(n)])
    return t, n, h2d, d2h


def decode_gemms_by_m(wl, stream, steps, warmup, pk):
    """The decode step's four matmuls at each token count M, timed as a graph
    of their own: {M: [us, fraction of HBM, fraction of the roofline]}.  The
    roofline time of a GEMM is the larger of its algorithmic bytes at the
    measured HBM rate and its flops at the dense fp8 peak; at M = 256 the two
    are within 10 % of each other (2·M flops per weight byte against a ridge
    near 560), so HBM alone understates how close that regime is to its
    bound."""
    out = {}
    hbm, fp8 = pk["hbm_gbs"] * 1e9, 2.0 * pk["bf16_tflops"] * 1e12
    for M in DECODE_MS:
        its = [it for it in wl.items if it["M"] == M]
        g = graph_of(lambda its=its: wl.run_gemm(its), stream)
        t, _ = time_graph(g, stream, steps, warmup)
        roof = sum(max(wl.gemm_bytes([it]) / hbm, wl.flops([it]) / fp8) for it in its)
        out[str(M)] = [r4(t * 1e6), r4(wl.gemm_bytes(its) / t / hbm), r4(roof / t)]
        del g
    return out


def run_ours(args):
    import torch
    ws_n, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = None
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        barrier = lambda: dist.barrier(device_ids=[local])  # noqa: E731
    import int8_w8a8_scaled_gb300 as w8
    from int8_w8a8_scaled_gb300 import _build
    _build.build()
    pk, pk_kind = peaks()
    stream = torch.cuda.Stream(device=dev)

    wl = DecodeWorkload(dev)
    g_step = graph_of(wl.run_step, stream)
    g_gemm = graph_of(wl.run_gemm, stream)
    g_quant = graph_of(wl.run_quant, stream)

    sampler = ClockSampler(local)
    sampler.start()
    t_sample, n_samples = timed(g_step.replay, stream, args.steps, args.warmup, barrier=barrier, device=dev)
    clocks = sampler.stop()
    t = max_over_ranks(t_sample, dev)
    flops_step = wl.flops()
    value = aggregate_tflops(flops_step, args.steps, t, ws_n)
    ms_per_step = t / args.steps * 1e3

    # the step's two kernel classes, each over its own timed samples
    t_gemm, _ = time_graph(g_gemm, stream, args.steps, args.warmup)
    t_quant, _ = time_graph(g_quant, stream, args.steps, args.warmup)
    hbm = pk["hbm_gbs"]
    gemm_gbs = wl.gemm_bytes() / t_gemm / 1e9
    quant_gbs = wl.quant_bytes() / t_quant / 1e9

    t_e2e, n_e2e, h2d, d2h = run_e2e(wl, stream, dev, args.steps, args.warmup, barrier)
    t_e2e = max_over_ranks(t_e2e, dev)
    e2e_val = aggregate_tflops(flops_step, args.steps, t_e2e, ws_n)
    del g_step, g_gemm, g_quant

    cfgs = {}
    if not args.main_only:
        w = max(3, args.warmup)
        st = max(3, min(args.steps, 50))
        cfgs["c3_prefill_fp8"] = measure_prefill_fp8(dev, st, w, stream, pk)
        cfgs["c4_int8_70b"] = measure_int8_70b(dev, st, w, stream, pk)
        cfgs["c5_kv_fp8"] = measure_kv(dev, st, w, stream, pk)
        cfgs["attn_fp8kv"] = measure_kv_attention(dev, st, w, stream, pk)
        cfgs["quant_prefill"] = measure_quant_prefill(dev, st, w, stream, pk)
    cfgs["c2_detail"] = {"gemm_us": r4(t_gemm * 1e6), "quant_us": r4(t_quant * 1e6),
                         "quant_gbs": r4(quant_gbs), "quant_frac": r4(quant_gbs / hbm),
                         "by_m": decode_gemms_by_m(wl, stream, args.steps, args.warmup, pk)}

    cpu = None
    if rank == 0 and args.gpus == 1 and not args.no_cpu_baseline:
        f, tc, rows, cores = oracle_decode_sample(args.cpu_budget)
        cpu = {"value": r4(f / tc / 1e12), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{rows} rows (M=1) x 4 projections: quant + exact matmul, {tc:.1f} s"}
        if not args.main_only:
            for key, fn in (("c3_prefill_fp8", cpu_prefill_sample), ("c4_int8_70b", cpu_int8_sample),
                            ("c5_kv_fp8", cpu_kv_full), ("attn_fp8kv", cpu_attention_sample),
                            ("quant_prefill", cpu_quant_prefill_sample)):
                cfgs[key]["cpu_baseline"] = fn()

    if rank == 0:
        tr = traffic_ratio_for("decode_gemm")
        line = {
            "metric": METRIC, "value": r4(value), "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r4(ms_per_step), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD,
                       "timing": f"CUDA graph of one step; median of {n_samples} samples of {args.steps} steps "
                                 f"(>= {MIN_TIMED_S} s timed); inputs > L2 (218 MB weights/step)",
                       "parallelism": "replicas" if ws_n > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": "w8a8_gemm_kernel (16 decode GEMMs)",
                         "achieved": r4(gemm_gbs), "peak": r4(hbm), "unit": "GB/s", "frac": r4(gemm_gbs / hbm),
                         "peak_kind": pk_kind,
                         "traffic": None if tr is None else r4(tr * wl.gemm_bytes() / wl.gemms_per_step())},
            "cpu_baseline": cpu,
            "e2e": {"value": r4(e2e_val), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "samples": n_e2e},
            "gpu_launches": wl.launches_per_step() * args.steps,
            "clocks": clocks,
            "configs": cfgs,
        }
        print(json.dumps(line, separators=(",", ":")), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--main-only", action="store_true", help="skip the other configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle time for the decode cpu_baseline")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run a few launches of one kernel on a small case (for ncu) and exit")
    ap.add_argument("--launches", type=int, default=5)
    ap.add_argument("--int8-routes", action="store_true",
                    help="time the warp-level MMA instructions an int8 matmul could use (the route choice) and exit")
    args = ap.parse_args()
    if args.int8_routes:
        return run_int8_routes()
    if args.profile_case:
        run_profile_case(args.profile_case, args.launches)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
