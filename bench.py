"""Benchmark of the fused MoE layer on GB300.

One step = one pass of the whole hot path over one batch of synthetic tokens:
route -> align/permute -> [FP8 quantise] -> gather -> gate/up GEMM + SiLU*mul
-> down GEMM + router weight -> ordered top-k reduce, each a CUDA kernel of
libgbmoe.so launched through its C ABI.

Default workload: the Mixtral-8x7B-shaped prefill layer in bf16 (M=4096 tokens,
K=4096, N=14336, E=8, top-2), synthetic seeded inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on host cores

Multi-GPU: the layer is data parallel over tokens and needs no exchange, so
N ranks run N independent replicas (weak scaling); ranks only meet at the
timing barriers.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

WORKLOADS = dict(WL.BY_NAME)
DEFAULT = WL.MIXTRAL_PREFILL.name
METRIC = "MoE-layer tokens/s and % of roofline (TFLOP/s or HBM GB/s) on 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _kernel_traffic(cfg, which: str):
    """DRAM bytes per launch of the dominant kernel on this workload, from a
    committed ncu summary profiles/<workload>.<which>.traffic.txt (lines
    'traffic_bytes_per_launch: <n>', 'source_file: <kernel source>' and
    'source_sha256: <its sha256>').  None when there is none, or when the
    kernel source has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{cfg.name}.{which}.traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for ln in f:
            if ":" in ln and not ln.startswith("#"):
                k, v = ln.split(":", 1)
                vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, vals.get("source_file", ""))
    if not os.path.isfile(src):
        return None
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    if vals.get("source_sha256") != h:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in samples taken
        between wall times t0 and t1 (all samples when not given)."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if t0 is not None and not (t0 - 0.1 <= ts <= t1 + 0.1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- GPU arm --

class Layer:
    """Device buffers of one Standard-format layer plus the staged launch
    sequence (the same kernels moe_forward launches, called one by one so
    the dominant GEMM can be timed with events on the launching stream)."""

    def __init__(self, cfg, device):
        import torch
        import mixture_experts_layer_count_gb300 as g
        self.g, self.torch, self.cfg = g, torch, cfg
        g.load()
        d = WL.make_inputs(cfg, device)
        self.x, self.logits, self.bias = d["x"], d["logits"], d["bias"]
        M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
        P = M * k
        self.fp8 = cfg.dtype != WL.BF16
        # one scale per weight row; per token (FP8_CHANNEL) or per tensor
        # (FP8_TENSOR) for the activations
        self.ch = cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR)
        self.tensor = cfg.dtype == WL.FP8_TENSOR
        if self.ch:
            self.w1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=device)
            self.w2 = torch.empty((E, K, N), dtype=torch.uint8, device=device)
            self.w1s = torch.empty((E, 2 * N), dtype=torch.float32, device=device)
            self.w2s = torch.empty((E, K), dtype=torch.float32, device=device)
            g.moe_quant_fp8_group(d["w1"].view(E * 2 * N, K), self.w1.view(E * 2 * N, K),
                                  self.w1s.view(E * 2 * N, 1), group=K)
            g.moe_quant_fp8_group(d["w2"].view(E * K, N), self.w2.view(E * K, N),
                                  self.w2s.view(E * K, 1), group=N)
            del d
            torch.cuda.empty_cache()
        elif self.fp8:
            self.w1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=device)
            self.w2 = torch.empty((E, K, N), dtype=torch.uint8, device=device)
            self.w1s = torch.empty((E, 2 * N // 128, K // 128), dtype=torch.float32, device=device)
            self.w2s = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device=device)
            g.moe_quant_fp8_block(d["w1"], self.w1, self.w1s)
            g.moe_quant_fp8_block(d["w2"], self.w2, self.w2s)
            del d
            torch.cuda.empty_cache()
        else:
            self.w1, self.w2, self.w1s, self.w2s = d["w1"], d["w2"], None, None
        i32, f32 = torch.int32, torch.float32
        self.ids = torch.empty((M, k), dtype=i32, device=device)
        self.wts = torch.empty((M, k), dtype=f32, device=device)
        self.counts = torch.empty(E, dtype=i32, device=device)
        self.offsets = torch.empty(E + 1, dtype=i32, device=device)
        self.sorted = torch.empty(P, dtype=i32, device=device)
        self.inv = torch.empty(P, dtype=i32, device=device)
        self.align_ws = g.workspace(g.WS_ALIGN, M, E, 0, 0, k, 0, device=device)
        adt = torch.uint8 if self.fp8 else torch.bfloat16
        sk = 1 if self.ch else K // 128   # scales per row of x / A
        self.A = torch.empty((P, K), dtype=adt, device=device)
        ld = (P + 3) // 4 * 4  # group-major FP8 row scales
        self.As = torch.empty((sk, ld), dtype=f32, device=device) if self.fp8 else None
        if self.ch:  # H in bf16 from gate/up, then its per-token e4m3 codes
            self.Hb = torch.empty((P, N), dtype=torch.bfloat16, device=device)
            self.H = torch.empty((P, N), dtype=torch.uint8, device=device)
            self.Hs = torch.empty((P, 1), dtype=f32, device=device)
        else:
            self.Hb = None
            self.H = torch.empty((P, N), dtype=adt, device=device)
            self.Hs = torch.empty((N // 128, ld), dtype=f32, device=device) if self.fp8 else None
        self.y = torch.empty((M, k, K), dtype=torch.bfloat16, device=device)
        self.out = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.err = torch.zeros(1, dtype=i32, device=device)
        self.amax = torch.zeros(2, dtype=i32, device=device) if self.tensor else None
        self.fwd_ws = g.workspace(g.WS_FORWARD, M, E, N, K, k, cfg.dtype, device=device)
        # route, 3 align, gather, gate/up, [quant H], down, reduce; e4m3
        # quantises x and gathers in one launch (per tensor: after a clear
        # and a maximum, as its H quant is a clear, a maximum and the codes)
        self.launches_per_step = 8 + (1 if self.ch else 0) + (4 if self.tensor else 0)

    def step(self, ev_gemm=None, mark=None):
        """One layer pass as its separate calls.  ev_gemm: a pair of events
        recorded around the gate/up GEMM; mark(name): called after each
        stage (the per-stage breakdown records an event there)."""
        g, c = self.g, self.cfg
        M, E, N, K, k = c.M, c.E, c.N, c.K, c.topk
        mark = mark or (lambda name: None)
        g.moe_topk_route(self.logits, self.bias, k, c.score_fn, c.n_groups, c.topk_groups,
                         c.renorm, self.ids, self.wts)
        mark("a1_route")
        g.moe_align_permute(self.ids, E, self.counts, self.offsets, self.sorted, self.inv,
                            self.align_ws, self.err)
        mark("a2_a3_count_align")
        if self.fp8 and not self.ch and not self.tensor:
            # 1 x 128 groups: quantised once, codes and scales written to the
            # permuted rows in the same pass
            g.moe_quant_fp8_group_permute(self.x, self.inv, k, self.A, self.As)
            mark("a4_a3_quant_permute")
        elif self.ch and not self.tensor:
            # one scale per token: likewise
            g.moe_quant_fp8_row_permute(self.x, self.inv, k, self.A, self.As.view(-1))
            mark("a4_a3_quant_permute")
        elif self.tensor:
            # one scale for the tensor: its maximum first, then the codes
            # written to the permuted rows
            g.moe_quant_fp8_tensor_permute(self.x, self.inv, k, self.A, self.As.view(-1),
                                           amax_ws=self.amax[0:1])
            mark("a4_a3_quant_permute")
        else:
            g.moe_permute_rows(self.x, None, self.sorted, self.offsets, k, E, c.dtype, self.A,
                               self.As)
            mark("a3_gather")
        if ev_gemm is not None:
            ev_gemm[0].record()
        g.moe_grouped_gemm_gate_up_silu(self.A, self.As, self.offsets, M, k, E, N, K, self.w1,
                                        self.w1s, c.dtype, self.Hb if self.ch else self.H,
                                        self.Hs, self.err)
        if ev_gemm is not None:
            ev_gemm[1].record()
        mark("a5_gate_up")
        if self.tensor:  # rows of pairs computed here: offsets[E]
            g.moe_quant_fp8_tensor(self.Hb, self.H, self.Hs, self.amax[1:2],
                                   n_rows=self.offsets[E:])
            mark("a4_quant_h")
        elif self.ch:
            g.moe_quant_fp8_group(self.Hb, self.H, self.Hs, group=N)
            mark("a4_quant_h")
        g.moe_grouped_gemm_down(self.H, self.Hs, self.sorted, self.offsets, self.wts, M, k, E,
                                N, K, self.w2, self.w2s, c.dtype, self.y, self.err)
        mark("a6_down")
        g.moe_unpermute_weighted_reduce(self.y, self.inv, M, k, K, self.out)
        mark("a7_reduce")

    def forward_public(self, x, logits, out):
        """The public one-call API on device tensors."""
        c = self.cfg
        self.g.moe_forward(x, logits, self.bias, c.N, c.E, c.topk, c.score_fn, c.n_groups,
                           c.topk_groups, c.renorm, c.dtype, self.w1, self.w1s, self.w2,
                           self.w2s, out, self.fwd_ws, err_word=self.err)


def stage_breakdown(layer, steps):
    """Mean device milliseconds of each stage of the separate-call layer over
    `steps` passes (events between consecutive calls on the launching
    stream; a pass apart from the timed region)."""
    import torch
    acc = {}
    for _ in range(steps):
        evs = []
        start = torch.cuda.Event(enable_timing=True)
        start.record()

        def mark(name, evs=evs):
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            evs.append((name, e))
        layer.step(mark=mark)
        torch.cuda.synchronize()
        prev = start
        for name, e in evs:
            acc[name] = acc.get(name, 0.0) + prev.elapsed_time(e)
            prev = e
    return {k: v / steps for k, v in acc.items()}


def graph_time(layer, steps):
    """Milliseconds per step of the one-call layer (moe_forward) captured
    once in a CUDA graph and replayed `steps` times, and of the same call
    launched eagerly."""
    import torch
    out = torch.empty_like(layer.out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            layer.forward_public(layer.x, layer.logits, out)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward_public(layer.x, layer.logits, out)
    for _ in range(3):
        graph.replay()
    t = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    torch.cuda.synchronize()
    t[0].record()
    for _ in range(steps):
        graph.replay()
    t[1].record()
    for _ in range(steps):
        layer.forward_public(layer.x, layer.logits, out)
    t[2].record()
    torch.cuda.synchronize()
    assert layer.err.item() == 0
    return t[0].elapsed_time(t[1]) / steps, t[1].elapsed_time(t[2]) / steps


def reduce_max(values, dist=None, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity with one
    process).  The only cross-rank operation of the benchmark."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(tokens_per_step, steps, world, max_ms):
    """Whole-job tokens/s of `world` independent replicas: every rank's
    tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / (max_ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def pipelined_e2e(steps, h2d, compute, d2h):
    """End-to-end steps as a serving loop runs them: step i's host-to-device
    copy (h2d(b)), the layer (compute(b)) and the device-to-host copy of its
    result (d2h(b)) go to three streams, on buffer set b = i % 2, so the
    copies of one step overlap the layer of its neighbour.  Events order a
    buffer's reuse: the copy into set b waits until the layer of step i - 2
    has read it, the layer waits for its inputs and for the copy-out of step
    i - 2.  Returns the milliseconds from the first copy-in to the last
    copy-out (events on both streams)."""
    import torch
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    for st in (s_in, s_run, s_out):
        st.wait_stream(torch.cuda.current_stream())
    t0.record(s_in)
    for i in range(steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["done"][b])
            h2d(b)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev["in"][b])
            if i >= 2:
                s_run.wait_event(ev["out"][b])
            compute(b)
            ev["done"][b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            d2h(b)
            ev["out"][b].record(s_out)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_run)
    t1.record(s_out)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def run_gpu(args, cfg):
    import torch
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    layer = Layer(cfg, dev)
    # warm-up (untimed)
    for _ in range(args.warmup):
        layer.step()
    torch.cuda.synchronize()
    assert layer.err.item() == 0, f"device error word {layer.err.item()}"

    steps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        wall0 = time.time()
        t0.record()
        for i in range(steps):
            layer.step(ev[i])
        t1.record()
        barrier()
        wall1 = time.time()
    ms = t0.elapsed_time(t1)
    gemm_ms = [a.elapsed_time(b) for a, b in ev]
    assert layer.err.item() == 0, f"device error word {layer.err.item()}"

    # end to end through the public one-call API: every step copies its inputs
    # in from pinned host memory and its output back, inside the timed region
    x_h = layer.x.cpu().pin_memory()
    lg_h = layer.logits.cpu().pin_memory()
    out_h = [torch.empty(layer.out.shape, dtype=layer.out.dtype).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(layer.x) for _ in range(2)]
    lg_d = [torch.empty_like(layer.logits) for _ in range(2)]
    out_d = [torch.empty_like(layer.out) for _ in range(2)]

    def h2d(b):
        x_d[b].copy_(x_h, non_blocking=True)
        lg_d[b].copy_(lg_h, non_blocking=True)

    def d2h(b):
        out_h[b].copy_(out_d[b], non_blocking=True)

    pipelined_e2e(max(2, args.warmup), h2d, lambda b: layer.forward_public(x_d[b], lg_d[b], out_d[b]),
                  d2h)
    barrier()
    e2e_ms = pipelined_e2e(steps, h2d,
                           lambda b: layer.forward_public(x_d[b], lg_d[b], out_d[b]), d2h)
    barrier()
    assert layer.err.item() == 0

    # per-stage breakdown and one-call graph / eager timing (outside the
    # timed region, on this rank)
    kernels_ms = stage_breakdown(layer, min(steps, 20))
    graph_ms, eager_call_ms = graph_time(layer, min(steps, 100))

    # max over ranks
    ms, e2e_ms, gemm_avg = reduce_max([ms, e2e_ms, float(np.mean(gemm_ms))], pg, device=dev)
    value = replica_throughput(cfg.M, steps, world, ms)
    e2e_value = replica_throughput(cfg.M, steps, world, e2e_ms)
    line = _line(args, cfg, layer, world, steps, ms, gemm_avg, e2e_ms,
                 clk.summary(wall0, wall1))
    line["value"] = value
    line["e2e"]["value"] = e2e_value
    line["kernels_ms"] = kernels_ms
    line["graph_ms_per_step"] = graph_ms
    line["one_call_eager_ms_per_step"] = eager_call_ms
    if rank != 0:
        return
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, layer, args.cpu_seconds)
    if world == 1 and not args.no_extras:
        del layer
        torch.cuda.empty_cache()
        line["per_workload"] = run_extras(args, dev, skip=cfg.name)
        if not args.no_features:
            line["features"] = run_features(args, dev)
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


EXTRA_WORKLOADS = [WL.TINY, WL.DSV3_DECODE, WL.DSV3_PREFILL_FP8, WL.BATCHED_MASKED,
                   WL.BATCHED_MASKED_FP8]


def run_extras(args, dev, skip=None):
    """The other workloads of the layer, each timed as the default one is
    (event-timed steps over resident inputs, clocks sampled inside the timed
    region) but without the end-to-end leg: tiny (launch-bound), DeepSeek-V3
    decode (weight-streaming, HBM-bound), DeepSeek-V3 prefill with e4m3 block
    scales, and the batched masked format replayed from a CUDA graph.  Only
    the tiny and decode entries carry a CPU leg: the oracle on all their
    tokens (seconds), the tiny one also on one thread."""
    import torch
    steps = max(20, min(args.steps, 200))
    warmup = max(3, min(args.warmup, 10))
    # the whole-workload oracle timings ride along where they take seconds
    cpu_full = not args.no_cpu_baseline and _dist()[0] == 1
    out = {}
    for cfg in EXTRA_WORKLOADS:
        if cfg.name == skip:
            continue
        t = time.time()
        if cfg.batched:
            entry = measure_batched_entry(cfg, dev, steps, warmup, cpu_full)
        else:
            entry = measure_standard_entry(cfg, dev, steps, warmup, cpu_full)
        entry["wall_s"] = time.time() - t
        out[cfg.name] = entry
        torch.cuda.empty_cache()
    return out


def _timed(fn, steps, warmup, dev):
    """Milliseconds per call of fn (whatever it enqueues, on any streams that
    join the current one), CUDA events over `steps` calls after `warmup`,
    with the clocks sampled in between."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        wall0 = time.time()
        t0.record()
        for _ in range(steps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        wall1 = time.time()
    return t0.elapsed_time(t1) / steps, clk.summary(wall0, wall1)


def _tc_roof(flop, ms, fp8, timed_s, what):
    peaks, src = _peaks()
    key = "bf16_tflops" if timed_s < 2.0 else "bf16_tflops_sustained"
    peak = peaks.get(key, FALLBACK_PEAKS[key]) * (2.0 if fp8 else 1.0)
    achieved = flop / (ms / 1e3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": None, "kernel": what,
            "peak_source": f"{src} {key}" + (" x2 (nominal fp8:bf16 dense ratio)" if fp8 else "")
                           + f" (timed region {timed_s:.2f} s)"}


# the wider features, each measured on a DeepSeek-V3-shaped workload
FEATURE_STANDARD = [(WL.DSV3_PREFILL_FP8CH, "e4m3, one scale per token and per weight row"),
                    (WL.DSV3_PREFILL_FP8T, "e4m3, one dynamic scale per activation tensor")]
SHARED_NS = 2048          # DeepSeek-V3's shared expert: intermediate size 2048
CHUNK = 2048              # tokens per chunk of the chunked layer


def run_features(args, dev):
    """The layer's wider features timed like the workloads above (event-timed calls over
    resident inputs, clocks sampled inside the timed region): the per-channel
    and per-tensor e4m3 layers; the block-scaled e4m3 layer with its shared
    expert overlapped on an auxiliary stream (and the same calls one after
    the other); that layer in chunks of 2048 tokens; and the worst-tokens EP
    layer of eight shards (route, e4m3 dispatch, eight masked expert GEMM
    pairs, combine) replayed from one CUDA graph."""
    import torch
    steps = max(20, min(args.steps, 100))
    warmup = max(3, min(args.warmup, 10))
    cpu_full = not args.no_cpu_baseline and _dist()[0] == 1
    out = {}
    for cfg, feature in FEATURE_STANDARD:
        t = time.time()
        e = measure_standard_entry(cfg, dev, steps, warmup, cpu_full)
        e["feature"] = feature
        e["wall_s"] = time.time() - t
        out[cfg.name] = e
        torch.cuda.empty_cache()
    t = time.time()
    sh, ch = measure_shared_and_chunked(WL.DSV3_PREFILL_FP8, dev, steps, warmup)
    sh["wall_s"] = ch["wall_s"] = time.time() - t
    out[WL.DSV3_PREFILL_FP8.name + "_shared_expert_overlapped"] = sh
    out[WL.DSV3_PREFILL_FP8.name + f"_chunked_{CHUNK}"] = ch
    torch.cuda.empty_cache()
    t = time.time()
    e = measure_ep_entry(WL.EP8_DSV3, dev, steps, warmup)
    e["wall_s"] = time.time() - t
    out[WL.EP8_DSV3.name + "_fp8"] = e
    torch.cuda.empty_cache()
    return out


def measure_shared_and_chunked(cfg, dev, steps, warmup):
    """The one-call e4m3 layer (moe_forward) with a shared expert of
    intermediate size SHARED_NS in block-scaled e4m3: routed alone, shared
    alone, both one after the other on one stream, and overlapped (the
    shared expert on an auxiliary stream, moe_forward_shared); then the
    routed layer in chunks of CHUNK tokens (moe_forward_chunked, a workspace
    sized for one chunk)."""
    import torch
    layer = Layer(cfg, dev)
    g = layer.g
    M, E, N, K, k = cfg.M, cfg.E, cfg.N, cfg.K, cfg.topk
    Ns = SHARED_NS
    gen = torch.Generator(device=dev).manual_seed(cfg.seed + 100)
    w1s = (torch.randn((2 * Ns, K), generator=gen, device=dev) / K ** 0.5).to(torch.bfloat16)
    w2s = (torch.randn((K, Ns), generator=gen, device=dev) / Ns ** 0.5).to(torch.bfloat16)
    q1 = torch.empty((2 * Ns, K), dtype=torch.uint8, device=dev)
    q2 = torch.empty((K, Ns), dtype=torch.uint8, device=dev)
    s1 = torch.empty((2 * Ns // 128, K // 128), dtype=torch.float32, device=dev)
    s2 = torch.empty((K // 128, Ns // 128), dtype=torch.float32, device=dev)
    g.moe_quant_fp8_block(w1s, q1, s1)
    g.moe_quant_fp8_block(w2s, q2, s2)
    del w1s, w2s
    out_sh = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    ws = layer.fwd_ws
    ws_sh = g.workspace(g.WS_SHARED, M, 1, Ns, K, 1, WL.FP8, device=dev)
    args = (layer.x, layer.logits, layer.bias, N, E, k, cfg.score_fn, cfg.n_groups,
            cfg.topk_groups, cfg.renorm, cfg.dtype, layer.w1, layer.w1s, layer.w2, layer.w2s)
    shk = dict(shared_dtype=WL.FP8, w1s_scales=s1, w2s_scales=s2, err_word=layer.err)
    aux = torch.cuda.Stream()
    ev_in, ev_out = torch.cuda.Event(), torch.cuda.Event()

    def routed():
        g.moe_forward(*args, layer.out, ws, err_word=layer.err)

    def shared():
        g.moe_shared_expert_forward(layer.x, Ns, q1, q2, out_sh, ws_sh, dtype=WL.FP8,
                                    w1s_scales=s1, w2s_scales=s2, err_word=layer.err)

    def serial():
        g.moe_forward_shared(*args, layer.out, ws, Ns, q1, q2, out_sh, ws_sh, **shk)

    def overlapped():
        g.moe_forward_shared(*args, layer.out, ws, Ns, q1, q2, out_sh, ws_sh, aux_stream=aux,
                             ev_input_ready=ev_in, ev_output_ready=ev_out, **shk)

    t_r, _ = _timed(routed, steps, warmup, dev)
    t_s, _ = _timed(shared, steps, warmup, dev)
    t_ser, _ = _timed(serial, steps, warmup, dev)
    t_ovl, clk = _timed(overlapped, steps, warmup, dev)
    routed_flop = 6.0 * K * N * cfg.P
    shared_flop = 6.0 * K * Ns * M
    sh = {"feature": "shared expert (block-scaled e4m3) overlapped on an auxiliary stream",
          "unit": "tokens/s", "value": M / (t_ovl / 1e3), "steps": steps,
          "ms_per_step": t_ovl, "serial_ms_per_step": t_ser, "routed_alone_ms": t_r,
          "shared_alone_ms": t_s, "overlap_saved_ms": t_ser - t_ovl,
          "layer_tflops": (routed_flop + shared_flop) / (t_ovl / 1e3) / 1e12,
          "roofline": _tc_roof(routed_flop + shared_flop, t_ovl, True, t_ovl * steps / 1e3,
                               "whole layer: routed experts + shared expert"),
          "clocks": clk, "config": {"M": M, "K": K, "N": N, "E": E, "topk": k,
                                    "shared_intermediate": Ns,
                                    "scales": _scales_desc(cfg)}}
    ws_c = g.workspace(g.WS_FORWARD, CHUNK, E, N, K, k, cfg.dtype, device=dev)

    def chunked():
        g.moe_forward_chunked(*args, layer.out, ws_c, CHUNK, err_word=layer.err)

    t_c, clk_c = _timed(chunked, steps, warmup, dev)
    torch.cuda.synchronize()
    assert layer.err.item() == 0, f"device error word {layer.err.item()}"
    ch = {"feature": "in-graph chunking (device-side counts per chunk)",
          "unit": "tokens/s", "value": M / (t_c / 1e3), "steps": steps,
          "ms_per_step": t_c, "unchunked_ms_per_step": t_r, "chunk_tokens": CHUNK,
          "workspace_bytes": ws_c.numel(), "unchunked_workspace_bytes": ws.numel(),
          "roofline": _tc_roof(routed_flop, t_c, True, t_c * steps / 1e3,
                               "whole layer, all chunks"),
          "clocks": clk_c, "config": {"M": M, "K": K, "N": N, "E": E, "topk": k,
                                      "scales": _scales_desc(cfg)}}
    del layer
    return sh, ch


def measure_ep_entry(cfg, dev, steps, warmup):
    """The worst-tokens EP layer of cfg.G shards in this GPU's memory, e4m3:
    route every shard's tokens, quantise them in 1 x 128 groups, dispatch
    the valid pairs into the experts' static receive blocks (device counts),
    run each shard's masked expert GEMMs on its block, combine -- captured
    once in a CUDA graph and replayed; the same sequence launched eagerly
    for comparison.  The roofline counts the valid pairs' expert work and
    the e4m3 weights of the experts that received rows."""
    import torch
    import mixture_experts_layer_count_gb300 as g
    g.load()
    G, M, K, N, E, k = cfg.G, cfg.M, cfg.K, cfg.N, cfg.E, cfg.topk
    W = cfg.worst_tokens
    El = E // G
    d = WL.make_ep_inputs(cfg, dev)
    q1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=dev)
    q2 = torch.empty((E, K, N), dtype=torch.uint8, device=dev)
    s1 = torch.empty((E, 2 * N // 128, K // 128), dtype=torch.float32, device=dev)
    s2 = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device=dev)
    g.moe_quant_fp8_block(d["w1"], q1, s1)
    g.moe_quant_fp8_block(d["w2"], q2, s2)
    del d["w1"], d["w2"]
    torch.cuda.empty_cache()
    i32, f32 = torch.int32, torch.float32
    x, logits, num_tokens = d["x"], d["logits"], d["num_tokens"]
    ids = torch.empty((G, M, k), dtype=i32, device=dev)
    wts = torch.empty((G, M, k), dtype=f32, device=dev)
    xq = torch.empty((G, M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty((G * M, K // 128), dtype=f32, device=dev)
    recv_x = torch.empty((E, W, K), dtype=torch.uint8, device=dev)
    recv_s = torch.empty((E * W, K // 128), dtype=f32, device=dev)
    recv_y = torch.empty((E, W, K), dtype=torch.bfloat16, device=dev)
    recv_counts = torch.empty(E, dtype=i32, device=dev)
    recv_pos = torch.empty((G, M, k), dtype=i32, device=dev)
    out = torch.empty((G, M, K), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=i32, device=dev)
    ws = g.workspace(g.WS_EP_DISPATCH, M, E, G, K, k, 0, device=dev)
    bws = [g.workspace(g.WS_BATCHED, W, El, N, K, 1, WL.FP8, device=dev) for _ in range(G)]

    def step():
        g.moe_topk_route(logits.view(G * M, E), None, k, cfg.score_fn, cfg.n_groups,
                         cfg.topk_groups, True, ids.view(G * M, k), wts.view(G * M, k))
        g.moe_quant_fp8_group(x.view(G * M, K), xq.view(G * M, K), xs)
        g.moe_ep_dispatch(xq, num_tokens, ids, E, W, recv_x, recv_counts, recv_pos, ws, err,
                          dtype=WL.FP8, x_scales=xs, recv_scales=recv_s)
        for r in range(G):
            sl = slice(r * El, (r + 1) * El)
            g.moe_batched_masked_experts(recv_x[sl], recv_counts[sl], N, q1[sl], q2[sl],
                                         recv_y[sl], bws[r], dtype=WL.FP8,
                                         x_b_scales=recv_s[r * El * W:(r + 1) * El * W],
                                         w1_scales=s1[sl], w2_scales=s2[sl], err_word=err)
        g.moe_ep_combine(recv_y, ids, recv_pos, wts, num_tokens, out)

    t_eager, _ = _timed(step, min(steps, 20), warmup, dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    t_graph, clk = _timed(graph.replay, steps, warmup, dev)
    torch.cuda.synchronize()
    assert err.item() == 0, f"device error word {err.item()}"
    counts = recv_counts.cpu().numpy()
    tokens = int(num_tokens.sum().item())
    pairs = int(counts.sum())
    flop = 6.0 * K * N * pairs
    touched = int((counts > 0).sum())
    wbytes = touched * (3 * N * K + (2 * N // 128 * (K // 128) + (K // 128) * (N // 128)) * 4)
    gbs = wbytes / (t_graph / 1e3) / 1e9
    peaks, src = _peaks()
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tc = _tc_roof(flop, t_graph, True, t_graph * steps / 1e3,
                  "EP layer: route, dispatch, 8 shards' masked e4m3 GEMMs, combine")
    roof = tc if tc["achieved"] / tc["peak"] >= gbs / hbm_peak else {
        "bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
        "frac": gbs / hbm_peak, "traffic": None, "kernel": tc["kernel"],
        "peak_source": f"{src} hbm_gbs (copy)"}
    roof["tensor_frac"] = tc["frac"]
    roof["hbm_frac"] = gbs / hbm_peak
    del graph
    return {"feature": "worst-tokens EP dispatch/combine, single-GPU form (8 shards)",
            "unit": "tokens/s", "value": tokens / (t_graph / 1e3), "steps": steps,
            "ms_per_step": t_graph, "graph_ms_per_step": t_graph,
            "eager_ms_per_step": t_eager, "valid_tokens": tokens, "valid_pairs": pairs,
            "experts_with_rows": touched, "roofline": roof, "clocks": clk,
            "config": {"G": G, "M_per_shard": M, "K": K, "N": N, "E": E, "topk": k,
                       "worst_tokens": W, "scales": "fp32, 1x128 activations / 128x128 weights"}}


def measure_standard_entry(cfg, dev, steps, warmup, cpu_full=False):
    import torch
    layer = Layer(cfg, dev)
    for _ in range(warmup):
        layer.step()
    torch.cuda.synchronize()
    assert layer.err.item() == 0, f"device error word {layer.err.item()}"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        wall0 = time.time()
        t0.record()
        for i in range(steps):
            layer.step(ev[i])
        t1.record()
        torch.cuda.synchronize()
        wall1 = time.time()
    ms = t0.elapsed_time(t1)
    assert layer.err.item() == 0, f"device error word {layer.err.item()}"
    gemm_avg = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    roof, touched = _roofline(cfg, layer, gemm_avg, ms / 1e3)
    graph_ms, eager_call_ms = graph_time(layer, min(steps, 100))
    eb = 1 if cfg.dtype != WL.BF16 else 2
    wbytes = touched * 3 * cfg.N * cfg.K * eb
    entry = {"unit": "tokens/s", "value": cfg.M * steps / (ms / 1e3), "steps": steps,
             "ms_per_step": ms / steps, "graph_ms_per_step": graph_ms,
             "one_call_eager_ms_per_step": eager_call_ms,
             "graph_tokens_per_s": cfg.M / (graph_ms / 1e3),
             "kernel_ms": gemm_avg, "kernels_ms": stage_breakdown(layer, min(steps, 20)),
             "layer_tflops": 6.0 * cfg.K * cfg.N * cfg.P / (ms / steps / 1e3) / 1e12,
             "roofline": roof, "clocks": clk.summary(wall0, wall1),
             "config": {"M": cfg.M, "K": cfg.K, "N": cfg.N, "E": cfg.E, "topk": cfg.topk,
                        "scales": _scales_desc(cfg),
                        "l2": ("no flush; working set > L2 (%.2f GB of expert weights per step)"
                               % (wbytes / 1e9)) if wbytes > L2_BYTES else
                              ("L2-resident: %.1f MB of expert weights, no flush (a "
                               "launch-latency case)" % (wbytes / 1e6))},
             "gpu_launches_per_step": layer.launches_per_step}
    if cpu_full and cfg.name in FULL_ORACLE_WORKLOADS:
        entry["cpu_baseline"] = cpu_baseline_full(cfg, layer)
    elif cpu_full and cfg.dtype != WL.FP8_TENSOR:
        entry["cpu_baseline"] = cpu_baseline_pairs(cfg, layer)
    del layer
    return entry


def measure_batched_entry(cfg, dev, steps, warmup, cpu_full=False):
    """One CUDA graph of moe_batched_masked_experts replayed over resident
    inputs; the roofline covers both grouped GEMM launches.  e4m3: x_b comes
    quantised (1 x 128 group scales, as the prepare step hands it to the
    experts) and the weights block-quantised, both before the timed region."""
    import torch
    import mixture_experts_layer_count_gb300 as g
    g.load()
    d = WL.make_inputs(cfg, dev)
    E, T, N, K = cfg.E, cfg.M, cfg.N, cfg.K
    cpu = cpu_baseline_batched(cfg, d) if cpu_full else None
    xb, counts, w1, w2 = d["x_b"], d["counts"], d["w1"], d["w2"]
    yb = torch.empty_like(xb)
    fp8 = cfg.dtype == WL.FP8
    kw = {}
    if fp8:
        q1 = torch.empty((E, 2 * N, K), dtype=torch.uint8, device=dev)
        q2 = torch.empty((E, K, N), dtype=torch.uint8, device=dev)
        s1 = torch.empty((E, 2 * N // 128, K // 128), dtype=torch.float32, device=dev)
        s2 = torch.empty((E, K // 128, N // 128), dtype=torch.float32, device=dev)
        g.moe_quant_fp8_block(w1, q1, s1)
        g.moe_quant_fp8_block(w2, q2, s2)
        xq = torch.empty((E, T, K), dtype=torch.uint8, device=dev)
        xs = torch.empty((E * T, K // 128), dtype=torch.float32, device=dev)
        g.moe_quant_fp8_group(xb.view(E * T, K), xq.view(E * T, K), xs)
        del d["w1"], d["w2"]
        w1, w2, xb = q1, q2, xq
        kw = dict(dtype=WL.FP8, x_b_scales=xs, w1_scales=s1, w2_scales=s2)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.WS_BATCHED, T, E, N, K, 1, cfg.dtype, device=dev)
    rows = int(counts.clamp(0, T).sum().item())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warmup):
            g.moe_batched_masked_experts(xb, counts, N, w1, w2, yb, ws, err_word=err, **kw)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.moe_batched_masked_experts(xb, counts, N, w1, w2, yb, ws, err_word=err, **kw)
    for _ in range(warmup):
        graph.replay()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        wall0 = time.time()
        t0.record()
        for _ in range(steps):
            graph.replay()
        t1.record()
        torch.cuda.synchronize()
        wall1 = time.time()
    ms = t0.elapsed_time(t1)
    assert err.item() == 0, f"device error word {err.item()}"
    peaks, src = _peaks()
    key = "bf16_tflops" if ms / 1e3 < 2.0 else "bf16_tflops_sustained"
    peak = peaks.get(key, FALLBACK_PEAKS[key]) * (2.0 if fp8 else 1.0)
    flop = 6.0 * K * N * rows
    achieved = flop / (ms / steps / 1e3) / 1e12
    touched = int((counts > 0).sum().item())
    eb = 1 if fp8 else 2
    wbytes = touched * 3 * N * K * eb
    hbm = (wbytes + rows * K * (eb + 2)) / (ms / steps / 1e3) / 1e9
    return {"unit": "rows/s", "value": rows * steps / (ms / 1e3), "steps": steps,
            "ms_per_step": ms / steps, "graph_ms_per_step": ms / steps,
            "kernel_ms": ms / steps,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "tensor_frac": achieved / peak,
                         "hbm_frac": hbm / peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
                         "traffic": None, "flop_per_launch": flop,
                         "kernel": "grouped GEMM gate/up + down (one graph replay)",
                         "peak_source": f"{src} {key} (timed region {ms / 1e3:.2f} s)"
                                        + (" x2 (nominal fp8:bf16 dense ratio)" if fp8 else "")},
            **({"cpu_baseline": cpu} if cpu else {}),
            "clocks": clk.summary(wall0, wall1),
            "config": {"E": E, "T": T, "K": K, "N": N, "valid_rows": rows,
                       "scales": _scales_desc(cfg),
                       "experts_with_rows": touched,
                       "l2": "no flush; working set > L2 (%.2f GB of expert weights per "
                             "step)" % (wbytes / 1e9)}}


def _scales_desc(cfg):
    return {WL.BF16: "none", WL.FP8: "fp32, 1x128 activations / 128x128 weights",
            WL.FP8_CHANNEL: "fp32, per token / per output channel",
            WL.FP8_TENSOR: "fp32, per activation tensor / per output channel"}[cfg.dtype]


def _gate_up_kernel_name(cfg):
    """Which kernel runs the gate/up GEMM of a Standard-format workload: the
    library's dispatch (block-scaled e4m3 on the FP8 kernel, per-channel e4m3
    on the 1-SM kernel; bf16 on CTA pairs when the experts average 128 rows
    or more)."""
    if cfg.dtype == WL.FP8:
        return "grouped_gemm_fp8_kernel"
    if cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR):
        return "grouped_gemm_kernel"
    pairs = cfg.M * cfg.topk >= 128 * cfg.E
    return "grouped_gemm_pair_kernel" if pairs else "grouped_gemm_kernel"


def _roofline(cfg, layer, gemm_avg, timed_s):
    """Roofline of the dominant kernel, the gate/up grouped GEMM (2/3 of the
    layer's FLOPs), from its mean event-timed duration gemm_avg (ms).
    Algorithmic bytes per launch: w1 (+ scales) of the experts with rows, the
    gathered A rows read and H written.  Both the tensor and the HBM
    fractions are given; `bound` names the larger roofline time."""
    peaks, src = _peaks()
    P = cfg.M * cfg.topk
    fp8 = cfg.dtype != WL.BF16
    ch = cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR)
    eb = 1 if fp8 else 2
    gemm_flop = 4.0 * cfg.K * cfg.N * P
    counts = layer.counts.cpu().numpy()
    touched = int((counts > 0).sum())
    w1_scales = (2 * cfg.N if ch else (2 * cfg.N // 128) * (cfg.K // 128)) * 4 if fp8 else 0
    gemm_bytes = (touched * 2 * cfg.N * cfg.K * eb            # w1 of the experts with rows
                  + touched * w1_scales
                  + P * cfg.K * eb                            # A rows read
                  + P * cfg.N * (2 if ch else eb))            # H written (bf16 before its quant)
    key = "bf16_tflops" if timed_s < 2.0 else "bf16_tflops_sustained"
    tc_peak = peaks.get(key, FALLBACK_PEAKS[key]) * (2.0 if fp8 else 1.0)
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tc_time = gemm_flop / (tc_peak * 1e12)
    hbm_time = gemm_bytes / (hbm_peak * 1e9)
    tflops = gemm_flop / (gemm_avg / 1e3) / 1e12
    gbs = gemm_bytes / (gemm_avg / 1e3) / 1e9
    if tc_time >= hbm_time:
        roof = {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": tflops / tc_peak,
                "peak_source": f"{src} {key}" + (" x2 (nominal fp8:bf16 dense ratio)" if fp8 else "")
                               + f" (timed region {timed_s:.2f} s)"}
    else:
        roof = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_source": f"{src} hbm_gbs (copy)"}
    roof.update({"traffic": _kernel_traffic(cfg, "gate_up"),
                 "kernel": _gate_up_kernel_name(cfg) + ", gate/up + SiLU*mul",
                 "kernel_ms": gemm_avg, "flop_per_launch": gemm_flop,
                 "alg_bytes_per_launch": gemm_bytes, "experts_with_rows": touched,
                 "tensor_frac": tflops / tc_peak, "hbm_frac": gbs / hbm_peak})
    return roof, touched


def _line(args, cfg, layer, world, steps, ms, gemm_avg, e2e_ms, clocks):
    """The JSON result line (value fields filled in by the caller)."""
    P = cfg.M * cfg.topk
    fp8 = cfg.dtype != WL.BF16
    eb = 1 if fp8 else 2
    roof, touched = _roofline(cfg, layer, gemm_avg, ms / 1e3)
    layer_flop = 6.0 * cfg.K * cfg.N * P
    return {
        "metric": METRIC,
        "value": None,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) activations and logits; N(0,1/K), N(0,1/N) weights)",
        "config": {"workload": cfg.name, "M": cfg.M, "K": cfg.K, "N": cfg.N, "E": cfg.E,
                   "topk": cfg.topk, "format": "standard", "scales": _scales_desc(cfg),
                   "l2": "no flush; working set > L2 (%.2f GB of expert weights read per step)" %
                         (touched * 3 * cfg.N * cfg.K * eb / 1e9),
                   "parallelism": f"{world} independent replica(s)"},
        "layer_tflops": layer_flop / (ms / steps / 1e3) / 1e12,
        "roofline": roof,
        "e2e": {"value": None, "unit": "tokens/s",
                "h2d_bytes_per_step": int(layer.x.numel() * 2 + layer.logits.numel() * 4),
                "d2h_bytes_per_step": int(layer.out.numel() * 2),
                "pipeline": "copy-in, moe_forward and copy-out of consecutive steps on three "
                            "streams, two buffer sets"},
        "gpu_launches": layer.launches_per_step * steps,
        "clocks": clocks,
    }


def run_gpu_batched(args, cfg):
    """BatchedExperts (E, T, K) masked by device counts, as it is used: one
    CUDA graph of moe_batched_masked_experts captured once and replayed
    (step = one replay over resident inputs).  Throughput counts the valid
    rows (a token routed to an expert); the roofline covers both grouped
    GEMM launches of the call (6*K*N FLOP per valid row)."""
    import torch
    import mixture_experts_layer_count_gb300 as g
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    g.load()
    d = WL.make_inputs(cfg, dev)
    E, T, N, K = cfg.E, cfg.M, cfg.N, cfg.K
    xb, counts, w1, w2 = d["x_b"], d["counts"], d["w1"], d["w2"]
    yb = torch.empty_like(xb)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = g.workspace(g.WS_BATCHED, T, E, N, K, 1, WL.BF16, device=dev)
    rows = int(counts.clamp(0, T).sum().item())

    def call(x, c, y):
        g.moe_batched_masked_experts(x, c, N, w1, w2, y, ws, err_word=err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(max(1, args.warmup)):
            call(xb, counts, yb)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(xb, counts, yb)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    steps = args.steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()
        wall0 = time.time()
        t0.record()
        for _ in range(steps):
            graph.replay()
        t1.record()
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()
        wall1 = time.time()
    ms = t0.elapsed_time(t1)
    assert err.item() == 0, f"device error word {err.item()}"
    # end to end: every step copies x_b and the counts in from pinned host
    # memory and y_b back, inside the timed region; a second graph over a
    # second buffer set lets the copies of one step overlap its neighbour
    xh = xb.cpu().pin_memory()
    ch = counts.cpu().pin_memory()
    yh = [torch.empty(yb.shape, dtype=yb.dtype).pin_memory() for _ in range(2)]
    xb2, counts2, yb2 = torch.empty_like(xb), counts.clone(), torch.empty_like(yb)
    xb2.copy_(xb)
    with torch.cuda.stream(s):
        call(xb2, counts2, yb2)
    torch.cuda.current_stream().wait_stream(s)
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph2):
        call(xb2, counts2, yb2)
    sets = [(xb, counts, yb, graph), (xb2, counts2, yb2, graph2)]

    def h2d(b):
        sets[b][0].copy_(xh, non_blocking=True)
        sets[b][1].copy_(ch, non_blocking=True)

    def d2h(b):
        yh[b].copy_(sets[b][2], non_blocking=True)

    e2e_steps = max(2, min(steps, 50))
    pipelined_e2e(2, h2d, lambda b: sets[b][3].replay(), d2h)
    e2e_ms = pipelined_e2e(e2e_steps, h2d, lambda b: sets[b][3].replay(), d2h)
    assert err.item() == 0
    ms, e2e_ms = reduce_max([ms, e2e_ms], pg, device=dev)
    if rank != 0:
        return
    peaks, src = _peaks()
    timed_s = ms / 1e3
    key = "bf16_tflops" if timed_s < 2.0 else "bf16_tflops_sustained"
    peak = peaks.get(key, FALLBACK_PEAKS[key])
    flop = 6.0 * K * N * rows
    achieved = flop / (ms / steps / 1e3) / 1e12
    touched = int((counts > 0).sum().item())
    line = {
        "metric": METRIC, "value": replica_throughput(rows, steps, world, ms),
        "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; padded rows N(0,10^2) garbage)",
        "config": {"workload": cfg.name, "E": E, "T": T, "K": K, "N": N,
                   "format": "batched_experts, CUDA graph replay",
                   "valid_rows": rows, "experts_with_rows": touched,
                   "l2": "no flush; working set > L2 (%.2f GB of expert weights per step)" %
                         (touched * 3 * N * K * 2 / 1e9),
                   "parallelism": f"{world} independent replica(s)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": ("grouped_gemm_pair_kernel" if T >= 128 else "grouped_gemm_kernel")
                               + ", gate/up + down (one graph replay)",
                     "peak_source": f"{src} {key} (timed region {timed_s:.2f} s)",
                     "flop_per_launch": flop},
        "e2e": {"value": rows * e2e_steps * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(xb.numel() * 2 + counts.numel() * 4),
                "d2h_bytes_per_step": int(yb.numel() * 2),
                "pipeline": "copy-in, graph replay and copy-out of consecutive steps on three "
                            "streams, two buffer sets (two captured graphs)"},
        "gpu_launches": 2 * steps,
        "clocks": clk.summary(wall0, wall1),
    }
    print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


# ------------------------------------------------------------ CPU oracle --

def _oracle_inputs(cfg, d, tokens):
    import oracle as orc
    rid, _, _ = orc.route(d["logits"].cpu().numpy(),
                          None if d["bias"] is None else d["bias"].cpu().numpy(),
                          cfg.topk, cfg.score_fn, cfg.n_groups, cfg.topk_groups, cfg.renorm)
    experts = np.unique(rid[tokens])
    blocks = {}
    for e in experts:
        b1 = WL.bf16_bits(d["w1"][e])
        b2 = WL.bf16_bits(d["w2"][e])
        if cfg.dtype == WL.BF16:
            blocks[int(e)] = (b1, b2)
        elif cfg.dtype in (WL.FP8_CHANNEL, WL.FP8_TENSOR):
            q1, s1 = orc.quant_fp8_group(b1, group=cfg.K)
            q2, s2 = orc.quant_fp8_group(b2, group=cfg.N)
            blocks[int(e)] = (q1, q2, s1[:, 0], s2[:, 0])
        else:
            q1, s1 = orc.quant_fp8_block(b1)
            q2, s2 = orc.quant_fp8_block(b2)
            blocks[int(e)] = (q1, q2, s1, s2)
    return orc.Weights(cfg.dtype, experts=blocks, E=cfg.E, N=cfg.N, K=cfg.K)


def _time_oracle(cfg, d, W, tokens, threads):
    import oracle as orc
    t = time.perf_counter()
    orc.moe_forward(WL.bf16_bits(d["x"]), d["logits"].cpu().numpy(),
                    None if d["bias"] is None else d["bias"].cpu().numpy(), cfg.topk,
                    cfg.score_fn, W, cfg.n_groups, cfg.topk_groups, cfg.renorm,
                    cfg.requant_h, tokens=tokens, nthreads=threads)
    return time.perf_counter() - t


_TENSOR_UNBOUNDED = ("per-tensor activation scales couple every token: the oracle computes "
                     "all tokens' hidden rows before any output, so no bounded token sample "
                     "of this workload exists")


# small enough for the whole oracle layer in seconds: every token, on all
# host cores and (the tiny one) on one
FULL_ORACLE_WORKLOADS = {WL.TINY.name: (0, 1), WL.DSV3_DECODE.name: (0,)}


def cpu_baseline_full(cfg, layer):
    """The oracle on every token of the workload, on the listed thread counts
    (0 = all host cores); weights copied to the host before the clock
    starts."""
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    d = {"x": layer.x, "logits": layer.logits, "bias": layer.bias}
    d.update(WL.make_weights(cfg, layer.x.device))
    tokens = np.arange(cfg.M)
    W = _oracle_inputs(cfg, d, tokens)
    res = {"kind": "oracle", "unit": "tokens/s",
           "sample": f"all {cfg.M} tokens of {cfg.name}, fp64 per-token loops"}
    for threads in FULL_ORACLE_WORKLOADS[cfg.name]:
        n = cores if threads == 0 else threads
        _time_oracle(cfg, d, W, tokens[:1], n)  # page the weights in
        dt = _time_oracle(cfg, d, W, tokens, n)
        if threads == 0:
            res.update({"value": cfg.M / dt, "cores": n, "seconds": dt})
        else:
            res[f"threads_{n}"] = {"value": cfg.M / dt, "cores": n, "seconds": dt}
    return res


def cpu_baseline_pairs(cfg, layer, n_experts=4, rows_per_expert=32):
    """The oracle's expert rows -- the per-pair work of the layer, each routed
    row through its expert (e4m3: h requantised) -- on the first rows routed
    to a few experts with rows, all host cores; pairs/s, tokens/s = pairs/s /
    topk, and the whole run extrapolated.  Only those experts' weights are
    prepared, so the sample stays seconds on a 256-expert layer."""
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    x = layer.x
    rid, _, _ = orc.route(layer.logits.cpu().numpy(),
                          None if layer.bias is None else layer.bias.cpu().numpy(),
                          cfg.topk, cfg.score_fn, cfg.n_groups, cfg.topk_groups, cfg.renorm)
    rng = np.random.default_rng(0)
    present = np.unique(rid)
    experts = np.sort(rng.choice(present, min(n_experts, len(present)), replace=False))
    wd = WL.make_weights(cfg, x.device)  # the workload's weights (on the device)
    T = rows_per_expert
    xb = np.zeros((len(experts), T, cfg.K), np.uint16)
    counts = np.zeros(len(experts), np.int32)
    blocks = {}
    for i, e in enumerate(experts):
        toks = np.flatnonzero((rid == e).any(axis=1))[:T]
        counts[i] = len(toks)
        xb[i, :len(toks)] = WL.bf16_bits(x[torch_index(toks, x.device)])
        b1, b2 = WL.bf16_bits(wd["w1"][int(e)]), WL.bf16_bits(wd["w2"][int(e)])
        if cfg.dtype == WL.FP8:
            q1, s1 = orc.quant_fp8_block(b1)
            q2, s2 = orc.quant_fp8_block(b2)
            blocks[i] = (q1, q2, s1, s2)
        elif cfg.dtype == WL.FP8_CHANNEL:
            q1, s1 = orc.quant_fp8_group(b1, group=cfg.K)
            q2, s2 = orc.quant_fp8_group(b2, group=cfg.N)
            blocks[i] = (q1, q2, s1[:, 0], s2[:, 0])
        else:
            blocks[i] = (b1, b2)
    W = orc.Weights(cfg.dtype, experts=blocks, E=len(experts), N=cfg.N, K=cfg.K)
    out = np.empty((len(experts), T, cfg.K), np.float64)
    t = time.perf_counter()
    _, n = orc.batched_experts(xb, counts, W, requant_h=cfg.requant_h, nthreads=cores, out=out)
    dt = time.perf_counter() - t
    del wd
    pairs_s = n / dt
    return {"value": pairs_s / cfg.topk, "unit": "tokens/s", "pairs_per_s": pairs_s,
            "cores": cores, "kind": "oracle",
            "sample": f"{n} routed rows of experts {experts.tolist()} of {cfg.name} through "
                      f"their experts (the per-pair work; routing and the reduce left out), "
                      f"fp64 loops, {cores} OpenMP threads, {dt:.2f} s",
            "full_run_s_extrapolated": cfg.P / pairs_s}


def torch_index(idx, device):
    import torch
    return torch.from_numpy(np.asarray(idx, np.int64)).to(device)


def cpu_baseline_batched(cfg, d, n_rows=128):
    """The oracle's BatchedExperts rows (each valid row through its expert)
    on a seeded sample of valid rows, all host cores; rows/s, and the whole
    run extrapolated."""
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    counts = d["counts"].clamp(0, cfg.M).cpu().numpy()
    valid = np.array([(e, r) for e in range(cfg.E) for r in range(int(counts[e]))], np.int32)
    rng = np.random.default_rng(0)
    rows = valid[np.sort(rng.choice(len(valid), min(n_rows, len(valid)), replace=False))]
    blocks = {}
    for e in np.unique(rows[:, 0]):
        b1, b2 = WL.bf16_bits(d["w1"][e]), WL.bf16_bits(d["w2"][e])
        if cfg.dtype == WL.FP8:
            q1, s1 = orc.quant_fp8_block(b1)
            q2, s2 = orc.quant_fp8_block(b2)
            blocks[int(e)] = (q1, q2, s1, s2)
        else:
            blocks[int(e)] = (b1, b2)
    W = orc.Weights(cfg.dtype, experts=blocks, E=cfg.E, N=cfg.N, K=cfg.K)
    xb = WL.bf16_bits(d["x_b"])
    out = np.empty((cfg.E, cfg.M, cfg.K), np.float64)  # only the sampled rows are written
    t = time.perf_counter()
    orc.batched_experts(xb, counts, W, rows=rows, requant_h=cfg.dtype == WL.FP8,
                        nthreads=cores, out=out)
    dt = time.perf_counter() - t
    return {"value": len(rows) / dt, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {len(valid)} valid rows of {cfg.name}, fp64 loops, "
                      f"{cores} OpenMP threads, {dt:.1f} s",
            "full_run_s_extrapolated": len(valid) * dt / len(rows)}


def cpu_baseline(cfg, layer, budget_s):
    """The oracle as it stands on the host cores, on a bounded token sample."""
    if cfg.dtype == WL.FP8_TENSOR:
        return {"unavailable": _TENSOR_UNBOUNDED}
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    d = {"x": layer.x, "logits": layer.logits, "bias": layer.bias}
    wd = WL.make_weights(cfg, layer.x.device)
    d.update(wd)
    rng = np.random.default_rng(0)
    probe = rng.choice(cfg.M, cores, replace=False)
    n_target = cores
    W = _oracle_inputs(cfg, d, np.arange(cfg.M))
    dt = _time_oracle(cfg, d, W, probe, cores)
    n_target = int(max(cores, min(cfg.M, cores * max(1, math.floor(budget_s / max(dt, 1e-3))))))
    tokens = rng.choice(cfg.M, n_target, replace=False)
    dt = _time_oracle(cfg, d, W, tokens, cores)
    return {"value": len(tokens) / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(tokens)} of {cfg.M} tokens of {cfg.name}, fp64 per-token loops, "
                      f"{cores} OpenMP threads, {dt:.1f} s"}


def run_reference(args, cfg):
    """--impl reference: the CPU oracle (this build's reference arm), timed
    per step on a bounded token sample of the same workload."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    if cfg.dtype == WL.FP8_TENSOR:
        print(json.dumps({"impl": "reference", "unavailable": _TENSOR_UNBOUNDED}), flush=True)
        return
    import torch
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = WL.make_inputs(cfg, dev)
    tokens_per_step = cores
    rng = np.random.default_rng(0)
    W = _oracle_inputs(cfg, d, np.arange(cfg.M))
    for _ in range(args.warmup):
        _time_oracle(cfg, d, W, rng.choice(cfg.M, 1, replace=False), cores)
    total = 0.0
    for _ in range(args.steps):
        total += _time_oracle(cfg, d, W, rng.choice(cfg.M, tokens_per_step, replace=False), cores)
    value = tokens_per_step * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if cfg.dtype == WL.BF16 else "fp8_e4m3", "data": "synthetic",
            "config": {"workload": cfg.name, "M": cfg.M, "K": cfg.K, "N": cfg.N, "E": cfg.E,
                       "topk": cfg.topk, "format": "standard", "scales": _scales_desc(cfg),
                       "sample_tokens_per_step": tokens_per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{tokens_per_step} tokens per step of {cfg.name}"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gbmoe", choices=["gbmoe", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-features", action="store_true",
                    help="leave out the features object (shared experts, chunking, EP, "
                         "per-channel and per-tensor e4m3)")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the chosen workload (no per_workload object)")
    args = ap.parse_args()
    cfg = WORKLOADS[args.workload]
    if args.impl == "reference":
        if cfg.batched:
            raise SystemExit("the reference arm times the Standard workloads")
        run_reference(args, cfg)
    elif cfg.batched:
        if cfg.dtype != WL.BF16:
            raise SystemExit("the e4m3 BatchedExperts workload is timed in the per_workload "
                             "object of the default line")
        run_gpu_batched(args, cfg)
    else:
        run_gpu(args, cfg)


if __name__ == "__main__":
    main()
