"""Benchmark of the MoE FFN layer forward on one GB300: MoE-layer tokens/s and
the roofline fraction of the layer and of its dominant kernel.

    python bench.py [--steps K] [--warmup W] [--workload decode --T 8] [--no-sweep] [--impl reference]

A step is one whole-layer forward (route, dispatch, gate_up GroupedMatmul with
SiLU*mul, down GroupedMatmul, combine, shared expert on the side stream) over
one batch of T synthetic tokens.  Inputs are seeded and synthetic with the
workload's shapes and distributions.  Expert weights rotate over R device
copies so that every step streams its experts' weights from HBM rather than
L2.  One forward per copy is captured in a CUDA graph (its output first
checked bit for bit against the eager forward) and the graphs are replayed
back to back; K replays are timed with CUDA events on the launching stream.

The headline line is the named workload (default: decode T=8) timed over
exactly K steps.  Unless --no-sweep is given, the line also carries
``workloads``: every decode, batched-decode and prefill shape of the metric,
each timed over its own step count (about a quarter second of replays), with
its layer roofline, its dominant kernel's roofline and the clock samples of
its own timed window.  Clocks are sampled every 20 ms over the whole
measurement phase.

One GPU only: the layer does not shard, and its prefill matmuls share operand
tiles between the two CTAs of a cluster by TMA multicast, which stays inside
one GPU's own memory.  ``--gpus N`` with N > 1 (or WORLD_SIZE > 1) is refused
before anything is built or loaded.

``--impl reference`` times the CPU oracle instead, on bounded samples of the
same workload (rank 0 only under torchrun).
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (decode T=1..256, prefill T=8K) and % of HBM/TC roofline"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# every shape of the metric, timed after the headline unless --no-sweep
SWEEP = [("decode", 1), ("decode", 4), ("decode", 8), ("batched_decode", 64), ("batched_decode", 256),
         ("prefill", 8192), ("large_prefill", 16384),
         # the same decode shapes with FP8 (e4m3, per-row scales) routed expert weights
         ("decode_w8", 1), ("decode_w8", 4), ("decode_w8", 8), ("batched_decode_w8", 64),
         ("batched_decode_w8", 256)]
SWEEP_SECONDS = 0.25          # timed replays per sweep workload
MIN_FORWARDS_PER_GRAPH = 8    # a model's decode step holds dozens of MoE layers in one graph
ONE_GPU = ("one GPU only: the layer does not shard, and its prefill matmuls share operand tiles between the two "
           "CTAs of a cluster by TMA multicast, which stays inside one GPU's own memory")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- algorithmic units

def is_w8(w) -> bool:
    """A workload with FP8 (e4m3) routed expert weights (per-row fp32 scales)."""
    return w.name.split("@")[0].endswith("_w8")


def expert_bytes(w) -> int:
    """Bytes of one routed expert's weights: 3 I H elements (2 or 1 bytes each)
    plus, for FP8, one fp32 scale per weight row (2I + H rows)."""
    return 3 * w.H * w.I + (2 * w.I + w.H) * 4 if is_w8(w) else 6 * w.H * w.I


def layer_units(w, nonempty):
    """Algorithmic bytes and FLOPs of one layer forward (intermediates not
    counted): weights of every expert that received a token, the shared expert,
    the router, x and out; FLOPs of the routed and shared MLPs and the router."""
    bytes_ = (expert_bytes(w) * nonempty + 6 * w.H * w.Is + 4 * w.E * w.H + 2 * w.T * w.H * 2)
    flops = 2 * w.T * w.k * 3 * w.H * w.I + 2 * w.T * 3 * w.H * w.Is + 2 * w.T * w.E * w.H
    return bytes_, flops


def routed_units(w, nonempty):
    """The routed path alone (router, dispatch, both routed matmuls, combine):
    weights of the non-empty experts, the router weights, x and out."""
    bytes_ = expert_bytes(w) * nonempty + 4 * w.E * w.H + 2 * w.T * w.H * 2
    flops = 2 * w.T * w.k * 3 * w.H * w.I + 2 * w.T * w.E * w.H
    return bytes_, flops


def gate_up_units(w, nonempty):
    """gate_up GroupedMatmul: reads the 2I x H weights of each non-empty expert
    (and their row scales, FP8) and the T*k dispatched rows, writes T*k rows of h."""
    rows = w.T * w.k
    wb = nonempty * 2 * w.I * (w.H + 4) if is_w8(w) else nonempty * 2 * w.I * w.H * 2
    bytes_ = wb + rows * w.H * 2 + rows * w.I * 2
    flops = 2 * rows * 2 * w.I * w.H
    return bytes_, flops


def tokens_per_s(tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput of `steps` steps of `tokens_per_step` tokens in `ms`."""
    return steps * tokens_per_step / (ms / 1e3)


def weight_copies(w) -> tuple[int, int]:
    """(R, touched bytes): R device copies of the expert weights, enough that R
    x the bytes one forward touches is at least 4 x L2."""
    touched = min(w.E, w.T * w.k) * expert_bytes(w) + 6 * w.H * w.Is
    return int(min(16, max(2, -(-4 * L2_BYTES // max(touched, 1))))), touched


def _routing_desc(w):
    if w.zipf_s is None and not w.n_empty:
        return f"router W ~ N(0,{w.sigma_router}), near-uniform"
    s = f"router W ~ N(0,{w.sigma_router}) + Zipf(s={w.zipf_s}) log-rank bias"
    return s + (f", {w.n_empty} experts forced empty" if w.n_empty else "")


def config_of(w) -> dict:
    """The workload's config dict (the same for both arms)."""
    R, touched = weight_copies(w)
    return {"workload": f"{w.name.split('@')[0]} T={w.T}", "T": w.T, "H": w.H, "E": w.E, "k": w.k, "I": w.I,
            "I_s": w.Is, "routing": _routing_desc(w), "parallelism": "one GPU (the layer does not shard)",
            "weights": ("routed experts e4m3 with per-row fp32 scales, shared expert bf16" if is_w8(w)
                        else "bf16"),
            "l2": f"expert weights rotate over {R} device copies ({R} x {touched / 1e6:.0f} MB touched >= 4 x L2); "
                  f"the timed CUDA graph holds consecutive forwards over the copies in turn (as consecutive MoE "
                  f"layers of a model run in one graph), replayed back to back"}


# ---------------------------------------------------------------- clocks

CLOCK_Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
           "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
           "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples every 20 ms for the whole measurement phase; window()
    summarises the samples whose own timestamps fall in a host-time window."""

    def __init__(self, index: int, period_ms: int = 20):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_Q}", "--format=csv,noheader,nounits",
                                          "-i", str(index), "-lms", str(period_ms)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx, pw = float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            active = [n for n, v in zip(_REASONS, f[5:9]) if v.lower() == "active"]
            self.samples.append((t, sm, mx, pw, active))

    def window(self, t0: float, t1: float, pad: float = 0.0) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        s = [x for x in list(self.samples) if t0 - pad <= x[0] <= t1 + pad]
        reasons = sorted({r for x in s for r in x[4]})
        return {"sm_mhz": statistics.median(x[1] for x in s) if s else None,
                "sm_max_mhz": max(x[2] for x in s) if s else None,
                "power_w_max": max(x[3] for x in s) if s else None, "reasons": reasons, "samples": len(s),
                "window_s": round(t1 - t0 + 2 * pad, 3)}

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()


# ---------------------------------------------------------------- CPU oracle timing

def time_oracle(w, inp, budget_s: float, max_tokens: int | None = None):
    """Oracle forward of tokens of the workload, token batches evaluated one by
    one until `budget_s` of wall time has passed; returns (tokens/s, cores,
    tokens done, seconds)."""
    from oracle import moe_oracle as om
    ids, wts, _ = om.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    T = w.T
    batch = T if T <= 16 else 8
    done, t0, c0 = 0, time.perf_counter(), time.process_time()
    rng = np.random.default_rng(1)
    while True:
        toks = np.arange(T) if batch == T else rng.choice(T, size=batch, replace=False)
        om.forward_tokens(inp, w.k, toks, routing=(ids, wts))
        done += len(toks)
        el = time.perf_counter() - t0
        if el >= budget_s or (max_tokens and done >= max_tokens):
            break
    el = time.perf_counter() - t0
    cores = (time.process_time() - c0) / el
    return done / el, cores, done, el


# ---------------------------------------------------------------- GPU arm

class WeightBed:
    """Device copies of one set of expert and shared weights; workloads with
    the same layer sizes (decode, batched decode and prefill) share them."""

    def __init__(self, w, seed, dev):
        import torch

        from moe_ffn_layer_gb300 import synth
        from moe_ffn_layer_gb300.layer import bf16_tensor
        self.dev = dev
        sgu, sd = synth.make_shared_weights(w, seed)
        b16 = lambda a: None if a is None else bf16_tensor(a, dev)
        if is_w8(w):
            wgu, swgu, wd, swd = synth.make_expert_weights_w8(w, seed)
            self.host = dict(w_gate_up=wgu, w_gate_up_scale=swgu, w_down=wd, w_down_scale=swd, ws_gate_up=sgu,
                             ws_down=sd)
            u8 = lambda a: torch.from_numpy(a).to(dev)
            # (gate_up, down, shared gate_up, shared down, gate_up scales, down scales)
            self.copies = [(u8(wgu), u8(wd), b16(sgu), b16(sd), torch.from_numpy(swgu).to(dev),
                            torch.from_numpy(swd).to(dev))]
        else:
            wgu, wd = synth.make_expert_weights(w, seed)
            self.host = dict(w_gate_up=wgu, w_down=wd, ws_gate_up=sgu, ws_down=sd)
            self.copies = [(b16(wgu), b16(wd), b16(sgu), b16(sd))]
        self._torch = torch

    def get(self, R):
        while len(self.copies) < R:
            t = self.copies[0]
            self.copies.append(tuple(None if a is None else a.clone() for a in t))
        return self.copies[:R]


def _timed_graph(graphs, stream, K, e0, e1, pre_s=0.0, post_s=0.0):
    """Replays graphs[i % R] K times between two events; optional untimed
    replays before and after (host-time bounded) keep the load steady around
    the timed region.  Returns (ms, t_start, t_end) in host time."""
    R = len(graphs)
    t_pre = time.time()
    if pre_s > 0:
        i = 0
        while time.time() - t_pre < pre_s:
            for _ in range(64):
                graphs[i % R].replay()
                i += 1
            stream.synchronize()
    e0.record(stream)
    for i in range(K):
        graphs[i % R].replay()
    e1.record(stream)
    e1.synchronize()
    t_post = time.time()
    if post_s > 0:
        i = 0
        while time.time() - t_post < post_s:
            for _ in range(64):
                graphs[i % R].replay()
                i += 1
            stream.synchronize()
    return e0.elapsed_time(e1), t_pre, time.time()


def measure(w, bed, args, clk, K, W, headline=False):
    import torch

    from moe_ffn_layer_gb300 import binding as B
    from moe_ffn_layer_gb300 import synth
    from moe_ffn_layer_gb300.layer import MoEFFN, bf16_tensor

    dev = bed.dev
    x_np, wr_np, b_np = synth.make_activations(w, args.seed)
    x = bf16_tensor(x_np, dev)
    wr = torch.from_numpy(wr_np).to(dev)
    b = None if b_np is None else torch.from_numpy(b_np).to(dev)
    R, _ = weight_copies(w)
    if args.copies:
        R = args.copies
    copies = bed.get(R)
    layers = [MoEFFN(w.k, wr, b, *c) for c in copies]   # (FP8 copies carry their scales last)
    outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for L, o in zip(layers, outs):          # eager forwards (set kernel attributes, size workspaces)
            L.forward(x, o, stream)
    stream.synchronize()
    launches = B.moe_last_launch_count()
    assert B.moe_last_device_error(stream) == 0
    eager0 = outs[0].clone()
    graphs = []
    for L, o in zip(layers, outs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            L.forward(x, o, torch.cuda.current_stream())
        graphs.append(g)
    torch.cuda.synchronize()
    outs[0].fill_(0)
    with torch.cuda.stream(stream):
        graphs[0].replay()
    stream.synchronize()
    graph_same = bool(torch.equal(outs[0].view(torch.int16), eager0.view(torch.int16)))

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(W):
            graphs[i % R].replay()
        stream.synchronize()
        if K is None:                           # sweep: about SWEEP_SECONDS of replays
            ms, _, _ = _timed_graph(graphs, stream, 2 * R, e0, e1)
            K = int(min(20000, max(20, SWEEP_SECONDS * 1e3 / max(ms / (2 * R), 1e-3))))
            K = -(-K // max(R, MIN_FORWARDS_PER_GRAPH)) * max(R, MIN_FORWARDS_PER_GRAPH)
        torch.cuda.synchronize()
        # one forward per graph, replayed back to back: every forward also pays
        # the gap between two graph launches (reported beside the value)
        ms1, _, _ = _timed_graph(graphs, stream, K, e0, e1)
    torch.cuda.synchronize()
    # The timed graph holds F consecutive forwards, forward j on weight copy
    # j mod R, as consecutive MoE layers of a model's decode step run inside
    # one graph; F is the smallest divisor of K not below R or
    # MIN_FORWARDS_PER_GRAPH (else K), so that the K timed steps are whole
    # replays.
    F = next((f for f in range(max(R, MIN_FORWARDS_PER_GRAPH), K + 1) if K % f == 0), K)
    gm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gm, stream=stream):
        cs = torch.cuda.current_stream()
        for j in range(F):
            layers[j % R].forward(x, outs[j % R], cs)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(-(-W // F)):
            gm.replay()
        stream.synchronize()
        ms, t0, t1 = _timed_graph([gm], stream, K // F, e0, e1, pre_s=0.15 if headline else 0.0,
                                  post_s=0.1 if headline else 0.0)
    torch.cuda.synchronize()
    clocks = clk.window(t0, t1, pad=0.03)
    assert B.moe_last_device_error(stream) == 0
    # every copy holds the same weights: each output of the timed graph equals the eager one
    graph_same = graph_same and all(torch.equal(o.view(torch.int16), eager0.view(torch.int16))
                                    for o in outs[:min(R, F)])
    value = tokens_per_s(w.T, K, ms)

    # the routing of this batch, through the route and permute calls
    ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
    rb = B.moe_route_workspace_bytes(w.T, w.H, w.E)
    pb = B.moe_permute_workspace_bytes(w.T, w.E)
    rws = torch.empty(max(rb, pb, 256), dtype=torch.uint8, device=dev)
    offs = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
    st = torch.empty(w.T * w.k, dtype=torch.int32, device=dev)
    inv = torch.empty(w.T * w.k, dtype=torch.int32, device=dev)
    xperm = torch.empty((w.T * w.k, w.H), dtype=torch.bfloat16, device=dev)
    B.moe_route(x, wr, b, w.T, w.H, w.E, w.k, ids, tw, rws, rb, stream)
    B.moe_permute(ids, x, w.T, w.H, w.E, w.k, offs, st, inv, xperm, rws, pb, stream)
    stream.synchronize()
    nonempty = int((offs[1:] - offs[:-1] > 0).sum().item())
    pk, pk_src = peaks()
    lbytes, lflops = layer_units(w, nonempty)
    step_s = ms / 1e3 / K
    hbm = pk["hbm_gbs"] * 1e9
    tc = pk["bf16_tflops_sustained"] * 1e12
    t_roof = max(lbytes / hbm, lflops / tc)
    layer_roof = {"bytes": lbytes, "flops": lflops, "nonempty_experts": nonempty,
                  "roofline_us": t_roof * 1e6, "step_us": step_s * 1e6, "frac": t_roof / step_s,
                  "bound": "hbm" if lbytes / hbm >= lflops / tc else "tensor",
                  "peaks": f"{pk_src}: {pk['hbm_gbs']} GB/s, {pk['bf16_tflops_sustained']} TFLOP/s sustained"}
    roof = dominant_kernel(w, copies, wr, b, x, offs, xperm, nonempty, pk, pk_src, stream, e0, e1, K)
    res = {"value": value, "ms_per_step": ms / K, "steps": K, "warmup": W, "layer_roofline": layer_roof,
           "forwards_per_graph": F, "ms_per_step_one_forward_per_graph": ms1 / K,
           "roofline": roof, "clocks": clocks, "launches_per_step": launches, "graph_matches_eager": graph_same,
           "config": config_of(w)}
    if headline:
        res["e2e"] = end_to_end(w, layers, outs, x, stream, e0, e1, K)
    del graphs
    return res


def dominant_kernel(w, copies, wr, b, x, offs, xperm, nonempty, pk, pk_src, stream, e0, e1, K):
    """The step's dominant work, timed alone back to back in one graph over the
    weight copies, in the configuration the layer itself runs.  Up to 16
    tokens: the routed path (the layer without its shared expert: router and
    dispatch, gate_up reading the dispatched rows of x through the sort, down,
    combine).  Above: the routed gate_up GroupedMatmul on the layer's
    dispatched rows."""
    import torch

    from moe_ffn_layer_gb300 import binding as B
    from moe_ffn_layer_gb300.layer import MoEFFN
    R = len(copies)
    M = max(20, min(400, K))
    if w.T <= 16:
        routed = [MoEFFN(w.k, wr, b, c[0], c[1], None, None, *c[4:]) for c in copies]
        o = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=x.device)
        # (an NVTX range, so that a profiler can pick out these launches: one
        # forward of the routed path per weight copy)
        torch.cuda.nvtx.range_push("routed_path_eager")
        for L in routed:
            L.forward(x, o, stream)
        torch.cuda.nvtx.range_pop()
        n_launch = None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cs = torch.cuda.current_stream()
            for i in range(M):
                routed[i % R].forward(x, o, cs)
                n_launch = B.moe_last_launch_count()
        kernel = "routed path (layer without its shared expert)"
        gb, gf = routed_units(w, nonempty)
    else:
        h = torch.empty((w.T * w.k, w.I), dtype=torch.bfloat16, device=x.device)
        gb_ws = B.moe_grouped_gemm_workspace_bytes(w.E, w.T * w.k, w.I, w.H, 1)
        g_ws = torch.zeros(max(gb_ws, 256), dtype=torch.uint8, device=x.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cs = torch.cuda.current_stream()
            for i in range(M):
                if is_w8(w):
                    B.moe_grouped_gemm_w8(xperm, copies[i % R][0], copies[i % R][4], offs, w.E, w.T * w.k, w.I, w.H,
                                          1, h, g_ws, gb_ws, cs)
                else:
                    B.moe_grouped_gemm(xperm, copies[i % R][0], offs, w.E, w.T * w.k, w.I, w.H, 1, h, g_ws, gb_ws,
                                       cs)
                n_launch = B.moe_last_launch_count()
        kernel = "grouped_gemm gate_up+SiLU*mul" + (" (e4m3 weights)" if is_w8(w) else "")
        gb, gf = gate_up_units(w, nonempty)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        g.replay()
        e1.record(stream)
    e1.synchronize()
    assert B.moe_last_device_error(stream) == 0
    k_us = e0.elapsed_time(e1) * 1e3 / M
    if w.T * w.k <= 64 * w.E:     # weight streaming: HBM-bound
        achieved = gb / (k_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"]}
    else:
        achieved = gf / (k_us * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"]}
    roof.update({"traffic": _traffic(w), "kernel": kernel, "us_per_launch": k_us, "launches": n_launch,
                 "algorithmic_bytes": gb, "algorithmic_flops": gf, "peak_source": pk_src + " (burst)"})
    return roof


def end_to_end(w, layers, outs, x, stream, e0, e1, K):
    """The same metric through the public call: pinned host x -> device,
    forward, out -> pinned host, every step, no graph."""
    import torch
    R = len(layers)
    xh = x.cpu().pin_memory()
    oh = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)
    KE = max(5, min(K, 200))
    with torch.cuda.stream(stream):
        for i in range(3):
            xd.copy_(xh, non_blocking=True)
            layers[i % R].forward(xd, outs[i % R], stream)
            oh.copy_(outs[i % R], non_blocking=True)
        stream.synchronize()
        e0.record(stream)
        for i in range(KE):
            xd.copy_(xh, non_blocking=True)
            layers[i % R].forward(xd, outs[i % R], stream)
            oh.copy_(outs[i % R], non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / KE
    return {"value": w.T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": w.T * w.H * 2,
            "d2h_bytes_per_step": w.T * w.H * 2, "ms_per_step": e2e_ms, "steps": KE,
            "path": "MoEFFN.forward (one moe_forward call), no graph"}


def run_gpu(args, w):
    import torch

    from moe_ffn_layer_gb300 import build as build_mod
    from moe_ffn_layer_gb300 import synth

    build_mod.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    clk = ClockSampler(0)
    beds = {}

    def bed_for(wl):
        key = (wl.H, wl.E, wl.I, wl.Is, wl.sigma_w, is_w8(wl))
        if key not in beds:
            if len(beds) >= 1:          # one set of weights on the device at a time
                beds.clear()
                torch.cuda.empty_cache()
            beds[key] = WeightBed(wl, args.seed, dev)
        return beds[key]

    try:
        head = measure(w, bed_for(w), args, clk, args.steps, args.warmup, headline=True)
        cpu = None
        if not args.no_cpu_baseline:
            inp = dict(zip(("x", "w_router", "bias"), synth.make_activations(w, args.seed)))
            inp.update(bed_for(w).host)
            tps, cores, ntok, el = time_oracle(w, inp, args.cpu_budget)
            cpu = {"value": tps, "unit": UNIT, "cores": round(cores, 2), "kind": "oracle",
                   "sample": f"{ntok} tokens of the same workload through the float64 oracle, token batches "
                             f"of {min(w.T, 8) if w.T > 16 else w.T}, {el:.1f} s wall; cores = CPU time / wall "
                             f"time (numpy BLAS pool of {os.cpu_count()} threads)"}
        sweep = {}
        if not args.no_sweep:
            for name, T in SWEEP:
                wl = synth.workload(name, T)
                r = measure(wl, bed_for(wl), args, clk, None, 5)
                sweep[r["config"]["workload"]] = {k: r[k] for k in ("value", "ms_per_step", "steps", "forwards_per_graph",
                                                                    "ms_per_step_one_forward_per_graph",
                                                                    "layer_roofline",
                                                                    "roofline", "clocks", "launches_per_step",
                                                                    "graph_matches_eager")}
    finally:
        clk.stop()

    result = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; workload shapes and distributions)",
        "config": head["config"], "clocks": head["clocks"], "e2e": head["e2e"],
        "gpu_launches": args.steps * head["launches_per_step"], "launches_per_step": head["launches_per_step"],
        "roofline": head["roofline"], "layer_roofline": head["layer_roofline"], "cpu_baseline": cpu,
        "graph_matches_eager": head["graph_matches_eager"],
        "forwards_per_graph": head["forwards_per_graph"],
        "ms_per_step_one_forward_per_graph": head["ms_per_step_one_forward_per_graph"],
        "clocks_note": "sampled every 20 ms; the headline window spans 0.15 s of untimed replays of the same "
                       "graphs before the timed steps and 0.1 s after them",
    }
    if sweep:
        result["workloads"] = sweep
    return result


# ---------------------------------------------------------------- reference arm

def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from moe_ffn_layer_gb300 import synth
    from oracle import moe_oracle as om
    inp = synth.make_inputs(w, args.seed)
    ids, wts, _ = om.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    # bounded sample per step: a few tokens, sized so the run ends in minutes
    t0 = time.perf_counter()
    om.forward_tokens(inp, w.k, np.arange(1), routing=(ids, wts))
    per_tok = max(time.perf_counter() - t0, 1e-3)
    n = int(max(1, min(w.T, 120.0 / (args.steps + args.warmup) / per_tok)))
    rng = np.random.default_rng(2)
    for _ in range(args.warmup):
        om.forward_tokens(inp, w.k, rng.choice(w.T, size=n, replace=False), routing=(ids, wts))
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(args.steps):
        om.forward_tokens(inp, w.k, rng.choice(w.T, size=n, replace=False), routing=(ids, wts))
    el = time.perf_counter() - t0
    cores = (time.process_time() - c0) / el
    value = args.steps * n / el
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; workload shapes and distributions)", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": round(cores, 2), "kind": "oracle",
                             "sample": f"{n} random tokens of the workload per step through the float64 oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _traffic(w):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    capture of the same kernel source, else None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(f"{w.name.split('@')[0]}@T{w.T}")
    if not e:
        return None
    src = os.path.join(ROOT, "moe_ffn_layer_gb300", "csrc", e.get("source", "grouped_gemm.cu"))
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if e.get("source_sha") != h:
        return None
    return e.get("dram_bytes_per_launch")


def refuse_multi_gpu(args) -> bool:
    """True (after printing one line) when asked for more than one GPU."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus <= 1 and world <= 1:
        return False
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps({"metric": METRIC, "unit": UNIT, "n_gpus": max(args.gpus, world), "impl": args.impl,
                          "unavailable": f"multi-GPU runs closed on this pool; {ONE_GPU}"}), flush=True)
    return True


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="time the named workload only")
    ap.add_argument("--copies", type=int, default=0, help="weight copies to rotate over (0: enough to defeat L2)")
    args = ap.parse_args()
    if args.impl == "own" and refuse_multi_gpu(args):
        return
    from moe_ffn_layer_gb300 import synth
    T = args.T if args.T is not None else (8 if args.workload == "decode" else None)
    w = synth.workload(args.workload, T)
    if args.steps is None:
        args.steps = 200 if args.impl == "own" else 20
    args.warmup = max(args.warmup, 3)
    res = run_reference(args, w) if args.impl == "reference" else run_gpu(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
