"""Benchmark of the MoE FFN layer forward on GB300: MoE-layer tokens/s and the
roofline fraction of the dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode --T 8] [--impl reference]

A step is one whole-layer forward (route, dispatch, gate_up GroupedMatmul with
SiLU*mul, down GroupedMatmul, combine, shared expert on the side stream) over
one batch of T synthetic tokens.  Inputs are seeded and synthetic with the
workload's shapes and distributions.  Expert weights rotate over R device
copies so that every step streams its experts' weights from HBM rather than L2.
One forward per copy is captured in a CUDA graph and the graphs are replayed
back to back; K replays are timed with CUDA events on the launching stream.

Under torchrun (N > 1) each rank runs its own replica of the layer on its GPU
(the layer does not shard: replicas only); rank 0 prints one JSON line with
value = tokens of all ranks / max time over ranks.

``--impl reference`` times the CPU oracle instead (rank 0 only), on bounded
samples of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (decode T=1..256, prefill T=8K) and % of HBM/TC roofline"
UNIT = "tokens/s"
DEFAULT_STEPS = {"tiny": 2000, "decode": 4000, "batched_decode": 2000, "prefill": 300, "large_prefill": 60}
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- algorithmic units

def layer_units(w, nonempty):
    """Algorithmic bytes and FLOPs of one layer forward (intermediates not
    counted): weights of every expert that received a token, the shared expert,
    the router, x and out; FLOPs of the routed and shared MLPs and the router."""
    bytes_ = (6 * w.H * w.I * nonempty + 6 * w.H * w.Is + 4 * w.E * w.H + 2 * w.T * w.H * 2)
    flops = 2 * w.T * w.k * 3 * w.H * w.I + 2 * w.T * 3 * w.H * w.Is + 2 * w.T * w.E * w.H
    return bytes_, flops


def gate_up_units(w, nonempty):
    """gate_up GroupedMatmul: reads the 2I x H weights of each non-empty expert
    and the T*k dispatched rows, writes T*k rows of h."""
    rows = w.T * w.k
    bytes_ = nonempty * 2 * w.I * w.H * 2 + rows * w.H * 2 + rows * w.I * 2
    flops = 2 * rows * 2 * w.I * w.H
    return bytes_, flops


# ---------------------------------------------------------------- clocks

CLOCK_Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
           "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
           "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_Q}", "--format=csv,noheader,nounits",
                                          "-i", str(index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
                pw.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(ms_local: float, tokens_per_rank: int, steps: int, world: int):
    """(tokens/s of all ranks together, ms of the slowest rank) for `steps`
    timed steps of `tokens_per_rank` tokens on every rank."""
    ms = max_over_ranks(ms_local, world)
    return world * steps * tokens_per_rank / (ms / 1e3), ms


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


# ---------------------------------------------------------------- main arm

def run_gpu(args, w):
    import torch

    from moe_ffn_layer_gb300 import binding as B
    from moe_ffn_layer_gb300 import build as build_mod
    from moe_ffn_layer_gb300 import synth
    from moe_ffn_layer_gb300.layer import MoEFFN, bf16_tensor

    build_mod.build()
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = synth.make_inputs(w, args.seed)
    base = MoEFFN.from_inputs(inp, w.k, dev)
    x = bf16_tensor(inp["x"], dev)

    # weight copies: R x touched bytes >= 4 x L2
    wgt_bytes = (2 * w.I * w.H + w.H * w.I) * 2
    touched = min(w.E, w.T * w.k) * wgt_bytes + 6 * w.H * w.Is
    R = int(min(16, max(2, -(-4 * L2_BYTES // max(touched, 1)))))
    if args.copies:
        R = args.copies
    layers = [base]
    for _ in range(R - 1):
        t = base.tensors
        layers.append(MoEFFN(w.k, t[0], t[1], t[2].clone(), t[3].clone(),
                             None if t[4] is None else t[4].clone(), None if t[5] is None else t[5].clone()))
    outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for L, o in zip(layers, outs):          # eager warm-up (sets kernel attributes, sizes workspaces)
            L.forward(x, o, stream)
    stream.synchronize()
    launches = B.moe_last_launch_count()
    assert B.moe_last_device_error(stream) == 0
    graphs = []
    for L, o in zip(layers, outs):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            L.forward(x, o, torch.cuda.current_stream())
        graphs.append(g)
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(W):
            graphs[i % R].replay()
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clk = ClockSampler(local) if rank == 0 else None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(K):
            graphs[i % R].replay()
        e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    clocks = clk.stop() if clk else None
    barrier(world)
    ms_local = e0.elapsed_time(e1)
    value, ms = whole_job(ms_local, w.T, K, world)
    assert B.moe_last_device_error(stream) == 0

    result = None
    if rank == 0:
        # the dispatched rows and expert offsets of this batch, through the
        # route and permute calls (the routing statistics come from the GPU path)
        ids = torch.empty((w.T, w.k), dtype=torch.int32, device=dev)
        tw = torch.empty((w.T, w.k), dtype=torch.float32, device=dev)
        rb = B.moe_route_workspace_bytes(w.T, w.H, w.E)
        pb = B.moe_permute_workspace_bytes(w.T, w.E)
        rws = torch.empty(max(rb, pb, 256), dtype=torch.uint8, device=dev)
        offs = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        st = torch.empty(w.T * w.k, dtype=torch.int32, device=dev)
        inv = torch.empty(w.T * w.k, dtype=torch.int32, device=dev)
        xperm = torch.empty((w.T * w.k, w.H), dtype=torch.bfloat16, device=dev)
        B.moe_route(x, base.tensors[0], base.tensors[1], w.T, w.H, w.E, w.k, ids, tw, rws, rb, stream)
        B.moe_permute(ids, x, w.T, w.H, w.E, w.k, offs, st, inv, xperm, rws, pb, stream)
        stream.synchronize()
        nonempty = int((offs[1:] - offs[:-1] > 0).sum().item())
        lbytes, lflops = layer_units(w, nonempty)
        pk, pk_src = peaks()
        step_s = ms / 1e3 / K
        hbm = pk["hbm_gbs"] * 1e9
        tc = pk["bf16_tflops_sustained"] * 1e12
        t_roof = max(lbytes / hbm, lflops / tc)
        layer_roof = {"bytes": lbytes, "flops": lflops, "nonempty_experts": nonempty,
                      "roofline_us": t_roof * 1e6, "step_us": step_s * 1e6, "frac": t_roof / step_s,
                      "bound": "hbm" if lbytes / hbm >= lflops / tc else "tensor",
                      "peaks": f"{pk_src}: {pk['hbm_gbs']} GB/s, {pk['bf16_tflops_sustained']} TFLOP/s sustained"}

        # dominant kernel: the routed gate_up GroupedMatmul, timed alone on the
        # layer's own dispatched rows, back to back in one graph over the weight copies
        h = torch.empty((w.T * w.k, w.I), dtype=torch.bfloat16, device=dev)
        gb_ws = B.moe_grouped_gemm_workspace_bytes(w.E, w.T * w.k, w.I, w.H, 1)
        g_ws = torch.zeros(max(gb_ws, 256), dtype=torch.uint8, device=dev)
        M = max(20, min(400, K))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cs = torch.cuda.current_stream()
            for i in range(M):
                B.moe_grouped_gemm(xperm, layers[i % R].tensors[2], offs, w.E, w.T * w.k, w.I, w.H, 1, h, g_ws,
                                   gb_ws, cs)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        assert B.moe_last_device_error(stream) == 0
        k_us = e0.elapsed_time(e1) * 1e3 / M
        gb, gf = gate_up_units(w, nonempty)
        if w.T * w.k <= 64 * w.E:     # weights-on-M form: weight streaming, HBM-bound
            achieved = gb / (k_us * 1e-6) / 1e9
            roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / pk["hbm_gbs"]}
        else:
            achieved = gf / (k_us * 1e-6) / 1e12
            roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / pk["bf16_tflops"]}
        roof.update({"traffic": _traffic(w), "kernel": "grouped_gemm gate_up+SiLU*mul", "us_per_launch": k_us,
                     "algorithmic_bytes": gb, "algorithmic_flops": gf, "peak_source": pk_src + " (burst)"})

        # end to end through the public call: pinned host x -> device, forward, out -> pinned host
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
        e2e = {"value": w.T / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": w.T * w.H * 2,
               "d2h_bytes_per_step": w.T * w.H * 2, "ms_per_step": e2e_ms,
               "path": "MoEFFN.forward (one moe_forward call), no graph"}

        cpu = None
        if not args.no_cpu_baseline:
            tps, cores, ntok, el = time_oracle(w, inp, args.cpu_budget)
            cpu = {"value": tps, "unit": UNIT, "cores": round(cores, 2), "kind": "oracle",
                   "sample": f"{ntok} tokens of the same workload through the float64 oracle, token batches "
                             f"of {min(w.T, 8) if w.T > 16 else w.T}, {el:.1f} s wall; cores = CPU time / wall time "
                             f"(numpy BLAS pool of {os.cpu_count()} threads)"}

        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded; workload shapes and distributions)",
            "config": {"workload": f"{w.name.split('@')[0]} T={w.T}", "T": w.T, "H": w.H, "E": w.E, "k": w.k,
                       "I": w.I, "I_s": w.Is, "routing": _routing_desc(w), "parallelism": f"replicas x{world}",
                       "l2": f"expert weights rotate over {R} device copies ({R} x {touched / 1e6:.0f} MB touched "
                             f">= 4 x L2); one CUDA graph per copy, replayed back to back"},
            "clocks": clocks, "e2e": e2e, "gpu_launches": K * launches, "launches_per_step": launches,
            "roofline": roof, "layer_roofline": layer_roof, "cpu_baseline": cpu,
        }
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def _routing_desc(w):
    if w.zipf_s is None and not w.n_empty:
        return f"router W ~ N(0,{w.sigma_router}), near-uniform"
    s = f"router W ~ N(0,{w.sigma_router}) + Zipf(s={w.zipf_s}) log-rank bias"
    return s + (f", {w.n_empty} experts forced empty" if w.n_empty else "")


def _traffic(w):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    capture of the same kernel source, else None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    src = os.path.join(ROOT, "moe_ffn_layer_gb300", "csrc", "grouped_gemm.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    d = json.load(open(p))
    e = d.get(f"{w.name.split('@')[0]}@T{w.T}")
    if not e or e.get("source_sha") != h:
        return None
    return e.get("dram_bytes_per_launch")


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
            "data": "synthetic (seeded; workload shapes and distributions)",
            "config": {"workload": f"{w.name.split('@')[0]} T={w.T}", "T": w.T, "H": w.H, "E": w.E, "k": w.k,
                       "I": w.I, "I_s": w.Is, "routing": _routing_desc(w)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": round(cores, 2), "kind": "oracle",
                             "sample": f"{n} random tokens of the workload per step through the float64 oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


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
    ap.add_argument("--copies", type=int, default=0, help="weight copies to rotate over (0: enough to defeat L2)")
    args = ap.parse_args()
    from moe_ffn_layer_gb300 import synth
    T = args.T if args.T is not None else (8 if args.workload == "decode" else None)
    w = synth.workload(args.workload, T)
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload] if args.impl == "own" else 20
    args.warmup = max(args.warmup, 3)
    res = run_reference(args, w) if args.impl == "reference" else run_gpu(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
