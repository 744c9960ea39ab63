"""Seeded layer cases shared by the GPU parity tests: the synthetic inputs of a
workload and the oracle's routing of them, cached per process."""
from __future__ import annotations

import functools

import numpy as np
import torch

from moe_ffn_layer_gb300 import synth
from moe_ffn_layer_gb300.layer import MoEFFN, bf16_tensor
from oracle import moe_oracle as om

# Output tolerance of the layer (bf16 output against the float64 oracle).
REL_FRO = 1e-2
MAX_ABS_FRAC = 2e-2
# Router weights: fp32 softmax of fp32 logits whose summation order differs
# from the oracle's by a few fp32 ulps of |l| <~ 4.
ROUTE_W_ATOL = 5e-6
# From 512 tokens on (E, H multiples of 64) the logits come from the tensor
# cores: exact bf16 products, but the tensor core's fp32 accumulation rounds
# less exactly than an FMA chain (measured logit error ~3e-5 at K = 3*2048);
# a weight moves by at most ~0.5 x the logit error.
ROUTE_W_ATOL_TC = 1e-4


def route_w_atol(T: int, H: int, E: int) -> float:
    return ROUTE_W_ATOL_TC if (T >= 512 and E % 64 == 0 and H % 64 == 0) else ROUTE_W_ATOL


@functools.lru_cache(maxsize=1)
def _weights(name: str, seed: int):
    w = synth.workload(name)
    return synth.make_expert_weights(w, seed) + synth.make_shared_weights(w, seed)


@functools.lru_cache(maxsize=4)
def _activations(name: str, T: int, seed: int):
    return synth.make_activations(synth.workload(name, T), seed)


def inputs(name: str, T: int, seed: int = 0) -> dict:
    """synth.make_inputs(workload(name, T), seed), with the expert weights
    (which do not depend on T) drawn once per workload."""
    x, wr, b = _activations(name, T, seed)
    wgu, wd, sgu, sd = _weights(name, seed)
    return dict(x=x, w_router=wr, bias=b, w_gate_up=wgu, w_down=wd, ws_gate_up=sgu, ws_down=sd)


@functools.lru_cache(maxsize=3)
def routing(name: str, T: int, seed: int = 0):
    w = synth.workload(name, T)
    inp = inputs(name, T, seed)
    ids, wts, logits = om.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    off, st, inv = om.permute(ids, w.E)
    return ids, wts, off, st, inv


_layers: dict = {}


def layer(name: str, T: int, seed: int = 0) -> MoEFFN:
    """Device copy of a workload's weights (one layer kept at a time: the
    large prefill layer alone holds 6.4 GB)."""
    wkey = (name, seed)
    if wkey not in _layers:
        _layers.clear()
        torch.cuda.empty_cache()
        w = synth.workload(name, T)
        _layers[wkey] = MoEFFN.from_inputs(inputs(name, T, seed), w.k, "cuda")
    return _layers[wkey]


def x_tensor(name: str, T: int, seed: int = 0) -> torch.Tensor:
    return bf16_tensor(inputs(name, T, seed)["x"], "cuda")


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close_layer(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    """The layer's output tolerance: relative Frobenius error <= 1e-2 and max
    abs error <= 2e-2 * max|ref|."""
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = gpu - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    bound = MAX_ABS_FRAC * np.abs(ref).max() if ref.size else 0.0
    assert rel <= REL_FRO, f"{what}: rel Frobenius error {rel:.3e} > {REL_FRO}"
    assert mx <= bound, f"{what}: max abs error {mx:.3e} > {bound:.3e}"
    return rel, mx
