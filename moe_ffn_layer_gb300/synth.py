"""Seeded synthetic inputs for the MoE FFN layer forward.

This module only draws numbers: hidden states, router weights, router bias and
expert weights, rounded to the storage types the layer reads (bf16 stored as
uint16 bit patterns, fp32 router; for the FP8 layer, e4m3 codes with one fp32
scale per weight row, the storage format of the weights).  It computes nothing of the layer itself.
The one place where it looks at the router is the near-tie guard: a token whose
k-th and (k+1)-th router logits lie closer than ``GAP`` gets its hidden row
redrawn, so that the choice of experts does not hinge on the summation order
of an fp32 dot product.  That guard evaluates the logits with a numpy float64
matrix product (a library primitive), on the exact values both sides read.

Workloads (``WORKLOADS``) follow the layer shapes of the MoE serving setting:
hidden size 2048 for the decode/prefill shapes (the size of the MoE model's
hidden state in "Ascend 910C LLM inference optimisation, part 2" (Dewu Tech),
section on the fused o_proj + AllReduce + RMSNorm operator), and E, k, I, I_s,
value distributions and routing skew as the benchmark shapes define them.

Stream layout (each stream is ``numpy.random.default_rng([seed, tag, sub])``):
tag 0 hidden x, 1 router W, 2 Zipf rank permutation, 3 forced-empty experts,
4 gate_up of expert e (sub=e), 5 down of expert e (sub=e), 6 shared gate_up,
7 shared down, 1000+t redraw attempt a of hidden row t (sub=a).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np

GAP = 1e-4  # minimum k-th vs (k+1)-th router logit gap (fp64) after the guard


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    Is: int
    sigma_router: float
    zipf_s: Optional[float] = None   # bias_e = -s * ln(rank_e)
    n_empty: int = 0                 # experts whose bias is -inf
    sigma_x: float = 1.0
    sigma_w: float = 0.02

    def with_T(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")


WORKLOADS = {
    # tiny layer: T=16, H=256, E=8, k=2, I=128, one shared expert I_s=256
    "tiny": Workload("tiny", 16, 256, 8, 2, 128, 256, sigma_router=0.1),
    # decode, c=1..8: near-uniform routing
    "decode": Workload("decode", 8, 2048, 128, 8, 768, 2048, sigma_router=0.02),
    # batched decode: Zipf(1.1) log-rank router bias
    "batched_decode": Workload("batched_decode", 256, 2048, 128, 8, 768, 2048,
                               sigma_router=0.02, zipf_s=1.1),
    # prefill: uniform routing, ~512 rows per expert
    "prefill": Workload("prefill", 8192, 2048, 128, 8, 768, 2048, sigma_router=0.02),
    # large prefill: Zipf(1.2) bias, 8 forced-empty experts, one hot expert
    "large_prefill": Workload("large_prefill", 16384, 4096, 256, 8, 1024, 4096,
                              sigma_router=0.02, zipf_s=1.2, n_empty=8),
    # the decode shapes with FP8 (e4m3, per-row scales) routed expert weights
    # (make_inputs_w8 / make_expert_weights_w8 draw them)
    "decode_w8": Workload("decode_w8", 8, 2048, 128, 8, 768, 2048, sigma_router=0.02),
    "batched_decode_w8": Workload("batched_decode_w8", 256, 2048, 128, 8, 768, 2048,
                                  sigma_router=0.02, zipf_s=1.1),
}

# every (workload, T) the parity tests cover at full size
FULL_SHAPES = [("tiny", 16), ("decode", 1), ("decode", 4), ("decode", 8),
               ("batched_decode", 64), ("batched_decode", 256),
               ("prefill", 8192), ("large_prefill", 16384)]


def workload(name: str, T: Optional[int] = None) -> Workload:
    w = WORKLOADS[name]
    return w.with_T(T) if T is not None and T != w.T else w


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + r) >> 16).astype(np.uint16)


# the 127 non-negative finite e4m3 values, ascending (code = index): exponent
# field e (bias 7) and mantissa m; e = 0 holds m * 2^-9
_E4M3_POS = np.array([(m * 2.0 ** -9) if (c >> 3) == 0 else (1 + m / 8.0) * 2.0 ** ((c >> 3) - 7)
                      for c in range(127) for m in [c & 7]], dtype=np.float64)


def f32_to_e4m3(v: np.ndarray) -> np.ndarray:
    """Round float32 values to e4m3 codes (uint8), to nearest, ties to the even
    code, magnitudes above 448 saturating to 448."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 126)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a == _E4M3_POS[hi], hi, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def quantize_rows_e4m3(w: np.ndarray):
    """Per-row (output channel) e4m3 quantisation of float32 weights [..., K]:
    scale = max|row| / 448 (fp32; 1 for an all-zero row), codes = e4m3(w /
    scale).  Returns (codes uint8 [..., K], scale float32 [...])."""
    w = np.asarray(w, dtype=np.float32)
    amax = np.abs(w).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    return f32_to_e4m3(w / scale[..., None]), scale


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, tag: int, sub: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, tag, sub])


def _normal_bf16(rng: np.random.Generator, shape, sigma: float, out: np.ndarray) -> None:
    v = rng.standard_normal(shape, dtype=np.float32)
    v *= np.float32(sigma)
    out[...] = f32_to_bf16_bits(v)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def router_bias(w: Workload, seed: int) -> Optional[np.ndarray]:
    """Per-expert fp32 router bias: -s*ln(rank) with a seeded rank permutation,
    and -inf on ``n_empty`` seeded experts; None when the workload has none."""
    if w.zipf_s is None and w.n_empty == 0:
        return None
    b = np.zeros(w.E, dtype=np.float64)
    if w.zipf_s is not None:
        ranks = _rng(seed, 2).permutation(w.E) + 1
        b = -w.zipf_s * np.log(ranks.astype(np.float64))
    if w.n_empty:
        empty = _rng(seed, 3).choice(w.E, size=w.n_empty, replace=False)
        b[empty] = -np.inf
    return b.astype(np.float32)


def _kth_gap(x_bits: np.ndarray, wr: np.ndarray, b: Optional[np.ndarray], k: int) -> np.ndarray:
    """fp64 gap between the k-th and (k+1)-th largest router logit of each row."""
    l = bf16_bits_to_f32(x_bits).astype(np.float64) @ wr.astype(np.float64).T
    if b is not None:
        l = l + b.astype(np.float64)
    part = -np.partition(-l, k, axis=1)[:, : k + 1]
    part.sort(axis=1)
    return part[:, 1] - part[:, 0]  # (k-th largest) - ((k+1)-th largest)


def make_activations(w: Workload, seed: int = 0):
    """Hidden states x (bf16 bits [T,H]), router W (fp32 [E,H]), bias (fp32 [E] or None),
    with the near-tie guard applied row by row."""
    x = np.empty((w.T, w.H), dtype=np.uint16)
    _normal_bf16(_rng(seed, 0), (w.T, w.H), w.sigma_x, x)
    wr = (_rng(seed, 1).standard_normal((w.E, w.H), dtype=np.float32)
          * np.float32(w.sigma_router)).astype(np.float32)
    b = router_bias(w, seed)
    if w.k < w.E:
        bad = np.nonzero(_kth_gap(x, wr, b, w.k) <= GAP)[0]
        for t in bad:
            for a in range(1000):
                row = np.empty((1, w.H), dtype=np.uint16)
                _normal_bf16(_rng(seed, 1000 + int(t), a), (1, w.H), w.sigma_x, row)
                if _kth_gap(row, wr, b, w.k)[0] > GAP:
                    x[t] = row[0]
                    break
            else:
                raise RuntimeError(f"near-tie guard: no redraw of row {t} cleared the gap")
    return x, wr, b


def make_expert_weights(w: Workload, seed: int = 0):
    """Routed expert weights: gate_up bf16 [E][2I][H] (rows 0..I-1 gate, I..2I-1 up)
    and down bf16 [E][H][I]; one seeded stream per expert, filled in parallel."""
    wgu = np.empty((w.E, 2 * w.I, w.H), dtype=np.uint16)
    wd = np.empty((w.E, w.H, w.I), dtype=np.uint16)

    def fill(e):
        _normal_bf16(_rng(seed, 4, e), (2 * w.I, w.H), w.sigma_w, wgu[e])
        _normal_bf16(_rng(seed, 5, e), (w.H, w.I), w.sigma_w, wd[e])

    with _cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(w.E)))
    return wgu, wd


def make_expert_weights_w8(w: Workload, seed: int = 0):
    """Routed expert weights in e4m3 with one fp32 scale per output row: the
    same fp32 draws as make_expert_weights, quantised row by row.  Returns
    (gate_up codes [E][2I][H], gate_up scales [E][2I], down codes [E][H][I],
    down scales [E][H])."""
    wgu = np.empty((w.E, 2 * w.I, w.H), dtype=np.uint8)
    sgu = np.empty((w.E, 2 * w.I), dtype=np.float32)
    wd = np.empty((w.E, w.H, w.I), dtype=np.uint8)
    sd = np.empty((w.E, w.H), dtype=np.float32)

    def fill(e):
        g = _rng(seed, 4, e).standard_normal((2 * w.I, w.H), dtype=np.float32) * np.float32(w.sigma_w)
        wgu[e], sgu[e] = quantize_rows_e4m3(g)
        d = _rng(seed, 5, e).standard_normal((w.H, w.I), dtype=np.float32) * np.float32(w.sigma_w)
        wd[e], sd[e] = quantize_rows_e4m3(d)

    with _cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(fill, range(w.E)))
    return wgu, sgu, wd, sd


def make_inputs_w8(w: Workload, seed: int = 0) -> dict:
    """All inputs of one layer forward with e4m3 routed expert weights (keys
    w_gate_up / w_down hold codes, w_gate_up_scale / w_down_scale the row
    scales); x, the router and the bf16 shared expert as make_inputs."""
    x, wr, b = make_activations(w, seed)
    wgu, sgu, wd, sd = make_expert_weights_w8(w, seed)
    shg, shd = make_shared_weights(w, seed)
    return dict(x=x, w_router=wr, bias=b, w_gate_up=wgu, w_gate_up_scale=sgu, w_down=wd, w_down_scale=sd,
                ws_gate_up=shg, ws_down=shd)


def make_shared_weights(w: Workload, seed: int = 0):
    """Shared expert: gate_up bf16 [2I_s][H], down bf16 [H][I_s] (None when I_s == 0)."""
    if w.Is == 0:
        return None, None
    sgu = np.empty((2 * w.Is, w.H), dtype=np.uint16)
    sd = np.empty((w.H, w.Is), dtype=np.uint16)
    _normal_bf16(_rng(seed, 6), sgu.shape, w.sigma_w, sgu)
    _normal_bf16(_rng(seed, 7), sd.shape, w.sigma_w, sd)
    return sgu, sd


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """All inputs of one layer forward as numpy arrays (bf16 as uint16 bits)."""
    x, wr, b = make_activations(w, seed)
    wgu, wd = make_expert_weights(w, seed)
    sgu, sd = make_shared_weights(w, seed)
    return dict(x=x, w_router=wr, bias=b, w_gate_up=wgu, w_down=wd,
                ws_gate_up=sgu, ws_down=sd)


def random_bf16(shape, seed: int, tag: int = 50, sigma: float = 1.0) -> np.ndarray:
    """Plain seeded N(0, sigma) bf16 bits, for operand-level tests."""
    out = np.empty(shape, dtype=np.uint16)
    _normal_bf16(_rng(seed, tag), shape, sigma, out)
    return out
