"""Pins of the CPU oracle against facts that do not come from the oracle itself:
a hand-derived closed-form example, brute-force fp64 top-k, the full-softmax
closed form, numpy's stable argsort, torch's dense SwiGLU, a brute-force dense
evaluation of every expert on every token, and invariants of the layer."""
import json
import math
import os

import numpy as np
import pytest
import torch

from moe_ffn_layer_gb300 import synth
from oracle import moe_oracle as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small_inputs(T=12, H=64, E=6, k=2, I=32, Is=48, seed=3, bias=False):
    w = synth.Workload("t", T, H, E, k, I, Is, sigma_router=0.3,
                       zipf_s=1.0 if bias else None, sigma_w=0.1)
    return w, synth.make_inputs(w, seed)


# ---------------------------------------------------------------- closed form

def _closed_form_inputs():
    g = json.load(open(os.path.join(GOLDEN, "closed_form.json")))
    val = {"ln3": math.log(3.0), "ln2": math.log(2.0)}
    wr = np.array([[val.get(v, v) if isinstance(v, str) else v for v in row]
                   for row in g["w_router"]], dtype=np.float32)
    b = lambda a: synth.f32_to_bf16_bits(np.array(a, dtype=np.float32))
    inp = dict(x=b(g["x"]), w_router=wr, bias=None, w_gate_up=b(g["w_gate_up"]),
               w_down=b(g["w_down"]), ws_gate_up=b(g["ws_gate_up"]), ws_down=b(g["ws_down"]))
    return g, inp


def test_closed_form_example():
    g, inp = _closed_form_inputs()
    r = om.forward(inp, k=2)
    np.testing.assert_array_equal(r["ids"], g["ids"])
    np.testing.assert_allclose(r["w"], g["weights"], rtol=0, atol=1e-6)
    np.testing.assert_array_equal(r["offsets"], g["offsets"])
    np.testing.assert_array_equal(r["sorted_token"], g["sorted_token"])
    np.testing.assert_array_equal(r["inv_perm"], g["inv_perm"])
    e = math.e
    s1, s2 = e / (e + 1), e * e / (e * e + 1)          # sigma(1), sigma(2)
    y00 = np.array([2 * s1, -2 * s1])
    y10 = -(1 - s1) * np.array([0.5, 2.0])
    y11 = 2 * s1 * np.array([0.5, 2.0])
    y21 = -2 * s2 * np.array([3.0, 1.0])
    sh0 = np.array([s1, s1])
    sh1 = np.array([2 * s2, 2 * s2])
    out0 = 0.75 * y00 + 0.25 * y10 + sh0
    out1 = 0.8 * y11 + 0.2 * y21 + sh1
    np.testing.assert_allclose(r["out"], np.stack([out0, out1]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(r["s"], np.stack([sh0, sh1]), rtol=0, atol=1e-12)
    # the per-token evaluation reaches the same numbers
    rt = om.forward_tokens(inp, 2, [1, 0])
    np.testing.assert_allclose(rt["out"], np.stack([out1, out0]), rtol=0, atol=1e-6)


# ---------------------------------------------------------------- router

@pytest.mark.parametrize("bias", [False, True])
def test_route_brute_force_topk(bias):
    w, inp = _small_inputs(bias=bias)
    ids, wts, l = om.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    x = om.bf16_to_f64(inp["x"])
    for t in range(w.T):
        # fp64 logits, full sort by (-logit, id): brute force
        lt = [sum(x[t, h] * float(inp["w_router"][e, h]) for h in range(w.H))
              + (float(inp["bias"][e]) if bias else 0.0) for e in range(w.E)]
        best = sorted(range(w.E), key=lambda e: (-lt[e], e))[: w.k]
        assert list(ids[t]) == sorted(best)
        assert abs(l[t] - np.array(lt)).max() < 1e-4


def test_route_full_softmax_closed_form():
    """softmax over all E, restricted to the chosen k and renormalised, equals the
    oracle's softmax over the k chosen logits (torch.softmax as the library)."""
    w, inp = _small_inputs(bias=True)
    ids, wts, l = om.route(inp["x"], inp["w_router"], inp["bias"], w.k)
    p = torch.softmax(torch.from_numpy(l.astype(np.float64)), dim=1).numpy()
    for t in range(w.T):
        q = p[t, ids[t]]
        np.testing.assert_allclose(wts[t], q / q.sum(), rtol=1e-12, atol=1e-15)
    assert np.all(wts > 0)
    np.testing.assert_allclose(wts.sum(1), 1.0, atol=1e-12)
    assert np.all(np.diff(ids, axis=1) > 0)   # distinct, ascending
    assert ids.min() >= 0 and ids.max() < w.E


def test_route_bias_decides_selection():
    """A large bias on one expert puts it in every token's top-k; a -inf bias keeps
    an expert out: the bias enters the selection."""
    w, inp = _small_inputs()
    b = np.zeros(w.E, dtype=np.float32)
    b[4] = 100.0
    b[1] = -np.inf
    ids, wts, _ = om.route(inp["x"], inp["w_router"], b, w.k)
    assert np.all((ids == 4).any(1))
    assert not np.any(ids == 1)
    # and into the weights: expert 4 takes nearly all of each token's weight
    assert np.all(wts[ids == 4] > 0.999)


def test_route_matches_torch_topk():
    w = synth.workload("decode", 8)
    x, wr, b = synth.make_activations(w)
    ids, wts, l = om.route(x, wr, b, w.k)
    l64 = torch.from_numpy(om.bf16_to_f64(x)) @ torch.from_numpy(wr.astype(np.float64)).T
    top = torch.topk(l64, w.k, dim=1).indices.sort(dim=1).values.numpy()
    np.testing.assert_array_equal(ids, top)


# ---------------------------------------------------------------- permute

@pytest.mark.parametrize("name,T", [("tiny", 16), ("batched_decode", 256)])
def test_permute_matches_stable_argsort(name, T):
    w = synth.workload(name, T)
    x, wr, b = synth.make_activations(w)
    ids, _, _ = om.route(x, wr, b, w.k)
    off, st, inv = om.permute(ids, w.E)
    key = ids.astype(np.int64) * w.T + np.arange(w.T)[:, None]
    order = np.argsort(key.ravel(), kind="stable")          # pair index t*k+j per row
    np.testing.assert_array_equal(st, order // w.k)
    np.testing.assert_array_equal(inv[order], np.arange(w.T * w.k))
    counts = np.bincount(ids.ravel(), minlength=w.E)
    assert counts.sum() == w.T * w.k
    np.testing.assert_array_equal(np.diff(off), counts)
    assert off[0] == 0 and off[-1] == w.T * w.k
    np.testing.assert_array_equal(np.sort(inv), np.arange(w.T * w.k))   # bijection
    np.testing.assert_array_equal(st[inv], np.repeat(np.arange(w.T), w.k))


def test_permute_handles_empty_experts():
    ids = np.array([[0, 3], [3, 5], [0, 5]], dtype=np.int32)
    off, st, inv = om.permute(ids, 7)
    np.testing.assert_array_equal(off, [0, 2, 2, 2, 4, 4, 6, 6])
    np.testing.assert_array_equal(st, [0, 2, 0, 1, 1, 2])
    np.testing.assert_array_equal(inv, [0, 2, 3, 4, 1, 5])


# ---------------------------------------------------------------- expert MLP

def _torch_swiglu(x, wgu, wd):
    n = wgu.shape[0] // 2
    return (torch.nn.functional.silu(x @ wgu[:n].T) * (x @ wgu[n:].T)) @ wd.T


def test_single_expert_is_dense_swiglu():
    """E=1, k=1: the layer is one SwiGLU MLP plus the shared one (torch CPU fp64)."""
    w = synth.Workload("t", 10, 64, 1, 1, 32, 16, sigma_router=0.1, sigma_w=0.1)
    inp = synth.make_inputs(w, 5)
    r = om.forward(inp, 1)
    f = lambda a: torch.from_numpy(om.bf16_to_f64(a))
    x = f(inp["x"])
    ref = _torch_swiglu(x, f(inp["w_gate_up"][0]), f(inp["w_down"][0])) + \
        _torch_swiglu(x, f(inp["ws_gate_up"]), f(inp["ws_down"]))
    np.testing.assert_allclose(r["w"], 1.0)
    np.testing.assert_allclose(r["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bias", [False, True])
def test_brute_force_dense_layer(bias):
    """Every expert on every token (torch fp64), masked by the routing weights from
    torch.topk + torch.softmax, plus the shared expert."""
    w, inp = _small_inputs(T=20, E=8, k=3, bias=bias)
    r = om.forward(inp, w.k)
    f = lambda a: torch.from_numpy(om.bf16_to_f64(a))
    x = f(inp["x"])
    l = torch.from_numpy(om.router_logits(inp["x"], inp["w_router"], inp["bias"]).astype(np.float64))
    top = torch.topk(l, w.k, dim=1).indices
    p = torch.softmax(l, dim=1)
    mask = torch.zeros_like(p).scatter_(1, top, 1.0)
    wdense = p * mask / (p * mask).sum(1, keepdim=True)
    out = _torch_swiglu(x, f(inp["ws_gate_up"]), f(inp["ws_down"]))
    for e in range(w.E):
        out = out + wdense[:, e:e + 1] * _torch_swiglu(x, f(inp["w_gate_up"][e]), f(inp["w_down"][e]))
    np.testing.assert_allclose(r["out"], out.numpy(), rtol=1e-10, atol=1e-12)
    # per-token evaluation agrees with the permuted evaluation
    rt = om.forward_tokens(inp, w.k, np.arange(w.T))
    np.testing.assert_allclose(rt["out"], r["out"], rtol=1e-12, atol=1e-13)


def test_identical_experts_invariant():
    """All experts equal: routed part = MLP(x) because each token's weights sum to 1."""
    w, inp = _small_inputs(E=5, k=3)
    inp["w_gate_up"][:] = inp["w_gate_up"][0]
    inp["w_down"][:] = inp["w_down"][0]
    inp["ws_gate_up"] = None
    inp["ws_down"] = None
    r = om.forward(inp, w.k)
    f = lambda a: torch.from_numpy(om.bf16_to_f64(a))
    ref = _torch_swiglu(f(inp["x"]), f(inp["w_gate_up"][0]), f(inp["w_down"][0]))
    np.testing.assert_allclose(r["out"], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_linear_in_down_weights_and_shared_zero():
    w, inp = _small_inputs()
    base = om.forward(inp, w.k)
    inp2 = dict(inp)
    inp2["w_down"] = synth.f32_to_bf16_bits(2 * om.bf16_to_f32(inp["w_down"]))  # exact in bf16
    inp2["ws_down"] = np.zeros_like(inp["ws_down"])
    r2 = om.forward(inp2, w.k)
    routed = base["out"] - base["s"]
    np.testing.assert_allclose(r2["out"], 2 * routed, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(r2["s"], 0)


def test_silu_special_values():
    v = np.array([0.0, 1.0, -1.0, 50.0, -800.0])
    s = om.silu(v)
    np.testing.assert_allclose(s[:3], [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e)], atol=1e-15)
    assert abs(s[3] - 50.0) < 1e-12 and s[4] == 0.0


def test_grouped_gemm_definition():
    rng = np.random.default_rng(1)
    a = synth.f32_to_bf16_bits(rng.standard_normal((9, 16)).astype(np.float32))
    wt = synth.f32_to_bf16_bits(rng.standard_normal((3, 8, 16)).astype(np.float32))
    off = np.array([0, 4, 4, 9])
    out = om.grouped_gemm(a, wt, off, 0)
    A, W = om.bf16_to_f64(a), om.bf16_to_f64(wt)
    for r in range(9):
        g = 0 if r < 4 else 2
        np.testing.assert_allclose(out[r], [sum(A[r, c] * W[g, n, c] for c in range(16)) for n in range(8)],
                                   rtol=1e-12, atol=1e-12)
    out1 = om.grouped_gemm(a, wt, off, 1)
    gate, up = A[:4] @ W[0, :4].T, A[:4] @ W[0, 4:].T
    np.testing.assert_allclose(out1[:4], gate * torch.sigmoid(torch.from_numpy(gate)).numpy() * up, rtol=1e-12)


# ---------------------------------------------------------------- FP8 expert weights

def test_e4m3_decoding_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = om.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.nonzero(nan)[0], [0x7F, 0xFF])
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # the format's landmarks: smallest subnormal, smallest normal, largest finite
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x7E] == 448.0 and got[0xFE] == -448.0


def test_w8_layer_equals_bf16_layer_on_exactly_representable_weights():
    """When every bf16 weight is an e4m3 value times a power-of-two row scale,
    the FP8 layer (codes and scales) and the bf16 layer are the same layer."""
    w = synth.Workload("w8", 9, 64, 6, 2, 32, 48, sigma_router=0.3)
    inp = synth.make_inputs(w, 5)
    rng = np.random.default_rng(6)
    vals = om.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    def rows(shape):
        codes = rng.integers(0, 0x7F, size=shape).astype(np.uint8) | (rng.integers(0, 2, size=shape) << 7).astype(np.uint8)
        scale = np.exp2(rng.integers(-12, -6, size=shape[:-1])).astype(np.float32)
        dense = (om.e4m3_to_f64(codes) * scale[..., None]).astype(np.float32)
        bits = synth.f32_to_bf16_bits(dense)
        assert np.array_equal(om.bf16_to_f64(bits), om.e4m3_to_f64(codes) * scale[..., None])   # exact in bf16
        return codes, scale, bits
    cgu, sgu, bgu = rows((w.E, 2 * w.I, w.H))
    cd, sd, bd = rows((w.E, w.H, w.I))
    inp_bf16 = dict(inp, w_gate_up=bgu, w_down=bd)
    inp_w8 = dict(inp, w_gate_up=cgu, w_gate_up_scale=sgu, w_down=cd, w_down_scale=sd)
    a, b = om.forward(inp_bf16, w.k), om.forward(inp_w8, w.k)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["h"], b["h"])
    t = np.array([0, 4, 8])
    assert np.array_equal(om.forward_tokens(inp_w8, w.k, t)["out"], om.forward_tokens(inp_bf16, w.k, t)["out"])
    off = a["offsets"]
    xp = inp["x"][a["sorted_token"]]
    assert np.array_equal(om.grouped_gemm(xp, cgu, off, 1, w_scale=sgu), om.grouped_gemm(xp, bgu, off, 1))


def test_w8_brute_force_dense_layer():
    """FP8 layer against a dense evaluation of every expert on every token
    (torch, float64 dequantised weights) masked by the routing weights."""
    w = synth.Workload("w8d", 10, 64, 6, 2, 32, 48, sigma_router=0.3)
    inp = synth.make_inputs_w8(w, 7)
    r = om.forward(inp, w.k)
    x = torch.from_numpy(om.bf16_to_f64(inp["x"]))
    dense = torch.zeros((w.T, w.H), dtype=torch.float64)
    for e in range(w.E):
        wgu = torch.from_numpy(om.dequant_w8(inp["w_gate_up"][e], inp["w_gate_up_scale"][e]))
        wd = torch.from_numpy(om.dequant_w8(inp["w_down"][e], inp["w_down_scale"][e]))
        y = (torch.nn.functional.silu(x @ wgu[:w.I].T) * (x @ wgu[w.I:].T)) @ wd.T
        mask = torch.zeros(w.T, dtype=torch.float64)
        for t in range(w.T):
            for j in range(w.k):
                if r["ids"][t, j] == e:
                    mask[t] = r["w"][t, j]
        dense += mask[:, None] * y
    sgu, sd = (torch.from_numpy(om.bf16_to_f64(a)) for a in (inp["ws_gate_up"], inp["ws_down"]))
    dense += (torch.nn.functional.silu(x @ sgu[:w.Is].T) * (x @ sgu[w.Is:].T)) @ sd.T
    np.testing.assert_allclose(r["out"], dense.numpy(), rtol=1e-10, atol=1e-12)
