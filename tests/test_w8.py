"""FP8 (e4m3) routed expert weights with one fp32 scale per weight row: the
grouped matmul and the layer forward against the float64 oracle on the same
codes and scales (the layer's tolerances), at every decode-sized workload, with
ragged groups, split-K and one-row groups; graph replay and repeat bits."""
import functools

import numpy as np
import pytest
import torch

from cases import assert_close_layer, to_f64
from moe_ffn_layer_gb300 import binding as B
from moe_ffn_layer_gb300 import build as build_mod
from moe_ffn_layer_gb300 import synth
from moe_ffn_layer_gb300.layer import MoEFFN, bf16_tensor
from oracle import moe_oracle as om

pytestmark = pytest.mark.gpu

W8_SHAPES = [("decode", 1), ("decode", 4), ("decode", 8), ("decode", 16), ("batched_decode", 64),
             ("batched_decode", 256)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield B.lib()
    torch.cuda.synchronize()


def stream():
    return torch.cuda.current_stream()


def no_device_error():
    assert B.moe_last_device_error(stream()) == 0


def u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


GEMM_CASES = [
    ([1, 0, 3, 16, 17, 64, 0, 2], 256, 128, 0),
    ([1, 0, 3, 16, 17, 64, 0, 2], 128, 192, 1),
    ([1, 0, 3, 16, 2, 0, 9, 1], 256, 512, 1),           # every group <= 16 rows: split-K applies
    ([1, 0, 3, 16, 2, 0, 9, 1], 384, 2048, 0),
    ([1] * 8 + [0] * 100 + [2, 16], 768, 2048, 1),      # decode-like gate_up
    ([1] * 8 + [0] * 100 + [2, 16], 2048, 768, 0),      # decode-like down
    ([100, 0, 5, 200, 1, 63, 65, 0], 384, 256, 1),      # groups over one 64-row chunk
    ([5], 2048, 768, 0),
    # stages pair the 64-wide K blocks: one block, and an odd count (the last stage half full)
    ([1, 0, 3, 16, 2, 0, 9, 1], 256, 64, 1),
    ([1, 0, 3, 16, 2, 0, 9, 1], 384, 320, 0),
    ([7, 64, 1, 0, 33], 128, 320, 1),
]


@pytest.mark.parametrize("use_ws", [False, True])
@pytest.mark.parametrize("rows,N,K,act", GEMM_CASES)
def test_grouped_gemm_w8(rows, N, K, act, use_ws):
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    rows_max = R + 3
    a_bits = synth.random_bf16((rows_max, K), seed=R + N, tag=91)
    wf = (np.random.default_rng(K + G).standard_normal((G, 2 * N if act else N, K)) * 0.05).astype(np.float32)
    codes, scale = synth.quantize_rows_e4m3(wf)
    ref = om.grouped_gemm(a_bits, codes, off, act, w_scale=scale)
    nb = B.moe_grouped_gemm_workspace_bytes(G, rows_max, N, K, act)
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda") if use_ws else None
    out = torch.full((rows_max, N), 1024.0, dtype=torch.bfloat16, device="cuda")
    a, w, s = bf16_tensor(a_bits, "cuda"), u8(codes), f32(scale)
    B.moe_grouped_gemm_w8(a, w, s, i32(off), G, rows_max, N, K, act, out, ws, nb if use_ws else 0, stream())
    no_device_error()
    got = to_f64(out)
    assert_close_layer(got[:R], ref[:R], f"w8 gemm rows={rows} N={N} K={K} act={act}")
    assert np.all(got[R:] == 1024.0)
    for r in np.linspace(0, R - 1, min(R, 16)).astype(int):
        scl = np.abs(ref[r]).max() + 1e-6
        assert np.abs(got[r] - ref[r]).max() <= 2e-2 * scl, r
    out2 = torch.full_like(out, 1024.0)
    B.moe_grouped_gemm_w8(a, w, s, i32(off), G, rows_max, N, K, act, out2, ws, nb if use_ws else 0, stream())
    no_device_error()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_grouped_gemm_w8_every_code_exact():
    """Every e4m3 code at every position of the tiles: token rows that are unit
    vectors pick single weights, so with power-of-two scales each output is one
    decoded code times its scale, exact in bf16, and must match bit for bit
    (codes 0x01..0x07 and 0x81..0x87 are the subnormals m * 2^-9)."""
    G, per, N, K = 4, 64, 128, 256
    off = (np.arange(G + 1) * per).astype(np.int32)
    R = G * per
    a = np.zeros((R, K), dtype=np.float32)
    a[np.arange(R), np.arange(R) % K] = 1.0
    a_bits = synth.f32_to_bf16_bits(a)
    n, k = np.meshgrid(np.arange(N), np.arange(K), indexing="ij")
    codes = np.stack([(n * 3 + k + 17 * g) % 256 for g in range(G)]).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00
    scale = np.ldexp(1.0, (np.arange(G * N) % 7) - 3).reshape(G, N).astype(np.float32)
    ref = om.grouped_gemm(a_bits, codes, off, 0, w_scale=scale)
    out = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm_w8(bf16_tensor(a_bits, "cuda"), u8(codes), f32(scale), i32(off), G, R, N, K, 0, out, None, 0,
                          stream())
    no_device_error()
    assert np.array_equal(to_f64(out), ref)
    assert len(np.unique(codes)) == 254


@pytest.mark.parametrize("act,N,K", [(1, 768, 2048), (0, 2048, 768), (1, 256, 512)])
def test_grouped_gemm_w8_one_row_groups(act, N, K):
    """Groups of one row (a token's k experts): the CUDA-core weight stream
    reading 1-byte weights."""
    rows = [1, 0, 1, 1, 0, 1]
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    a_bits = synth.random_bf16((1, K), seed=K, tag=92)
    wf = (np.random.default_rng(N).standard_normal((G, 2 * N if act else N, K)) * 0.05).astype(np.float32)
    codes, scale = synth.quantize_rows_e4m3(wf)
    off1 = np.array([0, 1], dtype=np.int32)
    for g in range(G):
        if rows[g] == 0:
            continue
        ref = om.grouped_gemm(a_bits, codes[g:g + 1], off1, act, w_scale=scale[g:g + 1])
        out = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        B.moe_grouped_gemm_w8(bf16_tensor(a_bits, "cuda"), u8(codes[g:g + 1]), f32(scale[g:g + 1]), None, 1, 1, N, K,
                              act, out, None, 0, stream())
        no_device_error()
        assert_close_layer(to_f64(out), ref, f"w8 one row g={g}")


@functools.lru_cache(maxsize=1)
def _w8_weights(name):
    w = synth.workload(name)
    return synth.make_expert_weights_w8(w, 0) + synth.make_shared_weights(w, 0)


@functools.lru_cache(maxsize=1)
def _w8_layer(name):
    w = synth.workload(name)
    wgu, sgu, wd, sd, shg, shd = _w8_weights(name)
    x, wr, b = synth.make_activations(w, 0)
    inp = dict(x=x, w_router=wr, bias=None, w_gate_up=wgu, w_gate_up_scale=sgu, w_down=wd, w_down_scale=sd,
               ws_gate_up=shg, ws_down=shd)
    return MoEFFN.from_inputs(inp, w.k, "cuda")


def _w8_inputs(name, T):
    w = synth.workload(name, T)
    x, wr, b = synth.make_activations(w, 0)
    wgu, sgu, wd, sd, shg, shd = _w8_weights(name)
    return dict(x=x, w_router=wr, bias=b, w_gate_up=wgu, w_gate_up_scale=sgu, w_down=wd, w_down_scale=sd,
                ws_gate_up=shg, ws_down=shd)


@pytest.mark.parametrize("name,T", W8_SHAPES)
def test_forward_w8(name, T):
    """Every output element of the FP8 layer against the oracle on the same
    codes and scales."""
    w = synth.workload(name, T)
    inp = _w8_inputs(name, T)
    ref = om.forward(inp, w.k)
    base = _w8_layer("decode")      # decode and batched decode share the expert weights
    b = None if inp["bias"] is None else f32(inp["bias"])
    L = MoEFFN(w.k, base.tensors[0], b, base.tensors[2], base.tensors[3], base.tensors[4], base.tensors[5],
               base.scales[0], base.scales[1])
    x = bf16_tensor(inp["x"], "cuda")
    out = L.forward(x).clone()
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"w8 {name} T={T}")
    again = L.forward(x)
    no_device_error()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    # the same forward captured in a CUDA graph and replayed
    g = torch.cuda.CUDAGraph()
    o = torch.zeros_like(out)
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        L.forward(x, o, torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(out.view(torch.int16), o.view(torch.int16))


@pytest.mark.parametrize("seed", range(16))
def test_forward_w8_random_shapes(seed):
    """Seeded random layer shapes with e4m3 routed weights, within the sizes the
    8-bit path takes (I and H multiples of 128, T*k <= 64 E): every output
    element against the oracle on the same codes and scales."""
    r = np.random.default_rng(2000 + seed)
    E = int(r.choice([4, 8, 16, 64, 128]))
    k = int(r.integers(1, min(E, 8) + 1))
    T = int(r.choice([t for t in (1, 2, 3, 5, 8, 13, 16, 24, 64, 200) if t * k <= 64 * E]))
    wl = synth.Workload(f"w8random{seed}", T, int(r.choice([128, 256, 512, 1024])), E, k,
                        int(r.choice([128, 256, 512])), int(r.choice([0, 128, 256])), sigma_router=0.1,
                        sigma_w=0.03, zipf_s=1.1 if r.random() < 0.4 else None)
    inp = synth.make_inputs_w8(wl, seed)
    ref = om.forward(inp, k)
    L = MoEFFN.from_inputs(inp, k, "cuda")
    out = L.forward(bf16_tensor(inp["x"], "cuda")).clone()
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"],
                       f"w8 T={T} H={wl.H} E={E} k={k} I={wl.I} I_s={wl.Is} zipf={wl.zipf_s}")


def test_forward_w8_refuses_prefill_sizes():
    base = _w8_layer("decode")
    x = torch.zeros((8192, 2048), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError) as e:
        base.forward(x)
    assert e.value.code == -2
