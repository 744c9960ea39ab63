"""Parity of each C-ABI call of the CUDA path with the CPU oracle, on seeded
inputs, at sizes that span several tiles with ragged tails and at the full
sizes of every workload (sampled rows where the oracle would take too long).

Bars: expert ids, offsets and permutation indices bit-exact; the layer's bf16
output within a relative Frobenius error of 1e-2 and a max abs error of
2e-2 * max|ref| of the float64 oracle."""
import time

import numpy as np
import pytest
import torch

from cases import (assert_close_layer, inputs, layer, route_w_atol, routing, to_f64, x_tensor)
from moe_ffn_layer_gb300 import binding as B
from moe_ffn_layer_gb300 import build as build_mod
from moe_ffn_layer_gb300 import synth
from moe_ffn_layer_gb300.layer import MoEFFN, bf16_tensor
from oracle import moe_oracle as om

# the grouped matmul's scratch keeps its counters in its first 64 KiB (moe_ffn.h)
COUNTER_REGION_BYTES = 64 * 1024

pytestmark = pytest.mark.gpu

SMALL_SHAPES = [s for s in synth.FULL_SHAPES if s[1] <= 256]
# prefill T=8192: the whole output against the oracle; large prefill: sampled rows
FULL_OUTPUT_SHAPES = SMALL_SHAPES + [("prefill", 8192)]
LARGE_SHAPES = [s for s in synth.FULL_SHAPES if s[1] > 8192]


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    L = B.lib()
    yield L
    torch.cuda.synchronize()


def stream():
    return torch.cuda.current_stream()


def no_device_error():
    assert B.moe_last_device_error(stream()) == 0


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


# ---------------------------------------------------------------- a1 route

@pytest.mark.parametrize("name,T", synth.FULL_SHAPES)
def test_route(name, T):
    w = synth.workload(name, T)
    inp = inputs(name, T)
    ids_ref, w_ref, *_ = routing(name, T)
    x = bf16_tensor(inp["x"], "cuda")
    wr = f32(inp["w_router"])
    b = None if inp["bias"] is None else f32(inp["bias"])
    ids = torch.empty((T, w.k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, w.k), dtype=torch.float32, device="cuda")
    nb = B.moe_route_workspace_bytes(T, w.H, w.E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.moe_route(x, wr, b, T, w.H, w.E, w.k, ids, tw, ws, nb, stream())
    no_device_error()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(tw.cpu().numpy(), w_ref, rtol=0, atol=route_w_atol(T, w.H, w.E))


@pytest.mark.parametrize("T,H,E,k", [(1, 256, 8, 2), (5, 520, 8, 3), (16, 2048, 64, 6), (16, 512, 512, 16),
                                     (3, 4096, 256, 8), (17, 256, 40, 4), (511, 256, 64, 4), (512, 256, 64, 4),
                                     (700, 192, 512, 16), (1000, 128, 40, 3)])
def test_route_shapes(T, H, E, k):
    """The one-launch decode router (T <= 16) across slice counts, E up to 512
    and k up to 16; the H-sliced fp32 routers for 16 < T < 512 (16-token chunks
    below 128 tokens, 64x64 tiles from 128); and the tensor-core router
    (three-term bf16 split of the fp32 weights) from T = 512 on, with a ragged
    last tile."""
    w = synth.Workload("r", T, H, E, k, 64, 0, sigma_router=0.3, zipf_s=1.0)
    x_np, wr_np, b_np = synth.make_activations(w, 4)
    ids_ref, w_ref, _ = om.route(x_np, wr_np, b_np, k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    nb = B.moe_route_workspace_bytes(T, H, E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.moe_route(bf16_tensor(x_np, "cuda"), f32(wr_np), f32(b_np), T, H, E, k, ids, tw, ws, nb, stream())
    no_device_error()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(tw.cpu().numpy(), w_ref, rtol=0, atol=route_w_atol(T, H, E))


def test_route_near_ties_tensor_core_path():
    """Experts with nearly equal router rows: most tokens have a k-th vs
    (k+1)-th logit gap below 1e-3 and about a third below the 5e-4 band in
    which the tensor-core router re-evaluates the boundary in fp32; the ids
    must equal the oracle's.  Tokens whose fp64 gap is below 2e-4 are dropped
    (closer calls depend on the fp32 summation order itself)."""
    H, E, k = 256, 64, 4
    rng = np.random.default_rng(21)
    x_bits = synth.random_bf16((4096, H), seed=21, tag=70)
    base = rng.standard_normal(H).astype(np.float32) * 0.1
    wr = (base[None, :] + 4e-4 * rng.standard_normal((E, H))).astype(np.float32)
    l64 = om.bf16_to_f64(x_bits) @ wr.astype(np.float64).T
    srt = np.sort(l64, axis=1)[:, ::-1]
    gap = srt[:, k - 1] - srt[:, k]
    keep = np.nonzero(gap > 2e-4)[0][:2048]
    assert len(keep) >= 1024 and np.mean(gap[keep] < 1e-3) > 0.5 and np.mean(gap[keep] < 5e-4) > 0.25
    x_np = np.ascontiguousarray(x_bits[keep])
    T = len(keep)
    ids_ref, w_ref, _ = om.route(x_np, wr, None, k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    nb = B.moe_route_workspace_bytes(T, H, E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.moe_route(bf16_tensor(x_np, "cuda"), f32(wr), None, T, H, E, k, ids, tw, ws, nb, stream())
    no_device_error()
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(tw.cpu().numpy(), w_ref, rtol=0, atol=route_w_atol(T, H, E))


# ---------------------------------------------------------------- a2 permute

def _permute(ids_np, x_np, E, H, with_x=True):
    T, k = ids_np.shape
    ids = i32(ids_np)
    x = bf16_tensor(x_np, "cuda") if with_x else None
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    st = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    xp = torch.empty((T * k, H), dtype=torch.bfloat16, device="cuda") if with_x else None
    nb = B.moe_permute_workspace_bytes(T, E)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    B.moe_permute(ids, x, T, H, E, k, off, st, inv, xp, ws, nb, stream())
    return off, st, inv, xp


@pytest.mark.parametrize("name,T", synth.FULL_SHAPES)
def test_permute(name, T):
    w = synth.workload(name, T)
    inp = inputs(name, T)
    ids, _, off_ref, st_ref, inv_ref = routing(name, T)
    off, st, inv, xp = _permute(ids, inp["x"], w.E, w.H)
    no_device_error()
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(st.cpu().numpy(), st_ref)
    np.testing.assert_array_equal(inv.cpu().numpy(), inv_ref)
    xp_bits = xp.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(xp_bits, inp["x"][st_ref])


@pytest.mark.parametrize("T", [255, 256, 257, 1000])
def test_permute_block_boundaries(T):
    """Both sort paths (one block for T <= 256, three passes above) around the
    block size, with skewed ids, against the oracle."""
    E, k = 37, 5
    rng = np.random.default_rng(T)
    p = 1.0 / np.arange(1, E + 1) ** 1.2
    p /= p.sum()
    # skewed, in no particular slot order
    ids = np.stack([rng.permutation(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]).astype(np.int32)
    off_ref, st_ref, inv_ref = om.permute(ids, E)
    off, st, inv, _ = _permute(ids, None, E, 64, with_x=False)
    no_device_error()
    np.testing.assert_array_equal(off.cpu().numpy(), off_ref)
    np.testing.assert_array_equal(st.cpu().numpy(), st_ref)
    np.testing.assert_array_equal(inv.cpu().numpy(), inv_ref)


def test_permute_rejects_bad_ids():
    """An id out of range or repeated within a token is recorded as a device
    check error; that token's pairs get row -1 and nothing is written out of
    bounds."""
    ids = np.array([[0, 1], [2, 9], [3, 3], [1, 2]], dtype=np.int32)
    off, st, inv, _ = _permute(ids, None, 4, 64, with_x=False)
    assert B.moe_last_device_error(stream()) == -6
    inv = inv.cpu().numpy().reshape(4, 2)
    assert (inv[1] == -1).all() and (inv[2] == -1).all()
    off = off.cpu().numpy()
    assert off[-1] == 4          # only tokens 0 and 3 were sorted
    assert B.moe_last_device_error(stream()) == 0   # read clears it


# ---------------------------------------------------------------- a3/a4 grouped GEMM

GEMM_CASES = [
    # (group rows, N, K, act): weights-on-M form (few rows per group) ...
    ([1, 0, 3, 16, 17, 64, 0, 2], 256, 128, 0),
    ([1, 0, 3, 16, 17, 64, 0, 2], 128, 192, 1),
    ([1, 0, 3, 16, 2, 0, 9, 1], 256, 512, 1),           # every group <= 16 rows: split-K applies
    ([1, 0, 3, 16, 2, 0, 9, 1], 384, 2048, 0),
    ([1] * 8 + [0] * 100 + [2, 16], 128, 1024, 1),      # few units, many groups
    ([5], 2048, 768, 0),
    ([100, 0, 5, 200, 1, 63, 65, 0], 384, 256, 1),     # groups over one 64-row chunk
    ([100, 0, 5, 200, 1, 63, 65, 0], 256, 128, 0),
    # more whole units than CTAs (groups over 16 rows): several units per CTA
    ([64] * 16 + [20, 40, 3], 2048, 128, 0),
    ([64] * 16 + [20, 40, 3], 2048, 128, 1),
    # ... and tokens-on-M form (many rows per group): ragged 128-row tiles
    ([127, 129, 0, 300], 256, 192, 1),
    ([127, 129, 0, 300], 192, 128, 0),
    ([127, 129, 0, 300], 384, 64, 0),
    ([128, 1, 255, 0, 257], 128, 256, 1),
    ([64, 1000], 192, 64, 1),
    ([513], 512, 128, 0),
    # multicast pairs over several weight blocks: single tiles, odd last tiles
    # beside tile pairs, an odd number of weight-block pairs
    ([127, 129, 0, 300, 385], 768, 128, 1),
    ([257, 0, 384, 1], 1024, 192, 0),
]


@pytest.mark.parametrize("use_ws", [False, True])
@pytest.mark.parametrize("rows,N,K,act", GEMM_CASES)
def test_grouped_gemm(rows, N, K, act, use_ws):
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    rows_max = R + 5           # rows past the last group must stay untouched
    a_bits = synth.random_bf16((rows_max, K), seed=R + N, tag=51)
    w_bits = synth.random_bf16((G, 2 * N if act else N, K), seed=K + G, tag=52, sigma=0.05)
    ref = om.grouped_gemm(a_bits, w_bits, off, act)
    a = bf16_tensor(a_bits, "cuda")
    w = bf16_tensor(w_bits, "cuda")
    nb = B.moe_grouped_gemm_workspace_bytes(G, rows_max, N, K, act)
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda") if use_ws else None
    out = torch.full((rows_max, N), 1024.0, dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm(a, w, i32(off), G, rows_max, N, K, act, out, ws, nb if use_ws else 0, stream())
    no_device_error()
    got = to_f64(out)
    assert_close_layer(got[:R], ref[:R], f"gemm rows={rows} N={N} K={K} act={act}")
    assert np.all(got[R:] == 1024.0)
    if use_ws:   # the scratch counters are back to zero, and a second call gives the same bits
        assert nb == 0 or int(ws[:COUNTER_REGION_BYTES].view(torch.int32).abs().sum()) == 0
        out2 = torch.full_like(out, 1024.0)
        B.moe_grouped_gemm(a, w, i32(off), G, rows_max, N, K, act, out2, ws, nb, stream())
        no_device_error()
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    # per-row check as well: no row may be far off even if the total is fine
    for r in np.linspace(0, R - 1, min(R, 16)).astype(int):
        scale = np.abs(ref[r]).max() + 1e-6
        assert np.abs(got[r] - ref[r]).max() <= 2e-2 * scale, r


@pytest.mark.parametrize("T,N,K,act", [(1, 256, 128, 1), (37, 128, 256, 0), (200, 256, 128, 1), (300, 128, 64, 0)])
def test_grouped_gemm_single_group_no_offsets(T, N, K, act):
    """G = 1 without an offsets array: the shared expert's form."""
    a_bits = synth.random_bf16((T, K), seed=T, tag=53)
    w_bits = synth.random_bf16((1, 2 * N if act else N, K), seed=N, tag=54, sigma=0.05)
    ref = om.grouped_gemm(a_bits, w_bits, np.array([0, T]), act)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    nb = B.moe_grouped_gemm_workspace_bytes(1, T, N, K, act)
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
    B.moe_grouped_gemm(bf16_tensor(a_bits, "cuda"), bf16_tensor(w_bits, "cuda"), None, 1, T, N, K, act, out, ws, nb,
                       stream())
    no_device_error()
    assert_close_layer(to_f64(out), ref, "single group")


def test_grouped_gemm_shapes_share_one_scratch():
    """Calls of different shapes use one scratch buffer in turn (sized for the
    largest); each gives the same bits as with a fresh zeroed scratch.  The
    second shape has more units than the first and splits too, so its ticket
    counters would sit where the first call left partial sums if the counter
    region depended on the shape."""
    seq = [([1, 2, 3, 1], 256, 2048, 1), ([1] * 40, 256, 2048, 0), ([1, 0, 3, 16, 2, 0, 9, 1], 384, 2048, 0),
           ([2] * 30, 128, 1024, 1), ([1, 2, 3, 1], 256, 2048, 1)]
    probs = []
    for i, (rows, N, K, act) in enumerate(seq):
        G = len(rows)
        off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
        R = int(off[-1])
        a = bf16_tensor(synth.random_bf16((R, K), seed=R + N + i, tag=55), "cuda")
        w = bf16_tensor(synth.random_bf16((G, 2 * N if act else N, K), seed=K + G, tag=56, sigma=0.03), "cuda")
        probs.append((a, w, i32(off), G, R, N, K, act))
    big = max(B.moe_grouped_gemm_workspace_bytes(G, R, N, K, act) for _, _, _, G, R, N, K, act in probs)
    shared = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for a, w, off, G, R, N, K, act in probs:
        out = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
        B.moe_grouped_gemm(a, w, off, G, R, N, K, act, out, shared, big, stream())
        no_device_error()
        nb = B.moe_grouped_gemm_workspace_bytes(G, R, N, K, act)
        fresh = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(out)
        B.moe_grouped_gemm(a, w, off, G, R, N, K, act, ref, fresh, nb, stream())
        no_device_error()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (G, R, N, K, act)


@pytest.mark.parametrize("rows,N,K,act", [
    ([1, 0, 2, 0, 1], 256, 512, 1), ([1, 0, 2, 0, 1], 512, 256, 0), ([0, 0, 4], 128, 2048, 1),
    ([1] * 4 + [0] * 60, 768, 2048, 1), ([1] * 4 + [0] * 60, 2048, 768, 0), ([3], 192, 64, 0), ([2, 2], 64, 128, 1),
    ([0, 1, 0], 768, 2048, 1), ([0, 0, 0, 1], 2048, 768, 0), ([1], 256, 512, 1), ([1], 192, 64, 0)])
def test_grouped_gemm_groups_of_at_most_four_rows(rows, N, K, act):
    """Groups of at most four rows with rows_max equal to the rows held (a
    single row runs on the CUDA cores, more on the tensor cores): every row
    checked against the oracle, and the call repeats bit for bit."""
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    a_bits = synth.random_bf16((R, K), seed=R + N + K, tag=57)
    w_bits = synth.random_bf16((G, 2 * N if act else N, K), seed=K + G, tag=58, sigma=0.05)
    ref = om.grouped_gemm(a_bits, w_bits, off, act)
    a = bf16_tensor(a_bits, "cuda")
    w = bf16_tensor(w_bits, "cuda")
    out = torch.full((R, N), 1024.0, dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm(a, w, i32(off), G, R, N, K, act, out, None, 0, stream())
    no_device_error()
    got = to_f64(out)
    assert_close_layer(got, ref, f"small groups rows={rows} N={N} K={K} act={act}")
    for r in range(R):
        scale = np.abs(ref[r]).max() + 1e-6
        assert np.abs(got[r] - ref[r]).max() <= 2e-2 * scale, r
    out2 = torch.empty_like(out)
    B.moe_grouped_gemm(a, w, i32(off), G, R, N, K, act, out2, None, 0, stream())
    no_device_error()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    if G == 1:   # no offsets: one group of R rows
        out3 = torch.empty_like(out)
        B.moe_grouped_gemm(a, w, None, 1, R, N, K, act, out3, None, 0, stream())
        no_device_error()
        assert torch.equal(out.view(torch.int16), out3.view(torch.int16))


def test_grouped_gemm_rejects_bad_offsets():
    """Offsets past rows_max or decreasing: the kernel records a device check
    error and computes nothing."""
    a = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2, 128, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((64, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    for bad in ([0, 10, 80], [0, 30, 20]):
        offs = i32(bad)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        B.moe_grouped_gemm(a, w, offs, 2, 64, 128, 64, 0, out, None, 0, stream())
        torch.cuda.synchronize()
        # the kernel leaves at once: no bounded wait ran out
        assert time.perf_counter() - t0 < 0.5
        assert B.moe_last_device_error(stream()) == -6
    assert torch.all(out == 7.0)


# ---------------------------------------------------------------- a6 combine

@pytest.mark.parametrize("name,T", [("tiny", 16), ("decode", 8), ("batched_decode", 256)])
def test_combine(name, T):
    w = synth.workload(name, T)
    _, wts, _, _, inv = routing(name, T)
    y_bits = synth.random_bf16((T * w.k, w.H), seed=T, tag=55)
    s_bits = synth.random_bf16((T, w.H), seed=T, tag=56)
    ref = om.combine(om.bf16_to_f64(y_bits), inv, wts, om.bf16_to_f64(s_bits))
    out = torch.empty((T, w.H), dtype=torch.bfloat16, device="cuda")
    B.moe_unpermute_combine(bf16_tensor(y_bits, "cuda"), i32(inv), f32(wts), bf16_tensor(s_bits, "cuda"), T, w.H,
                            w.k, out, stream())
    no_device_error()
    got = to_f64(out)
    # fp32 accumulation, one rounding to bf16: within one bf16 ulp of the exact sum
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=1e-5)
    # without the shared row
    B.moe_unpermute_combine(bf16_tensor(y_bits, "cuda"), i32(inv), f32(wts), None, T, w.H, w.k, out, stream())
    ref0 = om.combine(om.bf16_to_f64(y_bits), inv, wts, None)
    np.testing.assert_allclose(to_f64(out), ref0, rtol=2.0 ** -8, atol=1e-5)


# ---------------------------------------------------------------- whole layer

@pytest.mark.parametrize("name,T", FULL_OUTPUT_SHAPES)
def test_forward_full(name, T):
    """Every output element of the layer against the float64 oracle (at
    prefill T=8192 the tokens-on-M matmuls run as CTA pairs, both pair modes:
    groups with an even and with an odd number of 128-row tiles)."""
    w = synth.workload(name, T)
    inp = inputs(name, T)
    ref = om.forward(inp, w.k)
    L = layer(name, T)
    out = L.forward(x_tensor(name, T))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"{name} T={T}")


def _sample_tokens(name, T, n=24):
    ids, _, off, st, _ = routing(name, T)
    rng = np.random.default_rng(7)
    pick = set(rng.choice(T, size=n, replace=False).tolist()) | {0, T - 1}
    counts = np.diff(off)
    hot = int(np.argmax(counts))
    # tokens at the ends of the hottest group and of a 128-row tile boundary inside it
    g0, g1 = int(off[hot]), int(off[hot + 1])
    for r in (g0, g1 - 1, min(g0 + 127, g1 - 1), min(g0 + 128, g1 - 1)):
        pick.add(int(st[r]))
    # groups whose last 128-row tile is odd (the pair shares that tile between two
    # weight blocks) and groups with an even tile count: first and last row of the last tile
    tiles = (counts + 127) // 128
    for parity in (1, 0):
        gs = [g for g in np.nonzero((tiles % 2 == parity) & (counts > 0))[0]]
        for g in gs[:6]:
            r0 = int(off[g]) + 128 * (int(tiles[g]) - 1)
            pick.add(int(st[r0]))
            pick.add(int(st[int(off[g + 1]) - 1]))
    return np.array(sorted(pick))


@pytest.mark.parametrize("name,T", LARGE_SHAPES)
def test_forward_sampled_full_size(name, T):
    """The large prefill layer: every output is finite, and sampled rows
    (random tokens, tokens at the hot group's tile boundaries, and the first
    and last rows of the last tile of groups with an odd and an even number of
    tiles) match the oracle evaluated token by token."""
    w = synth.workload(name, T)
    inp = inputs(name, T)
    ids, wts, *_ = routing(name, T)
    L = layer(name, T)
    out = L.forward(x_tensor(name, T))
    no_device_error()
    toks = _sample_tokens(name, T)
    ref = om.forward_tokens(inp, w.k, toks, routing=(ids, wts))
    got = out[torch.from_numpy(toks).cuda()]
    assert torch.isfinite(out.float()).all()
    assert_close_layer(to_f64(got), ref["out"], f"{name} T={T} sampled")


@pytest.mark.parametrize("T", [4, 16])
def test_forward_decode_sizes_of_the_wide_layer(T):
    """Decode batches of the H=4096, E=256, I=1024 layer (the large-prefill
    layer): the one-launch router with its dispatch, gmm1 reading the rows of x
    by TMA gather4, gmm2."""
    w = synth.workload("large_prefill", T)
    ref = om.forward(inputs("large_prefill", T), w.k)
    out = layer("large_prefill", T).forward(x_tensor("large_prefill", T))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"large-prefill layer T={T}")


@pytest.mark.parametrize("T", [2, 12, 16])
def test_forward_decode_sizes(T):
    """Decode batch sizes between and beyond the benchmark's (up to the
    largest batch the one-launch router handles)."""
    w = synth.workload("decode", T)
    ref = om.forward(inputs("decode", T), w.k)
    out = layer("decode", T).forward(x_tensor("decode", T))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"decode T={T}")


def test_forward_one_hot_expert_and_empty_experts():
    """Every token routed to one expert (a group of T rows spanning several
    128-row tiles with a ragged tail) while most experts stay empty; T above
    the one-block permute size."""
    wl = synth.Workload("hot", 300, 256, 16, 2, 128, 128, sigma_router=0.1)
    inp = synth.make_inputs(wl, 11)
    bias = np.zeros(wl.E, dtype=np.float32)
    bias[5] = 50.0
    bias[[0, 1, 2, 3]] = -np.inf
    inp["bias"] = bias
    ref = om.forward(inp, wl.k)
    assert (np.diff(ref["offsets"])[5] == wl.T)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    out = L.forward(bf16_tensor(inp["x"], "cuda"))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], "hot expert")


@pytest.mark.parametrize("T,I", [(12, 64), (16, 192), (3, 128)])
def test_forward_decode_gathered_rows(T, I):
    """At decode sizes the first matmul reads the dispatched rows of x through
    sorted_token (TMA gather4) in both tile forms: I a multiple of 128 gives the
    weights-on-M form, otherwise tokens-on-M."""
    wl = synth.Workload("gather", T, 128, 8, 2, I, 64, sigma_router=0.2, sigma_w=0.05)
    inp = synth.make_inputs(wl, 13)
    ref = om.forward(inp, wl.k)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    out = L.forward(bf16_tensor(inp["x"], "cuda"))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"gathered rows T={T} I={I}")


def test_forward_one_token_wide_expert():
    """One token with wide experts (I = 8192, K of gmm2 eight times the
    decode layer's): gmm1 on the CUDA cores, then gmm2 and the combine in one
    launch."""
    wl = synth.Workload("wide", 1, 256, 8, 8, 8192, 64, sigma_router=0.1, sigma_w=0.02)
    inp = synth.make_inputs(wl, 17)
    ref = om.forward(inp, wl.k)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    out = L.forward(bf16_tensor(inp["x"], "cuda"))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], "one token, I = 8192")


def test_forward_without_shared_expert():
    wl = synth.Workload("noshared", 40, 128, 8, 2, 64, 0, sigma_router=0.1)
    inp = synth.make_inputs(wl, 12)
    ref = om.forward(inp, wl.k)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    out = L.forward(bf16_tensor(inp["x"], "cuda"))
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], "no shared expert")


def test_forward_batches_of_different_sizes_share_one_workspace():
    """One layer object keeps one workspace (sized for its largest batch) and
    runs batches of different sizes in turn, across both router paths and both
    tile forms; each output has the same bits as the same batch run through a
    fresh workspace."""
    wl = synth.Workload("vary", 300, 512, 16, 4, 1024, 128, sigma_router=0.1, sigma_w=0.03)
    inp = synth.make_inputs(wl, 21)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    x = bf16_tensor(inp["x"], "cuda")
    L.workspace(wl.T)
    for T in [300, 8, 64, 1, 16, 200, 8, 3]:
        got = L.forward(x[:T]).clone()
        no_device_error()
        fresh = MoEFFN.from_inputs(inp, wl.k, "cuda")
        ref = fresh.forward(x[:T])
        no_device_error()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), T


@pytest.mark.parametrize("T,H,E,k", [(700, 512, 8, 2), (100, 256, 2, 2)])
def test_forward_matches_standalone_calls(T, H, E, k):
    """At sizes where both matmuls take the tokens-on-M form (no split-K), the
    layer output has the same bits as the standalone calls (route, permute,
    both matmuls, shared expert, combine), and matches the oracle.  T = 100
    takes the one-block sort."""
    wl = synth.Workload("standalone", T, H, E, k, 256, 128, sigma_router=0.1, sigma_w=0.03)
    inp = synth.make_inputs(wl, 23)
    ref = om.forward(inp, wl.k)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    x = bf16_tensor(inp["x"], "cuda")
    out = L.forward(x).clone()
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"forward T={T}")
    wr, bias, wgu, wd, sgu, sd = L.tensors
    rows = T * k
    dev = "cuda"
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    tw = torch.empty((T, k), dtype=torch.float32, device=dev)
    rb, pb = B.moe_route_workspace_bytes(T, H, E), B.moe_permute_workspace_bytes(T, E)
    rws = torch.empty(max(rb, 256), dtype=torch.uint8, device=dev)
    pws = torch.empty(max(pb, 256), dtype=torch.uint8, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    st = torch.empty(rows, dtype=torch.int32, device=dev)
    inv = torch.empty(rows, dtype=torch.int32, device=dev)
    xp = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    h = torch.empty((rows, wl.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((rows, H), dtype=torch.bfloat16, device=dev)
    hs = torch.empty((T, wl.Is), dtype=torch.bfloat16, device=dev)
    sh = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    out2 = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    B.moe_route(x, wr, bias, T, H, E, k, ids, tw, rws, rb, stream())
    B.moe_permute(ids, x, T, H, E, k, offs, st, inv, xp, pws, pb, stream())
    B.moe_grouped_gemm(xp, wgu, offs, E, rows, wl.I, H, 1, h, None, 0, stream())
    B.moe_grouped_gemm(h, wd, offs, E, rows, H, wl.I, 0, y, None, 0, stream())
    B.moe_grouped_gemm(x, sgu, None, 1, T, wl.Is, H, 1, hs, None, 0, stream())
    B.moe_grouped_gemm(hs, sd, None, 1, T, H, wl.Is, 0, sh, None, 0, stream())
    B.moe_unpermute_combine(y, inv, tw, sh, T, H, k, out2, stream())
    no_device_error()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("case", ["decode", "no_shared", "k12"])
def test_forward_one_token_matches_standalone_calls(case):
    """One token: the layer runs gmm2 and the combine as one launch (k <= 8);
    its output has the same bits as the standalone calls (route, one-row
    gate_up and down per slot, the shared expert, combine), and matches the
    oracle.  k = 12 keeps the two launches."""
    if case == "decode":
        wl = synth.workload("decode", 1)
    elif case == "no_shared":
        wl = synth.Workload("one", 1, 512, 16, 4, 256, 0, sigma_router=0.1, sigma_w=0.03)
    else:
        wl = synth.Workload("one", 1, 256, 32, 12, 128, 64, sigma_router=0.1, sigma_w=0.03)
    inp = synth.make_inputs(wl, 31)
    ref = om.forward(inp, wl.k)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    x = bf16_tensor(inp["x"], "cuda")
    out = L.forward(x).clone()
    no_device_error()
    assert_close_layer(to_f64(out), ref["out"], f"one token {case}")
    H, E, k, I, Is = wl.H, wl.E, wl.k, wl.I, wl.Is
    wr, bias, wgu, wd, sgu, sd = L.tensors
    dev = "cuda"
    ids = torch.empty((1, k), dtype=torch.int32, device=dev)
    tw = torch.empty((1, k), dtype=torch.float32, device=dev)
    rb = B.moe_route_workspace_bytes(1, H, E)
    rws = torch.empty(max(rb, 256), dtype=torch.uint8, device=dev)
    B.moe_route(x, wr, bias, 1, H, E, k, ids, tw, rws, rb, stream())
    nb = max(B.moe_grouped_gemm_workspace_bytes(1, 1, n_, k_, a_)
             for n_, k_, a_ in [(I, H, 1), (H, I, 0), (max(Is, 64), H, 1), (H, max(Is, 64), 0)])
    gws = torch.zeros(max(nb, 256), dtype=torch.uint8, device=dev)
    y = torch.empty((k, H), dtype=torch.bfloat16, device=dev)
    h = torch.empty((1, I), dtype=torch.bfloat16, device=dev)
    for j, g in enumerate(ids[0].tolist()):
        B.moe_grouped_gemm(x, wgu[g:g + 1], None, 1, 1, I, H, 1, h, gws, nb, stream())
        B.moe_grouped_gemm(h, wd[g:g + 1], None, 1, 1, H, I, 0, y[j:j + 1], gws, nb, stream())
    sh = None
    if Is:
        hs = torch.empty((1, Is), dtype=torch.bfloat16, device=dev)
        sh = torch.empty((1, H), dtype=torch.bfloat16, device=dev)
        B.moe_grouped_gemm(x, sgu, None, 1, 1, Is, H, 1, hs, gws, nb, stream())
        B.moe_grouped_gemm(hs, sd, None, 1, 1, H, Is, 0, sh, gws, nb, stream())
    out2 = torch.empty((1, H), dtype=torch.bfloat16, device=dev)
    inv = torch.arange(k, dtype=torch.int32, device=dev)   # y is in slot order
    B.moe_unpermute_combine(y, inv, tw, sh, 1, H, k, out2, stream())
    no_device_error()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


DISPATCH_CASES = [("decode", 1), ("decode", 4), ("decode", 8), ("decode", 16), ("tiny", 16),
                  ("batched_decode", 64)]


@pytest.mark.parametrize("name,T", DISPATCH_CASES)
def test_forward_dispatch_bit_exact(name, T):
    """The routing and dispatch the layer forward itself computed (read from
    its workspace): expert ids, offsets, sorted tokens and the inverse
    permutation bit-exact against the oracle, weights within the router
    tolerance."""
    w = synth.workload(name, T)
    ids_ref, w_ref, off_ref, st_ref, inv_ref = routing(name, T)
    L = layer(name, T)
    ws = L.workspace(T)
    ws.fill_(0)        # every region below must be written by this call
    L.forward(x_tensor(name, T))
    no_device_error()
    o = B.moe_workspace_layout(L.dims, T)
    Tk = T * w.k

    def region(off, n, dtype):
        return ws[off:off + n * 4].view(dtype).cpu().numpy()

    np.testing.assert_array_equal(region(o.topk_ids, Tk, torch.int32).reshape(T, w.k), ids_ref)
    np.testing.assert_allclose(region(o.topk_w, Tk, torch.float32).reshape(T, w.k), w_ref, rtol=0,
                               atol=route_w_atol(T, w.H, w.E))
    np.testing.assert_array_equal(region(o.expert_offsets, w.E + 1, torch.int32), off_ref)
    np.testing.assert_array_equal(region(o.sorted_token, Tk, torch.int32), st_ref)
    np.testing.assert_array_equal(region(o.inv_perm, Tk, torch.int32), inv_ref)
    ws.fill_(0)        # leave the workspace as the layer expects it (counters zero)


def _random_layer(seed: int):
    """A seeded layer shape within the supported ranges (H, I, I_s multiples
    of 64; k <= min(E, 16)), with or without router bias and shared expert."""
    r = np.random.default_rng(1000 + seed)
    E = int(r.choice([2, 4, 8, 16, 32, 64, 256]))
    k = int(r.integers(1, min(E, 16) + 1)) if r.random() < 0.3 else int(r.integers(1, min(E, 8) + 1))
    wl = synth.Workload(f"random{seed}", int(r.choice([1, 2, 3, 5, 7, 9, 13, 16, 17, 33, 64, 100, 257, 600])),
                        int(r.choice([128, 256, 384, 512, 1024])), E, k, int(r.choice([64, 128, 192, 256, 512])),
                        int(r.choice([0, 64, 128, 256])), sigma_router=0.1, sigma_w=0.03,
                        zipf_s=1.1 if r.random() < 0.4 else None)
    return wl


@pytest.mark.parametrize("seed", range(48))
def test_forward_random_shapes(seed):
    """Seeded random layer shapes (batch size, hidden and expert sizes, experts,
    top-k, shared expert or none, skewed routing or not): the layer output
    within the layer tolerance of the oracle, and the dispatch the forward
    computed (read from its workspace) bit-exact."""
    wl = _random_layer(seed)
    T = wl.T
    inp = synth.make_inputs(wl, seed)
    ref = om.forward(inp, wl.k)
    ids_ref, w_ref, _ = om.route(inp["x"], inp["w_router"], inp["bias"], wl.k)
    off_ref, st_ref, inv_ref = om.permute(ids_ref, wl.E)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    ws = L.workspace(T)
    out = L.forward(bf16_tensor(inp["x"], "cuda")).clone()
    no_device_error()
    shape = f"T={T} H={wl.H} E={wl.E} k={wl.k} I={wl.I} I_s={wl.Is} zipf={wl.zipf_s}"
    assert_close_layer(to_f64(out), ref["out"], shape)
    o = B.moe_workspace_layout(L.dims, T)
    Tk = T * wl.k

    def region(off, n, dtype):
        return ws[off:off + n * 4].view(dtype).cpu().numpy()

    np.testing.assert_array_equal(region(o.topk_ids, Tk, torch.int32).reshape(T, wl.k), ids_ref, err_msg=shape)
    np.testing.assert_array_equal(region(o.expert_offsets, wl.E + 1, torch.int32), off_ref, err_msg=shape)
    np.testing.assert_array_equal(region(o.sorted_token, Tk, torch.int32), st_ref, err_msg=shape)
    np.testing.assert_array_equal(region(o.inv_perm, Tk, torch.int32), inv_ref, err_msg=shape)


@pytest.mark.parametrize("name,T", [("decode", 1), ("decode", 8), ("batched_decode", 256), ("prefill", 8192)])
def test_forward_graph_replay_matches_eager(name, T):
    """The forward captured in a CUDA graph (as the benchmark times it) and
    replayed gives the same bits as the eager call."""
    L = layer(name, T)
    x = x_tensor(name, T)
    eager = L.forward(x).clone()
    no_device_error()
    s = torch.cuda.Stream()
    out = torch.zeros_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.forward(x, out, torch.cuda.current_stream())
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        no_device_error()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_operands_outside_device_memory_are_refused():
    """The matmuls read their operands with TMA (the prefill form multicasts
    them between the CTAs of a cluster): host memory, pinned or not, is refused
    on the host before any launch."""
    G, R, N, K = 2, 600, 512, 128          # tokens-on-M with 256-wide blocks: the pair form
    w = torch.zeros((G, 2 * N, K), dtype=torch.bfloat16, device="cuda")
    a = torch.zeros((R, K), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((R, N), dtype=torch.bfloat16, device="cuda")
    offs = i32(np.array([0, 300, 600]))
    B.moe_grouped_gemm(a, w, offs, G, R, N, K, 1, out, None, 0, stream())     # device memory: runs
    no_device_error()
    a_pinned = torch.zeros((R, K), dtype=torch.bfloat16).pin_memory()
    a_host = np.zeros((R, K), dtype=np.uint16)
    for bad in (a_pinned.data_ptr(), a_host.ctypes.data):
        with pytest.raises(B.MoEError) as e:
            B.moe_grouped_gemm(bad, w, offs, G, R, N, K, 1, out, None, 0, stream())
        assert e.value.code == -2
        with pytest.raises(B.MoEError) as e:
            B.moe_grouped_gemm(a, bad, offs, G, R, N, K, 1, out, None, 0, stream())
        assert e.value.code == -2
        with pytest.raises(B.MoEError) as e:
            B.moe_grouped_gemm_noalloc(bad, w, offs, G, R, N, K, 1, out, stream())
        assert e.value.code == -2
    # the layer forward: x in host memory
    L = layer("tiny", 16)
    x_pinned = torch.zeros((16, 256), dtype=torch.bfloat16).pin_memory()
    ws = L.workspace(16)
    o = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.moe_forward(L.dims, L.weights, x_pinned, 16, o, ws, ws.numel(), stream(), L.side, L.ev_fork, L.ev_join)
    assert e.value.code == -2
    no_device_error()


@pytest.mark.parametrize("T", [4, 9])
def test_forward_shared_expert_as_leading_phase(T):
    """4 to 9 tokens: the shared expert leads the routed matmul launches (its
    gate_up before the gate_up launch waits on the router), no side stream:
    four launches, the oracle's output, the same bits on a second call and
    through a CUDA graph."""
    L = layer("tiny", T)
    x = x_tensor("tiny", T)
    ref = om.forward(inputs("tiny", T), synth.workload("tiny", T).k)
    a = L.forward(x).clone()
    assert B.moe_last_launch_count() == 4   # router with dispatch, gate_up, down, combine
    no_device_error()
    assert_close_layer(to_f64(a), ref["out"], f"tiny T={T}")
    b = L.forward(x).clone()
    g_out = torch.empty_like(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.forward(x, g_out, s)   # (sizes the workspace on this stream before capture)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.forward(x, g_out, torch.cuda.current_stream())
    g_out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    no_device_error()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), g_out.view(torch.int16))


def test_forward_repeatable_and_launch_count():
    """Two calls give identical bits; the launch count is what the call reports."""
    L = layer("tiny", 16)
    x = x_tensor("tiny", 16)
    a = L.forward(x).clone()
    n = B.moe_last_launch_count()
    b = L.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # shared gate_up and down; router with dispatch, gate_up, down, combine
    assert n == 6
