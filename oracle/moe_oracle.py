"""CPU oracle for the MoE FFN layer forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and
its binding) never calls it, and it shares no code with that path: it reads
the same seeded inputs and nothing else.

What it computes, step by step, as plain definitions (numpy; float64 except
where the layer fixes another precision):

* The layer: routed experts, then the shared expert, then a reduction, where
  the shared expert reads the same hidden states and does not depend on the
  routed path ("Ascend 910C LLM inference optimisation, part 2" (Dewu Tech),
  section "MoE multi-stream overlap": the MoE layer's order routed GroupedMatmul
  -> shared expert -> AllReduce, the shared expert's independence, and its
  gate_up (part 1) and down (part 2) matmuls on the same hidden_states).  The
  AllReduce is the identity at one tensor-parallel rank.
* The routed side runs dispatch -> gmm1 (gate_up) -> activation -> gmm2 (down)
  -> combine (same page and section, the dispatch/combine/gmm2 events).
* Router, activation and combine weights are fixed by the layer's definition
  of the benchmark shapes, not by the page: fp32 router logits x.Wr^T + b,
  the k largest logits per token, weights = softmax over those k logits (equal
  to the full softmax over E renormalised over the chosen k), SiLU(gate)*up,
  output = sum_j w_j * expert_j(x) + shared(x).

Readings where the definition leaves a choice: top-k ties go to the lower
expert id; a token's chosen ids are reported in ascending id order; rows of the
permuted layout are grouped by expert (ascending) and, within an expert, by
token (ascending).  The router's top-k decision is taken on fp32 logits, the
precision the layer fixes for the router; everything after it is float64.

FP8 expert weights (the w8a8_dynamic matmul configuration of the xLLM PR
"FlashComm1 + matmul-reduce-scatter", configuration section, read for the
weight side only): each routed expert's weight rows are stored as e4m3 codes
(OCP 8-bit float: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
exponent 0 holding the subnormals m * 2^-9, codes 0x7f/0xff NaN, no infinity)
with one fp32 scale per row (output channel): W[n][k] = e4m3(q[n][k]) * s[n].
The layer is the same layer with those weights; activations stay bf16 and the
shared expert stays bf16 (the MoE page keeps it unquantised).

Parity pins (tests/test_oracle.py): brute-force fp64 top-k, the full-softmax
closed form, numpy's stable argsort for the permutation, a dense SwiGLU MLP in
torch for E=1, a brute-force dense evaluation of every expert on every token
masked by the routing weights, the identical-experts invariant, linearity in the
down weights, a hand-derived closed-form example (tests/golden/), torch's
float8_e4m3fn decoding of every code, and the FP8 layer equal to the bf16
layer when the bf16 weights are exactly e4m3 codes times their row scales.
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# storage types
# ----------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as uint16 bit patterns."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of e4m3 codes (uint8): sign bit 7, exponent bits 6..3 (bias
    7), mantissa bits 2..0; exponent 0 gives m * 2^-9, otherwise
    (1 + m/8) * 2^(e-7); 0x7f and 0xff are NaN."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def dequant_w8(codes: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Weights of e4m3 codes [..., rows, K] with one fp32 scale per row
    [..., rows]: value times scale, float64 (exact)."""
    return e4m3_to_f64(codes) * np.asarray(scale, dtype=np.float32).astype(np.float64)[..., None]


def is_w8(inp: dict) -> bool:
    """The routed expert weights are e4m3 codes with row scales."""
    return "w_gate_up_scale" in inp


def expert_gate_up(inp: dict, e: int) -> np.ndarray:
    """float64 gate_up weights [2I][H] of routed expert e."""
    if is_w8(inp):
        return dequant_w8(inp["w_gate_up"][e], inp["w_gate_up_scale"][e])
    return bf16_to_f64(inp["w_gate_up"][e])


def expert_down(inp: dict, e: int) -> np.ndarray:
    """float64 down weights [H][I] of routed expert e."""
    if is_w8(inp):
        return dequant_w8(inp["w_down"][e], inp["w_down_scale"][e])
    return bf16_to_f64(inp["w_down"][e])


# ----------------------------------------------------------------------------
# a1: router
# ----------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, w_router: np.ndarray, bias) -> np.ndarray:
    """fp32 logits l[t, e] = sum_h x[t, h] * Wr[e, h] + b[e] (fp32 matrix product)."""
    l = bf16_to_f32(x_bits) @ np.asarray(w_router, dtype=np.float32).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32)[None, :]
    return l.astype(np.float32)


def route(x_bits, w_router, bias, k: int):
    """Top-k expert choice and renormalised softmax weights per token.

    Returns (ids int32 [T, k] ascending per row, weights float64 [T, k],
    fp32 logits [T, E]).
    """
    l = router_logits(x_bits, w_router, bias)
    T, E = l.shape
    ids = np.empty((T, k), dtype=np.int32)
    wts = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        # descending logit, ties to the lower id: a stable sort of -l
        order = np.argsort(-l[t].astype(np.float64), kind="stable")[:k]
        chosen = np.sort(order)
        sel = l[t, chosen].astype(np.float64)
        m = sel.max()
        p = np.exp(sel - m)
        ids[t] = chosen
        wts[t] = p / p.sum()
    return ids, wts, l


# ----------------------------------------------------------------------------
# a2: permute (counting sort by expert, then token)
# ----------------------------------------------------------------------------

def permute(ids: np.ndarray, E: int):
    """Counting sort of the T*k (token, slot) pairs by (expert, token).

    Returns expert_offsets int32 [E+1] (exclusive prefix of the per-expert
    counts), sorted_token int32 [T*k] (token of each permuted row) and
    inv_perm int32 [T*k] (permuted row of pair (t, j) at index t*k + j).
    """
    T, k = ids.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[ids[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E].copy()
    sorted_token = np.empty(T * k, dtype=np.int32)
    inv_perm = np.empty(T * k, dtype=np.int32)
    for t in range(T):                       # tokens in ascending order
        for j in range(k):
            e = ids[t, j]
            r = cursor[e]
            cursor[e] += 1
            sorted_token[r] = t
            inv_perm[t * k + j] = r
    return offsets.astype(np.int32), sorted_token, inv_perm


# ----------------------------------------------------------------------------
# a3/a4/a5: expert MLP pieces
# ----------------------------------------------------------------------------

def silu(v: np.ndarray) -> np.ndarray:
    """SiLU(v) = v * sigmoid(v) = v / (1 + exp(-v))."""
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def gate_up(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """gmm1 + activation for one expert: W (float64) is [2N][K], rows 0..N-1
    gate, N..2N-1 up; returns SiLU(a.Wg^T) * (a.Wu^T), float64 [rows, N]."""
    n = w.shape[0] // 2
    g = a @ w[:n].T
    u = a @ w[n:].T
    return silu(g) * u


def down(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """gmm2 for one expert: h.Wd^T with Wd (float64) [N_out][K]."""
    return h @ w.T


def grouped_gemm(a_bits: np.ndarray, w_bits: np.ndarray, offsets: np.ndarray, act: int, w_scale=None):
    """Rows [off_g, off_{g+1}) of A times group g's weights (W[g] K-major).

    act 0: out = A_g . W_g^T (W [G][N][K]); act 1: out = SiLU(A_g.Wg^T)*(A_g.Wu^T)
    (W [G][2N][K]).  W is bf16 bits, or e4m3 codes when w_scale ([G][rows]
    fp32, one per weight row) is given.  float64 [rows, N]; rows past
    offsets[G] are left at 0.
    """
    a = bf16_to_f64(a_bits)
    G = w_bits.shape[0]
    n_out = w_bits.shape[1] // 2 if act == 1 else w_bits.shape[1]
    out = np.zeros((a.shape[0], n_out), dtype=np.float64)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            w = bf16_to_f64(w_bits[g]) if w_scale is None else dequant_w8(w_bits[g], w_scale[g])
            out[r0:r1] = gate_up(a[r0:r1], w) if act == 1 else (a[r0:r1] @ w.T)
    return out


def shared_expert(x: np.ndarray, ws_gate_up_bits, ws_down_bits) -> np.ndarray:
    """Shared expert on the hidden states: down(gate_up(x)); zero when absent."""
    if ws_gate_up_bits is None:
        return np.zeros_like(x)
    return down(gate_up(x, bf16_to_f64(ws_gate_up_bits)), bf16_to_f64(ws_down_bits))


# ----------------------------------------------------------------------------
# a6: combine, and the whole layer
# ----------------------------------------------------------------------------

def combine(y: np.ndarray, inv_perm: np.ndarray, w: np.ndarray, s) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y[inv_perm[t*k + j]] + s[t]."""
    T, k = w.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[inv_perm.reshape(T, k)[:, j]]
    if s is not None:
        out += s
    return out


def forward(inp: dict, k: int) -> dict:
    """Whole layer in the routed order dispatch -> gmm1 -> act -> gmm2 -> combine,
    plus the shared expert.  Returns every intermediate (float64 where real)."""
    x = bf16_to_f64(inp["x"])
    E = inp["w_gate_up"].shape[0]
    ids, wts, logits = route(inp["x"], inp["w_router"], inp["bias"], k)
    offsets, sorted_token, inv_perm = permute(ids, E)
    x_perm = x[sorted_token]
    I = inp["w_gate_up"].shape[1] // 2
    h = np.zeros((x_perm.shape[0], I))
    y = np.zeros((x_perm.shape[0], x.shape[1]))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            h[r0:r1] = gate_up(x_perm[r0:r1], expert_gate_up(inp, e))
            y[r0:r1] = down(h[r0:r1], expert_down(inp, e))
    s = shared_expert(x, inp["ws_gate_up"], inp["ws_down"])
    out = combine(y, inv_perm, wts, s)
    return dict(ids=ids, w=wts, logits=logits, offsets=offsets, sorted_token=sorted_token,
                inv_perm=inv_perm, h=h, y=y, s=s, out=out)


def forward_tokens(inp: dict, k: int, tokens, routing=None) -> dict:
    """Output rows of the listed tokens only, each computed on its own:
    out[t] = sum_j w[t, j] * down_e(gate_up_e(x[t])) + shared(x[t]).

    ``routing`` = (ids, weights) from ``route`` may be passed to skip re-routing.
    Returns dict(tokens, out [n, H], s [n, H], h/y per (token, slot)).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    if routing is None:
        ids, wts, _ = route(inp["x"], inp["w_router"], inp["bias"], k)
    else:
        ids, wts = routing
    x = bf16_to_f64(inp["x"][tokens])
    n, H = x.shape
    I = inp["w_gate_up"].shape[1] // 2
    h = np.zeros((n, k, I))
    y = np.zeros((n, k, H))
    by_expert: dict = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            by_expert.setdefault(int(ids[t, j]), []).append((i, j))
    for e, pairs in by_expert.items():
        rows = np.array([i for i, _ in pairs])
        he = gate_up(x[rows], expert_gate_up(inp, e))
        ye = down(he, expert_down(inp, e))
        for q, (i, j) in enumerate(pairs):
            h[i, j] = he[q]
            y[i, j] = ye[q]
    s = shared_expert(x, inp["ws_gate_up"], inp["ws_down"])
    out = np.einsum("nj,njh->nh", wts[tokens], y) + s
    return dict(tokens=tokens, out=out, s=s, h=h, y=y, ids=ids[tokens], w=wts[tokens])
