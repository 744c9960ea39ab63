"""The seeded input generator: determinism, the near-tie guard and the routing
statistics each workload is defined by."""
import numpy as np
import pytest

from moe_ffn_layer_gb300 import synth


def _logits64(x, wr, b):
    l = synth.bf16_bits_to_f32(x).astype(np.float64) @ wr.astype(np.float64).T
    return l if b is None else l + b.astype(np.float64)


def test_bf16_rounding_round_to_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    back = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    np.testing.assert_array_equal(back[:4], np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], dtype=np.float32))


def test_deterministic():
    w = synth.workload("tiny")
    a, b = synth.make_inputs(w, 0), synth.make_inputs(w, 0)
    for key in a:
        if a[key] is not None:
            np.testing.assert_array_equal(a[key], b[key])
    c = synth.make_inputs(w, 1)
    assert not np.array_equal(a["x"], c["x"])


@pytest.mark.parametrize("name,T", synth.FULL_SHAPES[:6])
def test_gap_guard(name, T):
    w = synth.workload(name, T)
    x, wr, b = synth.make_activations(w)
    l = np.sort(_logits64(x, wr, b), axis=1)[:, ::-1]
    assert np.all(l[:, w.k - 1] - l[:, w.k] > synth.GAP)


def test_routing_skew_batched_decode():
    w = synth.workload("batched_decode", 64)
    x, wr, b = synth.make_activations(w)
    ids = np.argsort(-_logits64(x, wr, b), axis=1)[:, : w.k]
    cnt = np.bincount(ids.ravel(), minlength=w.E)
    assert (cnt <= 3).mean() > 0.6            # most experts get 0-3 tokens
    assert np.sort(cnt)[-3:].min() >= 12      # a few get dozens


def test_large_prefill_bias():
    w = synth.workload("large_prefill")
    b = synth.router_bias(w, 0)
    assert np.isneginf(b).sum() == 8
    fin = b[np.isfinite(b)]
    assert fin.max() == 0.0                   # rank 1 -> -s*ln(1) = 0
    np.testing.assert_allclose(np.sort(-fin / 1.2)[:3], np.log([1, 2, 3]), rtol=1e-6)


def test_e4m3_rounding_matches_torch():
    """To nearest, ties to even, subnormals, signs; up to the largest finite
    value (above it torch returns NaN, the quantiser never goes there)."""
    import torch
    pos = synth._E4M3_POS.astype(np.float32)
    v = np.concatenate([np.random.default_rng(0).standard_normal(100000).astype(np.float32) * np.float32(60),
                        (pos[:-1] + pos[1:]) / 2, -pos, pos, np.array([0.0, -0.0, 2.0 ** -11, 3 * 2.0 ** -11], np.float32)])
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.f32_to_e4m3(v), ref)
    assert synth.f32_to_e4m3(np.array([1e9, -500.0], np.float32)).tolist() == [0x7E, 0xFE]   # saturates


def test_row_quantisation():
    w = np.random.default_rng(1).standard_normal((64, 256)).astype(np.float32) * np.float32(0.02)
    w[3] = 0
    codes, scale = synth.quantize_rows_e4m3(w)
    assert scale.dtype == np.float32 and scale[3] == 1.0 and np.all(codes[3] == 0)
    live = np.arange(64) != 3
    # the largest magnitude of every row maps to the largest code
    assert np.all((codes[live] & 0x7F).max(axis=1) == 0x7E)
    from oracle import moe_oracle as om
    deq = om.dequant_w8(codes, scale)
    rel = np.abs(deq[live] - w[live]) / (np.abs(w[live]).max(axis=1, keepdims=True))
    # at most half a step of the top binade (256..448, step 32): 16 / 448 of the row's largest magnitude
    assert rel.max() <= 16 / 448 + 1e-7


def test_w8_weights_are_seeded_and_follow_the_bf16_draws():
    w = synth.Workload("q", 4, 128, 4, 2, 64, 64, sigma_router=0.1)
    a = synth.make_expert_weights_w8(w, 3)
    b = synth.make_expert_weights_w8(w, 3)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    from oracle import moe_oracle as om
    wgu, wd = synth.make_expert_weights(w, 3)
    # same draws: the dequantised weights sit within one e4m3 step of the bf16 ones
    d = om.dequant_w8(a[0], a[1]) - om.bf16_to_f64(wgu)
    assert np.abs(d).max() <= 0.07 * np.abs(om.bf16_to_f64(wgu)).max()
