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
