"""Host-side pieces of bench.py that need no GPU: the algorithmic units the
roofline fractions divide by, and the reference arm (the CPU oracle) on a
bounded sample."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_ffn_layer_gb300 import synth  # noqa: E402


def test_layer_units_decode_t1():
    """Decode T=1 with 8 non-empty experts: 6*H*I*8 + 6*H*I_s + 4*E*H + 4*T*H bytes."""
    w = synth.workload("decode", 1)
    b, f = bench.layer_units(w, 8)
    assert b == 6 * 2048 * 768 * 8 + 6 * 2048 * 2048 + 4 * 128 * 2048 + 4 * 2048
    assert b == 101_720_064
    assert f == 2 * 8 * 3 * 2048 * 768 + 2 * 3 * 2048 * 2048 + 2 * 128 * 2048


def test_gate_up_units_prefill():
    w = synth.workload("prefill")
    b, f = bench.gate_up_units(w, 128)
    rows = 8192 * 8
    assert f == 2 * rows * 2 * 768 * 2048          # 412.3 GFLOP
    assert b == 128 * 2 * 768 * 2048 * 2 + rows * 2048 * 2 + rows * 768 * 2


def test_routed_units_drop_the_shared_expert():
    w = synth.workload("decode", 1)
    b, f = bench.routed_units(w, 8)
    lb, lf = bench.layer_units(w, 8)
    assert lb - b == 6 * 2048 * 2048 and lf - f == 2 * 3 * 2048 * 2048


def test_weight_copies_defeat_l2():
    for name, T in bench.SWEEP:
        w = synth.workload(name, T)
        R, touched = bench.weight_copies(w)
        assert 2 <= R <= 16 and (R * touched >= 4 * bench.L2_BYTES or R == 16)


def test_reference_arm_runs_the_oracle(monkeypatch):
    monkeypatch.setenv("RANK", "0")
    args = type("A", (), dict(steps=2, warmup=1, seed=0, gpus=1))()
    w = synth.workload("tiny")
    r = bench.run_reference(args, w)
    assert r["impl"] == "reference" and r["unit"] == "tokens/s" and r["value"] > 0
    assert r["cpu_baseline"]["kind"] == "oracle" and r["e2e"]["h2d_bytes_per_step"] == 0
    # the reference arm reports the same config dict as the GPU arm
    assert r["config"] == bench.config_of(w)
