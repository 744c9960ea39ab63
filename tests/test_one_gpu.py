"""bench.py runs on one GPU only: asked for more (--gpus N or WORLD_SIZE > 1),
it prints one 'unavailable' line and exits 0 before it builds or loads the
library (the layer does not shard, and its prefill matmuls multicast operand
tiles inside clusters of one GPU).  The whole-job arithmetic of one rank."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       env=env, timeout=120, cwd=ROOT)
    return r


@pytest.mark.parametrize("args,env", [(["--gpus", "2"], {}), (["--gpus", "8", "--steps", "3"], {}),
                                      ([], {"WORLD_SIZE": "2", "RANK": "0"})])
def test_more_than_one_gpu_is_refused_before_loading(args, env):
    r = _run(args, env)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert "unavailable" in d and "one GPU" in d["unavailable"] and "value" not in d
    # nothing was built or imported: the refusal comes before torch and the library
    assert "Traceback" not in r.stderr


def test_other_ranks_print_nothing():
    r = _run([], {"WORLD_SIZE": "2", "RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_tokens_per_second_of_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.tokens_per_s(16, 10, 4.0) == pytest.approx(10 * 16 / 4e-3)


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    from moe_ffn_layer_gb300 import synth
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=0, seed=0, gpus=2))()
    assert bench.run_reference(args, synth.workload("tiny")) is None
