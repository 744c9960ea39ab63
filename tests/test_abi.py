"""The C-ABI library builds, loads without a GPU, exports exactly the entry
points the header declares, and rejects bad arguments on the host before any
launch (every call here returns before touching the device)."""
import ctypes
import os
import re
import subprocess

import pytest

from moe_ffn_layer_gb300 import binding as B
from moe_ffn_layer_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_ffn.h")


def header_functions():
    src = open(HEADER).read()
    return set(re.findall(r"^MOE_API\s+\w+\s+(moe_\w+)\(", src, flags=re.M))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def test_header_declares_the_five_calls():
    names = header_functions()
    for n in ["moe_route", "moe_permute", "moe_grouped_gemm", "moe_unpermute_combine", "moe_forward"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.library_path()], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert exported == names, exported ^ names
    assert set(B._SIGS) == names


def test_workspace_queries(lib):
    d = B.moe_dims(2048, 128, 8, 768, 2048)
    small = B.moe_workspace_bytes(d, 1)
    big = B.moe_workspace_bytes(d, 8192)
    assert 0 < small < big
    # holds at least x_perm, h and y of the routed path (bf16)
    Tk = 8192 * 8
    assert big >= Tk * (2048 + 768 + 2048) * 2
    assert big % 256 == 0
    assert B.moe_workspace_bytes(B.moe_dims(2048, 128, 8, 700, 2048), 1) == 0   # I % 64 != 0
    assert B.moe_route_workspace_bytes(16, 2048, 128) >= 16 * 128 * 4
    assert B.moe_permute_workspace_bytes(256, 128) == 0          # one-block path needs none
    assert B.moe_permute_workspace_bytes(4096, 128) >= 16 * 128 * 4
    # split-K scratch only for the weights-on-M form (few rows per group)
    assert B.moe_grouped_gemm_workspace_bytes(128, 64, 768, 2048, 1) > 0
    assert B.moe_grouped_gemm_workspace_bytes(128, 65536, 768, 2048, 1) == 0
    assert B.moe_grouped_gemm_workspace_bytes(128, 64, 768, 2048, 1) >= 128 * 64 * 4


def test_workspace_layout(lib):
    """The regions where the layer forward leaves its routing and dispatch lie
    inside its workspace, 256-byte aligned, large enough and disjoint."""
    for dims, T in [(B.moe_dims(2048, 128, 8, 768, 2048), 8), (B.moe_dims(256, 8, 2, 128, 256), 16),
                    (B.moe_dims(2048, 128, 8, 768, 2048), 8192), (B.moe_dims(256, 8, 2, 128, 0), 1)]:
        total = B.moe_workspace_bytes(dims, T)
        o = B.moe_workspace_layout(dims, T)
        Tk = T * dims.k
        regions = sorted([(o.topk_ids, Tk * 4), (o.topk_w, Tk * 4), (o.expert_offsets, (dims.E + 1) * 4),
                          (o.sorted_token, Tk * 4), (o.inv_perm, Tk * 4)])
        for (a, n), (b, _) in zip(regions, regions[1:]):
            assert a + n <= b
        for a, n in regions:
            assert a % 256 == 0 and a + n <= total
    assert _rc(B.moe_workspace_layout, B.moe_dims(2048, 128, 8, 700, 2048), 8) == -2
    assert _rc(B.moe_workspace_layout, B.moe_dims(2048, 128, 8, 768, 2048), -1) == -1


def test_wait_limit_setter_needs_no_device(lib):
    assert B.moe_debug_set_wait_limit_ns(0) == 0
    assert B.moe_debug_set_wait_limit_ns(2_000_000_000) == 0


def _rc(fn, *args):
    with pytest.raises(B.MoEError) as e:
        fn(*args)
    return e.value.code


def test_host_side_argument_checks(lib):
    INVALID, UNSUP = -1, -2
    fake = 1 << 20    # never dereferenced: every call below returns before a launch
    # grouped GEMM: N, K multiples of 64; act 0/1; groups need offsets unless G == 1
    assert _rc(B.moe_grouped_gemm, fake, fake, fake, 8, 64, 100, 64, 0, fake, None, 0, None) == UNSUP
    assert _rc(B.moe_grouped_gemm, fake, fake, fake, 8, 64, 128, 96, 0, fake, None, 0, None) == UNSUP
    assert _rc(B.moe_grouped_gemm, fake, fake, fake, 8, 64, 128, 64, 2, fake, None, 0, None) == INVALID
    assert _rc(B.moe_grouped_gemm, fake, fake, None, 8, 64, 128, 64, 0, fake, None, 0, None) == INVALID
    assert _rc(B.moe_grouped_gemm, fake, fake, fake, 2000, 64, 128, 64, 0, fake, None, 0, None) == UNSUP
    assert _rc(B.moe_grouped_gemm, fake + 8, fake, fake, 8, 64, 128, 64, 0, fake, None, 0, None) == UNSUP
    assert B.moe_grouped_gemm(fake, fake, fake, 8, 0, 128, 64, 0, fake, None, 0, None) == 0    # no rows: no-op
    # split-K scratch must be 256-byte aligned
    assert _rc(B.moe_grouped_gemm, fake, fake, fake, 8, 64, 128, 64, 0, fake, fake + 16, 1 << 20, None) == UNSUP
    # router: k <= E, E <= 512, k <= 16, H % 8
    assert _rc(B.moe_route, fake, fake, None, 4, 64, 8, 9, fake, fake, fake, 1 << 20, None) == INVALID
    assert _rc(B.moe_route, fake, fake, None, 4, 64, 1024, 8, fake, fake, fake, 1 << 20, None) == UNSUP
    assert _rc(B.moe_route, fake, fake, None, 4, 64, 64, 17, fake, fake, fake, 1 << 20, None) == UNSUP
    assert _rc(B.moe_route, fake, fake, None, 4, 60, 64, 8, fake, fake, fake, 1 << 20, None) == UNSUP
    assert _rc(B.moe_route, fake, fake, None, 4, 64, 64, 8, fake, fake, fake, 16, None) == -3   # workspace
    assert B.moe_route(None, None, None, 0, 64, 64, 8, None, None, None, 0, None) == 0      # T == 0
    # permute
    assert _rc(B.moe_permute, fake, fake, 4, 64, 8, 9, fake, fake, fake, fake, None, 0, None) == INVALID
    assert _rc(B.moe_permute, fake, fake, 4, 60, 8, 2, fake, fake, fake, fake, None, 0, None) == UNSUP
    assert _rc(B.moe_permute, fake, fake, 4096, 64, 8, 2, fake, fake, fake, fake, None, 0, None) == -3
    # combine
    assert _rc(B.moe_unpermute_combine, fake, fake, fake, None, 4, 60, 2, fake, None) == UNSUP
    assert _rc(B.moe_unpermute_combine, fake, fake, fake, None, 4, 64, 17, fake, None) == UNSUP
    assert _rc(B.moe_unpermute_combine, None, fake, fake, None, 4, 64, 2, fake, None) == INVALID
    # forward: shapes, missing shared-expert plumbing, workspace
    w = B.moe_weights(fake, None, fake, fake, fake, fake)
    assert _rc(B.moe_forward, B.moe_dims(2048, 128, 8, 700, 2048), w, fake, 1, fake, fake, 1 << 30,
               fake, fake, fake, fake) == UNSUP
    assert _rc(B.moe_forward, B.moe_dims(2048, 128, 8, 768, 2048), w, fake, 1, fake, fake, 1 << 30,
               fake, None, fake, fake) == INVALID
    assert _rc(B.moe_forward, B.moe_dims(2048, 128, 8, 768, 2048), w, fake, 1, fake, fake, 64,
               fake, fake, fake, fake) == -3
    assert B.moe_forward(B.moe_dims(2048, 128, 8, 768, 2048), w, None, 0, None, None, 0, None, None, None,
                         None) == 0


def test_w8_calls_refuse_shapes_outside_the_weight_stream(lib):
    """FP8 weights serve the weights-on-M (decode-sized) shapes: larger batches
    are refused on the host, before anything is launched."""
    fake = 1 << 20
    # 300 rows over 2 groups: more than 64 rows per group -> tokens-on-M
    assert _rc(B.moe_grouped_gemm_w8, fake, fake, fake, fake, 2, 300, 256, 128, 1, fake, None, 0, None) == -2
    assert _rc(B.moe_grouped_gemm_w8, fake, fake, None, fake, 2, 64, 256, 128, 1, fake, None, 0, None) == -1
    d = B.moe_dims(2048, 128, 8, 768, 2048)
    w8 = B.moe_weights_w8(fake, None, fake, fake, fake, fake, fake, fake)
    assert _rc(B.moe_forward_w8, d, w8, fake, 8192, fake, fake, 1 << 40, fake, fake, fake, fake) == -2   # prefill
    no_scales = B.moe_weights_w8(fake, None, fake, None, fake, None, fake, fake)
    assert _rc(B.moe_forward_w8, d, no_scales, fake, 8, fake, fake, 1 << 30, fake, fake, fake, fake) == -1


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.moe_last_launch_count()
