"""The bounded-wait path, on the GPU without a fault.  With the wait limit at 0
every wait that is not already complete expires at once: the grouped matmul
records MOE_ERR_TIMEOUT, drains the copies it issued, frees its tensor memory
and exits without writing its output.  With the limit restored, the next call
gives the same bits as before (for the layer, once its workspace is zeroed
again, as after any device error)."""
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

DEFAULT_NS = 2_000_000_000
TIMEOUT = -5


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield B.lib()
    B.moe_debug_set_wait_limit_ns(DEFAULT_NS)


@pytest.mark.parametrize("rows,N,K,act", [([8], 128, 1024, 1), ([5], 128, 2048, 0)])
def test_wait_limit_expires_and_next_call_is_clean(rows, N, K, act):
    """One group of a few rows and one 128-row weight block: the weights-on-M
    form on a single CTA (no pair, no split)."""
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    a_bits = synth.random_bf16((R, K), seed=R + K, tag=81)
    w_bits = synth.random_bf16((G, 2 * N if act else N, K), seed=N, tag=82, sigma=0.05)
    a, w = bf16_tensor(a_bits, "cuda"), bf16_tensor(w_bits, "cuda")
    offs = torch.from_numpy(off).cuda()
    s = torch.cuda.current_stream()
    fresh = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm(a, w, offs, G, R, N, K, act, fresh, None, 0, s)
    assert B.moe_last_device_error(s) == 0
    assert_close_layer(to_f64(fresh), om.grouped_gemm(a_bits, w_bits, off, act), "before")

    out = torch.full((R, N), 5.0, dtype=torch.bfloat16, device="cuda")
    try:
        B.moe_debug_set_wait_limit_ns(0)
        B.moe_grouped_gemm(a, w, offs, G, R, N, K, act, out, None, 0, s)
    finally:
        B.moe_debug_set_wait_limit_ns(DEFAULT_NS)
    assert B.moe_last_device_error(s) == TIMEOUT
    assert B.moe_last_device_error(s) == 0          # the read cleared it
    assert torch.all(out == 5.0)                     # the abandoned launch wrote nothing

    again = torch.empty_like(fresh)
    B.moe_grouped_gemm(a, w, offs, G, R, N, K, act, again, None, 0, s)
    assert B.moe_last_device_error(s) == 0
    assert torch.equal(again.view(torch.int16), fresh.view(torch.int16))


def test_layer_forward_after_a_timeout_is_clean():
    wl = synth.Workload("dec", 4, 512, 16, 4, 256, 128, sigma_router=0.1, sigma_w=0.03)
    inp = synth.make_inputs(wl, 19)
    L = MoEFFN.from_inputs(inp, wl.k, "cuda")
    x = bf16_tensor(inp["x"], "cuda")
    s = torch.cuda.current_stream()
    fresh = L.forward(x).clone()
    assert B.moe_last_device_error(s) == 0
    assert_close_layer(to_f64(fresh), om.forward(inp, wl.k)["out"], "before")
    try:
        B.moe_debug_set_wait_limit_ns(0)
        L.forward(x)
    finally:
        B.moe_debug_set_wait_limit_ns(DEFAULT_NS)
    assert B.moe_last_device_error(s) == TIMEOUT
    # after a device error the workspace is zeroed again (split-K tickets of the
    # abandoned shared-expert matmuls may be left taken)
    L.workspace(wl.T).zero_()
    again = L.forward(x)
    assert B.moe_last_device_error(s) == 0
    assert torch.equal(again.view(torch.int16), fresh.view(torch.int16))
