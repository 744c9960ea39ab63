"""moe_grouped_gemm_noalloc: the grouped matmul for callers that cannot
allocate device memory (its split-K scratch is a fixed array inside the
library).  Its output must match moe_grouped_gemm's on the same inputs, call
after call, since every call reuses the same array, and the float64 oracle
within the layer's tolerance.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from cases import assert_close_layer, to_f64
from moe_ffn_layer_gb300 import binding as B
from moe_ffn_layer_gb300 import build as build_mod
from moe_ffn_layer_gb300 import synth
from moe_ffn_layer_gb300.layer import bf16_tensor
from oracle import moe_oracle as om

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return B.lib()


CASES = [
    # (rows per group, N, K, act): decode-like groups of a few rows (split-K
    # runs in the fixed scratch), a down-like shape, and groups too large to split
    ([1, 2, 0, 1, 3, 1, 0, 2, 1, 1, 4, 0, 1, 2, 1, 1], 768, 2048, 1),
    ([1, 2, 0, 1, 3, 1, 0, 2, 1, 1, 4, 0, 1, 2, 1, 1], 2048, 768, 0),
    ([8] * 16, 384, 1024, 1),
    ([300, 0, 129], 256, 192, 1),
    ([1] * 64, 2048, 768, 0),   # 1024 units of one row each
]


@pytest.mark.parametrize("rows,N,K,act", CASES)
def test_noalloc_matches_grouped_gemm(rows, N, K, act):
    G = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    a_bits = synth.random_bf16((R, K), seed=R + K, tag=61)
    w_bits = synth.random_bf16((G, 2 * N if act else N, K), seed=N + G, tag=62, sigma=0.03)
    a = bf16_tensor(a_bits, "cuda")
    w = bf16_tensor(w_bits, "cuda")
    oracle = om.grouped_gemm(a_bits, w_bits, off, act)
    offs = torch.from_numpy(off).cuda()
    s = torch.cuda.current_stream()
    nb = B.moe_grouped_gemm_workspace_bytes(G, R, N, K, act)
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
    ref = torch.empty((R, N), dtype=torch.bfloat16, device="cuda")
    B.moe_grouped_gemm(a, w, offs, G, R, N, K, act, ref, ws, nb, s)
    n_ref = B.moe_last_launch_count()
    ref64 = to_f64(ref)
    outs = []
    for _ in range(2):   # two calls in a row on the same fixed scratch
        out = torch.full((R, N), 3.0, dtype=torch.bfloat16, device="cuda")
        B.moe_grouped_gemm_noalloc(a, w, offs, G, R, N, K, act, out, s)
        assert B.moe_last_launch_count() == n_ref >= 1
        assert B.moe_last_device_error(s) == 0
        got = to_f64(out)
        assert_close_layer(got, ref64, f"noalloc rows={rows} N={N} K={K} act={act}")
        assert_close_layer(got, oracle, f"noalloc vs oracle rows={rows} N={N} K={K} act={act}")
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_noalloc_refuses_bad_arguments_before_launch():
    """Argument errors are refused on the host, before anything is launched
    (the pointers below are never dereferenced)."""
    fake = 1 << 20
    for args, code in [
        ((fake, fake, fake, 0, 16, 256, 64, 1, fake, None), -1),       # no groups
        ((fake, fake, None, 4, 16, 256, 64, 1, fake, None), -1),       # several groups need offsets
        ((fake, fake, fake, 4, 16, 200, 64, 1, fake, None), -2),       # N not a multiple of 64
        ((fake, fake, fake, 4, 16, 256, 96, 1, fake, None), -2),       # K not a multiple of 64
        ((fake + 8, fake, fake, 4, 16, 256, 64, 1, fake, None), -2),   # A not 16-byte aligned
    ]:
        with pytest.raises(B.MoEError) as e:
            B.moe_grouped_gemm_noalloc(*args)
        assert e.value.code == code, args

