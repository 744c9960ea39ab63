"""A MoE FFN layer held on one CUDA device: its weights, the side stream and the
two events of the shared-expert fork/join, and a workspace sized for the
largest batch seen so far.  PyTorch provides the memory, streams and events;
``forward`` is one call of the C entry point ``moe_forward``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """bf16 tensor from uint16 bit patterns (no rounding)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


class MoEFFN:
    """Weights (device tensors): w_router fp32 [E,H]; router_bias fp32 [E] or
    None; w_gate_up bf16 [E,2I,H]; w_down bf16 [E,H,I]; ws_gate_up bf16
    [2I_s,H] and ws_down bf16 [H,I_s], or None for a layer without a shared
    expert.  With s_gate_up fp32 [E,2I] and s_down fp32 [E,H] the routed
    weights are e4m3 codes (uint8 tensors of the same shapes) with one scale
    per weight row, and forward() calls moe_forward_w8."""

    def __init__(self, k: int, w_router, router_bias, w_gate_up, w_down, ws_gate_up=None, ws_down=None,
                 s_gate_up=None, s_down=None):
        E, twoI, H = w_gate_up.shape
        I_s = 0 if ws_gate_up is None else ws_gate_up.shape[0] // 2
        self.H, self.E, self.k, self.I, self.I_s = H, E, k, twoI // 2, I_s
        self.device = w_gate_up.device
        self.tensors = (w_router, router_bias, w_gate_up, w_down, ws_gate_up, ws_down)
        self.scales = None if s_gate_up is None else (s_gate_up, s_down)
        self.dims = B.moe_dims(H, E, k, twoI // 2, I_s)
        if self.scales is None:
            self.weights = B.moe_weights(*(B.ptr(t) for t in self.tensors))
        else:
            self.weights = B.moe_weights_w8(*(B.ptr(t) for t in (w_router, router_bias, w_gate_up, s_gate_up, w_down,
                                                                 s_down, ws_gate_up, ws_down)))
        self.side = torch.cuda.Stream(self.device)
        self.ev_fork = torch.cuda.Event()
        self.ev_join = torch.cuda.Event()
        # torch creates an event's CUDA object on its first record
        s = torch.cuda.current_stream(self.device)
        self.ev_fork.record(s)
        self.ev_join.record(s)
        self._ws = None

    @classmethod
    def from_inputs(cls, inp: dict, k: int, device="cuda") -> "MoEFFN":
        """From the numpy arrays of ``synth.make_inputs`` (bf16 as uint16 bits)
        or ``synth.make_inputs_w8`` (e4m3 codes as uint8 with row scales)."""
        f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
        b16 = lambda a: None if a is None else bf16_tensor(a, device)
        if "w_gate_up_scale" in inp:
            u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.uint8)).to(device)
            return cls(k, f32(inp["w_router"]), f32(inp["bias"]), u8(inp["w_gate_up"]), u8(inp["w_down"]),
                       b16(inp["ws_gate_up"]), b16(inp["ws_down"]), f32(inp["w_gate_up_scale"]),
                       f32(inp["w_down_scale"]))
        return cls(k, f32(inp["w_router"]), f32(inp["bias"]), b16(inp["w_gate_up"]), b16(inp["w_down"]),
                   b16(inp["ws_gate_up"]), b16(inp["ws_down"]))

    def workspace_bytes(self, T: int) -> int:
        return B.moe_workspace_bytes(self.dims, T)

    def workspace(self, T: int) -> torch.Tensor:
        """Workspace for batches of up to T tokens, zero-filled when allocated
        (the library keeps its scratch counters zero from call to call)."""
        need = self.workspace_bytes(T)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """out[T,H] bf16 = MoE FFN layer of x[T,H] bf16, launched on `stream`
        (default: the current stream) with the shared expert on the side stream."""
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device)
        stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        ws = self.workspace(T)
        call = B.moe_forward if self.scales is None else B.moe_forward_w8
        call(self.dims, self.weights, x, T, out, ws, ws.numel(), stream, self.side, self.ev_fork, self.ev_join)
        return out

    __call__ = forward
