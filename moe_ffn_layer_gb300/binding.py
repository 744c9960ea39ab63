"""ctypes binding of the MoE FFN C ABI (``include/moe_ffn.h``).

Argument marshalling only: every function here has the name and argument
order of the C entry point, turns torch tensors into device pointers and
streams into handles, calls the library and raises ``MoEError`` on a non-zero
status.  All work runs in the library's CUDA kernels.  There is no other
implementation to fall back on: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_CUDA", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_DEVICE_CHECK"}


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS.get(code, 'unknown')})")
        self.code = code


class moe_dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int), ("I", ctypes.c_int),
                ("I_s", ctypes.c_int)]


class moe_weights_w8(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p),
                ("s_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("ws_gate_up", ctypes.c_void_p), ("ws_down", ctypes.c_void_p)]


class moe_workspace_offsets(ctypes.Structure):
    _fields_ = [("topk_ids", ctypes.c_size_t), ("topk_w", ctypes.c_size_t), ("expert_offsets", ctypes.c_size_t),
                ("sorted_token", ctypes.c_size_t), ("inv_perm", ctypes.c_size_t)]


class moe_weights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("ws_gate_up", ctypes.c_void_p), ("ws_down", ctypes.c_void_p)]


_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "moe_route_workspace_bytes": (_Z, [_I, _I, _I]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_permute_workspace_bytes": (_Z, [_I, _I]),
    "moe_permute": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_grouped_gemm_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "moe_grouped_gemm": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_grouped_gemm_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_grouped_gemm_w8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _Z, _P]),
    "moe_unpermute_combine": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_workspace_bytes": (_Z, [ctypes.POINTER(moe_dims), _I]),
    "moe_forward": (_I, [ctypes.POINTER(moe_dims), ctypes.POINTER(moe_weights), _P, _I, _P, _P, _Z, _P, _P, _P,
                         _P]),
    "moe_forward_w8": (_I, [ctypes.POINTER(moe_dims), ctypes.POINTER(moe_weights_w8), _P, _I, _P, _P, _Z, _P, _P,
                            _P, _P]),
    "moe_last_device_error": (_I, [_P]),
    "moe_last_launch_count": (_I, []),
    "moe_workspace_layout": (_I, [ctypes.POINTER(moe_dims), _I, ctypes.POINTER(moe_workspace_offsets)]),
    "moe_debug_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"MoE FFN library not built ({path}); run moe_ffn_layer_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def ptr(t) -> int | None:
    """Device pointer of a tensor (None -> NULL); ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def handle(s) -> int | None:
    """cudaStream_t / cudaEvent_t of a torch stream or event (None -> NULL)."""
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    if hasattr(s, "cuda_event"):
        return s.cuda_event
    raise TypeError(f"not a stream or event: {type(s)}")


def _check(fn: str, rc: int) -> int:
    if rc != 0:
        raise MoEError(fn, rc)
    return rc


def moe_route_workspace_bytes(T: int, H: int, E: int) -> int:
    return lib().moe_route_workspace_bytes(T, H, E)


def moe_route(x, w_router, bias, T, H, E, k, topk_ids, topk_w, ws, ws_bytes, stream) -> int:
    return _check("moe_route", lib().moe_route(ptr(x), ptr(w_router), ptr(bias), T, H, E, k, ptr(topk_ids),
                                               ptr(topk_w), ptr(ws), ws_bytes, handle(stream)))


def moe_permute_workspace_bytes(T: int, E: int) -> int:
    return lib().moe_permute_workspace_bytes(T, E)


def moe_permute(topk_ids, x, T, H, E, k, expert_offsets, sorted_token, inv_perm, x_perm, ws, ws_bytes,
                stream) -> int:
    return _check("moe_permute", lib().moe_permute(ptr(topk_ids), ptr(x), T, H, E, k, ptr(expert_offsets),
                                                   ptr(sorted_token), ptr(inv_perm), ptr(x_perm), ptr(ws),
                                                   ws_bytes, handle(stream)))


def moe_grouped_gemm_workspace_bytes(G, rows_max, N, K, act) -> int:
    return lib().moe_grouped_gemm_workspace_bytes(G, rows_max, N, K, act)


def moe_grouped_gemm(a, w, group_offsets, G, rows_max, N, K, act, out, ws, ws_bytes, stream) -> int:
    return _check("moe_grouped_gemm", lib().moe_grouped_gemm(ptr(a), ptr(w), ptr(group_offsets), G, rows_max, N, K,
                                                             act, ptr(out), ptr(ws), ws_bytes, handle(stream)))


def moe_grouped_gemm_noalloc(a, w, group_offsets, G, rows_max, N, K, act, out, stream) -> int:
    return _check("moe_grouped_gemm_noalloc", lib().moe_grouped_gemm_noalloc(ptr(a), ptr(w), ptr(group_offsets), G,
                                                                             rows_max, N, K, act, ptr(out),
                                                                             handle(stream)))


def moe_grouped_gemm_w8(a, w, w_scale, group_offsets, G, rows_max, N, K, act, out, ws, ws_bytes, stream) -> int:
    return _check("moe_grouped_gemm_w8", lib().moe_grouped_gemm_w8(ptr(a), ptr(w), ptr(w_scale), ptr(group_offsets),
                                                                   G, rows_max, N, K, act, ptr(out), ptr(ws),
                                                                   ws_bytes, handle(stream)))


def moe_unpermute_combine(y, inv_perm, topk_w, shared, T, H, k, out, stream) -> int:
    return _check("moe_unpermute_combine", lib().moe_unpermute_combine(ptr(y), ptr(inv_perm), ptr(topk_w),
                                                                       ptr(shared), T, H, k, ptr(out),
                                                                       handle(stream)))


def moe_workspace_bytes(dims: moe_dims, T: int) -> int:
    return lib().moe_workspace_bytes(ctypes.byref(dims), T)


def moe_forward(dims: moe_dims, weights: moe_weights, x, T, out, ws, ws_bytes, stream, side, ev_fork,
                ev_join) -> int:
    return _check("moe_forward", lib().moe_forward(ctypes.byref(dims), ctypes.byref(weights), ptr(x), T, ptr(out),
                                                   ptr(ws), ws_bytes, handle(stream), handle(side),
                                                   handle(ev_fork), handle(ev_join)))


def moe_forward_w8(dims: moe_dims, weights: moe_weights_w8, x, T, out, ws, ws_bytes, stream, side, ev_fork,
                   ev_join) -> int:
    return _check("moe_forward_w8", lib().moe_forward_w8(ctypes.byref(dims), ctypes.byref(weights), ptr(x), T,
                                                         ptr(out), ptr(ws), ws_bytes, handle(stream), handle(side),
                                                         handle(ev_fork), handle(ev_join)))


def moe_last_device_error(stream) -> int:
    return lib().moe_last_device_error(handle(stream))


def moe_last_launch_count() -> int:
    return lib().moe_last_launch_count()


def moe_workspace_layout(dims: moe_dims, T: int) -> moe_workspace_offsets:
    out = moe_workspace_offsets()
    _check("moe_workspace_layout", lib().moe_workspace_layout(ctypes.byref(dims), T, ctypes.byref(out)))
    return out


def moe_debug_set_wait_limit_ns(ns: int) -> int:
    return _check("moe_debug_set_wait_limit_ns", lib().moe_debug_set_wait_limit_ns(ns))
