"""Thin Python binding of libmoe_gb300 (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors (or raw integer addresses) for the pointer arguments, passes their
device addresses straight through, and raises MoeError on a non-OK status.
No step of the layer runs in Python.  Loading fails loudly if the compiled
library is absent: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_TIMEOUT = 5
MOE_ERR_DEVICE_INDEX = 6

OP_ROUTE, OP_PERMUTE, OP_EXPERT_FFN_FWD, OP_EXPERT_FFN_BWD, OP_ROUTER_BWD, \
    OP_LAYER_FWD, OP_LAYER_BWD, OP_LAYER_FWD_FP8, OP_LAYER_BWD_FP8 = range(9)

HEADER = os.path.join(_build.ROOT, "include", "moe.h")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("h", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("sar", ctypes.c_int32)]


def dims(T, h, f, E, k, has_bias=False, capacity=0, sar=False) -> moe_dims:
    return moe_dims(int(T), int(h), int(f), int(E), int(k), int(bool(has_bias)), int(capacity),
                    int(bool(sar)))


def dims_of(cfg, has_bias=None, capacity=0, sar=False) -> moe_dims:
    hb = cfg.zipf_s > 0 if has_bias is None else has_bias
    return dims(cfg.T, cfg.h, cfg.f, cfg.E, cfg.k, hb, capacity, sar)


def capacity_for(T, k, E, factor: float) -> int:
    """moe_capacity_for: the per-expert capacity for a capacity factor."""
    c = load().moe_capacity_for(int(T), int(k), int(E), float(factor))
    if c < 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_capacity_for")
    return int(c)


_LIB = None
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_D = ctypes.POINTER(moe_dims)

_SIGS = {
    "moe_workspace_bytes": (_SZ, [_D, _I]),
    "moe_saved_bytes": (_SZ, [_D]),
    "moe_route": (_I, [_D, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_noalloc": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_permute_local": (_I, [_D, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                               _P, _SZ, _P]),
    "moe_unpermute": (_I, [_D, _P, _P, _P, _P]),
    "moe_expert_ffn_fwd": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_combine": (_I, [_D, _P, _P, _P, _P, _P]),
    "moe_expert_ffn_bwd": (_I, [_D] + [_P] * 17 + [_P, _SZ, _P]),
    "moe_router_bwd": (_I, [_D] + [_P] * 11 + [_P, _SZ, _P]),
    "moe_layer_fwd": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_layer_bwd": (_I, [_D] + [_P] * 12 + [_P, _SZ, _P]),
    "moe_saved_view": (_P, [_D, _P, ctypes.c_char_p]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_read_device_status": (_I, [_P, _P]),
    "moe_clear_device_status": (_I, [_P, _P]),
    "moe_profile_events": (_I, [_P, _I]),
    "moe_profile_kernel_name": (ctypes.c_char_p, [_I]),
    "moe_kernel_launches": (ctypes.c_int64, []),
    "moe_test_fail_launch_after": (None, [ctypes.c_int]),
    "moe_selftest_wait_timeout": (_I, [_P, ctypes.c_uint32, _P]),
    "moe_fp8_weight_bytes": (_SZ, [_D]),
    "moe_quantize_weights_fp8": (_I, [_D, _P, _P, _P, _P, _P]),
    "moe_fp8_weight_view": (_P, [_D, _P, ctypes.c_char_p]),
    "moe_quantize_rows_fp8": (_I, [_P, ctypes.c_int64, ctypes.c_int32, _P, ctypes.c_int32,
                                   ctypes.c_int64, _P, _P, _P]),
    "moe_layer_fwd_fp8": (_I, [_D, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_fp8_bwd_weight_bytes": (_SZ, [_D]),
    "moe_quantize_weights_fp8_bwd": (_I, [_D, _P, _P, _P, _P]),
    "moe_fp8_bwd_weight_view": (_P, [_D, _P, ctypes.c_char_p]),
    "moe_layer_bwd_fp8": (_I, [_D] + [_P] * 11 + [_P, _SZ, _P]),
    "moe_version": (ctypes.c_char_p, []),
    "moe_capacity_for": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_double]),
}


def declared_symbols() -> list[str]:
    """Entry points declared in include/moe.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def load(path: str | None = None, build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the compiled library (once).  Raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"libmoe_gb300 not built ({path} missing); run build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _addr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_version() -> str:
    return load().moe_version().decode()


def moe_workspace_bytes(d: moe_dims, op: int) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(d), int(op)))


def moe_saved_bytes(d: moe_dims) -> int:
    return int(load().moe_saved_bytes(ctypes.byref(d)))


def moe_saved_view(d: moe_dims, saved, name: str) -> int:
    """Device address of a named tensor inside a `saved` context."""
    p = load().moe_saved_view(ctypes.byref(d), _addr(saved), name.encode())
    if not p:
        raise MoeError(MOE_ERR_INVALID_ARG, f"moe_saved_view({name})")
    return int(p)


def moe_route(d, x, Wg, b, topk_idx, gates, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_route(ctypes.byref(d), _addr(x), _addr(Wg), _addr(b), _addr(topk_idx),
                            _addr(gates), _addr(ws), ws_bytes, _stream(stream)), "moe_route")


def moe_permute(d, topk_idx, x, counts, offsets, perm_src, perm_dst, x_perm, ws,
                ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_permute(ctypes.byref(d), _addr(topk_idx), _addr(x), _addr(counts),
                              _addr(offsets), _addr(perm_src), _addr(perm_dst), _addr(x_perm),
                              _addr(ws), ws_bytes, _stream(stream)), "moe_permute")


def moe_permute_noalloc(d, topk_idx, x, counts, offsets, perm_src, perm_dst, x_perm,
                        stream=None):
    _check(load().moe_permute_noalloc(ctypes.byref(d), _addr(topk_idx), _addr(x), _addr(counts),
                                      _addr(offsets), _addr(perm_src), _addr(perm_dst),
                                      _addr(x_perm), _stream(stream)), "moe_permute_noalloc")


def moe_permute_local(d, topk_idx, e_lo, e_hi, x, counts, offsets, perm_src, perm_dst, x_perm,
                      ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_permute_local(ctypes.byref(d), _addr(topk_idx), int(e_lo), int(e_hi),
                                    _addr(x), _addr(counts), _addr(offsets), _addr(perm_src),
                                    _addr(perm_dst), _addr(x_perm), _addr(ws), ws_bytes,
                                    _stream(stream)), "moe_permute_local")


def moe_unpermute(d, perm_dst, rows_perm, rows_assign, stream=None):
    _check(load().moe_unpermute(ctypes.byref(d), _addr(perm_dst), _addr(rows_perm),
                                _addr(rows_assign), _stream(stream)), "moe_unpermute")


def moe_expert_ffn_fwd(d, x, perm_src, offsets, W1, W3, W2, A, B, H, O, ws, ws_bytes=None,
                       stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_ffn_fwd(ctypes.byref(d), _addr(x), _addr(perm_src), _addr(offsets),
                                     _addr(W1), _addr(W3), _addr(W2), _addr(A), _addr(B),
                                     _addr(H), _addr(O), _addr(ws), ws_bytes, _stream(stream)),
           "moe_expert_ffn_fwd")


def moe_combine(d, O, gates, perm_dst, y, stream=None):
    _check(load().moe_combine(ctypes.byref(d), _addr(O), _addr(gates), _addr(perm_dst), _addr(y),
                              _stream(stream)), "moe_combine")


def moe_expert_ffn_bwd(d, x, dy, gates, perm_src, offsets, W1, W3, W2, A, B, H, O, dX_perm, dg,
                       dW1, dW3, dW2, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    args = [x, dy, gates, perm_src, offsets, W1, W3, W2, A, B, H, O, dX_perm, dg, dW1, dW3, dW2]
    _check(load().moe_expert_ffn_bwd(ctypes.byref(d), *[_addr(a) for a in args], _addr(ws),
                                     ws_bytes, _stream(stream)), "moe_expert_ffn_bwd")


def moe_router_bwd(d, x, Wg, topk_idx, gates, dg, dX_perm, perm_src, perm_dst, offsets, dx, dWg,
                   ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    args = [x, Wg, topk_idx, gates, dg, dX_perm, perm_src, perm_dst, offsets, dx, dWg]
    _check(load().moe_router_bwd(ctypes.byref(d), *[_addr(a) for a in args], _addr(ws),
                                 ws_bytes, _stream(stream)), "moe_router_bwd")


def moe_layer_fwd(d, x, Wg, b, W1, W3, W2, y, saved, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_layer_fwd(ctypes.byref(d), _addr(x), _addr(Wg), _addr(b), _addr(W1),
                                _addr(W3), _addr(W2), _addr(y), _addr(saved), _addr(ws),
                                ws_bytes, _stream(stream)), "moe_layer_fwd")


def moe_layer_bwd(d, x, dy, Wg, W1, W3, W2, saved, dx, dWg, dW1, dW3, dW2, ws, ws_bytes=None,
                  stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    args = [x, dy, Wg, W1, W3, W2, saved, dx, dWg, dW1, dW3, dW2]
    _check(load().moe_layer_bwd(ctypes.byref(d), *[_addr(a) for a in args], _addr(ws), ws_bytes,
                                _stream(stream)), "moe_layer_bwd")


def moe_read_device_status(ws, stream=None) -> int:
    return int(load().moe_read_device_status(_addr(ws), _stream(stream)))


def moe_clear_device_status(ws, stream=None):
    _check(load().moe_clear_device_status(_addr(ws), _stream(stream)), "moe_clear_device_status")


def moe_profile_events(events_array_addr: int | None, capacity: int) -> int:
    return int(load().moe_profile_events(events_array_addr, int(capacity)))


def moe_profile_kernel_name(i: int) -> str:
    return load().moe_profile_kernel_name(int(i)).decode()


def moe_selftest_wait_timeout(ws, limit_us: int, stream=None):
    _check(load().moe_selftest_wait_timeout(_addr(ws), int(limit_us), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_kernel_launches() -> int:
    return int(load().moe_kernel_launches())


def moe_test_fail_launch_after(n: int) -> None:
    load().moe_test_fail_launch_after(int(n))


def moe_fp8_weight_bytes(d) -> int:
    return int(load().moe_fp8_weight_bytes(ctypes.byref(d)))


def moe_quantize_weights_fp8(d, W1, W3, W2, qw, stream=None):
    _check(load().moe_quantize_weights_fp8(ctypes.byref(d), _addr(W1), _addr(W3), _addr(W2),
                                           _addr(qw), _stream(stream)), "moe_quantize_weights_fp8")


def moe_fp8_weight_view(d, qw, name: str) -> int:
    p = load().moe_fp8_weight_view(ctypes.byref(d), _addr(qw), name.encode())
    if not p:
        raise MoeError(MOE_ERR_INVALID_ARG, f"moe_fp8_weight_view({name})")
    return int(p)


def moe_quantize_rows_fp8(inp, rows, n, idx, div, src_rows, q, scale, stream=None):
    _check(load().moe_quantize_rows_fp8(_addr(inp), int(rows), int(n), _addr(idx), int(div),
                                        int(src_rows), _addr(q), _addr(scale), _stream(stream)),
           "moe_quantize_rows_fp8")


def moe_layer_fwd_fp8(d, x, Wg, b, qw, y, saved, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_layer_fwd_fp8(ctypes.byref(d), _addr(x), _addr(Wg), _addr(b), _addr(qw),
                                    _addr(y), _addr(saved), _addr(ws), ws_bytes, _stream(stream)),
           "moe_layer_fwd_fp8")


def moe_fp8_bwd_weight_bytes(d) -> int:
    return int(load().moe_fp8_bwd_weight_bytes(ctypes.byref(d)))


def moe_quantize_weights_fp8_bwd(d, W1, W3, qwb, stream=None):
    _check(load().moe_quantize_weights_fp8_bwd(ctypes.byref(d), _addr(W1), _addr(W3),
                                               _addr(qwb), _stream(stream)),
           "moe_quantize_weights_fp8_bwd")


def moe_fp8_bwd_weight_view(d, qwb, name: str) -> int:
    p = load().moe_fp8_bwd_weight_view(ctypes.byref(d), _addr(qwb), name.encode())
    if not p:
        raise MoeError(MOE_ERR_INVALID_ARG, f"moe_fp8_bwd_weight_view({name})")
    return int(p)


def moe_layer_bwd_fp8(d, x, dy, Wg, W2, qwb, saved, dx, dWg, dW1, dW3, dW2, ws, ws_bytes=None,
                      stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_layer_bwd_fp8(ctypes.byref(d), _addr(x), _addr(dy), _addr(Wg), _addr(W2),
                                    _addr(qwb),
                                    _addr(saved), _addr(dx), _addr(dWg), _addr(dW1), _addr(dW3),
                                    _addr(dW2), _addr(ws), ws_bytes, _stream(stream)),
           "moe_layer_bwd_fp8")

