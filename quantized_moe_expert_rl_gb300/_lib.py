"""ctypes binding of librlmoe.so (include/rl_moe.h).

Argument marshalling only: every function here has the name of a C entry point, turns
tensors (or None) into raw pointers, calls the library, and raises RlError on a non-OK
status.  All compute happens in the CUDA kernels.  The library must have been built
(`quantized_moe_expert_rl_gb300.build.build()`); loading fails loudly if it is missing.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

RL_OK, RL_ERR_INVALID, RL_ERR_UNSUPPORTED, RL_ERR_CUDA, RL_ERR_TIMEOUT = 0, 1, 2, 3, 4
RL_NO_EARLY_OUT = 0x7FFFFFFF
RL_DEVERR_SLOT_ALIGN, RL_DEVERR_WAIT_TIMEOUT, RL_DEVERR_BAD_ID, RL_DEVERR_MISSING, RL_DEVERR_RANGE = 1, 2, 4, 8, 16
RL_DEVERR_NAN = 32
STATUS_NAMES = {0: "RL_OK", 1: "RL_ERR_INVALID", 2: "RL_ERR_UNSUPPORTED", 3: "RL_ERR_CUDA", 4: "RL_ERR_TIMEOUT"}

# every symbol include/rl_moe.h declares
EXPORTS = ("rl_abi_version", "rl_last_error", "rl_record_bytes", "rl_rmsnorm", "rl_route_workspace_bytes",
           "rl_route", "rl_resolve_slots", "moe_decode_workspace_bytes", "moe_decode",
           "rl_build_pairs_workspace_bytes", "rl_build_pairs", "moe_prefill_workspace_bytes",
           "moe_prefill_chunk", "moe_prefill_chunk_f32", "moe_decode_static", "moe_decode_stack_workspace_bytes",
           "moe_decode_stack", "rl_fill_workspace_bytes", "rl_fill_missing", "rl_host_device_pointer",
           "moe_decode_stack_fill", "moe_decode_layer")


class RlShape(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("n_layers", ctypes.c_int32)]

    @classmethod
    def of(cls, hidden, n_experts, top_k, inter, n_layers):
        return cls(hidden, n_experts, top_k, inter, n_layers)


class RlError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load librlmoe.so (no fallback: raises if the CUDA library was not built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library {p} not built; run quantized_moe_expert_rl_gb300.build.build()")
    L = ctypes.CDLL(p)
    i32, u64p, vp, sz, f32 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    shp = ctypes.POINTER(RlShape)
    sig = {
        "rl_abi_version": (i32, []),
        "rl_last_error": (ctypes.c_char_p, []),
        "rl_record_bytes": (sz, [shp]),
        "rl_rmsnorm": (i32, [vp, vp, i32, i32, f32, vp]),
        "rl_route_workspace_bytes": (sz, [shp, i32]),
        "rl_route": (i32, [shp, i32, i32, vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "rl_resolve_slots": (i32, [shp, i32, i32, vp, vp, vp, vp]),
        "moe_decode_workspace_bytes": (sz, [shp]),
        "moe_decode": (i32, [shp, i32, vp, f32, vp, vp, vp, vp, i32, vp, vp, sz, vp]),
        "moe_decode_static": (i32, [shp, i32, vp, f32, vp, vp, vp, vp, i32, vp, vp]),
        "moe_decode_stack_workspace_bytes": (sz, [shp]),
        "moe_decode_stack": (i32, [shp, i32, i32, vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, sz,
                                   vp]),
        "rl_build_pairs_workspace_bytes": (sz, [shp, i32]),
        "rl_build_pairs": (i32, [shp, i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_prefill_workspace_bytes": (sz, [shp, i32]),
        "moe_prefill_chunk": (i32, [shp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, sz, vp]),
        "moe_prefill_chunk_f32": (i32, [shp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, sz, vp]),
        "moe_decode_stack_fill": (i32, [shp, i32, i32, vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        vp, vp, sz, vp]),
        "moe_decode_layer": (i32, [shp, i32, vp, f32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "rl_fill_workspace_bytes": (sz, [shp]),
        "rl_fill_missing": (i32, [shp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "rl_host_device_pointer": (i32, [vp, ctypes.POINTER(ctypes.c_uint64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    del u64p
    if path is None:
        _lib = L
    return L


def ptr(t) -> int | None:
    """Raw address of a device tensor / int / None (NULL).  The library reads every buffer as
    a dense array on the device, so a strided view or a host tensor is refused here rather
    than read wrongly."""
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {t.stride()} is not contiguous")
    if t.device.type != "cuda":
        raise ValueError(f"tensor on {t.device} passed where a device buffer is expected")
    return t.data_ptr() or None


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check(fn: str, st: int) -> None:
    if st != RL_OK:
        raise RlError(st, fn, load().rl_last_error().decode())


def rl_abi_version() -> int:
    return load().rl_abi_version()


def rl_record_bytes(shape: RlShape) -> int:
    return load().rl_record_bytes(ctypes.byref(shape))


def rl_rmsnorm(x, xn, T, H, eps, stream=None):
    _check("rl_rmsnorm", load().rl_rmsnorm(ptr(x), ptr(xn), T, H, eps, _stream(stream)))


def rl_route_workspace_bytes(shape, T) -> int:
    return load().rl_route_workspace_bytes(ctypes.byref(shape), T)


def rl_route(shape, layer, T, x, norm_eps, w_router, bias, residency, ids, weights, slots, miss, ctrl,
             logits_out=None, ws=None, ws_bytes=0, stream=None):
    _check("rl_route", load().rl_route(ctypes.byref(shape), layer, T, ptr(x), float(norm_eps), ptr(w_router), ptr(bias),
                                       ptr(residency), ptr(ids), ptr(weights), ptr(slots), ptr(miss), ptr(ctrl),
                                       ptr(logits_out), ptr(ws), ws_bytes, _stream(stream)))


def rl_fill_workspace_bytes(shape) -> int:
    return load().rl_fill_workspace_bytes(ctypes.byref(shape))


def rl_fill_missing(shape, layer, T, ids, slots, residency, src, dst, filled, first_early_out, ctrl, ws, ws_bytes,
                    stream=None):
    _check("rl_fill_missing", load().rl_fill_missing(ctypes.byref(shape), layer, T, ptr(ids), ptr(slots),
                                                     ptr(residency), ptr(src), ptr(dst), ptr(filled),
                                                     ptr(first_early_out), ptr(ctrl), ptr(ws), ws_bytes,
                                                     _stream(stream)))


def rl_host_device_pointer(host_ptr: int) -> int:
    out = ctypes.c_uint64(0)
    _check("rl_host_device_pointer", load().rl_host_device_pointer(host_ptr, ctypes.byref(out)))
    return int(out.value)


def rl_resolve_slots(shape, layer, T, ids, residency, slots, stream=None):
    _check("rl_resolve_slots", load().rl_resolve_slots(ctypes.byref(shape), layer, T, ptr(ids), ptr(residency),
                                                       ptr(slots), _stream(stream)))


def moe_decode_workspace_bytes(shape) -> int:
    return load().moe_decode_workspace_bytes(ctypes.byref(shape))


def moe_decode(shape, layer, x, norm_eps, slots, weights, codebook, y, accumulate, ctrl, ws, ws_bytes, stream=None):
    _check("moe_decode", load().moe_decode(ctypes.byref(shape), layer, ptr(x), float(norm_eps), ptr(slots), ptr(weights),
                                           ptr(codebook), ptr(y), int(accumulate), ptr(ctrl), ptr(ws), ws_bytes,
                                           _stream(stream)))


def moe_decode_static(shape, layer, x, norm_eps, slots, weights, codebook, y, accumulate, ctrl, stream=None):
    _check("moe_decode_static", load().moe_decode_static(ctypes.byref(shape), layer, ptr(x), float(norm_eps),
                                                         ptr(slots), ptr(weights), ptr(codebook), ptr(y),
                                                         int(accumulate), ptr(ctrl), _stream(stream)))


def moe_decode_stack_workspace_bytes(shape) -> int:
    return load().moe_decode_stack_workspace_bytes(ctypes.byref(shape))


def moe_decode_stack(shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids, weights, slots,
                     miss, ctrl, logits_out, x_hist, pregate, pregate_hits, ws, ws_bytes, stream=None):
    _check("moe_decode_stack", load().moe_decode_stack(
        ctypes.byref(shape), layer0, n_layers, ptr(x), float(norm_eps), ptr(w_router), ptr(bias), ptr(residency),
        ptr(codebook), ptr(ids), ptr(weights), ptr(slots), ptr(miss), ptr(ctrl), ptr(logits_out), ptr(x_hist),
        int(pregate), ptr(pregate_hits), ptr(ws), ws_bytes, _stream(stream)))


def moe_decode_stack_fill(shape, layer0, n_layers, x, norm_eps, w_router, bias, residency, codebook, ids, weights,
                          slots, miss, ctrl, logits_out, x_hist, fill_src, fill_dst, filled, ws, ws_bytes, stream=None):
    _check("moe_decode_stack_fill", load().moe_decode_stack_fill(
        ctypes.byref(shape), layer0, n_layers, ptr(x), float(norm_eps), ptr(w_router), ptr(bias), ptr(residency),
        ptr(codebook), ptr(ids), ptr(weights), ptr(slots), ptr(miss), ptr(ctrl), ptr(logits_out), ptr(x_hist),
        ptr(fill_src), ptr(fill_dst), ptr(filled), ptr(ws), ws_bytes, _stream(stream)))


def moe_decode_layer(shape, layer, x, norm_eps, w_router, bias, residency, codebook, ids, weights, slots, miss, ctrl,
                     logits_out, y, ws, ws_bytes, stream=None):
    _check("moe_decode_layer", load().moe_decode_layer(
        ctypes.byref(shape), layer, ptr(x), float(norm_eps), ptr(w_router), ptr(bias), ptr(residency), ptr(codebook),
        ptr(ids), ptr(weights), ptr(slots), ptr(miss), ptr(ctrl), ptr(logits_out), ptr(y), ptr(ws), ws_bytes,
        _stream(stream)))


def rl_build_pairs_workspace_bytes(shape, T) -> int:
    return load().rl_build_pairs_workspace_bytes(ctypes.byref(shape), T)


def rl_build_pairs(shape, layer, T, ids, offs, pair_tok, pair_k, ctrl, ws=None, ws_bytes=0, stream=None):
    _check("rl_build_pairs", load().rl_build_pairs(ctypes.byref(shape), layer, T, ptr(ids), ptr(offs),
                                                   ptr(pair_tok), ptr(pair_k), ptr(ctrl), ptr(ws), ws_bytes,
                                                   _stream(stream)))


def moe_prefill_workspace_bytes(shape, T) -> int:
    return load().moe_prefill_workspace_bytes(ctypes.byref(shape), T)


def moe_prefill_chunk(shape, layer, T, xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate,
                      ctrl, ws, ws_bytes, stream=None):
    _check("moe_prefill_chunk", load().moe_prefill_chunk(
        ctypes.byref(shape), layer, T, ptr(xn), ptr(offs), ptr(pair_tok), ptr(pair_k), ptr(slots), ptr(weights),
        ptr(codebook), ptr(y), int(accumulate), ptr(ctrl), ptr(ws), ws_bytes, _stream(stream)))


def moe_prefill_chunk_f32(shape, layer, T, xn, offs, pair_tok, pair_k, slots, weights, codebook, y, accumulate,
                          ctrl, ws, ws_bytes, stream=None):
    _check("moe_prefill_chunk_f32", load().moe_prefill_chunk_f32(
        ctypes.byref(shape), layer, T, ptr(xn), ptr(offs), ptr(pair_tok), ptr(pair_k), ptr(slots), ptr(weights),
        ptr(codebook), ptr(y), int(accumulate), ptr(ctrl), ptr(ws), ws_bytes, _stream(stream)))
