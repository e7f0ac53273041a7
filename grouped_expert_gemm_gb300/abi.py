"""ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Functions keep the C names.  Tensor arguments are torch tensors (or None for a
NULL pointer) whose ``data_ptr()`` is passed through; ``stream`` defaults to
torch's current CUDA stream.  Every computation happens in the CUDA library;
nothing here falls back to another implementation.  A non-OK status raises
MoeError; loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4

MOE_DEV_NONFINITE_LOGIT = 1
MOE_DEV_BAD_EXPERT_ID = 2
MOE_DEV_BAD_HEADER_ID = 4
MOE_DEV_BAD_ROW = 8
MOE_DEV_TIMEOUT = 16
MOE_DEV_NONFINITE_INPUT = 32
MOE_DEV_BAD_MAP = 64

MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID_GROUP = 1
MOE_WAVE_STRIPE = 0
MOE_WAVE_DESTMOD = 1
MOE_POOL_EMPTY = 0xFFFF
MOE_ROUTE_MASKED = -1
MOE_BIAS_SIGN = 0
MOE_BIAS_PROPORTIONAL = 1
MOE_SCALE_ROW = 0
MOE_SCALE_BLOCK128 = 128
MOE_PAYLOAD_BF16 = 0
MOE_PAYLOAD_FP8_ROW = 1
MOE_PAYLOAD_FP8_BLOCK128 = 2

EXPORTED = [
    "moe_version", "moe_status_string", "moe_capacity", "moe_route", "moe_sigmoid_det",
    "moe_permute_workspace_size", "moe_permute", "moe_permute_noalloc",
    "moe_grouped_swiglu_workspace_size",
    "moe_grouped_swiglu", "moe_grouped_gate_up", "moe_grouped_down", "moe_grouped_down_chained",
    "moe_grouped_swiglu_onepass", "moe_grouped_swiglu_onepass_taken",
    "moe_combine", "moe_pool_pack_workspace_size", "moe_pool_pack",
    "moe_pool_compact_workspace_size", "moe_pool_compact", "moe_pool_compact_rotated",
    "moe_compose_map",
    "moe_combine_backward", "moe_unpermute_grad", "moe_load_stats", "moe_bias_update",
    "moe_bucket_stage", "moe_route_bucket", "moe_permute_bucket", "moe_combine_bucket",
    "moe_payload_bytes", "moe_quantize_fp8", "moe_dequantize_fp8", "moe_permute_fp8",
    "moe_grouped_gate_up_fp8", "moe_grouped_gate_up_gather", "moe_expert_demand", "moe_validate_permutation",
    "moe_validate_pools_workspace_size", "moe_validate_pools",
    "moe_validate_compact_workspace_size", "moe_validate_compact", "moe_debug_wait_timeout",
    "moe_decode_workspace_size", "moe_decode_layer",
]


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


class RouteParams(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("route_scale", ctypes.c_float)]


class PoolParams(ctypes.Structure):
    _fields_ = [("n_dest", ctypes.c_int32), ("local_per_dest", ctypes.c_int32),
                ("n_waves", ctypes.c_int32), ("pool_cap", ctypes.c_int32),
                ("wave_policy", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_version": (_I32, []),
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_capacity": (_I64, [_I64, _I64, _I64, _I64]),
    "moe_route": (_I32, [ctypes.POINTER(RouteParams), _P, _P, _P, _P, _P, _P]),
    "moe_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "moe_decode_layer": (_I32, [ctypes.POINTER(RouteParams), _I32, _I32, _I32, _P, _P, _P, _P, _P,
                                _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                _P]),
    "moe_sigmoid_det": (_I32, [_I64, _P, _P, _P]),
    "moe_permute_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "moe_permute": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                           _P, _P]),
    "moe_permute_noalloc": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _P]),
    "moe_grouped_swiglu_workspace_size": (_SZ, [_I32, _I32]),
    "moe_grouped_swiglu": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                  _P, _P]),
    "moe_grouped_gate_up": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_down": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_down_chained": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_swiglu_onepass": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P, _P]),
    "moe_grouped_swiglu_onepass_taken": (_I32, [_I32, _I32, _I32, _I32]),
    "moe_combine": (_I32, [_I32, _I32, _I32, _P, _I64, _P, _P, _P, _I32, _P, _P, _P]),
    "moe_pool_pack_workspace_size": (_SZ, [ctypes.POINTER(PoolParams), _I32, _I32]),
    "moe_pool_pack": (_I32, [ctypes.POINTER(PoolParams), _I32, _I32, _I32, _I32, _P, _P, _P, _P,
                             _P, _P, _P, _SZ, _P, _P]),
    "moe_pool_compact_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "moe_pool_compact": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                _P]),
    "moe_pool_compact_rotated": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                        _SZ, _P, _P]),
    "moe_compose_map": (_I32, [_I64, _P, _P, _I64, _P, _P, _P]),
    "moe_combine_backward": (_I32, [_I32, _I32, _I32, _P, _P, _I64, _P, _P, _P, _P, _P, _P]),
    "moe_unpermute_grad": (_I32, [_I32, _I32, _I32, _P, _I64, _P, _P, _I32, _P, _P]),
    "moe_load_stats": (_I32, [_I32, _P, _P, _P]),
    "moe_bucket_stage": (_I32, [_I32, _I32, _I32, _P, _P, _P, _P, _P, _P]),
    "moe_route_bucket": (_I32, [ctypes.POINTER(RouteParams), _P, _P, _P, _P, _P, _P, _P]),
    "moe_permute_bucket": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  _P, _SZ, _P, _P]),
    "moe_combine_bucket": (_I32, [_I32, _I32, _I32, _P, _P, _I64, _P, _P, _P, _I32, _P, _P, _P]),
    "moe_bias_update": (_I32, [_I32, _P, _P, ctypes.c_float, _I32, _P]),
    "moe_payload_bytes": (_I64, [_I64, _I32, _I32]),
    "moe_quantize_fp8": (_I32, [_I64, _I32, _I32, _P, _P, _P, _P, _P]),
    "moe_dequantize_fp8": (_I32, [_I64, _I32, _I32, _P, _P, _P, _P]),
    "moe_permute_fp8": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _P, _P, _SZ, _P, _P]),
    "moe_grouped_gate_up_fp8": (_I32, [_I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P]),
    "moe_grouped_gate_up_gather": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P]),
    "moe_expert_demand": (_I32, [_I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "moe_validate_permutation": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P]),
    "moe_validate_pools_workspace_size": (_SZ, [ctypes.POINTER(PoolParams)]),
    "moe_validate_pools": (_I32, [ctypes.POINTER(PoolParams), _I32, _I32, _I32, _P, _P, _P, _P,
                                  _P, _SZ, _P, _P]),
    "moe_validate_compact_workspace_size": (_SZ, [_I32, _I32]),
    "moe_validate_compact": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P,
                                    _P]),
    "moe_debug_wait_timeout": (_I32, [_I64, _P, _P]),
}

_lib: Optional[ctypes.CDLL] = None
_launches = [0]


def launch_count() -> int:
    """Kernels launched through this binding so far (each call knows its launch count)."""
    return _launches[0]


def _count(n: int):
    _launches[0] += n


def library_path() -> str:
    return _build.LIBPATH


def lib() -> ctypes.CDLL:
    """Load the CUDA library (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run grouped_expert_gemm_gb300.build.build())")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != MOE_OK:
        raise MoeError(fn, st, lib().moe_status_string(st).decode())


# ----------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def moe_version() -> int:
    return lib().moe_version()


def moe_capacity(cf_num: int, cf_den: int, assignments: int, slots: int) -> int:
    return lib().moe_capacity(cf_num, cf_den, assignments, slots)


def moe_route(p: RouteParams, logits, sel_bias, topk_ids, gates, dev_status=None, stream=None):
    _check("moe_route", lib().moe_route(ctypes.byref(p), _ptr(logits), _ptr(sel_bias),
                                        _ptr(topk_ids), _ptr(gates), _ptr(dev_status),
                                        _stream(stream)))
    _count(1 if p.T > 0 else 0)


def moe_sigmoid_det(n: int, z, s, stream=None):
    _check("moe_sigmoid_det", lib().moe_sigmoid_det(n, _ptr(z), _ptr(s), _stream(stream)))
    _count(1 if n > 0 else 0)


def _permute_launches(T: int, k: int, copy: bool = True) -> int:
    """Kernels one permute call launches: the tile histogram runs only with several tiles,
    the row copy only when rows are copied (not for the maps-only form) and as a launch
    of its own only above 16 routes (below, the rank block copies them)."""
    R = T * k
    if R <= 0:
        return 1
    per_tile = max(2048, -(-R // 128))
    return (3 if -(-R // per_tile) > 1 else 2) - (0 if copy and R > 16 else 1)


def moe_permute_workspace_size(T: int, k: int, E: int) -> int:
    return lib().moe_permute_workspace_size(T, k, E)


def moe_permute(T, d, E, k, capacity, topk_ids, x, x_perm, counts, offsets, row_to_route,
                route_to_row, n_dropped, ws, ws_bytes, dev_status=None, stream=None):
    _check("moe_permute", lib().moe_permute(
        T, d, E, k, capacity, _ptr(topk_ids), _ptr(x), _ptr(x_perm), _ptr(counts), _ptr(offsets),
        _ptr(row_to_route), _ptr(route_to_row), _ptr(n_dropped), _ptr(ws), ws_bytes,
        _ptr(dev_status), _stream(stream)))
    _count(_permute_launches(T, k, x is not None))


def moe_permute_noalloc(T, d, E, k, capacity, topk_ids, x, x_perm, counts, offsets, row_to_route,
                        route_to_row, n_dropped, dev_status=None, stream=None):
    """moe_permute without a workspace: scratch is a fixed 64 KiB device array of the library.
    Calls that overlap on the GPU race on it; the first call on a device should precede
    any stream capture."""
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(
        T, d, E, k, capacity, _ptr(topk_ids), _ptr(x), _ptr(x_perm), _ptr(counts), _ptr(offsets),
        _ptr(row_to_route), _ptr(route_to_row), _ptr(n_dropped), _ptr(dev_status),
        _stream(stream)))
    _count(_permute_launches(T, k, x is not None))


def moe_grouped_swiglu_workspace_size(max_rows: int, I: int) -> int:
    return lib().moe_grouped_swiglu_workspace_size(max_rows, I)


def moe_grouped_swiglu(n_seg, d, I, max_rows, x, seg_begin, seg_count, w_gate, w_up, w_down, y,
                       ws, ws_bytes, dev_status=None, stream=None):
    _check("moe_grouped_swiglu", lib().moe_grouped_swiglu(
        n_seg, d, I, max_rows, _ptr(x), _ptr(seg_begin), _ptr(seg_count), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(y), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))
    _count(2 if max_rows > 0 else 0)


def moe_grouped_swiglu_onepass_taken(n_seg, d, I, max_rows) -> bool:
    return bool(lib().moe_grouped_swiglu_onepass_taken(n_seg, d, I, max_rows))


def moe_grouped_swiglu_onepass(n_seg, d, I, max_rows, x, seg_begin, seg_count, w_gate, w_up,
                               w_down, h, y, sync, dev_status=None, stream=None):
    _check("moe_grouped_swiglu_onepass", lib().moe_grouped_swiglu_onepass(
        n_seg, d, I, max_rows, _ptr(x), _ptr(seg_begin), _ptr(seg_count), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(h), _ptr(y), _ptr(sync), _ptr(dev_status),
        _stream(stream)))
    if max_rows > 0:
        _count(1 if moe_grouped_swiglu_onepass_taken(n_seg, d, I, max_rows) else 2)


def moe_grouped_gate_up(n_seg, d, I, max_rows, x, seg_begin, seg_count, w_gate, w_up, h,
                        dev_status=None, stream=None):
    _check("moe_grouped_gate_up", lib().moe_grouped_gate_up(
        n_seg, d, I, max_rows, _ptr(x), _ptr(seg_begin), _ptr(seg_count), _ptr(w_gate),
        _ptr(w_up), _ptr(h), _ptr(dev_status), _stream(stream)))
    _count(1 if max_rows > 0 else 0)


def moe_payload_bytes(rows: int, d: int, payload: int) -> int:
    return lib().moe_payload_bytes(rows, d, payload)


def fp8_scale_groups(d: int, group: int) -> int:
    """Scales per row for a scale group setting (MOE_SCALE_ROW or MOE_SCALE_BLOCK128)."""
    return 1 if group == MOE_SCALE_ROW else -(-d // 128)


def moe_quantize_fp8(n, d, group, x, q, scales, dev_status=None, stream=None):
    _check("moe_quantize_fp8", lib().moe_quantize_fp8(
        n, d, group, _ptr(x), _ptr(q), _ptr(scales), _ptr(dev_status), _stream(stream)))
    _count(1 if n > 0 else 0)


def moe_dequantize_fp8(n, d, group, q, scales, x, stream=None):
    _check("moe_dequantize_fp8", lib().moe_dequantize_fp8(
        n, d, group, _ptr(q), _ptr(scales), _ptr(x), _stream(stream)))
    _count(1 if n > 0 else 0)


def moe_permute_fp8(T, d, E, k, capacity, group, topk_ids, q, scales, q_perm, scales_perm, counts,
                    offsets, row_to_route, route_to_row, n_dropped, ws, ws_bytes, dev_status=None,
                    stream=None):
    _check("moe_permute_fp8", lib().moe_permute_fp8(
        T, d, E, k, capacity, group, _ptr(topk_ids), _ptr(q), _ptr(scales), _ptr(q_perm),
        _ptr(scales_perm), _ptr(counts), _ptr(offsets), _ptr(row_to_route), _ptr(route_to_row),
        _ptr(n_dropped), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))
    _count(_permute_launches(T, k))


def moe_grouped_gate_up_gather(n_seg, d, I, max_rows, T, k, x, row_to_route, seg_begin,
                               seg_count, w_gate, w_up, h, dev_status=None, stream=None):
    _check("moe_grouped_gate_up_gather", lib().moe_grouped_gate_up_gather(
        n_seg, d, I, max_rows, T, k, _ptr(x), _ptr(row_to_route), _ptr(seg_begin),
        _ptr(seg_count), _ptr(w_gate), _ptr(w_up), _ptr(h), _ptr(dev_status), _stream(stream)))
    _count(1 if max_rows > 0 else 0)


def moe_grouped_gate_up_fp8(n_seg, d, I, max_rows, group, xq, scales, seg_begin, seg_count,
                            w_gate, w_up, h, dev_status=None, stream=None):
    _check("moe_grouped_gate_up_fp8", lib().moe_grouped_gate_up_fp8(
        n_seg, d, I, max_rows, group, _ptr(xq), _ptr(scales), _ptr(seg_begin), _ptr(seg_count),
        _ptr(w_gate), _ptr(w_up), _ptr(h), _ptr(dev_status), _stream(stream)))
    _count(1 if max_rows > 0 else 0)


def moe_grouped_down(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y, dev_status=None,
                     stream=None):
    _check("moe_grouped_down", lib().moe_grouped_down(
        n_seg, I, d, max_rows, _ptr(h), _ptr(seg_begin), _ptr(seg_count), _ptr(w_down), _ptr(y),
        _ptr(dev_status), _stream(stream)))
    _count(1 if max_rows > 0 else 0)


def moe_grouped_down_chained(n_seg, I, d, max_rows, h, seg_begin, seg_count, w_down, y,
                             dev_status=None, stream=None):
    """moe_grouped_down right after this library's gate/up pass on the same stream and
    segment table (see include/moe.h for the precondition)."""
    _check("moe_grouped_down_chained", lib().moe_grouped_down_chained(
        n_seg, I, d, max_rows, _ptr(h), _ptr(seg_begin), _ptr(seg_count), _ptr(w_down), _ptr(y),
        _ptr(dev_status), _stream(stream)))
    _count(1 if max_rows > 0 else 0)


def moe_combine(T, k, d, y, y_rows, route_to_row, gates, shared_y, accumulate, out,
                dev_status=None, stream=None):
    _check("moe_combine", lib().moe_combine(
        T, k, d, _ptr(y), y_rows, _ptr(route_to_row), _ptr(gates), _ptr(shared_y),
        int(accumulate), _ptr(out), _ptr(dev_status), _stream(stream)))
    _count(1 if T > 0 else 0)


def moe_pool_pack_workspace_size(p: PoolParams, T: int, k: int) -> int:
    return lib().moe_pool_pack_workspace_size(ctypes.byref(p), T, k)


def moe_pool_pack(p: PoolParams, T, d, k, wave, topk_ids, x, pools, route_to_poolrow, pool_fill,
                  sender_drops, ws, ws_bytes, dev_status=None, stream=None):
    _check("moe_pool_pack", lib().moe_pool_pack(
        ctypes.byref(p), T, d, k, wave, _ptr(topk_ids), _ptr(x), _ptr(pools),
        _ptr(route_to_poolrow), _ptr(pool_fill), _ptr(sender_drops), _ptr(ws), ws_bytes,
        _ptr(dev_status), _stream(stream)))
    _count(3 if T > 0 else 2)


def moe_pool_compact_workspace_size(n_src: int, pool_cap: int, n_local: int) -> int:
    return lib().moe_pool_compact_workspace_size(n_src, pool_cap, n_local)


def moe_pool_compact(n_src, pool_cap, d, n_local, local_cap, pools, compact, local_counts,
                     poolrow_to_row, receiver_drops, ws, ws_bytes, dev_status=None, stream=None):
    _check("moe_pool_compact", lib().moe_pool_compact(
        n_src, pool_cap, d, n_local, local_cap, _ptr(pools), _ptr(compact), _ptr(local_counts),
        _ptr(poolrow_to_row), _ptr(receiver_drops), _ptr(ws), ws_bytes, _ptr(dev_status),
        _stream(stream)))
    _count(3)


def moe_pool_compact_rotated(n_src, pool_cap, d, n_local, local_cap, first_source, pools, compact,
                             local_counts, poolrow_to_row, receiver_drops, ws, ws_bytes,
                             dev_status=None, stream=None):
    _check("moe_pool_compact_rotated", lib().moe_pool_compact_rotated(
        n_src, pool_cap, d, n_local, local_cap, first_source, _ptr(pools), _ptr(compact),
        _ptr(local_counts), _ptr(poolrow_to_row), _ptr(receiver_drops), _ptr(ws), ws_bytes,
        _ptr(dev_status), _stream(stream)))
    _count(3)


def moe_compose_map(n, a, b, b_len, out, dev_status=None, stream=None):
    _check("moe_compose_map", lib().moe_compose_map(n, _ptr(a), _ptr(b), b_len, _ptr(out),
                                                    _ptr(dev_status), _stream(stream)))
    _count(1 if n > 0 else 0)


def moe_combine_backward(T, k, d, dout, y, y_rows, route_to_row, gates, dy, dgates,
                         dev_status=None, stream=None):
    _check("moe_combine_backward", lib().moe_combine_backward(
        T, k, d, _ptr(dout), _ptr(y), y_rows, _ptr(route_to_row), _ptr(gates), _ptr(dy),
        _ptr(dgates), _ptr(dev_status), _stream(stream)))
    _count(1 if T > 0 else 0)


def moe_unpermute_grad(T, k, d, dx_perm, rows, route_to_row, dx, accumulate=0, dev_status=None,
                       stream=None):
    _check("moe_unpermute_grad", lib().moe_unpermute_grad(
        T, k, d, _ptr(dx_perm), rows, _ptr(route_to_row), _ptr(dx), int(accumulate),
        _ptr(dev_status), _stream(stream)))
    _count(1 if T > 0 else 0)


def moe_load_stats(U, counts, stats, stream=None):
    _check("moe_load_stats", lib().moe_load_stats(U, _ptr(counts), _ptr(stats), _stream(stream)))
    _count(1)


def moe_bias_update(E, counts, bias, u, rule=MOE_BIAS_SIGN, stream=None):
    _check("moe_bias_update", lib().moe_bias_update(E, _ptr(counts), _ptr(bias), float(u), rule,
                                                    _stream(stream)))
    _count(1)


def moe_bucket_stage(T, E, d, logits, x, logits_dst, x_dst, valid_tokens, stream=None):
    _check("moe_bucket_stage", lib().moe_bucket_stage(
        T, E, d, _ptr(logits), _ptr(x), _ptr(logits_dst), _ptr(x_dst), _ptr(valid_tokens),
        _stream(stream)))
    _count(1)


def moe_route_bucket(p: RouteParams, valid_tokens, logits, sel_bias, topk_ids, gates,
                     dev_status=None, stream=None):
    _check("moe_route_bucket", lib().moe_route_bucket(
        ctypes.byref(p), _ptr(valid_tokens), _ptr(logits), _ptr(sel_bias), _ptr(topk_ids),
        _ptr(gates), _ptr(dev_status), _stream(stream)))
    _count(1 if p.T > 0 else 0)


def moe_permute_bucket(T, d, E, k, capacity, valid_tokens, topk_ids, x, x_perm, counts, offsets,
                       row_to_route, route_to_row, n_dropped, ws, ws_bytes, dev_status=None,
                       stream=None):
    _check("moe_permute_bucket", lib().moe_permute_bucket(
        T, d, E, k, capacity, _ptr(valid_tokens), _ptr(topk_ids), _ptr(x), _ptr(x_perm),
        _ptr(counts), _ptr(offsets), _ptr(row_to_route), _ptr(route_to_row), _ptr(n_dropped),
        _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))
    _count(_permute_launches(T, k, x is not None))


def moe_combine_bucket(T, k, d, valid_tokens, y, y_rows, route_to_row, gates, shared_y,
                       accumulate, out, dev_status=None, stream=None):
    _check("moe_combine_bucket", lib().moe_combine_bucket(
        T, k, d, _ptr(valid_tokens), _ptr(y), y_rows, _ptr(route_to_row), _ptr(gates),
        _ptr(shared_y), int(accumulate), _ptr(out), _ptr(dev_status), _stream(stream)))
    _count(1 if T > 0 else 0)


def moe_decode_workspace_size(T, d, E, k, I) -> int:
    return lib().moe_decode_workspace_size(T, d, E, k, I)


def moe_decode_layer(p: RouteParams, d, I, capacity, valid_tokens, logits, sel_bias, x, w_gate,
                     w_up, w_down, topk_ids, gates, counts, offsets, row_to_route, route_to_row,
                     n_dropped, x_perm, h, y, out, ws, ws_bytes, dev_status=None, stream=None):
    _check("moe_decode_layer", lib().moe_decode_layer(
        ctypes.byref(p), d, I, capacity, _ptr(valid_tokens), _ptr(logits), _ptr(sel_bias),
        _ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(topk_ids), _ptr(gates),
        _ptr(counts), _ptr(offsets), _ptr(row_to_route), _ptr(route_to_row), _ptr(n_dropped),
        _ptr(x_perm), _ptr(h), _ptr(y), _ptr(out), _ptr(ws), ws_bytes, _ptr(dev_status),
        _stream(stream)))
    _count(1)


def moe_expert_demand(T, k, E, valid_tokens, topk_ids, demand, dev_status=None, stream=None):
    _check("moe_expert_demand", lib().moe_expert_demand(
        T, k, E, _ptr(valid_tokens), _ptr(topk_ids), _ptr(demand), _ptr(dev_status),
        _stream(stream)))
    _count(1 if T > 0 else 0)


def moe_validate_permutation(T, E, k, capacity, valid_tokens, topk_ids, counts, offsets,
                             row_to_route, route_to_row, n_dropped, dev_status, stream=None):
    _check("moe_validate_permutation", lib().moe_validate_permutation(
        T, E, k, capacity, _ptr(valid_tokens), _ptr(topk_ids), _ptr(counts), _ptr(offsets),
        _ptr(row_to_route), _ptr(route_to_row), _ptr(n_dropped), _ptr(dev_status),
        _stream(stream)))
    _count(2 if T > 0 else 1)


def moe_validate_pools_workspace_size(p: PoolParams) -> int:
    return lib().moe_validate_pools_workspace_size(ctypes.byref(p))


def moe_validate_pools(p: PoolParams, T, d, k, topk_ids, pools, route_to_poolrow, pool_fill, ws,
                       ws_bytes, dev_status, stream=None):
    _check("moe_validate_pools", lib().moe_validate_pools(
        ctypes.byref(p), T, d, k, _ptr(topk_ids), _ptr(pools), _ptr(route_to_poolrow),
        _ptr(pool_fill), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))
    _count(3)


def moe_validate_compact_workspace_size(n_local: int, local_cap: int) -> int:
    return lib().moe_validate_compact_workspace_size(n_local, local_cap)


def moe_validate_compact(n_src, pool_cap, d, n_local, local_cap, pools, local_counts,
                         poolrow_to_row, ws, ws_bytes, dev_status, stream=None, first_source=0):
    _check("moe_validate_compact", lib().moe_validate_compact(
        n_src, pool_cap, d, n_local, local_cap, first_source, _ptr(pools), _ptr(local_counts),
        _ptr(poolrow_to_row), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))
    _count(4)


def moe_debug_wait_timeout(limit_ns, dev_status, stream=None):
    _check("moe_debug_wait_timeout", lib().moe_debug_wait_timeout(
        int(limit_ns), _ptr(dev_status), _stream(stream)))
    _count(1)
