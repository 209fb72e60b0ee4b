"""Python binding of libspc, the GB300 decode-time hot path of SpeCache.

Every ``spc_*`` function here has the name and arguments of the C entry point
in ``include/spc.h`` and only marshals arguments: torch tensors become device
pointers, the stream defaults to torch's current stream, and a non-OK status
raises ``SpcError``.  All computation runs in the CUDA kernels of
``libspc.so``; there is no other implementation behind these names.  If the
library has not been built the import fails: build it with
``python -c "import __graft_entry__ as g; g.build()"``.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

__all__ = [
    "Dims", "SpcError", "spc_abi_version", "spc_num_quantized", "spc_records_bytes", "spc_resid_bytes",
    "spc_quantize_kv", "spc_attn_workspace_bytes", "spc_decode_attn2", "spc_merged_attn", "spc_topk_select",
    "spc_topk_select_prev", "spc_merged_attn_fetch_prev", "spc_host_gather_prev", "spc_decode_step_prev",
    "spc_host_gather", "spc_merged_attn_noalloc", "spc_merged_attn_fetch", "spc_attn_kernel_count",
    "spc_decode_step_kernel_count", "spc_decode_step_on_chip", "spc_decode_step", "spc_step_workspace_bytes",
    "spc_read_device_status", "spc_append_kv", "spc_offload_kv", "lib_path",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libspc.so")

if not os.path.exists(lib_path):
    raise ImportError(f"{lib_path} is missing: the CUDA library must be built (see __graft_entry__.build())")
_lib = C.CDLL(lib_path)

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape", 3: "CUDA error",
          4: "host pointer is not mapped pinned memory", 5: "workspace too small",
          6: "a kernel's bounded wait ran out"}


class SpcError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = f"{fn}: {STATUS.get(status, status)}"
        if status == 3:
            msg += f" (cudaError {_lib.spc_last_cuda_error()})"
        super().__init__(msg)


class spc_dims(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("D", C.c_int32),
                ("bits", C.c_int32), ("group", C.c_int32), ("N", C.c_int32), ("R", C.c_int32),
                ("q_groups_cap", C.c_int32), ("resid_cap", C.c_int32), ("scale", C.c_float)]


def Dims(B, Hq, Hkv, N, R, bits, q_groups_cap=None, resid_cap=None, scale=None, D=128, group=32) -> spc_dims:
    """Shape of one layer's cache (see spc_dims in include/spc.h).  The default
    capacities hold exactly the N_q quantised tokens and the r = N - N_q
    residual rows that spc_num_quantized reports for the shape."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    probe = spc_dims(B, Hq, Hkv, D, bits, group, N, R, max(N, 0) // 32 + 1, max(N, 0), scale)
    nq = max(int(_lib.spc_num_quantized(C.byref(probe))), 0)  # -1: an invalid shape, which every call refuses
    if q_groups_cap is None:
        q_groups_cap = nq // 32
    if resid_cap is None:
        resid_cap = N - nq
    return spc_dims(B, Hq, Hkv, D, bits, group, N, R, q_groups_cap, resid_cap, scale)


_P = C.c_void_p
_D = C.POINTER(spc_dims)
_sig = {
    "spc_abi_version": (C.c_int32, []),
    "spc_status_string": (C.c_char_p, [C.c_int]),
    "spc_last_cuda_error": (C.c_int32, []),
    "spc_num_quantized": (C.c_int32, [_D]),
    "spc_records_bytes": (C.c_size_t, [_D]),
    "spc_resid_bytes": (C.c_size_t, [_D]),
    "spc_quantize_kv": (C.c_int, [_D, _P, _P, _P, _P, _P]),
    "spc_attn_workspace_bytes": (C.c_size_t, [_D, C.c_int32]),
    "spc_decode_attn2": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "spc_merged_attn": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, _P, C.c_size_t, _P]),
    "spc_merged_attn_noalloc": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, _P]),
    "spc_merged_attn_fetch": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, _P, C.c_size_t,
                                        _P, C.c_int64, _P, C.c_int32, _P, _P]),
    "spc_topk_select": (C.c_int, [_D, _P, _P, C.c_int32, _P, _P, _P]),
    "spc_topk_select_prev": (C.c_int, [_D, _P, _P, C.c_int32, _P, _P, _P, C.c_int32, _P, _P]),
    "spc_merged_attn_fetch_prev": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, _P, C.c_size_t,
                                             _P, C.c_int64, _P, C.c_int32, _P, _P, _P, C.c_int32, _P]),
    "spc_host_gather": (C.c_int, [_D, _P, C.c_int64, _P, C.c_int32, _P, C.c_int32, _P]),
    "spc_host_gather_prev": (C.c_int, [_D, _P, C.c_int64, _P, C.c_int32, _P, _P, _P, C.c_int32, C.c_int32, _P]),
    "spc_append_kv": (C.c_int, [_D, _P, _P, _P, _P, _P, C.c_int64, _P]),
    "spc_offload_kv": (C.c_int, [_D, _P, _P, _P, C.c_int64, _P]),
    "spc_step_workspace_bytes": (C.c_size_t, [_D, C.c_int32]),
    "spc_attn_kernel_count": (C.c_int32, [_D, C.c_int32, C.c_int32]),
    "spc_decode_step_kernel_count": (C.c_int32, [_D, C.c_int32, C.c_int32, C.c_int32]),
    "spc_decode_step_on_chip": (C.c_int32, [_D, C.c_int32, C.c_int32, C.c_int32]),
    "spc_decode_step": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, C.c_int32, _P, _P, _P,
                                  C.c_size_t, _P, C.c_int64, _P, C.c_int32, _P, _P]),
    "spc_decode_step_prev": (C.c_int, [_D, _P, _P, _P, _P, _P, _P, _P, C.c_int32, _P, _P, _P, C.c_int32, _P, _P,
                                       _P, _P, C.c_size_t, _P, C.c_int64, _P, C.c_int32, _P, _P, _P, C.c_int32,
                                       _P]),
    "spc_read_device_status": (C.c_int, [_P, _D, _P]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, st):
    if st != 0:
        raise SpcError(fn, st)


def spc_abi_version() -> int:
    return int(_lib.spc_abi_version())


def spc_num_quantized(d) -> int:
    return int(_lib.spc_num_quantized(C.byref(d)))


def spc_records_bytes(d) -> int:
    return int(_lib.spc_records_bytes(C.byref(d)))


def spc_resid_bytes(d) -> int:
    return int(_lib.spc_resid_bytes(C.byref(d)))


def spc_attn_workspace_bytes(d, k_max=0) -> int:
    return int(_lib.spc_attn_workspace_bytes(C.byref(d), int(k_max)))


def spc_step_workspace_bytes(d, k_max=0) -> int:
    return int(_lib.spc_step_workspace_bytes(C.byref(d), int(k_max)))


def spc_attn_kernel_count(d, k=0, fetch_k=0) -> int:
    return int(_lib.spc_attn_kernel_count(C.byref(d), int(k), int(fetch_k)))


def spc_decode_step_kernel_count(d, k, fetch_k, next_k) -> int:
    return int(_lib.spc_decode_step_kernel_count(C.byref(d), int(k), int(fetch_k), int(next_k)))


def spc_decode_step_on_chip(d, k, fetch_k, next_k) -> int:
    """1 if spc_decode_step may be called with spec_logits=None (logits kept in TMEM)."""
    return int(_lib.spc_decode_step_on_chip(C.byref(d), int(k), int(fetch_k), int(next_k)))


def spc_decode_step(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, next_k, next_idx,
                    next_bitmap, ws, ws_bytes=None, fetch_host_kv=None, fetch_n_cap=0, fetch_idx=None, fetch_k=0,
                    fetch_staging=None, stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_decode_step",
           _lib.spc_decode_step(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(kv_self), _ptr(idx),
                                _ptr(bitmap),
                                _ptr(staging), int(k), _ptr(o), _ptr(lse), _ptr(spec_logits), int(next_k),
                                _ptr(next_idx), _ptr(next_bitmap), _ptr(ws), ws_bytes, _ptr(fetch_host_kv),
                                int(fetch_n_cap), _ptr(fetch_idx), int(fetch_k), _ptr(fetch_staging),
                                _stream(stream)))


def spc_decode_step_prev(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, next_k, next_idx,
                         next_bitmap, next_src, ws, ws_bytes=None, fetch_host_kv=None, fetch_n_cap=0, fetch_idx=None,
                         fetch_k=0, fetch_staging=None, fetch_src=None, fetch_prev_staging=None, fetch_prev_k=0,
                         stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_decode_step_prev",
           _lib.spc_decode_step_prev(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(kv_self), _ptr(idx),
                                     _ptr(bitmap), _ptr(staging), int(k), _ptr(o), _ptr(lse), _ptr(spec_logits),
                                     int(next_k), _ptr(next_idx), _ptr(next_bitmap), _ptr(next_src), _ptr(ws),
                                     ws_bytes, _ptr(fetch_host_kv), int(fetch_n_cap), _ptr(fetch_idx), int(fetch_k),
                                     _ptr(fetch_staging), _ptr(fetch_src), _ptr(fetch_prev_staging),
                                     int(fetch_prev_k), _stream(stream)))


def spc_read_device_status(ws, d, stream=None) -> int:
    """0, or SPC_ERR_TIMEOUT (6) if a bounded wait in spc_decode_step ran out (the word is cleared)."""
    return int(_lib.spc_read_device_status(_ptr(ws), C.byref(d), _stream(stream)))


def spc_quantize_kv(d, k, v, records, resid, stream=None):
    _check("spc_quantize_kv", _lib.spc_quantize_kv(C.byref(d), _ptr(k), _ptr(v), _ptr(records), _ptr(resid),
                                                   _stream(stream)))


def spc_decode_attn2(d, records, resid, q, o, lse, spec_logits, ws, ws_bytes=None, stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_decode_attn2", _lib.spc_decode_attn2(C.byref(d), _ptr(records), _ptr(resid), _ptr(q),
                                                     _ptr(kv_self), _ptr(o), _ptr(lse), _ptr(spec_logits),
                                                     _ptr(ws), ws_bytes, _stream(stream)))


def spc_merged_attn(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, ws, ws_bytes=None,
                    stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_merged_attn", _lib.spc_merged_attn(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(kv_self),
                                                   _ptr(idx), _ptr(bitmap), _ptr(staging), int(k), _ptr(o),
                                                   _ptr(lse), _ptr(spec_logits), _ptr(ws), ws_bytes,
                                                   _stream(stream)))


def spc_merged_attn_fetch(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, ws, fetch_host_kv,
                          fetch_n_cap, fetch_idx, fetch_k, fetch_staging, ws_bytes=None, stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_merged_attn_fetch",
           _lib.spc_merged_attn_fetch(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(kv_self), _ptr(idx),
                                      _ptr(bitmap),
                                      _ptr(staging), int(k), _ptr(o), _ptr(lse), _ptr(spec_logits), _ptr(ws),
                                      ws_bytes, _ptr(fetch_host_kv), int(fetch_n_cap), _ptr(fetch_idx),
                                      int(fetch_k), _ptr(fetch_staging), _stream(stream)))


def spc_merged_attn_fetch_prev(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, ws,
                               fetch_host_kv, fetch_n_cap, fetch_idx, fetch_k, fetch_staging, fetch_src,
                               fetch_prev_staging, fetch_prev_k, ws_bytes=None, stream=None, kv_self=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check("spc_merged_attn_fetch_prev",
           _lib.spc_merged_attn_fetch_prev(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(kv_self),
                                           _ptr(idx), _ptr(bitmap), _ptr(staging), int(k), _ptr(o), _ptr(lse),
                                           _ptr(spec_logits), _ptr(ws), ws_bytes, _ptr(fetch_host_kv),
                                           int(fetch_n_cap), _ptr(fetch_idx), int(fetch_k), _ptr(fetch_staging),
                                           _ptr(fetch_src), _ptr(fetch_prev_staging), int(fetch_prev_k),
                                           _stream(stream)))


def spc_merged_attn_noalloc(d, records, resid, q, idx, bitmap, staging, k, o, lse, spec_logits, stream=None):
    """spc_merged_attn with the library's built-in workspace (for callers that cannot allocate)."""
    _check("spc_merged_attn_noalloc",
           _lib.spc_merged_attn_noalloc(C.byref(d), _ptr(records), _ptr(resid), _ptr(q), _ptr(idx), _ptr(bitmap),
                                        _ptr(staging), int(k), _ptr(o), _ptr(lse), _ptr(spec_logits),
                                        _stream(stream)))


def spc_topk_select(d, spec_logits, lse, k, idx, bitmap, stream=None):
    _check("spc_topk_select", _lib.spc_topk_select(C.byref(d), _ptr(spec_logits), _ptr(lse), int(k), _ptr(idx),
                                                   _ptr(bitmap), _stream(stream)))


def spc_topk_select_prev(d, spec_logits, lse, k, idx, bitmap, prev_idx, prev_k, src, stream=None):
    _check("spc_topk_select_prev",
           _lib.spc_topk_select_prev(C.byref(d), _ptr(spec_logits), _ptr(lse), int(k), _ptr(idx), _ptr(bitmap),
                                     _ptr(prev_idx), int(prev_k), _ptr(src), _stream(stream)))


def spc_append_kv(d, k_new, v_new, records, resid, host_kv=None, n_cap=0, stream=None):
    _check("spc_append_kv", _lib.spc_append_kv(C.byref(d), _ptr(k_new), _ptr(v_new), _ptr(records), _ptr(resid),
                                               _ptr(host_kv), int(n_cap), _stream(stream)))


def spc_offload_kv(d, k, v, host_kv, n_cap, stream=None):
    _check("spc_offload_kv", _lib.spc_offload_kv(C.byref(d), _ptr(k), _ptr(v), _ptr(host_kv), int(n_cap),
                                                 _stream(stream)))


def spc_host_gather(d, host_kv, n_cap, idx, k, staging, max_ctas=0, stream=None):
    _check("spc_host_gather", _lib.spc_host_gather(C.byref(d), _ptr(host_kv), int(n_cap), _ptr(idx), int(k),
                                                   _ptr(staging), int(max_ctas), _stream(stream)))


def spc_host_gather_prev(d, host_kv, n_cap, idx, k, staging, src, prev_staging, prev_k, max_ctas=0, stream=None):
    _check("spc_host_gather_prev",
           _lib.spc_host_gather_prev(C.byref(d), _ptr(host_kv), int(n_cap), _ptr(idx), int(k), _ptr(staging),
                                     _ptr(src), _ptr(prev_staging), int(prev_k), int(max_ctas), _stream(stream)))
