"""GPU twin of synth.kv_layer: the same bytes, made on the device.

Used for workloads too large to draw on the host (the 32-layer, 32K-token
cache is 34 GB of bf16).  A test checks it against the numpy generator.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

import synth

_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspc_synth.so")
_lib = None
_tables = {}


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise ImportError(f"{_LIB} is missing: build it with __graft_entry__.build()")
        _lib = C.CDLL(_LIB)
        _lib.spc_synth_kv.restype = C.c_int32
        _lib.spc_synth_kv.argtypes = [C.c_uint64, C.c_uint64, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p]
    return _lib


def _device_tables(device):
    key = str(device)
    if key not in _tables:
        th = torch.from_numpy(synth.THRESH.view(np.int64).copy()).to(device)
        vals = torch.from_numpy(synth.VALS.view(np.int16).copy()).to(device)
        _tables[key] = (th, vals)
    return _tables[key]


def kv_layer_into(seed: int, layer: int, K: torch.Tensor, V: torch.Tensor, stream=None):
    """Fill device bf16-bit tensors K, V [B, Hkv, N, D] (dtype int16/uint16/bfloat16)."""
    lib = _load()
    B, Hkv, N, D = K.shape
    th, vals = _device_tables(K.device)
    outl = torch.from_numpy(synth.outlier_channels(seed, layer, Hkv, D)).to(K.device)
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream.cuda_stream
    kk = int(synth.stream_key(seed, synth.TID_K, layer))
    kv = int(synth.stream_key(seed, synth.TID_V, layer))
    err = lib.spc_synth_kv(kk, kv, B, Hkv, N, D, outl.data_ptr(), th.data_ptr(), vals.data_ptr(), len(synth.THRESH),
                           K.data_ptr() if K is not None else None, V.data_ptr() if V is not None else None, s)
    if err != 0:
        raise RuntimeError(f"spc_synth_kv failed with cudaError {err}")
    # keep the outlier table alive until the kernel has read it
    torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
