"""ctypes wrapper of the plain C oracle (spc_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path
(``bit_kv_cache_spc_gb300``) never does.  All arithmetic lives in the C file;
this module only allocates numpy arrays and marshals arguments.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "spc_oracle.c")
LIB = os.path.join(HERE, "libspc_oracle.so")

_lib = None


class orc_dims(C.Structure):
    _fields_ = [("B", C.c_int32), ("Hq", C.c_int32), ("Hkv", C.c_int32), ("D", C.c_int32),
                ("bits", C.c_int32), ("N", C.c_int32), ("R", C.c_int32), ("group", C.c_int32),
                ("scale", C.c_double)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add, OpenMP)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "spc_oracle.h"))):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", "-Wall", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        P = C.c_void_p
        L.orc_nq.restype = C.c_int32
        L.orc_nq.argtypes = [C.POINTER(orc_dims)]
        L.orc_quant_params.argtypes = [C.c_int32, C.c_int32, C.c_float, C.c_float,
                                       C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.orc_quant_code.restype = C.c_uint8
        L.orc_quant_code.argtypes = [C.c_int32, C.c_float, C.c_float, C.c_float]
        L.orc_dequant.restype = C.c_double
        L.orc_dequant.argtypes = [C.c_int32, C.c_int32, C.c_uint16, C.c_uint16, C.c_int32]
        L.orc_quantize.argtypes = [C.POINTER(orc_dims), C.c_int32, P, P, P, P, P, P]
        L.orc_record_bytes.restype = C.c_int64
        L.orc_record_bytes.argtypes = [C.c_int32]
        L.orc_unit_bytes.restype = C.c_int64
        L.orc_unit_bytes.argtypes = [C.c_int32, C.c_int32]
        L.orc_units_cap.restype = C.c_int32
        L.orc_units_cap.argtypes = [C.c_int32, C.c_int32]
        L.orc_pack.argtypes = [C.POINTER(orc_dims), P, P, P, P, P, P, C.c_int32, C.c_int32, P, P]
        L.orc_attention.argtypes = [C.POINTER(orc_dims), C.c_int32, P, P, P, P, P, P, P, P,
                                    C.c_int32, P, P, P, P]
        L.orc_topk.argtypes = [C.POINTER(orc_dims), P, C.c_int32, P, P]
        L.orc_gather.argtypes = [C.POINTER(orc_dims), P, C.c_int64, P, C.c_int32, P]
        L.orc_append.argtypes = [C.POINTER(orc_dims), C.c_int32, C.c_int32, P, P, P, P, P, C.c_int64]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def dims(B, Hq, Hkv, N, R, bits, D=128, scale=None, group=32) -> orc_dims:
    assert group in (32, 64)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(D)))
    return orc_dims(B, Hq, Hkv, D, bits, N, R, group, scale)


def nq(d: orc_dims) -> int:
    return int(lib().orc_nq(C.byref(d)))


def quant_params(bits: int, lo: float, hi: float, mode: int = 0):
    z, s = C.c_float(), C.c_float()
    lib().orc_quant_params(bits, mode, lo, hi, C.byref(z), C.byref(s))
    return z.value, s.value


def quant_code(bits: int, x: float, z: float, s: float) -> int:
    return int(lib().orc_quant_code(bits, x, z, s))


def dequant(bits: int, lo_bits: int, hi_bits: int, code: int, mode: int = 0) -> float:
    return float(lib().orc_dequant(bits, mode, lo_bits, hi_bits, code))


def quantize(d: orc_dims, K, V, mode: int = 0):
    """Logical codes and min/max (see spc_oracle.h)."""
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    n_q = nq(d)
    kcode = np.zeros((d.B, d.Hkv, n_q, d.D), np.uint8)
    vcode = np.zeros((d.B, d.Hkv, n_q, d.D), np.uint8)
    kmm = np.zeros((d.B, d.Hkv, n_q // d.group, d.D, 2), np.uint16)
    vmm = np.zeros((d.B, d.Hkv, n_q, d.D // d.group, 2), np.uint16)
    lib().orc_quantize(C.byref(d), mode, _p(K), _p(V), _p(kcode), _p(kmm), _p(vcode), _p(vmm))
    return {"kcode": kcode, "kmm": kmm, "vcode": vcode, "vmm": vmm}


def record_bytes(bits: int, group: int = 32) -> int:
    """Bytes of one record: a 32-token group at g = 32, a 64-token group at g = 64."""
    return int(lib().orc_unit_bytes(bits, group))


def records_per_pair(group: int, q_groups_cap: int) -> int:
    """Records per (b, hkv) for a capacity of q_groups_cap 32-token groups."""
    return int(lib().orc_units_cap(group, q_groups_cap))


def pack(d: orc_dims, qz, K, V, q_groups_cap=None, resid_cap=None):
    """Byte layout of C' (records) and the residual window, as the library stores them."""
    assert d.D == 128, "the packed layout is defined for head dim 128"
    n_q = nq(d)
    q_groups_cap = n_q // 32 if q_groups_cap is None else q_groups_cap
    resid_cap = (d.N - n_q) if resid_cap is None else resid_cap
    rec = np.zeros((d.B, d.Hkv, records_per_pair(d.group, q_groups_cap), record_bytes(d.bits, d.group)), np.uint8)
    res = np.zeros((d.B, d.Hkv, max(resid_cap, 0), 2, d.D), np.uint16)
    Kc, Vc = _c(K, np.uint16), _c(V, np.uint16)  # held until the call returns
    lib().orc_pack(C.byref(d), _p(qz["kcode"]), _p(qz["kmm"]), _p(qz["vcode"]), _p(qz["vmm"]),
                   _p(Kc), _p(Vc), q_groups_cap, resid_cap, _p(rec), _p(res))
    return rec, res


def attention(d: orc_dims, q, qz, K, V, idx=None, mode: int = 0, kv_self=None):
    """fp64 o [B,2,Hq,D], lse [B,2,Hq], S [B,Hkv,N_q] of the two-query attention.
    kv_self: bf16 bits [B,Hkv,2,D] or None, the speculative token's own key and
    value row, seen by the speculative query only."""
    q = _c(q, np.uint16)
    K = _c(K, np.uint16)
    V = _c(V, np.uint16)
    if kv_self is not None:
        kv_self = _c(kv_self, np.uint16)
    n_q = nq(d)
    k = 0
    if idx is not None:
        idx = _c(idx, np.int32)
        k = idx.shape[-1]
    o = np.zeros((d.B, 2, d.Hq, d.D), np.float64)
    lse = np.zeros((d.B, 2, d.Hq), np.float64)
    S = np.zeros((d.B, d.Hkv, n_q), np.float64)
    lib().orc_attention(C.byref(d), mode, _p(q), _p(qz["kcode"]), _p(qz["kmm"]), _p(qz["vcode"]),
                        _p(qz["vmm"]), _p(K), _p(V), _p(idx), k, _p(kv_self), _p(o), _p(lse), _p(S))
    return o, lse, S


def topk(d: orc_dims, S, k: int):
    """idx int32 [B,Hkv,k] ascending (-1 padded) and bitmap u32 [B,Hkv,ceil(N_q/32)]."""
    S = _c(S, np.float64)
    n_q = nq(d)
    idx = np.zeros((d.B, d.Hkv, k), np.int32)
    bm = np.zeros((d.B, d.Hkv, (n_q + 31) // 32), np.uint32)
    lib().orc_topk(C.byref(d), _p(S), k, _p(idx), _p(bm))
    return idx, bm


def append(d: orc_dims, records, resid, k_new, v_new, host=None):
    """Decode-time append of token d.N, in place on the packed cache (records
    as pack() lays them out, resid [B,Hkv,resid_cap,2,D] bf16) and, if given,
    the host cache [B,Hkv,n_cap,2,D].  The caller then advances d.N."""
    for a in (records, resid) + (() if host is None else (host,)):
        assert a.flags["C_CONTIGUOUS"], "append works in place on contiguous arrays"
    kn, vn = _c(k_new, np.uint16), _c(v_new, np.uint16)  # held until the call returns
    q_groups_cap = int(records.shape[2]) * (2 if d.group == 64 else 1)
    lib().orc_append(C.byref(d), q_groups_cap, int(resid.shape[2]), _p(kn), _p(vn),
                     _p(records), _p(resid), _p(host), 0 if host is None else int(host.shape[2]))


def gather(d: orc_dims, host, idx):
    """staging bf16 [B,Hkv,k,2,D] from host bf16 [B,Hkv,n_cap,2,D]."""
    host = _c(host, np.uint16)
    idx = _c(idx, np.int32)
    k = idx.shape[-1]
    st = np.zeros((d.B, d.Hkv, k, 2, d.D), np.uint16)
    lib().orc_gather(C.byref(d), _p(host), host.shape[2], _p(idx), k, _p(st))
    return st
