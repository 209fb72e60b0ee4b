"""Seeded synthetic inputs for the SpeCache decode path (numpy side).

This module draws the numbers; it holds none of the method's arithmetic.  The
oracle, the tests and the benchmark all take their inputs from here (or from
the CUDA twin of the same generator in ``synth/synth.cu``, which is checked to
give identical bytes), so both sides of every parity check see the same data.

Generator definition (both implementations follow it exactly):

* ``mix64`` is the SplitMix64 output function (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014; constants as in
  Vigna's public-domain splitmix64.c):
  z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31.
* A stream key is ``key = mix64(seed + GAMMA)`` followed, for every id in the
  stream's id tuple, by ``key = mix64(key ^ (id + GAMMA))`` (all mod 2**64),
  GAMMA = 0x9E3779B97F4A7C15.
* Element i (0-based) of a stream is ``r_i = mix64(key + (i + 1) * GAMMA)``,
  i.e. the i-th SplitMix64 output from state ``key``.
* A bf16 standard-normal draw from r: sign = r >> 63, u = r & (2**63 - 1),
  magnitude = VALS[#{j : THRESH[j] <= u}] from ``normal_bf16_table.npz``
  (see ``make_normal_table.py``): exactly N(0,1) rounded to nearest bf16, up
  to 2**-63 in probability.

Workload recipe (shapes of the pages' LLaMA-2-7B / LLaMA-3-8B / Mistral-7B
attention layers, SpeCache page, section 4):

* K, V for layer l: bf16 [B, Hkv, N, D], element (b,h,n,c) is draw number
  ((b*Hkv + h)*N + n)*D + c of streams (seed, TID_K, l) and (seed, TID_V, l).
* 4 outlier key channels per (layer, KV head), the same for every token and
  batch row, are multiplied by 8 (exact in bf16).  They are picked by a partial
  Fisher-Yates shuffle of 0..D-1 driven by draws h*4 .. h*4+3 of stream
  (seed, TID_OUTLIER, l): for i in 0..3, swap(perm[i], perm[i + r % (D - i)]).
* Queries for layer l: bf16 [B, 2, Hq, D]; the real query q[b,0,h,c] is draw
  (b*Hq + h)*D + c of stream (seed, TID_Q, l); the speculative query is
  bf16_rne(f32(q) + f32(0.1) * f32(z)) with z the same draw of stream
  (seed, TID_QSPEC, l), i.e. the real query plus N(0, 0.1^2) noise, computed
  in IEEE binary32 without fused multiply-add.
"""
from __future__ import annotations

import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)
MASK63 = np.uint64((1 << 63) - 1)

TID_K = 1
TID_V = 2
TID_Q = 3
TID_QSPEC = 4
TID_OUTLIER = 5

N_OUTLIERS = 4
OUTLIER_GAIN = 8.0
SPEC_NOISE_STD = 0.1

_HERE = os.path.dirname(os.path.abspath(__file__))
_TABLE = np.load(os.path.join(_HERE, "normal_bf16_table.npz"))
THRESH: np.ndarray = _TABLE["thresh"].astype(np.uint64)
VALS: np.ndarray = _TABLE["vals"].astype(np.uint16)


def mix64(z):
    """SplitMix64 output function on uint64 scalars or arrays (wrapping)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * M1
        z = z ^ (z >> np.uint64(27))
        z = z * M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, *ids: int) -> np.uint64:
    with np.errstate(over="ignore"):
        key = mix64(np.uint64(seed) + GAMMA)
        for i in ids:
            key = mix64(key ^ (np.uint64(i) + GAMMA))
    return np.uint64(key)


def uniform_u64(key, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the stream with key ``key``."""
    i = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (i + np.uint64(1)) * GAMMA)


def normal_bf16_from_u64(r: np.ndarray) -> np.ndarray:
    sign = (r >> np.uint64(63)).astype(np.uint16)
    u = r & MASK63
    j = np.searchsorted(THRESH, u, side="right")
    return VALS[j] | (sign << np.uint16(15))


def normal_bf16(key, start: int, count: int) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws start .. start+count-1."""
    out = np.empty(count, dtype=np.uint16)
    step = 1 << 22
    for s in range(0, count, step):
        n = min(step, count - s)
        out[s:s + n] = normal_bf16_from_u64(uniform_u64(key, start + s, n))
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round binary32 to bf16 (nearest, ties to even); inputs are finite."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = u + np.uint64(0x7FFF) + lsb
    return (u >> np.uint64(16)).astype(np.uint16)


def outlier_channels(seed: int, layer: int, Hkv: int, D: int = 128) -> np.ndarray:
    """int32 [Hkv, 4]: the outlier key channels of each KV head of a layer."""
    key = stream_key(seed, TID_OUTLIER, layer)
    out = np.empty((Hkv, N_OUTLIERS), dtype=np.int32)
    for h in range(Hkv):
        r = uniform_u64(key, h * N_OUTLIERS, N_OUTLIERS)
        perm = list(range(D))
        for i in range(N_OUTLIERS):
            j = i + int(r[i] % np.uint64(D - i))
            perm[i], perm[j] = perm[j], perm[i]
        out[h] = perm[:N_OUTLIERS]
    return out


def kv_slice(seed: int, layer: int, B: int, Hkv: int, N: int, D: int,
             b: int, h: int, n0: int = 0, n1: int | None = None):
    """K and V rows n0..n1-1 of (b, h) as bf16 bits, shape [n1-n0, D] each."""
    n1 = N if n1 is None else n1
    start = ((b * Hkv + h) * N + n0) * D
    count = (n1 - n0) * D
    k = normal_bf16(stream_key(seed, TID_K, layer), start, count).reshape(n1 - n0, D)
    v = normal_bf16(stream_key(seed, TID_V, layer), start, count).reshape(n1 - n0, D)
    ch = outlier_channels(seed, layer, Hkv, D)[h]
    k[:, ch] = f32_to_bf16_rne(bf16_to_f32(k[:, ch]) * np.float32(OUTLIER_GAIN))
    return k, v


def kv_layer(seed: int, layer: int, B: int, Hkv: int, N: int, D: int = 128):
    """Full K, V of one layer: bf16 bits [B, Hkv, N, D] each."""
    K = np.empty((B, Hkv, N, D), dtype=np.uint16)
    V = np.empty((B, Hkv, N, D), dtype=np.uint16)
    for b in range(B):
        for h in range(Hkv):
            K[b, h], V[b, h] = kv_slice(seed, layer, B, Hkv, N, D, b, h)
    return K, V


def queries(seed: int, layer: int, B: int, Hq: int, D: int = 128) -> np.ndarray:
    """bf16 bits [B, 2, Hq, D]: index 0 the real query, 1 the speculative one."""
    cnt = B * Hq * D
    q = normal_bf16(stream_key(seed, TID_Q, layer), 0, cnt).reshape(B, Hq, D)
    z = normal_bf16(stream_key(seed, TID_QSPEC, layer), 0, cnt).reshape(B, Hq, D)
    noise = np.float32(SPEC_NOISE_STD) * bf16_to_f32(z)
    spec = f32_to_bf16_rne(bf16_to_f32(q) + noise)
    return np.stack([q, spec], axis=1)
