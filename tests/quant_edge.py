"""Adversarial inputs for the quantiser: groups built to sit on its decision
boundaries and at the edges of binary32 arithmetic.

Every key group (one channel over `group` tokens) and every value group (one
token over `group` channels) is filled from one of the patterns below, taken
in turn, so that each pattern lands on both axes and at every bit position of
the packed record.  Only bf16 bit patterns are produced here; the arithmetic
that decides codes lives in the oracle and in the kernels.

Patterns:
  midpoint1   1-bit boundary: min, max and values exactly at (min + max) / 2,
              where (x - z) / s = 1/2, and one bf16 step either side of it
  halfstep2   2-bit boundary: min = 0 or -1, max = 3 * 2^e, values at
              min + (i + 1/2) s exactly
  third2      2-bit with s = (max - min) / 3 not exact in binary32, values
              next to min + (i + 1/2) s (the quotient lands within 1e-5 of a
              half integer)
  constant    min = max (s = 0)
  zeros       +0 and -0, alone and with one small value
  subnormal   bf16 subnormals (and zero): s is subnormal, 1/s overflows
  tiny        min and max one bf16 step apart, at random exponents
  near_max    magnitudes next to the largest finite bf16, one sign (3 min + max
              overflows) or both signs (max - min overflows)
  wide        values spanning 2^-20 .. 2^20 with both signs
  absorbed    min = -max exactly (a zero midpoint) with tiny values of both
              signs around 0 (2^-40 .. 2^-20 of max) and zeros: x - z
              rounds to -z in binary32 for a run of them, so the 1-bit code
              changes far from the midpoint in bf16 order
  normal      N(0, 1) rounded to bf16 (control)
"""
from __future__ import annotations

import numpy as np

import synth

BF16_MAX = 0x7F7F  # largest finite bf16


def _bf16(x):
    return synth.f32_to_bf16_rne(np.asarray(x, np.float32)).astype(np.uint16)


def _neighbours(b):
    """The bf16 patterns one step below and one step above pattern b in value."""
    b = int(b)
    if b & 0x8000:  # negative: a larger magnitude is a smaller value
        up = 0x0001 if b == 0x8000 else b - 1
        return [np.uint16(b + 1), np.uint16(up)]
    down = 0x8001 if b == 0 else b - 1
    return [np.uint16(down), np.uint16(b + 1)]


def _fill(rng, L, values):
    """L patterns drawn from `values`, each of them at least once when L allows."""
    values = np.asarray(values, np.uint16)
    out = rng.choice(values, size=L)
    m = min(L, len(values))
    pos = rng.permutation(L)[:m]
    out[pos] = values[:m]
    return out


def _pattern(name, rng, L):
    if name == "midpoint1":
        e = int(rng.integers(-6, 6))
        lo = -float(rng.integers(1, 64)) * 2.0 ** e
        hi = lo + 2.0 * float(rng.integers(1, 64)) * 2.0 ** e  # even width: the midpoint is on the grid
        mid = _bf16((lo + hi) / 2)
        vals = [_bf16(lo), _bf16(hi), mid] + _neighbours(mid)
        # keep the group's extremes as stated
        v = synth.bf16_to_f32(np.array(vals, np.uint16))
        vals = [b for b, x in zip(vals, v) if lo <= x <= hi]
        return _fill(rng, L, vals)
    if name == "halfstep2":
        e = int(rng.integers(-8, 8))
        s = 2.0 ** e
        lo = float(rng.choice([0.0, -s]))
        hi = lo + 3 * s
        return _fill(rng, L, _bf16([lo, hi] + [lo + (i + 0.5) * s for i in range(3)] + [lo + i * s for i in range(4)]))
    if name == "third2":
        e = int(rng.integers(-6, 6))
        lo = float(rng.integers(-40, 40)) * 2.0 ** e
        hi = lo + float(rng.integers(1, 40)) * 2.0 ** e
        s = (hi - lo) / 3.0
        cand = [lo + (i + 0.5) * s for i in range(3)]
        b = _bf16(cand)
        vals = [_bf16(lo), _bf16(hi)]
        for x in b:  # the nearest bf16 values and their neighbours
            vals += [x] + _neighbours(x)
        v = synth.bf16_to_f32(np.array(vals, np.uint16))
        vals = [bb for bb, x in zip(vals, v) if np.isfinite(x) and lo <= x <= hi]
        return _fill(rng, L, vals)
    if name == "constant":
        return np.full(L, _bf16(rng.normal()), np.uint16)
    if name == "zeros":
        if rng.integers(0, 2):
            return _fill(rng, L, [0x0000, 0x8000])
        return _fill(rng, L, [0x0000, 0x8000, _bf16(float(rng.choice([-1, 1])) * 2.0 ** -10)])
    if name == "subnormal":
        mant = rng.integers(1, 128, size=4).astype(np.uint16)
        sign = rng.integers(0, 2, size=4).astype(np.uint16) << 15
        vals = list((mant | sign).astype(np.uint16)) + [0x0000, 0x0001, 0x8001]
        if rng.integers(0, 2):  # adjacent subnormals only
            a = int(rng.integers(1, 127))
            vals = [a, a + 1]
        return _fill(rng, L, vals)
    if name == "tiny":
        a = _bf16(float(rng.choice([-1, 1])) * 2.0 ** float(rng.integers(-120, 120)) * (1 + rng.random()))
        return _fill(rng, L, [a, _neighbours(a)[1]])
    if name == "near_max":
        pos = [BF16_MAX, BF16_MAX - 1, BF16_MAX - 5, 0x7F00, 0x7E80]
        neg = [p | 0x8000 for p in pos]
        kind = int(rng.integers(0, 3))
        vals = pos if kind == 0 else neg if kind == 1 else pos[:3] + neg[:3]
        return _fill(rng, L, vals)
    if name == "absorbed":
        a = float(2.0 ** rng.integers(-6, 6) * (1 + rng.integers(0, 128) / 128.0))
        tiny = a * np.power(2.0, rng.uniform(-40, -20, size=12)) * rng.choice([-1, 1], size=12)
        return _fill(rng, L, list(_bf16([a, -a])) + list(_bf16(tiny)) + [0x0000, 0x8000])
    if name == "wide":
        x = np.power(2.0, rng.uniform(-20, 20, size=L)) * rng.choice([-1, 1], size=L)
        return _bf16(x)
    assert name == "normal"
    return _bf16(rng.normal(size=L))


PATTERNS = ["midpoint1", "halfstep2", "third2", "constant", "zeros", "subnormal", "tiny", "near_max", "wide",
            "absorbed", "normal"]


def edge_kv(seed, B, Hkv, N, group=32, D=128):
    """bf16 K, V ([B, Hkv, N, D] uint16) whose groups follow PATTERNS in turn."""
    rng = np.random.default_rng(seed)
    K = np.zeros((B, Hkv, N, D), np.uint16)
    V = np.zeros((B, Hkv, N, D), np.uint16)
    i = 0
    for b in range(B):
        for h in range(Hkv):
            for g0 in range(0, N - group + 1, group):  # key groups: a channel over `group` tokens
                for c in range(D):
                    K[b, h, g0:g0 + group, c] = _pattern(PATTERNS[i % len(PATTERNS)], rng, group)
                    i += 1
            for n in range(N):  # value groups: a token over `group` channels
                for c0 in range(0, D, group):
                    V[b, h, n, c0:c0 + group] = _pattern(PATTERNS[i % len(PATTERNS)], rng, group)
                    i += 1
            # the tail that stays in the residual window: random
            tail = N - (N // group) * group
            if tail:
                K[b, h, N - tail:] = _bf16(rng.normal(size=(tail, D)))
    return K, V
