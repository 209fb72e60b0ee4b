"""Write synth/normal_bf16_table.npz: the inverse-CDF table behind synth.normal_bf16.

The table makes "a standard normal sample rounded to bf16" a pure integer
function of a 63-bit uniform, so the numpy and CUDA generators give identical
bytes on any machine.

Before trimming, entry j of VALS is the j-th non-negative bf16 bit pattern
(0x0000 = 0.0 up to 0x4180 = 16.0) and THRESH[j] is floor(P(|X| < m_j) * 2**63)
for X ~ N(0,1), where m_j is the midpoint between VALS[j] and VALS[j+1], i.e. the
round-to-nearest boundary between the two bf16 magnitudes.  A uniform u in
[0, 2**63) maps to the magnitude VALS[#{j : THRESH[j] <= u}].  Magnitudes that
no u can reach (threshold 0 below, saturated thresholds above) are trimmed;
len(VALS) == len(THRESH) + 1 always.  P(|X| > 16) is below 2**-180.

The CDF is evaluated with mpmath at 60 significant digits, which makes the
table independent of the platform's libm.  Run:  python synth/make_normal_table.py
"""
import os

import mpmath
import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "normal_bf16_table.npz")
LAST = 0x4180  # bf16 bit pattern of 16.0


def bf16_bits_to_float(bits: int) -> mpmath.mpf:
    f32 = np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]
    return mpmath.mpf(float(f32))


def build():
    mpmath.mp.dps = 60
    vals = np.arange(0, LAST + 1, dtype=np.uint16)
    two63 = mpmath.mpf(2) ** 63
    thresh = np.zeros(LAST, dtype=np.uint64)
    sqrt2 = mpmath.sqrt(2)
    prev = bf16_bits_to_float(0)
    for j in range(LAST):
        nxt = bf16_bits_to_float(j + 1)
        mid = (prev + nxt) / 2
        p = mpmath.erf(mid / sqrt2)  # P(|X| < mid)
        t = int(mpmath.floor(p * two63))
        thresh[j] = np.uint64(min(t, (1 << 63) - 1))
        prev = nxt
    assert np.all(np.diff(thresh.astype(object)) >= 0)
    # Magnitudes whose threshold is 0 can never be drawn (every u passes
    # them), and only the first saturated threshold can matter: trim both ends.
    lo = int(np.count_nonzero(thresh == 0))
    top = np.uint64((1 << 63) - 1)
    hi = int(np.argmax(thresh == top)) + 1 if np.any(thresh == top) else LAST
    np.savez(OUT, thresh=thresh[lo:hi], vals=vals[lo:hi + 1])
    return OUT


if __name__ == "__main__":
    print(build())
