"""The quantiser on adversarial groups, bit for bit against the oracle.

The kernel decides most codes by multiplying by the correctly rounded
reciprocal of s and falls back to the IEEE quotient near a rounding boundary;
these groups sit on the boundaries (1-bit midpoints, exact and inexact 2-bit
half steps), have no range (constant groups, +0 / -0), live in the subnormal
range (s subnormal, 1/s overflowing) or next to the largest bf16 (3 min + max
or max - min overflowing binary32).  Records (codes and min/max words) and
residual rows must equal the oracle's bytes exactly, through the C ABI, for
both bit widths and both group sizes.
"""
import numpy as np
import pytest
import torch

import oracle
from quant_edge import edge_kv
from spc_cases import GpuLayer, odims

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("bits", [1, 2])
def test_quantiser_edge_groups_bit_exact(bits, group):
    B, Hkv = 2, 2
    N = 20 * group + 39  # R = 32: N_q = 20 g, a 39-row residual window
    cfg = dict(B=B, Hq=Hkv, Hkv=Hkv, N=N, R=32, bits=bits, k=0, group=group)
    K, V = edge_kv(100 + 10 * bits + group, B, Hkv, N, group)
    q = np.zeros((B, 2, Hkv, 128), np.uint16)
    g = GpuLayer(cfg, K=K, V=V, q=q, host=False)
    d = odims(cfg)
    qz = oracle.quantize(d, K, V)
    rec, res = oracle.pack(d, qz, K, V)
    torch.cuda.synchronize()
    got = g.records.cpu().numpy()[:rec.size]
    bad = np.flatnonzero(got != rec.reshape(-1))
    assert bad.size == 0, f"{bad.size} record bytes differ, first at {bad[:8]}"
    r = N - g.nq
    got_res = g.resid.cpu().numpy().view(np.uint16).reshape(B, Hkv, -1, 2, 128)[:, :, :r]
    assert np.array_equal(got_res, res[:, :, :r])
