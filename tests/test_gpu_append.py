"""Parity of the decode-time append (spc_append_kv) with the oracle.

A run of single-token appends, crossing at least one flush of the residual
window into a new record, is compared byte for byte with the oracle's append
(records, window, host cache), and the appended cache then decodes like the
oracle's attention over all tokens.  At the configuration-4 shape one append
that flushes is checked on sampled (batch, KV head) pairs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from spc_cases import OUT_TOL, b2f, out_err

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=2, Hkv=3, Hq=6, R=16, bits=1, N0=50, T=45),
    dict(B=2, Hkv=3, Hq=6, R=16, bits=2, N0=75, T=40),
    dict(B=1, Hkv=2, Hq=8, R=0, bits=1, N0=20, T=50),     # R = 0: the new row completes the flushed group
    dict(B=1, Hkv=2, Hq=8, R=128, bits=2, N0=100, T=70),  # starts with no quantised token
    dict(B=2, Hkv=2, Hq=8, R=16, bits=1, N0=40, T=90, group=64),  # g = 64: 64-row flushes
    dict(B=1, Hkv=3, Hq=6, R=0, bits=2, N0=10, T=60, group=64),
]


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"b{c['bits']}_R{c['R']}_N{c['N0']}+{c['T']}_g{c.get('group', 32)}")
def test_append_sequence_matches_oracle(c):
    import bit_kv_cache_spc_gb300 as spc
    B, Hkv, Hq, R, bits, N0, T = (c[x] for x in ("B", "Hkv", "Hq", "R", "bits", "N0", "T"))
    group = c.get("group", 32)
    N1 = N0 + T
    D = 128
    K, V = synth.kv_layer(5, bits, B, Hkv, N1)
    cap, rcap, n_cap = N1 // 32 + 2, R + group, N1 + 2
    scale = float(np.float32(1.0 / math.sqrt(D)))
    d = spc.Dims(B, Hq, Hkv, N0, R, bits, q_groups_cap=cap, resid_cap=rcap, scale=scale, group=group)
    rec = torch.zeros(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
    res = torch.zeros(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
    spc.spc_quantize_kv(d, dev16(K[:, :, :N0]), dev16(V[:, :, :N0]), rec, res)
    host = torch.zeros((B, Hkv, n_cap, 2, D), dtype=torch.int16, pin_memory=True)
    host[:, :, :N0] = torch.from_numpy(np.stack([K[:, :, :N0], V[:, :, :N0]], axis=3).view(np.int16))
    Kn = dev16(K.transpose(2, 0, 1, 3))  # [N1, B, Hkv, D]: token n's rows contiguous
    Vn = dev16(V.transpose(2, 0, 1, 3))

    od = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N0, R=R, bits=bits, scale=scale, group=group)
    qz = oracle.quantize(od, K[:, :, :N0], V[:, :, :N0])
    orec, ores = oracle.pack(od, qz, K[:, :, :N0], V[:, :, :N0], q_groups_cap=cap, resid_cap=rcap)
    ohost = np.zeros((B, Hkv, n_cap, 2, D), np.uint16)
    ohost[:, :, :N0] = np.stack([K[:, :, :N0], V[:, :, :N0]], axis=3)
    flushes = 0
    for n in range(N0, N1):
        before = oracle.nq(od)
        spc.spc_append_kv(d, Kn[n], Vn[n], rec, res, host, n_cap)
        d.N += 1
        oracle.append(od, orec, ores, K[:, :, n], V[:, :, n], ohost)
        od.N += 1
        flushes += oracle.nq(od) > before
    torch.cuda.synchronize()
    assert flushes >= 1
    nq1 = oracle.nq(od)
    assert spc.spc_num_quantized(d) == nq1
    r1 = N1 - nq1
    got_rec = rec.cpu().numpy().reshape(B, Hkv, oracle.records_per_pair(group, cap), -1)
    assert np.array_equal(got_rec[:, :, :nq1 // group], orec[:, :, :nq1 // group])
    got_res = res.cpu().numpy().view(np.uint16).reshape(B, Hkv, rcap, 2, D)
    assert np.array_equal(got_res[:, :, :r1], ores[:, :, :r1])
    assert np.array_equal(host.numpy().view(np.uint16), ohost)

    # the appended cache decodes like the oracle's attention over all N1 tokens
    q = synth.queries(5, 0, B, Hq)
    G = Hq // Hkv
    o = torch.zeros((B, 2, Hq, D), dtype=torch.int16, device="cuda")
    lse = torch.zeros((B, 2, Hq), dtype=torch.float32, device="cuda")
    lg = torch.zeros((B, Hkv, G, cap * 32), dtype=torch.float32, device="cuda")
    ws = torch.zeros(spc.spc_attn_workspace_bytes(d, 0), dtype=torch.uint8, device="cuda")
    spc.spc_decode_attn2(d, rec, res, dev16(q), o, lse, lg, ws)
    od1 = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N1, R=R, bits=bits, scale=scale, group=group)
    oo, lo, _ = oracle.attention(od1, q, oracle.quantize(od1, K, V), K, V)
    torch.cuda.synchronize()
    assert out_err(b2f(o.cpu().numpy()), oo) <= OUT_TOL
    assert np.max(np.abs(lse.cpu().numpy() - lo)) <= 1e-3


def test_append_flush_at_config4_shape_sampled():
    """LLaMA-3-8B shape (B=8, 32/8 heads, R=128, 1 bit): token 32799 completes
    group 1020, so the append flushes; sampled pairs against the oracle."""
    import bit_kv_cache_spc_gb300 as spc
    import synth.gpu
    B, Hq, Hkv, R, bits, D = 8, 32, 8, 128, 1, 128
    N1 = 32800
    N0 = N1 - 1
    K1 = torch.empty((B, Hkv, N1, D), dtype=torch.int16, device="cuda")
    V1 = torch.empty_like(K1)
    synth.gpu.kv_layer_into(0, 3, K1, V1)
    cap, rcap = N1 // 32 + 1, R + 32
    d = spc.Dims(B, Hq, Hkv, N0, R, bits, q_groups_cap=cap, resid_cap=rcap)
    rec = torch.zeros(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
    res = torch.zeros(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
    spc.spc_quantize_kv(d, K1[:, :, :N0].contiguous(), V1[:, :, :N0].contiguous(), rec, res)
    nq0 = spc.spc_num_quantized(d)
    spc.spc_append_kv(d, K1[:, :, N0].contiguous(), V1[:, :, N0].contiguous(), rec, res)
    d.N += 1
    nq1 = spc.spc_num_quantized(d)
    assert (nq0, nq1) == (32640, 32672)
    torch.cuda.synchronize()
    RB = oracle.record_bytes(bits)
    got_rec = rec.view(B, Hkv, cap, RB)
    got_res = res.view(B, Hkv, rcap, 2, D)
    for (b, h) in [(0, 0), (3, 5), (7, 7)]:
        kk, vv = synth.kv_slice(0, 3, B, Hkv, N1, D, b, h)
        od = oracle.dims(B=1, Hq=Hq // Hkv, Hkv=1, N=N1, R=R, bits=bits)
        orec, ores = oracle.pack(od, oracle.quantize(od, kk[None, None], vv[None, None]), kk[None, None],
                                 vv[None, None], q_groups_cap=cap, resid_cap=rcap)
        g = nq1 // 32 - 1
        assert np.array_equal(got_rec[b, h, g].cpu().numpy(), orec[0, 0, g])
        r1 = N1 - nq1
        assert np.array_equal(got_res[b, h, :r1].cpu().numpy().view(np.uint16), ores[0, 0, :r1])
