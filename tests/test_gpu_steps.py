"""The per-layer steps of the SpeCache page (Algorithms 1-3) end to end
against the oracle: the prefill's quantise + offload, the pre-decoding step
(append, single-query attention, ArgTopK, Pre-fetch) and two decoding steps
(append, merged two-query attention with the fetched rows, ArgTopK over the
speculative row, Pre-fetch)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from spc_cases import OUT_TOL, b2f, check_topk_sets, out_err

pytestmark = pytest.mark.gpu


def dev16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("n_extra", [0, 5])
def test_prefill_layer_quantises_and_offloads(n_extra):
    """Offload(C): the host cache holds every K then V row, bit for bit (one
    strided copy when the host rows are contiguous, per-(b, hkv) copies when
    n_cap > N); the low-bit cache is the quantiser's."""
    import bit_kv_cache_spc_gb300 as spc
    from bit_kv_cache_spc_gb300.steps import prefill_layer
    B, Hq, Hkv, N, R, bits = 2, 8, 2, 1000, 40, 1
    K, V = synth.kv_layer(7, 0, B, Hkv, N)
    d = spc.Dims(B, Hq, Hkv, N, R, bits)
    rec = torch.zeros(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
    res = torch.zeros(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
    n_cap = N + n_extra
    host = torch.full((B, Hkv, n_cap, 2, 128), -1, dtype=torch.int16, pin_memory=True)
    copy_stream = torch.cuda.Stream()
    done = prefill_layer(d, dev16(K), dev16(V), rec, res, host, n_cap, copy_stream=copy_stream)
    done.synchronize()
    torch.cuda.synchronize()
    h = host.numpy().view(np.uint16)
    assert np.array_equal(h[:, :, :N], np.stack([K, V], axis=3))
    assert np.all(h[:, :, N:] == 0xFFFF)
    od = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=bits)
    orec, ores = oracle.pack(od, oracle.quantize(od, K, V), K, V)
    assert np.array_equal(rec.cpu().numpy(), orec.reshape(-1))
    r = N - oracle.nq(od)
    assert np.array_equal(res.cpu().numpy().view(np.uint16).reshape(B, Hkv, -1, 2, 128)[:, :, :r], ores[:, :, :r])


@pytest.mark.parametrize("keep", [False, True])
def test_predecode_then_two_decode_steps_match_oracle(keep):
    """Algorithm 2 then Algorithm 3 twice on one layer.  Token 999 completes a
    group at the pre-decoding step (a flush).  At every step the GPU's outputs
    are compared with the oracle's attention over the same cache and the same
    substituted rows, its selection with the oracle's ArgTopK, and the staged
    rows with the host cache at the selected positions.  keep: the rows the
    previous selection staged are copied from its staging buffer, not
    re-read from the host."""
    import bit_kv_cache_spc_gb300 as spc
    from bit_kv_cache_spc_gb300.steps import decode_layer, predecode_layer
    B, Hq, Hkv, R, bits, k = 2, 8, 2, 40, 1, 33
    G = Hq // Hkv
    N0, steps = 999, 2
    N1 = N0 + 1 + steps
    scale = float(np.float32(1.0 / math.sqrt(128)))
    K, V = synth.kv_layer(9, 0, B, Hkv, N1)
    cap, rcap, n_cap = N1 // 32 + 1, R + 32, N1 + 1
    d = spc.Dims(B, Hq, Hkv, N0, R, bits, q_groups_cap=cap, resid_cap=rcap, scale=scale)
    rec = torch.zeros(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
    res = torch.zeros(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
    spc.spc_quantize_kv(d, dev16(K[:, :, :N0]), dev16(V[:, :, :N0]), rec, res)
    host = torch.zeros((B, Hkv, n_cap, 2, 128), dtype=torch.int16, pin_memory=True)
    host[:, :, :N0] = torch.from_numpy(np.stack([K[:, :, :N0], V[:, :, :N0]], axis=3).view(np.int16))
    Kn, Vn = dev16(K.transpose(2, 0, 1, 3)), dev16(V.transpose(2, 0, 1, 3))  # [token][B][Hkv][D]
    o = torch.zeros((B, 2, Hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.zeros((B, 2, Hq), dtype=torch.float32, device="cuda")
    lg = torch.zeros((B, Hkv, G, cap * 32), dtype=torch.float32, device="cuda")
    # the workspace is sized for the largest cache the steps reach
    ws_bytes = spc.spc_attn_workspace_bytes(spc.Dims(B, Hq, Hkv, N1, R, bits, q_groups_cap=cap, resid_cap=rcap), k)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    idx = [torch.zeros((B, Hkv, k), dtype=torch.int32, device="cuda") for _ in range(2)]
    bm = [torch.zeros((B, Hkv, cap), dtype=torch.int32, device="cuda") for _ in range(2)]
    st = [torch.zeros((B, Hkv, k, 2, 128), dtype=torch.int16, device="cuda") for _ in range(2)]
    q2 = torch.empty((B, 2, Hq, 128), dtype=torch.int16, device="cuda")
    src = torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda") if keep else None

    def oracle_check(n_tokens, q, sub_idx):
        od = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=n_tokens, R=R, bits=bits, scale=scale)
        Kc, Vc = K[:, :, :n_tokens], V[:, :, :n_tokens]
        oo, lo, S = oracle.attention(od, q, oracle.quantize(od, Kc, Vc), Kc, Vc, idx=sub_idx)
        return od, oo, lo, S

    # ---- pre-decoding: token N0's query alone ----
    q1 = synth.queries(9, 0, B, Hq)[:, 0]
    predecode_layer(d, rec, res, host, n_cap, dev16(q1), Kn[N0], Vn[N0], k, idx[0], bm[0], st[0], o, lse, lg, ws,
                    ws_bytes, q2)
    torch.cuda.synchronize()
    assert d.N == N0 + 1
    od, oo, lo, S = oracle_check(N0 + 1, np.stack([q1, q1], axis=1), None)
    got = b2f(o.cpu().numpy())
    assert out_err(got, oo) <= OUT_TOL
    io, _ = oracle.topk(od, S, k)
    sel = idx[0].cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            check_topk_sets(sel[b, h], io[b, h], S[b, h], k)
            assert np.array_equal(st[0].cpu().numpy().view(np.uint16)[b, h],
                                  np.stack([K, V], axis=3)[b, h, sel[b, h]])

    # ---- decoding steps: the real token plus a speculative token ----
    cur = 0
    for t in range(steps):
        n = N0 + 1 + t  # this step's real token joins the cache first
        q = synth.queries(9, 1 + t, B, Hq)
        used = idx[cur].cpu().numpy()
        decode_layer(d, rec, res, host, n_cap, dev16(q), Kn[n], Vn[n], k, idx[cur], bm[cur], st[cur],
                     idx[1 - cur], bm[1 - cur], st[1 - cur], o, lse, lg, ws, ws_bytes, src=src)
        torch.cuda.synchronize()
        assert d.N == n + 1
        od, oo, lo, S = oracle_check(n + 1, q, used)
        assert out_err(b2f(o.cpu().numpy()), oo) <= OUT_TOL
        assert np.max(np.abs(lse.cpu().numpy() - lo)) <= 1e-3
        io, _ = oracle.topk(od, S, k)
        sel = idx[1 - cur].cpu().numpy()
        staged = st[1 - cur].cpu().numpy().view(np.uint16)
        for b in range(B):
            for h in range(Hkv):
                check_topk_sets(sel[b, h], io[b, h], S[b, h], k)
                assert np.array_equal(staged[b, h], np.stack([K, V], axis=3)[b, h, sel[b, h]])
        cur = 1 - cur
    assert np.array_equal(host.numpy().view(np.uint16)[:, :, :N1], np.stack([K, V], axis=3))
