"""spc_decode_step: the merged attention with ArgTopK fused at its end.

Its outputs must equal, bit for bit, those of the separate calls it replaces
(spc_merged_attn[_fetch] then spc_topk_select on the same inputs): the scores
are computed with the same operations in the same order, and the selection
rule (ties to the lower position) is exact.  A wait that nothing releases
must run out and be reported, not hang.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from spc_cases import GpuLayer

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=2, Hq=8, Hkv=2, N=1000, R=40, bits=1, k=33),       # ragged residual
    dict(B=2, Hq=4, Hkv=2, N=2080, R=128, bits=2, k=20),      # G = 2, 2-bit
    dict(B=1, Hq=4, Hkv=4, N=300, R=64, bits=2, k=7),         # G = 1
    dict(B=1, Hq=4, Hkv=1, N=96, R=32, bits=1, k=200),        # k > N_q
    dict(B=2, Hq=8, Hkv=2, N=40000, R=128, bits=1, k=400),    # many chunks
    dict(B=8, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328),   # the LLaMA-3-8B decode shape
    dict(B=2, Hq=8, Hkv=2, N=4200, R=40, bits=1, k=41, group=64),   # g = 64 records
    dict(B=1, Hq=4, Hkv=2, N=2100, R=64, bits=2, k=20, group=64),   # g = 64, 2-bit
]


def cid(c):
    return f"B{c['B']}_Hq{c['Hq']}_Hkv{c['Hkv']}_N{c['N']}_b{c['bits']}_k{c['k']}_g{c.get('group', 32)}"


def prepare(cfg, seed=3):
    g = GpuLayer(cfg, seed=seed, host=cfg["N"] <= 40000)
    k = cfg["k"]
    o0, lse0, lg0 = g.attn2()
    idx, bm = g.topk(lg0, lse0, k)
    idx, bm = idx.contiguous(), bm.contiguous()
    if g.host is not None:
        g.gather(idx, k)
    return g, idx, bm


@pytest.mark.parametrize("cfg", CASES, ids=cid)
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("with_self", [False, True])
def test_decode_step_equals_separate_calls(cfg, in_place, with_self):
    import bit_kv_cache_spc_gb300 as spc
    g, idx, bm = prepare(cfg)
    k = cfg["k"]
    ks = None
    if with_self:  # the speculative token's own key/value row
        K1, V1 = synth.kv_layer(15, 0, cfg["B"], cfg["Hkv"], 1)
        ks = torch.from_numpy(np.stack([K1[:, :, 0], V1[:, :, 0]], axis=2).view(np.int16).copy()).cuda()
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k, kv_self=ks)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, k)
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    o, lse, lg = g.new_out()
    if in_place:
        nidx, nbm = idx.clone(), bm.clone()
        src_idx, src_bm = nidx, nbm
    else:
        nidx = torch.full_like(idx, -9)
        nbm = torch.full_like(bm, 0x77)
        src_idx, src_bm = idx, bm
    for rep in range(2):  # the second call checks that the workspace's control words were reset
        if rep == 1 and in_place:
            src_idx.copy_(idx)
            src_bm.copy_(bm)
        spc.spc_decode_step(g.d, g.records, g.resid, g.q, src_idx, src_bm, g.staging, k, o, lse, lg, k, nidx, nbm, ws,
                            kv_self=ks)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        assert torch.equal(lg[..., :g.nq], ref_lg[..., :g.nq])
        assert torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)
    assert spc.spc_read_device_status(ws, g.d) == 0


def test_decode_step_with_fetch_job():
    """The pre-fetch riding along is copied exactly, and the results are unchanged."""
    import bit_kv_cache_spc_gb300 as spc
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    g, idx, bm = prepare(cfg, seed=5)
    k = cfg["k"]
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, k)
    K2, V2 = synth.kv_layer(9, 1, cfg["B"], cfg["Hkv"], 500)
    host2 = torch.from_numpy(np.stack([K2, V2], axis=3).view(np.int16)).pin_memory()
    rng = np.random.default_rng(4)
    fk = 70
    fidx = np.sort(rng.choice(500, size=(cfg["B"], cfg["Hkv"], fk)), axis=-1).astype(np.int32)
    fidx[1, 0, 2] = -1
    fst = torch.zeros((cfg["B"], cfg["Hkv"], fk, 2, 128), dtype=torch.int16, device="cuda")
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    o, lse, lg = g.new_out()
    nidx, nbm = torch.empty_like(idx), torch.empty_like(bm)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, lg, k, nidx, nbm, ws,
                        fetch_host_kv=host2, fetch_n_cap=500, fetch_idx=torch.from_numpy(fidx).cuda(), fetch_k=fk,
                        fetch_staging=fst)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)
    d2 = oracle.dims(B=cfg["B"], Hq=cfg["Hq"], Hkv=cfg["Hkv"], N=500, R=0, bits=1)
    want = oracle.gather(d2, np.stack([K2, V2], axis=3), fidx)
    assert np.array_equal(fst.cpu().numpy().view(np.uint16), want)


def test_decode_step_falls_back_when_the_selection_does_not_fit():
    """next_k too large for the attention's shared memory: the selection runs
    as its own launch, with the same results."""
    import bit_kv_cache_spc_gb300 as spc
    cfg = dict(B=1, Hq=4, Hkv=1, N=70000, R=128, bits=1, k=40)
    g, idx, bm = prepare(cfg, seed=6)
    k, nk = cfg["k"], 5000
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, nk)
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, nk), dtype=torch.uint8, device="cuda")
    o, lse, lg = g.new_out()
    nidx = torch.empty((1, 1, nk), dtype=torch.int32, device="cuda")
    nbm = torch.empty_like(bm)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, lg, nk, nidx, nbm, ws)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)


def test_decode_step_wait_that_nothing_releases_runs_out():
    """With (b, hkv) 0's ticket preset so that none of its CTAs is ever the
    last, the log-sum-exp is never published: every wait of that (b, hkv)
    must end at its time limit, and the fault is reported once."""
    import bit_kv_cache_spc_gb300 as spc
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    g, idx, bm = prepare(cfg, seed=7)
    k = cfg["k"]
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[0] = 1 << 20  # ticket of (b, hkv) 0
    o, lse, lg = g.new_out()
    nidx, nbm = torch.empty_like(idx), torch.empty_like(bm)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, lg, k, nidx, nbm, ws)
    torch.cuda.synchronize()
    assert spc.spc_read_device_status(ws, g.d) == 6  # SPC_ERR_TIMEOUT
    assert spc.spc_read_device_status(ws, g.d) == 0  # cleared by the read


ONCHIP = [c for c in CASES if c["k"] > 0]


@pytest.mark.parametrize("cfg", ONCHIP, ids=cid)
@pytest.mark.parametrize("with_self", [False, True])
def test_decode_step_with_logits_on_chip_equals_separate_calls(cfg, with_self):
    """spec_logits=None: each CTA keeps its chunk's speculative logits in TMEM
    from the low-bit loop to its selection.  Outputs, selection and bitmap
    must equal the separate calls' bit for bit."""
    import bit_kv_cache_spc_gb300 as spc
    g, idx, bm = prepare(cfg, seed=8)
    k = cfg["k"]
    if spc.spc_decode_step_on_chip(g.d, k, 0, k) != 1:
        pytest.skip("this shape keeps its logits in device memory")
    ks = None
    if with_self:
        K1, V1 = synth.kv_layer(16, 0, cfg["B"], cfg["Hkv"], 1)
        ks = torch.from_numpy(np.stack([K1[:, :, 0], V1[:, :, 0]], axis=2).view(np.int16).copy()).cuda()
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k, kv_self=ks)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, k)
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    o, lse, _ = g.new_out()
    nidx = torch.full_like(idx, -9)
    nbm = torch.full_like(bm, 0x77)
    for _ in range(2):  # the workspace's control words are reset by each call
        spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, None, k, nidx, nbm, ws,
                            kv_self=ks)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
        assert torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)
    assert spc.spc_read_device_status(ws, g.d) == 0


def test_decode_step_on_chip_with_fetch_job_and_limits():
    """On-chip logits with a pre-fetch riding along; the LLaMA-3-8B decode
    shape qualifies, a shape whose warps hold more than 32 groups does not
    and refuses spec_logits=None."""
    import bit_kv_cache_spc_gb300 as spc
    d4 = spc.Dims(8, 32, 8, 32768, 128, 1)
    assert spc.spc_decode_step_on_chip(d4, 328, 328, 328) == 1
    big = spc.Dims(4, 32, 8, 131072, 128, 1)
    assert spc.spc_decode_step_on_chip(big, 1311, 0, 1311) == 0
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    g, idx, bm = prepare(cfg, seed=9)
    k = cfg["k"]
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, k)
    K2, V2 = synth.kv_layer(10, 1, cfg["B"], cfg["Hkv"], 500)
    host2 = torch.from_numpy(np.stack([K2, V2], axis=3).view(np.int16)).pin_memory()
    rng = np.random.default_rng(6)
    fk = 70
    fidx = np.sort(rng.choice(500, size=(cfg["B"], cfg["Hkv"], fk)), axis=-1).astype(np.int32)
    fst = torch.zeros((cfg["B"], cfg["Hkv"], fk, 2, 128), dtype=torch.int16, device="cuda")
    assert spc.spc_decode_step_on_chip(g.d, k, fk, k) == 1
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    o, lse, _ = g.new_out()
    nidx, nbm = torch.empty_like(idx), torch.empty_like(bm)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, None, k, nidx, nbm, ws,
                        fetch_host_kv=host2, fetch_n_cap=500, fetch_idx=torch.from_numpy(fidx).cuda(), fetch_k=fk,
                        fetch_staging=fst)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)
    d2 = oracle.dims(B=cfg["B"], Hq=cfg["Hq"], Hkv=cfg["Hkv"], N=500, R=0, bits=1)
    assert np.array_equal(fst.cpu().numpy().view(np.uint16), oracle.gather(d2, np.stack([K2, V2], axis=3), fidx))
    # a shape that cannot keep its logits on chip refuses a missing logits buffer
    cfgb = dict(B=4, Hq=32, Hkv=8, N=131072, R=128, bits=1, k=1311)
    gb = GpuLayer(cfgb, host=False)
    wsb = torch.zeros(spc.spc_step_workspace_bytes(gb.d, cfgb["k"]), dtype=torch.uint8, device="cuda")
    ob, lseb, _ = gb.new_out()
    ib = torch.zeros((4, 8, cfgb["k"]), dtype=torch.int32, device="cuda")
    bb = torch.zeros((4, 8, gb.d.q_groups_cap), dtype=torch.int32, device="cuda")
    with pytest.raises(spc.SpcError) as e:
        spc.spc_decode_step(gb.d, gb.records, gb.resid, gb.q, ib, bb, gb.staging, cfgb["k"], ob, lseb, None, cfgb["k"],
                            ib, bb, wsb)
    assert e.value.status == 2


def test_decode_step_on_chip_wait_that_nothing_releases_runs_out():
    """The same run-out with the logits on chip: the CTAs that waited still
    score their chunk from tensor memory and release it, and the fault is
    reported once."""
    import bit_kv_cache_spc_gb300 as spc
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    g, idx, bm = prepare(cfg, seed=7)
    k = cfg["k"]
    assert spc.spc_decode_step_on_chip(g.d, k, 0, k) == 1
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    ws.view(torch.int32)[0] = 1 << 20  # ticket of (b, hkv) 0
    o, lse, _ = g.new_out()
    nidx, nbm = torch.empty_like(idx), torch.empty_like(bm)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, None, k, nidx, nbm, ws)
    torch.cuda.synchronize()
    assert spc.spc_read_device_status(ws, g.d) == 6  # SPC_ERR_TIMEOUT
    assert spc.spc_read_device_status(ws, g.d) == 0
    # the device is still usable: a clean call on a fresh workspace matches the separate calls
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k)
    ref_idx, ref_bm = g.topk(ref_lg, ref_lse, k)
    ws2 = torch.zeros_like(ws)
    spc.spc_decode_step(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, None, k, nidx, nbm, ws2)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(nidx, ref_idx) and torch.equal(nbm, ref_bm)
