"""Pre-fetch that keeps the rows already staged (SpeCache page, section 3,
pre-fetching and offloading during decoding: the used 16-bit rows outside the
new top-k are evicted, so the rows inside it stay).

spc_topk_select_prev says where each selected position sat in the previous
selection; spc_merged_attn_fetch_prev copies those rows from the previous
staging buffer and reads only the others from the host.  Checked here: src
against a search of the previous selection (both top-k paths), the routing of
every staged row, and a two-layer decode pipeline with double-buffered staging
that must reproduce the pipeline that re-fetches every row, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synth
import bit_kv_cache_spc_gb300 as spc
from spc_cases import GpuLayer

pytestmark = pytest.mark.gpu


def want_src(idx, prev):
    """Index of each entry of idx in prev (ascending, -1 padded), else -1."""
    out = np.full(idx.shape, -1, np.int32)
    for r in np.ndindex(idx.shape[:-1]):
        p = prev[r]
        valid = p[p >= 0]
        for j, v in enumerate(idx[r]):
            if v < 0:
                continue
            i = np.searchsorted(valid, v)
            if i < len(valid) and valid[i] == v:
                out[r + (j,)] = i
    return out


@pytest.mark.parametrize("B,Hq,Hkv,N,k,prev_k", [(2, 8, 2, 32768, 328, 328), (1, 4, 2, 16384, 164, 200),
                                                 (1, 4, 2, 65536 + 128, 2500, 2500), (2, 4, 4, 1000, 900, 40),
                                                 (1, 4, 2, 32768, 328, 3000)])
def test_topk_prev_src(B, Hq, Hkv, N, k, prev_k):
    """idx and bitmap as spc_topk_select's; src the previous slot of every
    selected position.  The previous selection is the top prev_k of nearby
    logits (partial overlap); k = 2500 takes the radix path; k = 900 of 864
    positions pads with -1; a previous selection of 3000 (more than the 2048
    the selection copies into shared memory) is searched in device memory."""
    rng = np.random.default_rng(N + k)
    d = spc.Dims(B, Hq, Hkv, N, 128, 1)
    G = Hq // Hkv
    nq = spc.spc_num_quantized(d)
    Lcap = d.q_groups_cap * 32
    lg = np.zeros((B, Hkv, G, Lcap), np.float32)
    lg[..., :nq] = (2.0 * rng.standard_normal((B, Hkv, G, nq))).astype(np.float32)
    lse = (8.0 + rng.standard_normal((B, 2, Hq))).astype(np.float32)
    lg_prev = lg.copy()
    lg_prev[..., :nq] += (0.7 * rng.standard_normal((B, Hkv, G, nq))).astype(np.float32)
    dev = lambda a: torch.from_numpy(a).cuda()
    prev = torch.full((B, Hkv, prev_k), -7, dtype=torch.int32, device="cuda")
    pbm = torch.zeros((B, Hkv, d.q_groups_cap), dtype=torch.int32, device="cuda")
    spc.spc_topk_select(d, dev(lg_prev), dev(lse), prev_k, prev, pbm)
    idx0 = torch.full((B, Hkv, k), -7, dtype=torch.int32, device="cuda")
    bm0 = torch.zeros_like(pbm)
    spc.spc_topk_select(d, dev(lg), dev(lse), k, idx0, bm0)
    idx = torch.full_like(idx0, -7)
    bm = torch.full_like(bm0, 0x5A5A)
    src = torch.full((B, Hkv, k), -7, dtype=torch.int32, device="cuda")
    spc.spc_topk_select_prev(d, dev(lg), dev(lse), k, idx, bm, prev, prev_k, src)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx0) and torch.equal(bm, bm0)
    got = src.cpu().numpy()
    want = want_src(idx.cpu().numpy(), prev.cpu().numpy())
    assert np.array_equal(got, want)
    shared = (got >= 0).sum()
    assert shared > 0
    if prev_k <= k:
        assert shared < (idx.cpu().numpy() >= 0).sum()  # a partial overlap, both kinds of rows present


@pytest.mark.parametrize("cfg", [dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41),
                                 dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=2, k=41),
                                 dict(B=2, Hq=8, Hkv=2, N=4200, R=40, bits=1, k=41, group=64),
                                 dict(B=1, Hq=4, Hkv=2, N=2100, R=64, bits=2, k=20, group=64)],
                         ids=lambda c: f"b{c['bits']}_g{c.get('group', 32)}")
def test_fetch_prev_routes_staged_rows(cfg):
    """A row whose src is >= 0 comes from the previous staging buffer, every
    other from the host cache: the previous buffer is filled from a second
    cache, so each output row shows where it was read.  The attention's own
    results are those of spc_merged_attn.  Every bit width and group size
    (the carried pre-fetch rides on each one's low-bit loop)."""
    g = GpuLayer(cfg, seed=3)
    B, Hkv, k = cfg["B"], cfg["Hkv"], cfg["k"]
    o0, lse0, lg0 = g.attn2()
    idx, bm = g.topk(lg0, lse0, k)
    g.gather(idx, k)
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, k)
    n2 = 600
    K2, V2 = synth.kv_layer(21, 1, B, Hkv, n2)
    K3, V3 = synth.kv_layer(22, 1, B, Hkv, n2)
    host2 = torch.from_numpy(np.stack([K2, V2], axis=3).view(np.int16)).pin_memory()
    other = np.stack([K3, V3], axis=3).view(np.uint16)  # [B][Hkv][n2][2][D]
    rng = np.random.default_rng(4)
    fk, pk = 70, 50
    fidx = np.sort(np.stack([np.stack([rng.choice(n2, fk, replace=False) for _ in range(Hkv)]) for _ in range(B)]),
                   axis=-1).astype(np.int32)
    pidx = np.sort(np.stack([np.stack([rng.choice(n2, pk, replace=False) for _ in range(Hkv)]) for _ in range(B)]),
                   axis=-1).astype(np.int32)
    src = want_src(fidx, pidx)
    assert (src >= 0).any() and (src < 0).any()
    prev = np.take_along_axis(other, pidx[..., None, None], axis=2)  # the previous rows, from the second cache
    prev_d = torch.from_numpy(prev.view(np.int16).copy()).cuda()
    fst = torch.zeros((B, Hkv, fk, 2, 128), dtype=torch.int16, device="cuda")
    o, lse, lg = g.new_out()
    spc.spc_merged_attn_fetch_prev(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, lg, g.ws, host2, n2,
                                   torch.from_numpy(fidx).cuda(), fk, fst, torch.from_numpy(src).cuda(), prev_d, pk)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert torch.equal(lg[..., :g.nq], ref_lg[..., :g.nq])
    got = fst.cpu().numpy().view(np.uint16)
    d2 = oracle.dims(B=B, Hq=cfg["Hq"], Hkv=Hkv, N=n2, R=0, bits=1)
    from_host = oracle.gather(d2, np.stack([K2, V2], axis=3), fidx)
    from_prev = np.take_along_axis(other, fidx[..., None, None], axis=2)
    want = np.where((src >= 0)[..., None, None], from_prev, from_host)
    assert np.array_equal(got, want)


def test_host_gather_prev_routes_staged_rows():
    """The standalone pre-fetch with kept rows: rows whose src is >= 0 come
    from the previous staging buffer (filled from a second cache), the others
    from the host cache; a bounded grid (max_ctas) gives the same rows."""
    B, Hq, Hkv, n2 = 2, 8, 4, 900
    d = spc.Dims(B, Hq, Hkv, n2, 128, 1)
    K2, V2 = synth.kv_layer(23, 0, B, Hkv, n2)
    K3, V3 = synth.kv_layer(24, 0, B, Hkv, n2)
    host = torch.from_numpy(np.stack([K2, V2], axis=3).view(np.int16)).pin_memory()
    other = np.stack([K3, V3], axis=3).view(np.uint16)
    rng = np.random.default_rng(5)
    fk, pk = 120, 90
    pick = lambda m: np.sort(np.stack([np.stack([rng.choice(n2, m, replace=False) for _ in range(Hkv)])
                                       for _ in range(B)]), axis=-1).astype(np.int32)
    fidx, pidx = pick(fk), pick(pk)
    src = want_src(fidx, pidx)
    assert (src >= 0).any() and (src < 0).any()
    prev_d = torch.from_numpy(np.take_along_axis(other, pidx[..., None, None], axis=2).view(np.int16).copy()).cuda()
    d2 = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=n2, R=0, bits=1)
    want = np.where((src >= 0)[..., None, None], np.take_along_axis(other, fidx[..., None, None], axis=2),
                    oracle.gather(d2, np.stack([K2, V2], axis=3), fidx))
    for max_ctas in (0, 3):
        st = torch.zeros((B, Hkv, fk, 2, 128), dtype=torch.int16, device="cuda")
        spc.spc_host_gather_prev(d, host, n2, torch.from_numpy(fidx).cuda(), fk, st, torch.from_numpy(src).cuda(),
                                 prev_d, pk, max_ctas=max_ctas)
        torch.cuda.synchronize()
        assert np.array_equal(st.cpu().numpy().view(np.uint16), want)


def test_two_layer_pipeline_with_kept_rows_equals_full_refetch():
    """Two layers, three decode steps, each layer's attention carrying the
    other layer's pre-fetch (layer 1 carries layer 0's selection of the same
    step, layer 0 the selection layer 1 made in the step before).  Pipeline A
    re-fetches every row into one staging buffer per layer; pipeline B keeps
    the staged rows: double-buffered selections and staging by step parity,
    spc_topk_select_prev and spc_merged_attn_fetch_prev.  Outputs, speculative
    logits and selections agree bit for bit at every call."""
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    B, Hkv, k, N = cfg["B"], cfg["Hkv"], cfg["k"], cfg["N"]
    L = [GpuLayer(cfg, seed=30 + l, layer=l) for l in range(2)]
    d = L[0].d
    zi = lambda: torch.full((B, Hkv, k), -1, dtype=torch.int32, device="cuda")
    zb = lambda: torch.zeros((B, Hkv, d.q_groups_cap), dtype=torch.int32, device="cuda")
    zs = lambda: torch.zeros((B, Hkv, k, 2, 128), dtype=torch.int16, device="cuda")
    idxA, bmA, stA = [zi(), zi()], [zb(), zb()], [zs(), zs()]
    idxB = [[zi(), zi()], [zi(), zi()]]  # [parity][layer]
    bmB = [[zb(), zb()], [zb(), zb()]]
    stB = [[zs(), zs()], [zs(), zs()]]
    src = [zi(), zi()]
    # pre-decoding: plain attention, the first selection and its gather (parity 0 for pipeline B)
    for l in range(2):
        o, lse, lg = L[l].attn2()
        spc.spc_topk_select(d, lg, lse, k, idxA[l], bmA[l])
        spc.spc_topk_select(d, lg, lse, k, idxB[0][l], bmB[0][l])
        spc.spc_host_gather(d, L[l].host, N, idxA[l], k, stA[l])
        spc.spc_host_gather(d, L[l].host, N, idxB[0][l], k, stB[0][l])
    torch.cuda.synchronize()
    reused = 0
    for t in range(3):
        P = t % 2
        for l in range(2):
            j = 1 - l
            oA, lseA, lgA = L[l].new_out()
            spc.spc_merged_attn_fetch(d, L[l].records, L[l].resid, L[l].q, idxA[l], bmA[l], stA[l], k, oA, lseA,
                                      lgA, L[l].ws, L[j].host, N, idxA[j], k, stA[j])
            oB, lseB, lgB = L[l].new_out()
            if l == 1:  # layer 0's selection of this step: written to parity 1 - P
                fidx, fout, fprev = idxB[1 - P][0], stB[1 - P][0], stB[P][0]
            else:  # layer 1's selection of the previous step (pre-decoding at t = 0): parity P
                fidx, fout, fprev = idxB[P][1], stB[P][1], stB[1 - P][1]
            spc.spc_merged_attn_fetch_prev(d, L[l].records, L[l].resid, L[l].q, idxB[P][l], bmB[P][l], stB[P][l],
                                           k, oB, lseB, lgB, L[l].ws, L[j].host, N, fidx, k, fout, src[j], fprev, k)
            torch.cuda.synchronize()
            assert torch.equal(oA, oB) and torch.equal(lseA, lseB), (t, l)
            assert torch.equal(lgA[..., :L[l].nq], lgB[..., :L[l].nq]), (t, l)
            spc.spc_topk_select(d, lgA, lseA, k, idxA[l], bmA[l])
            spc.spc_topk_select_prev(d, lgB, lseB, k, idxB[1 - P][l], bmB[1 - P][l], idxB[P][l], k, src[l])
            torch.cuda.synchronize()
            assert torch.equal(idxA[l], idxB[1 - P][l]) and torch.equal(bmA[l], bmB[1 - P][l]), (t, l)
            reused += int((src[l] >= 0).sum())
    # layer 0's rows fetched in the last step (t = 2, written to parity 1) match the full re-fetch
    assert torch.equal(stA[0], stB[1][0])
    assert reused > 0


@pytest.mark.parametrize("cfg,on_chip", [
    (dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41), True),
    (dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41), False),
    (dict(B=8, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328), True),   # the LLaMA-3-8B decode shape
    (dict(B=2, Hq=8, Hkv=2, N=40000, R=128, bits=1, k=400), False),   # many chunks
    (dict(B=1, Hq=4, Hkv=2, N=40000, R=128, bits=1, k=3000), False),  # the selection in its own launch
], ids=lambda c: str(c) if isinstance(c, bool) else f"B{c['B']}_N{c['N']}_k{c['k']}")
def test_decode_step_prev_equals_separate_calls(cfg, on_chip):
    """spc_decode_step_prev against spc_merged_attn_fetch_prev followed by
    spc_topk_select_prev on the same inputs: outputs, selection, bitmap, the
    selection's slots in the call's own idx and the kept-row pre-fetch of
    another layer's rows, bit for bit; with the logits on chip and in device
    memory, and with a selection too large to ride on the attention."""
    g = GpuLayer(cfg, seed=12)
    B, Hkv, k = cfg["B"], cfg["Hkv"], cfg["k"]
    o0, lse0, lg0 = g.attn2()
    idx, bm = g.topk(lg0, lse0, k)
    idx, bm = idx.contiguous(), bm.contiguous()
    g.gather(idx, k)
    n2, fk, pk = 700, 60, 45
    if on_chip and spc.spc_decode_step_on_chip(g.d, k, fk, k) != 1:
        pytest.skip("this shape keeps its logits in device memory")
    K2, V2 = synth.kv_layer(25, 1, B, Hkv, n2)
    K3, V3 = synth.kv_layer(26, 1, B, Hkv, n2)
    host2 = torch.from_numpy(np.stack([K2, V2], axis=3).view(np.int16)).pin_memory()
    other = np.stack([K3, V3], axis=3).view(np.uint16)
    rng = np.random.default_rng(7)
    pick = lambda m: np.sort(np.stack([np.stack([rng.choice(n2, m, replace=False) for _ in range(Hkv)])
                                       for _ in range(B)]), axis=-1).astype(np.int32)
    fidx, pidx = pick(fk), pick(pk)
    src = torch.from_numpy(want_src(fidx, pidx)).cuda()
    prev_d = torch.from_numpy(np.take_along_axis(other, pidx[..., None, None], axis=2).view(np.int16).copy()).cuda()
    fidx_d = torch.from_numpy(fidx).cuda()
    # the separate calls
    fst_r = torch.zeros((B, Hkv, fk, 2, 128), dtype=torch.int16, device="cuda")
    o_r, lse_r, lg_r = g.new_out()
    spc.spc_merged_attn_fetch_prev(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o_r, lse_r, lg_r, g.ws, host2,
                                   n2, fidx_d, fk, fst_r, src, prev_d, pk)
    nidx_r = torch.full_like(idx, -7)
    nbm_r = torch.full_like(bm, 0x77)
    nsrc_r = torch.full_like(idx, -7)
    spc.spc_topk_select_prev(g.d, lg_r, lse_r, k, nidx_r, nbm_r, idx, k, nsrc_r)
    # the fused step
    ws = torch.zeros(spc.spc_step_workspace_bytes(g.d, k), dtype=torch.uint8, device="cuda")
    fst = torch.zeros_like(fst_r)
    o, lse, lg = g.new_out()
    nidx, nbm, nsrc = torch.full_like(idx, -9), torch.full_like(bm, 0x55), torch.full_like(idx, -9)
    spc.spc_decode_step_prev(g.d, g.records, g.resid, g.q, idx, bm, g.staging, k, o, lse, None if on_chip else lg, k,
                             nidx, nbm, nsrc, ws, fetch_host_kv=host2, fetch_n_cap=n2, fetch_idx=fidx_d, fetch_k=fk,
                             fetch_staging=fst, fetch_src=src, fetch_prev_staging=prev_d, fetch_prev_k=pk)
    torch.cuda.synchronize()
    assert torch.equal(o, o_r) and torch.equal(lse, lse_r)
    if not on_chip:
        assert torch.equal(lg[..., :g.nq], lg_r[..., :g.nq])
    assert torch.equal(nidx, nidx_r) and torch.equal(nbm, nbm_r) and torch.equal(nsrc, nsrc_r)
    assert np.array_equal(nsrc.cpu().numpy(), want_src(nidx.cpu().numpy(), idx.cpu().numpy()))
    assert (nsrc.cpu().numpy() >= 0).any()
    assert torch.equal(fst, fst_r)
    assert spc.spc_read_device_status(ws, g.d) == 0
