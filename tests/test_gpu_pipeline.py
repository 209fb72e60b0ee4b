"""The multi-layer decode schedule (bit_kv_cache_spc_gb300.pipeline) against
the same steps run layer after layer on one stream.

In the schedule, layer l's attention carries the pre-fetch of another layer's
selection and the top-k runs on a second stream; with kept rows the
selections and staging alternate by step parity and only new rows are read
from the host.  Per step, every layer must still attend over the rows of its
own previous selection and select from its own speculative logits, so the
outputs, selections and bitmaps equal those of the plain per-layer sequence
(gather, merged attention, top-k) bit for bit, and the staged rows equal the
oracle's gather of the host cache.
"""
import numpy as np
import pytest
import torch

import oracle
import bit_kv_cache_spc_gb300 as spc
from bit_kv_cache_spc_gb300.pipeline import DecodePipeline
from spc_cases import GpuLayer, odims

pytestmark = pytest.mark.gpu


def make_pipeline(cfg, n_layers, lag, keep, seed=40):
    layers = [GpuLayer(cfg, seed=seed + l, layer=l) for l in range(n_layers)]
    d, k = layers[0].d, cfg["k"]
    outs = [g.new_out() for g in layers]
    ws = torch.zeros(spc.spc_attn_workspace_bytes(d, k), dtype=torch.uint8, device="cuda")
    pipe = DecodePipeline(d, k, [g.records for g in layers], [g.resid for g in layers], [g.host for g in layers],
                          cfg["N"], [g.q for g in layers], [x[0] for x in outs], [x[1] for x in outs],
                          [x[2] for x in outs], ws, ws.numel(), lag=lag, keep=keep)
    return layers, pipe


@pytest.mark.parametrize("keep", [True, False], ids=["kept_rows", "refetch"])
@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("n_layers,lag", [(3, 2), (4, 3), (2, 1)])
def test_pipeline_equals_layer_by_layer(keep, graph, n_layers, lag):
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    k = cfg["k"]
    layers, pipe = make_pipeline(cfg, n_layers, lag, keep)
    pipe.predecode()
    torch.cuda.synchronize()
    # the reference's own pre-decoding selection of every layer
    ref = []
    for l, g in enumerate(layers):
        o0, lse0, lg0 = g.attn2()
        idx, bm = g.topk(lg0, lse0, k)
        ref.append((idx.contiguous(), bm.contiguous()))
        assert torch.equal(pipe.idx[0][l], ref[l][0]) and torch.equal(pipe.bitmap[0][l], ref[l][1]), l
    graphs = pipe.capture() if graph else None
    kept = 0
    for t in range(4):
        if graph:
            graphs.replay()
        else:
            pipe.step()
        torch.cuda.synchronize()
        nidx, nbm = pipe.selection(pipe.parity)  # the selections the next step reads
        for l, g in enumerate(layers):
            g.gather(ref[l][0], k)
            ro, rlse, rlg = g.merged(ref[l][0], ref[l][1], k)
            assert torch.equal(pipe.o[l], ro) and torch.equal(pipe.lse[l], rlse), (t, l)
            assert torch.equal(pipe.logits[l][..., :g.nq], rlg[..., :g.nq]), (t, l)
            idx, bm = g.topk(rlg, rlse, k)
            ref[l] = (idx.contiguous(), bm.contiguous())
            assert torch.equal(nidx[l], ref[l][0]) and torch.equal(nbm[l], ref[l][1]), (t, l)
        # the first L - lag layers' new rows are staged within the step (the others ride on the next step)
        P = pipe.parity if keep else 0
        for l in range(n_layers - pipe.lag):
            host = layers[l].host.numpy().view(np.uint16)
            want = oracle.gather(odims(cfg), host, ref[l][0].cpu().numpy())
            got = pipe.staging[P][l].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want), (t, l)
        if keep:
            kept += sum(int((s >= 0).sum()) for s in pipe.src)
    assert (kept > 0) == keep
    frac = pipe.kept_fraction()
    assert (frac is None) != keep and (frac is None or 0.0 < frac <= 1.0)


@pytest.mark.parametrize("bits,group,Hq", [(2, 32, 8), (1, 64, 8), (2, 64, 8), (1, 32, 4), (1, 32, 2)],
                         ids=["b2g32", "b1g64", "b2g64", "G2", "G1"])
def test_pipeline_other_codes(bits, group, Hq):
    """The schedule with 2-bit codes, 64-token groups and query groups of 1
    and 2 heads, kept rows, as graphs: outputs and selections bit-identical
    to the layer-by-layer calls."""
    cfg = dict(B=2, Hq=Hq, Hkv=2, N=4096 + 96, R=128, bits=bits, k=41, group=group)
    k = cfg["k"]
    layers, pipe = make_pipeline(cfg, 3, 2, True, seed=90)
    pipe.predecode()
    torch.cuda.synchronize()
    ref = []
    for g in layers:
        o0, lse0, lg0 = g.attn2()
        idx, bm = g.topk(lg0, lse0, k)
        ref.append((idx.contiguous(), bm.contiguous()))
    graphs = pipe.capture()
    for t in range(3):
        graphs.replay()
        torch.cuda.synchronize()
        nidx, nbm = pipe.selection(pipe.parity)
        for l, g in enumerate(layers):
            g.gather(ref[l][0], k)
            ro, rlse, rlg = g.merged(ref[l][0], ref[l][1], k)
            assert torch.equal(pipe.o[l], ro) and torch.equal(pipe.lse[l], rlse), (t, l)
            idx, bm = g.topk(rlg, rlse, k)
            ref[l] = (idx.contiguous(), bm.contiguous())
            assert torch.equal(nidx[l], ref[l][0]) and torch.equal(nbm[l], ref[l][1]), (t, l)


def test_pipeline_hooks_bracket_every_call():
    """on_attention / on_topk run before and after each layer's call, on the
    stream the call is enqueued on; without the selection no top-k hook runs."""
    cfg = dict(B=1, Hq=4, Hkv=1, N=1024, R=64, bits=1, k=24)
    layers, pipe = make_pipeline(cfg, 3, 2, True)
    pipe.predecode()
    seen = []
    pipe.enqueue(parity=0, on_attention=lambda l, w, s: seen.append(("a", l, w, s is pipe.main)),
                 on_topk=lambda l, w, s: seen.append(("t", l, w, s is pipe.side)))
    want = []
    for l in range(3):
        want += [("a", l, 0, True), ("a", l, 1, True), ("t", l, 0, True), ("t", l, 1, True)]
    assert seen == want
    seen.clear()
    pipe.enqueue(parity=1, topk=False, on_attention=lambda l, w, s: seen.append(l),
                 on_topk=lambda l, w, s: seen.append(-1))
    assert seen == [0, 0, 1, 1, 2, 2]
    torch.cuda.synchronize()


def test_pipeline_refuses_a_lag_that_reads_its_own_fetch():
    cfg = dict(B=1, Hq=4, Hkv=1, N=1024, R=64, bits=1, k=24)
    for n_layers, lag in ((2, 2), (3, 0), (1, 1)):
        with pytest.raises(ValueError):
            make_pipeline(cfg, n_layers, lag, True)


def test_pipeline_at_the_llama3_8b_decode_shape():
    """The timed schedule at the LLaMA-3-8B decode shape (B=8, 32/8 heads,
    32K context, 1 bit, k=328: the benchmark's launch configuration), three
    layers, kept rows, captured as graphs: outputs and selections bit-identical
    to the layer-by-layer calls, and the staged rows of one sampled
    (b, KV head) per step equal to the oracle's gather of the host cache."""
    cfg = dict(B=8, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328)
    k, n_layers = cfg["k"], 3
    layers, pipe = make_pipeline(cfg, n_layers, 2, True, seed=60)
    pipe.predecode()
    torch.cuda.synchronize()
    ref = []
    for l, g in enumerate(layers):
        o0, lse0, lg0 = g.attn2()
        idx, bm = g.topk(lg0, lse0, k)
        ref.append((idx.contiguous(), bm.contiguous()))
    graphs = pipe.capture()
    d1 = odims(cfg, B=1, Hkv=1, Hq=cfg["Hq"] // cfg["Hkv"])
    for t in range(3):
        graphs.replay()
        torch.cuda.synchronize()
        nidx, nbm = pipe.selection(pipe.parity)
        for l, g in enumerate(layers):
            g.gather(ref[l][0], k)
            ro, rlse, rlg = g.merged(ref[l][0], ref[l][1], k)
            assert torch.equal(pipe.o[l], ro) and torch.equal(pipe.lse[l], rlse), (t, l)
            idx, bm = g.topk(rlg, rlse, k)
            ref[l] = (idx.contiguous(), bm.contiguous())
            assert torch.equal(nidx[l], ref[l][0]) and torch.equal(nbm[l], ref[l][1]), (t, l)
        b, h = (3 * t + 1) % cfg["B"], (5 * t + 2) % cfg["Hkv"]
        host = layers[0].host[b:b + 1, h:h + 1].numpy().view(np.uint16)
        want = oracle.gather(d1, host, ref[0][0][b:b + 1, h:h + 1].cpu().numpy())
        got = pipe.staging[pipe.parity][0][b:b + 1, h:h + 1].cpu().numpy().view(np.uint16)
        assert np.array_equal(got, want), t
    assert 0.0 < pipe.kept_fraction() <= 1.0


def test_readme_decode_example():
    """The README's decode example, as written there, at a small shape: the
    prefill through steps.prefill_layer, the pipeline's pre-decoding step and
    graph replays with new queries written in place; every layer's outputs
    and selections then equal the layer-by-layer calls on the same caches."""
    import synth
    import synth.gpu
    from bit_kv_cache_spc_gb300.steps import prefill_layer
    B, Hq, Hkv, N, R, bits, L, T = 2, 8, 2, 4096, 128, 1, 3, 3
    d = spc.Dims(B, Hq, Hkv, N, R, bits)
    k = 41
    dev = "cuda"
    K, V = [], []
    for l in range(L):
        Kt = torch.empty((B, Hkv, N, 128), dtype=torch.int16, device=dev)
        Vt = torch.empty_like(Kt)
        synth.gpu.kv_layer_into(70, l, Kt, Vt)
        K.append(Kt)
        V.append(Vt)
    # --- as in the README ---
    records = [torch.empty(spc.spc_records_bytes(d), dtype=torch.uint8, device=dev) for _ in range(L)]
    resid = [torch.empty(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device=dev) for _ in range(L)]
    host = [torch.empty((B, Hkv, N, 2, 128), dtype=torch.int16, pin_memory=True) for _ in range(L)]
    for l in range(L):
        prefill_layer(d, K[l], V[l], records[l], resid[l], host[l], N)
    q = [torch.empty((B, 2, Hq, 128), dtype=torch.int16, device=dev) for _ in range(L)]
    o = [torch.empty((B, 2, Hq, 128), dtype=torch.int16, device=dev) for _ in range(L)]
    lse = [torch.empty((B, 2, Hq), dtype=torch.float32, device=dev) for _ in range(L)]
    logits = [torch.empty((B, Hkv, Hq // Hkv, d.q_groups_cap * 32), dtype=torch.float32, device=dev)
              for _ in range(L)]
    ws = torch.zeros(spc.spc_attn_workspace_bytes(d, k), dtype=torch.uint8, device=dev)
    queries = lambda t, l: torch.from_numpy(synth.queries(80 + t, l, B, Hq).view(np.int16).copy()).to(dev)
    for l in range(L):
        q[l].copy_(queries(0, l))
    pipe = DecodePipeline(d, k, records, resid, host, N, q, o, lse, logits, ws, ws.numel())
    pipe.predecode()
    graphs = pipe.capture()
    # --- the reference: the same caches, one layer after another ---
    cfg = dict(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=bits, k=k)
    ref_layers = [GpuLayer(cfg, seed=70, layer=l) for l in range(L)]
    ref = []
    for l, g in enumerate(ref_layers):
        g.q.copy_(queries(0, l))
        o0, lse0, lg0 = g.attn2()
        idx, bm = g.topk(lg0, lse0, k)
        ref.append((idx.contiguous(), bm.contiguous()))
    for t in range(1, T + 1):
        for l in range(L):
            q[l].copy_(queries(t, l))
        graphs.replay()
        torch.cuda.synchronize()
        nidx, nbm = pipe.selection(pipe.parity)
        for l, g in enumerate(ref_layers):
            g.q.copy_(queries(t, l))
            g.gather(ref[l][0], k)
            ro, rlse, rlg = g.merged(ref[l][0], ref[l][1], k)
            assert torch.equal(o[l], ro) and torch.equal(lse[l], rlse), (t, l)
            idx, bm = g.topk(rlg, rlse, k)
            ref[l] = (idx.contiguous(), bm.contiguous())
            assert torch.equal(nidx[l], ref[l][0]) and torch.equal(nbm[l], ref[l][1]), (t, l)
