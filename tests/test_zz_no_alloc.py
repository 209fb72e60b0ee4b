"""The allocation-free attention entry point.

Some callers of this library cannot allocate device memory (a plug-in inside
a host that owns the allocator, or a path that must not synchronise the way
cudaMalloc can), so spc_merged_attn_noalloc runs the merged attention with a
workspace built into the library.  This checks it through the C ABI against
spc_merged_attn with a caller workspace, on two calls in a row (the built-in
buffer keeps the previous call's contents): both run the same kernels on the
same workspace layout, so the results must be identical bit for bit.  Also
that argument errors return spc_merged_attn's statuses and a shape too large
for the buffer is refused.  The file is named to be collected last.
"""
import pytest
import torch

import synth
from spc_cases import GpuLayer

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_variant_on_two_calls():
    import bit_kv_cache_spc_gb300 as spc
    cfg = dict(B=2, Hq=8, Hkv=2, N=4096, R=128, bits=1, k=41)
    K, V = synth.kv_layer(4, 0, cfg["B"], cfg["Hkv"], cfg["N"])
    g = GpuLayer(cfg, K=K, V=V, q=synth.queries(4, 0, cfg["B"], cfg["Hq"]))
    o0, lse0, lg0 = g.attn2()
    idx, bm = g.topk(lg0, lse0, cfg["k"])
    g.gather(idx, cfg["k"])
    ref_o, ref_lse, ref_lg = g.merged(idx, bm, cfg["k"])
    for _ in range(2):
        o, lse, lg = g.new_out()
        spc.spc_merged_attn_noalloc(g.d, g.records, g.resid, g.q, idx, bm, g.staging, cfg["k"], o, lse, lg)
        torch.cuda.synchronize()
        nq = g.nq
        assert torch.equal(o, ref_o)
        assert torch.equal(lse, ref_lse)
        assert torch.equal(lg[..., :nq], ref_lg[..., :nq])


def test_noalloc_refuses_shapes_beyond_its_buffer():
    import bit_kv_cache_spc_gb300 as spc
    d = spc.Dims(64, 256, 64, 262144, 128, 1)  # needs far more than the built-in buffer
    assert spc.spc_attn_workspace_bytes(d, 0) > (8 << 20)
    with pytest.raises(spc.SpcError) as e:
        spc.spc_merged_attn_noalloc(d, 16, 16, 16, 16, 16, 16, 1, 16, 16, 16)
    assert e.value.status == 5
    # argument errors come first, with spc_merged_attn's statuses
    g8 = spc.Dims(1, 64, 8, 1024, 32, 1)  # G = 8: unsupported shape
    with pytest.raises(spc.SpcError) as e:
        spc.spc_merged_attn_noalloc(g8, 16, 16, 16, 16, 16, 16, 1, 16, 16, 16)
    assert e.value.status == 2
    with pytest.raises(spc.SpcError) as e:  # misaligned output
        spc.spc_merged_attn_noalloc(spc.Dims(1, 4, 1, 1024, 32, 1), 16, 16, 16, 16, 16, 16, 1, 17, 16, 16)
    assert e.value.status == 1
