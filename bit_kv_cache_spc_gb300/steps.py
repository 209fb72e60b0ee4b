"""The SpeCache page's per-layer steps (Algorithms 1-3) as sequences of the
library's C-ABI calls.

Nothing here computes: every step runs in libspc's kernels or copy-engine
copies; this module only orders the calls on the caller's streams and keeps
the cache length in the dims struct.

    prefill_layer   Algorithm 1: Quant(K), Quant(V) into the low-bit cache,
                    then Offload(C) of the 16-bit K/V to the pinned host cache
                    on a copy stream (section 3, "Prefilling").
    predecode_layer Algorithm 2: append the first token's K/V, attention of
                    its single query over the cache, ArgTopK over that
                    attention, Pre-fetch of the selected 16-bit rows.
    decode_layer    Algorithm 3: the append (and offload) of the real token's
                    K/V, the two-query attention over C' with the fetched rows
                    substituted, ArgTopK over the speculative row, Pre-fetch.
"""
from __future__ import annotations

import torch

from . import (spc_append_kv, spc_decode_attn2, spc_host_gather, spc_host_gather_prev, spc_merged_attn,
               spc_offload_kv, spc_quantize_kv, spc_topk_select, spc_topk_select_prev)


def prefill_layer(d, k, v, records, resid, host_kv, n_cap, stream=None, copy_stream=None):
    """Quantise the layer's K and V (bf16 [B][Hkv][N][D], device) into
    records/resid on `stream`, and offload them to host_kv on `copy_stream`
    (default: `stream`).  Returns the event after which k and v may be freed."""
    stream = torch.cuda.current_stream() if stream is None else stream
    copy_stream = stream if copy_stream is None else copy_stream
    spc_quantize_kv(d, k, v, records, resid, stream=stream.cuda_stream)
    ready = torch.cuda.Event()
    ready.record(stream)
    copy_stream.wait_event(ready)
    spc_offload_kv(d, k, v, host_kv, n_cap, stream=copy_stream.cuda_stream)
    done = torch.cuda.Event()
    done.record(copy_stream)
    return done


def predecode_layer(d, records, resid, host_kv, n_cap, q1, k1, v1, k, idx, bitmap, staging, o, lse, logits, ws,
                    ws_bytes, q2, stream=None, fetch_stream=None):
    """Algorithm 2 for one layer.  q1: bf16 [B][Hq][D]; k1, v1: bf16
    [B][Hkv][D], the first generated token's rows.  The token's K/V joins the
    cache (d.N is advanced) and is offloaded to host_kv; the single query's
    attention is the two-query attention with both rows equal to q1 (q2 is a
    [B][2][Hq][D] scratch tensor), so its second row is the real token's and
    feeds ArgTopK.  The Pre-fetch runs on `fetch_stream` (default: `stream`)
    after the selection; the returned event marks its end."""
    stream = torch.cuda.current_stream() if stream is None else stream
    fetch_stream = stream if fetch_stream is None else fetch_stream
    s = stream.cuda_stream
    spc_append_kv(d, k1, v1, records, resid, host_kv, n_cap, stream=s)
    d.N += 1
    with torch.cuda.stream(stream):
        q2.copy_(q1.unsqueeze(1).expand(-1, 2, -1, -1))
    spc_decode_attn2(d, records, resid, q2, o, lse, logits, ws, ws_bytes, stream=s)
    spc_topk_select(d, logits, lse, k, idx, bitmap, stream=s)
    selected = torch.cuda.Event()
    selected.record(stream)
    fetch_stream.wait_event(selected)
    spc_host_gather(d, host_kv, n_cap, idx, k, staging, stream=fetch_stream.cuda_stream)
    fetched = torch.cuda.Event()
    fetched.record(fetch_stream)
    return fetched


def decode_layer(d, records, resid, host_kv, n_cap, q, k_t, v_t, k, idx, bitmap, staging, next_idx, next_bitmap,
                 next_staging, o, lse, logits, ws, ws_bytes, stream=None, fetch_stream=None, kv_self=None,
                 src=None):
    """Algorithm 3 for one layer.  The real token's K/V (k_t, v_t: bf16
    [B][Hkv][D]) first joins the cache and is offloaded (d.N is advanced), so
    both queries see it; q: bf16 [B][2][Hq][D] (the real token, then the
    speculative token).  idx/bitmap/staging hold the rows fetched for this
    step (selected at the previous step); the merged attention substitutes
    them, the speculative row's probabilities select next_idx/next_bitmap,
    and their Pre-fetch into next_staging runs on `fetch_stream`.  The
    speculative token's own K/V (kv_self: bf16 [B][Hkv][2][D], optional) is
    seen by the speculative query only and is not part of the cache.  With
    src (int32 [B][Hkv][k], scratch), the rows of the new selection that this
    step's selection already staged are copied from `staging` and only the
    others are read from the host (the used rows outside the new top-k are
    the ones evicted); next_staging is the same either way.  Returns the
    event that ends the Pre-fetch."""
    stream = torch.cuda.current_stream() if stream is None else stream
    fetch_stream = stream if fetch_stream is None else fetch_stream
    s = stream.cuda_stream
    spc_append_kv(d, k_t, v_t, records, resid, host_kv, n_cap, stream=s)
    d.N += 1
    spc_merged_attn(d, records, resid, q, idx, bitmap, staging, k, o, lse, logits, ws, ws_bytes, stream=s,
                    kv_self=kv_self)
    if src is None:
        spc_topk_select(d, logits, lse, k, next_idx, next_bitmap, stream=s)
    else:
        spc_topk_select_prev(d, logits, lse, k, next_idx, next_bitmap, idx, k, src, stream=s)
    selected = torch.cuda.Event()
    selected.record(stream)
    fetch_stream.wait_event(selected)
    if src is None:
        spc_host_gather(d, host_kv, n_cap, next_idx, k, next_staging, stream=fetch_stream.cuda_stream)
    else:
        spc_host_gather_prev(d, host_kv, n_cap, next_idx, k, next_staging, src, staging, k,
                             stream=fetch_stream.cuda_stream)
    fetched = torch.cuda.Event()
    fetched.record(fetch_stream)
    return fetched
