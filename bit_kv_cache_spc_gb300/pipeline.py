"""The decode step of every layer (SpeCache page, section 3 "Decoding",
Algorithm 3, applied layer after layer) in the schedule that measured fastest
on one GB300.

Per layer l, on a high-priority main stream, the merged attention of layer l
over C' U C_kappa carries the Pre-fetch of layer (l - lag)'s new selection on
its own copy pipeline (spc_merged_attn_fetch[_prev]); the layer's ArgTopK runs
on a low-priority side stream once the attention is done, in the SMs that the
attentions leave idle.  Layer l's attention waits only for layer (l - lag)'s
top-k, and every layer's rows are staged before that layer's attention of the
next step (the last lag layers' rows ride on the next step's first
attentions).

With the staged rows kept (keep=True, the pages' eviction rule: the used
16-bit rows outside the new top-k are evicted, the others stay), the
selections and staging buffers alternate between two copies by step parity:
the step of parity P reads copy P and writes the next selection and its rows
into copy 1 - P, and a pre-fetch copies the rows its layer's previous
selection already staged from device memory (spc_topk_select_prev reports
where each row sat) instead of reading them from the host.

Every call is an entry point of the library; this module only orders them on
two streams with events (and resets the previous-slot arrays at the
pre-decoding step), so a step can be captured into a CUDA graph (one graph
per parity when rows are kept).  The per-layer sequential form of
Algorithms 1-3 is in steps.py.
"""
from __future__ import annotations

import torch

from . import (spc_decode_attn2, spc_host_gather, spc_merged_attn, spc_merged_attn_fetch,
               spc_merged_attn_fetch_prev, spc_topk_select, spc_topk_select_prev)


class DecodePipeline:
    """The decode step of L layers of one shape d with k fetched rows each.

    Per layer l (lists of L tensors, all on the device but host):
      records[l], resid[l]: the layer's low-bit cache and bf16 residual window;
      host[l]: the layer's pinned, mapped 16-bit cache [B][Hkv][n_cap][2][D];
      q[l]: bf16 [B][2][Hq][D] (the real token, then the speculative token);
      o[l], lse[l], logits[l]: the merged attention's outputs (logits: the
        speculative row, [B][Hkv][G][q_groups_cap * 32] fp32).
    ws, ws_bytes: one attention workspace (spc_attn_workspace_bytes(d, k)),
    zero-filled once.  The selections, the staging buffers and, with kept
    rows, the previous-slot arrays are allocated here unless given (idx,
    bitmap, staging: two copies each with keep, a list per copy; src: per
    layer).  1 <= lag <= L - 1: at lag = L a layer's attention would carry
    the fetch of its own staging, which it reads; lag = 1 makes each
    attention wait for the top-k just before it.
    """

    def __init__(self, d, k, records, resid, host, n_cap, q, o, lse, logits, ws, ws_bytes, lag=2, keep=True,
                 main=None, side=None, idx=None, bitmap=None, staging=None, src=None):
        L = len(records)
        if L < 2 or not 1 <= lag <= L - 1:
            raise ValueError(f"the schedule needs at least 2 layers and 1 <= lag <= L - 1 (L = {L}, lag = {lag})")
        self.d, self.k, self.L, self.n_cap = d, k, L, n_cap
        self.records, self.resid, self.host, self.q = records, resid, host, q
        self.o, self.lse, self.logits, self.ws, self.ws_bytes = o, lse, logits, ws, ws_bytes
        self.lag = lag
        self.keep = keep
        dev = records[0].device
        B, Hkv = d.B, d.Hkv
        copies = 2 if keep else 1
        if idx is None:
            idx = [[torch.full((B, Hkv, k), -1, dtype=torch.int32, device=dev) for _ in range(L)]
                   for _ in range(copies)]
        if bitmap is None:
            bitmap = [[torch.zeros((B, Hkv, d.q_groups_cap), dtype=torch.int32, device=dev) for _ in range(L)]
                      for _ in range(copies)]
        if staging is None:
            staging = [[torch.zeros((B, Hkv, k, 2, d.D), dtype=torch.int16, device=dev) for _ in range(L)]
                       for _ in range(copies)]
        if keep and src is None:
            src = [torch.full((B, Hkv, k), -1, dtype=torch.int32, device=dev) for _ in range(L)]
        self.idx, self.bitmap, self.staging, self.src = idx, bitmap, staging, src
        self.main = torch.cuda.Stream(priority=-1) if main is None else main
        self.side = torch.cuda.Stream(priority=0) if side is None else side
        self.attended = [torch.cuda.Event() for _ in range(L)]
        self.selected = [torch.cuda.Event() for _ in range(L)]
        self.parity = 0  # the copy the next step() or StepGraphs.replay() reads

    def predecode(self, stream=None):
        """Algorithm 2 for every layer, on `stream` (default: main): the
        low-bit attention of the queries (the caller passes the pre-decoding
        queries in q), the first selection and its gather, into copy 0; the
        next step reads copy 0."""
        s = self.main if stream is None else stream
        s.wait_stream(torch.cuda.current_stream())  # the caches written on the caller's stream
        d, k = self.d, self.k
        self.parity = 0
        for l in range(self.L):
            if self.keep:
                with torch.cuda.stream(s):
                    self.src[l].fill_(-1)  # the first pre-fetches find no staged rows
            spc_decode_attn2(d, self.records[l], self.resid[l], self.q[l], self.o[l], self.lse[l], self.logits[l],
                             self.ws, self.ws_bytes, stream=s)
            spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[0][l], self.bitmap[0][l], stream=s)
            spc_host_gather(d, self.host[l], self.n_cap, self.idx[0][l], k, self.staging[0][l], stream=s)

    def enqueue(self, parity=0, fetch=True, topk=True, on_attention=None, on_topk=None):
        """One decode step on the two streams (capturable into a CUDA graph).
        parity: the copy this step reads (kept rows; 0 otherwise), the steps
        alternating 0, 1, 0, ...  fetch=False leaves the pre-fetch out (the
        staging already filled); topk=False leaves the selection out.
        on_attention(l, when, stream) / on_topk(l, when, stream), when 0 or 1,
        run just before / after layer l's attention or top-k is enqueued."""
        d, k, L, lag = self.d, self.k, self.L, self.lag
        main, side = self.main, self.side
        P = parity if self.keep else 0
        for l in range(L):
            j = (l - lag) % L
            idx, bitmap, staging = self.idx[P][l], self.bitmap[P][l], self.staging[P][l]
            if not self.keep:
                f_idx, f_out, f_prev = self.idx[0][j], self.staging[0][j], None
            elif l >= lag:  # layer j's selection of this step, written to the other copy
                f_idx, f_out, f_prev = self.idx[1 - P][j], self.staging[1 - P][j], self.staging[P][j]
            else:  # layer j's selection of the previous step
                f_idx, f_out, f_prev = self.idx[P][j], self.staging[P][j], self.staging[1 - P][j]
            if topk and l >= lag:  # layers L-lag .. L-1 were selected by the previous step, which has completed
                main.wait_event(self.selected[j])
            if on_attention:
                on_attention(l, 0, main)
            if fetch and self.keep:
                spc_merged_attn_fetch_prev(d, self.records[l], self.resid[l], self.q[l], idx, bitmap, staging, k,
                                           self.o[l], self.lse[l], self.logits[l], self.ws, self.host[j],
                                           self.n_cap, f_idx, k, f_out, self.src[j], f_prev, k,
                                           ws_bytes=self.ws_bytes, stream=main)
            elif fetch:
                spc_merged_attn_fetch(d, self.records[l], self.resid[l], self.q[l], idx, bitmap, staging, k,
                                      self.o[l], self.lse[l], self.logits[l], self.ws, self.host[j], self.n_cap,
                                      f_idx, k, f_out, ws_bytes=self.ws_bytes, stream=main)
            else:
                spc_merged_attn(d, self.records[l], self.resid[l], self.q[l], idx, bitmap, staging, k, self.o[l],
                                self.lse[l], self.logits[l], self.ws, self.ws_bytes, stream=main)
            if on_attention:
                on_attention(l, 1, main)
            if not topk:
                continue
            self.attended[l].record(main)
            side.wait_event(self.attended[l])
            if on_topk:
                on_topk(l, 0, side)
            if self.keep:
                spc_topk_select_prev(d, self.logits[l], self.lse[l], k, self.idx[1 - P][l], self.bitmap[1 - P][l],
                                     idx, k, self.src[l], stream=side)
            else:
                spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[0][l], self.bitmap[0][l], stream=side)
            if on_topk:
                on_topk(l, 1, side)
            self.selected[l].record(side)
        if topk:
            for l in range(L):  # join the side stream before the step ends
                main.wait_event(self.selected[l])

    def step(self, **hooks):
        """Enqueue the next decode step (the current parity) and advance the
        parity; returns at once (the work runs on the two streams)."""
        self.main.wait_stream(torch.cuda.current_stream())
        self.enqueue(parity=self.parity, **hooks)
        torch.cuda.current_stream().wait_stream(self.main)
        self.parity ^= 1 if self.keep else 0

    def capture(self, **hooks):
        """The decode step captured as CUDA graphs, one per parity (one with
        the staged rows not kept); StepGraphs.replay() runs the next one."""
        self.main.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        graphs = []
        for P in ((0, 1) if self.keep else (0,)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.main):
                g.capture_begin(capture_error_mode="relaxed")
                self.enqueue(parity=P, **hooks)
                g.capture_end()
            graphs.append(g)
        torch.cuda.synchronize()
        return StepGraphs(self, graphs)

    def selection(self, parity):
        """The selections (idx, bitmap per layer) that the step of `parity`
        reads: the ones the step before it wrote."""
        P = parity if self.keep else 0
        return self.idx[P], self.bitmap[P]

    def kept_fraction(self):
        """Of the rows the last step's pre-fetches staged, the fraction copied
        from the previous staging instead of read from the host (None without
        kept rows)."""
        if not self.keep:
            return None
        torch.cuda.current_stream().wait_stream(self.main)
        n = sum(int((s >= 0).sum().item()) for s in self.src)
        return n / float(sum(s.numel() for s in self.src))


class StepGraphs:
    """A pipeline's step graphs by parity.  replay() runs the graph of the
    pipeline's current parity on its main stream and advances the parity, so
    that graphs and step() calls can be mixed."""

    def __init__(self, pipe, graphs):
        self.pipe, self.graphs = pipe, graphs

    def replay(self):
        pipe = self.pipe
        pipe.main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(pipe.main):
            self.graphs[pipe.parity if pipe.keep else 0].replay()
        torch.cuda.current_stream().wait_stream(pipe.main)
        pipe.parity ^= 1 if pipe.keep else 0
