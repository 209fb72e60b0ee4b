#!/usr/bin/env python
"""Benchmark of the SpeCache decode hot path on GB300.

Workload: one decode step of LLaMA-3-8B's attention over all 32 layers
(batch 8, 32 query / 8 KV heads, head dim 128, 32K context, 1-bit cache,
top-1% = 328 fetched rows per KV head).  Per layer: the merged two-query
attention over C' U C_kappa, which in the same launch pre-fetches the bf16
rows that layer l-2's top-k selected from pinned host memory, and the
speculative top-k, which runs on a low-priority second stream beside the next
layer's attention.  A step is captured once as a CUDA graph and replayed.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(workload="llama3-8b decode step, 32 layers x attention, B=8, Hq=32, Hkv=8, D=128, "
                         "N=32768, 1-bit, residual 128, top-1% (k=328)",
                B=8, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328, layers=32)
METRIC = "decode attn steps/s and HBM GB/s (% of peak) at 32K ctx, 1-bit, top-1%"  # value: steps/s; GB/s: roofline
# DRAM bytes (read + write) of one merged-attention call of this workload (attn_kernel + combine_kernel, the
# carried pre-fetch included, as the default placement runs it), from an ncu capture of the attention sources
# whose digest is recorded beside it; reported as null when the sources compiled now differ from those, or for
# another placement's call.
ATTN_TRAFFIC = {"bytes_per_call": 178306816, "sources_sha256": "84d63584d9f24b86"}
ATTN_SOURCES = ("attention.cuh", "attn_b1g32.cu", "attention.cu", "common.cuh", "select.cuh")


def attention_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for name in ATTN_SOURCES:
        with open(os.path.join(ROOT, "bit_kv_cache_spc_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def attention_traffic():
    """The captured DRAM traffic of one attention call, if it was taken on the sources built now."""
    if ATTN_TRAFFIC["sources_sha256"] is not None and ATTN_TRAFFIC["sources_sha256"] == attention_sources_sha256():
        return ATTN_TRAFFIC["bytes_per_call"]
    return None


def synth_queries(seed, layer, W):
    import synth
    return synth.queries(seed, layer, W["B"], W["Hq"])


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["spc", "reference"], default="spc")
    p.add_argument("--layers", type=int, default=WORKLOAD["layers"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-pairs", type=int, default=0,
                   help="(b, kv-head) pairs in the oracle sample (0: as many as host cores, at least 16)")
    p.add_argument("--no-configs", dest="configs", action="store_false",
                   help="skip the per-configuration points (configurations 1-3 and the 48 of configuration 5)")
    p.add_argument("--oracle-1core", action="store_true",
                   help="(internal) time the oracle on the two small configurations, one thread, and exit")
    p.add_argument("--prefetch", choices=["side", "fused", "step", "overlap"], default="overlap",
                   help="pre-fetch as a small side-stream kernel, or carried by the next layer's attention "
                        "(then top-k as its own launch), or 'step': one spc_decode_step launch per layer "
                        "(attention + carried pre-fetch + fused top-k)")
    p.add_argument("--gather-ctas", type=int, default=32, help="grid of the side-stream pre-fetch kernel")
    p.add_argument("--refetch-all", action="store_true",
                   help="overlap placement: fetch every selected row from the host each step, instead of keeping "
                        "the rows that the layer's previous selection already staged")
    p.add_argument("--prefetch-lag", type=int, default=2,
                   help="overlap placement: layer l's attention carries the pre-fetch of layer l-LAG's selection")
    p.add_argument("--profile-call", choices=["attn2", "merged", "merged_fetch", "topk", "gather"], default=None,
                   help="(profiling) one decode layer of the workload: run its calls once, then this call "
                        "--profile-reps times, and exit; a profiler captures the call's kernels")
    p.add_argument("--profile-reps", type=int, default=4)
    args = p.parse_args()
    if args.layers < 2 and args.prefetch != "side" and args.impl == "spc" and args.profile_call is None:
        # a carried pre-fetch rides on another layer's attention: with one layer it would write the
        # staging rows that the same attention reads
        p.error("--prefetch fused|step|overlap needs at least 2 layers (--prefetch side runs one)")
    return args


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region
    (every 25 ms, so that a timed region of a few tens of milliseconds still
    holds samples)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        self.started = False
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        # the sampler's first line comes before the timed region and is dropped: every kept sample is
        # taken while the timed work runs
        import select
        ready, _, _ = select.select([self.proc.stdout], [], [], 5.0)
        if ready:
            self.started = bool(self.proc.stdout.readline())
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        return False

    def summary(self):
        if not getattr(self, "rows", None):
            why = "nvidia-smi unavailable" if self.proc is None or not self.started else \
                "no nvidia-smi sample during the timed region"
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [why], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def record_external(ev, stream):
    """Record a timing event so that it survives CUDA graph capture."""
    ev.record(stream)


def make_timing_event(torch):
    try:
        return torch.cuda.Event(enable_timing=True, external=True), record_external
    except TypeError:
        pass
    # older torch: record through the CUDA runtime with cudaEventRecordExternal
    lib = None
    with open("/proc/self/maps") as f:
        for line in f:
            if "libcudart.so" in line:
                lib = ctypes.CDLL(line.split()[-1])
                break
    if lib is None:
        lib = ctypes.CDLL("libcudart.so")
    lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
    ev = torch.cuda.Event(enable_timing=True)
    ev.record()  # create the underlying event
    torch.cuda.synchronize()

    def rec(e, stream):
        err = lib.cudaEventRecordWithFlags(ctypes.c_void_p(e.cuda_event), ctypes.c_void_p(stream.cuda_stream), 1)
        if err != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed: {err}")
    return ev, rec


# ------------------------------------------------------------------ the GPU workload

class GraphPair:
    """The graphs of one step for the two buffer parities; each replay runs
    the graph of the owner's current parity and flips it, so that every graph
    pair of the owner stays in step with the buffers."""

    def __init__(self, owner, graphs):
        self.owner, self.graphs = owner, graphs

    def replay(self):
        self.graphs[self.owner.parity].replay()
        self.owner.parity ^= 1


class DecodeStep:
    def __init__(self, W, layers, seed=0, mode="fused", gather_ctas=32, lag=2, keep_staged=True):
        import torch

        import bit_kv_cache_spc_gb300 as spc
        import synth
        import synth.gpu
        self.torch, self.spc = torch, spc
        B, Hq, Hkv, N, R, bits, k = (W[x] for x in ("B", "Hq", "Hkv", "N", "R", "bits", "k"))
        self.W, self.L, self.k = W, layers, k
        self.G = Hq // Hkv
        self.d = spc.Dims(B, Hq, Hkv, N, R, bits, scale=float(np.float32(1.0 / math.sqrt(128))))
        d = self.d
        dev = torch.device("cuda")
        self.nq = spc.spc_num_quantized(d)
        self.Lcap = d.q_groups_cap * 32
        self.records = [torch.empty(spc.spc_records_bytes(d), dtype=torch.uint8, device=dev) for _ in range(layers)]
        self.resid = [torch.empty(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device=dev) for _ in range(layers)]
        self.host = [torch.empty((B, Hkv, N, 2, 128), dtype=torch.int16, pin_memory=True) for _ in range(layers)]
        Kt = torch.empty((B, Hkv, N, 128), dtype=torch.int16, device=dev)
        Vt = torch.empty_like(Kt)
        for l in range(layers):
            synth.gpu.kv_layer_into(seed, l, Kt, Vt)
            spc.spc_quantize_kv(d, Kt, Vt, self.records[l], self.resid[l])
            self.host[l].copy_(torch.stack([Kt, Vt], dim=3), non_blocking=False)
        del Kt, Vt
        qn = np.stack([synth.queries(seed, l, B, Hq) for l in range(layers)])
        self.q_host = torch.from_numpy(qn.view(np.int16).copy()).pin_memory()
        self.q = self.q_host.to(dev)
        self.o = torch.zeros((layers, B, 2, Hq, 128), dtype=torch.int16, device=dev)
        self.o_host = torch.empty_like(self.o, device="cpu").pin_memory()
        self.lse = torch.zeros((layers, B, 2, Hq), dtype=torch.float32, device=dev)
        self.logits = torch.zeros((layers, B, Hkv, self.G, self.Lcap), dtype=torch.float32, device=dev)
        self.idx = torch.zeros((layers, B, Hkv, k), dtype=torch.int32, device=dev)
        self.bitmap = torch.zeros((layers, B, Hkv, d.q_groups_cap), dtype=torch.int32, device=dev)
        self.staging = torch.zeros((layers, B, Hkv, k, 2, 128), dtype=torch.int16, device=dev)
        # Overlap placement: the rows still staged from a layer's previous selection are kept.  Selections
        # and staging alternate between two buffers by step parity (the previous ones are read while the
        # next are written); src[l] says where each newly selected row of layer l sat in its previous
        # selection (-1: read it from the host).
        self.keep = keep_staged and mode in ("overlap", "step")
        self.parity = 0
        if self.keep:
            self.idx_b = [self.idx, torch.full_like(self.idx, -1)]
            self.bitmap_b = [self.bitmap, torch.zeros_like(self.bitmap)]
            self.staging_b = [self.staging, torch.zeros_like(self.staging)]
            self.src = torch.full((layers, B, Hkv, k), -1, dtype=torch.int32, device=dev)
        self.ws_bytes = spc.spc_attn_workspace_bytes(d, k)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)  # zero-filled once
        self.ws_step_bytes = spc.spc_step_workspace_bytes(d, k)
        # the fused step keeps the speculative logits on chip (TMEM) when the shape allows it
        self.step_onchip = spc.spc_decode_step_on_chip(d, k, k, k) == 1
        self.ws_step = torch.zeros(self.ws_step_bytes, dtype=torch.uint8, device=dev)  # zero-filled once
        self.main = torch.cuda.Stream(priority=-1 if mode == "overlap" else 0)
        self.side = torch.cuda.Stream(priority=-1)
        self.side_lo = torch.cuda.Stream(priority=0)
        self.attended = [torch.cuda.Event() for _ in range(layers)]
        self.selected = [torch.cuda.Event() for _ in range(layers)]
        self.gathered = [torch.cuda.Event() for _ in range(layers)]
        self.mode = mode
        self.gather_ctas = gather_ctas
        self.lag = max(1, min(lag, layers - 1))
        self.pipe = None
        if mode == "overlap":
            from bit_kv_cache_spc_gb300.pipeline import DecodePipeline
            self.pipe = DecodePipeline(d, k, self.records, self.resid, self.host, N, self.q, self.o, self.lse,
                                       self.logits, self.ws, self.ws_bytes, lag=self.lag, keep=self.keep,
                                       main=self.main, side=self.side_lo,
                                       idx=self.idx_b if self.keep else [self.idx],
                                       bitmap=self.bitmap_b if self.keep else [self.bitmap],
                                       staging=self.staging_b if self.keep else [self.staging],
                                       src=self.src if self.keep else None)
        self.t0, self.rec = make_timing_event(torch)
        self.attn_ev = [(make_timing_event(torch)[0], make_timing_event(torch)[0]) for _ in range(layers)]
        self.topk_ev = [(make_timing_event(torch)[0], make_timing_event(torch)[0]) for _ in range(layers)]
        # pre-decoding step: plain low-bit attention, first top-k and prefetch
        with torch.cuda.stream(self.main):
            for l in range(layers):
                spc.spc_decode_attn2(d, self.records[l], self.resid[l], self.q[l], self.o[l], self.lse[l],
                                     self.logits[l], self.ws, self.ws_bytes, stream=self.main)
                spc.spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[l], self.bitmap[l],
                                    stream=self.main)
                spc.spc_host_gather(d, self.host[l], N, self.idx[l], k, self.staging[l], stream=self.main)
        torch.cuda.synchronize()
        # attention, top-k, and the gather (its own launch, or riding on the next attention)
        attn_f = spc.spc_attn_kernel_count(d, k, k)  # the attention call's kernels, carrying a pre-fetch
        attn = spc.spc_attn_kernel_count(d, k, 0)
        step = spc.spc_decode_step_kernel_count(d, k, k, k)
        self.launches_per_step = layers * {"side": attn + 2, "fused": attn_f + 1, "step": step,
                                           "overlap": attn_f + 1}[mode]
        self.graph = None

    def enqueue(self, timed=False, parity=0):
        self.capture_parity = parity
        if self.mode == "fused":
            return self.enqueue_fused(timed)
        if self.mode == "step":
            return self.enqueue_step(timed, parity=self.capture_parity)
        if self.mode == "overlap":
            return self.enqueue_overlap(timed, parity=self.capture_parity)
        return self.enqueue_side(timed)

    def enqueue_overlap(self, timed=False, fetch=True, topk=True, parity=0):
        """One decode step of the library's two-stream schedule
        (bit_kv_cache_spc_gb300.pipeline.DecodePipeline): layer l's merged
        attention on the high-priority main stream carries the pre-fetch of
        layer (l - lag)'s selection, and each top-k runs on a low-priority
        stream after its layer's attention; with the staged rows kept, the
        step of this parity reads buffer `parity` and writes the other.
        fetch=False: the same step with the staging buffers already filled and
        no pre-fetch (the overlap test's reference).  topk=False: the merged
        attentions alone, back to back on one stream (their kernel time).
        timed: events around every attention and top-k."""
        hooks = {}
        if timed:
            hooks = dict(on_attention=lambda l, w, s: self.rec(self.attn_ev[l][w], s),
                         on_topk=lambda l, w, s: self.rec(self.topk_ev[l][w], s))
        self.pipe.enqueue(parity=parity, fetch=fetch, topk=topk, **hooks)

    def enqueue_step(self, timed=False, parity=0):
        """One decode step on one stream, one launch per layer: spc_decode_step
        runs the merged attention over C' U C_kappa, carries the pre-fetch of
        layer l-1's selection and ends with the speculative top-k.  Without
        kept rows the selection replaces idx[l] / bitmap[l] in place; with them
        (self.keep, spc_decode_step_prev) the step of this parity reads buffer
        `parity` and writes the next selection into the other, and a pre-fetch
        copies the rows its layer's previous selection staged from HBM."""
        spc, d, k = self.spc, self.d, self.k
        main, L = self.main, self.L
        P = parity
        for l in range(L):
            j = (l - 1) % L
            if timed:
                self.rec(self.attn_ev[l][0], main)
            logits = None if self.step_onchip else self.logits[l]
            if self.keep:
                if l >= 1:  # layer j's selection of this step, written to the other parity
                    f_idx, f_out, f_prev = self.idx_b[1 - P][j], self.staging_b[1 - P][j], self.staging_b[P][j]
                else:  # layer L-1's selection of the previous step
                    f_idx, f_out, f_prev = self.idx_b[P][j], self.staging_b[P][j], self.staging_b[1 - P][j]
                spc.spc_decode_step_prev(d, self.records[l], self.resid[l], self.q[l], self.idx_b[P][l],
                                         self.bitmap_b[P][l], self.staging_b[P][l], k, self.o[l], self.lse[l], logits,
                                         k, self.idx_b[1 - P][l], self.bitmap_b[1 - P][l], self.src[l], self.ws_step,
                                         self.ws_step_bytes, fetch_host_kv=self.host[j], fetch_n_cap=self.W["N"],
                                         fetch_idx=f_idx, fetch_k=k, fetch_staging=f_out, fetch_src=self.src[j],
                                         fetch_prev_staging=f_prev, fetch_prev_k=k, stream=main)
            else:
                spc.spc_decode_step(d, self.records[l], self.resid[l], self.q[l], self.idx[l], self.bitmap[l],
                                    self.staging[l], k, self.o[l], self.lse[l], logits, k, self.idx[l],
                                    self.bitmap[l], self.ws_step, self.ws_step_bytes, fetch_host_kv=self.host[j],
                                    fetch_n_cap=self.W["N"], fetch_idx=self.idx[j], fetch_k=k,
                                    fetch_staging=self.staging[j], stream=main)
            if timed:
                self.rec(self.attn_ev[l][1], main)
                self.rec(self.topk_ev[l][0], main)
                self.rec(self.topk_ev[l][1], main)

    def enqueue_side(self, timed=False):
        """One decode step.  Layer l: the merged attention over C' U C_kappa and
        the speculative top-k on the main stream; the pre-fetch of layer l's new
        selection on a high-priority side stream with a small persistent grid,
        so that it shares the SMs with layer l+1's attention while the host link
        works.  The next step's attention of layer l waits for that pre-fetch."""
        spc, d, k = self.spc, self.d, self.k
        main, side, L = self.main, self.side, self.L
        for l in range(L):
            main.wait_event(self.gathered[l])
            if timed:
                self.rec(self.attn_ev[l][0], main)
            spc.spc_merged_attn(d, self.records[l], self.resid[l], self.q[l], self.idx[l], self.bitmap[l],
                                self.staging[l], k, self.o[l], self.lse[l], self.logits[l], self.ws, self.ws_bytes,
                                stream=main)
            if timed:
                self.rec(self.attn_ev[l][1], main)
                self.rec(self.topk_ev[l][0], main)
            spc.spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[l], self.bitmap[l], stream=main)
            if timed:
                self.rec(self.topk_ev[l][1], main)
            self.selected[l].record(main)
            side.wait_event(self.selected[l])
            spc.spc_host_gather(d, self.host[l], self.W["N"], self.idx[l], k, self.staging[l],
                                max_ctas=self.gather_ctas, stream=side)
            self.gathered[l].record(side)
        for l in range(L):  # join the side stream before the step ends
            main.wait_event(self.gathered[l])

    def enqueue_fused(self, timed=False):
        """One decode step on one stream.  Layer l: the merged attention over
        C' U C_kappa, carrying the pre-fetch of layer l-1's new selection (layer
        L-1's for l = 0, from the previous step), then the speculative top-k.
        The rows fetched during layer l's attention are read by layer l-1's
        attention of the next step, so the host link works behind the SMs."""
        spc, d, k = self.spc, self.d, self.k
        main, L = self.main, self.L
        for l in range(L):
            j = (l - 1) % L  # the layer whose selection is pre-fetched now
            if timed:
                self.rec(self.attn_ev[l][0], main)
            spc.spc_merged_attn_fetch(d, self.records[l], self.resid[l], self.q[l], self.idx[l], self.bitmap[l],
                                      self.staging[l], k, self.o[l], self.lse[l], self.logits[l], self.ws,
                                      self.host[j], self.W["N"], self.idx[j], k, self.staging[j],
                                      ws_bytes=self.ws_bytes, stream=main)
            if timed:
                self.rec(self.attn_ev[l][1], main)
                self.rec(self.topk_ev[l][0], main)
            spc.spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[l], self.bitmap[l], stream=main)
            if timed:
                self.rec(self.topk_ev[l][1], main)

    def enqueue_serial(self):
        """The non-speculative decode step that SpeCache's speculation replaces
        (the exact token's own attention decides the rows to fetch): per layer,
        the low-bit attention of the real token (both query rows equal), its
        ArgTopK, the gather of those rows on the critical path, then the merged
        attention with them."""
        spc, d, k = self.spc, self.d, self.k
        main, L = self.main, self.L
        for l in range(L):
            spc.spc_decode_attn2(d, self.records[l], self.resid[l], self.q_serial[l], self.o[l], self.lse[l],
                                 self.logits[l], self.ws, self.ws_bytes, stream=main)
            spc.spc_topk_select(d, self.logits[l], self.lse[l], k, self.idx[l], self.bitmap[l], stream=main)
            spc.spc_host_gather(d, self.host[l], self.W["N"], self.idx[l], k, self.staging[l], stream=main)
            spc.spc_merged_attn(d, self.records[l], self.resid[l], self.q_serial[l], self.idx[l], self.bitmap[l],
                                self.staging[l], k, self.o[l], self.lse[l], self.logits[l], self.ws, self.ws_bytes,
                                stream=main)

    def time_serial(self, steps, warmup):
        """Steps/s of the non-speculative step, captured as its own graph."""
        torch = self.torch
        self.q_serial = self.q[:, :, :1].expand(-1, -1, 2, -1, -1).contiguous()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.main):
            g.capture_begin(capture_error_mode="relaxed")
            self.enqueue_serial()
            g.capture_end()
        with torch.cuda.stream(self.main):
            for _ in range(max(3, warmup)):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.main)
        with torch.cuda.stream(self.main):
            for _ in range(steps):
                g.replay()
        e1.record(self.main)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        del g
        return {"value": 1000.0 / ms, "unit": "steps/s", "ms_per_step": ms,
                "what": "per layer: low-bit attention of the real token, its top-k, the gather on the critical path, "
                        "merged attention (no speculative token, no overlap)"}

    def capture(self):
        """Two graphs of the same step: the one that is timed has nothing
        between the kernels (so each launch may overlap its predecessor's
        tail), the other records events around every attention and top-k for
        the per-layer breakdown."""
        torch = self.torch
        self.main.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        self.graph = self.capture_step(lambda P: self.enqueue(timed=False, parity=P))
        self.graph_timed = self.capture_step(lambda P: self.enqueue(timed=True, parity=P))

    def capture_step(self, enqueue):
        """The step's graph; with the staged rows kept, one graph per step
        parity, replayed in turn (GraphPair)."""
        if not self.keep:
            return self.capture_graph(lambda: enqueue(0))
        return GraphPair(self, [self.capture_graph(lambda: enqueue(0)), self.capture_graph(lambda: enqueue(1))])

    def capture_graph(self, enqueue):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.main):
            g.capture_begin(capture_error_mode="relaxed")
            enqueue()
            g.capture_end()
        torch.cuda.synchronize()
        return g

    def time_graph(self, g, reps, warmup=3):
        """ms per replay of graph g: `reps` replays back to back between two
        events on the main stream, after `warmup` replays."""
        torch = self.torch
        with torch.cuda.stream(self.main):
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.main)
        with torch.cuda.stream(self.main):
            for _ in range(reps):
                g.replay()
        e1.record(self.main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def replay(self):
        with self.torch.cuda.stream(self.main):
            self.graph.replay()

    def replay_timed(self):
        with self.torch.cuda.stream(self.main):
            self.graph_timed.replay()

    def kept_fraction(self):
        """Of the rows the last step's pre-fetches staged, the fraction copied
        from the previous staging instead of read from the host (None when
        every row is read from the host)."""
        if not self.keep:
            return None
        self.torch.cuda.synchronize()
        return float((self.src >= 0).sum().item()) / float(self.src.numel())

    def attn_ms(self):
        return [s.elapsed_time(e) for (s, e) in self.attn_ev]

    def topk_ms(self):
        return [s.elapsed_time(e) for (s, e) in self.topk_ev]


def host_link_probe(step, reps=20):
    """The pre-fetch alone against the host link: one layer's gather of the
    selected 16-bit rows (zero-copy loads from pinned host memory) timed in
    isolation, next to a contiguous pinned host-to-device copy of 1 GiB (the
    copy engines' rate) and the same kernel reading contiguous rows; the
    faster of the two is the link's measured peak."""
    torch = step.torch
    W, d, k = step.W, step.d, step.k
    s = step.main
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for _ in range(3):
            step.spc.spc_host_gather(d, step.host[0], W["N"], step.idx[0], k, step.staging[0], stream=s)
        e0.record(s)
        for _ in range(reps):
            step.spc.spc_host_gather(d, step.host[0], W["N"], step.idx[0], k, step.staging[0], stream=s)
        e1.record(s)
    torch.cuda.synchronize()
    g_ms = e0.elapsed_time(e1) / reps
    g_bytes = W["B"] * W["Hkv"] * k * 512
    src = step.host[0].view(-1)
    dst = torch.empty(src.numel(), dtype=src.dtype, device="cuda")
    with torch.cuda.stream(s):
        dst.copy_(src, non_blocking=True)
        e0.record(s)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize()
    c_ms = e0.elapsed_time(e1) / 3
    c_gbs = src.numel() * src.element_size() / (c_ms / 1000.0) / 1e9
    del dst
    # zero-copy loads of contiguous rows: the same kernel over the first 8192 rows of every (b, kv-head)
    kc = min(8192, W["N"])
    idx_c = torch.arange(kc, dtype=torch.int32, device="cuda").expand(W["B"], W["Hkv"], kc).contiguous()
    st_c = torch.empty((W["B"], W["Hkv"], kc, 2, 128), dtype=torch.int16, device="cuda")
    with torch.cuda.stream(s):
        step.spc.spc_host_gather(d, step.host[0], W["N"], idx_c, kc, st_c, stream=s)
        e0.record(s)
        for _ in range(3):
            step.spc.spc_host_gather(d, step.host[0], W["N"], idx_c, kc, st_c, stream=s)
        e1.record(s)
    torch.cuda.synchronize()
    z_ms = e0.elapsed_time(e1) / 3
    z_gbs = st_c.numel() * st_c.element_size() / (z_ms / 1000.0) / 1e9
    del st_c, idx_c
    g_gbs = g_bytes / (g_ms / 1000.0) / 1e9
    peak = max(c_gbs, z_gbs)
    return {"kernel": "spc_host_gather, one layer", "bytes_per_launch": g_bytes, "avg_launch_us": g_ms * 1000.0,
            "achieved_gbs": g_gbs, "host_link_peak_gbs": peak,
            "copy_engine_contiguous_gbs": c_gbs, "zero_copy_contiguous_gbs": z_gbs,
            "peak_source": "measured: the faster of a contiguous pinned host-to-device copy of 1 GiB and the "
                           f"same kernel reading {kc} contiguous rows of every (b, kv-head)",
            "frac": g_gbs / peak}


def append_probe(W, reps=20):
    """Decode-time append of one token to one layer of the workload's cache
    (spc_append_kv, host offload included), timed without and with a flush:
    at N = 32768 the window grows; at N = 32799 the new token completes a
    group, which is quantised into a record and dropped from the window."""
    import torch
    import bit_kv_cache_spc_gb300 as spc
    import synth.gpu
    B, Hq, Hkv, R, bits = (W[x] for x in ("B", "Hq", "Hkv", "R", "bits"))
    N1 = W["N"] + 32
    K = torch.empty((B, Hkv, N1, 128), dtype=torch.int16, device="cuda")
    V = torch.empty_like(K)
    synth.gpu.kv_layer_into(0, 0, K, V)
    host = torch.empty((B, Hkv, N1, 2, 128), dtype=torch.int16, pin_memory=True)
    out = {}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for tag, N in (("no_flush", W["N"]), ("flush", W["N"] + 31)):
        d = spc.Dims(B, Hq, Hkv, N, R, bits, q_groups_cap=N1 // 32, resid_cap=R + 32)
        rec = torch.empty(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
        res = torch.empty(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
        kn, vn = K[:, :, N].contiguous(), V[:, :, N].contiguous()
        ts = []
        for i in range(reps + 3):
            spc.spc_quantize_kv(d, K[:, :, :N].contiguous(), V[:, :, :N].contiguous(), rec, res)
            e0.record()
            spc.spc_append_kv(d, kn, vn, rec, res, host, N1)
            e1.record()
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1000.0)
        out[f"{tag}_us"] = statistics.median(ts)
    del K, V, host
    out["note"] = "one layer, B*Hkv rows of 512 B to the window and to pinned host memory; a flush codes one group per (b, kv-head)"
    return out


def prefill_probe(W, layers=4, reps=3):
    """The prefill's per-layer tail (Algorithm 1): spc_quantize_kv of one
    layer's K/V, and Offload(C) of those 16-bit rows to pinned host memory on
    a copy stream; then `layers` layers pipelined (layer l+1's quantisation
    while layer l's rows travel to the host)."""
    import torch
    import bit_kv_cache_spc_gb300 as spc
    import synth.gpu
    from bit_kv_cache_spc_gb300.steps import prefill_layer
    B, Hq, Hkv, N, R, bits = (W[x] for x in ("B", "Hq", "Hkv", "N", "R", "bits"))
    d = spc.Dims(B, Hq, Hkv, N, R, bits)
    K = torch.empty((B, Hkv, N, 128), dtype=torch.int16, device="cuda")
    V = torch.empty_like(K)
    synth.gpu.kv_layer_into(0, 0, K, V)
    rec = torch.empty(spc.spc_records_bytes(d), dtype=torch.uint8, device="cuda")
    res = torch.empty(spc.spc_resid_bytes(d) // 2, dtype=torch.int16, device="cuda")
    host = torch.empty((B, Hkv, N, 2, 128), dtype=torch.int16, pin_memory=True)
    main, copy = torch.cuda.current_stream(), torch.cuda.Stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    q_us, o_us = [], []
    for _ in range(reps + 1):
        ev[0].record(main)
        spc.spc_quantize_kv(d, K, V, rec, res)
        ev[1].record(main)
        ev[2].record(main)
        spc.spc_offload_kv(d, K, V, host, N)
        ev[3].record(main)
        torch.cuda.synchronize()
        q_us.append(ev[0].elapsed_time(ev[1]) * 1000.0)
        o_us.append(ev[2].elapsed_time(ev[3]) * 1000.0)
    qu, ou = statistics.median(q_us[1:]), statistics.median(o_us[1:])
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(main)
    for _ in range(layers):
        prefill_layer(d, K, V, rec, res, host, N, stream=main, copy_stream=copy)
    main.wait_stream(copy)
    t1.record(main)
    torch.cuda.synchronize()
    pipe_us = t0.elapsed_time(t1) * 1000.0 / layers
    host_bytes = K.numel() * 2 * 2
    q_bytes = host_bytes + spc.spc_records_bytes(d)
    del K, V, host
    return {"quantize_us": qu, "quantize_gbs": q_bytes / (qu * 1e-6) / 1e9,
            "offload_us": ou, "offload_gbs": host_bytes / (ou * 1e-6) / 1e9,
            "pipelined_us_per_layer": pipe_us, "layers": layers,
            "note": "one layer of the workload: quantise (HBM) and Offload(C) of 1.07 GB to pinned host memory "
                    "(copy engines, device-to-host); the pipeline overlaps the next layer's quantisation"}


def attention_bytes_per_layer(W, nq):
    """Algorithmic HBM bytes of one merged-attention call (one layer): the
    low-bit copy, the residual and fetched 16-bit rows read, q read and o
    written."""
    beta = 64 if W["bits"] == 1 else 96
    bh = W["B"] * W["Hkv"]
    r = W["N"] - nq
    qo = W["B"] * 2 * W["Hq"] * 128 * 2 * 2  # q read + o written
    return bh * (nq * beta + r * 512 + W["k"] * 512) + qo


# ------------------------------------------------------------------ CPU oracle timing

def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


_KV_CACHE = {}


def kv_pair(seed, layer, B, Hkv, N, b, h):
    """The seeded K, V rows of one (b, kv-head), generated once per process."""
    import synth
    key = (seed, layer, B, Hkv, N, b, h)
    if key not in _KV_CACHE:
        if len(_KV_CACHE) > 64:
            _KV_CACHE.clear()
        _KV_CACHE[key] = synth.kv_slice(seed, layer, B, Hkv, N, 128, b, h)
    return _KV_CACHE[key]


class OracleSample:
    """The oracle's per-layer decode work (merged attention, top-k, gather) on
    `pairs` (b, kv-head) pairs of one layer of the workload.  Inputs, the
    quantisation and the first selection are prepared once; run() times the rest."""

    def __init__(self, W, pairs, seed=0, layer=0, k=None):
        import oracle
        import synth
        self.oracle = oracle
        B, Hq, Hkv, N = W["B"], W["Hq"], W["Hkv"], W["N"]
        G = Hq // Hkv
        sel = [(p // Hkv, p % Hkv) for p in range(min(pairs, B * Hkv))]
        qall = synth.queries(seed, layer, B, Hq)
        Ks, Vs, qs = [], [], []
        for (b, h) in sel:
            kk, vv = kv_pair(seed, layer, B, Hkv, N, b, h)
            Ks.append(kk)
            Vs.append(vv)
            qs.append(qall[b, :, h * G:(h + 1) * G])
        self.P = len(sel)
        self.pairs_per_layer = B * Hkv
        self.K = np.stack(Ks)[:, None]  # the pairs as P sequences with one KV head each
        self.V = np.stack(Vs)[:, None]
        self.q = np.stack(qs)
        self.d = oracle.dims(B=self.P, Hq=G, Hkv=1, N=N, R=W["R"], bits=W["bits"],
                             scale=float(np.float32(1 / math.sqrt(128))), group=W.get("group", 32))
        self.qz = oracle.quantize(self.d, self.K, self.V)
        _, _, S0 = oracle.attention(self.d, self.q, self.qz, self.K, self.V)
        self.k = W["k"] if k is None else k
        self.idx, _ = oracle.topk(self.d, S0, self.k)
        self.host = np.stack([self.K, self.V], axis=3)
        self.layers = W.get("layers", 1)
        self.scale_to_step = (B * Hkv / self.P) * self.layers
        self.threads = min(self.P, host_cores())

    def run(self):
        o = self.oracle
        t = time.perf_counter()
        o.gather(self.d, self.host, self.idx)
        _, _, S1 = o.attention(self.d, self.q, self.qz, self.K, self.V, idx=self.idx)
        o.topk(self.d, S1, self.k)
        return time.perf_counter() - t

    def steps_per_s(self, seconds):
        return 1.0 / (seconds * self.scale_to_step)

    def layer_ms(self, seconds):
        """ms for the whole layer (all B * Hkv pairs) at the sample's rate."""
        return 1000.0 * seconds * self.pairs_per_layer / self.P


# ------------------------------------------------------------------ the other configurations

CONFIGS = {  # shapes of the pages' Mistral-7B / LLaMA-2-7B layers and a one-head layer
    "c1": dict(workload="one layer, B=1, 1 query / 1 KV head, N=1024, 1-bit, residual 32, k=16",
               B=1, Hq=1, Hkv=1, N=1024, R=32, bits=1, ks=[16], pairs=1),
    "c2": dict(workload="Mistral-7B layer, B=1, 32 query / 8 KV heads, N=32768, 1-bit, residual 128, k=328 (1%)",
               B=1, Hq=32, Hkv=8, N=32768, R=128, bits=1, ks=[328], pairs=8),
    "c3": dict(workload="LLaMA-2-7B layer, B=16, 32 query / 32 KV heads (MHA), N=2048, 2-bit, residual 128, k=64",
               B=16, Hq=32, Hkv=32, N=2048, R=128, bits=2, ks=[64], pairs=16),
}


def c5_points():
    """Configuration 5: the LLaMA-3-8B layer shape at B in {1, 4}, N in {4K, 16K,
    64K, 128K}, 1 and 2 bits, k = 0.5%, 1% and 4% of N (k = ceil(p N))."""
    pts = []
    for B in (1, 4):
        for N in (4096, 16384, 65536, 131072):
            for bits in (1, 2):
                ks = [int(math.ceil(round(p * N, 6))) for p in (0.005, 0.01, 0.04)]
                pts.append(dict(workload=f"LLaMA-3-8B layer, B={B}, N={N}, {bits}-bit", B=B, Hq=32, Hkv=8, N=N,
                                R=128, bits=bits, ks=ks, pairs=1))
    return pts


class LayerRig:
    """One layer of a configuration resident on the device (the low-bit cache
    and residual window, the pinned 16-bit host cache, the queries and every
    output buffer), driven through the library's public calls.  Each call is
    timed alone with CUDA events after an L2 flush (a 256 MB write, more than
    the 129 MB L2), with the host queued ahead by a short GPU spin so that no
    launch waits for the host."""

    FLUSH_BYTES = 256 << 20

    def __init__(self, cfg, seed=0, layer=0):
        import torch

        import bit_kv_cache_spc_gb300 as spc
        import synth
        import synth.gpu
        self.torch, self.spc = torch, spc
        B, Hq, Hkv, N, R, bits = (cfg[x] for x in ("B", "Hq", "Hkv", "N", "R", "bits"))
        self.cfg = cfg
        self.kmax = max(cfg["ks"])
        self.G = Hq // Hkv
        self.d = spc.Dims(B, Hq, Hkv, N, R, bits, scale=float(np.float32(1.0 / math.sqrt(128))),
                          group=cfg.get("group", 32))
        d = self.d
        dev = torch.device("cuda")
        self.nq = spc.spc_num_quantized(d)
        self.K = torch.empty((B, Hkv, N, 128), dtype=torch.int16, device=dev)
        self.V = torch.empty_like(self.K)
        synth.gpu.kv_layer_into(seed, layer, self.K, self.V)
        self.records = torch.empty(max(spc.spc_records_bytes(d), 16), dtype=torch.uint8, device=dev)
        self.resid = torch.empty(max(spc.spc_resid_bytes(d) // 2, 8), dtype=torch.int16, device=dev)
        spc.spc_quantize_kv(d, self.K, self.V, self.records, self.resid)
        self.host = torch.empty((B, Hkv, N, 2, 128), dtype=torch.int16, pin_memory=True)
        self.host.copy_(torch.stack([self.K, self.V], dim=3))
        self.q = torch.from_numpy(synth.queries(seed, layer, B, Hq).view(np.int16).copy()).to(dev)
        self.o = torch.zeros((B, 2, Hq, 128), dtype=torch.int16, device=dev)
        self.lse = torch.zeros((B, 2, Hq), dtype=torch.float32, device=dev)
        self.logits = torch.zeros((B, Hkv, self.G, max(d.q_groups_cap * 32, 1)), dtype=torch.float32, device=dev)
        self.idx = torch.zeros((B, Hkv, max(self.kmax, 1)), dtype=torch.int32, device=dev)
        self.bitmap = torch.zeros((B, Hkv, max(d.q_groups_cap, 1)), dtype=torch.int32, device=dev)
        self.staging = torch.zeros((B, Hkv, max(self.kmax, 1), 2, 128), dtype=torch.int16, device=dev)
        self.ws_bytes = spc.spc_attn_workspace_bytes(d, self.kmax)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)  # zero-filled once
        self.ws_step_bytes = spc.spc_step_workspace_bytes(d, self.kmax)
        self.ws_step = torch.zeros(max(self.ws_step_bytes, 16), dtype=torch.uint8, device=dev)  # zero-filled once
        self.flush = torch.empty(self.FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream()
        torch.cuda.synchronize()

    # the calls of one decode step of this layer
    def quantize(self):
        self.spc.spc_quantize_kv(self.d, self.K, self.V, self.records, self.resid, stream=self.stream)

    def attn2(self):
        self.spc.spc_decode_attn2(self.d, self.records, self.resid, self.q, self.o, self.lse, self.logits, self.ws,
                                  self.ws_bytes, stream=self.stream)

    def topk(self, k):
        self.spc.spc_topk_select(self.d, self.logits, self.lse, k, self.idx, self.bitmap, stream=self.stream)

    def gather(self, k):
        self.spc.spc_host_gather(self.d, self.host, self.cfg["N"], self.idx, k, self.staging, stream=self.stream)

    def merged(self, k):
        self.spc.spc_merged_attn(self.d, self.records, self.resid, self.q, self.idx, self.bitmap, self.staging, k,
                                 self.o, self.lse, self.logits, self.ws, self.ws_bytes, stream=self.stream)

    def decode_step(self, k):
        """One decode step of the layer: the merged attention over C' U C_kappa,
        its top-k and the pre-fetch of the new selection (for the next step)."""
        self.merged(k)
        self.topk(k)
        self.gather(k)

    def decode_step_fused(self, k):
        """The same step through spc_decode_step: the merged attention and its
        top-k in one launch where the selection fits the attention's shared
        memory (the logits kept on chip where allowed), else as the library's
        two launches; then the pre-fetch of the new selection."""
        spc, d = self.spc, self.d
        logits = None if spc.spc_decode_step_on_chip(d, k, 0, k) == 1 else self.logits
        spc.spc_decode_step(d, self.records, self.resid, self.q, self.idx, self.bitmap, self.staging, k, self.o,
                            self.lse, logits, k, self.idx, self.bitmap, self.ws_step, self.ws_step_bytes,
                            stream=self.stream)
        self.gather(k)

    def time_us(self, fn, reps=10):
        """Median device time of fn (its kernels back to back), one call per
        L2 flush."""
        torch = self.torch
        s = self.stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        out = []
        with torch.cuda.stream(s):
            for i in range(reps + 2):
                self.flush.fill_(i)
                torch.cuda._sleep(200000)  # the host enqueues fn while the GPU spins
                e0.record(s)
                fn()
                e1.record(s)
                e1.synchronize()
                if i >= 2:
                    out.append(e0.elapsed_time(e1) * 1000.0)
        return statistics.median(out)

    def graph_us(self, fn, reps=10):
        """Median latency of fn captured as one CUDA graph and replayed, one
        replay per L2 flush."""
        torch = self.torch
        s = self.stream
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.capture_begin(capture_error_mode="relaxed")
            fn()
            g.capture_end()
        us = self.time_us(g.replay, reps)
        del g
        return us


def low_bit_bytes_per_token(bits, group=32):
    """Bytes per token and KV head of the low-bit copy: codes plus a bf16
    (min, max) pair per group of keys and of values."""
    return {(1, 32): 64, (2, 32): 96, (1, 64): 48, (2, 64): 80}[(bits, group)]


def attention_bytes(cfg, nq, k):
    """Algorithmic HBM bytes of one merged-attention call: the low-bit copy,
    the residual and fetched 16-bit rows read, q read and o written."""
    beta = low_bit_bytes_per_token(cfg["bits"], cfg.get("group", 32))
    bh = cfg["B"] * cfg["Hkv"]
    r = cfg["N"] - nq
    qo = cfg["B"] * 2 * cfg["Hq"] * 128 * 2 * 2
    return bh * (nq * beta + r * 512 + k * 512) + qo


def measure_config(cfg, peak_gbs, oracle_on=True, reps=10, rig=None):
    """Per-call device times of one configuration (its layer), bytes, HBM and
    host-link fractions, and the oracle's time on a sample of the same layer."""
    rig = LayerRig(cfg) if rig is None else rig
    out = []
    q_us = rig.time_us(rig.quantize, reps=max(3, reps // 3))
    bh = cfg["B"] * cfg["Hkv"]
    q_bytes = bh * cfg["N"] * 512 + bh * rig.nq * low_bit_bytes_per_token(cfg["bits"], cfg.get("group", 32))
    a2_us = rig.time_us(rig.attn2, reps)
    for k in cfg["ks"]:
        rig.attn2()
        rig.topk(k)
        rig.gather(k)
        rig.torch.cuda.synchronize()
        t_us = rig.time_us(lambda: rig.topk(k), reps)
        g_us = rig.time_us(lambda: rig.gather(k), reps)
        m_us = rig.time_us(lambda: rig.merged(k), reps)
        step_us = rig.graph_us(lambda: rig.decode_step(k), reps)
        fused_us = rig.graph_us(lambda: rig.decode_step_fused(k), reps)
        mb = attention_bytes(cfg, rig.nq, k)
        a2b = attention_bytes(cfg, rig.nq, 0)
        gb = bh * k * 512
        pt = {"B": cfg["B"], "N": cfg["N"], "bits": cfg["bits"], "group": cfg.get("group", 32), "k": k,
              "low_bit_bytes_per_token": low_bit_bytes_per_token(cfg["bits"], cfg.get("group", 32)),
              "decode_step_graph_us": step_us, "decode_step_fused_graph_us": fused_us,
              "decode_step_fused_launches": rig.spc.spc_decode_step_kernel_count(rig.d, k, 0, k),
              "merged_us": m_us, "attn2_us": a2_us, "topk_us": t_us,
              "gather_us": g_us, "quantize_us": q_us,
              "merged_bytes": mb, "merged_hbm_frac": mb / (m_us * 1e-6) / 1e9 / peak_gbs,
              "attn2_hbm_frac": a2b / (a2_us * 1e-6) / 1e9 / peak_gbs,
              "quantize_hbm_frac": q_bytes / (q_us * 1e-6) / 1e9 / peak_gbs,
              "gather_bytes": gb, "gather_gbs": gb / (g_us * 1e-6) / 1e9}
        if oracle_on:
            ref = OracleSample(dict(cfg, k=k, layers=1), cfg["pairs"], k=k)
            secs = [ref.run() for _ in range(2 if cfg["N"] >= 65536 else 3)]
            dt = statistics.median(secs)
            pt["oracle_ms_per_layer"] = ref.layer_ms(dt)
            pt["oracle_sample"] = (f"merged attention + top-k + gather of {ref.P} of {ref.pairs_per_layer} "
                                   f"(b, kv-head) pairs, {ref.threads} threads, scaled to the layer")
        out.append(pt)
    return out


def measure_configs(peak_gbs, oracle_on=True, log=None):
    """Configurations 1-3 and the 48 points of configuration 5, one line each."""
    import torch
    res = {}
    for name, cfg in CONFIGS.items():
        try:
            res[name] = dict(workload=cfg["workload"], points=measure_config(cfg, peak_gbs, oracle_on))
        except Exception as e:  # a failed configuration is reported, not fatal to the bench
            res[name] = {"workload": cfg["workload"], "error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    pts = []
    for cfg in c5_points():
        try:
            pts += measure_config(cfg, peak_gbs, oracle_on)
        except Exception as e:
            pts.append({"B": cfg["B"], "N": cfg["N"], "bits": cfg["bits"], "error": f"{type(e).__name__}: {e}"})
        torch.cuda.empty_cache()
    for bits in (1, 2):  # group size 64 (the appendix's LongBench runs) on one LLaMA-3-8B decode layer
        cfg = dict(workload=f"LLaMA-3-8B decode layer at g = 64, B=8, 32/8 heads, N=32768, {bits}-bit, k=328",
                   B=8, Hq=32, Hkv=8, N=32768, R=128, bits=bits, ks=[328], pairs=16, group=64)
        name = f"g64_{bits}bit"
        try:
            res[name] = dict(workload=cfg["workload"], points=measure_config(cfg, peak_gbs, oracle_on))
        except Exception as e:
            res[name] = {"workload": cfg["workload"], "error": f"{type(e).__name__}: {e}"}
        torch.cuda.empty_cache()
    res["c5"] = dict(workload="LLaMA-3-8B layer (32 query / 8 KV heads), B in {1, 4}, N in {4096, 16384, 65536, "
                              "131072}, 1 and 2 bits, k = 0.5 / 1 / 4 % of N", points=pts)
    return res


# ------------------------------------------------------------------ ranks

SMALL_CONFIGS = {  # the oracle's single-core timing (one layer each)
    "c1": dict(B=1, Hq=1, Hkv=1, N=1024, R=32, bits=1, k=16, layers=1),
    "c2": dict(B=1, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328, layers=1),
}


def oracle_single_core():
    """The oracle's decode work (merged attention, top-k, gather) on the whole
    of each small configuration, in a child process with one OpenMP thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-1core"], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"exit {r.returncode}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def max_over_ranks(value_ms, world, device):
    """The slowest rank's time: every rank's value reduced with MAX (one rank: itself)."""
    if world <= 1:
        return value_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, steps, total_ms):
    """Whole-job steps/s: each of the `world` ranks runs `steps` steps of its own
    replica of the workload (weak scaling; the path has no exchange step)."""
    return world * steps / (total_ms / 1000.0)


# ------------------------------------------------------------------ main

def profile_call(W, call, reps):
    """One decode layer of the workload resident on the device: the low-bit
    cache, the first attention, its top-k and the gather of the selection;
    then `call` reps times back to back (merged_fetch carries the pre-fetch of
    a second layer's selection).  Prints one line and exits."""
    import torch
    cfg = dict(workload=W["workload"], B=W["B"], Hq=W["Hq"], Hkv=W["Hkv"], N=W["N"], R=W["R"], bits=W["bits"],
               ks=[W["k"]], pairs=1)
    k = W["k"]
    rig = LayerRig(cfg)
    rig.attn2()
    rig.topk(k)
    rig.gather(k)
    other = None
    if call == "merged_fetch":
        other = LayerRig(cfg, layer=1)
        other.attn2()
        other.topk(k)
    fst = torch.zeros_like(rig.staging)
    fns = {"attn2": rig.attn2, "merged": lambda: rig.merged(k), "topk": lambda: rig.topk(k),
           "gather": lambda: rig.gather(k),
           "merged_fetch": lambda: rig.spc.spc_merged_attn_fetch(
               rig.d, rig.records, rig.resid, rig.q, rig.idx, rig.bitmap, rig.staging, k, rig.o, rig.lse,
               rig.logits, rig.ws, other.host, W["N"], other.idx, k, fst, ws_bytes=rig.ws_bytes, stream=rig.stream)}
    torch.cuda.synchronize()
    for _ in range(reps):
        fns[call]()
    torch.cuda.synchronize()
    print(json.dumps({"profile_call": call, "reps": reps, "workload": W["workload"]}))


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    W = dict(WORKLOAD)
    W["layers"] = args.layers

    if args.profile_call:
        profile_call(W, args.profile_call, args.profile_reps)
        return

    if args.oracle_1core:
        out = {}
        for name, cfg in SMALL_CONFIGS.items():
            ref = OracleSample(cfg, cfg["B"] * cfg["Hkv"])
            secs = [ref.run() for _ in range(5)]
            out[f"{name}_ms_per_layer"] = 1000.0 * statistics.median(secs)
        out["threads"] = 1
        print(json.dumps(out))
        return

    if args.impl == "reference":
        if rank != 0:
            return
        pairs = args.cpu_pairs or min(W["B"] * W["Hkv"], max(16, host_cores()))
        ref = OracleSample(W, pairs)
        for _ in range(args.warmup):
            ref.run()
        secs = [ref.run() for _ in range(max(1, args.steps))]
        dt = statistics.median(secs)
        v = ref.steps_per_s(dt)
        sample = (f"each of the {args.steps} timed 'steps' is one run of the CPU oracle's merged attention + top-k + "
                  f"gather on {ref.P} of {W['B'] * W['Hkv']} (b, kv-head) pairs of one layer "
                  f"({dt:.2f} s median), extrapolated x{ref.scale_to_step:g} "
                  f"({W['B'] * W['Hkv']} / {ref.P} pairs x {W['layers']} layers) to a decode step")
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / v, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": W["workload"]},
                "measured": {"seconds_per_sample": dt, "samples": len(secs), "sample_pairs": ref.P,
                             "pairs_per_layer": W["B"] * W["Hkv"], "layers": W["layers"],
                             "scale_to_step": ref.scale_to_step, "threads": ref.threads,
                             "host_cores": host_cores(),
                             "note": "value and ms_per_step are extrapolated from the sample, not timed steps"},
                "cpu_baseline": {"value": v, "unit": "steps/s", "cores": ref.threads, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    peaks, peak_src = measured_peaks()

    step = DecodeStep(W, args.layers, mode=args.prefetch, gather_ctas=args.gather_ctas, lag=args.prefetch_lag,
                      keep_staged=not args.refetch_all)
    step.capture()
    for _ in range(max(3, args.warmup)):
        step.replay()
    torch.cuda.synchronize()

    # ---- device-resident timed region ----
    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        start.record(step.main)
        for _ in range(args.steps):
            step.replay()
        end.record(step.main)
        barrier()
    # per-layer breakdown: the graph with events between the kernels, replayed after the timed region
    for _ in range(3):
        step.replay_timed()
    torch.cuda.synchronize()
    per_layer = step.attn_ms()
    per_layer_topk = step.topk_ms()
    total_ms = max_over_ranks(start.elapsed_time(end), world, "cuda")
    ms_per_step = total_ms / args.steps
    kept_timed = step.kept_fraction()
    value = job_throughput(world, args.steps, total_ms)
    launches_per_step = step.launches_per_step

    # ---- end to end: each step's queries in from pinned host memory (a different set every step, so the
    # selections and the fetched host rows change), outputs back, every step ----
    n_sets = 8
    q_sets = torch.from_numpy(np.stack([np.stack([synth_queries(s_, l, W) for l in range(args.layers)])
                                        for s_ in range(n_sets)]).view(np.int16).copy()).pin_memory()
    h2d = step.q_host.numel() * step.q_host.element_size()
    d2h = step.o.numel() * step.o.element_size()
    for i in range(args.warmup):  # the same loop untimed: first use of the pinned query sets and output buffer
        with torch.cuda.stream(step.main):
            step.q.copy_(q_sets[i % n_sets], non_blocking=True)
            step.graph.replay()
            step.o_host.copy_(step.o, non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(step.main)
    for i in range(args.steps):
        with torch.cuda.stream(step.main):
            step.q.copy_(q_sets[i % n_sets], non_blocking=True)
            step.graph.replay()
            step.o_host.copy_(step.o, non_blocking=True)
    e1.record(step.main)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
    e2e = {"value": job_throughput(world, args.steps, e2e_ms), "unit": "steps/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h,
           "note": f"queries rotate over {n_sets} seeded sets, so every step selects and fetches other host rows"}
    # the same rotation with the query sets already in HBM (a device copy per step): what fresh
    # selections cost the step, without the host copies
    q_dev = q_sets.to("cuda")
    barrier()
    e0.record(step.main)
    for i in range(args.steps):
        with torch.cuda.stream(step.main):
            step.q.copy_(q_dev[i % n_sets], non_blocking=True)
            step.graph.replay()
    e1.record(step.main)
    barrier()
    fresh_ms = e0.elapsed_time(e1) / args.steps
    kept_fresh = step.kept_fraction()
    step.q.copy_(q_dev[0])
    del q_dev
    torch.cuda.synchronize()

    # ---- overlap test: the step with the pre-fetch against the same step with the staging buffers already
    # filled and no pre-fetch; the two graphs alternate, twice each ----
    L = args.layers
    overlap = None
    if args.prefetch == "overlap":
        g_nofetch = step.capture_step(lambda P: step.enqueue_overlap(fetch=False, parity=P))
        t_f, t_n = [], []
        for _ in range(2):
            t_f.append(step.time_graph(step.graph, reps=max(5, args.steps)))
            t_n.append(step.time_graph(g_nofetch, reps=max(5, args.steps)))
        del g_nofetch
        tf, tn = statistics.mean(t_f), statistics.mean(t_n)
        overlap = {"steps_per_s_with_prefetch": 1000.0 / tf, "steps_per_s_staging_preloaded": 1000.0 / tn,
                   "delta_pct": 100.0 * (tf - tn) / tn, "hidden": (tf - tn) / tn <= 0.02,
                   "prefetch_bytes_per_step": W["B"] * W["Hkv"] * W["k"] * 512 * L,
                   "prefetch_host_bytes_per_step": W["B"] * W["Hkv"] * W["k"] * 512 * L * (1.0 - (kept_timed or 0.0)),
                   "link_bound_ms_per_step": None,
                   "what": "the step as timed, against the same step with every layer's selected rows already in "
                           "HBM and no pre-fetch (spc_merged_attn instead of spc_merged_attn_fetch); 'hidden' is "
                           "a difference of 2% or less"}
    # the host copies of e2e alone, per step
    e0.record(step.main)
    for i in range(args.steps):
        with torch.cuda.stream(step.main):
            step.q.copy_(q_sets[i % n_sets], non_blocking=True)
            step.o_host.copy_(step.o, non_blocking=True)
    e1.record(step.main)
    torch.cuda.synchronize()
    e2e["host_copies_ms_per_step"] = e0.elapsed_time(e1) / args.steps
    step.q.copy_(q_sets[0])
    torch.cuda.synchronize()

    # ---- roofline of the dominant call (merged attention, one layer per call) ----
    # Its live duration is taken from the timed step itself: the layers' attention calls are the only work on
    # the step's main stream (each top-k runs beside them on a second stream), so the main stream's time per
    # layer bounds one call's duration from above (waits for a top-k, if any, are counted against it).
    bytes_layer = attention_bytes_per_layer(W, step.nq)
    attn_avg_ms = ms_per_step / L
    dur_src = (f"the timed step's main stream per layer ({ms_per_step:.4f} ms / {L}): CUDA events on the launching "
               f"stream around {args.steps} graph replays in which the {L} attention calls are that stream's only "
               f"work")
    achieved = bytes_layer / (attn_avg_ms / 1000.0) / 1e9
    pf_bytes = W["B"] * W["Hkv"] * W["k"] * 512 if args.prefetch in ("fused", "step", "overlap") else 0
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"],
            "traffic": attention_traffic() if args.prefetch == "overlap" else None,  # captured on that call
            "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of attn_kernel and combine_kernel "
                              "for one call, from an ncu capture of this build's attention sources (null when "
                              "the sources differ from the captured ones)",
            "kernel": {"side": "spc_merged_attn (attn_kernel + combine_kernel), one layer",
                       "fused": "spc_merged_attn_fetch (attn_kernel + combine_kernel; the previous layer's "
                                "pre-fetch riding along), one layer",
                       "overlap": "spc_merged_attn_fetch (attn_kernel + combine_kernel; the pre-fetch of the layer "
                                  "two before riding along), one layer",
                       "step": "spc_decode_step (attention + combine + top-k, the previous layer's pre-fetch "
                               "riding along), one layer"}[args.prefetch],
            "algorithmic_bytes_per_launch": bytes_layer, "avg_launch_ms": attn_avg_ms,
            "duration_source": dur_src,
            "prefetch_bytes_per_launch": pf_bytes,
            "prefetch_host_bytes_per_launch": pf_bytes * (1.0 - (kept_timed or 0.0)),
            "prefetch_note": "the carried pre-fetch rows (read over the host link, written to HBM) are not in the "
                             "algorithmic bytes; they are accounted against the host link in 'gather'",
            "peak_source": f"{peak_src} hbm_gbs (burst copy)",
            "step_hbm_gbs": bytes_layer * L / (ms_per_step / 1000.0) / 1e9,
            "step_hbm_frac": bytes_layer * L / (ms_per_step / 1000.0) / 1e9 / peaks["hbm_gbs"]}

    gather = host_link_probe(step, reps=20)
    if overlap is not None:
        overlap["link_bound_ms_per_step"] = (overlap["prefetch_host_bytes_per_step"] /
                                             (gather["host_link_peak_gbs"] * 1e6))
    append = append_probe(W) if rank == 0 else None
    serial = step.time_serial(max(5, args.steps // 4), args.warmup) if rank == 0 else None
    prefill = prefill_probe(W) if rank == 0 else None
    peak_hbm = peaks["hbm_gbs"]
    del step
    torch.cuda.empty_cache()
    configs = measure_configs(peak_hbm, oracle_on=not args.no_cpu_baseline) if (rank == 0 and args.configs) \
        else None

    line = {"metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16-mma/f32", "data": "synthetic",
            "config": {"workload": W["workload"], "layers": W["layers"], "batch": W["B"], "context": W["N"],
                       "bits": W["bits"], "k": W["k"], "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (4.3 GB low-bit cache per step, 129 MB L2); no flush",
                       "graph": "one CUDA graph per step",
                       "replay": "every timed step replays the same queries; the selection then alternates with "
                                 "period two (a fetched row's exact logit replaces its low-bit estimate in the "
                                 "next step): consecutive steps share 38% of their selected rows, steps two apart "
                                 "all of them (see e2e and fresh_queries for changing queries); the decode-time "
                                 "append of the new token is not in the step (see append)",
                       "prefetch": {"side": f"side stream, {args.gather_ctas} CTAs",
                                    "fused": "fused into the next layer's attention",
                                    "step": "fused into the next layer's attention, which also ends with "
                                            "the top-k (spc_decode_step, speculative logits kept in TMEM)",
                                    "overlap": "fused into the attention two layers on; top-k on a "
                                               "low-priority stream beside the next attention"}[args.prefetch] +
                                   ("; the rows that the layer's previous selection already staged are copied "
                                    "from HBM, the others read from the host" if kept_timed is not None else "")},
            "roofline": roof, "overlap": overlap, "gather": gather,
            "prefetch_rows": None if kept_timed is None else {
                "kept": kept_timed, "kept_fresh_queries": kept_fresh,
                "what": "of the rows each step's pre-fetches stage, the fraction that the layer's previous "
                        "selection had staged already (copied from HBM; the rest come over the host link): "
                        "in the timed step, and with the queries rotating over unrelated seeded sets"},
            "fresh_queries": {"value": 1000.0 / fresh_ms, "unit": "steps/s",
                              "what": "the step with the queries rotating over 8 seeded sets already in HBM"},
            "per_layer_us": {"attention": statistics.mean(per_layer) * 1000.0,
                             "topk": statistics.mean(per_layer_topk) * 1000.0,
                             "note": "CUDA events around each call inside a copy of the step's graph (the events "
                                     "break the programmatic overlap of neighbouring launches, so these run a few "
                                     "microseconds longer than in the timed step)"},
            "append": append,
            "nonspeculative_baseline": serial,
            "prefill": prefill, "configs": configs, "clocks": clk.summary(), "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps}
    if rank == 0 and not args.no_cpu_baseline:
        pairs = args.cpu_pairs or min(W["B"] * W["Hkv"], max(16, host_cores()))
        ref = OracleSample(W, pairs)
        secs = []
        while sum(secs) < 10.0 and len(secs) < 1000:  # about 10 s of oracle work
            secs.append(ref.run())
        dt = statistics.median(secs)
        line["cpu_baseline"] = {"value": ref.steps_per_s(dt), "unit": "steps/s", "cores": ref.threads,
                                "host_cores": host_cores(), "kind": "oracle",
                                "sample": f"merged attention + top-k + gather of {ref.P} (b, kv-head) pairs of one "
                                          f"layer, {len(secs)} runs in {sum(secs):.1f} s (median {dt:.3f} s), "
                                          f"scaled to {W['B'] * W['Hkv']} pairs x {W['layers']} layers",
                                "sample_pairs": ref.P, "pairs_per_layer": W["B"] * W["Hkv"], "layers": W["layers"],
                                "measured_s_per_sample": dt, "scale_to_step": ref.scale_to_step,
                                "single_core": oracle_single_core()}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
