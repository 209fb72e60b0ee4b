"""Shared helpers of the GPU parity tests: the five workload configurations,
runners for the CUDA path (through the C ABI) and for the CPU oracle, and the
comparison rules (codes bit-exact; top-k sets equal except within 1e-5
relative of the k-th score; outputs within 2e-3 max-abs of the fp64 oracle)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth

# Workloads (shapes of the pages' LLaMA-2-7B / LLaMA-3-8B / Mistral-7B layers).
CONFIGS = {
    "c1": dict(B=1, Hq=1, Hkv=1, N=1024, R=32, bits=1, k=16),
    "c2": dict(B=1, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328),
    "c3": dict(B=16, Hq=32, Hkv=32, N=2048, R=128, bits=2, k=64),
    "c4": dict(B=8, Hq=32, Hkv=8, N=32768, R=128, bits=1, k=328, layers=32),
}
SEED = 0
OUT_TOL = 2e-3     # max-abs on bf16 outputs against the fp64 oracle
TOPK_REL = 1e-5    # boundary band for top-k set differences


def bf16_half_ulp(x) -> np.ndarray:
    """Half a bf16 unit in the last place at |x| (bf16 keeps 8 significant bits)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 0.5 * np.power(2.0, e - 7)


def out_err(got_bf16_as_f64, ref) -> float:
    """Error of a bf16 output against the fp64 oracle beyond the output format's
    own rounding: max(|got - ref| - half_ulp_bf16(ref)).  The bound OUT_TOL
    applies to this quantity (2e-3 on the kernel's fp32 result; the bf16 store
    adds up to half an ulp, which alone exceeds 2e-3 once |o| >= 1)."""
    return float(np.max(np.abs(got_bf16_as_f64 - ref) - bf16_half_ulp(ref)))


def k_from_fraction(p: float, N: int) -> int:
    return int(math.ceil(round(p * N, 6)))


def c5_cases():
    out = []
    for B in (1, 4):
        for N in (4096, 16384, 65536, 131072):
            for bits in (1, 2):
                for p in (0.005, 0.01, 0.04):
                    out.append(dict(B=B, Hq=32, Hkv=8, N=N, R=128, bits=bits, k=k_from_fraction(p, N)))
    return out


def b2f(bits) -> np.ndarray:
    return synth.bf16_to_f32(np.asarray(bits).view(np.uint16)).astype(np.float64)


def odims(cfg, B=None, Hkv=None, Hq=None):
    B = cfg["B"] if B is None else B
    Hkv = cfg["Hkv"] if Hkv is None else Hkv
    Hq = cfg["Hq"] if Hq is None else Hq
    return oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=cfg["N"], R=cfg["R"], bits=cfg["bits"],
                       scale=float(np.float32(1.0 / math.sqrt(128))), group=cfg.get("group", 32))


def interleave_host(K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """[B,Hkv,N,D] x 2 -> the 16-bit cache row format [B,Hkv,N,2,D]."""
    return np.ascontiguousarray(np.stack([K, V], axis=3))


class GpuLayer:
    """One layer's cache and buffers on the device, driven through the C ABI."""

    def __init__(self, cfg, K=None, V=None, seed=SEED, layer=0, kcap=None, host=True, q=None):
        import bit_kv_cache_spc_gb300 as spc
        self.spc = spc
        self.cfg = cfg
        B, Hq, Hkv, N, R, bits = (cfg[x] for x in ("B", "Hq", "Hkv", "N", "R", "bits"))
        self.G = Hq // Hkv
        self.d = spc.Dims(B, Hq, Hkv, N, R, bits, scale=float(np.float32(1.0 / math.sqrt(128))),
                          group=cfg.get("group", 32))
        self.nq = spc.spc_num_quantized(self.d)
        dev = torch.device("cuda")
        if K is None:
            import synth.gpu
            Kt = torch.empty((B, Hkv, N, 128), dtype=torch.int16, device=dev)
            Vt = torch.empty_like(Kt)
            synth.gpu.kv_layer_into(seed, layer, Kt, Vt)
        else:
            Kt = torch.from_numpy(np.ascontiguousarray(K).view(np.int16)).to(dev)
            Vt = torch.from_numpy(np.ascontiguousarray(V).view(np.int16)).to(dev)
        self.K, self.V = Kt, Vt
        self.records = torch.zeros(max(spc.spc_records_bytes(self.d), 16), dtype=torch.uint8, device=dev)
        self.resid = torch.zeros(max(spc.spc_resid_bytes(self.d) // 2, 8), dtype=torch.int16, device=dev)
        spc.spc_quantize_kv(self.d, Kt, Vt, self.records, self.resid)
        qn = synth.queries(seed, layer, B, Hq) if q is None else q
        self.q_np = qn
        self.q = torch.from_numpy(qn.view(np.int16).copy()).to(dev)
        self.Lcap = self.d.q_groups_cap * 32
        self.kcap = cfg["k"] if kcap is None else kcap
        # zero-filled once, as the workspace contract asks
        self.ws = torch.zeros(max(spc.spc_attn_workspace_bytes(self.d, max(self.kcap, self.nq)), 16),
                              dtype=torch.uint8, device=dev)
        self.host = None
        if host:
            self.host = torch.empty((B, Hkv, N, 2, 128), dtype=torch.int16, pin_memory=True)
            self.host.copy_(torch.stack([Kt, Vt], dim=3).cpu())
        self.staging = torch.zeros((B, Hkv, max(self.kcap, 1), 2, 128), dtype=torch.int16, device=dev)

    def new_out(self):
        B, Hq, Hkv = self.cfg["B"], self.cfg["Hq"], self.cfg["Hkv"]
        o = torch.zeros((B, 2, Hq, 128), dtype=torch.int16, device="cuda")
        lse = torch.zeros((B, 2, Hq), dtype=torch.float32, device="cuda")
        lg = torch.full((B, Hkv, self.G, max(self.Lcap, 1)), float("nan"), dtype=torch.float32, device="cuda")
        return o, lse, lg

    def attn2(self, kv_self=None):
        o, lse, lg = self.new_out()
        self.spc.spc_decode_attn2(self.d, self.records, self.resid, self.q, o, lse, lg, self.ws, kv_self=kv_self)
        return o, lse, lg

    def merged(self, idx, bitmap, k, kv_self=None):
        o, lse, lg = self.new_out()
        self.spc.spc_merged_attn(self.d, self.records, self.resid, self.q, idx, bitmap, self.staging, k, o, lse, lg,
                                 self.ws, kv_self=kv_self)
        return o, lse, lg

    def topk(self, lg, lse, k):
        B, Hkv = self.cfg["B"], self.cfg["Hkv"]
        idx = torch.full((B, Hkv, max(k, 1)), -7, dtype=torch.int32, device="cuda")
        bm = torch.full((B, Hkv, max(self.d.q_groups_cap, 1)), 0xDEAD, dtype=torch.int32, device="cuda")
        self.spc.spc_topk_select(self.d, lg, lse, k, idx, bm)
        return idx[..., :k], bm[..., :self.d.q_groups_cap]

    def gather(self, idx, k, max_ctas=0):
        self.spc.spc_host_gather(self.d, self.host, self.cfg["N"], idx, k, self.staging, max_ctas)


class PairOracle:
    """The oracle on one (b, hkv) of a configuration, as a 1 x 1 sub-problem on
    the same seeded inputs; the pair's K/V, queries and quantisation are made
    once and shared by every attention call."""

    def __init__(self, cfg, b, hk, K=None, V=None, seed=SEED, layer=0):
        B, Hq, Hkv, N = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"]
        G = Hq // Hkv
        if K is None:
            k, v = synth.kv_slice(seed, layer, B, Hkv, N, 128, b, hk)
        else:
            k, v = K[b, hk], V[b, hk]
        self.K, self.V = k[None, None], v[None, None]
        self.q = synth.queries(seed, layer, B, Hq)[b:b + 1, :, hk * G:(hk + 1) * G]
        self.d = odims(cfg, B=1, Hkv=1, Hq=G)
        self.qz = oracle.quantize(self.d, self.K, self.V)

    def attention(self, idx=None):
        """(o [2, G, D], lse [2, G], S [N_q]) with the 16-bit rows at idx (or none)."""
        o, lse, S = oracle.attention(self.d, self.q, self.qz, self.K, self.V,
                                     idx=None if idx is None else np.asarray(idx)[None, None])
        return o[0], lse[0], S[0, 0]

    def topk(self, S, k):
        io, _ = oracle.topk(self.d, S[None, None], k)
        return io[0, 0]


def oracle_pair(cfg, b, hk, K=None, V=None, idx=None, seed=SEED, layer=0):
    """Oracle outputs of one (b, hkv) of a configuration (a 1 x 1 sub-problem)."""
    p = PairOracle(cfg, b, hk, K=K, V=V, seed=seed, layer=layer)
    o, lse, S = p.attention(idx)
    return dict(d=p.d, K=p.K, V=p.V, qz=p.qz, o=o, lse=lse, S=S)


def check_topk_sets(idx_gpu, idx_orc, S_orc, k):
    """Sets equal except for positions whose oracle score lies within TOPK_REL of
    the oracle's k-th score; ascending order and -1 padding are exact."""
    nq = S_orc.shape[-1]
    keff = min(k, nq)
    g = np.asarray(idx_gpu)
    assert np.all(g[keff:] == -1)
    g = g[:keff]
    assert np.all(np.diff(g) > 0), "indices not strictly ascending"
    o = np.asarray(idx_orc)[:keff]
    if keff == 0:
        return 0
    sk = S_orc[o].min()
    diff = set(g.tolist()) ^ set(o.tolist())
    for n in diff:
        assert abs(S_orc[n] - sk) <= TOPK_REL * sk, f"position {n}: S={S_orc[n]!r} vs k-th {sk!r}"
    return len(diff)


def bitmap_from_idx(idx, n_words):
    bm = np.zeros(n_words, np.uint32)
    for n in idx:
        if n >= 0:
            bm[n // 32] |= np.uint32(1) << np.uint32(n % 32)
    return bm
