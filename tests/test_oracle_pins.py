"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: the hand
worked examples under tests/golden (from the SpeCache page's formulas), the
half-interval geometry the page states, exact rational arithmetic, library
routines (torch's scaled-dot-product attention and softmax in fp64, numpy's
lexsort), closed-form byte counts the page prints, and invariants of softmax
attention.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f2b(x):
    """Exact bf16 bits of a float that is representable in bf16."""
    b = synth.f32_to_bf16_rne(np.asarray(x, np.float32))
    assert np.all(synth.bf16_to_f32(b) == np.asarray(x, np.float32)), "not a bf16 value"
    return b


def b2f(b):
    return synth.bf16_to_f32(np.asarray(b, np.uint16)).astype(np.float64)


def read_golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append([s.split() for s in line.split("|")])
    return rows


def quantize_key_group(bits, values, mode=0, group=32):
    """Quantise one key group (`group` tokens of channel 0) holding `values` (padded)."""
    vals = list(values) + [values[0]] * (group - len(values))
    N = group
    d = oracle.dims(B=1, Hq=1, Hkv=1, N=N, R=0, bits=bits, group=group)
    K = np.zeros((1, 1, N, 128), np.uint16)
    K[0, 0, :, 0] = f2b(np.array(vals, np.float32))
    V = np.zeros_like(K)
    qz = oracle.quantize(d, K, V, mode=mode)
    codes = qz["kcode"][0, 0, :len(values), 0].astype(int)
    lo, hi = qz["kmm"][0, 0, 0, 0]
    deq = [oracle.dequant(bits, int(lo), int(hi), int(c), mode) for c in codes]
    return codes, deq, b2f(lo), b2f(hi)


@pytest.mark.parametrize("name,bits", [("quant_1bit_worked.txt", 1), ("quant_2bit_worked.txt", 2)])
def test_golden_worked_examples(name, bits):
    for (mm, vals, codes, deq) in read_golden(name):
        lo, hi = float(mm[0]), float(mm[1])
        values = [float(v) for v in vals]
        # pad with min and max so the group's extremes are the stated ones
        group = values + [lo, hi]
        got_codes, got_deq, glo, ghi = quantize_key_group(bits, group)
        assert (glo, ghi) == (lo, hi)
        assert list(got_codes[:len(values)]) == [int(c) for c in codes]
        assert got_deq[:len(values)] == [float(x) for x in deq]


def random_bf16_group(rng, n, lo_exp=-3, hi_exp=3):
    """bf16 values whose exponents stay within a small range (P1's premise)."""
    mant = rng.integers(128, 256, size=n)
    exp = rng.integers(lo_exp, hi_exp + 1, size=n)
    sign = rng.choice([-1.0, 1.0], size=n)
    return (sign * mant.astype(np.float64) / 128.0 * np.power(2.0, exp)).astype(np.float32)


def test_p1_one_bit_lands_on_half_interval_centres():
    """Page 1 section 3: values below the midpoint dequantise to the centre of
    [min, mid), values above it to the centre of (mid, max], exactly."""
    rng = np.random.default_rng(1)
    for _ in range(200):
        vals = random_bf16_group(rng, 32)
        codes, deq, lo, hi = quantize_key_group(1, list(vals))
        lo_f, hi_f = Fraction(lo), Fraction(hi)
        mid = (lo_f + hi_f) / 2
        low_centre = (lo_f + mid) / 2
        high_centre = (mid + hi_f) / 2
        for x, c, xd in zip(vals, codes, deq):
            xf = Fraction(float(x))
            want = 0 if xf <= mid else 1
            assert c == want
            assert Fraction(xd) == (low_centre if c == 0 else high_centre)


def test_p1_centres_minimise_uniform_error():
    """The page's reason for the new z, s: under a uniform distribution on
    [min, max] the two half-interval centres minimise the mean squared error.
    Moving either reconstruction level away from the oracle's value raises it."""
    codes, deq, lo, hi = quantize_key_group(1, [-1.0, 3.0])
    levels = sorted(set(deq))
    x = np.linspace(lo, hi, 200001)

    def mse(l0, l1):
        return np.mean(np.minimum((x - l0) ** 2, (x - l1) ** 2))

    base = mse(*levels)
    for d0, d1 in [(0.05, 0), (-0.05, 0), (0, 0.05), (0, -0.05)]:
        assert mse(levels[0] + d0, levels[1] + d1) > base
    # original KIVI 1-bit (z = min, s = max - min) gives a strictly larger error
    _, deq_kivi, _, _ = quantize_key_group(1, [-1.0, 3.0], mode=1)
    assert mse(*sorted(set(deq_kivi))) > base


@pytest.mark.parametrize("group", [32, 64])
def test_p2_two_bit_nearest_grid_point(group):
    """KIVI 2-bit: the code is the nearest point of {min + i*s}, s=(max-min)/3,
    min and max taken over the whole group (32 or 64 tokens)."""
    rng = np.random.default_rng(2)
    for _ in range(200 if group == 32 else 100):
        vals = random_bf16_group(rng, group)
        codes, deq, lo, hi = quantize_key_group(2, list(vals), group=group)
        lo_f, hi_f = Fraction(lo), Fraction(hi)
        for x, c in zip(vals, codes):
            if hi_f == lo_f:
                assert c == 0
                continue
            t = 3 * (Fraction(float(x)) - lo_f) / (hi_f - lo_f)
            fl = math.floor(t)
            if t - fl == Fraction(1, 2):
                assert c in (fl, fl + 1)  # exact ties: either neighbour is nearest
            else:
                assert c == min(max(round(t), 0), 3)


def test_p3_original_kivi_one_bit_gives_min_and_max():
    """Page 1 section 3: with the original KIVI rule at 1 bit every X' is max X or min X."""
    rng = np.random.default_rng(3)
    vals = random_bf16_group(rng, 32)
    codes, deq, lo, hi = quantize_key_group(1, list(vals), mode=1)
    assert set(deq) <= {lo, hi}
    two = quantize_key_group(1, [0.5, 2.0] * 16)
    assert two[0][0] != two[0][1]  # SpeCache's rule separates a two-valued group


def test_constant_group_and_value_axis():
    """min == max gives code 0 and X' = the constant; value groups run over channels."""
    d = oracle.dims(B=1, Hq=1, Hkv=1, N=32, R=0, bits=1)
    K = np.full((1, 1, 32, 128), f2b(np.float32(0.75)), np.uint16)
    V = np.zeros_like(K)
    V[0, 0, 5, 32:64] = f2b(np.float32(-2.0))
    V[0, 0, 5, 40] = f2b(np.float32(1.0))
    qz = oracle.quantize(d, K, V)
    assert np.all(qz["kcode"] == 0)
    assert oracle.dequant(1, int(qz["kmm"][0, 0, 0, 3, 0]), int(qz["kmm"][0, 0, 0, 3, 1]), 0) == 0.75
    lo, hi = qz["vmm"][0, 0, 5, 1]
    assert (b2f(lo), b2f(hi)) == (-2.0, 1.0)
    assert qz["vcode"][0, 0, 5, 40] == 1 and qz["vcode"][0, 0, 5, 33] == 0
    assert tuple(qz["vmm"][0, 0, 5, 0]) == (0, 0)  # -0.0/+0.0 stored as +0.0


def test_residual_split():
    for N, R, want in [(1024, 32, 992), (32768, 128, 32640), (100, 64, 32), (64, 64, 0), (10, 64, 0),
                       (2048, 128, 1920)]:
        assert oracle.nq(oracle.dims(B=1, Hq=1, Hkv=1, N=N, R=R, bits=1)) == want


def dequant_tensors(d, qz):
    """Dequantised K', V' of the oracle's own codes (fp64), for library comparisons."""
    nq = oracle.nq(d)
    kmm = b2f(qz["kmm"])
    vmm = b2f(qz["vmm"])
    klo = np.repeat(kmm[..., 0], d.group, axis=2)
    khi = np.repeat(kmm[..., 1], d.group, axis=2)
    vlo = np.repeat(vmm[..., 0], d.group, axis=3)
    vhi = np.repeat(vmm[..., 1], d.group, axis=3)
    if d.bits == 1:
        kz, ks = (3 * klo + khi) / 4, (khi - klo) / 2
        vz, vs = (3 * vlo + vhi) / 4, (vhi - vlo) / 2
    else:
        kz, ks = klo, (khi - klo) / 3
        vz, vs = vlo, (vhi - vlo) / 3
    Kd = qz["kcode"].astype(np.float64) * ks + kz
    Vd = qz["vcode"].astype(np.float64) * vs + vz
    assert Kd.shape[2] == nq
    return Kd, Vd


def sdpa_reference(d, q, Keff, Veff):
    """torch's attention and softmax in fp64 over the effective K, V rows."""
    G = d.Hq // d.Hkv
    qf = torch.from_numpy(b2f(q))  # [B,2,Hq,D]
    Kt = torch.from_numpy(Keff).repeat_interleave(G, dim=1)  # [B,Hq,N,D]
    Vt = torch.from_numpy(Veff).repeat_interleave(G, dim=1)
    qh = qf.permute(0, 2, 1, 3)  # [B,Hq,2,D]
    o = torch.nn.functional.scaled_dot_product_attention(qh, Kt, Vt, scale=d.scale)
    logits = torch.einsum("bhid,bhnd->bhin", qh, Kt) * d.scale
    lse = torch.logsumexp(logits, dim=-1)
    p = torch.softmax(logits, dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.permute(0, 2, 1).numpy(), p.numpy()


@pytest.mark.parametrize("bits,B,Hq,Hkv,N,R,group", [(1, 1, 4, 1, 160, 64, 32), (2, 2, 2, 2, 96, 32, 32),
                                                     (1, 1, 8, 2, 200, 40, 32), (1, 1, 4, 1, 230, 40, 64),
                                                     (2, 1, 8, 2, 300, 64, 64)])
def test_p6_attention_matches_library_on_tiny_inputs(bits, B, Hq, Hkv, N, R, group):
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=bits, group=group)
    K, V = synth.kv_layer(7, 0, B, Hkv, N)
    q = synth.queries(7, 0, B, Hq)
    qz = oracle.quantize(d, K, V)
    nq = oracle.nq(d)
    Kd, Vd = dequant_tensors(d, qz)
    Keff = np.concatenate([Kd, b2f(K)[:, :, nq:]], axis=2)
    Veff = np.concatenate([Vd, b2f(V)[:, :, nq:]], axis=2)
    o_ref, lse_ref, p_ref = sdpa_reference(d, q, Keff, Veff)
    o, lse, S = oracle.attention(d, q, qz, K, V)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    G = Hq // Hkv
    S_ref = p_ref[:, :, 1, :nq].reshape(B, Hkv, G, nq).sum(axis=2)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("bits,Hq,Hkv,N,R", [(1, 4, 1, 160, 64), (2, 8, 2, 200, 40)])
def test_p11_speculative_self_row_is_seen_by_the_speculative_query_only(bits, Hq, Hkv, N, R):
    """Algorithm 3 attends over [K, K_t] with the new tokens' rows; the
    speculative token follows T_t, so with its own key/value row given, query
    row 1 attends over N + 1 rows and row 0 over the N cache rows (torch's
    fp64 attention with a causal mask), and row 0 is bit-identical to the
    call without the row."""
    B = 2
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=bits)
    K, V = synth.kv_layer(13, 0, B, Hkv, N)
    q = synth.queries(13, 0, B, Hq)
    K1, V1 = synth.kv_layer(14, 0, B, Hkv, 1)
    kv_self = np.stack([K1[:, :, 0], V1[:, :, 0]], axis=2)  # [B,Hkv,2,D]
    qz = oracle.quantize(d, K, V)
    nq = oracle.nq(d)
    Kd, Vd = dequant_tensors(d, qz)
    Keff = np.concatenate([Kd, b2f(K)[:, :, nq:], b2f(kv_self)[:, :, None, 0]], axis=2)  # N + 1 rows
    Veff = np.concatenate([Vd, b2f(V)[:, :, nq:], b2f(kv_self)[:, :, None, 1]], axis=2)
    G = Hq // Hkv
    qh = torch.from_numpy(b2f(q)).permute(0, 2, 1, 3)  # [B,Hq,2,D]
    Kt = torch.from_numpy(Keff).repeat_interleave(G, dim=1)
    Vt = torch.from_numpy(Veff).repeat_interleave(G, dim=1)
    mask = torch.ones((2, N + 1), dtype=torch.bool)
    mask[0, N] = False  # T_t does not see the speculative token's row
    o_ref = torch.nn.functional.scaled_dot_product_attention(qh, Kt, Vt, attn_mask=mask, scale=d.scale)
    logits = (torch.einsum("bhid,bhnd->bhin", qh, Kt) * d.scale).masked_fill(~mask, float("-inf"))
    lse_ref = torch.logsumexp(logits, dim=-1).permute(0, 2, 1).numpy()
    p_ref = torch.softmax(logits, dim=-1).numpy()
    o, lse, S = oracle.attention(d, q, qz, K, V, kv_self=kv_self)
    np.testing.assert_allclose(o, o_ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    S_ref = p_ref[:, :, 1, :nq].reshape(B, Hkv, G, nq).sum(axis=2)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-13)
    o0, lse0, S0 = oracle.attention(d, q, qz, K, V)
    assert np.array_equal(o[:, 0], o0[:, 0]) and np.array_equal(lse[:, 0], lse0[:, 0])
    assert np.abs(o[:, 1] - o0[:, 1]).max() > 1e-4 and np.all(S < S0 + 1e-15)  # the row takes probability


def test_p4_all_positions_fetched_equals_full_precision_attention():
    """Page 1 section 3: C' U C_kappa replaces the low-bit rows by the 16-bit
    ones, so fetching every position gives plain bf16 attention."""
    B, Hq, Hkv, N, R = 1, 4, 2, 192, 64
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=1)
    K, V = synth.kv_layer(11, 0, B, Hkv, N)
    q = synth.queries(11, 0, B, Hq)
    qz = oracle.quantize(d, K, V)
    nq = oracle.nq(d)
    idx = np.broadcast_to(np.arange(nq, dtype=np.int32), (B, Hkv, nq)).copy()
    o, lse, S = oracle.attention(d, q, qz, K, V, idx=idx)
    o_ref, lse_ref, _ = sdpa_reference(d, q, b2f(K), b2f(V))
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    # and the low-bit attention is measurably different (the substitution matters)
    o0, _, _ = oracle.attention(d, q, qz, K, V)
    assert np.abs(o0 - o_ref).max() > 1e-3


def test_p5_k0_is_plain_low_bit_attention_and_padding_is_ignored():
    B, Hq, Hkv, N, R = 1, 4, 1, 160, 32
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=1)
    K, V = synth.kv_layer(5, 0, B, Hkv, N)
    q = synth.queries(5, 0, B, Hq)
    qz = oracle.quantize(d, K, V)
    a = oracle.attention(d, q, qz, K, V)
    b = oracle.attention(d, q, qz, K, V, idx=np.zeros((B, Hkv, 0), np.int32))
    c = oracle.attention(d, q, qz, K, V, idx=np.full((B, Hkv, 4), -1, np.int32))
    for x, y, z in zip(a, b, c):
        assert np.array_equal(x, y) and np.array_equal(x, z)


def test_p9_softmax_invariants():
    B, Hq, Hkv, N = 1, 4, 1, 128
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=0, bits=1)
    K, V = synth.kv_layer(3, 0, B, Hkv, N)
    q = synth.queries(3, 0, B, Hq)
    qz = oracle.quantize(d, K, V)
    o, lse, S = oracle.attention(d, q, qz, K, V)
    # no residual: the speculative row sums to 1 per query head
    np.testing.assert_allclose(S.sum(axis=-1), Hq // Hkv, rtol=1e-13)
    # the same V row at every position, constant within each 32-channel value
    # group (so quantisation is lossless), comes back exactly
    row = np.repeat(f2b(np.array([0.5, -1.25, 3.0, 0.0], np.float32)), 32)
    Vc = np.broadcast_to(row, V.shape).copy()
    qzc = oracle.quantize(d, K, Vc)
    oc, _, _ = oracle.attention(d, q, qzc, K, Vc)
    np.testing.assert_allclose(oc, np.broadcast_to(b2f(Vc[:, 0, 0, :])[:, None, None, :], oc.shape), atol=1e-12)
    # permuting whole 32-token groups permutes S and leaves o, lse unchanged
    perm = np.array([2, 0, 3, 1])
    tok = (perm[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
    Kp, Vp = K[:, :, tok], V[:, :, tok]
    qzp = oracle.quantize(d, Kp, Vp)
    op, lsep, Sp = oracle.attention(d, q, qzp, Kp, Vp)
    np.testing.assert_allclose(op, o, atol=1e-12)
    np.testing.assert_allclose(lsep, lse, atol=1e-12)
    np.testing.assert_allclose(Sp, S[:, :, tok], atol=1e-15)


def test_topk_matches_library_sort_with_ties():
    rng = np.random.default_rng(4)
    B, Hkv, nq = 2, 3, 320
    d = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=nq, R=0, bits=1)
    S = rng.integers(0, 40, size=(B, Hkv, nq)).astype(np.float64) / 7.0  # many ties
    for k in (0, 1, 17, 64, 320, 400):
        idx, bm = oracle.topk(d, S, k)
        keff = min(k, nq)
        for b in range(B):
            for h in range(Hkv):
                order = np.lexsort((np.arange(nq), -S[b, h]))
                want = np.sort(order[:keff])
                assert np.array_equal(idx[b, h, :keff], want)
                assert np.all(idx[b, h, keff:] == -1)
                bits = np.unpackbits(bm[b, h].view(np.uint8), bitorder="little")[:nq]
                assert np.array_equal(np.flatnonzero(bits), want)


def test_p10_single_head_topk_is_topk_by_logit():
    B, Hq, Hkv, N, R = 1, 1, 1, 288, 32
    d = oracle.dims(B=B, Hq=Hq, Hkv=Hkv, N=N, R=R, bits=1)
    K, V = synth.kv_layer(9, 0, B, Hkv, N)
    q = synth.queries(9, 0, B, Hq)
    qz = oracle.quantize(d, K, V)
    _, _, S = oracle.attention(d, q, qz, K, V)
    Kd, _ = dequant_tensors(d, qz)
    logits = torch.from_numpy(Kd[0, 0]) @ torch.from_numpy(b2f(q[0, 1, 0]))
    idx, _ = oracle.topk(d, S, 20)
    want = np.sort(np.lexsort((np.arange(len(logits)), -logits.numpy()))[:20])
    assert np.array_equal(idx[0, 0], want)


def test_p7_gather_is_an_exact_row_copy():
    rng = np.random.default_rng(6)
    B, Hkv, ncap, k = 2, 3, 500, 37
    d = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=ncap, R=0, bits=1)
    host = rng.integers(0, 1 << 16, size=(B, Hkv, ncap, 2, 128), dtype=np.uint16)
    idx = np.sort(rng.choice(ncap, size=(B, Hkv, k)), axis=-1).astype(np.int32)
    st = oracle.gather(d, host, idx)
    for b in range(B):
        for h in range(Hkv):
            assert st[b, h].tobytes() == host[b, h, idx[b, h]].tobytes()


def test_p8_compression_ratio_matches_printed_values():
    """Figure 4 caption: 0.13 (Mistral, 32k) and 0.14 (LLaMA-3, 8k) at g = 32.
    The low-bit copy stores codes plus a bf16 (min, max) pair per 32 values."""
    for (row,) in read_golden("compression_ratio.txt"):
        model, ctx, resid, bits, printed = row
        ctx, resid, bits = int(ctx), int(resid), int(bits)
        d = oracle.dims(B=1, Hq=1, Hkv=1, N=ctx, R=resid, bits=bits)
        nq = oracle.nq(d)
        gpu_bytes = nq // 32 * oracle.record_bytes(bits) + (ctx - nq) * 2 * 128 * 2
        ratio = gpu_bytes / (ctx * 2 * 128 * 2)
        assert round(ratio, 2) == float(printed)
    # fp32 metadata would not reproduce the printed ratios
    assert round((32640 * (32 + 64) + 128 * 512) / (32768 * 512), 2) != 0.13


def test_pack_places_every_bit_exactly_once():
    """The packed layout is a bijection between (token, channel, plane) and bits."""
    for bits in (1, 2):
        d = oracle.dims(B=1, Hq=1, Hkv=1, N=32, R=0, bits=bits)
        K = np.zeros((1, 1, 32, 128), np.uint16)
        V = np.zeros_like(K)
        base = oracle.quantize(d, K, V)
        seen_k = set()
        seen_v = set()
        for p in range(bits):
            for n in range(0, 32, 3):
                for c in range(0, 128, 5):
                    for which in ("kcode", "vcode"):
                        qz = {k: v.copy() for k, v in base.items()}
                        qz[which][0, 0, n, c] = 1 << p
                        rec, _ = oracle.pack(d, qz, K, V)
                        on = np.flatnonzero(np.unpackbits(rec[0, 0, 0]))
                        assert len(on) == 1
                        (seen_k if which == "kcode" else seen_v).add(int(on[0]))
        assert len(seen_k) == len(seen_v) == bits * 11 * 26


def code_word_rule(p, kc, vc, kcode, vcode, n0):
    """The code-word rule of the header, restated: every bit of the K and V code
    planes kc, vc of the 32 tokens n0 .. n0+31 against the logical codes."""
    for L in range(32):
        a, t = L >> 2, L & 3
        for j in range(4):
            kw, vw = int(kc[128 * p + 4 * L + j]), int(vc[128 * p + 4 * L + j])
            for b in range(32):
                v = (b + 21) % 32
                n, q = v % 4, v // 4
                i, h = (4 - q % 4) % 4, 1 if 1 <= q <= 4 else 0
                e = 4 * j + i
                tok, ch = 8 * n + a, 16 * (e >> 1) + 8 * (e & 1) + 2 * t + h
                assert (kw >> b) & 1 == (int(kcode[n0 + tok, ch]) >> p) & 1
                tok = 16 * (j >> 1) + 8 * (j & 1) + 2 * t + (b >> 4)
                ch = 16 * ((b & 15) >> 1) + 8 * (b & 1) + a
                assert (vw >> b) & 1 == (int(vcode[n0 + tok, ch]) >> p) & 1


@pytest.mark.parametrize("bits", [1, 2])
def test_pack_follows_the_documented_index_rule(bits):
    """Every bit and metadata word of the packed records, read back with the
    index rule as the library's header states it (restated here), equals the
    logical codes and (min, max) of the quantiser."""
    B, Hkv, N = 1, 1, 64
    d = oracle.dims(B=B, Hq=1, Hkv=Hkv, N=N, R=0, bits=bits)
    K, V = synth.kv_layer(21, 0, B, Hkv, N)
    qz = oracle.quantize(d, K, V)
    rec, _ = oracle.pack(d, qz, K, V)
    kcode, vcode, kmm, vmm = qz["kcode"][0, 0], qz["vcode"][0, 0], qz["kmm"][0, 0], qz["vmm"][0, 0]
    assert kcode.max() > 0 and vcode.max() > 0
    for g in range(N // 32):
        w = np.frombuffer(rec[0, 0, g].tobytes(), dtype="<u4")
        kc, km, vc, vm = w[:128 * bits], w[128 * bits:128 * bits + 128], w[128 * bits + 128:256 * bits + 128], \
            w[256 * bits + 128:]
        for p in range(bits):
            code_word_rule(p, kc, vc, kcode, vcode, 32 * g)
        for t in range(4):
            for m in range(32):
                ch = 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1) + (m & 1)
                assert int(km[32 * t + m]) == int(kmm[g, ch, 0]) | (int(kmm[g, ch, 1]) << 16)
                tok = 16 * (m >> 4) + 8 * ((m >> 3) & 1) + 2 * t + ((m >> 2) & 1)
                assert int(vm[32 * t + m]) == int(vmm[32 * g + tok, m & 3, 0]) | (int(vmm[32 * g + tok, m & 3, 1]) << 16)


@pytest.mark.parametrize("bits", [1, 2])
def test_pack_follows_the_documented_index_rule_g64(bits):
    """The same for g = 64, whose records hold a 64-token group each with its
    metadata once: both halves' code planes by the 32-token word rule, the keys'
    (min, max) over 64 tokens, two value (min, max) words per token (channels
    0..63 and 64..127), 48 (1 bit) or 80 (2 bits) bytes per token."""
    B, Hkv, N = 1, 1, 128
    d = oracle.dims(B=B, Hq=1, Hkv=Hkv, N=N, R=0, bits=bits, group=64)
    K, V = synth.kv_layer(23, 0, B, Hkv, N)
    qz = oracle.quantize(d, K, V)
    rec, _ = oracle.pack(d, qz, K, V)
    assert rec.shape[2] == N // 64 and rec.shape[3] == 64 * (48 if bits == 1 else 80)
    kcode, vcode, kmm, vmm = qz["kcode"][0, 0], qz["vcode"][0, 0], qz["kmm"][0, 0], qz["vmm"][0, 0]
    for u in range(N // 64):
        w = np.frombuffer(rec[0, 0, u].tobytes(), dtype="<u4")
        P = 128 * bits  # words of one half's code planes
        km = w[2 * P:2 * P + 128]
        vm = w[2 * P + 128 + 2 * P:]
        for hf in range(2):
            kc = w[hf * P:(hf + 1) * P]
            vc = w[2 * P + 128 + hf * P:2 * P + 128 + (hf + 1) * P]
            for p in range(bits):
                code_word_rule(p, kc, vc, kcode, vcode, 64 * u + 32 * hf)
            for m in range(32):
                tok = 64 * u + 32 * hf + 16 * ((m >> 2) & 1) + 8 * ((m >> 1) & 1) + 2 * (m >> 3) + (m & 1)
                for c in range(2):
                    assert int(vm[64 * hf + 2 * m + c]) == int(vmm[tok, c, 0]) | (int(vmm[tok, c, 1]) << 16)
        for t in range(4):
            for m in range(32):
                ch = 16 * (m >> 2) + 2 * t + 8 * ((m >> 1) & 1) + (m & 1)
                assert int(km[32 * t + m]) == int(kmm[u, ch, 0]) | (int(kmm[u, ch, 1]) << 16)


@pytest.mark.parametrize("bits,R,N0,T,group", [(1, 8, 30, 45, 32), (2, 8, 71, 40, 32), (1, 0, 0, 70, 32),
                                               (2, 128, 100, 70, 32), (1, 16, 40, 90, 64), (2, 0, 10, 60, 64)])
def test_append_one_token_at_a_time_equals_quantising_the_sequence(bits, R, N0, T, group):
    """Decode-time append (SpeCache section 3, Algorithm 3): after tokens
    N0 .. N0+T-1 join one by one, the packed cache must be the one that
    quantising all N0+T tokens at once gives (group boundaries and codes
    depend only on the tokens), and the host cache must hold every row.  The
    runs cross at least one flush; R = 0 flushes the group the new row
    completes."""
    B, Hkv, D = 2, 2, 128
    N1 = N0 + T
    K, V = synth.kv_layer(11, bits, B, Hkv, N1, D)
    cap = N1 // 32 + 2
    rcap = R + group
    d = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=N0, R=R, bits=bits, group=group)
    qz = oracle.quantize(d, K[:, :, :N0], V[:, :, :N0])
    rec, res = oracle.pack(d, qz, K[:, :, :N0], V[:, :, :N0], q_groups_cap=cap, resid_cap=rcap)
    host = np.zeros((B, Hkv, N1 + 3, 2, D), np.uint16)
    host[:, :, :N0] = np.stack([K[:, :, :N0], V[:, :, :N0]], axis=3)
    flushes = 0
    for n in range(N0, N1):
        before = oracle.nq(d)
        oracle.append(d, rec, res, K[:, :, n], V[:, :, n], host)
        d.N += 1
        flushes += oracle.nq(d) > before
    assert flushes >= 1
    d1 = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=N1, R=R, bits=bits, group=group)
    nq1 = oracle.nq(d1)
    rec1, res1 = oracle.pack(d1, oracle.quantize(d1, K, V), K, V, q_groups_cap=cap, resid_cap=rcap)
    assert np.array_equal(rec[:, :, :nq1 // group], rec1[:, :, :nq1 // group])
    assert np.array_equal(res[:, :, :N1 - nq1], res1[:, :, :N1 - nq1])
    assert np.array_equal(host[:, :, :N1], np.stack([K, V], axis=3))
    assert not host[:, :, N1:].any()


@pytest.mark.parametrize("bits", [1, 2])
def test_g64_equals_g32_when_both_halves_of_every_group_span_the_same_range(bits):
    """A 64-token key group whose two 32-token halves have the same per-channel
    (min, max), and a 64-channel value group whose two halves share theirs,
    quantise exactly as with g = 32 (a code depends only on the value and its
    group's min and max): the codes must coincide and each 64-group's (min, max)
    must be both of its 32-groups'."""
    B, Hkv, N, D = 1, 2, 256, 128
    K, V = synth.kv_layer(13, bits, B, Hkv, N, D)
    rng = np.random.default_rng(5)
    for g in range(N // 64):  # second half of each 64-token block: a permutation of the first
        perm = rng.permutation(32)
        K[:, :, 64 * g + 32:64 * g + 64] = K[:, :, 64 * g + perm]
    for c0 in (0, 64):  # channels c0+32..c0+63: a permutation of c0..c0+31, per token
        perm = rng.permutation(32)
        V[..., c0 + 32:c0 + 64] = V[..., c0 + perm]
    qz = {}
    for group in (32, 64):
        d = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=N, R=0, bits=bits, group=group)
        qz[group] = oracle.quantize(d, K, V)
    assert np.array_equal(qz[32]["kcode"], qz[64]["kcode"]) and np.array_equal(qz[32]["vcode"], qz[64]["vcode"])
    assert np.array_equal(qz[32]["kmm"][:, :, 0::2], qz[64]["kmm"])
    assert np.array_equal(qz[32]["kmm"][:, :, 1::2], qz[64]["kmm"])
    assert np.array_equal(qz[32]["vmm"][:, :, :, 0::2], qz[64]["vmm"])
    assert np.array_equal(qz[32]["vmm"][:, :, :, 1::2], qz[64]["vmm"])
    # and an ordinary input does differ (the pin is not vacuous)
    K2, V2 = synth.kv_layer(13, bits, B, Hkv, N, D)
    out = []
    for group in (32, 64):
        d = oracle.dims(B=B, Hq=Hkv, Hkv=Hkv, N=N, R=0, bits=bits, group=group)
        out.append(oracle.quantize(d, K2, V2)["kcode"])
    assert not np.array_equal(out[0], out[1])


def test_binary32_edge_readings():
    """Groups at the edges of binary32, worked by hand from IEEE-754 rules:
    subnormal ranges quantise like any other; 3 min + max overflowing makes
    z = +inf (every code 0) or -inf (every code the top code); max - min
    overflowing makes s = +inf, so a finite x - z gives the quotient 0 and an
    infinite one no number, which takes code 0 (the reading for a quotient
    that is not a number)."""
    big = float(b2f(0x7F7F))          # largest finite bf16
    big1 = float(b2f(0x7F7E))         # the next one down
    sub = float(b2f(0x0001))          # smallest bf16 subnormal, 2^-133
    # lo = 0, hi = 2^-133: s = 2^-134, z = 2^-135; quotients -1/2 and 3/2
    codes, _, lo, hi = quantize_key_group(1, [0.0, sub, 0.0, sub])
    assert (lo, hi) == (0.0, sub) and list(codes) == [0, 1, 0, 1]
    # 2-bit on {0, 2^-133 .. 3 * 2^-133}: s = 2^-133 exactly, codes are the multiples
    codes, _, _, _ = quantize_key_group(2, [0.0, sub, 2 * sub, 3 * sub])
    assert list(codes) == [0, 1, 2, 3]
    for bits in (1, 2):
        codes, _, _, _ = quantize_key_group(bits, [big, big1, big])
        top = 0 if bits == 1 else 3  # 2-bit: z = min, nothing overflows, max gets the top code
        assert list(codes) == [top, 0, top]
    codes, _, _, _ = quantize_key_group(1, [-big, -big1, -big])  # z = -inf: x - z = +inf
    assert list(codes) == [1, 1, 1]
    codes, _, _, _ = quantize_key_group(1, [-big, big, -big1])    # z = -inf, s = +inf: inf / inf
    assert list(codes) == [0, 0, 0]
    codes, _, _, _ = quantize_key_group(2, [-big, big, 0.0])      # s = +inf: 0, inf / inf, finite / inf
    assert list(codes) == [0, 0, 0]
    codes, _, _, _ = quantize_key_group(1, [-float(b2f(0x7E80)), big, 1.0])  # z finite, s = +inf
    assert list(codes) == [0, 0, 0]
