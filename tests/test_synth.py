"""The seeded input generator: published SplitMix64 values and the bf16 normal draw."""
import numpy as np
from scipy import stats

import synth


def test_splitmix64_reference_outputs():
    # first outputs of SplitMix64 from state 0 (Vigna's splitmix64.c)
    got = [int(x) for x in synth.uniform_u64(np.uint64(0), 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_table_is_monotone_and_trimmed():
    assert np.all(np.diff(synth.THRESH.astype(np.float64)) >= 0)
    assert len(synth.VALS) == len(synth.THRESH) + 1
    v = synth.bf16_to_f32(synth.VALS)
    assert np.all(np.diff(v) > 0) and v[0] > 0


def test_normal_draw_matches_standard_normal():
    x = synth.bf16_to_f32(synth.normal_bf16(synth.stream_key(0, 99), 0, 1 << 21)).astype(np.float64)
    n = len(x)
    for a in (0.25, 1.0, 2.0, 3.0):
        p = stats.norm.cdf(a) - stats.norm.cdf(-a)
        emp = np.mean(np.abs(x) < a)
        assert abs(emp - p) < 5 * np.sqrt(p * (1 - p) / n)
    assert abs(x.mean()) < 5 / np.sqrt(n)
    assert abs(x.std() - 1) < 5e-3
    # every draw is a bf16 value already (rounding happened in the table)
    xf = x.astype(np.float32)
    assert np.array_equal(synth.bf16_to_f32(synth.f32_to_bf16_rne(xf)), xf)


def test_slices_are_consistent_with_full_layer():
    B, Hkv, N = 2, 3, 96
    K, V = synth.kv_layer(0, 4, B, Hkv, N)
    k, v = synth.kv_slice(0, 4, B, Hkv, N, 128, 1, 2, 40, 70)
    assert np.array_equal(K[1, 2, 40:70], k) and np.array_equal(V[1, 2, 40:70], v)


def test_outliers_and_spec_query():
    B, Hkv, N = 1, 8, 64
    K, _ = synth.kv_layer(0, 0, B, Hkv, N)
    ch = synth.outlier_channels(0, 0, Hkv)
    assert all(len(set(c)) == 4 for c in ch)
    kf = np.abs(synth.bf16_to_f32(K)).mean(axis=2)  # [B,Hkv,D]
    for h in range(Hkv):
        big = kf[0, h, ch[h]].mean()
        rest = np.delete(kf[0, h], ch[h]).mean()
        assert 5 < big / rest < 12
    q = synth.queries(0, 0, 2, 32)
    d = synth.bf16_to_f32(q[:, 1]).astype(np.float64) - synth.bf16_to_f32(q[:, 0])
    assert 0.08 < d.std() < 0.12
