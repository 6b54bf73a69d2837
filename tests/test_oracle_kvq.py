"""Pins of the oracle's reduced-precision KV-cache functions (bf16 and fp8
E4M3 caches, the latter with per-tensor k_scale / v_scale, as in the
launchers paged_decode_attn_bf16 / paged_decode_attn_fp8 of the page
"prefill_attn_a.rs", layers/ops).  The element formats are pinned to values their
definitions fix: E4M3 has 1 sign bit, 4 exponent bits with bias 7 and 3
fraction bits, subnormals at exponent field 0 (frac * 2^-9), NaN at
S.1111.111, no infinity and a largest finite magnitude of 448; bfloat16 is
the upper half of a binary32.  The attention over such caches is pinned to
the fp32 attention oracle on the exactly dequantized cache and to the
one-row case."""
import numpy as np
import pytest

import oracle


def test_e4m3_decode_fixed_points():
    codes = np.array([0x00, 0x01, 0x07, 0x08, 0x09, 0x38, 0x3C, 0x3F, 0x40, 0x77, 0x7E, 0x80, 0xB8, 0xFE], np.uint8)
    want = [0.0, 2.0**-9, 7 * 2.0**-9, 2.0**-6, 1.125 * 2.0**-6, 1.0, 1.5, 1.875, 2.0, 1.875 * 2.0**7, 448.0, -0.0,
            -1.0, -448.0]
    got = oracle.e4m3_to_f32(codes)
    assert np.array_equal(got, np.array(want, np.float32))
    assert np.signbit(got[11])
    assert np.isnan(oracle.e4m3_to_f32(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_is_monotone_and_complete():
    v = oracle.e4m3_to_f32(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)  # 0x00 .. 0x7E strictly increasing
    assert v[0] == 0.0 and v[-1] == 448.0
    # negative codes mirror the positive ones
    neg = oracle.e4m3_to_f32(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)


def test_e4m3_encode_round_trip_ties_and_saturation():
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_from_f32(oracle.e4m3_to_f32(finite)), finite)
    x = np.array([1.0625, 1.1875, 2.0**-10, 3 * 2.0**-10, 1000.0, -1e30, 460.0, 432.0, -432.0, 1.06250006],
                 np.float32)
    # ties go to the even code: 1.0625 between 1 (0x38) and 1.125 (0x39) -> 0x38;
    # 1.1875 between 0x39 and 1.25 (0x3A) -> 0x3A; 2^-10 between 0 and 0x01 -> 0;
    # 3*2^-10 between 0x01 and 0x02 -> 0x02; 432 between 416 (0x7D) and 448 -> 0x7E;
    # magnitudes beyond 448 saturate; just above a tie rounds up
    want = [0x38, 0x3A, 0x00, 0x02, 0x7E, 0xFE, 0x7E, 0x7E, 0xFE, 0x39]
    assert list(oracle.e4m3_from_f32(x)) == want
    assert oracle.e4m3_from_f32(np.array([np.nan], np.float32))[0] == 0x7F


def test_e4m3_encode_divides_by_the_scale():
    x = np.array([0.5, -0.75, 4.48, 10.0], np.float32)
    s = np.float32(0.01)
    codes = oracle.e4m3_from_f32(x, float(s))
    assert np.array_equal(codes, oracle.e4m3_from_f32(x / s))
    assert codes[3] == 0x7E  # 1000 saturates


def test_e4m3_encode_is_nearest():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1.0, 100.0], 20000)).astype(np.float32)
    x = x[np.abs(x) < 448]
    c = oracle.e4m3_from_f32(x)
    v = oracle.e4m3_to_f32(c).astype(np.float64)
    grid = oracle.e4m3_to_f32(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    best = np.min(np.abs(np.abs(x.astype(np.float64))[:, None] - grid[None, :]), axis=1)
    assert np.array_equal(np.abs(v - x), best)


def test_bf16_round_to_nearest_even():
    big = np.finfo(np.float32).max  # 0x7F7FFFFF: above bf16's largest finite value -> infinity
    x = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, 1 + 2.0**-8 + 2.0**-20, -1.5, big, 3.0e38, 0.0], np.float32)
    assert list(oracle.bf16_from_f32(x)) == [0x3F80, 0x3F82, 0x3F81, 0xBFC0, 0x7F80, 0x7F62, 0x0000]
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(b)
    keep = ~np.isnan(f)
    assert np.array_equal(oracle.bf16_from_f32(f[keep]), b[keep])


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
def test_attention_kvq_equals_fp32_oracle_on_dequantized_cache(kind):
    rng = np.random.default_rng(11 + kind)
    H, KV, hd, C, T = 8, 2, 64, 40, 37
    q = rng.standard_normal(H * hd).astype(np.float32)
    k = rng.standard_normal((KV, C, hd)).astype(np.float32)
    v = rng.standard_normal((KV, C, hd)).astype(np.float32)
    if kind == oracle.KV_BF16:
        kc, vc = oracle.bf16_from_f32(k), oracle.bf16_from_f32(v)
        kd, vd = oracle.bf16_to_f32(kc), oracle.bf16_to_f32(vc)
        ks = vs = 1.0
    else:
        ks, vs = 2.0**-6, 2.0**-5  # powers of two: code * scale is exact in fp32
        kc, vc = oracle.e4m3_from_f32(k, ks), oracle.e4m3_from_f32(v, vs)
        kd, vd = oracle.e4m3_to_f32(kc) * np.float32(ks), oracle.e4m3_to_f32(vc) * np.float32(vs)
    got = oracle.attention_kvq(q, kc, vc, H, KV, T, C, hd, kind, ks, vs)
    want = oracle.attention(q, kd, vd, H, KV, T, C, hd)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
def test_attention_kvq_one_row_returns_the_value_row(kind):
    rng = np.random.default_rng(3)
    H, KV, hd, C = 4, 2, 64, 8
    q = rng.standard_normal(H * hd).astype(np.float32)
    if kind == oracle.KV_BF16:
        kc = oracle.bf16_from_f32(rng.standard_normal((KV, C, hd)).astype(np.float32))
        vc = oracle.bf16_from_f32(rng.standard_normal((KV, C, hd)).astype(np.float32))
        row = oracle.bf16_to_f32(vc[:, 0])
        vs = 1.0
    else:
        kc = rng.integers(0, 0x7E, (KV, C, hd)).astype(np.uint8)
        vc = rng.integers(0, 0x7E, (KV, C, hd)).astype(np.uint8)
        vs = 0.37
        row = (oracle.e4m3_to_f32(vc[:, 0]).astype(np.float64) * np.float64(np.float32(vs))).astype(np.float32)
    out = oracle.attention_kvq(q, kc, vc, H, KV, 1, C, hd, kind, 0.5, vs).reshape(H, hd)
    for h in range(H):
        assert np.array_equal(out[h], row[h * KV // H])


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
def test_kv_store_kvq_writes_only_row_pos(kind):
    rng = np.random.default_rng(4)
    KV, C, hd, pos = 2, 6, 64, 3
    dt = np.uint16 if kind == oracle.KV_BF16 else np.uint8
    kc = rng.integers(0, 100, (KV, C, hd)).astype(dt)
    vc = kc.copy()
    k0, v0 = kc.copy(), vc.copy()
    k = rng.standard_normal(KV * hd).astype(np.float32)
    v = rng.standard_normal(KV * hd).astype(np.float32)
    oracle.kv_store_kvq(kc, vc, k, v, pos, KV, C, hd, kind, 0.01, 0.02)
    enc = (lambda x, s: oracle.bf16_from_f32(x)) if kind == oracle.KV_BF16 else oracle.e4m3_from_f32
    assert np.array_equal(kc[:, pos].ravel(), enc(k, 0.01)) and np.array_equal(vc[:, pos].ravel(), enc(v, 0.02))
    rest = [t for t in range(C) if t != pos]
    assert np.array_equal(kc[:, rest], k0[:, rest]) and np.array_equal(vc[:, rest], v0[:, rest])


def _pool_from_contiguous(cache, block_size, perm):
    """cache [KV, C, hd] -> pool [num_blocks, KV, block_size, hd] with logical block i at physical perm[i]."""
    KV, C, hd = cache.shape
    nb = C // block_size
    pool = np.zeros((len(perm), KV, block_size, hd), cache.dtype)
    for i in range(nb):
        pool[perm[i]] = cache[:, i * block_size:(i + 1) * block_size].transpose(0, 1, 2)
    return pool


def test_paged_attention_with_identity_table_equals_contiguous():
    rng = np.random.default_rng(21)
    H, KV, hd, bs, nb = 8, 2, 64, 16, 6
    C = bs * nb
    q = rng.standard_normal(H * hd).astype(np.float32)
    k = rng.standard_normal((KV, C, hd)).astype(np.float32)
    v = rng.standard_normal((KV, C, hd)).astype(np.float32)
    perm = np.arange(nb)
    kp, vp = _pool_from_contiguous(k, bs, perm), _pool_from_contiguous(v, bs, perm)
    for T in (1, 15, 16, 17, 90, 96):
        got = oracle.attention_paged(q, kp, vp, perm[None, :], [T], 1, H, KV, hd, bs, nb, 0)
        assert np.array_equal(got, oracle.attention(q, k, v, H, KV, T, C, hd)), T


def test_paged_attention_is_invariant_to_block_placement():
    rng = np.random.default_rng(22)
    H, KV, hd, bs, nb = 4, 2, 64, 32, 5
    C = bs * nb
    q = rng.standard_normal(2 * H * hd).astype(np.float32)
    k = rng.standard_normal((KV, C, hd)).astype(np.float32)
    v = rng.standard_normal((KV, C, hd)).astype(np.float32)
    ident = np.arange(nb)
    perm = rng.permutation(2 * nb)[:nb]  # a pool twice as large, blocks scattered
    kp1, vp1 = _pool_from_contiguous(k, bs, ident), _pool_from_contiguous(v, bs, ident)
    kp2 = np.zeros((2 * nb, KV, bs, hd), np.float32)
    vp2 = np.zeros_like(kp2)
    kp2[perm], vp2[perm] = kp1, vp1
    lens = [150, 37]
    t1 = np.stack([ident, ident]).astype(np.int32)
    t2 = np.stack([perm, perm]).astype(np.int32)
    a = oracle.attention_paged(q, kp1, vp1, t1, lens, 2, H, KV, hd, bs, nb, 0)
    b = oracle.attention_paged(q, kp2, vp2, t2, lens, 2, H, KV, hd, bs, nb, 0)
    assert np.array_equal(a, b)


def test_paged_attention_window_equals_attention_over_the_last_rows():
    rng = np.random.default_rng(23)
    H, KV, hd, bs, nb = 4, 1, 64, 16, 8
    C = bs * nb
    q = rng.standard_normal(H * hd).astype(np.float32)
    k = rng.standard_normal((KV, C, hd)).astype(np.float32)
    v = rng.standard_normal((KV, C, hd)).astype(np.float32)
    perm = np.arange(nb)
    kp, vp = _pool_from_contiguous(k, bs, perm), _pool_from_contiguous(v, bs, perm)
    T = 100
    for W in (1, 7, 33, 99, 100, 500):
        got = oracle.attention_paged(q, kp, vp, perm[None, :], [T], 1, H, KV, hd, bs, nb, W)
        lo = max(0, T - W)
        want = oracle.attention(q, np.ascontiguousarray(k[:, lo:T]), np.ascontiguousarray(v[:, lo:T]), H, KV, T - lo,
                                T - lo, hd)
        assert np.array_equal(got, want), W
