"""Pins of the oracle to facts outside itself (no GPU).

Each test checks an oracle function against something the format definition,
the mathematics or an independent library fixes: exhaustive or structured
comparison with numpy's IEEE binary16 conversion, hand-built blocks whose
weights follow from the field layout by hand, closed forms, invariants, and
brute force over exact integers.  A plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a missing scale) fails at
least one of them.
"""
import math

import numpy as np
import pytest

import oracle
from quantized_weight_attention_gb300 import synth


# --------------------------------------------------------------------------
# fp16 codec vs numpy's binary16 (an independent IEEE implementation)
# --------------------------------------------------------------------------
def test_f16_to_f32_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32_array(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_f32_to_f16_structured_and_random():
    # every sign/exponent, every upper-10-bit fraction, and low-13-bit
    # fractions at and around the round-to-nearest-even tie
    se = np.arange(512, dtype=np.uint32) << np.uint32(23)
    hi = np.arange(1024, dtype=np.uint32) << np.uint32(13)
    lo = np.array([0, 1, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x0800, 0x17FF], np.uint32)
    bits = (se[:, None, None] | hi[None, :, None] | lo[None, None, :]).ravel()
    rng = np.random.default_rng(1234)
    bits = np.concatenate([bits, rng.integers(0, 2**32, 1 << 20, dtype=np.uint64).astype(np.uint32)])
    x = bits.view(np.float32)
    got = oracle.f32_to_f16_array(x)
    with np.errstate(over="ignore", invalid="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


def test_f32_to_f16_hand_cases():
    assert oracle.f32_to_f16(1.0) == 0x3C00
    assert oracle.f32_to_f16(-2.0) == 0xC000
    assert oracle.f32_to_f16(65504.0) == 0x7BFF
    assert oracle.f32_to_f16(65519.99) == 0x7BFF
    assert oracle.f32_to_f16(65520.0) == 0x7C00          # tie rounds to even -> inf
    assert oracle.f32_to_f16(2.0 ** -24) == 0x0001        # smallest subnormal
    assert oracle.f32_to_f16(2.0 ** -25) == 0x0000        # tie to even -> 0
    assert oracle.f32_to_f16(1.5 * 2.0 ** -25) == 0x0001
    assert oracle.f32_to_f16(1.0 + 2.0 ** -11) == 0x3C00  # tie, even stays
    assert oracle.f32_to_f16(1.0 + 3 * 2.0 ** -11) == 0x3C02


# --------------------------------------------------------------------------
# Block codecs on hand-built bytes (expected weights worked out by hand from
# the field layout: d fp16 LE at byte 0, qh u32 LE at 2, qs at 6)
# --------------------------------------------------------------------------
def _q5(d16, qh, qs):
    b = np.zeros(22, np.uint8)
    b[0], b[1] = d16 & 0xFF, d16 >> 8
    for i in range(4):
        b[2 + i] = (qh >> (8 * i)) & 0xFF
    b[6:22] = qs
    return b


def test_q5_0_hand_blocks():
    one = 0x3C00
    w = oracle.dequant_q5_0(_q5(one, 0, np.zeros(16, np.uint8)))[0]
    assert np.all(w == -16.0)
    w = oracle.dequant_q5_0(_q5(one, 0xFFFFFFFF, np.full(16, 0xFF, np.uint8)))[0]
    assert np.all(w == 15.0)
    for j in range(16):
        qs = np.zeros(16, np.uint8)
        qs[j] = 0x0F
        w = oracle.dequant_q5_0(_q5(one, 0, qs))[0]
        want = np.full(32, -16.0, np.float32)
        want[j] = -1.0
        assert np.array_equal(w, want), j
        qs[j] = 0xF0
        w = oracle.dequant_q5_0(_q5(one, 0, qs))[0]
        want = np.full(32, -16.0, np.float32)
        want[j + 16] = -1.0
        assert np.array_equal(w, want), j
    for k in range(32):
        w = oracle.dequant_q5_0(_q5(one, 1 << k, np.zeros(16, np.uint8)))[0]
        want = np.full(32, -16.0, np.float32)
        want[k] = 0.0
        assert np.array_equal(w, want), k
    # d = -2.0 (0xC000): code 3 in element 5 (low nibble 3, qh bit clear) -> (3-16)*-2 = 26
    qs = np.zeros(16, np.uint8)
    qs[5] = 0x03
    w = oracle.dequant_q5_0(_q5(0xC000, 0xFFFFFFFF & ~(1 << 5), qs))[0]
    want = np.full(32, 0.0, np.float32)  # other elements: code 16 -> 0
    want[5] = 26.0
    assert np.array_equal(w, want)


def test_q8_0_hand_blocks():
    b = np.zeros(34, np.uint8)
    b[0], b[1] = 0x00, 0x38  # 0x3800 = 0.5
    b[2:] = (np.arange(32) - 16).astype(np.int8).view(np.uint8)
    w = oracle.dequant_q8_0(b)[0]
    assert np.array_equal(w, (np.arange(32) - 16) * 0.5)
    b[2:] = np.array([-128] * 32, np.int8).view(np.uint8)
    assert np.all(oracle.dequant_q8_0(b)[0] == -64.0)


def test_unpack_matches_input_packer():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 32, (64, 32), dtype=np.uint8)
    d16 = rng.integers(0, 0x7C00, 64).astype(np.uint16)
    q, d = oracle.unpack_q5_0(synth.pack_q5_0(codes, d16))
    assert np.array_equal(q, codes.astype(np.int32) - 16)
    assert np.array_equal(d, d16.view(np.float16).astype(np.float32))
    c8 = rng.integers(-128, 128, (64, 32)).astype(np.int8)
    q, d = oracle.unpack_q8_0(synth.pack_q8_0(c8, d16))
    assert np.array_equal(q, c8.astype(np.int32))


def test_golden_q5_0_fixture():
    """tests/golden/q5_0_blocks.txt: hand-derived weights of hand-built blocks."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "q5_0_blocks.txt")
    cases = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        hexbytes, weights = line.split("|")
        blk = np.frombuffer(bytes.fromhex(hexbytes.strip()), np.uint8)
        want = np.array([float(v) for v in weights.split()], np.float32)
        got = oracle.dequant_q5_0(blk)[0]
        assert np.array_equal(got, want), line
        cases += 1
    assert cases >= 4


# --------------------------------------------------------------------------
# Q8_0 activation quantizer
# --------------------------------------------------------------------------
def _q8_fields(y):
    y = y.reshape(-1, 34)
    d16 = y[:, 0].astype(np.uint16) | (y[:, 1].astype(np.uint16) << 8)
    return d16, y[:, 2:].view(np.int8).astype(np.int32)


def test_q8_0_ties_round_half_away():
    x = np.zeros(32, np.float32)
    x[0] = 127.0                    # amax = 127 -> d = 1, 1/d = 1 exactly
    x[1:7] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5]
    d16, q = _q8_fields(oracle.quantize_q8_0(x))
    assert d16[0] == 0x3C00
    assert list(q[0, :7]) == [127, 3, -3, 1, -1, 2, -2]


def test_q8_0_zero_block_and_extremes():
    x = np.zeros(64, np.float32)
    x[32:] = np.linspace(-3, 7, 32, dtype=np.float32)
    d16, q = _q8_fields(oracle.quantize_q8_0(x))
    assert d16[0] == 0 and np.all(q[0] == 0)
    assert q[1, np.argmax(np.abs(x[32:]))] == 127
    x[32 + 5] = -9.0
    d16, q = _q8_fields(oracle.quantize_q8_0(x))
    assert q[1, 5] == -127


def test_q8_0_scale_and_rounding_bound():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(32 * 500) * rng.uniform(1e-3, 1e3, 500).repeat(32)).astype(np.float32)
    d16, q = _q8_fields(oracle.quantize_q8_0(x))
    xb = x.reshape(-1, 32)
    d = (np.abs(xb).max(1) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(d16, d.astype(np.float16).view(np.uint16))
    # nearest integer to x/d, up to the fp32 rounding of x * (1/d)
    assert np.all(np.abs(q - xb.astype(np.float64) / d[:, None].astype(np.float64)) <= 0.5 + 1e-5)
    assert np.all(np.abs(q) <= 127)


# --------------------------------------------------------------------------
# Block dots and GEMV against exact integer / float64 arithmetic on codes the
# test itself chose
# --------------------------------------------------------------------------
def _codes_case(rng, M, K, q8):
    nb = K // 32
    if q8:
        cw = rng.integers(-128, 128, (M * nb, 32)).astype(np.int8)
    else:
        cw = rng.integers(0, 32, (M * nb, 32), dtype=np.uint8)
    dw = (rng.uniform(0.5, 1.5, M * nb) * 1e-2).astype(np.float16)
    cx = rng.integers(-127, 128, (nb, 32)).astype(np.int8)
    dx = (rng.uniform(0.5, 1.5, nb) * 1e-1).astype(np.float16)
    W = (synth.pack_q8_0(cw, dw.view(np.uint16)) if q8 else synth.pack_q5_0(cw, dw.view(np.uint16)))
    xq = synth.pack_q8_0(cx, dx.view(np.uint16))
    wint = cw.astype(np.int64) - (0 if q8 else 16)
    return W.ravel(), xq.ravel(), wint.reshape(M, nb, 32), dw.astype(np.float64).reshape(M, nb), \
        cx.astype(np.int64), dx.astype(np.float64)


@pytest.mark.parametrize("q8", [False, True])
def test_block_dots_brute_force(q8):
    rng = np.random.default_rng(11 + q8)
    M, K = 7, 96
    W, xq, wint, _, cx, _ = _codes_case(rng, M, K, q8)
    got = oracle.block_dots(W, xq, M, K, q8)
    want = np.einsum("mbj,bj->mb", wint, cx)
    assert np.array_equal(got, want)
    # extremes: every code at its most negative / positive
    nb = 1
    cw = np.full((1, 32), 0 if not q8 else -128, np.int64)
    Wx = (synth.pack_q8_0(cw.astype(np.int8), [0x3C00]) if q8 else synth.pack_q5_0(cw.astype(np.uint8), [0x3C00]))
    xx = synth.pack_q8_0(np.full((1, 32), -128, np.int8), [0x3C00])
    assert oracle.block_dots(Wx.ravel(), xx.ravel(), 1, 32, q8)[0, 0] == 32 * (-128 if q8 else -16) * -128


@pytest.mark.parametrize("q8", [False, True])
def test_gemv_vs_float64_dequant_matmul(q8):
    rng = np.random.default_rng(21 + q8)
    M, K = 37, 160   # M != K: a transposed operand would not even fit
    W, xq, wint, dw, cx, dx = _codes_case(rng, M, K, q8)
    bias = rng.standard_normal(M).astype(np.float32)
    Wd = (wint * dw[:, :, None]).reshape(M, K)
    xd = (cx * dx[:, None]).reshape(K)
    exact = Wd @ xd
    y = oracle.gemv(W, xq, bias, M, K, q8)
    y0 = oracle.gemv(W, xq, None, M, K, q8)
    assert np.array_equal(y0, exact.astype(np.float32)) or np.allclose(y0, exact, rtol=2e-7, atol=0)
    assert np.allclose(y, (exact.astype(np.float32) + bias), rtol=0, atol=2e-6 * (np.abs(exact) + np.abs(bias)).max())


# --------------------------------------------------------------------------
# RMSNorm closed forms
# --------------------------------------------------------------------------
def test_rmsnorm_constant_vector_closed_form():
    D, c, eps = 256, 0.75, 1e-6
    x = np.full(D, c, np.float32)
    g = np.linspace(0.5, 1.5, D).astype(np.float32)
    y, rstd = oracle.rmsnorm(x, g, eps)
    want_rstd = np.float32(1.0 / math.sqrt(c * c + np.float64(np.float32(eps))))
    assert rstd == want_rstd
    assert np.array_equal(y, (x * want_rstd) * g)


def test_rmsnorm_power_of_two_scale_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(896).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(896)).astype(np.float32)
    y1, r1 = oracle.rmsnorm(x, g, 0.0)
    y2, r2 = oracle.rmsnorm(x * np.float32(8.0), g, 0.0)
    assert r2 == r1 / 8 and np.array_equal(y1, y2)
    # mean over D, not a sum: doubling D with a copy leaves rstd unchanged
    y3, r3 = oracle.rmsnorm(np.concatenate([x, x]), np.concatenate([g, g]), 0.0)
    assert abs(r3 - r1) <= 1e-7 * r1


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------
def test_rope_position_zero_is_identity():
    cos, sin = synth.rope_tables(8, 64, 1e4)
    rng = np.random.default_rng(4)
    q = rng.standard_normal(4 * 64).astype(np.float32)
    k = rng.standard_normal(2 * 64).astype(np.float32)
    q2, k2 = oracle.rope(q, k, cos, sin, 0, 4, 2, 64)
    assert np.array_equal(q, q2) and np.array_equal(k, k2)


def test_rope_pairs_d_with_d_plus_half():
    hd, cap = 8, 2
    cos = np.zeros((cap, hd // 2), np.float32)
    sin = np.ones((cap, hd // 2), np.float32)
    q = np.zeros(hd, np.float32)
    q[0] = 1.0
    q[5] = 2.0
    q2, _ = oracle.rope(q, None, cos, sin, 1, 1, 0, hd)
    # (a, b) -> (a cos - b sin, a sin + b cos) = (-b, a) on pairs (d, d + 4)
    want = np.zeros(hd, np.float32)
    want[4] = 1.0
    want[1] = -2.0
    assert np.array_equal(q2, want)


def test_rope_hd2_closed_form_and_norms():
    phi = 0.3
    cos = np.array([[1.0], [math.cos(phi)]], np.float32)
    sin = np.array([[0.0], [math.sin(phi)]], np.float32)
    q = np.array([0.7, -1.3], np.float32)
    q2, _ = oracle.rope(q, None, cos, sin, 1, 1, 0, 2)
    c, s = np.float32(math.cos(phi)), np.float32(math.sin(phi))
    assert np.allclose(q2, [0.7 * c + 1.3 * s, 0.7 * s - 1.3 * c], rtol=1e-6)
    cos, sin = synth.rope_tables(64, 64, 1e4)
    rng = np.random.default_rng(9)
    q = rng.standard_normal(3 * 64).astype(np.float32)
    q2, _ = oracle.rope(q, None, cos, sin, 37, 3, 0, 64)
    a, b = q.reshape(3, 2, 32), q2.reshape(3, 2, 32)
    assert np.allclose((a ** 2).sum(1), (b ** 2).sum(1), rtol=1e-5)


def test_rope_relative_position():
    cos, sin = synth.rope_tables(128, 64, 1e4)
    rng = np.random.default_rng(10)
    q = rng.standard_normal(64).astype(np.float32)
    k = rng.standard_normal(64).astype(np.float32)
    def rot(v, p):
        return oracle.rope(v, None, cos, sin, p, 1, 0, 64)[0].astype(np.float64)
    assert abs(rot(q, 20) @ rot(k, 20) - q.astype(np.float64) @ k) < 1e-4
    assert abs(rot(q, 30) @ rot(k, 20) - rot(q, 15) @ rot(k, 5)) < 1e-4


# --------------------------------------------------------------------------
# KV store
# --------------------------------------------------------------------------
def test_kv_store_writes_only_row_pos():
    KV, C, hd = 3, 10, 32
    kc = np.zeros((KV, C, hd), np.float32)
    vc = np.zeros((KV, C, hd), np.float32)
    k = np.arange(KV * hd, dtype=np.float32) + 1
    v = -k
    oracle.kv_store(kc, vc, k, v, 6, KV, C, hd)
    assert np.array_equal(kc[:, 6, :], k.reshape(KV, hd))
    assert np.array_equal(vc[:, 6, :], v.reshape(KV, hd))
    kc[:, 6, :] = 0
    vc[:, 6, :] = 0
    assert not kc.any() and not vc.any()


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
def _cache(rng, KV, C, hd, T):
    kc = np.zeros((KV, C, hd), np.float32)
    vc = np.zeros((KV, C, hd), np.float32)
    kc[:, :T] = rng.standard_normal((KV, T, hd))
    vc[:, :T] = rng.standard_normal((KV, T, hd))
    return kc, vc


def test_attention_single_row_returns_v_exactly_and_head_map():
    rng = np.random.default_rng(12)
    H, KV, C, hd = 6, 3, 5, 32
    kc, vc = _cache(rng, KV, C, hd, 1)
    q = rng.standard_normal(H * hd).astype(np.float32)
    o = oracle.attention(q, kc, vc, H, KV, 1, C, hd).reshape(H, hd)
    for h in range(H):
        assert np.array_equal(o[h], vc[h * KV // H, 0]), h   # heads 0,1 -> kv 0; 2,3 -> 1; 4,5 -> 2
    o = oracle.attention(q, kc, vc, 3, 3, 1, C, hd).reshape(3, hd)   # MHA: KV == H
    for h in range(3):
        assert np.array_equal(o[h], vc[h, 0])


def test_attention_constant_keys_give_mean_of_values():
    rng = np.random.default_rng(13)
    H, KV, C, hd, T = 4, 2, 40, 64, 33
    kc, vc = _cache(rng, KV, C, hd, T)
    kc[:, :T] = kc[:, :1]
    q = rng.standard_normal(H * hd).astype(np.float32)
    o = oracle.attention(q, kc, vc, H, KV, T, C, hd).reshape(H, hd)
    for h in range(H):
        assert np.allclose(o[h], vc[h // 2, :T].astype(np.float64).mean(0), rtol=0, atol=1e-6)


def test_attention_two_rows_sigmoid_closed_form():
    hd, C = 64, 4
    a, c = 1.7, 2.3
    q = np.zeros(hd, np.float32)
    q[0] = a
    kc = np.zeros((1, C, hd), np.float32)
    kc[0, 1, 0] = c
    vc = np.zeros((1, C, hd), np.float32)
    rng = np.random.default_rng(14)
    vc[0, :2] = rng.standard_normal((2, hd))
    o = oracle.attention(q, kc, vc, 1, 1, 2, C, hd)
    s1 = np.float32(a) * np.float32(c) / math.sqrt(hd)     # the 1/sqrt(hd) scale
    w1 = 1.0 / (1.0 + math.exp(-s1))
    want = vc[0, 0].astype(np.float64) + w1 * (vc[0, 1].astype(np.float64) - vc[0, 0])
    assert np.allclose(o, want, rtol=0, atol=1e-6)


def test_attention_permutation_and_shift_invariance():
    rng = np.random.default_rng(15)
    H, KV, C, hd, T = 4, 2, 24, 32, 19
    kc, vc = _cache(rng, KV, C, hd, T)
    q = rng.standard_normal(H * hd).astype(np.float32)
    o = oracle.attention(q, kc, vc, H, KV, T, C, hd)
    perm = rng.permutation(T)
    kp, vp = kc.copy(), vc.copy()
    kp[:, :T] = kc[:, perm]
    vp[:, :T] = vc[:, perm]
    assert np.allclose(oracle.attention(q, kp, vp, H, KV, T, C, hd), o, rtol=0, atol=1e-6)
    ks = kc.copy()
    ks[:, :T] += np.float32(0.5)   # same offset for every row -> same score shift
    o2 = oracle.attention(q, ks, vc, H, KV, T, C, hd)
    assert np.allclose(o2, o, rtol=0, atol=1e-5)
    # rows beyond T are never read
    kc2 = kc.copy()
    kc2[:, T:] = 1e30
    assert np.array_equal(oracle.attention(q, kc2, vc, H, KV, T, C, hd), o)


def test_attention_dominant_row():
    hd, C, T = 32, 8, 6
    q = np.zeros(hd, np.float32)
    q[3] = 1.0
    kc = np.zeros((1, C, hd), np.float32)
    kc[0, 4, 3] = 400.0     # score 400/sqrt(32) ~ 70.7 above the rest
    vc = np.random.default_rng(16).standard_normal((1, C, hd)).astype(np.float32)
    o = oracle.attention(q, kc, vc, 1, 1, T, C, hd)
    assert np.allclose(o, vc[0, 4], rtol=0, atol=1e-20 + 1e-6)


# --------------------------------------------------------------------------
# The layer
# --------------------------------------------------------------------------
def _tiny(seed=0):
    w = synth.WORKLOADS["tiny"]
    L = synth.make_layer(w, np.random.Generator(np.random.PCG64(seed)))
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    return w, L, cos, sin


def test_layer_equals_step_by_step_composition():
    w, L, cos, sin = _tiny()
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    out, t = oracle.decode_layer(L.x, L.x, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc,
                                 cos, sin, w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, taps=True)
    # the page's steps, one call each
    xn, _ = oracle.rmsnorm(L.x, L.gamma, w.eps)
    xq = oracle.quantize_q8_0(xn)
    q = oracle.gemv(L.wq, xq, L.bq, w.QD, w.D, False)
    k = oracle.gemv(L.wk, xq, L.bk, w.KD, w.D, False)
    v = oracle.gemv(L.wv, xq, L.bv, w.KD, w.D, True)
    q, k = oracle.rope(q, k, cos, sin, w.pos, w.H, w.KV, w.hd)
    kc2, vc2 = L.k_cache.copy(), L.v_cache.copy()
    oracle.kv_store(kc2, vc2, k, v, w.pos, w.KV, w.capacity, w.hd)
    attn = oracle.attention(q, kc2, vc2, w.H, w.KV, w.pos + 1, w.capacity, w.hd)
    aq = oracle.quantize_q8_0(attn)
    o = oracle.gemv(L.wo, aq, L.bo, w.D, w.QD, False) + L.x
    assert np.array_equal(t["xq"], xq) and np.array_equal(t["q"], q) and np.array_equal(t["k"], k)
    assert np.array_equal(t["v"], v) and np.array_equal(t["attn"], attn) and np.array_equal(t["aq"], aq)
    assert np.array_equal(out, o)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def test_layer_zero_weights_give_residual():
    w, L, cos, sin = _tiny(1)
    z5 = np.zeros_like(L.wq)
    z8 = np.zeros_like(L.wv)
    zo = np.zeros_like(L.wo)
    zb = lambda a: np.zeros_like(a)
    res = np.random.default_rng(2).standard_normal(w.D).astype(np.float32)
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    out = oracle.decode_layer(L.x, res, z5, np.zeros_like(L.wk), z8, zo, L.gamma, zb(L.bq), zb(L.bk), zb(L.bv),
                              zb(L.bo), kc, vc, cos, sin, w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
    assert np.array_equal(out, res)
    assert not kc[:, w.pos].any() and not vc[:, w.pos].any()   # zero k, v stored at pos
    bo = np.full(w.D, 0.25, np.float32)
    out = oracle.decode_layer(L.x, res, z5, np.zeros_like(L.wk), z8, zo, L.gamma, None, None, None, bo,
                              kc, vc, cos, sin, w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
    assert np.array_equal(out, (np.float32(0) + bo) + res)
