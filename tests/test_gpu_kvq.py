"""Parity of the decode attention over bf16 and fp8 E4M3 KV caches
(ck_attn_decode_gqa_bf16 / _fp8) and of the matching KV stores
(ck_kv_store_bf16 / _fp8) with the oracle.

Bit-exact: the codes the stores write.  Floating point (the attention
output, over caches encoded by the oracle): max |err| <= 1e-3 * max |ref|
and relative L2 error <= 1e-4.  Cases span one row, ragged tails, every query
group size, both stage heights and long splits."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
import quantized_weight_attention_gb300 as q  # noqa: E402

pytestmark = pytest.mark.gpu


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref).max() if got.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert err <= 1e-3 * scale and rel <= 1e-4, f"{what}: max|err| {err:.3e} > {1e-3 * scale:.3e} or relL2 {rel:.3e}"


@pytest.fixture(scope="module")
def dev(cuda_ok):
    from quantized_weight_attention_gb300 import build as kb
    kb.build()
    q.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def T(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def H(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def ok(rc):
    assert rc == q.CK_OK, q.ck_status_string(rc)


def encode(kind, x, scale):
    return oracle.bf16_from_f32(x) if kind == oracle.KV_BF16 else oracle.e4m3_from_f32(x, scale)


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
def test_kv_store_codes_bit_exact(dev, kind):
    rng = np.random.default_rng(30 + kind)
    KV, C, hd, pos = 4, 9, 128, 5
    n = KV * hd
    k = (rng.standard_normal(n) * rng.choice([1e-4, 1.0, 30.0, 1e3], n)).astype(np.float32)
    v = (rng.standard_normal(n) * rng.choice([1e-4, 1.0, 30.0, 1e3], n)).astype(np.float32)
    ks, vs = 0.05, 0.02
    if kind == oracle.KV_BF16:
        k[:4] = [1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 2.0**-8), np.finfo(np.float32).max]  # ties, overflow
    else:
        k[:6] = np.array([1.0625, 1.1875, 2.0**-10, 3 * 2.0**-10, 1e6, -1e6], np.float32) * np.float32(ks)
    dt = np.uint16 if kind == oracle.KV_BF16 else np.uint8
    kc0 = rng.integers(0, 120, (KV, C, hd)).astype(dt)
    vc0 = rng.integers(0, 120, (KV, C, hd)).astype(dt)
    kc, vc = T(kc0, dev), T(vc0, dev)
    if kind == oracle.KV_BF16:
        ok(q.ck_kv_store_bf16(kc, vc, T(k, dev), T(v, dev), pos, KV, C, hd))
    else:
        ok(q.ck_kv_store_fp8(kc, vc, T(k, dev), T(v, dev), pos, KV, C, hd, ks, vs))
    rk, rv = kc0.copy(), vc0.copy()
    oracle.kv_store_kvq(rk, rv, k, v, pos, KV, C, hd, kind, ks, vs)
    assert np.array_equal(H(kc), rk) and np.array_equal(H(vc), rv)


# (head_dim, H, KV, rows attended, capacity)
CASES = [
    (64, 8, 8, 1, 16),          # one row, MHA
    (64, 8, 2, 37, 64),         # ragged tail of one short split
    (128, 12, 4, 300, 320),     # G = 3 (run masked in the G = 4 kernel)
    (128, 28, 4, 1025, 1088),   # G = 7
    (128, 32, 4, 8193, 8256),   # G = 8, the 8K length
    (64, 16, 2, 20011, 20016),  # long splits of a head_dim 64 cache
    (128, 28, 4, 32769, 32832), # 32K rows: large stages
    (128, 4, 4, 129, 192),      # G = 1: a full 128-row tile and a one-row tile
    (128, 8, 4, 257, 320),      # G = 2: three tiles, the two row groups unevenly loaded
    (128, 16, 2, 128, 128),     # G = 8: exactly one tile, the cache full
]


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
@pytest.mark.parametrize("hd,Hq,KV,Tn,C", CASES)
def test_attention_kvq_matches_oracle(dev, kind, hd, Hq, KV, Tn, C):
    rng = np.random.default_rng(1000 * hd + Tn + 7 * kind)
    qv = rng.standard_normal(Hq * hd).astype(np.float32)
    k = rng.standard_normal((KV, C, hd)).astype(np.float32)
    v = rng.standard_normal((KV, C, hd)).astype(np.float32)
    ks = float(np.abs(k).max() / 448.0 * 1.01)
    vs = float(np.abs(v).max() / 448.0 * 1.01)
    kc, vc = encode(kind, k, ks), encode(kind, v, vs)
    # rows past the attended ones hold NaN codes: they must never be read
    nan = 0x7FC0 if kind == oracle.KV_BF16 else 0x7F
    kc[:, Tn:] = nan
    vc[:, Tn:] = nan
    ref = oracle.attention_kvq(qv, kc, vc, Hq, KV, Tn, C, hd, kind, ks, vs)
    nbytes = q.ck_attn_scratch_size(Hq, KV, C, hd)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(Hq * hd, dtype=torch.float32, device=dev)
    if kind == oracle.KV_BF16:
        ok(q.ck_attn_decode_gqa_bf16(T(qv, dev), T(kc, dev), T(vc, dev), out, Hq, KV, Tn, C, hd, scratch, nbytes))
    else:
        ok(q.ck_attn_decode_gqa_fp8(T(qv, dev), T(kc, dev), T(vc, dev), out, Hq, KV, Tn, C, hd, ks, vs, scratch,
                                    nbytes))
    assert_close(H(out), ref, f"kind {kind} hd {hd} H {Hq} KV {KV} T {Tn}")
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0


def test_attention_kvq_rejects_bad_arguments(dev):
    x = torch.zeros(4096, dtype=torch.float32, device=dev)
    c = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    nb = q.ck_attn_scratch_size(8, 2, 64, 64)
    s = torch.empty(nb, dtype=torch.uint8, device=dev)
    assert q.ck_attn_decode_gqa_fp8(x, c, c, x, 8, 2, 16, 64, 64, 0.0, 1.0, s, nb) == q.CK_EINVAL
    assert q.ck_attn_decode_gqa_fp8(x, c, c, x, 8, 2, 16, 64, 64, 1.0, float("nan"), s, nb) == q.CK_EINVAL
    assert q.ck_attn_decode_gqa_bf16(x, c, c, x, 8, 2, 16, 64, 96, s, nb) == q.CK_EINVAL
    assert q.ck_attn_decode_gqa_bf16(x, c, c, x, 8, 2, 65, 64, 64, s, nb) == q.CK_ERANGE
    assert q.ck_kv_store_fp8(c, c, x, x, 3, 2, 16, 64, -1.0, 1.0) == q.CK_EINVAL
    assert q.ck_kv_store_bf16(c, c, x, x, 16, 2, 16, 64) == q.CK_ERANGE
