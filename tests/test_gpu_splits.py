"""Parity of the decode attention at explicit split counts
(ck_attn_decode_gqa_split) with the oracle.

Every split count must give the oracle's attention within the layer's
tolerance (max |err| <= 1e-3 * max |ref|, relative L2 <= 1e-4): one split,
ragged splits, one split per SM and more splits than rows (empty splits), on
fp32, bf16 and fp8 caches."""
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


def run(dev, qv, kc, vc, H_, KV, rows, C, hd, kind, splits, ks=1.0, vs=1.0):
    nb = (q.ck_attn_split_scratch_size(H_, KV, hd, splits) if splits > 0
          else q.ck_attn_scratch_size(H_, KV, rows, hd))
    assert nb > 0
    sc = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.full((H_ * hd,), float("nan"), dtype=torch.float32, device=dev)
    ok(q.ck_attn_decode_gqa_split(T(qv, dev), kc, vc, out, H_, KV, rows, C, hd, kind, ks, vs, splits, sc, nb))
    return H(out)


@pytest.mark.parametrize("rows", [1025, 8193])
def test_split_counts_fp32(dev, rows):
    """The 7B-shaped heads (28 / 4, hd 128) over 1,025 and 8,193 rows at
    split counts from 1 to 1024 and the built-in choice (0)."""
    H_, KV, hd, C = 28, 4, 128, rows + 7
    rng = np.random.default_rng(rows)
    kc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    vc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    kc0[:, rows:] = np.nan
    vc0[:, rows:] = np.nan
    qv = rng.standard_normal(H_ * hd).astype(np.float32)
    ref = oracle.attention(qv, kc0, vc0, H_, KV, rows, C, hd)
    kc, vc = T(kc0, dev), T(vc0, dev)
    for S in (1, 2, 7, 38, 152, 1024, 0):
        assert_close(run(dev, qv, kc, vc, H_, KV, rows, C, hd, 0, S), ref, f"{rows} rows, {S} splits")


@pytest.mark.parametrize("kind", [oracle.KV_BF16, oracle.KV_FP8])
def test_split_counts_reduced_caches(dev, kind):
    H_, KV, hd, rows, C = 28, 4, 128, 3001, 3008
    rng = np.random.default_rng(40 + kind)
    ks, vs = 0.01, 0.02
    x = rng.standard_normal((2, KV, C, hd)).astype(np.float32)
    if kind == oracle.KV_BF16:
        kc0, vc0 = oracle.bf16_from_f32(x[0]), oracle.bf16_from_f32(x[1])
    else:
        kc0, vc0 = oracle.e4m3_from_f32(x[0], ks), oracle.e4m3_from_f32(x[1], vs)
    qv = rng.standard_normal(H_ * hd).astype(np.float32)
    ref = oracle.attention_kvq(qv, kc0, vc0, H_, KV, rows, C, hd, kind, ks, vs)
    kc, vc = T(kc0, dev), T(vc0, dev)
    for S in (1, 5, 300, 0):
        assert_close(run(dev, qv, kc, vc, H_, KV, rows, C, hd, kind, S, ks, vs), ref, f"kind {kind}, {S} splits")


def test_one_row_many_splits_returns_v0(dev):
    """One attended row over 1024 splits (1023 empty): the output is row 0 of
    V for every head (weight exp(0) / 1)."""
    H_, KV, hd, C = 8, 2, 64, 16
    rng = np.random.default_rng(3)
    kc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    vc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    qv = rng.standard_normal(H_ * hd).astype(np.float32)
    got = run(dev, qv, T(kc0, dev), T(vc0, dev), H_, KV, 1, C, hd, 0, 1024).reshape(H_, hd)
    for h in range(H_):
        np.testing.assert_allclose(got[h], vc0[h // (H_ // KV), 0], rtol=1e-6, atol=0)


def test_split_argument_errors(dev):
    H_, KV, hd, C = 8, 2, 64, 16
    z = torch.zeros((KV, C, hd), dtype=torch.float32, device=dev)
    qv = torch.zeros(H_ * hd, dtype=torch.float32, device=dev)
    out = torch.zeros(H_ * hd, dtype=torch.float32, device=dev)
    nb = q.ck_attn_split_scratch_size(H_, KV, hd, 64)
    sc = torch.empty(nb, dtype=torch.uint8, device=dev)
    call = lambda S, kind=0, bytes_=nb, ks=1.0: q.ck_attn_decode_gqa_split(qv, z, z, out, H_, KV, 8, C, hd, kind, ks,
                                                                            ks, S, sc, bytes_)
    assert call(-1) == q.CK_EINVAL and call(1025) == q.CK_EINVAL
    assert call(64, kind=3) == q.CK_EINVAL
    assert call(64, kind=2, ks=0.0) == q.CK_EINVAL
    assert call(65) == q.CK_ESCRATCH
    assert call(64, bytes_=nb - 257) == q.CK_ESCRATCH
    assert q.ck_attn_split_scratch_size(H_, KV, hd, 0) == 0 and q.ck_attn_split_scratch_size(H_, KV, hd, 1025) == 0
    ok(call(64))
