"""Parity of the paged decode attention with a sliding window
(ck_attn_decode_gqa_paged) with the oracle: fp32, bf16 and fp8 E4M3 pools,
block tables scattering each sequence over the pool, ragged lengths, block
sizes that do and do not divide the stage height, windows shorter and longer
than the sequences.  Floating point: max |err| <= 1e-3 * max |ref| and
relative L2 <= 1e-4.  Table entries and lengths out of range raise CK_ERANGE
in the status word and are not read."""
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


def make_pools(rng, kind, nblk, KV, bs, hd):
    k = rng.standard_normal((nblk, KV, bs, hd)).astype(np.float32)
    v = rng.standard_normal((nblk, KV, bs, hd)).astype(np.float32)
    ks = float(np.abs(k).max() / 448 * 1.01)
    vs = float(np.abs(v).max() / 448 * 1.01)
    if kind == 1:
        return oracle.bf16_from_f32(k), oracle.bf16_from_f32(v), 1.0, 1.0
    if kind == 2:
        return oracle.e4m3_from_f32(k, ks), oracle.e4m3_from_f32(v, vs), ks, vs
    return k, v, 1.0, 1.0


def run_case(dev, kind, B, Hq, KV, hd, bs, maxb, lens, window, seed, nblk=None):
    rng = np.random.default_rng(seed)
    nblk = nblk or B * maxb + 3
    kp, vp, ks, vs = make_pools(rng, kind, nblk, KV, bs, hd)
    tables = rng.permutation(nblk)[:B * maxb].reshape(B, maxb).astype(np.int32)
    lens = np.asarray(lens, np.int32)
    qv = rng.standard_normal(B * Hq * hd).astype(np.float32)
    ref = oracle.attention_paged(qv, kp, vp, tables, lens, B, Hq, KV, hd, bs, maxb, window, kind, ks, vs)
    nbytes = q.ck_attn_paged_scratch_size(B, Hq, KV, hd, bs, maxb, window)
    assert nbytes > 0
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.full((B * Hq * hd,), float("nan"), dtype=torch.float32, device=dev)
    rc = q.ck_attn_decode_gqa_paged(T(qv, dev), T(kp, dev), T(vp, dev), out, T(tables, dev), T(lens, dev), B, Hq, KV,
                                    hd, bs, maxb, nblk, window, kind, ks, vs, scratch, nbytes)
    assert rc == q.CK_OK, q.ck_status_string(rc)
    assert_close(H(out), ref, f"kind {kind} bs {bs} lens {list(lens)} window {window}")
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_paged_short_ragged_sequences(dev, kind):
    run_case(dev, kind, 6, 8, 2, 64, 16, 8, [1, 15, 16, 17, 128, 0], 0, seed=40 + kind)


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("window", [0, 1, 100, 1000, 5000])
def test_paged_7b_heads_windows(dev, kind, window):
    run_case(dev, kind, 3, 28, 4, 128, 32, 40, [1280, 700, 33], window, seed=50 + kind + window)


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_paged_long_splits_large_blocks(dev, kind):
    run_case(dev, kind, 2, 32, 4, 128, 128, 80, [10240, 5000], 0, seed=60 + kind)
    run_case(dev, kind, 2, 32, 4, 128, 128, 80, [10240, 5000], 4096, seed=61 + kind)


@pytest.mark.parametrize("bs", [8, 48])
@pytest.mark.parametrize("kind", [0, 1])
def test_paged_block_sizes_straddling_stages(dev, kind, bs):
    run_case(dev, kind, 3, 16, 4, 128, bs, 700 // bs + 2, [700, 301, bs + 1], 0, seed=70 + bs + kind)
    run_case(dev, kind, 2, 16, 4, 64, bs, 4000 // bs + 2, [4000, 2222], 0, seed=71 + bs + kind)


def test_paged_out_of_range_entries_are_flagged_not_read(dev):
    rng = np.random.default_rng(80)
    B, Hq, KV, hd, bs, maxb = 2, 8, 2, 64, 16, 4
    nblk = 8
    kp, vp, _, _ = make_pools(rng, 0, nblk, KV, bs, hd)
    tables = np.array([[0, 1, 2, 3], [4, 5, 1000, 7]], np.int32)  # one entry outside the pool
    lens = np.array([40, 60], np.int32)
    qv = rng.standard_normal(B * Hq * hd).astype(np.float32)
    nbytes = q.ck_attn_paged_scratch_size(B, Hq, KV, hd, bs, maxb, 0)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(B * Hq * hd, dtype=torch.float32, device=dev)
    q.ck_device_status()
    assert q.ck_attn_decode_gqa_paged(T(qv, dev), T(kp, dev), T(vp, dev), out, T(tables, dev), T(lens, dev), B, Hq,
                                      KV, hd, bs, maxb, nblk, 0, 0, 1.0, 1.0, scratch, nbytes) == q.CK_OK
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    # sequence 0 does not touch the bad entry: exact as the oracle
    ref0 = oracle.attention_paged(qv[:Hq * hd], kp, vp, tables[:1], lens[:1], 1, Hq, KV, hd, bs, maxb, 0)
    assert_close(H(out)[:Hq * hd], ref0, "sequence 0")
    lens2 = np.array([40, maxb * bs + 1], np.int32)  # longer than its table
    assert q.ck_attn_decode_gqa_paged(T(qv, dev), T(kp, dev), T(vp, dev), out, T(tables[:, :4] % nblk, dev),
                                      T(lens2, dev), B, Hq, KV, hd, bs, maxb, nblk, 0, 0, 1.0, 1.0, scratch,
                                      nbytes) == q.CK_OK
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    assert np.all(H(out)[Hq * hd:] == 0.0)  # nothing attended: zeros


def test_paged_rejects_bad_arguments(dev):
    x = torch.zeros(4096, dtype=torch.float32, device=dev)
    i = torch.zeros(64, dtype=torch.int32, device=dev)
    nb = q.ck_attn_paged_scratch_size(2, 8, 2, 64, 16, 4, 0)
    s = torch.empty(nb, dtype=torch.uint8, device=dev)
    args = lambda **kw: dict(dict(batch=2, H=8, KV=2, hd=64, bs=16, maxb=4, nblk=8, win=0, kind=0, ks=1.0, vs=1.0,
                                  nbytes=nb), **kw)
    def call(a):
        return q.ck_attn_decode_gqa_paged(x, x, x, x, i, i, a["batch"], a["H"], a["KV"], a["hd"], a["bs"], a["maxb"],
                                          a["nblk"], a["win"], a["kind"], a["ks"], a["vs"], s, a["nbytes"])
    assert call(args(batch=0)) == q.CK_EINVAL
    assert call(args(bs=0)) == q.CK_EINVAL
    assert call(args(win=-1)) == q.CK_EINVAL
    assert call(args(kind=3)) == q.CK_EINVAL
    assert call(args(kind=1, hd=96, H=6, KV=2)) == q.CK_EINVAL
    assert call(args(kind=2, ks=0.0)) == q.CK_EINVAL
    assert call(args(nbytes=16)) == q.CK_ESCRATCH


@pytest.mark.parametrize("kind", [1, 2])
def test_paged_tensor_core_kernel_flags_bad_entries(dev, kind):
    """The same checks on the head_dim 128 bf16 / fp8 kernel (scores and P.V on
    the tensor cores): an entry outside the pool is flagged and the other
    sequence stays exact; a length past the table is flagged and gives zeros."""
    rng = np.random.default_rng(90 + kind)
    B, Hq, KV, hd, bs, maxb = 2, 28, 4, 128, 64, 4
    nblk = 8
    kp, vp, ks, vs = make_pools(rng, kind, nblk, KV, bs, hd)
    tables = np.array([[0, 1, 2, 3], [4, 5, 1000, 7]], np.int32)
    lens = np.array([200, 230], np.int32)
    qv = rng.standard_normal(B * Hq * hd).astype(np.float32)
    nbytes = q.ck_attn_paged_scratch_size(B, Hq, KV, hd, bs, maxb, 0)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(B * Hq * hd, dtype=torch.float32, device=dev)
    q.ck_device_status()
    assert q.ck_attn_decode_gqa_paged(T(qv, dev), T(kp, dev), T(vp, dev), out, T(tables, dev), T(lens, dev), B, Hq,
                                      KV, hd, bs, maxb, nblk, 0, kind, ks, vs, scratch, nbytes) == q.CK_OK
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    ref0 = oracle.attention_paged(qv[:Hq * hd], kp, vp, tables[:1], lens[:1], 1, Hq, KV, hd, bs, maxb, 0, kind, ks,
                                  vs)
    assert_close(H(out)[:Hq * hd], ref0, "sequence 0")
    lens2 = np.array([200, maxb * bs + 1], np.int32)
    assert q.ck_attn_decode_gqa_paged(T(qv, dev), T(kp, dev), T(vp, dev), out, T(tables[:, :4] % nblk, dev),
                                      T(lens2, dev), B, Hq, KV, hd, bs, maxb, nblk, 0, kind, ks, vs, scratch,
                                      nbytes) == q.CK_OK
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    assert np.all(H(out)[Hq * hd:] == 0.0)
