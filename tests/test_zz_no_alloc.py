"""The attention entry point for callers that cannot allocate device memory.

Some callers of this library own no device allocator of their own: their
memory belongs to a host framework's pool or to a fixed budget, or they run a
decode loop where a cudaMalloc (which can synchronize the device) is not
acceptable.  ck_attn_decode_gqa_noalloc serves them by keeping its split-KV
partials in a buffer built into the library.  These tests call it through
the C ABI and check it against ck_attn_decode_gqa, which takes caller
scratch, within the parity tolerance of the other GPU tests, on two calls in
a row (the second with a different shape, so it also shows that what the
first call left in the shared buffer does not leak into the next result).

The file name makes pytest collect it last."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
import quantized_weight_attention_gb300 as q  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    from quantized_weight_attention_gb300 import build as kb
    kb.build()
    q.lib()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _close(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err <= 1e-3 * np.abs(ref).max() and rel <= 1e-4, (err, rel)


def _case(dev, Hh, KV, hd, Tn, C, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    kc = torch.zeros((KV, C, hd), dtype=torch.float32)
    vc = torch.zeros((KV, C, hd), dtype=torch.float32)
    kc[:, :Tn] = torch.randn((KV, Tn, hd), generator=g)
    vc[:, :Tn] = torch.randn((KV, Tn, hd), generator=g)
    qv = torch.randn(Hh * hd, generator=g)
    return qv.to(dev), kc.to(dev), vc.to(dev)


def _with_scratch(dev, qv, kc, vc, Hh, KV, hd, Tn, C):
    n = q.ck_attn_scratch_size(Hh, KV, C, hd)
    scratch = torch.empty(n, dtype=torch.uint8, device=dev)
    out = torch.empty(Hh * hd, dtype=torch.float32, device=dev)
    assert q.ck_attn_decode_gqa(qv, kc, vc, out, Hh, KV, Tn, C, hd, scratch, n) == q.CK_OK
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_attention_matches_scratch_version_twice(dev):
    shapes = [(28, 4, 128, 8193, 8256), (14, 2, 64, 1025, 2048)]
    for i, (Hh, KV, hd, Tn, C) in enumerate(shapes):
        qv, kc, vc = _case(dev, Hh, KV, hd, Tn, C, 100 + i)
        out = torch.full((Hh * hd,), float("nan"), dtype=torch.float32, device=dev)
        assert q.ck_attn_decode_gqa_noalloc(qv, kc, vc, out, Hh, KV, Tn, C, hd) == q.CK_OK
        torch.cuda.synchronize()
        _close(out.cpu().numpy(), _with_scratch(dev, qv, kc, vc, Hh, KV, hd, Tn, C))
    rc, st = q.ck_device_status()
    assert rc == q.CK_OK and st == q.CK_OK


def test_noalloc_rejects_bad_arguments_before_launch(dev):
    qv, kc, vc = _case(dev, 4, 2, 64, 17, 64, 7)
    out = torch.empty(256, dtype=torch.float32, device=dev)
    assert q.ck_attn_decode_gqa_noalloc(qv, kc, vc, out, 4, 2, 65, 64, 64) == q.CK_ERANGE
    assert q.ck_attn_decode_gqa_noalloc(None, kc, vc, out, 4, 2, 17, 64, 64) == q.CK_EINVAL
    assert q.ck_attn_decode_gqa_noalloc(qv, kc, vc, out, 5, 2, 17, 64, 64) == q.CK_EINVAL
