"""The C ABI without a GPU: the library builds and loads, exports every entry
point that include/ck_decode.h declares, and rejects invalid arguments on the
host before anything is launched (no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

import quantized_weight_attention_gb300 as q
from quantized_weight_attention_gb300 import build as kb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ck_decode.h")

A = 1 << 20          # a 16-byte aligned fake address: never dereferenced
MIS = (1 << 20) + 4  # misaligned


@pytest.fixture(scope="module", autouse=True)
def built():
    kb.build()
    return q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ck_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 15, names
    L = ctypes.CDLL(q.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_binding_covers_every_declared_function():
    for n in declared_functions():
        assert callable(getattr(q, n, None)), n


def test_status_strings():
    for rc in (q.CK_OK, q.CK_EINVAL, q.CK_ERANGE, q.CK_ESCRATCH, q.CK_EALIGN, q.CK_ECUDA, q.CK_ETIMEOUT):
        assert q.ck_status_string(rc).startswith("CK_")
    assert q.ck_status_string(12345) == "unknown status"


def test_quantize_validation():
    assert q.ck_quantize_q8_0(None, A, 32, 0) == q.CK_EINVAL
    assert q.ck_quantize_q8_0(A, A, 33, 0) == q.CK_EINVAL
    assert q.ck_quantize_q8_0(A, A, 0, 0) == q.CK_EINVAL
    assert q.ck_quantize_q8_0(MIS, A, 32, 0) == q.CK_EALIGN


def test_gemv_validation():
    for f in (q.ck_gemv_q5_0_q8_0, q.ck_gemv_q8_0_q8_0):
        assert f(A, A, A, None, 4, 48, 0) == q.CK_EINVAL
        assert f(A, A, A, None, 0, 64, 0) == q.CK_EINVAL
        assert f(A, None, A, None, 4, 64, 0) == q.CK_EINVAL
        assert f(A, A, A, MIS, 4, 64, 0) == q.CK_EALIGN
    for f in (q.ck_block_dots_q5_0_q8_0, q.ck_block_dots_q8_0_q8_0):
        assert f(A, A, A, 4, 40, 0) == q.CK_EINVAL
        assert f(MIS, A, A, 4, 64, 0) == q.CK_EALIGN


def test_rope_and_store_validation():
    assert q.ck_rope_inplace(A, A, A, A, 64, 4, 2, 64, 64, 0) == q.CK_ERANGE
    assert q.ck_rope_inplace(A, A, A, A, -1, 4, 2, 64, 64, 0) == q.CK_ERANGE
    assert q.ck_rope_inplace(A, A, A, A, 0, 4, 2, 63, 64, 0) == q.CK_EINVAL
    assert q.ck_rope_inplace(None, A, A, A, 0, 4, 2, 64, 64, 0) == q.CK_EINVAL
    assert q.ck_kv_store(A, A, A, A, 64, 2, 64, 64, 0) == q.CK_ERANGE
    assert q.ck_kv_store(A, A, A, None, 0, 2, 64, 64, 0) == q.CK_EINVAL


def test_attention_validation():
    ok = dict(num_heads=4, num_kv_heads=2, kv_tokens=17, cache_capacity=64, head_dim=64)

    def call(**kw):
        a = dict(ok, **kw)
        return q.ck_attn_decode_gqa(A, A, A, A, a["num_heads"], a["num_kv_heads"], a["kv_tokens"],
                                    a["cache_capacity"], a["head_dim"], A, 1 << 30, 0)
    assert call(kv_tokens=0) == q.CK_ERANGE
    assert call(kv_tokens=65) == q.CK_ERANGE
    assert call(num_heads=5) == q.CK_EINVAL          # H % KV != 0
    assert call(num_heads=18, num_kv_heads=2) == q.CK_EINVAL   # group of 9 > 8
    assert call(head_dim=48) == q.CK_EINVAL
    assert call(head_dim=160) == q.CK_EINVAL
    assert q.ck_attn_decode_gqa(A, A, A, A, 4, 2, 17, 64, 64, None, 0, 0) == q.CK_ESCRATCH
    assert q.ck_attn_decode_gqa(A, A, A, A, 4, 2, 17, 64, 64, A, 16, 0) == q.CK_ESCRATCH
    assert q.ck_attn_scratch_size(5, 2, 100, 64) == 0
    assert q.ck_attn_scratch_size(4, 2, 100, 64) > 0


def _layer(**kw):
    a = dict(out=A + 4096, x=A, res=A, pos=16, D=256, H=4, KV=2, hd=64, C=64, scratch=A, nbytes=1 << 30, dpos=None)
    a.update(kw)
    args = [a["out"], a["x"], a["res"], A, A, A, A, A, None, None, None, None, A, A, A, A]
    if a["dpos"] is None:
        return q.ck_decode_layer(*args, a["pos"], a["D"], a["H"], a["KV"], a["hd"], a["C"], 1e-6, a["scratch"],
                                 a["nbytes"], 0)
    return q.ck_decode_layer_devpos(*args, a["dpos"], a["D"], a["H"], a["KV"], a["hd"], a["C"], 1e-6, a["scratch"],
                                    a["nbytes"], 0)


def test_layer_validation():
    assert _layer(pos=64) == q.CK_ERANGE
    assert _layer(pos=-1) == q.CK_ERANGE
    assert _layer(D=250) == q.CK_EINVAL
    assert _layer(H=6, KV=4) == q.CK_EINVAL
    assert _layer(scratch=None) == q.CK_ESCRATCH
    assert _layer(nbytes=100) == q.CK_ESCRATCH
    assert _layer(scratch=MIS) == q.CK_EALIGN
    assert _layer(x=MIS) == q.CK_EALIGN
    assert _layer(out=A) == q.CK_EINVAL            # out aliases x
    assert _layer(dpos=MIS) == q.CK_EALIGN
    assert q.ck_decode_layer_devpos(*([A] * 16), None, 256, 4, 2, 64, 64, 1e-6, A, 1 << 30, 0) == q.CK_EINVAL
    assert q.ck_decode_layer_scratch_size(250, 4, 2, 64, 64) == 0
    assert q.ck_decode_layer_scratch_offset(9, 256, 4, 2, 64, 64) == (1 << 64) - 1


def test_scratch_offsets_are_disjoint_and_inside():
    D, H, KV, hd, C = 3584, 28, 4, 128, 8256
    total = q.ck_decode_layer_scratch_size(D, H, KV, hd, C)
    offs = [q.ck_decode_layer_scratch_offset(t, D, H, KV, hd, C) for t in range(4)]
    sizes = [H * hd * 4, D // 32 * 34, H * hd * 4, H * hd // 32 * 34]
    spans = sorted(zip(offs, sizes))
    for (o1, s1), (o2, _) in zip(spans, spans[1:]):
        assert o1 + s1 <= o2
    assert all(o % 256 == 0 for o in offs)
    assert spans[-1][0] + spans[-1][1] <= total


def _batched(**kw):
    a = dict(out=A + 4096, x=A, res=A, kcs=A, vcs=A, dpos=A, B=3, D=256, H=4, KV=2, hd=64, C=64, scratch=A,
             nbytes=1 << 30)
    a.update(kw)
    return q.ck_decode_layer_batched(a["out"], a["x"], a["res"], A, A, A, A, A, None, None, None, None, a["kcs"],
                                     a["vcs"], A, A, a["dpos"], a["B"], a["D"], a["H"], a["KV"], a["hd"], a["C"],
                                     1e-6, a["scratch"], a["nbytes"], 0)


def test_batched_validation():
    """Every bad argument is refused on the host, before any launch."""
    assert _batched(B=0) == q.CK_EINVAL
    assert _batched(B=1025) == q.CK_EINVAL
    assert _batched(D=224) == q.CK_EINVAL          # embed_dim not a multiple of 256
    assert _batched(D=4352) == q.CK_EINVAL         # more than 128 blocks per row
    assert _batched(H=2, hd=64) == q.CK_EINVAL     # num_heads*head_dim = 128
    assert _batched(H=6, KV=4) == q.CK_EINVAL
    assert _batched(hd=48) == q.CK_EINVAL
    assert _batched(kcs=None) == q.CK_EINVAL
    assert _batched(dpos=None) == q.CK_EINVAL
    assert _batched(dpos=MIS) == q.CK_EALIGN
    assert _batched(scratch=None) == q.CK_ESCRATCH
    assert _batched(nbytes=100) == q.CK_ESCRATCH
    assert _batched(scratch=MIS) == q.CK_EALIGN
    assert _batched(out=A) == q.CK_EINVAL           # out aliases x
    assert q.ck_decode_layer_batched_scratch_size(0, 256, 4, 2, 64, 64) == 0
    assert q.ck_decode_layer_batched_scratch_offset(9, 3, 256, 4, 2, 64, 64) == (1 << 64) - 1


def test_batched_scratch_offsets_are_disjoint_and_inside():
    Bn, D, H, KV, hd, C = 64, 3584, 28, 4, 128, 16448
    total = q.ck_decode_layer_batched_scratch_size(Bn, D, H, KV, hd, C)
    offs = [q.ck_decode_layer_batched_scratch_offset(t, Bn, D, H, KV, hd, C) for t in range(4)]
    sizes = [Bn * H * hd * 4, Bn * D // 32 * 34, Bn * H * hd * 4, Bn * H * hd // 32 * 34]
    spans = sorted(zip(offs, sizes))
    for (o1, s1), (o2, _) in zip(spans, spans[1:]):
        assert o1 + s1 <= o2
    assert all(o % 256 == 0 for o in offs)
    assert spans[-1][0] + spans[-1][1] <= total
