"""The oracle: ctypes access to ``oracle/ck_ref.c``.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product (the CUDA library and its
Python binding) never imports this package, and this package never imports
the product: the two share no code, only the bytes of inputs and outputs.

Every function follows the page "mega_fused_attention_decode_q5_0.c"
(C-Kernel-Engine), serial kernel, in the order STEP 1 (RMSNorm) to STEP 8
(O projection + residual); see ``ck_ref.c`` for the reading of each step that
the page declares without printing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ck_ref.c")
_LIB = os.path.join(_HERE, "libck_ref.so")
_lock = threading.Lock()
_lib = None

QK = 32
Q5_0_BYTES = 22
Q8_0_BYTES = 34

_CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-Wall"]


def build(force: bool = False) -> str:
    """Compile ``ck_ref.c`` into ``libck_ref.so`` with gcc (host code only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i = ctypes.c_int
            f = ctypes.c_float
            L.ref_f16_to_f32.restype = f
            L.ref_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.ref_f32_to_f16.restype = ctypes.c_uint16
            L.ref_f32_to_f16.argtypes = [f]
            L.ref_f32_to_f16_n.argtypes = [P, P, ctypes.c_long]
            L.ref_f16_to_f32_n.argtypes = [P, P, ctypes.c_long]
            L.ref_unpack_q5_0.argtypes = [P, P, P]
            L.ref_unpack_q8_0.argtypes = [P, P, P]
            L.ref_dequant_q5_0.argtypes = [P, P]
            L.ref_dequant_q8_0.argtypes = [P, P]
            L.ref_quantize_row_q8_0.argtypes = [P, P, i]
            L.ref_block_dot_q5_0_q8_0.restype = ctypes.c_int32
            L.ref_block_dot_q5_0_q8_0.argtypes = [P, P]
            L.ref_block_dot_q8_0_q8_0.restype = ctypes.c_int32
            L.ref_block_dot_q8_0_q8_0.argtypes = [P, P]
            L.ref_block_dots.argtypes = [P, P, P, i, i, i]
            L.ref_gemv.argtypes = [P, P, P, P, i, i, i]
            L.ref_bf16_to_f32.restype = f
            L.ref_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.ref_f32_to_bf16.restype = ctypes.c_uint16
            L.ref_f32_to_bf16.argtypes = [f]
            L.ref_e4m3_to_f32.restype = f
            L.ref_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            L.ref_f32_to_e4m3.restype = ctypes.c_uint8
            L.ref_f32_to_e4m3.argtypes = [f]
            L.ref_f32_to_bf16_n.argtypes = [P, P, ctypes.c_long]
            L.ref_f32_to_e4m3_n.argtypes = [P, f, P, ctypes.c_long]
            L.ref_e4m3_to_f32_n.argtypes = [P, P, ctypes.c_long]
            L.ref_attention_kvq.argtypes = [P, P, P, P, i, i, i, i, i, i, f, f]
            L.ref_kv_store_kvq.argtypes = [P, P, P, P, i, i, i, i, i, f, f]
            L.ref_attention_paged.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, i, f, f]
            L.ref_rmsnorm.restype = f
            L.ref_rmsnorm.argtypes = [P, P, P, i, f]
            L.ref_rope.argtypes = [P, P, P, P, i, i, i, i]
            L.ref_kv_store.argtypes = [P, P, P, P, i, i, i, i]
            L.ref_attention.argtypes = [P, P, P, P, i, i, i, i, i]
            L.ref_decode_layer.argtypes = [P] * 16 + [i] * 6 + [f] + [P] * 6
            L.ref_prefill_layer.argtypes = [P] * 16 + [i] * 7 + [f] + [P] * 6
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


# --- fp16 -------------------------------------------------------------------
def f16_to_f32(h: int) -> float:
    return lib().ref_f16_to_f32(int(h))


def f32_to_f16(x: float) -> int:
    return int(lib().ref_f32_to_f16(float(x)))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    x = _f32(x).ravel()
    h = np.empty(x.size, np.uint16)
    lib().ref_f32_to_f16_n(_p(x), _p(h), x.size)
    return h


def f16_to_f32_array(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    x = np.empty(h.size, np.float32)
    lib().ref_f16_to_f32_n(_p(h), _p(x), h.size)
    return x


# --- block codecs ------------------------------------------------------------
def unpack_q5_0(blocks: np.ndarray):
    """Q5_0 bytes [..., 22] -> (codes int32 [..., 32] in [-16, 15], d float32 [...])."""
    b = _u8(blocks).reshape(-1, Q5_0_BYTES)
    q = np.empty((b.shape[0], QK), np.int32)
    d = np.empty(b.shape[0], np.float32)
    L = lib()
    for r in range(b.shape[0]):
        L.ref_unpack_q5_0(_p(b[r]), _p(q[r]), _p(d[r:r + 1]))
    return q, d


def unpack_q8_0(blocks: np.ndarray):
    b = _u8(blocks).reshape(-1, Q8_0_BYTES)
    q = np.empty((b.shape[0], QK), np.int32)
    d = np.empty(b.shape[0], np.float32)
    L = lib()
    for r in range(b.shape[0]):
        L.ref_unpack_q8_0(_p(b[r]), _p(q[r]), _p(d[r:r + 1]))
    return q, d


def dequant_q5_0(blocks: np.ndarray) -> np.ndarray:
    b = _u8(blocks).reshape(-1, Q5_0_BYTES)
    w = np.empty((b.shape[0], QK), np.float32)
    L = lib()
    for r in range(b.shape[0]):
        L.ref_dequant_q5_0(_p(b[r]), _p(w[r]))
    return w


def dequant_q8_0(blocks: np.ndarray) -> np.ndarray:
    b = _u8(blocks).reshape(-1, Q8_0_BYTES)
    w = np.empty((b.shape[0], QK), np.float32)
    L = lib()
    for r in range(b.shape[0]):
        L.ref_dequant_q8_0(_p(b[r]), _p(w[r]))
    return w


# --- hot-path steps ----------------------------------------------------------
def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """fp32 [n] (n % 32 == 0) -> Q8_0 bytes [n/32 * 34]."""
    x = _f32(x).ravel()
    assert x.size % QK == 0
    y = np.empty(x.size // QK * Q8_0_BYTES, np.uint8)
    lib().ref_quantize_row_q8_0(_p(x), _p(y), x.size)
    return y


def block_dots(W: np.ndarray, xq: np.ndarray, M: int, K: int, w_is_q8: bool) -> np.ndarray:
    out = np.empty((M, K // QK), np.int32)
    lib().ref_block_dots(_p(out), _p(_u8(W)), _p(_u8(xq)), M, K, int(w_is_q8))
    return out


def gemv(W: np.ndarray, xq: np.ndarray, bias, M: int, K: int, w_is_q8: bool) -> np.ndarray:
    y = np.empty(M, np.float32)
    b = None if bias is None else _f32(bias)
    lib().ref_gemv(_p(y), _p(_u8(W)), _p(_u8(xq)), _p(b), M, K, int(w_is_q8))
    return y


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float):
    x = _f32(x)
    y = np.empty_like(x)
    rstd = lib().ref_rmsnorm(_p(x), _p(_f32(gamma)), _p(y), x.size, float(eps))
    return y, np.float32(rstd)


def rope(q, k, rope_cos, rope_sin, pos: int, H: int, KV: int, hd: int):
    q = None if q is None else _f32(q).copy()
    k = None if k is None else _f32(k).copy()
    lib().ref_rope(_p(q), _p(k), _p(_f32(rope_cos)), _p(_f32(rope_sin)), pos, H, KV, hd)
    return q, k


def kv_store(k_cache, v_cache, k, v, pos: int, KV: int, capacity: int, hd: int):
    """In place on k_cache / v_cache (float32, C-contiguous)."""
    assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float32 and v_cache.flags.c_contiguous
    lib().ref_kv_store(_p(k_cache), _p(v_cache), _p(_f32(k)), _p(_f32(v)), pos, KV, capacity, hd)


def attention(q, k_cache, v_cache, H: int, KV: int, T: int, capacity: int, hd: int) -> np.ndarray:
    out = np.empty(H * hd, np.float32)
    lib().ref_attention(_p(_f32(q)), _p(_f32(k_cache)), _p(_f32(v_cache)), _p(out), H, KV, T, capacity, hd)
    return out


# ---- reduced-precision KV caches (bf16; fp8 E4M3 with per-tensor scales) ----
KV_BF16, KV_FP8 = 1, 2


def bf16_from_f32(x) -> np.ndarray:
    """bfloat16 bit patterns of x (round to nearest, ties to even)."""
    x = _f32(x)
    y = np.empty(x.size, np.uint16)
    lib().ref_f32_to_bf16_n(_p(x), _p(y), x.size)
    return y.reshape(x.shape)


def bf16_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_from_f32(x, scale: float = 1.0) -> np.ndarray:
    """E4M3 codes of x / scale (round to nearest even, saturated to +-448)."""
    x = _f32(x)
    y = np.empty(x.size, np.uint8)
    lib().ref_f32_to_e4m3_n(_p(x), float(scale), _p(y), x.size)
    return y.reshape(x.shape)


def e4m3_to_f32(c) -> np.ndarray:
    c = np.ascontiguousarray(c, np.uint8)
    y = np.empty(c.size, np.float32)
    lib().ref_e4m3_to_f32_n(_p(c), _p(y), c.size)
    return y.reshape(c.shape)


def attention_kvq(q, k_cache, v_cache, H: int, KV: int, T: int, capacity: int, hd: int, kind: int,
                  k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Decode attention over a bf16 (kind 1) or E4M3 (kind 2) cache [KV, capacity, hd]."""
    dt = np.uint16 if kind == KV_BF16 else np.uint8
    kc = np.ascontiguousarray(k_cache, dt)
    vc = np.ascontiguousarray(v_cache, dt)
    out = np.empty(H * hd, np.float32)
    lib().ref_attention_kvq(_p(_f32(q)), _p(kc), _p(vc), _p(out), H, KV, T, capacity, hd, kind, float(k_scale),
                            float(v_scale))
    return out


def kv_store_kvq(k_cache, v_cache, k, v, pos: int, KV: int, capacity: int, hd: int, kind: int,
                 k_scale: float = 1.0, v_scale: float = 1.0):
    """STEP 6 into a reduced cache, in place."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    lib().ref_kv_store_kvq(_p(k_cache), _p(v_cache), _p(_f32(k)), _p(_f32(v)), pos, KV, capacity, hd, kind,
                           float(k_scale), float(v_scale))


def attention_paged(q, k_pool, v_pool, block_tables, seq_lens, B: int, H: int, KV: int, hd: int, block_size: int,
                    max_blocks: int, window: int, kind: int = 0, k_scale: float = 1.0,
                    v_scale: float = 1.0) -> np.ndarray:
    """Paged decode attention: pools [num_blocks, KV, block_size, hd] of fp32 (kind 0), bf16 (1) or E4M3 (2);
    block_tables int32 [B, max_blocks]; seq_lens int32 [B]; window 0 = all rows."""
    dt = {0: np.float32, 1: np.uint16, 2: np.uint8}[kind]
    kp = np.ascontiguousarray(k_pool, dt)
    vp = np.ascontiguousarray(v_pool, dt)
    bt = np.ascontiguousarray(block_tables, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    out = np.empty(B * H * hd, np.float32)
    lib().ref_attention_paged(_p(_f32(q)), _p(kp), _p(vp), _p(out), _p(bt), _p(sl), B, H, KV, hd, block_size,
                              max_blocks, window, kind, float(k_scale), float(v_scale))
    return out


def decode_layer(x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos, rope_sin,
                 pos: int, D: int, H: int, KV: int, hd: int, capacity: int, eps: float, taps: bool = False):
    """One decode step; k_cache / v_cache (float32, C-contiguous) are updated in place.

    Returns ``out`` or, with ``taps``, ``(out, dict_of_intermediates)``.
    """
    assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float32 and v_cache.flags.c_contiguous
    out = np.empty(D, np.float32)
    t = None
    if taps:
        t = dict(xq=np.empty(D // QK * Q8_0_BYTES, np.uint8), q=np.empty(H * hd, np.float32),
                 k=np.empty(KV * hd, np.float32), v=np.empty(KV * hd, np.float32),
                 attn=np.empty(H * hd, np.float32), aq=np.empty(H * hd // QK * Q8_0_BYTES, np.uint8))
    g = (lambda n: _p(t[n])) if taps else (lambda n: None)
    opt = lambda a: None if a is None else _p(_f32(a))
    lib().ref_decode_layer(_p(out), _p(_f32(x)), _p(_f32(residual)), _p(_u8(wq)), _p(_u8(wk)), _p(_u8(wv)),
                           _p(_u8(wo)), _p(_f32(gamma)), opt(bq), opt(bk), opt(bv), opt(bo), _p(k_cache),
                           _p(v_cache), _p(_f32(rope_cos)), _p(_f32(rope_sin)), pos, D, H, KV, hd, capacity,
                           float(eps), g("xq"), g("q"), g("k"), g("v"), g("attn"), g("aq"))
    return (out, t) if taps else out


def prefill_layer(x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos, rope_sin,
                  pos: int, n: int, D: int, H: int, KV: int, hd: int, capacity: int, eps: float, taps: bool = False):
    """The causal multi-token form: n tokens [n, D] at positions pos..pos+n-1.

    k_cache / v_cache (float32, C-contiguous) get rows pos..pos+n-1 in place.
    Returns ``out`` [n, D] or, with ``taps``, ``(out, dict_of_intermediates)``
    whose entries are the decode layer's taps, one row per token.
    """
    assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float32 and v_cache.flags.c_contiguous
    assert 0 <= pos and pos + n <= capacity and n >= 1
    out = np.empty((n, D), np.float32)
    t = None
    if taps:
        t = dict(xq=np.empty((n, D // QK * Q8_0_BYTES), np.uint8), q=np.empty((n, H * hd), np.float32),
                 k=np.empty((n, KV * hd), np.float32), v=np.empty((n, KV * hd), np.float32),
                 attn=np.empty((n, H * hd), np.float32), aq=np.empty((n, H * hd // QK * Q8_0_BYTES), np.uint8))
    g = (lambda nm: _p(t[nm])) if taps else (lambda nm: None)
    opt = lambda a: None if a is None else _p(_f32(a))
    lib().ref_prefill_layer(_p(out), _p(_f32(x)), _p(_f32(residual)), _p(_u8(wq)), _p(_u8(wk)), _p(_u8(wv)),
                            _p(_u8(wo)), _p(_f32(gamma)), opt(bq), opt(bk), opt(bv), opt(bo), _p(k_cache),
                            _p(v_cache), _p(_f32(rope_cos)), _p(_f32(rope_sin)), pos, n, D, H, KV, hd, capacity,
                            float(eps), g("xq"), g("q"), g("k"), g("v"), g("attn"), g("aq"))
    return (out, t) if taps else out
