"""GB300 (sm_103a) single-token attention decode step with Q5_0 / Q8_0 weights.

Python binding of ``libck_decode.so`` (C ABI in ``include/ck_decode.h``).
Each ``ck_*`` function below has the name and argument order of the C entry
point and only marshals arguments: tensors become device pointers, ``stream``
defaults to torch's current CUDA stream.  Every step runs in the library's
CUDA kernels; there is no other implementation behind these names, and a
missing library raises instead of falling back.

Entry points follow the page "mega_fused_attention_decode_q5_0.c"
(C-Kernel-Engine): quantize_row_q8_0, the Q5_0 / Q8_0 GEMVs, apply_rope_inline,
the KV-cache store, attention_forward_decode_head_major_gqa_flash, and the
whole mega-fused layer step.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "CK_OK", "CK_EINVAL", "CK_ERANGE", "CK_ESCRATCH", "CK_EALIGN", "CK_ECUDA", "CK_ETIMEOUT", "CkError",
    "lib", "check", "ck_status_string", "ck_quantize_q8_0", "ck_gemv_q5_0_q8_0", "ck_gemv_q8_0_q8_0",
    "ck_rope_inplace", "ck_kv_store", "ck_attn_scratch_size", "ck_attn_decode_gqa",
    "ck_prefill_layer_scratch_size", "ck_prefill_layer_scratch_offset", "ck_prefill_layer",
    "ck_prefill_layer_devpos",
    "ck_attn_split_scratch_size", "ck_attn_decode_gqa_split",
    "ck_attn_prefill_scratch_size", "ck_attn_prefill_gqa",
    "ck_decode_layer_scratch_size", "ck_decode_layer", "ck_decode_layer_devpos", "ck_device_status",
    "ck_block_dots_q5_0_q8_0", "ck_block_dots_q8_0_q8_0", "LIB_PATH", "ck_decode_layer_scratch_offset",
    "CK_TAP_Q", "CK_TAP_XQ8", "CK_TAP_ATTN", "CK_TAP_AQ8", "ck_attn_decode_gqa_noalloc",
    "CK_ATTN_NOALLOC_MAX_BYTES", "ck_attn_decode_gqa_bf16", "ck_attn_decode_gqa_fp8", "ck_kv_store_bf16",
    "ck_kv_store_fp8", "ck_attn_paged_scratch_size", "ck_attn_decode_gqa_paged",
]

CK_OK, CK_EINVAL, CK_ERANGE, CK_ESCRATCH, CK_EALIGN, CK_ECUDA, CK_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libck_decode.so")
_lib = None
_lock = threading.Lock()


class CkError(RuntimeError):
    pass


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "ck_status_string": (ctypes.c_char_p, [_I]),
    "ck_quantize_q8_0": (_I, [_P, _P, _I, _P]),
    "ck_gemv_q5_0_q8_0": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "ck_gemv_q8_0_q8_0": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "ck_rope_inplace": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "ck_kv_store": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "ck_attn_scratch_size": (_SZ, [_I, _I, _I, _I]),
    "ck_attn_decode_gqa": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "ck_attn_decode_gqa_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "ck_attn_decode_gqa_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _P, _SZ, _P]),
    "ck_kv_store_bf16": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "ck_kv_store_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _F, _F, _P]),
    "ck_attn_paged_scratch_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "ck_attn_decode_gqa_paged": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _P, _SZ,
                                      _P]),
    "ck_attn_decode_gqa_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "ck_decode_layer_scratch_size": (_SZ, [_I, _I, _I, _I, _I]),
    "ck_decode_layer": (_I, [_P] * 16 + [_I] * 6 + [_F, _P, _SZ, _P]),
    "ck_decode_layer_devpos": (_I, [_P] * 17 + [_I] * 5 + [_F, _P, _SZ, _P]),
    "ck_device_status": (_I, [_P, _P]),
    "ck_decode_layer_scratch_offset": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "ck_decode_layer_batched_scratch_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "ck_decode_layer_batched": (_I, [_P] * 17 + [_I] * 6 + [_F, _P, _SZ, _P]),
    "ck_decode_layer_batched_scratch_offset": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "ck_prefill_layer_scratch_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "ck_prefill_layer_scratch_offset": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "ck_prefill_layer": (_I, [_P] * 16 + [_I] * 7 + [_F, _P, _SZ, _P]),
    "ck_prefill_layer_devpos": (_I, [_P] * 17 + [_I] * 6 + [_F, _P, _SZ, _P]),
    "ck_attn_split_scratch_size": (_SZ, [_I, _I, _I, _I]),
    "ck_attn_prefill_scratch_size": (_SZ, [_I, _I, _I, _I]),
    "ck_attn_prefill_gqa": (_I, [_P] * 4 + [_I] * 6 + [_P, _SZ, _P]),
    "ck_attn_decode_gqa_split": (_I, [_P] * 4 + [_I] * 6 + [_F, _F, _I, _P, _SZ, _P]),
    "ck_block_dots_q5_0_q8_0": (_I, [_P, _P, _P, _I, _I, _P]),
    "ck_block_dots_q8_0_q8_0": (_I, [_P, _P, _P, _I, _I, _P]),
}


def lib():
    """The loaded CUDA library; raises CkError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise CkError(f"{LIB_PATH} is missing: build it with quantized_weight_attention_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def ck_status_string(rc: int) -> str:
    return lib().ck_status_string(rc).decode()


def check(rc: int) -> int:
    if rc != CK_OK:
        raise CkError(ck_status_string(rc))
    return rc


def ck_quantize_q8_0(x, y_q8, n: int, stream=None) -> int:
    return lib().ck_quantize_q8_0(_ptr(x), _ptr(y_q8), n, _stream(stream))


def ck_gemv_q5_0_q8_0(y, W, x_q8, bias, M: int, K: int, stream=None) -> int:
    return lib().ck_gemv_q5_0_q8_0(_ptr(y), _ptr(W), _ptr(x_q8), _ptr(bias), M, K, _stream(stream))


def ck_gemv_q8_0_q8_0(y, W, x_q8, bias, M: int, K: int, stream=None) -> int:
    return lib().ck_gemv_q8_0_q8_0(_ptr(y), _ptr(W), _ptr(x_q8), _ptr(bias), M, K, _stream(stream))


def ck_rope_inplace(q, k, rope_cos, rope_sin, pos: int, num_heads: int, num_kv_heads: int, head_dim: int,
                    cache_capacity: int, stream=None) -> int:
    return lib().ck_rope_inplace(_ptr(q), _ptr(k), _ptr(rope_cos), _ptr(rope_sin), pos, num_heads, num_kv_heads,
                                 head_dim, cache_capacity, _stream(stream))


def ck_kv_store(k_cache, v_cache, k, v, pos: int, num_kv_heads: int, cache_capacity: int, head_dim: int,
                stream=None) -> int:
    return lib().ck_kv_store(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), pos, num_kv_heads, cache_capacity,
                             head_dim, _stream(stream))


def ck_attn_scratch_size(num_heads: int, num_kv_heads: int, max_kv_tokens: int, head_dim: int) -> int:
    return lib().ck_attn_scratch_size(num_heads, num_kv_heads, max_kv_tokens, head_dim)


def ck_attn_decode_gqa(q, k_cache, v_cache, out, num_heads: int, num_kv_heads: int, kv_tokens: int,
                       cache_capacity: int, head_dim: int, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().ck_attn_decode_gqa(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), num_heads, num_kv_heads,
                                    kv_tokens, cache_capacity, head_dim, _ptr(scratch), scratch_bytes,
                                    _stream(stream))


def ck_attn_decode_gqa_bf16(q, k_cache, v_cache, out, num_heads: int, num_kv_heads: int, kv_tokens: int,
                            cache_capacity: int, head_dim: int, scratch, scratch_bytes: int, stream=None) -> int:
    """ck_attn_decode_gqa over bf16 caches (head_dim 64 or 128)."""
    return lib().ck_attn_decode_gqa_bf16(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), num_heads, num_kv_heads,
                                         kv_tokens, cache_capacity, head_dim, _ptr(scratch), scratch_bytes,
                                         _stream(stream))


def ck_attn_decode_gqa_fp8(q, k_cache, v_cache, out, num_heads: int, num_kv_heads: int, kv_tokens: int,
                           cache_capacity: int, head_dim: int, k_scale: float, v_scale: float, scratch,
                           scratch_bytes: int, stream=None) -> int:
    """ck_attn_decode_gqa over fp8 E4M3 caches: k = code * k_scale, v = code * v_scale."""
    return lib().ck_attn_decode_gqa_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), num_heads, num_kv_heads,
                                        kv_tokens, cache_capacity, head_dim, float(k_scale), float(v_scale),
                                        _ptr(scratch), scratch_bytes, _stream(stream))


def ck_kv_store_bf16(k_cache, v_cache, k, v, pos: int, num_kv_heads: int, cache_capacity: int, head_dim: int,
                     stream=None) -> int:
    return lib().ck_kv_store_bf16(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), pos, num_kv_heads,
                                  cache_capacity, head_dim, _stream(stream))


def ck_kv_store_fp8(k_cache, v_cache, k, v, pos: int, num_kv_heads: int, cache_capacity: int, head_dim: int,
                    k_scale: float, v_scale: float, stream=None) -> int:
    return lib().ck_kv_store_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k), _ptr(v), pos, num_kv_heads, cache_capacity,
                                 head_dim, float(k_scale), float(v_scale), _stream(stream))


def ck_attn_paged_scratch_size(batch: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                               max_blocks_per_seq: int, sliding_window: int) -> int:
    return lib().ck_attn_paged_scratch_size(batch, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                            sliding_window)


def ck_attn_decode_gqa_paged(q, k_pool, v_pool, out, block_tables, seq_lens, batch: int, num_heads: int,
                             num_kv_heads: int, head_dim: int, block_size: int, max_blocks_per_seq: int,
                             num_blocks: int, sliding_window: int, kv_dtype: int, k_scale: float, v_scale: float,
                             scratch, scratch_bytes: int, stream=None) -> int:
    """Paged decode attention with an optional sliding window (kv_dtype 0 fp32, 1 bf16, 2 fp8 E4M3)."""
    return lib().ck_attn_decode_gqa_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out), _ptr(block_tables),
                                          _ptr(seq_lens), batch, num_heads, num_kv_heads, head_dim, block_size,
                                          max_blocks_per_seq, num_blocks, sliding_window, kv_dtype, float(k_scale),
                                          float(v_scale), _ptr(scratch), scratch_bytes, _stream(stream))


CK_ATTN_NOALLOC_MAX_BYTES = 2 * 1024 * 1024


def ck_attn_decode_gqa_noalloc(q, k_cache, v_cache, out, num_heads: int, num_kv_heads: int, kv_tokens: int,
                               cache_capacity: int, head_dim: int, stream=None) -> int:
    """ck_attn_decode_gqa without a scratch argument, for callers that cannot
    allocate device memory: the partials live in a buffer built into the
    library (shared by all calls; overlapping calls on the GPU race)."""
    return lib().ck_attn_decode_gqa_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), num_heads,
                                            num_kv_heads, kv_tokens, cache_capacity, head_dim, _stream(stream))


def ck_decode_layer_scratch_size(embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                 cache_capacity: int) -> int:
    return lib().ck_decode_layer_scratch_size(embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity)


def ck_decode_layer(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos, rope_sin,
                    pos: int, embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int, cache_capacity: int,
                    eps: float, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().ck_decode_layer(
        _ptr(out), _ptr(x), _ptr(residual), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(bq), _ptr(bk),
        _ptr(bv), _ptr(bo), _ptr(k_cache), _ptr(v_cache), _ptr(rope_cos), _ptr(rope_sin), pos, embed_dim, num_heads,
        num_kv_heads, head_dim, cache_capacity, eps, _ptr(scratch), scratch_bytes, _stream(stream))


def ck_decode_layer_devpos(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                           rope_sin, d_pos, embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int,
                           cache_capacity: int, eps: float, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().ck_decode_layer_devpos(
        _ptr(out), _ptr(x), _ptr(residual), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(bq), _ptr(bk),
        _ptr(bv), _ptr(bo), _ptr(k_cache), _ptr(v_cache), _ptr(rope_cos), _ptr(rope_sin), _ptr(d_pos), embed_dim,
        num_heads, num_kv_heads, head_dim, cache_capacity, eps, _ptr(scratch), scratch_bytes, _stream(stream))


def ck_device_status(stream=None) -> tuple[int, int]:
    """(call status, device status): the device status word, read and cleared."""
    v = ctypes.c_int(0)
    rc = lib().ck_device_status(ctypes.addressof(v), _stream(stream))
    return rc, v.value


CK_TAP_Q, CK_TAP_XQ8, CK_TAP_ATTN, CK_TAP_AQ8 = 0, 1, 2, 3


def ck_decode_layer_scratch_offset(tap: int, embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                   cache_capacity: int) -> int:
    return lib().ck_decode_layer_scratch_offset(tap, embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity)


def ck_decode_layer_batched_scratch_size(batch: int, embed_dim: int, num_heads: int, num_kv_heads: int,
                                        head_dim: int, cache_capacity: int) -> int:
    return lib().ck_decode_layer_batched_scratch_size(batch, embed_dim, num_heads, num_kv_heads, head_dim,
                                                      cache_capacity)


def ck_decode_layer_batched(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_caches, v_caches, rope_cos,
                            rope_sin, d_pos, batch: int, embed_dim: int, num_heads: int, num_kv_heads: int,
                            head_dim: int, cache_capacity: int, eps: float, scratch, scratch_bytes: int,
                            stream=None) -> int:
    """k_caches / v_caches: device arrays of `batch` cache pointers (e.g. int64 tensors of data_ptr()s)."""
    return lib().ck_decode_layer_batched(
        _ptr(out), _ptr(x), _ptr(residual), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(bq), _ptr(bk),
        _ptr(bv), _ptr(bo), _ptr(k_caches), _ptr(v_caches), _ptr(rope_cos), _ptr(rope_sin), _ptr(d_pos), batch,
        embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps, _ptr(scratch), scratch_bytes,
        _stream(stream))


def ck_decode_layer_batched_scratch_offset(tap: int, batch: int, embed_dim: int, num_heads: int, num_kv_heads: int,
                                           head_dim: int, cache_capacity: int) -> int:
    return lib().ck_decode_layer_batched_scratch_offset(tap, batch, embed_dim, num_heads, num_kv_heads, head_dim,
                                                        cache_capacity)


def ck_prefill_layer_devpos(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos,
                            rope_sin, d_pos, n_tokens: int, embed_dim: int, num_heads: int, num_kv_heads: int,
                            head_dim: int, cache_capacity: int, eps: float, scratch, scratch_bytes: int,
                            stream=None) -> int:
    """ck_prefill_layer with the chunk's first position in device memory (int32 tensor)."""
    return lib().ck_prefill_layer_devpos(
        _ptr(out), _ptr(x), _ptr(residual), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(bq), _ptr(bk),
        _ptr(bv), _ptr(bo), _ptr(k_cache), _ptr(v_cache), _ptr(rope_cos), _ptr(rope_sin), _ptr(d_pos), n_tokens,
        embed_dim, num_heads, num_kv_heads, head_dim, cache_capacity, eps, _ptr(scratch), scratch_bytes,
        _stream(stream))


def ck_attn_prefill_scratch_size(num_heads: int, num_kv_heads: int, head_dim: int, cache_capacity: int) -> int:
    return lib().ck_attn_prefill_scratch_size(num_heads, num_kv_heads, head_dim, cache_capacity)


def ck_attn_prefill_gqa(q_, k_cache, v_cache, out, pos: int, n_tokens: int, num_heads: int, num_kv_heads: int,
                        head_dim: int, cache_capacity: int, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().ck_attn_prefill_gqa(_ptr(q_), _ptr(k_cache), _ptr(v_cache), _ptr(out), pos, n_tokens, num_heads,
                                     num_kv_heads, head_dim, cache_capacity, _ptr(scratch), scratch_bytes,
                                     _stream(stream))


def ck_attn_split_scratch_size(num_heads: int, num_kv_heads: int, head_dim: int, splits: int) -> int:
    return lib().ck_attn_split_scratch_size(num_heads, num_kv_heads, head_dim, splits)


def ck_attn_decode_gqa_split(q_, k_cache, v_cache, out, num_heads: int, num_kv_heads: int, kv_tokens: int,
                             cache_capacity: int, head_dim: int, kv_dtype: int, k_scale: float, v_scale: float,
                             splits: int, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().ck_attn_decode_gqa_split(_ptr(q_), _ptr(k_cache), _ptr(v_cache), _ptr(out), num_heads, num_kv_heads,
                                          kv_tokens, cache_capacity, head_dim, kv_dtype, k_scale, v_scale, splits,
                                          _ptr(scratch), scratch_bytes, _stream(stream))


def ck_prefill_layer_scratch_size(n_tokens: int, embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                  cache_capacity: int) -> int:
    return lib().ck_prefill_layer_scratch_size(n_tokens, embed_dim, num_heads, num_kv_heads, head_dim,
                                               cache_capacity)


def ck_prefill_layer_scratch_offset(tap: int, n_tokens: int, embed_dim: int, num_heads: int, num_kv_heads: int,
                                    head_dim: int, cache_capacity: int) -> int:
    return lib().ck_prefill_layer_scratch_offset(tap, n_tokens, embed_dim, num_heads, num_kv_heads, head_dim,
                                                 cache_capacity)


def ck_prefill_layer(out, x, residual, wq, wk, wv, wo, gamma, bq, bk, bv, bo, k_cache, v_cache, rope_cos, rope_sin,
                     pos: int, n_tokens: int, embed_dim: int, num_heads: int, num_kv_heads: int, head_dim: int,
                     cache_capacity: int, eps: float, scratch, scratch_bytes: int, stream=None) -> int:
    """n_tokens consecutive tokens of one sequence at positions pos.. (causal); x / out [n_tokens, embed_dim]."""
    return lib().ck_prefill_layer(
        _ptr(out), _ptr(x), _ptr(residual), _ptr(wq), _ptr(wk), _ptr(wv), _ptr(wo), _ptr(gamma), _ptr(bq), _ptr(bk),
        _ptr(bv), _ptr(bo), _ptr(k_cache), _ptr(v_cache), _ptr(rope_cos), _ptr(rope_sin), pos, n_tokens, embed_dim,
        num_heads, num_kv_heads, head_dim, cache_capacity, eps, _ptr(scratch), scratch_bytes, _stream(stream))


def ck_block_dots_q5_0_q8_0(isum, W, x_q8, M: int, K: int, stream=None) -> int:
    return lib().ck_block_dots_q5_0_q8_0(_ptr(isum), _ptr(W), _ptr(x_q8), M, K, _stream(stream))


def ck_block_dots_q8_0_q8_0(isum, W, x_q8, M: int, K: int, stream=None) -> int:
    return lib().ck_block_dots_q8_0_q8_0(_ptr(isum), _ptr(W), _ptr(x_q8), M, K, _stream(stream))
