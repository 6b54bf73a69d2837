"""Seeded synthetic inputs for the decode-attention layer.

This module draws inputs only.  It holds no step of the decode path: the
weight packers below turn fp32 draws into Q5_0 / Q8_0 *input bytes* (the
decode step receives weights already quantized and never packs them), and
the RoPE tables are inputs the caller passes in.  Both the CUDA path (through
the tests and the benchmark) and the oracle (through the tests) consume what
it makes; it imports neither.

Recipe (one numpy ``Generator(PCG64(seed))`` per workload, draws in this
order): gamma = 1 + N(0, 0.1); Wq, Wk, Wv, Wo fp32 N(0, 0.02) then packed;
bq, bk, bv, bo N(0, 0.01); x N(0, 1); K cache then V cache N(0, 1) in rows
0 .. pos-1 of each KV head (rows >= pos are zero).  The batched workload
draws its per-sequence lengths first.  Block formats: Q5_0 = 22 bytes
{fp16 d, u32 qh, 16 bytes of nibbles}, code q in [0, 31], weight (q-16)*d;
Q8_0 = 34 bytes {fp16 d, 32 x int8}, weight q*d; element j < 16 of a Q5_0
block sits in the low nibble of byte j and bit j of qh, element j + 16 in the
high nibble of byte j and bit j + 16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK = 32
Q5_0_BYTES = 22
Q8_0_BYTES = 34


# --------------------------------------------------------------------------
# Workloads.  Shapes follow a Qwen2-family attention layer: D=256 tiny,
# D=896 with 14/2 heads and D=3584 with 28/4 heads, head_dim 64 / 64 / 128.
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    D: int
    H: int
    KV: int
    hd: int
    pos: int            # position of the new token = rows already in the cache
    capacity: int       # cache rows per KV head
    theta: float
    seed: int
    layers: int = 1
    batch: int = 1      # independent sequences (batched workload)
    kv_lo: int = 0      # batched: per-sequence lengths uniform in [kv_lo, kv_hi]
    kv_hi: int = 0
    eps: float = 1e-6

    @property
    def QD(self):
        return self.H * self.hd

    @property
    def KD(self):
        return self.KV * self.hd

    def weight_bytes(self) -> int:
        """Bytes of the four quantized weight matrices of one layer."""
        nb_d, nb_q = self.D // QK, self.QD // QK
        return (self.QD * nb_d * Q5_0_BYTES + self.KD * nb_d * Q5_0_BYTES + self.KD * nb_d * Q8_0_BYTES
                + self.D * nb_q * Q5_0_BYTES)

    def kv_read_bytes(self, tokens: int) -> int:
        """Bytes of K and V cache rows read to attend over ``tokens`` rows."""
        return tokens * self.KD * 4 * 2


WORKLOADS = {
    "tiny": Workload("tiny", 256, 4, 2, 64, pos=16, capacity=64, theta=1e4, seed=0),
    "small1k": Workload("small1k", 896, 14, 2, 64, pos=1024, capacity=2048, theta=1e6, seed=1),
    "7b8k": Workload("7b8k", 3584, 28, 4, 128, pos=8192, capacity=8192 + 64, theta=1e6, seed=2),
    "stack32k": Workload("stack32k", 3584, 28, 4, 128, pos=32768, capacity=32768 + 64, theta=1e6, seed=3,
                         layers=28),
    "batched64": Workload("batched64", 3584, 28, 4, 128, pos=0, capacity=16384 + 64, theta=1e6, seed=4,
                          batch=64, kv_lo=512, kv_hi=16384),
}


# --------------------------------------------------------------------------
# Input packers (fp32 draws -> block bytes).  Input synthesis only.
# --------------------------------------------------------------------------
def pack_q5_0(codes: np.ndarray, d16: np.ndarray) -> np.ndarray:
    """codes uint8 [n, 32] in [0, 31], d16 uint16 [n] -> bytes [n, 22]."""
    c = np.asarray(codes, np.uint32).reshape(-1, QK)
    n = c.shape[0]
    out = np.zeros((n, Q5_0_BYTES), np.uint8)
    d = np.asarray(d16, np.uint16).reshape(n)
    out[:, 0] = d & 0xFF
    out[:, 1] = d >> 8
    qh = np.zeros(n, np.uint32)
    for j in range(QK):
        qh |= ((c[:, j] >> 4) & 1) << np.uint32(j)
    for i in range(4):
        out[:, 2 + i] = (qh >> np.uint32(8 * i)) & 0xFF
    out[:, 6:22] = ((c[:, :16] & 0xF) | ((c[:, 16:] & 0xF) << 4)).astype(np.uint8)
    return out


def pack_q8_0(codes: np.ndarray, d16: np.ndarray) -> np.ndarray:
    """codes int8 [n, 32], d16 uint16 [n] -> bytes [n, 34]."""
    c = np.asarray(codes, np.int8).reshape(-1, QK)
    n = c.shape[0]
    out = np.zeros((n, Q8_0_BYTES), np.uint8)
    d = np.asarray(d16, np.uint16).reshape(n)
    out[:, 0] = d & 0xFF
    out[:, 1] = d >> 8
    out[:, 2:] = c.view(np.uint8)
    return out


def weights_to_q5_0(w: np.ndarray) -> np.ndarray:
    """fp32 [M, K] -> Q5_0 bytes [M, K/32 * 22].

    Per block: m = the element of largest magnitude (first on ties), d = -m/16,
    code = min(31, trunc(x/d + 16.5)); uses the full code range [0, 31].
    """
    M, K = w.shape
    b = w.astype(np.float32).reshape(-1, QK)
    idx = np.argmax(np.abs(b), axis=1)
    m = b[np.arange(b.shape[0]), idx]
    d = (m / np.float32(-16.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    q = np.minimum(31, np.trunc(b * inv[:, None] + np.float32(16.5))).astype(np.int64)
    q = np.clip(q, 0, 31).astype(np.uint8)
    d16 = d.astype(np.float16).view(np.uint16)
    return pack_q5_0(q, d16).reshape(M, K // QK * Q5_0_BYTES)


def weights_to_q8_0(w: np.ndarray) -> np.ndarray:
    """fp32 [M, K] -> Q8_0 bytes [M, K/32 * 34] (d = amax/127, codes rounded half-to-even)."""
    M, K = w.shape
    b = w.astype(np.float32).reshape(-1, QK)
    d = (np.abs(b).max(axis=1) / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(d[:, None] != 0, np.rint(b / d[:, None]), 0)
    q = np.clip(q, -127, 127).astype(np.int8)
    d16 = d.astype(np.float16).view(np.uint16)
    return pack_q8_0(q, d16).reshape(M, K // QK * Q8_0_BYTES)


def random_q5_0(rng: np.random.Generator, M: int, K: int, d_scale: float = 1e-3) -> np.ndarray:
    """Uniformly random codes and qh bits with positive and negative fp16 scales."""
    n = M * K // QK
    codes = rng.integers(0, 32, size=(n, QK), dtype=np.uint8)
    d = (rng.uniform(0.25, 1.0, n) * d_scale * rng.choice([-1.0, 1.0], n)).astype(np.float16)
    return pack_q5_0(codes, d.view(np.uint16)).reshape(M, K // QK * Q5_0_BYTES)


def random_q8_0(rng: np.random.Generator, M: int, K: int, d_scale: float = 1e-3) -> np.ndarray:
    n = M * K // QK
    codes = rng.integers(-128, 128, size=(n, QK), dtype=np.int16).astype(np.int8)
    d = (rng.uniform(0.25, 1.0, n) * d_scale * rng.choice([-1.0, 1.0], n)).astype(np.float16)
    return pack_q8_0(codes, d.view(np.uint16)).reshape(M, K // QK * Q8_0_BYTES)


def rope_tables(capacity: int, hd: int, theta: float):
    """cos/sin [capacity, hd/2] fp32: angle p * theta^(-2i/hd), computed in double."""
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.arange(capacity, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# --------------------------------------------------------------------------
# One layer's inputs.
# --------------------------------------------------------------------------
@dataclass
class LayerInputs:
    gamma: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    wv: np.ndarray
    wo: np.ndarray
    bq: np.ndarray
    bk: np.ndarray
    bv: np.ndarray
    bo: np.ndarray
    x: np.ndarray
    k_cache: np.ndarray   # [KV, capacity, hd]
    v_cache: np.ndarray
    extra: dict = field(default_factory=dict)


def _normal(rng, shape, std, mean=0.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std) + np.float32(mean)).astype(np.float32)


def draw_weights(rng: np.random.Generator, w: Workload):
    gamma = _normal(rng, w.D, 0.1, 1.0)
    wq = weights_to_q5_0(_normal(rng, (w.QD, w.D), 0.02))
    wk = weights_to_q5_0(_normal(rng, (w.KD, w.D), 0.02))
    wv = weights_to_q8_0(_normal(rng, (w.KD, w.D), 0.02))
    wo = weights_to_q5_0(_normal(rng, (w.D, w.QD), 0.02))
    bq = _normal(rng, w.QD, 0.01)
    bk = _normal(rng, w.KD, 0.01)
    bv = _normal(rng, w.KD, 0.01)
    bo = _normal(rng, w.D, 0.01)
    return gamma, wq, wk, wv, wo, bq, bk, bv, bo


def draw_cache(rng: np.random.Generator, w: Workload, filled: int):
    kc = np.zeros((w.KV, w.capacity, w.hd), np.float32)
    vc = np.zeros((w.KV, w.capacity, w.hd), np.float32)
    kc[:, :filled, :] = _normal(rng, (w.KV, filled, w.hd), 1.0)
    vc[:, :filled, :] = _normal(rng, (w.KV, filled, w.hd), 1.0)
    return kc, vc


def make_layer(w: Workload, rng: np.random.Generator | None = None, pos: int | None = None) -> LayerInputs:
    """All inputs of one decode step of one layer at ``pos`` (default: the workload's)."""
    rng = rng if rng is not None else np.random.Generator(np.random.PCG64(w.seed))
    pos = w.pos if pos is None else pos
    gamma, wq, wk, wv, wo, bq, bk, bv, bo = draw_weights(rng, w)
    x = _normal(rng, w.D, 1.0)
    kc, vc = draw_cache(rng, w, pos)
    return LayerInputs(gamma, wq, wk, wv, wo, bq, bk, bv, bo, x, kc, vc)


def batched_lengths(w: Workload, rng: np.random.Generator) -> np.ndarray:
    """Per-sequence prior lengths (= each sequence's pos), uniform in [kv_lo, kv_hi]."""
    return rng.integers(w.kv_lo, w.kv_hi + 1, size=w.batch).astype(np.int32)
