"""Pins of the oracle's multi-token (prefill) layer, no GPU.

The prefill form is checked against facts outside its own code:
- one token is the decode layer (pinned on its own in test_oracle_pins);
- n tokens equal n decode steps taken one after the other, so a wrong causal
  row count, position or store row fails;
- its attention tap equals a dense causal-masked softmax written with numpy
  matrix products in float64;
- outputs and cache rows of early tokens do not move when later tokens change;
- zero weights give each token its own residual row.
"""
import numpy as np

import oracle
from quantized_weight_attention_gb300 import synth


def _case(n, seed=0):
    w = synth.WORKLOADS["tiny"]
    rng = np.random.Generator(np.random.PCG64(seed))
    L = synth.make_layer(w, rng)
    X = rng.standard_normal((n, w.D)).astype(np.float32)
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    return w, L, X, cos, sin


def _prefill(w, L, X, cos, sin, res=None, taps=False, kc=None, vc=None):
    kc = L.k_cache.copy() if kc is None else kc
    vc = L.v_cache.copy() if vc is None else vc
    r = oracle.prefill_layer(X, X if res is None else res, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv,
                             L.bo, kc, vc, cos, sin, w.pos, X.shape[0], w.D, w.H, w.KV, w.hd, w.capacity, w.eps,
                             taps=taps)
    return r, kc, vc


def test_prefill_one_token_is_the_decode_layer():
    w, L, X, cos, sin = _case(1)
    out, kc, vc = _prefill(w, L, X, cos, sin)
    kc2, vc2 = L.k_cache.copy(), L.v_cache.copy()
    ref = oracle.decode_layer(X[0], X[0], L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc2, vc2,
                              cos, sin, w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
    assert np.array_equal(out[0], ref)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def test_prefill_equals_sequential_decode_steps():
    n = 9
    w, L, X, cos, sin = _case(n, seed=1)
    out, kc, vc = _prefill(w, L, X, cos, sin)
    kc2, vc2 = L.k_cache.copy(), L.v_cache.copy()
    for i in range(n):
        ref = oracle.decode_layer(X[i], X[i], L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc2, vc2,
                                  cos, sin, w.pos + i, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
        assert np.array_equal(out[i], ref), i
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)


def test_prefill_attention_is_dense_causal_softmax():
    n = 12
    w, L, X, cos, sin = _case(n, seed=2)
    (out, t), kc, vc = _prefill(w, L, X, cos, sin, taps=True)
    G, hd, T = w.H // w.KV, w.hd, w.pos + n
    # the stored rows are the k / v taps; rows past the chunk are untouched
    for i in range(n):
        assert np.array_equal(kc[:, w.pos + i].reshape(-1), t["k"][i])
        assert np.array_equal(vc[:, w.pos + i].reshape(-1), t["v"][i])
    assert np.array_equal(kc[:, T:], L.k_cache[:, T:]) and np.array_equal(vc[:, T:], L.v_cache[:, T:])
    Q = t["q"].astype(np.float64).reshape(n, w.H, hd)
    # query token i sits at row pos + i and may see rows 0 .. pos + i
    mask = np.arange(T)[None, :] > (w.pos + np.arange(n))[:, None]
    for h in range(w.H):
        K = kc[h // G, :T].astype(np.float64)
        V = vc[h // G, :T].astype(np.float64)
        S = (Q[:, h] @ K.T) / np.sqrt(hd)
        S[mask] = -np.inf
        P = np.exp(S - S.max(axis=1, keepdims=True))
        O = (P @ V) / P.sum(axis=1, keepdims=True)
        got = t["attn"].reshape(n, w.H, hd)[:, h].astype(np.float64)
        np.testing.assert_allclose(got, O, rtol=2e-6, atol=1e-6 * np.abs(O).max())
    # a mask off by one (token i seeing row pos + i + 1) moves the result
    S = (Q[:, 0] @ kc[0, :T].astype(np.float64).T) / np.sqrt(hd)
    S[np.arange(T)[None, :] > (w.pos + np.arange(n) + 1)[:, None]] = -np.inf
    P = np.exp(S - S.max(axis=1, keepdims=True))
    wrong = (P @ vc[0, :T].astype(np.float64)) / P.sum(axis=1, keepdims=True)
    assert np.abs(t["attn"].reshape(n, w.H, hd)[:-1, 0] - wrong[:-1]).max() > 1e-3


def test_prefill_is_causal():
    n = 10
    w, L, X, cos, sin = _case(n, seed=3)
    out, kc, vc = _prefill(w, L, X, cos, sin)
    for i in (0, 4, 8):
        X2 = X.copy()
        X2[i + 1:] = np.random.default_rng(10 + i).standard_normal((n - i - 1, w.D)).astype(np.float32)
        out2, kc2, vc2 = _prefill(w, L, X2, cos, sin)
        assert np.array_equal(out2[:i + 1], out[:i + 1])
        assert not np.array_equal(out2[i + 1:], out[i + 1:])
        assert np.array_equal(kc2[:, :w.pos + i + 1], kc[:, :w.pos + i + 1])
        assert np.array_equal(vc2[:, :w.pos + i + 1], vc[:, :w.pos + i + 1])


def test_prefill_zero_weights_give_each_token_its_residual():
    n = 5
    w, L, X, cos, sin = _case(n, seed=4)
    res = np.random.default_rng(5).standard_normal((n, w.D)).astype(np.float32)
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    out = oracle.prefill_layer(X, res, np.zeros_like(L.wq), np.zeros_like(L.wk), np.zeros_like(L.wv),
                               np.zeros_like(L.wo), L.gamma, None, None, None, None, kc, vc, cos, sin, w.pos, n,
                               w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
    assert np.array_equal(out, res)
    assert not kc[:, w.pos:w.pos + n].any() and not vc[:, w.pos:w.pos + n].any()
