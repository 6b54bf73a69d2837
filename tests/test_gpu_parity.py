"""Parity of the CUDA path (through the C ABI) with the oracle, on one GPU.

Bit-exact: Q8_0 quantization bytes, per-block int32 dots, the quantized
activations inside the layer, RoPE and the KV store.  Floating point (GEMV
outputs, q, attention output, stored rows, layer output): max |err| <=
1e-3 * max |ref| and relative L2 error <= 1e-4.  Shapes span several tiles,
ragged tails and the degenerate cases (one cache row, a full cache, MHA)."""
import numpy as np
import pytest

import oracle
from quantized_weight_attention_gb300 import synth

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


# --------------------------------------------------------------------------
# Q8_0 quantization: bit-exact
# --------------------------------------------------------------------------
def _quant_cases():
    rng = np.random.default_rng(100)
    cases = [rng.standard_normal(32).astype(np.float32),
             (rng.standard_normal(3584) * 3).astype(np.float32),
             (rng.standard_normal(32 * 1001) * rng.uniform(1e-4, 1e3, 1001).repeat(32)).astype(np.float32)]
    ties = np.zeros((64, 32), np.float32)
    ties[:, 0] = 127.0
    ties[:, 1:] = (rng.integers(-126, 126, (64, 31)) + 0.5).astype(np.float32)
    cases.append(ties.ravel())
    z = np.zeros(96, np.float32)
    z[64:] = 1e-30                         # fp16 scale underflows to 0
    z[32:64] = np.linspace(-1e7, 1e7, 32)  # fp16 scale overflows to inf
    cases.append(z)
    return cases


@pytest.mark.parametrize("ci", range(5))
def test_quantize_q8_0_bitexact(dev, ci):
    x = _quant_cases()[ci]
    y = torch.empty(x.size // 32 * 34, dtype=torch.uint8, device=dev)
    ok(q.ck_quantize_q8_0(T(x, dev), y, x.size))
    assert np.array_equal(H(y), oracle.quantize_q8_0(x))


# --------------------------------------------------------------------------
# block dots (bit-exact) and GEMV (tolerance)
# --------------------------------------------------------------------------
SHAPES = [(1, 32), (7, 96), (33, 256), (64, 896), (130, 3584), (512, 3584), (3584, 3584), (5, 8192)]


def _wx(M, K, q8, seed):
    rng = np.random.default_rng(seed)
    W = synth.random_q8_0(rng, M, K) if q8 else synth.random_q5_0(rng, M, K)
    xq = synth.random_q8_0(rng, 1, K, d_scale=1e-1).ravel()
    return W, xq


@pytest.mark.parametrize("q8", [False, True])
@pytest.mark.parametrize("M,K", SHAPES)
def test_block_dots_bitexact(dev, M, K, q8):
    W, xq = _wx(M, K, q8, 7 * M + K + q8)
    isum = torch.empty((M, K // 32), dtype=torch.int32, device=dev)
    f = q.ck_block_dots_q8_0_q8_0 if q8 else q.ck_block_dots_q5_0_q8_0
    ok(f(isum, T(W, dev), T(xq, dev), M, K))
    assert np.array_equal(H(isum), oracle.block_dots(W, xq, M, K, q8))


@pytest.mark.parametrize("q8", [False, True])
@pytest.mark.parametrize("M,K", SHAPES + [(4608, 3584), (896, 896)])
def test_gemv_parity(dev, M, K, q8):
    W, xq = _wx(M, K, q8, 11 * M + K + q8)
    bias = np.random.default_rng(M).standard_normal(M).astype(np.float32) * 0.01
    f = q.ck_gemv_q8_0_q8_0 if q8 else q.ck_gemv_q5_0_q8_0
    Wd, xd = T(W, dev), T(xq, dev)
    y = torch.empty(M, dtype=torch.float32, device=dev)
    ok(f(y, Wd, xd, T(bias, dev), M, K))
    assert_close(H(y), oracle.gemv(W, xq, bias, M, K, q8), f"gemv {M}x{K} q8={q8}")
    ok(f(y, Wd, xd, None, M, K))
    assert_close(H(y), oracle.gemv(W, xq, None, M, K, q8), f"gemv nobias {M}x{K}")


def test_gemv_realistic_weights(dev):
    """Weights quantized from N(0, 0.02) and an activation quantized from N(0, 1)."""
    rng = np.random.default_rng(3)
    M, K = 3584, 3584
    W = synth.weights_to_q5_0(rng.standard_normal((M, K)).astype(np.float32) * 0.02)
    xq = oracle.quantize_q8_0(rng.standard_normal(K).astype(np.float32))
    y = torch.empty(M, dtype=torch.float32, device=dev)
    ok(q.ck_gemv_q5_0_q8_0(y, T(W, dev), T(xq, dev), None, M, K))
    assert_close(H(y), oracle.gemv(W, xq, None, M, K, False), "realistic gemv")


# --------------------------------------------------------------------------
# RoPE and KV store: bit-exact (same fp32 operations, no contraction)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("Hh,KV,hd,C,pos", [(4, 2, 64, 64, 16), (28, 4, 128, 8256, 8192), (3, 0, 2, 5, 4),
                                            (14, 2, 64, 2048, 0)])
def test_rope_bitexact(dev, Hh, KV, hd, C, pos):
    rng = np.random.default_rng(hd + pos)
    cos, sin = synth.rope_tables(C, hd, 1e6)
    qv = rng.standard_normal(Hh * hd).astype(np.float32)
    kv = rng.standard_normal(max(KV, 1) * hd).astype(np.float32)[:KV * hd]
    qd, kd = T(qv, dev), (T(kv, dev) if KV else None)
    ok(q.ck_rope_inplace(qd, kd, T(cos, dev), T(sin, dev), pos, Hh, KV, hd, C))
    rq, rk = oracle.rope(qv, kv if KV else None, cos, sin, pos, Hh, KV, hd)
    assert np.array_equal(H(qd), rq)
    if KV:
        assert np.array_equal(H(kd), rk)


def test_kv_store_bitexact(dev):
    rng = np.random.default_rng(1)
    KV, C, hd, pos = 4, 100, 128, 77
    kc = rng.standard_normal((KV, C, hd)).astype(np.float32)
    vc = rng.standard_normal((KV, C, hd)).astype(np.float32)
    k = rng.standard_normal(KV * hd).astype(np.float32)
    v = rng.standard_normal(KV * hd).astype(np.float32)
    kcd, vcd = T(kc, dev), T(vc, dev)
    ok(q.ck_kv_store(kcd, vcd, T(k, dev), T(v, dev), pos, KV, C, hd))
    oracle.kv_store(kc, vc, k, v, pos, KV, C, hd)
    assert np.array_equal(H(kcd), kc) and np.array_equal(H(vcd), vc)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
ATT = [(4, 2, 64, 17, 64), (14, 2, 64, 1025, 2048), (28, 4, 128, 8193, 8256), (8, 8, 32, 5, 8),
       (6, 2, 96, 100, 128), (8, 1, 256, 300, 512), (4, 4, 128, 33, 33), (2, 1, 64, 64, 64), (7, 1, 128, 4097, 5000)]
# Splits long enough (at 8 KV heads) for the ~16 KB stages of every head_dim,
# each ending in a partial stage; rows past kv_tokens are NaN.
ATT_LONG = [(16, 8, 32, 20011, 20016), (56, 8, 64, 10003, 10010), (24, 8, 96, 6203, 6210), (64, 8, 128, 5011, 5016),
            (8, 8, 256, 2517, 2520)]


def _attn_case(Hh, KV, hd, Tn, C, seed):
    rng = np.random.default_rng(seed)
    kc = np.zeros((KV, C, hd), np.float32)
    vc = np.zeros((KV, C, hd), np.float32)
    kc[:, :Tn] = rng.standard_normal((KV, Tn, hd))
    vc[:, :Tn] = rng.standard_normal((KV, Tn, hd))
    if C > Tn:  # rows past kv_tokens must never be read
        kc[:, Tn:] = np.nan
        vc[:, Tn:] = np.nan
    qv = rng.standard_normal(Hh * hd).astype(np.float32)
    return qv, kc, vc


def _gpu_attn(dev, qv, kc, vc, Hh, KV, hd, Tn, C):
    nbytes = q.ck_attn_scratch_size(Hh, KV, C, hd)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(Hh * hd, dtype=torch.float32, device=dev)
    ok(q.ck_attn_decode_gqa(T(qv, dev), T(kc, dev), T(vc, dev), out, Hh, KV, Tn, C, hd, scratch, nbytes))
    return H(out)


@pytest.mark.parametrize("Hh,KV,hd,Tn,C", ATT + ATT_LONG)
def test_attention_parity(dev, Hh, KV, hd, Tn, C):
    qv, kc, vc = _attn_case(Hh, KV, hd, Tn, C, Hh * 1000 + Tn)
    got = _gpu_attn(dev, qv, kc, vc, Hh, KV, hd, Tn, C)
    ref = oracle.attention(qv, np.nan_to_num(kc), np.nan_to_num(vc), Hh, KV, Tn, C, hd)
    assert_close(got, ref, f"attention {Hh}/{KV} hd={hd} T={Tn}")


def test_attention_single_row_is_v_exactly(dev):
    Hh, KV, hd, C = 28, 4, 128, 16
    qv, kc, vc = _attn_case(Hh, KV, hd, 1, C, 5)
    got = _gpu_attn(dev, qv, kc, vc, Hh, KV, hd, 1, C).reshape(Hh, hd)
    for h in range(Hh):
        assert np.array_equal(got[h], vc[h * KV // Hh, 0])


# --------------------------------------------------------------------------
# the layer
# --------------------------------------------------------------------------
class GpuLayer:
    def __init__(self, dev, w, L, cos, sin):
        self.dev, self.w = dev, w
        t = lambda a: T(a, dev)
        self.x, self.gamma = t(L.x), t(L.gamma)
        self.wq, self.wk, self.wv, self.wo = t(L.wq), t(L.wk), t(L.wv), t(L.wo)
        self.bq, self.bk, self.bv, self.bo = t(L.bq), t(L.bk), t(L.bv), t(L.bo)
        self.kc, self.vc = t(L.k_cache), t(L.v_cache)
        self.cos, self.sin = t(cos), t(sin)
        self.out = torch.empty(w.D, dtype=torch.float32, device=dev)
        self.nbytes = q.ck_decode_layer_scratch_size(w.D, w.H, w.KV, w.hd, w.capacity)
        self.scratch = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    def args(self, x=None, residual=None):
        x = self.x if x is None else x
        r = x if residual is None else residual
        return (self.out, x, r, self.wq, self.wk, self.wv, self.wo, self.gamma, self.bq, self.bk, self.bv, self.bo,
                self.kc, self.vc, self.cos, self.sin)

    def run(self, pos, x=None):
        w = self.w
        ok(q.ck_decode_layer(*self.args(x), pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, self.scratch,
                             self.nbytes))

    def tap(self, which, n, dtype):
        w = self.w
        off = q.ck_decode_layer_scratch_offset(which, w.D, w.H, w.KV, w.hd, w.capacity)
        nb = n * np.dtype(dtype).itemsize
        return self.scratch[off:off + nb].cpu().numpy().view(dtype)


def _layer_inputs(name, pos=None, seed=None):
    w = synth.WORKLOADS[name]
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    L = synth.make_layer(w, rng, pos=pos)
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    return w, L, cos, sin


@pytest.mark.parametrize("name", ["tiny", "small1k", "7b8k"])
def test_layer_parity(dev, name):
    w, L, cos, sin = _layer_inputs(name)
    g = GpuLayer(dev, w, L, cos, sin)
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    ref, taps = oracle.decode_layer(L.x, L.x, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc, cos,
                                    sin, w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, taps=True)
    g.run(w.pos)
    out = H(g.out)
    # the quantized normed activation: bit-exact
    assert np.array_equal(g.tap(q.CK_TAP_XQ8, w.D // 32 * 34, np.uint8), taps["xq"])
    assert_close(g.tap(q.CK_TAP_Q, w.QD, np.float32), taps["q"], "q")
    # stored rows (k after RoPE, v) and untouched rows
    gk, gv = H(g.kc), H(g.vc)
    assert_close(gk[:, w.pos].ravel(), taps["k"], "stored k")
    assert_close(gv[:, w.pos].ravel(), taps["v"], "stored v")
    others = np.arange(w.capacity) != w.pos
    assert np.array_equal(gk[:, others], kc[:, others]) and np.array_equal(gv[:, others], vc[:, others])
    attn = g.tap(q.CK_TAP_ATTN, w.QD, np.float32)
    assert_close(attn, taps["attn"], "attention output")
    # the O-projection input is the oracle quantizer applied to the GPU's own attention output
    aq = g.tap(q.CK_TAP_AQ8, w.QD // 32 * 34, np.uint8)
    assert np.array_equal(aq, oracle.quantize_q8_0(attn))
    assert_close(out, ref, f"layer output {name}")
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0


def test_layer_decode_sequence_graph_devpos(dev):
    """Four successive tokens replayed from one captured graph (position read
    on the device) match the oracle's sequential decode, and a replay equals
    an eager call bit for bit."""
    w, L, cos, sin = _layer_inputs("tiny", pos=10)
    g = GpuLayer(dev, w, L, cos, sin)
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    d_pos = torch.zeros(1, dtype=torch.int32, device=dev)
    x_in = torch.empty(w.D, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        d_pos.fill_(10)  # warm-up call outside capture (state restored below)
        ok(q.ck_decode_layer_devpos(*g.args(x_in), d_pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, g.scratch,
                                    g.nbytes, s))
    torch.cuda.synchronize()
    g.kc.copy_(T(L.k_cache, dev))
    g.vc.copy_(T(L.v_cache, dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        ok(q.ck_decode_layer_devpos(*g.args(x_in), d_pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, g.scratch,
                                    g.nbytes, s))
    rng = np.random.default_rng(77)
    for step in range(4):
        pos = 10 + step
        xs = rng.standard_normal(w.D).astype(np.float32)
        x_in.copy_(T(xs, dev))
        d_pos.fill_(pos)
        graph.replay()
        got = H(g.out)
        ref = oracle.decode_layer(xs, xs, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc, cos, sin,
                                  pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
        assert_close(got, ref, f"graph step {step}")
    # replay == eager, bit for bit, from the same state
    kc0, vc0 = g.kc.clone(), g.vc.clone()
    d_pos.fill_(20)
    graph.replay()
    o_graph = H(g.out).copy()
    k_graph = H(g.kc).copy()
    g.kc.copy_(kc0)
    g.vc.copy_(vc0)
    g.run(20, x_in)
    assert np.array_equal(H(g.out), o_graph) and np.array_equal(H(g.kc), k_graph)


def test_chained_steps_in_one_graph_match_eager(dev):
    """Several 7B-shaped steps over independent copies captured in one graph,
    so each step's kernels launch early behind the previous step's.  Every
    attention CTA here streams more tiles than its ring has stages.  The
    replays must finish with a clean device status and equal the eager
    results bit for bit."""
    w, L, cos, sin = _layer_inputs("7b8k")
    copies = [GpuLayer(dev, w, L, cos, sin) for _ in range(3)]
    for g in copies:
        g.run(w.pos)
    torch.cuda.synchronize()
    eager = [H(g.out).copy() for g in copies]
    q.ck_device_status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for g in copies:
            ok(q.ck_decode_layer(*g.args(), w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, g.scratch, g.nbytes, s))
    for g in copies:
        g.out.zero_()
    for _ in range(30):
        graph.replay()
    torch.cuda.synchronize()
    rc, st = q.ck_device_status()
    assert rc == q.CK_OK and st == q.CK_OK, st
    for g, e in zip(copies, eager):
        assert np.array_equal(H(g.out), e)


def test_layer_devpos_out_of_range_writes_nothing(dev):
    w, L, cos, sin = _layer_inputs("tiny")
    g = GpuLayer(dev, w, L, cos, sin)
    g.out.fill_(7.0)
    d_pos = torch.full((1,), w.capacity, dtype=torch.int32, device=dev)
    q.ck_device_status()
    ok(q.ck_decode_layer_devpos(*g.args(), d_pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, g.scratch, g.nbytes))
    assert np.all(H(g.out) == 7.0)
    assert np.array_equal(H(g.kc), L.k_cache) and np.array_equal(H(g.vc), L.v_cache)
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    assert q.ck_device_status()[1] == 0


def test_layer_edge_positions(dev):
    """pos = 0 (attends one row) and pos = capacity - 1 (the full cache)."""
    for pos in (0, 63):
        w, L, cos, sin = _layer_inputs("tiny", pos=pos)
        g = GpuLayer(dev, w, L, cos, sin)
        kc, vc = L.k_cache.copy(), L.v_cache.copy()
        ref = oracle.decode_layer(L.x, L.x, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc, cos,
                                  sin, pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
        g.run(pos)
        assert_close(H(g.out), ref, f"pos {pos}")


def test_stack_of_layers_chained(dev):
    """Three 7B-shaped layers with independent weights and caches at 32K context,
    residuals chained, against the oracle's chain."""
    base = synth.WORKLOADS["stack32k"]
    rng = np.random.Generator(np.random.PCG64(base.seed))
    cos, sin = synth.rope_tables(base.capacity, base.hd, base.theta)
    x = rng.standard_normal(base.D).astype(np.float32)
    xg = T(x, dev)
    xr = x.copy()
    for layer in range(3):
        L = synth.make_layer(base, rng)
        g = GpuLayer(dev, base, L, cos, sin)
        g.run(base.pos, xg)
        xg = g.out.clone()
        kc, vc = L.k_cache, L.v_cache
        xr = oracle.decode_layer(xr, xr, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc, cos, sin,
                                 base.pos, base.D, base.H, base.KV, base.hd, base.capacity, base.eps)
        assert_close(H(xg), xr, f"stack layer {layer}")
