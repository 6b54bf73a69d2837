"""Parity of the multi-token (prefill) layer, ck_prefill_layer, with the oracle.

The chunk's tokens must match the oracle's prefill form token by token, under
the layer's tolerances: bit-exact Q8_0 activations; max |err| <= 1e-3 * max |ref|
and relative L2 <= 1e-4 for floats.  The O-projection input is checked in
situ: it must be the oracle quantizer applied to the GPU's own attention
output.  A code of that input may legitimately differ from the oracle's where
the two attention outputs straddle a rounding boundary (one step of a block's
scale d); the layer output is then checked against the oracle's O projection
of the GPU's own codes, and end to end wherever no code differs, and the
number of differing codes is bounded.  Cache rows from pos + n_tokens on are
NaN, so a read of a row that is not yet part of the sequence shows up in the
results."""
import dataclasses

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


def H_(t):
    return H(t)


def H(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def ok(rc):
    assert rc == q.CK_OK, q.ck_status_string(rc)


class Chunk:
    """n tokens of one sequence at positions pos..pos+n-1 over a cache whose
    rows 0..pos-1 are filled and the rest NaN."""

    def __init__(self, dev, w, pos, n, seed):
        self.dev, self.w, self.pos, self.n = dev, w, pos, n
        rng = np.random.Generator(np.random.PCG64(seed))
        (self.gamma, self.wq, self.wk, self.wv, self.wo, self.bq, self.bk, self.bv,
         self.bo) = synth.draw_weights(rng, w)
        self.x = rng.standard_normal((n, w.D)).astype(np.float32)
        kc, vc = synth.draw_cache(rng, w, pos)
        kc[:, pos:] = np.nan
        vc[:, pos:] = np.nan
        self.kc0, self.vc0 = kc, vc
        self.cos, self.sin = synth.rope_tables(w.capacity, w.hd, w.theta)
        t = lambda a: T(a, dev)
        self.g = dict(gamma=t(self.gamma), wq=t(self.wq), wk=t(self.wk), wv=t(self.wv), wo=t(self.wo), bq=t(self.bq),
                      bk=t(self.bk), bv=t(self.bv), bo=t(self.bo), cos=t(self.cos), sin=t(self.sin), x=t(self.x))
        self.kc, self.vc = t(kc), t(vc)
        self.out = torch.empty((n, w.D), dtype=torch.float32, device=dev)
        self.nbytes = q.ck_prefill_layer_scratch_size(n, w.D, w.H, w.KV, w.hd, w.capacity)
        assert self.nbytes > 0
        self.scratch = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    def call(self, x=None, pos=None, n=None, out=None, kc=None, vc=None, nbytes=None):
        g, w = self.g, self.w
        x = g["x"] if x is None else x
        return q.ck_prefill_layer(self.out if out is None else out, x, x, g["wq"], g["wk"], g["wv"], g["wo"],
                                  g["gamma"], g["bq"], g["bk"], g["bv"], g["bo"], self.kc if kc is None else kc,
                                  self.vc if vc is None else vc, g["cos"], g["sin"],
                                  self.pos if pos is None else pos, self.n if n is None else n, w.D, w.H, w.KV, w.hd,
                                  w.capacity, w.eps, self.scratch, self.nbytes if nbytes is None else nbytes)

    def tap(self, which, width, dtype):
        w = self.w
        off = q.ck_prefill_layer_scratch_offset(which, self.n, w.D, w.H, w.KV, w.hd, w.capacity)
        nb = self.n * width * np.dtype(dtype).itemsize
        return self.scratch[off:off + nb].cpu().numpy().view(dtype).reshape(self.n, width)

    def check(self):
        w, p, n = self.w, self.pos, self.n
        kc, vc = self.kc0.copy(), self.vc0.copy()
        ref, taps = oracle.prefill_layer(self.x, self.x, self.wq, self.wk, self.wv, self.wo, self.gamma, self.bq,
                                         self.bk, self.bv, self.bo, kc, vc, self.cos, self.sin, p, n, w.D, w.H, w.KV,
                                         w.hd, w.capacity, w.eps, taps=True)
        out = H(self.out)
        xq = self.tap(q.CK_TAP_XQ8, w.D // 32 * 34, np.uint8)
        qt = self.tap(q.CK_TAP_Q, w.QD, np.float32)
        at = self.tap(q.CK_TAP_ATTN, w.QD, np.float32)
        aq = self.tap(q.CK_TAP_AQ8, w.QD // 32 * 34, np.uint8)
        gk, gv = H(self.kc), H(self.vc)
        assert np.array_equal(xq, taps["xq"]), "quantized inputs"
        assert np.array_equal(gk[:, :p], self.kc0[:, :p]) and np.array_equal(gv[:, :p], self.vc0[:, :p]), "old rows"
        assert np.all(np.isnan(gk[:, p + n:])) and np.all(np.isnan(gv[:, p + n:])), "rows past the chunk"
        flips = 0
        for i in range(n):
            assert_close(qt[i], taps["q"][i], f"token {i}: q")
            assert_close(gk[:, p + i].ravel(), taps["k"][i], f"token {i}: stored k")
            assert_close(gv[:, p + i].ravel(), taps["v"][i], f"token {i}: stored v")
            assert_close(at[i], taps["attn"][i], f"token {i}: attention output")
            assert np.array_equal(aq[i], oracle.quantize_q8_0(at[i])), f"token {i}: O-projection input"
            # the O projection + bias + residual on the GPU's own codes
            stage = oracle.gemv(self.wo, aq[i], self.bo, w.D, w.QD, False) + self.x[i]
            assert_close(out[i], stage, f"token {i}: layer output (O projection of its own codes)")
            codes_g = aq[i].reshape(-1, 34)[:, 2:]
            codes_o = taps["aq"][i].reshape(-1, 34)[:, 2:]
            nf = int(np.count_nonzero(codes_g != codes_o))
            flips += nf
            if nf == 0:
                assert_close(out[i], ref[i], f"token {i}: layer output")
        assert flips <= max(2, n * w.QD // 500), f"{flips} O-projection input codes differ from the oracle's"
        rc, st = q.ck_device_status()
        assert rc == 0 and st == 0


@pytest.mark.parametrize("pos,n", [(16, 5), (0, 1), (0, 64), (40, 24), (63, 1)])
def test_prefill_tiny(dev, pos, n):
    """The small layer: a chunk after 16 rows, a lone first token, the whole
    capacity from an empty cache, a chunk that ends on the last row, the last
    row alone."""
    c = Chunk(dev, synth.WORKLOADS["tiny"], pos, n, seed=31 + pos + n)
    ok(c.call())
    c.check()


@pytest.mark.parametrize("pos,n", [(1000, 37), (8092, 100)])
def test_prefill_7b_shape(dev, pos, n):
    """The 7B-shaped layer: a ragged chunk of 37 tokens, and 100 tokens (more
    than one 64-token projection tile) ending at row 8191."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=8192)
    c = Chunk(dev, w, pos, n, seed=41 + n)
    ok(c.call())
    c.check()


def test_prefill_one_token_matches_decode_layer(dev):
    """One token equals ck_decode_layer at the same position (other kernels
    for the projections: equal within the tolerance)."""
    w = synth.WORKLOADS["tiny"]
    c = Chunk(dev, w, 20, 1, seed=51)
    ok(c.call())
    kc, vc = T(c.kc0, dev), T(c.vc0, dev)
    nbytes = q.ck_decode_layer_scratch_size(w.D, w.H, w.KV, w.hd, w.capacity)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    o = torch.empty(w.D, dtype=torch.float32, device=dev)
    g = c.g
    ok(q.ck_decode_layer(o, g["x"][0], g["x"][0], g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"], g["bk"],
                         g["bv"], g["bo"], kc, vc, g["cos"], g["sin"], 20, w.D, w.H, w.KV, w.hd, w.capacity, w.eps,
                         scratch, nbytes))
    assert_close(H(c.out)[0], H(o), "layer output")
    assert_close(H(c.kc)[:, 20], H(kc)[:, 20], "stored k")
    assert_close(H(c.vc)[:, 20], H(vc)[:, 20], "stored v")


def test_prefill_is_causal_on_the_device(dev):
    """Changing the tokens after token i leaves outputs 0..i bit-identical (the
    same call shape runs the same arithmetic) and moves the later ones."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=2048)
    c = Chunk(dev, w, 700, 24, seed=61)
    ok(c.call())
    base = H(c.out).copy()
    i = 9
    x2 = c.g["x"].clone()
    x2[i + 1:] = torch.randn((c.n - i - 1, w.D), generator=torch.Generator(device=dev).manual_seed(5), device=dev)
    c.kc.copy_(T(c.kc0, dev))
    c.vc.copy_(T(c.vc0, dev))
    ok(c.call(x=x2))
    got = H(c.out)
    assert np.array_equal(got[:i + 1], base[:i + 1])
    assert not np.array_equal(got[i + 1:], base[i + 1:])


def test_prefill_two_chunks_equal_one(dev):
    """A prompt prefilled as 8 + 12 tokens equals the same 20 tokens in one call
    (within the tolerance: the call shapes differ)."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=1024)
    c = Chunk(dev, w, 300, 20, seed=71)
    ok(c.call())
    one, k1, v1 = H(c.out).copy(), H(c.kc).copy(), H(c.vc).copy()
    c.kc.copy_(T(c.kc0, dev))
    c.vc.copy_(T(c.vc0, dev))
    out2 = torch.empty_like(c.out)
    for p0, m in ((300, 8), (308, 12)):
        nb = q.ck_prefill_layer_scratch_size(m, w.D, w.H, w.KV, w.hd, w.capacity)
        sc = torch.empty(nb, dtype=torch.uint8, device=dev)
        xs = c.g["x"][p0 - 300:p0 - 300 + m].contiguous()
        o = torch.empty((m, w.D), dtype=torch.float32, device=dev)
        g = c.g
        ok(q.ck_prefill_layer(o, xs, xs, g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"], g["bk"], g["bv"],
                              g["bo"], c.kc, c.vc, g["cos"], g["sin"], p0, m, w.D, w.H, w.KV, w.hd, w.capacity, w.eps,
                              sc, nb))
        out2[p0 - 300:p0 - 300 + m] = o
    two = H(out2)
    for i in range(20):
        assert_close(two[i], one[i], f"token {i}")
    assert_close(H(c.kc)[:, 300:320], k1[:, 300:320], "stored k")
    assert_close(H(c.vc)[:, 300:320], v1[:, 300:320], "stored v")


def test_prefill_argument_errors(dev):
    """Host validation: nothing is launched and nothing written."""
    w = synth.WORKLOADS["tiny"]
    c = Chunk(dev, w, 10, 4, seed=81)
    c.out.fill_(3.0)
    assert c.call(pos=w.capacity - 3) == q.CK_ERANGE       # rows 61..64: one past the end
    assert c.call(pos=-1) == q.CK_ERANGE
    assert c.call(n=0) == q.CK_EINVAL
    assert c.call(n=1025) == q.CK_EINVAL
    assert c.call(nbytes=c.nbytes - 1) == q.CK_ESCRATCH
    assert c.call(out=c.g["x"]) == q.CK_EINVAL               # out aliases x
    flat = torch.empty(c.kc.numel() + 1, dtype=torch.float32, device=dev)
    assert c.call(kc=flat[1:].view(c.kc.shape)) == q.CK_EALIGN
    assert np.all(H(c.out) == 3.0)
    assert np.array_equal(H(c.kc), c.kc0, equal_nan=True)
    assert q.ck_prefill_layer_scratch_size(0, w.D, w.H, w.KV, w.hd, w.capacity) == 0


@pytest.mark.parametrize("D,H,KV,pos,n,C", [
    (3584, 28, 4, 0, 1, 256),     # one token, no prefix
    (3584, 28, 4, 0, 16, 256),    # exactly one 128-row query tile (16 tokens x 8 head slots)
    (3584, 28, 4, 5, 17, 256),    # a second tile holding one token
    (3584, 28, 4, 100, 64, 200),  # ends at row 163 of a 200-row cache: ragged last key tile
    (2048, 16, 4, 333, 70, 512),  # query groups of 4 (32 tokens per tile)
    (2048, 16, 2, 50, 20, 128),   # groups of 8 over two KV heads
])
def test_prefill_tensor_core_attention_shapes(dev, D, H, KV, pos, n, C):
    """head_dim 128: the chunk's attention runs on the tensor cores; tiles of
    query rows and key rows with ragged ends, several group sizes."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], D=D, H=H, KV=KV, hd=128, capacity=C)
    c = Chunk(dev, w, pos, n, seed=91 + n + pos)
    ok(c.call())
    c.check()


@pytest.mark.parametrize("H,KV,pos,n,C", [(28, 4, 0, 1, 64), (28, 4, 130, 33, 200), (16, 2, 7000, 300, 7300),
                                          (8, 8, 10, 70, 96), (32, 2, 64, 64, 128), (28, 4, 0, 1024, 1024)])
def test_attn_prefill_alone(dev, H, KV, pos, n, C):
    """ck_attn_prefill_gqa against the oracle's decode attention over pos + i + 1
    rows for sampled tokens (groups of 7, 8, 1 and 16; a 7,300-row cache; a
    1,024-token chunk from an empty cache filling it: 256 CTAs)."""
    hd = 128
    rng = np.random.default_rng(pos + n + H)
    kc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    vc0 = rng.standard_normal((KV, C, hd)).astype(np.float32)
    kc0[:, pos + n:] = np.nan
    vc0[:, pos + n:] = np.nan
    qv = (rng.standard_normal((n, H * hd)) * 1.5).astype(np.float32)
    nb = q.ck_attn_prefill_scratch_size(H, KV, hd, C)
    assert nb > 0
    sc = torch.empty(nb, dtype=torch.uint8, device=dev)
    out = torch.full((n, H * hd), float("nan"), dtype=torch.float32, device=dev)
    ok(q.ck_attn_prefill_gqa(T(qv, dev), T(kc0, dev), T(vc0, dev), out, pos, n, H, KV, hd, C, sc, nb))
    got = H_(out)
    for i in sorted({0, n // 2, n - 1} | set(range(0, n, max(1, n // 12)))):
        ref = oracle.attention(qv[i], kc0, vc0, H, KV, pos + i + 1, C, hd)
        assert_close(got[i], ref, f"token {i}")
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0


def test_attn_prefill_argument_errors(dev):
    H, KV, hd, C = 28, 4, 128, 64
    z = torch.zeros((KV, C, hd), dtype=torch.float32, device=dev)
    qv = torch.zeros((8, H * hd), dtype=torch.float32, device=dev)
    out = torch.zeros_like(qv)
    nb = q.ck_attn_prefill_scratch_size(H, KV, hd, C)
    sc = torch.empty(nb, dtype=torch.uint8, device=dev)
    f = lambda pos=0, n=8, hd_=hd, bytes_=nb: q.ck_attn_prefill_gqa(qv, z, z, out, pos, n, H, KV, hd_, C, sc, bytes_)
    assert f(pos=57) == q.CK_ERANGE and f(pos=-1) == q.CK_ERANGE
    assert f(n=0) == q.CK_EINVAL and f(hd_=64) == q.CK_EINVAL
    assert f(bytes_=nb - 257) == q.CK_ESCRATCH
    assert q.ck_attn_prefill_scratch_size(H, KV, 64, C) == 0
    ok(f(pos=56))


def _devpos_call(c, pos_t, x=None, out=None):
    g, w = c.g, c.w
    x = g["x"] if x is None else x
    return q.ck_prefill_layer_devpos(c.out if out is None else out, x, x, g["wq"], g["wk"], g["wv"], g["wo"],
                                     g["gamma"], g["bq"], g["bk"], g["bv"], g["bo"], c.kc, c.vc, g["cos"], g["sin"],
                                     pos_t, c.n, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, c.scratch, c.nbytes)


@pytest.mark.parametrize("shape", ["7b", "tiny"])
def test_prefill_devpos_equals_host_position(dev, shape):
    """The position read on the device gives the same bits as the host
    position (tensor-core attention at head_dim 128, decode path at 64)."""
    if shape == "7b":
        w, pos, n = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=1024), 300, 20
    else:
        w, pos, n = synth.WORKLOADS["tiny"], 16, 9
    c = Chunk(dev, w, pos, n, seed=101)
    ok(c.call())
    ref_out, ref_k, ref_v = H(c.out).copy(), H(c.kc).copy(), H(c.vc).copy()
    c.kc.copy_(T(c.kc0, dev))
    c.vc.copy_(T(c.vc0, dev))
    c.out.fill_(0.0)
    ok(_devpos_call(c, torch.tensor([pos], dtype=torch.int32, device=dev)))
    assert np.array_equal(H(c.out), ref_out)
    assert np.array_equal(H(c.kc), ref_k, equal_nan=True) and np.array_equal(H(c.vc), ref_v, equal_nan=True)
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0


@pytest.mark.parametrize("shape", ["7b", "tiny"])
def test_prefill_devpos_out_of_range_writes_nothing(dev, shape):
    if shape == "7b":
        w, n = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=256), 16
    else:
        w, n = synth.WORKLOADS["tiny"], 5
    c = Chunk(dev, w, 10, n, seed=102)
    c.out.fill_(7.0)
    q.ck_device_status()  # clear
    ok(_devpos_call(c, torch.tensor([w.capacity - n + 1], dtype=torch.int32, device=dev)))
    assert np.all(H(c.out) == 7.0)
    assert np.array_equal(H(c.kc), c.kc0, equal_nan=True) and np.array_equal(H(c.vc), c.vc0, equal_nan=True)
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    assert _devpos_call(c, None) == q.CK_EINVAL


def test_prefill_devpos_graph_replay_moves_the_chunk(dev):
    """One captured graph prefills two consecutive chunks of 8 tokens (the
    position advanced on the device between replays); the result equals two
    host-position calls."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=512)
    n, p0 = 8, 200
    c = Chunk(dev, w, p0, 2 * n, seed=103)  # 16 tokens of input, two chunks of 8
    nb = q.ck_prefill_layer_scratch_size(n, w.D, w.H, w.KV, w.hd, w.capacity)
    g = c.g
    # reference: two host-position calls
    sc = torch.empty(nb, dtype=torch.uint8, device=dev)
    ref = []
    for k in range(2):
        xs = g["x"][k * n:(k + 1) * n].contiguous()
        o = torch.empty((n, w.D), dtype=torch.float32, device=dev)
        ok(q.ck_prefill_layer(o, xs, xs, g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"], g["bk"], g["bv"],
                              g["bo"], c.kc, c.vc, g["cos"], g["sin"], p0 + k * n, n, w.D, w.H, w.KV, w.hd,
                              w.capacity, w.eps, sc, nb))
        ref.append(H(o).copy())
    ref_k, ref_v = H(c.kc).copy(), H(c.vc).copy()
    # the graph
    c.kc.copy_(T(c.kc0, dev))
    c.vc.copy_(T(c.vc0, dev))
    xin = torch.empty((n, w.D), dtype=torch.float32, device=dev)
    oo = torch.empty((n, w.D), dtype=torch.float32, device=dev)
    dpos = torch.tensor([p0], dtype=torch.int32, device=dev)
    st = torch.cuda.Stream(device=dev)
    xin.copy_(g["x"][:n])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        rc = q.ck_prefill_layer_devpos(oo, xin, xin, g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"], g["bk"],
                                       g["bv"], g["bo"], c.kc, c.vc, g["cos"], g["sin"], dpos, n, w.D, w.H, w.KV,
                                       w.hd, w.capacity, w.eps, sc, nb, st.cuda_stream)
    ok(rc)
    got = []
    for k in range(2):
        xin.copy_(g["x"][k * n:(k + 1) * n])
        dpos.fill_(p0 + k * n)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        got.append(H(oo).copy())
    for k in range(2):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(H(c.kc), ref_k, equal_nan=True) and np.array_equal(H(c.vc), ref_v, equal_nan=True)
    rc, st2 = q.ck_device_status()
    assert rc == 0 and st2 == 0
