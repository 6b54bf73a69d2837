"""Parity of the batched decode step (ck_decode_layer_batched) with the oracle:
every checked sequence must match the oracle's single-sequence decode step on
that sequence's own cache and position, under the same tolerances as the
single-sequence layer (bit-exact Q8_0 activations; max |err| <= 1e-3 *
max |ref| and relative L2 <= 1e-4 for floats).  Cache rows past each
sequence's position are NaN: the step must never read them."""
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


def H(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def ok(rc):
    assert rc == q.CK_OK, q.ck_status_string(rc)


class Batch:
    """A batch of sequences sharing one layer; caches drawn on the host (small
    cases) or on the device with a seeded generator (large ones)."""

    def __init__(self, dev, w, pos, seed, host_caches=True):
        self.dev, self.w = dev, w
        self.pos = np.asarray(pos, np.int32)
        B = self.B = len(pos)
        rng = np.random.Generator(np.random.PCG64(seed))
        (self.gamma, self.wq, self.wk, self.wv, self.wo, self.bq, self.bk, self.bv,
         self.bo) = synth.draw_weights(rng, w)
        self.x = rng.standard_normal((B, w.D)).astype(np.float32)
        self.cos, self.sin = synth.rope_tables(w.capacity, w.hd, w.theta)
        t = lambda a: T(a, dev)
        self.g = dict(gamma=t(self.gamma), wq=t(self.wq), wk=t(self.wk), wv=t(self.wv), wo=t(self.wo), bq=t(self.bq),
                      bk=t(self.bk), bv=t(self.bv), bo=t(self.bo), cos=t(self.cos), sin=t(self.sin), x=t(self.x))
        self.kc, self.vc = [], []
        gen = torch.Generator(device=dev)
        for s in range(B):
            shape = (w.KV, w.capacity, w.hd)
            if host_caches:
                kc, vc = synth.draw_cache(rng, w, int(pos[s]))
                kc[:, pos[s] + 1:] = np.nan
                vc[:, pos[s] + 1:] = np.nan
                self.kc.append(t(kc))
                self.vc.append(t(vc))
            else:
                gen.manual_seed(seed * 1000 + s)
                kc = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
                vc = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
                kc[:, :pos[s]].normal_(generator=gen)
                vc[:, :pos[s]].normal_(generator=gen)
                self.kc.append(kc)
                self.vc.append(vc)
        self.kptr = torch.tensor([c.data_ptr() for c in self.kc], dtype=torch.int64, device=dev)
        self.vptr = torch.tensor([c.data_ptr() for c in self.vc], dtype=torch.int64, device=dev)
        self.d_pos = T(self.pos, dev)
        self.out = torch.empty((B, w.D), dtype=torch.float32, device=dev)
        self.nbytes = q.ck_decode_layer_batched_scratch_size(B, w.D, w.H, w.KV, w.hd, w.capacity)
        assert self.nbytes > 0
        self.scratch = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    def host_cache(self, s):
        return H(self.kc[s]).copy(), H(self.vc[s]).copy()

    def run(self, stream=None):
        g, w = self.g, self.w
        ok(q.ck_decode_layer_batched(self.out, g["x"], g["x"], g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"],
                                     g["bq"], g["bk"], g["bv"], g["bo"], self.kptr, self.vptr, g["cos"], g["sin"],
                                     self.d_pos, self.B, w.D, w.H, w.KV, w.hd, w.capacity, w.eps, self.scratch,
                                     self.nbytes, stream))

    def tap(self, which, n, dtype):
        w = self.w
        off = q.ck_decode_layer_batched_scratch_offset(which, self.B, w.D, w.H, w.KV, w.hd, w.capacity)
        nb = self.B * n * np.dtype(dtype).itemsize
        return self.scratch[off:off + nb].cpu().numpy().view(dtype).reshape(self.B, n)

    def check(self, pre, sample):
        """pre[s] = (kc, vc) host copies taken before the step."""
        w = self.w
        out = H(self.out)
        xq = self.tap(q.CK_TAP_XQ8, w.D // 32 * 34, np.uint8)
        qt = self.tap(q.CK_TAP_Q, w.QD, np.float32)
        at = self.tap(q.CK_TAP_ATTN, w.QD, np.float32)
        aq = self.tap(q.CK_TAP_AQ8, w.QD // 32 * 34, np.uint8)
        for s in sample:
            kc, vc = pre[s]
            p = int(self.pos[s])
            ref, taps = oracle.decode_layer(self.x[s], self.x[s], self.wq, self.wk, self.wv, self.wo, self.gamma,
                                            self.bq, self.bk, self.bv, self.bo, kc, vc, self.cos, self.sin, p, w.D,
                                            w.H, w.KV, w.hd, w.capacity, w.eps, taps=True)
            assert np.array_equal(xq[s], taps["xq"]), f"seq {s}: quantized input"
            assert_close(qt[s], taps["q"], f"seq {s}: q")
            gk, gv = H(self.kc[s]), H(self.vc[s])
            assert_close(gk[:, p].ravel(), taps["k"], f"seq {s}: stored k")
            assert_close(gv[:, p].ravel(), taps["v"], f"seq {s}: stored v")
            assert np.array_equal(gk[:, :p], kc[:, :p]) and np.array_equal(gv[:, :p], vc[:, :p]), f"seq {s}: rows"
            assert_close(at[s], taps["attn"], f"seq {s}: attention output")
            assert np.array_equal(aq[s], oracle.quantize_q8_0(at[s])), f"seq {s}: O-projection input"
            assert_close(out[s], ref, f"seq {s}: layer output")
        rc, st = q.ck_device_status()
        assert rc == 0 and st == 0


def test_batched_tiny_ragged(dev):
    """Seven sequences of the small layer at positions from 0 to capacity - 1."""
    w = synth.WORKLOADS["tiny"]
    b = Batch(dev, w, [0, 1, 16, 31, 40, 62, 63], seed=21)
    pre = [b.host_cache(s) for s in range(b.B)]
    b.run()
    b.check(pre, range(b.B))


def test_batched_7b_shape_long_and_short(dev):
    """Six 7B-shaped sequences from 1 to 9951 attended rows: the attention
    takes its 16 KB stages (planned from the capacity) for short and long
    sequences alike, and splits end in partial stages."""
    w = dataclasses.replace(synth.WORKLOADS["7b8k"], capacity=10016)
    b = Batch(dev, w, [0, 100, 1000, 5000, 9000, 9950], seed=22)
    pre = [b.host_cache(s) for s in range(b.B)]
    b.run()
    b.check(pre, range(b.B))


def test_batched64_config_sampled(dev):
    """The 64-sequence workload (lengths uniform in [512, 16384]) in one call;
    the shortest, the longest and four more sequences against the oracle."""
    w = synth.WORKLOADS["batched64"]
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lens = synth.batched_lengths(w, rng)
    b = Batch(dev, w, lens, seed=w.seed, host_caches=False)
    sample = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 1, 17, 40, 63})
    pre = {s: b.host_cache(s) for s in sample}
    b.run()
    b.check(pre, sample)


def test_batched_matches_single_sequence_calls(dev):
    """The batched step equals ck_decode_layer_devpos run on each sequence
    alone (same kernels for the attention; the projections differ only in
    the order of fp32 accumulation, so compare within the tolerance)."""
    w = synth.WORKLOADS["tiny"]
    b = Batch(dev, w, [5, 33, 60], seed=23)
    pre = [b.host_cache(s) for s in range(b.B)]
    b.run()
    out = H(b.out)
    g = b.g
    nbytes = q.ck_decode_layer_scratch_size(w.D, w.H, w.KV, w.hd, w.capacity)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for s in range(b.B):
        kc, vc = T(pre[s][0], dev), T(pre[s][1], dev)
        o = torch.empty(w.D, dtype=torch.float32, device=dev)
        dpos = b.d_pos[s:s + 1].clone()  # its own (16-byte aligned) allocation
        ok(q.ck_decode_layer_devpos(o, g["x"][s], g["x"][s], g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"],
                                    g["bq"], g["bk"], g["bv"], g["bo"], kc, vc, g["cos"], g["sin"], dpos, w.D, w.H,
                                    w.KV, w.hd, w.capacity, w.eps, scratch, nbytes))
        assert_close(out[s], H(o), f"seq {s}")
        assert_close(H(b.kc[s])[:, b.pos[s]], H(kc)[:, b.pos[s]], f"seq {s}: stored k")
        assert_close(H(b.vc[s])[:, b.pos[s]], H(vc)[:, b.pos[s]], f"seq {s}: stored v")


def test_batched_out_of_range_position_writes_nothing(dev):
    """A sequence whose device position is the capacity writes nothing of its
    own; the others are unaffected; the status word reports CK_ERANGE."""
    w = synth.WORKLOADS["tiny"]
    b = Batch(dev, w, [10, 20, 30], seed=24)
    pre = [b.host_cache(s) for s in range(b.B)]
    b.pos[1] = w.capacity
    b.d_pos.copy_(T(b.pos, dev))
    b.out.fill_(7.0)
    q.ck_device_status()
    b.run()
    out = H(b.out)
    assert np.all(out[1] == 7.0)
    kc1, vc1 = H(b.kc[1]), H(b.vc[1])
    same = lambda u, v: np.array_equal(np.nan_to_num(u, nan=1234.5), np.nan_to_num(v, nan=1234.5))
    assert same(kc1, pre[1][0]) and same(vc1, pre[1][1])
    rc, st = q.ck_device_status()
    assert rc == 0 and st == q.CK_ERANGE
    for s in (0, 2):
        ref = oracle.decode_layer(b.x[s], b.x[s], b.wq, b.wk, b.wv, b.wo, b.gamma, b.bq, b.bk, b.bv, b.bo,
                                  pre[s][0], pre[s][1], b.cos, b.sin, int(b.pos[s]), w.D, w.H, w.KV, w.hd, w.capacity,
                                  w.eps)
        assert_close(out[s], ref, f"seq {s}")
