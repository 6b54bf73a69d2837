#!/usr/bin/env python3
"""Decode-step benchmark of the Q5_0/Q8_0 attention layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

A step is one decode step of the layer (RMSNorm -> Q8_0 -> Q/K/V GEMVs ->
RoPE -> KV store -> GQA attention -> Q8_0 -> O GEMV + residual) for one token.
Default workload: the 7B-class layer at 8K context (D=3584, 28/4 heads,
head_dim 128, 8193 cache rows attended).  Inputs are seeded synthetic data.
Each step uses the next of R byte-identical replicas of weights + caches, so
the bytes touched between two uses of a replica exceed the 129 MB L2.

Device timing: K steps replayed from CUDA graphs (R steps per graph), CUDA
events on the replay stream, barrier + synchronize on both sides, max over
ranks.  e2e: the same steps through the C-ABI call with the input copied from
pinned host memory and the output read back every step.  Under torchrun each
rank runs its own replica set ("replicas only": the decode step of one
sequence has no data-parallel split that needs a collective).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode layer-steps/s (tokens/s) and achieved HBM GB/s vs GB300 peak"
L2_BYTES = 129 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60000)
    p.add_argument("--warmup", type=int, default=600)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="7b8k",
                   choices=["tiny", "small1k", "7b8k", "stack32k", "batched64", "attn32k", "paged64", "prefill512"])
    p.add_argument("--kv-dtype", default="bf16", choices=["f32", "bf16", "fp8"],
                   help="attn32k / paged64: cache element type (fp8 = E4M3 with per-tensor scales)")
    p.add_argument("--window", type=int, default=0, help="paged64: sliding window (0: every row)")
    p.add_argument("--rows", type=int, default=0, help="attn32k: rows attended (default 32769)")
    p.add_argument("--splits", type=int, default=-1,
                   help="attn32k: split count through ck_attn_decode_gqa_split (0: its built-in choice)")
    p.add_argument("--block-size", type=int, default=64, help="paged64: rows per cache block")
    p.add_argument("--layers", type=int, default=0, help="stack32k: layers in the stack (default: all 28)")
    p.add_argument("--kv-cap", type=int, default=0,
                   help="batched64: cap every cache at this many rows (a small case for profilers; not the workload)")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle CPU baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# --------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo")
        pg = dist
    return ws, rank, local, pg


def barrier(pg, torch):
    if pg is not None:
        pg.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(pg, torch, v: float) -> float:
    """The largest of the ranks' values (the slowest rank's time)."""
    if pg is None:
        return v
    dev = "cuda" if torch.cuda.is_available() and pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id, self.rows, self.proc = gpu_id, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        num = lambda x: x.replace(".", "", 1).isdigit()
        ok = [r for r in self.rows if len(r) >= 8]
        sm = [float(r[0]) for r in ok if num(r[0])]
        mx = [float(r[1]) for r in ok if num(r[1])]
        pw = [float(r[2]) for r in ok if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in ok for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm), "power_w_max": max(pw) if pw else None}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def launches_per_layer(w) -> int:
    """Kernels one ck_decode_layer call launches: the Q/K/V projection (which
    also normalizes when D/32 is a multiple of 8, else a separate RMSNorm +
    quantize kernel runs first), the attention split, its combine, and the
    O-projection."""
    return 4 if (w.D // 32) % 8 == 0 else 5


def profiled_traffic(key: str, source: str):
    """DRAM bytes per launch of kernel@workload `key` from a committed ncu
    summary, if it was taken on the kernel source as it is now (same hash);
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        src = open(os.path.join(ROOT, source), "rb").read()
        entry = d.get(key)
        if entry and entry.get("source_sha256") == hashlib.sha256(src).hexdigest():
            return entry.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# --------------------------------------------------------------------------
# the workload on the device
# --------------------------------------------------------------------------
class Source:
    """Device copies of one seeded layer (the replicas clone it)."""

    def __init__(self, torch, w, dev):
        from quantized_weight_attention_gb300 import synth
        L = synth.make_layer(w)
        cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
        T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        self.t = dict(x=T(L.x), gamma=T(L.gamma), wq=T(L.wq), wk=T(L.wk), wv=T(L.wv), wo=T(L.wo), bq=T(L.bq),
                      bk=T(L.bk), bv=T(L.bv), bo=T(L.bo), kc=T(L.k_cache), vc=T(L.v_cache), cos=T(cos), sin=T(sin))


class Replica:
    """An independent byte copy of one layer's weights, caches and scratch."""

    def __init__(self, torch, q, src, w, dev):
        self.w = w
        self.t = {k: v.clone() for k, v in src.t.items()}
        self.out = torch.empty(w.D, dtype=torch.float32, device=dev)
        self.nbytes = q.ck_decode_layer_scratch_size(w.D, w.H, w.KV, w.hd, w.capacity)
        self.scratch = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)

    def call(self, q, stream, x=None):
        w, t = self.w, self.t
        xx = t["x"] if x is None else x
        return q.ck_decode_layer(self.out, xx, xx, t["wq"], t["wk"], t["wv"], t["wo"], t["gamma"], t["bq"], t["bk"],
                                 t["bv"], t["bo"], t["kc"], t["vc"], t["cos"], t["sin"], w.pos, w.D, w.H, w.KV, w.hd,
                                 w.capacity, w.eps, self.scratch, self.nbytes, stream)


def step_bytes(w):
    """Algorithmic bytes of one step: quantized weights + the K and V rows attended."""
    return w.weight_bytes() + w.kv_read_bytes(w.pos + 1)


def gpu_uuid(torch, dev):
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"


def run_ours(args, ws, rank, local, pg):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_attention_gb300 as q
    from quantized_weight_attention_gb300 import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.config == "attn32k":
        return run_attn_kv(args, ws, pg, torch, q, synth, dev)
    if args.config == "paged64":
        return run_paged(args, ws, pg, torch, q, synth, dev)
    if args.config == "prefill512":
        return run_prefill(args, ws, pg, torch, q, synth, dev)
    w = synth.WORKLOADS[args.config]
    if args.config == "stack32k":
        return run_stack(args, ws, pg, torch, q, synth, dev)
    if args.config == "batched64":
        return run_batched(args, ws, pg, torch, q, synth, dev)
    src = Source(torch, w, dev)
    per_replica = w.weight_bytes() + 2 * w.KV * w.capacity * w.hd * 4 + 4 * w.D * 8
    R = max(3, -(-int(2.5 * L2_BYTES) // per_replica))
    reps = [Replica(torch, q, src, w, dev) for _ in range(R)]
    del src
    stream = torch.cuda.Stream(device=dev)
    for r in reps:  # eager first calls (kernel attributes are set outside capture), checked
        q.check(r.call(q, stream.cuda_stream))
    torch.cuda.synchronize()
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                q.check(reps[i % R].call(q, stream.cuda_stream))
        return g

    g_full = capture(R)
    K, W = args.steps, max(args.warmup, 3)
    rem = K % R
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(-(-W // R)):
            g_full.replay()
    W = -(-W // R) * R
    torch.cuda.synchronize()

    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        ev0.record(stream)
        for _ in range(K // R):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    value = ws * K / sec

    # ---- dominant kernel: the attention over the cache (one C-ABI call:
    # split + combine), N calls back to back in a CUDA graph over the rotating
    # replicas' caches, timed with CUDA events around graph replays
    att_bytes = w.kv_read_bytes(w.pos + 1)
    att_scr = q.ck_attn_scratch_size(w.H, w.KV, w.capacity, w.hd)
    att_scratch = torch.empty(att_scr, dtype=torch.uint8, device=dev)
    att_out = torch.empty(w.H * w.hd, dtype=torch.float32, device=dev)
    qoff = q.ck_decode_layer_scratch_offset(q.CK_TAP_Q, w.D, w.H, w.KV, w.hd, w.capacity)
    qtap = [r.scratch[qoff:qoff + w.H * w.hd * 4].view(torch.float32) for r in reps]

    def att_calls(n):
        for i in range(n):
            r = reps[i % R]
            q.check(q.ck_attn_decode_gqa(qtap[i % R], r.t["kc"], r.t["vc"], att_out, w.H, w.KV, w.pos + 1,
                                         w.capacity, w.hd, att_scratch, att_scr, stream.cuda_stream))

    with torch.cuda.stream(stream):
        att_calls(R)
    torch.cuda.synchronize()
    g_att = torch.cuda.CUDAGraph()
    n_att = 4 * R
    with torch.cuda.graph(g_att, stream=stream):
        att_calls(n_att)
    durs = []
    with torch.cuda.stream(stream):
        g_att.replay()
        for _ in range(9):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(5):
                g_att.replay()
            b.record(stream)
            b.synchronize()
            durs.append(a.elapsed_time(b) / (5 * n_att))
    att_ms = statistics.median(durs)
    peak, peak_kind = measured_peaks()
    achieved = att_bytes / (att_ms / 1e3) / 1e9

    # ---- e2e through the C ABI with host buffers
    Ke = min(K, 20000)
    xh = reps[0].t["x"].cpu().pin_memory()
    outh = torch.empty((R, w.D), dtype=torch.float32).pin_memory()
    xdev = [torch.empty(w.D, dtype=torch.float32, device=dev) for _ in range(R)]
    torch.cuda.synchronize()
    barrier(pg, torch)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(Ke):
            j = i % R
            xdev[j].copy_(xh, non_blocking=True)
            q.check(reps[j].call(q, stream.cuda_stream, x=xdev[j]))
            outh[j].copy_(reps[j].out, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    barrier(pg, torch)
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1))
    e2e_value = ws * Ke / (e2e_ms / 1e3)
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "layer-steps/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": round(ms / K, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 dot (dp4a) + fp32", "data": "synthetic",
        "config": {"workload": f"{w.name}: one decode step of a D={w.D}, {w.H}/{w.KV}-head, head_dim {w.hd} layer "
                               f"at pos {w.pos} ({w.pos + 1} cache rows attended, capacity {w.capacity}); "
                               f"Q5_0 Wq/Wk/Wo, Q8_0 Wv, fp32 head-major KV cache",
                   "l2": f"inputs larger than L2: {R} replicas of weights+caches rotated, "
                         f"{R * per_replica / 2**20:.0f} MiB touched between reuses",
                   "graph_steps": R, "parallelism": f"replicas x{ws}"},
        "step_hbm_gbs": round(step_bytes(w) * ws * K / sec / 1e9, 1),
        "step_bytes": step_bytes(w),
        "roofline": {"kernel": "attention (k_attn_split + k_attn_combine: one ck_attn_decode_gqa call, "
                               "calls back to back in a CUDA graph)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                     "bytes_per_launch": att_bytes, "ms_per_launch": round(att_ms, 6),
                     "traffic": profiled_traffic(f"k_attn_split@{args.config}",
                                                 "quantized_weight_attention_gb300/csrc/ck_attn_kernels.cuh")},
        "e2e": {"value": round(e2e_value, 1), "unit": "layer-steps/s", "h2d_bytes_per_step": w.D * 4,
                "d2h_bytes_per_step": w.D * 4, "steps": Ke,
                "how": "per step: pinned x -> device, ck_decode_layer, out -> pinned host (one stream)"},
        "gpu_launches": launches_per_layer(w) * K,
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


def run_stack(args, ws, pg, torch, q, synth, dev):
    """28 layers of the 7B shape at 32K context: one token through the stack per step."""
    w = synth.WORKLOADS["stack32k"]
    nlayers = args.layers if args.layers > 0 else w.layers
    rng = np.random.Generator(np.random.PCG64(w.seed))
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    gen = torch.Generator(device=dev)
    layers = []
    for layer in range(nlayers):
        gamma, wq, wk, wv, wo, bq, bk, bv, bo = synth.draw_weights(rng, w)
        gen.manual_seed(w.seed * 1000 + layer)
        kc = torch.zeros((w.KV, w.capacity, w.hd), dtype=torch.float32, device=dev)
        vc = torch.zeros_like(kc)
        kc[:, :w.pos].normal_(generator=gen)
        vc[:, :w.pos].normal_(generator=gen)
        layers.append(dict(gamma=T(gamma), wq=T(wq), wk=T(wk), wv=T(wv), wo=T(wo), bq=T(bq), bk=T(bk), bv=T(bv),
                           bo=T(bo), kc=kc, vc=vc))
    cosd, sind = T(cos), T(sin)
    x0 = T(rng.standard_normal(w.D).astype(np.float32))
    bufs = [torch.empty(w.D, dtype=torch.float32, device=dev) for _ in range(2)]
    nbytes = q.ck_decode_layer_scratch_size(w.D, w.H, w.KV, w.hd, w.capacity)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def token():
        x = x0
        for i, Lr in enumerate(layers):
            out = bufs[i % 2]
            q.check(q.ck_decode_layer(out, x, x, Lr["wq"], Lr["wk"], Lr["wv"], Lr["wo"], Lr["gamma"], Lr["bq"],
                                      Lr["bk"], Lr["bv"], Lr["bo"], Lr["kc"], Lr["vc"], cosd, sind, w.pos, w.D, w.H,
                                      w.KV, w.hd, w.capacity, w.eps, scratch, nbytes, stream.cuda_stream))
            x = out

    with torch.cuda.stream(stream):
        token()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        token()
    K, W = args.steps, max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for _ in range(W):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        ev0.record(stream)
        for _ in range(K):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    per_tok = nlayers * step_bytes(w)
    peak, peak_kind = measured_peaks()
    ach = per_tok * ws * K / sec / 1e9
    return {"metric": METRIC, "value": round(ws * K / sec, 2), "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8 dot (dp4a) + fp32", "data": "synthetic",
            "config": {"workload": f"stack32k: {nlayers} layers of the D=3584 28/4-head layer, one token at pos "
                                   "32768, one CUDA graph per token",
                       "l2": f"{per_tok / 1e9:.2f} GB per step >> L2"},
            "step_hbm_gbs": round(ach, 1), "step_bytes": per_tok,
            "roofline": {"kernel": "whole token step", "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(ach / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                         "traffic": None},
            "gpu_launches": launches_per_layer(w) * nlayers * K, "clocks": clocks}


KV_ES = {"f32": 4, "bf16": 2, "fp8": 1}
ATTN_ROWS = 32769  # the 32K-context attention of the 7B-shaped layer (pos 32768)


def attn_kv_shape(synth, rows=0):
    w = synth.WORKLOADS["7b8k"]
    rows = rows or ATTN_ROWS
    return w.H, w.KV, w.hd, rows, rows + 63


def run_attn_kv(args, ws, pg, torch, q, synth, dev):
    """The decode attention of the 7B-shaped layer at 32,769 rows over an fp32,
    bf16 or fp8 E4M3 cache: one C-ABI attention call per step, calls back to
    back in a CUDA graph over replicated caches (more bytes than L2)."""
    H, KV, hd, Tn, C = attn_kv_shape(synth, args.rows)
    dt, es = args.kv_dtype, KV_ES[args.kv_dtype]
    S = args.splits
    kv_bytes = 2 * KV * Tn * hd * es
    per_rep = 2 * KV * C * hd * es
    R = max(3, -(-int(2.5 * L2_BYTES) // per_rep))
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    ks = vs = 0.01
    reps = []
    for r in range(R):
        if dt == "fp8":  # finite E4M3 codes, random sign
            mk = lambda: (torch.randint(0, 0x7F, (KV, C, hd), generator=gen, device=dev, dtype=torch.int32) |
                          (torch.randint(0, 2, (KV, C, hd), generator=gen, device=dev, dtype=torch.int32) << 7)
                          ).to(torch.uint8)
        else:
            f = torch.float32 if dt == "f32" else torch.bfloat16
            mk = lambda: torch.randn((KV, C, hd), generator=gen, device=dev, dtype=torch.float32).to(f)
        reps.append((mk(), mk()))
    qv = torch.randn(H * hd, generator=gen, device=dev, dtype=torch.float32)
    out = torch.empty(H * hd, dtype=torch.float32, device=dev)
    nbytes = max(q.ck_attn_scratch_size(H, KV, C, hd), q.ck_attn_split_scratch_size(H, KV, hd, max(S, 1)))
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(i, qin=None, o=None):
        kc, vc = reps[i % R]
        qq = qv if qin is None else qin
        oo = out if o is None else o
        if S >= 0:
            return q.ck_attn_decode_gqa_split(qq, kc, vc, oo, H, KV, Tn, C, hd, {"f32": 0, "bf16": 1, "fp8": 2}[dt],
                                              ks, vs, S, scratch, nbytes, stream.cuda_stream)
        if dt == "f32":
            return q.ck_attn_decode_gqa(qq, kc, vc, oo, H, KV, Tn, C, hd, scratch, nbytes, stream.cuda_stream)
        if dt == "bf16":
            return q.ck_attn_decode_gqa_bf16(qq, kc, vc, oo, H, KV, Tn, C, hd, scratch, nbytes, stream.cuda_stream)
        return q.ck_attn_decode_gqa_fp8(qq, kc, vc, oo, H, KV, Tn, C, hd, ks, vs, scratch, nbytes,
                                        stream.cuda_stream)

    with torch.cuda.stream(stream):
        for i in range(R):
            q.check(call(i))
    torch.cuda.synchronize()
    n_g = 4 * R
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_g):
            q.check(call(i))
    K = max(1, -(-args.steps // n_g)) * n_g  # whole graph replays
    K = min(K, 40 * n_g)
    W = max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for _ in range(-(-W // n_g)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(K // n_g):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    ach = kv_bytes * ws * K / sec / 1e9
    peak, peak_kind = measured_peaks()
    # e2e: q from pinned host memory, the output back, every call
    Ke = min(K, 2000)
    qh = qv.cpu().pin_memory()
    oh = torch.empty(H * hd, dtype=torch.float32).pin_memory()
    qd = torch.empty_like(qv)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(Ke):
            qd.copy_(qh, non_blocking=True)
            q.check(call(i, qd))
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1))
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    line = {"metric": "decode attention calls/s and achieved HBM GB/s vs GB300 peak", "value": round(ws * K / sec, 1),
            "unit": "attention-calls/s", "n_gpus": ws, "steps": K, "warmup": W, "ms_per_step": round(ms / K, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"f32": "f32", "bf16": "bf16 cache, f32 math", "fp8": "fp8 e4m3 cache, f32 math"}[dt],
            "data": "synthetic",
            "config": {"workload": f"attn32k: decode attention of the 28/4-head hd 128 layer over {Tn} rows of a "
                                   f"{dt} cache (fp8: per-tensor scales {ks}, {vs}), one C-ABI call per step"
                                   + (f", ck_attn_decode_gqa_split with splits={S}" if S >= 0 else ""),
                       "l2": f"inputs larger than L2: {R} cache replicas rotated "
                             f"({R * per_rep / 2**20:.0f} MiB)"},
            "step_hbm_gbs": round(ach, 1), "step_bytes": kv_bytes,
            "roofline": {"kernel": "attention (split + combine, one call)", "bound": "hbm", "achieved": round(ach, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                         "peak_kind": f"{peak_kind} hbm_gbs",
                         "traffic": profiled_traffic(
                             (f"k_attn_split@attn{Tn}_{dt}" if dt == "f32" else f"k_attn_tc@attn{Tn}_{dt}")
                             + ("" if S < 0 else f"_s{S}"),
                             "quantized_weight_attention_gb300/csrc/" +
                             ("ck_attn_kernels.cuh" if dt == "f32" else "ck_attn_tc.cu"))},
            "e2e": {"value": round(ws * Ke / (e2e_ms / 1e3), 1), "unit": "attention-calls/s",
                    "h2d_bytes_per_step": H * hd * 4, "d2h_bytes_per_step": H * hd * 4, "steps": Ke,
                    "how": "per call: pinned q -> device, the attention call, out -> pinned host"},
            "gpu_launches": 2 * K, "clocks": clocks}
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        line["cpu_baseline"] = cpu_baseline_attn(synth, dt, args.cpu_seconds, args.rows)
    return line


def cpu_baseline_attn(synth, dt, budget_s, rows=0):
    """The oracle attention over the same shape and cache type, calls until the budget."""
    import oracle
    oracle.lib()
    H, KV, hd, Tn, C = attn_kv_shape(synth, rows)
    rng = np.random.default_rng(7)
    qv = rng.standard_normal(H * hd).astype(np.float32)
    if dt == "fp8":
        kc = (rng.integers(0, 0x7F, (KV, C, hd)) | (rng.integers(0, 2, (KV, C, hd)) << 7)).astype(np.uint8)
        vc = kc[::-1].copy()
    else:
        k = rng.standard_normal((KV, C, hd)).astype(np.float32)
        kc = oracle.bf16_from_f32(k) if dt == "bf16" else k
        vc = kc[::-1].copy()
    n, t0 = 0, time.perf_counter()
    while True:
        if dt == "f32":
            oracle.attention(qv, kc, vc, H, KV, Tn, C, hd)
        else:
            oracle.attention_kvq(qv, kc, vc, H, KV, Tn, C, hd, oracle.KV_BF16 if dt == "bf16" else oracle.KV_FP8,
                                 0.01, 0.01)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(n / el, 4), "unit": "attention-calls/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} full attention calls ({Tn} rows, {dt} cache) by the single-threaded C oracle, "
                      f"{el:.1f} s, cpu: {cpu_model()}"}


def paged_plan(synth, bs):
    """The batched64 sequences (lengths from its seed) in a pool of bs-row
    blocks placed in a shuffled order: tables [B, max_blocks], lengths [B]."""
    w = synth.WORKLOADS["batched64"]
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lens = synth.batched_lengths(w, rng).astype(np.int32)
    maxb = -(-int(w.kv_hi + 1) // bs)
    need = [-(-int(n) // bs) for n in lens]
    nblk = int(sum(need))
    order = np.random.Generator(np.random.PCG64(w.seed + 1)).permutation(nblk).astype(np.int32)
    tables = np.zeros((w.batch, maxb), np.int32)
    o = 0
    for b, k in enumerate(need):
        tables[b, :k] = order[o:o + k]
        o += k
    return w, lens, tables, maxb, nblk


def run_paged(args, ws, pg, torch, q, synth, dev):
    """Paged decode attention for the 64 batched64 sequences: one C-ABI call
    per step (a token for every sequence), the pool holding exactly their rows
    in shuffled blocks."""
    bs, dt, win = args.block_size, args.kv_dtype, args.window
    w, lens, tables, maxb, nblk = paged_plan(synth, bs)
    B, H, KV, hd = w.batch, w.H, w.KV, w.hd
    es = KV_ES[dt]
    kind = {"f32": 0, "bf16": 1, "fp8": 2}[dt]
    gen = torch.Generator(device=dev)
    gen.manual_seed(9)
    shape = (nblk, KV, bs, hd)
    if dt == "fp8":
        mk = lambda: (torch.randint(0, 0x7F, shape, generator=gen, device=dev, dtype=torch.int32) |
                      (torch.randint(0, 2, shape, generator=gen, device=dev, dtype=torch.int32) << 7)).to(torch.uint8)
    else:
        f = torch.float32 if dt == "f32" else torch.bfloat16
        mk = lambda: torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(f)
    kp, vp = mk(), mk()
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    td, ld = T(tables), T(lens)
    qv = torch.randn(B * H * hd, generator=gen, device=dev, dtype=torch.float32)
    out = torch.empty(B * H * hd, dtype=torch.float32, device=dev)
    nbytes = q.ck_attn_paged_scratch_size(B, H, KV, hd, bs, maxb, win)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ks = vs = 0.01

    def call(qin=None):
        return q.ck_attn_decode_gqa_paged(qv if qin is None else qin, kp, vp, out, td, ld, B, H, KV, hd, bs, maxb,
                                          nblk, win, kind, ks, vs, scratch, nbytes, stream.cuda_stream)

    with torch.cuda.stream(stream):
        q.check(call())
    torch.cuda.synchronize()
    n_g = 10
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n_g):
            q.check(call())
    K = min(max(1, -(-args.steps // n_g)) * n_g, 400)
    W = max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for _ in range(-(-W // n_g)):
            g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(K // n_g):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    rows = int(sum(min(int(n), win) if win > 0 else int(n) for n in lens))
    kv_bytes = rows * KV * hd * es * 2
    ach = kv_bytes * ws * K / sec / 1e9
    peak, peak_kind = measured_peaks()
    Ke = min(K, 200)
    qh = qv.cpu().pin_memory()
    oh = torch.empty(B * H * hd, dtype=torch.float32).pin_memory()
    qd = torch.empty_like(qv)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            qd.copy_(qh, non_blocking=True)
            q.check(call(qd))
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1))
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    line = {"metric": "paged decode attention tokens/s and achieved HBM GB/s vs GB300 peak",
            "value": round(ws * B * K / sec, 1), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {"f32": "f32", "bf16": "bf16 cache, f32 math", "fp8": "fp8 e4m3 cache, f32 math"}[dt],
            "data": "synthetic",
            "config": {"workload": f"paged64: the 64 batched64 sequences (lengths uniform in [{w.kv_lo}, {w.kv_hi}], "
                                   f"sum {int(sum(lens))}) in a pool of {nblk} blocks of {bs} rows ({dt}), "
                                   f"shuffled; window {win or 'none'} ({rows} rows attended); one call per step",
                       "l2": f"{kv_bytes / 1e9:.2f} GB per step >> L2"},
            "step_hbm_gbs": round(ach, 1), "step_bytes": kv_bytes,
            "roofline": {"kernel": "paged attention (split + combine, one call)", "bound": "hbm",
                         "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                         "peak_kind": f"{peak_kind} hbm_gbs", "traffic": None},
            "e2e": {"value": round(ws * B * Ke / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": B * H * hd * 4, "d2h_bytes_per_step": B * H * hd * 4, "steps": Ke,
                    "how": "per call: pinned q [B, H*hd] -> device, the paged attention call, out -> pinned host"},
            "gpu_launches": 2 * K, "clocks": clocks}
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        line["cpu_baseline"] = cpu_baseline_paged(synth, dt, bs, win, args.cpu_seconds)
    return line


def cpu_baseline_paged(synth, dt, bs, win, budget_s):
    """The oracle paged attention sequence by sequence (the same lengths and
    block size) until the budget: tokens/s over the sequences done."""
    import oracle
    oracle.lib()
    w, lens, tables, maxb, nblk = paged_plan(synth, bs)
    H, KV, hd = w.H, w.KV, w.hd
    kind = {"f32": 0, "bf16": 1, "fp8": 2}[dt]
    rng = np.random.default_rng(9)
    done, el = 0, 0.0
    for b in range(w.batch):
        need = -(-int(lens[b]) // bs)
        if dt == "fp8":
            kp = (rng.integers(0, 0x7F, (need, KV, bs, hd)) | (rng.integers(0, 2, (need, KV, bs, hd)) << 7)
                  ).astype(np.uint8)
        else:
            kf = rng.standard_normal((need, KV, bs, hd)).astype(np.float32)
            kp = oracle.bf16_from_f32(kf) if dt == "bf16" else kf
        qv = rng.standard_normal(H * hd).astype(np.float32)
        tbl = np.arange(need, dtype=np.int32)[None, :]
        t0 = time.perf_counter()
        oracle.attention_paged(qv, kp, kp, tbl, [int(lens[b])], 1, H, KV, hd, bs, need, win, kind, 0.01, 0.01)
        el += time.perf_counter() - t0
        done += 1
        if el >= budget_s:
            break
    return {"value": round(done / el, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of the 64 sequences (paged, {dt}, block {bs}, window {win or 'none'}) by the "
                      f"single-threaded C oracle, {el:.1f} s, cpu: {cpu_model()}"}


PREFILL_POS, PREFILL_N = 7680, 512  # the last 512-token chunk of an 8192-token prompt
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12  # fp32 FMA lanes x 2 flops x max SM clock


def prefill_workload(synth):
    return dataclasses.replace(synth.WORKLOADS["7b8k"], pos=PREFILL_POS)


def prefill_attn_flops(pos, n, H, hd):
    """QK and PV, 2 flops per multiply-add each: token i sees pos + i + 1 rows."""
    rows = n * pos + n * (n + 1) // 2
    return 4 * rows * H * hd


def run_prefill(args, ws, pg, torch, q, synth, dev):
    """The 7B-shaped layer prefilling tokens 7680..8191 of a prompt in one
    ck_prefill_layer call per step (512 tokens, causal over the cache);
    replicas of weights and caches rotate to keep the working set over L2."""
    w = prefill_workload(synth)
    P, n = PREFILL_POS, PREFILL_N
    rng = np.random.Generator(np.random.PCG64(w.seed))
    gamma, wq, wk, wv, wo, bq, bk, bv, bo = synth.draw_weights(rng, w)
    x0 = rng.standard_normal((n, w.D)).astype(np.float32)
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    per_rep = w.weight_bytes() + 2 * w.KV * w.capacity * w.hd * 4
    R = max(1, -(-3 * l2 // per_rep))
    gen = torch.Generator(device=dev)
    reps = []
    for r in range(R):
        g = dict(gamma=T(gamma), wq=T(wq), wk=T(wk), wv=T(wv), wo=T(wo), bq=T(bq), bk=T(bk), bv=T(bv), bo=T(bo))
        gen.manual_seed(w.seed * 100 + r)
        g["kc"] = torch.zeros((w.KV, w.capacity, w.hd), dtype=torch.float32, device=dev)
        g["vc"] = torch.zeros_like(g["kc"])
        g["kc"][:, :P].normal_(generator=gen)
        g["vc"][:, :P].normal_(generator=gen)
        reps.append(g)
    cosd, sind = T(cos), T(sin)
    xd = T(x0)
    out = torch.empty((n, w.D), dtype=torch.float32, device=dev)
    nbytes = q.ck_prefill_layer_scratch_size(n, w.D, w.H, w.KV, w.hd, w.capacity)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(g, xin):
        q.check(q.ck_prefill_layer(out, xin, xin, g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"], g["bk"],
                                   g["bv"], g["bo"], g["kc"], g["vc"], cosd, sind, P, n, w.D, w.H, w.KV, w.hd,
                                   w.capacity, w.eps, scratch, nbytes, stream.cuda_stream))

    with torch.cuda.stream(stream):
        step(reps[0], xd)
    torch.cuda.synchronize()
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for g in reps:
            step(g, xd)
    K = max(1, -(-min(args.steps, 400) // R)) * R
    W = max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for _ in range(-(-W // R)):
            graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(K // R):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    fl = prefill_attn_flops(P, n, w.H, w.hd)
    ach = fl * K / sec / 1e12

    # the chunk's attention alone (ck_attn_prefill_gqa: K / V image + the
    # tensor-core kernel), on the replicas' caches, calls in a CUDA graph
    qa = torch.randn((n, w.H * w.hd), generator=gen, device=dev, dtype=torch.float32)
    oa = torch.empty_like(qa)
    anb = q.ck_attn_prefill_scratch_size(w.H, w.KV, w.hd, w.capacity)
    asc = torch.empty(anb, dtype=torch.uint8, device=dev)

    def attn(g):
        q.check(q.ck_attn_prefill_gqa(qa, g["kc"], g["vc"], oa, P, n, w.H, w.KV, w.hd, w.capacity, asc, anb,
                                      stream.cuda_stream))

    ag = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ag, stream=stream):
        for g in reps:
            attn(g)
    with torch.cuda.stream(stream):
        for _ in range(2):
            ag.replay()
    torch.cuda.synchronize()
    Ka = max(1, K // R) * R
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a0.record(stream)
        for _ in range(Ka // R):
            ag.replay()
        a1.record(stream)
    a1.synchronize()
    attn_ms = max_over_ranks(pg, torch, a0.elapsed_time(a1)) / Ka
    attn_tf = fl / (attn_ms / 1e3) / 1e12
    bf16_peak = 1941.2
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak, bf16_kind = float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except (OSError, KeyError, ValueError):
        bf16_peak, bf16_kind = 1900.0, "fallback bf16"

    # e2e: the chunk's rows from pinned host memory, its output rows back
    Ke = min(K, 50)
    xh = torch.from_numpy(x0).pin_memory()
    oh = torch.empty((n, w.D), dtype=torch.float32).pin_memory()
    xe = torch.empty((n, w.D), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(Ke):
            xe.copy_(xh, non_blocking=True)
            step(reps[i % R], xe)
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1))
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    line = {"metric": "prefill tokens/s of the layer (causal chunk over the cache)",
            "value": round(ws * n * K / sec, 1), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8/int5 codes: exact integer block dots (tcgen05 f16); attention in bf16 hi/lo pairs "
                     "(tcgen05, fp32 accumulation)", "data": "synthetic",
            "config": {"workload": f"prefill512: the D=3584 28/4-head hd=128 layer, tokens {P}..{P + n - 1} of one "
                                   f"sequence in one ck_prefill_layer call per step (causal: token i attends "
                                   f"{P} + i + 1 rows)",
                       "l2": f"{R} replicas of weights + caches ({per_rep / 1e6:.0f} MB each) in rotation"},
            "attn_flops_per_step": fl, "step_attn_tflops": round(ach, 2),
            "attn_alone": {"ms_per_call": round(attn_ms, 5), "calls": Ka,
                           "how": "ck_attn_prefill_gqa on the same chunk and caches, calls in a CUDA graph"},
            "roofline": {"kernel": "prefill attention (K/V image + tcgen05 kernel, one ck_attn_prefill_gqa call)",
                         "bound": "tensor", "achieved": round(attn_tf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(attn_tf / bf16_peak, 4),
                         "peak_kind": f"{bf16_kind}; the split-precision operands take 3 bf16 MMAs per product, "
                                      f"so this kernel's algorithmic ceiling is 1/3 of the peak",
                         "traffic": profiled_traffic("k_pf_attn@prefill512",
                                                     "quantized_weight_attention_gb300/csrc/ck_prefill_attn.cu")},
            "e2e": {"value": round(ws * n * Ke / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": n * w.D * 4, "d2h_bytes_per_step": n * w.D * 4, "steps": Ke,
                    "how": "per step: pinned x [n, D] -> device, ck_prefill_layer, out -> pinned host"},
            "gpu_launches": 6 * K, "clocks": clocks}
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        line["cpu_baseline"] = cpu_baseline_prefill(synth, args.cpu_seconds)
    return line


def cpu_baseline_prefill(synth, budget_s):
    """The oracle's prefill form on the first m tokens of the chunk (m sized
    from a 4-token probe to fill about budget_s): tokens/s."""
    import oracle
    oracle.lib()
    w = prefill_workload(synth)
    P = PREFILL_POS
    rng = np.random.Generator(np.random.PCG64(w.seed))
    gamma, wq, wk, wv, wo, bq, bk, bv, bo = synth.draw_weights(rng, w)
    x0 = rng.standard_normal((PREFILL_N, w.D)).astype(np.float32)
    kc, vc = synth.draw_cache(rng, w, P)
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)

    def run(m):
        k2, v2 = kc.copy(), vc.copy()
        t0 = time.perf_counter()
        oracle.prefill_layer(x0[:m], x0[:m], wq, wk, wv, wo, gamma, bq, bk, bv, bo, k2, v2, cos, sin, P, m, w.D, w.H,
                             w.KV, w.hd, w.capacity, w.eps)
        return time.perf_counter() - t0

    t4 = run(4)
    m = int(min(PREFILL_N, max(4, budget_s / max(t4 / 4, 1e-6))))
    el = run(m)
    return {"value": round(m / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"tokens {P}..{P + m - 1} ({m} of the 512) by the single-threaded C oracle's prefill form, "
                      f"{el:.1f} s, cpu: {cpu_model()}"}


def run_batched(args, ws, pg, torch, q, synth, dev):
    """64 sequences of the 7B-shaped layer with ragged caches (lengths uniform
    in [512, 16384]): one ck_decode_layer_batched call per step."""
    w = synth.WORKLOADS["batched64"]
    B = w.batch
    rng = np.random.Generator(np.random.PCG64(w.seed))
    lens = synth.batched_lengths(w, rng)
    gamma, wq, wk, wv, wo, bq, bk, bv, bo = synth.draw_weights(rng, w)
    x0 = rng.standard_normal((B, w.D)).astype(np.float32)
    capped = ""
    if args.kv_cap > 0:
        w = dataclasses.replace(w, capacity=min(w.capacity, args.kv_cap))
        lens = np.minimum(lens, w.capacity - 1).astype(np.int32)
        capped = f" (caches capped at {w.capacity} rows: a profiling case)"
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    g = dict(gamma=T(gamma), wq=T(wq), wk=T(wk), wv=T(wv), wo=T(wo), bq=T(bq), bk=T(bk), bv=T(bv), bo=T(bo),
             cos=T(cos), sin=T(sin))
    gen = torch.Generator(device=dev)
    kcs, vcs = [], []
    for s in range(B):
        gen.manual_seed(w.seed * 1000 + s)
        kc = torch.zeros((w.KV, w.capacity, w.hd), dtype=torch.float32, device=dev)
        vc = torch.zeros_like(kc)
        kc[:, :lens[s]].normal_(generator=gen)
        vc[:, :lens[s]].normal_(generator=gen)
        kcs.append(kc)
        vcs.append(vc)
    kptr = torch.tensor([c.data_ptr() for c in kcs], dtype=torch.int64, device=dev)
    vptr = torch.tensor([c.data_ptr() for c in vcs], dtype=torch.int64, device=dev)
    d_pos = T(lens)
    xd = T(x0)
    out = torch.empty((B, w.D), dtype=torch.float32, device=dev)
    nbytes = q.ck_decode_layer_batched_scratch_size(B, w.D, w.H, w.KV, w.hd, w.capacity)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(xin):
        q.check(q.ck_decode_layer_batched(out, xin, xin, g["wq"], g["wk"], g["wv"], g["wo"], g["gamma"], g["bq"],
                                          g["bk"], g["bv"], g["bo"], kptr, vptr, g["cos"], g["sin"], d_pos, B, w.D,
                                          w.H, w.KV, w.hd, w.capacity, w.eps, scratch, nbytes, stream.cuda_stream))

    with torch.cuda.stream(stream):
        step(xd)
    torch.cuda.synchronize()
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(xd)
    K, W = min(args.steps, 2000), max(args.warmup, 3)
    with torch.cuda.stream(stream):
        for _ in range(W):
            graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid(torch, dev))
    sampler.start()
    time.sleep(0.3)
    barrier(pg, torch)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        ev0.record(stream)
        for _ in range(K):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(pg, torch)
    clocks = sampler.stop()
    ms = max_over_ranks(pg, torch, ev0.elapsed_time(ev1))
    sec = ms / 1e3
    kv_bytes = int(sum((int(n) + 1) * w.KV * w.hd * 4 * 2 for n in lens))
    per_step = w.weight_bytes() + kv_bytes
    peak, peak_kind = measured_peaks()
    ach = per_step * ws * K / sec / 1e9

    # e2e: the B input rows from pinned host memory, the B output rows back
    Ke = min(K, 200)
    xh = torch.from_numpy(x0).pin_memory()
    oh = torch.empty((B, w.D), dtype=torch.float32).pin_memory()
    xe = torch.empty((B, w.D), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            xe.copy_(xh, non_blocking=True)
            step(xe)
            oh.copy_(out, non_blocking=True)
        e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(pg, torch, e0.elapsed_time(e1))
    rc, st = q.ck_device_status()
    assert rc == 0 and st == 0, (rc, st)
    line = {"metric": METRIC, "value": round(ws * B * K / sec, 1), "unit": "tokens/s", "n_gpus": ws, "steps": K,
            "warmup": W, "ms_per_step": round(ms / K, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8/int5 codes: exact integer block dots (tcgen05 f16, dp4a), fp32",
            "data": "synthetic",
            "config": {"workload": f"batched64: {B} sequences of the D=3584 28/4-head layer sharing its weights, "
                                   f"cache lengths uniform in [{w.kv_lo}, {w.kv_hi}] (sum {int(sum(lens))}), "
                                   f"one ck_decode_layer_batched call per step{capped}",
                       "l2": f"{per_step / 1e9:.2f} GB per step >> L2"},
            "step_hbm_gbs": round(ach, 1), "step_bytes": per_step,
            "roofline": {"kernel": "whole batched step", "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(ach / peak, 4), "peak_kind": f"{peak_kind} hbm_gbs",
                         "traffic": None},
            "e2e": {"value": round(ws * B * Ke / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": B * w.D * 4, "d2h_bytes_per_step": B * w.D * 4, "steps": Ke,
                    "how": "per step: pinned x [B, D] -> device, ck_decode_layer_batched, out -> pinned host"},
            "gpu_launches": 5 * K, "clocks": clocks}
    if not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        line["cpu_baseline"] = cpu_baseline_batched(w, lens, gamma, wq, wk, wv, wo, bq, bk, bv, bo, x0, cos, sin,
                                                    args.cpu_seconds)
    return line


def cpu_baseline_batched(w, lens, gamma, wq, wk, wv, wo, bq, bk, bv, bo, x0, cos, sin, budget_s):
    """The oracle's decode step run sequence after sequence (each on its own
    cache) until budget_s: tokens/s over the sequences done (cache drawing is
    not timed)."""
    import oracle
    oracle.lib()
    rng = np.random.Generator(np.random.PCG64(w.seed + 100))
    done, el = 0, 0.0
    for s in range(w.batch):
        kc = np.zeros((w.KV, w.capacity, w.hd), np.float32)
        vc = np.zeros((w.KV, w.capacity, w.hd), np.float32)
        n = int(lens[s])
        kc[:, :n] = rng.standard_normal((w.KV, n, w.hd), dtype=np.float32)
        vc[:, :n] = rng.standard_normal((w.KV, n, w.hd), dtype=np.float32)
        t0 = time.perf_counter()
        oracle.decode_layer(x0[s], x0[s], wq, wk, wv, wo, gamma, bq, bk, bv, bo, kc, vc, cos, sin, n, w.D, w.H, w.KV,
                            w.hd, w.capacity, w.eps)
        el += time.perf_counter() - t0
        done += 1
        if el >= budget_s:
            break
    return {"value": round(done / el, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} of the {w.batch} sequences' decode steps (cache lengths "
                      f"{', '.join(str(int(v)) for v in lens[:done])}) by the single-threaded C oracle, "
                      f"{el:.1f} s, cpu: {cpu_model()}"}


# --------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------
def oracle_steps(w, budget_s: float, max_steps: int | None = None):
    """Times full oracle decode steps of workload w until budget_s (at least
    one step) or max_steps.  Returns (steps, seconds)."""
    import oracle
    from quantized_weight_attention_gb300 import synth
    L = synth.make_layer(w)
    cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
    kc, vc = L.k_cache.copy(), L.v_cache.copy()
    oracle.lib()
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_layer(L.x, L.x, L.wq, L.wk, L.wv, L.wo, L.gamma, L.bq, L.bk, L.bv, L.bo, kc, vc, cos, sin,
                            w.pos, w.D, w.H, w.KV, w.hd, w.capacity, w.eps)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps is not None and n >= max_steps):
            return n, el


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(w, budget_s):
    n, el = oracle_steps(w, budget_s)
    return {"value": round(n / el, 3), "unit": "layer-steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} full decode steps of the {w.name} layer by the single-threaded C oracle "
                      f"(double accumulation), {el:.1f} s, cpu: {cpu_model()}"}


def run_reference(args, ws):
    from quantized_weight_attention_gb300 import synth
    if args.config == "prefill512":  # the oracle prefill form, as the CPU baseline
        cb = cpu_baseline_prefill(synth, 30.0)
        return {"impl": "reference", "metric": "prefill tokens/s of the layer (causal chunk over the cache)",
                "value": cb["value"], "unit": "tokens/s", "n_gpus": ws, "steps": 1, "warmup": 0,
                "ms_per_step": round(1e3 * PREFILL_N / cb["value"], 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64 accumulation (C oracle)", "data": "synthetic",
                "config": {"workload": "prefill512 (same as the GPU arm)"},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
    if args.config == "paged64":  # the oracle paged attention, as the CPU baseline
        cb = cpu_baseline_paged(synth, args.kv_dtype, args.block_size, args.window, 60.0)
        return {"impl": "reference", "metric": "paged decode attention tokens/s and achieved HBM GB/s vs GB300 peak",
                "value": cb["value"], "unit": "tokens/s", "n_gpus": ws, "steps": 1, "warmup": 0,
                "ms_per_step": round(1e3 * 64 / cb["value"], 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64 accumulation (C oracle)", "data": "synthetic",
                "config": {"workload": f"paged64, {args.kv_dtype} cache (same as the GPU arm)"},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
    if args.config == "attn32k":  # the oracle attention, as the CPU baseline
        cb = cpu_baseline_attn(synth, args.kv_dtype, 60.0, args.rows)
        return {"impl": "reference", "metric": "decode attention calls/s and achieved HBM GB/s vs GB300 peak",
                "value": cb["value"], "unit": "attention-calls/s", "n_gpus": ws, "steps": 1, "warmup": 0,
                "ms_per_step": round(1e3 / cb["value"], 3), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64 accumulation (C oracle)", "data": "synthetic",
                "config": {"workload": f"attn32k, {args.kv_dtype} cache (same as the GPU arm)"},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "attention-calls/s",
                                            "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    w = synth.WORKLOADS[args.config]
    if args.config == "batched64":  # the oracle sequence after sequence, within a few minutes
        rng = np.random.Generator(np.random.PCG64(w.seed))
        lens = synth.batched_lengths(w, rng)
        gamma, wq, wk, wv, wo, bq, bk, bv, bo = synth.draw_weights(rng, w)
        x0 = rng.standard_normal((w.batch, w.D)).astype(np.float32)
        cos, sin = synth.rope_tables(w.capacity, w.hd, w.theta)
        cb = cpu_baseline_batched(w, lens, gamma, wq, wk, wv, wo, bq, bk, bv, bo, x0, cos, sin, 120.0)
        return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": ws,
                "steps": 1, "warmup": 0, "ms_per_step": round(1e3 * w.batch / cb["value"], 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64 accumulation (C oracle)", "data": "synthetic",
                "config": {"workload": f"{w.name} (same as the GPU arm)"},
                "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
    # each step is one full oracle decode step; the number timed is capped so
    # that warm-up + timed steps end within a few minutes
    budget = 150.0
    _, per = oracle_steps(w, 0.0, max_steps=1)
    per = max(per, 1e-6)
    W = min(max(args.warmup, 0), int(20.0 / per))
    if W:
        oracle_steps(w, 1e9, max_steps=W)
    K = max(1, min(args.steps, int(budget / per)))
    n, el = oracle_steps(w, 1e9, max_steps=K)
    v = n / el
    unit = "tokens/s" if args.config == "stack32k" else "layer-steps/s"
    if args.config == "stack32k":
        v /= w.layers
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": unit, "n_gpus": ws, "steps": n,
            "warmup": W, "ms_per_step": round(1e3 * el / n, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 accumulation (C oracle)", "data": "synthetic",
            "config": {"workload": f"{w.name} (same as the GPU arm)",
                       "note": f"{n} of the requested {args.steps} steps timed to stay within {budget:.0f} s"},
            "cpu_baseline": {"value": round(v, 4), "unit": unit, "cores": 1, "kind": "oracle",
                             "sample": f"{n} full decode layer steps, single-threaded, cpu: {cpu_model()}"},
            "e2e": {"value": round(v, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":  # rank 0 alone; the other ranks exit without work
        ws, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
        if rank == 0:
            print(json.dumps(run_reference(args, ws)), flush=True)
        return
    ws, rank, local, pg = dist_setup()
    line = run_ours(args, ws, rank, local, pg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
