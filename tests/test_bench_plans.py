"""Host-side plans of bench.py's workloads (no GPU): the paged pool of the
paged64 workload and the prefill chunk's flop count."""
import numpy as np

import bench
from quantized_weight_attention_gb300 import synth


def test_paged_plan_uses_every_block_once():
    for bs in (16, 64):
        w, lens, tables, maxb, nblk = bench.paged_plan(synth, bs)
        assert len(lens) == w.batch and tables.shape == (w.batch, maxb)
        need = [-(-int(n) // bs) for n in lens]
        assert sum(need) == nblk and maxb * bs >= int(lens.max())
        used = np.concatenate([tables[b, :k] for b, k in enumerate(need)])
        assert np.array_equal(np.sort(used), np.arange(nblk))  # a permutation of the pool
        assert not np.array_equal(used, np.arange(nblk))        # shuffled, not contiguous
        # the lengths are those of the batched64 workload
        rng = np.random.Generator(np.random.PCG64(w.seed))
        assert np.array_equal(lens, synth.batched_lengths(w, rng))


def test_prefill_flops_count_each_attended_row():
    H, hd = 28, 128
    # token i sees pos + i + 1 rows; 4 flops per row element and head
    assert bench.prefill_attn_flops(0, 1, H, hd) == 4 * 1 * H * hd
    assert bench.prefill_attn_flops(10, 3, H, hd) == 4 * (11 + 12 + 13) * H * hd
    brute = sum(4 * (7680 + i + 1) * H * hd for i in range(512))
    assert bench.prefill_attn_flops(7680, 512, H, hd) == brute
