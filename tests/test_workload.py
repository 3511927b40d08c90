"""Host-side checks of the seeded input generator (no method arithmetic)."""
import math

import numpy as np

from mla_prefix_cache_gb300 import workload as W


def test_block_pool_and_sentinels():
    wl = W.make_workload("w", 2, [100, 64], [30, 1], seed=0)
    seq = wl.seq_lens
    need = [math.ceil(s / 64) for s in seq]
    used = np.concatenate([wl.block_table[r, :n] for r, n in enumerate(need)])
    assert len(set(used.tolist())) == len(used)                       # no block shared
    assert wl.num_blocks == sum(need) + math.ceil(0.1 * sum(need))    # 10 % spare
    assert (wl.block_table[1, need[1]:] == -1).all()
    bits = wl.kv_cache
    nan = (bits & 0x7FFF) > 0x7F80
    spare = sorted(set(range(wl.num_blocks)) - set(used.tolist()))
    assert nan[spare].all()
    # tail slots of the last block of request 0 (130 tokens -> block 2 slots 2..63)
    assert nan[wl.block_table[0, 2], 2:].all() and not nan[wl.block_table[0, 2], :2].any()
    assert not nan[wl.block_table[1, 0]].any()


def test_fp8_pool_and_scale():
    wl = W.make_workload("f", 1, [64], [65], kv_dtype="fp8_e4m3", seed=1)
    assert wl.kv_cache.shape[-1] == 640 and wl.kv_cache.dtype == np.uint8
    b1 = wl.block_table[0, 2]
    assert (wl.kv_cache[b1, 1:, :512] == 0x7F).all()                  # e4m3 NaN sentinel
    assert wl.kv_scale > 0


def test_reloc_segments():
    wl = W.make_workload("r", 1, [256], [3], doc_len=64, seed=2)
    assert wl.segments.tolist() == [[0, 0, 64, 0], [0, 64, 64, 64], [0, 128, 64, 128], [0, 192, 64, 192]]
    assert wl.q_pos.tolist() == [256, 257, 258]


def test_flop_formula_against_derived_totals():
    # Derived totals for the tiny and DeepSeek-V3 8K workloads:
    # up-projection 2*512*256*H per token, attention 2*(192+128)*H per visible pair.
    assert W.tiny().algorithmic_flops() == 320 * 262144 * 8 + 64 * 256 * 640 * 8 + 64 * 65 // 2 * 640 * 8
    assert abs(W.tiny().algorithmic_flops() - 7.66e8) / 7.66e8 < 1e-3
    wl = W.make_workload("v", 128, [8192], [2048], seed=1)
    assert abs(wl.algorithmic_flops() - 1.89e12) / 1.89e12 < 5e-3


def test_seeded_determinism():
    a = W.make_workload("a", 2, [64], [5], seed=3)
    b = W.make_workload("a", 2, [64], [5], seed=3)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.kv_cache, b.kv_cache)
    assert np.array_equal(a.kv_b_proj, b.kv_b_proj)
