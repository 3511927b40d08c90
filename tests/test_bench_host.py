"""Host-side accounting of bench.py (no GPU): the executed tensor-core FLOPs
of the fused kernel's plan, against closed forms worked out by hand."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_prefix_cache_gb300 import workload as W  # noqa: E402

UP = 2.0 * 512 * 256          # per token and head
ATT = 2.0 * (192 + 128)       # per (query, key, head)


def test_executed_flops_tiny_by_hand():
    # C = 256, E = 64, chunk 128: the chunks and the extend join into one piece
    # [0, 320) = 3 tiles of 128 keys; 2 producer passes of 256 tokens; one
    # consumer pair (M = 256 rows, one of its query tiles empty) over 3 tiles.
    wl = W.tiny()
    H = 8
    expect = H * (2 * 256 * UP + 3 * 256 * 128 * ATT)
    assert bench.executed_flops(wl) == expect


def test_executed_flops_documents_by_hand():
    # two relocated documents of 64 tokens (separate pieces: different RoPE
    # offsets) and 130 new tokens: pieces [0, 64), [64, 128), [128, 258)
    wl = W.make_workload("d", 2, [128], [130], chunk=64, seed=1, doc_len=64)
    H = 2
    up = H * UP * 256 * (1 + 1 + 1)                 # 1, 1 and ceil(ceil(130/128)/2) = 1 passes
    # consumer pair: query tiles 0 (rows 0..127) and 1 (rows 128..129)
    # documents: 1 tile each; extend piece [128, 258): tile 1 of the pair sees all 130 keys -> 2 tiles
    att = H * 256 * 128 * ATT * (1 + 1 + 2)
    assert bench.executed_flops(wl) == up + att


def test_executed_at_least_algorithmic():
    for name in ("tiny", "v3_8k"):
        wl = W.by_name(name)
        assert bench.executed_flops(wl) >= wl.algorithmic_flops()
