"""C-ABI checks that need no GPU: the library loads, exports every symbol that
include/mla.h declares, and its host-side validation and planner behave."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_prefix_cache_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, n


def test_status_strings(lib):
    assert _lib.status_string(0) == "MLA_OK"
    assert _lib.status_string(5) == "MLA_ERR_WORKSPACE"
    assert lib.mla_abi_version() == 1


def _ws(lib, seq, cu, H, segs=None, chunk=128, parts=3):
    sl, k1 = _lib.i32_host(seq)
    cq, k2 = _lib.i32_host(cu)
    sp, ns, k3 = _lib.segments_host(segs)
    return lib.mla_prefill_workspace_size(len(k1), sl, cq, H, sp, ns, chunk, parts)


def _up(x, a=256):
    return (x + a - 1) // a * a


def fused_layout(pieces, heads, slots, total_q, seq_lens, ring_depth=128, ring_lanes=None, max_tiles=None,
                 min_pairs=None):
    """Workspace of the fused path: 256 B header, per-job ring flags, the K/V
    ring lanes (`ring_lanes` x `ring_depth` 128-token bf16 tiles, shared by
    the jobs in turn, then the K_nope residual tiles of each lane's first 16
    slots), the gathered rows (1152 B per token, whole 64-token
    blocks), then partial states."""
    jobs = pieces * heads
    if ring_lanes is None:   # 32 MiB of the longest piece's tiles, or 76 pairs over a job's fewest, within [4, 64]
        fit = (32 << 20) // (128 * 256 * 2 * min(max_tiles, ring_depth))
        ring_lanes = max(4, min(64, max(fit, 76 // min_pairs)))
    ring_lanes = min(ring_lanes, jobs)       # no more lanes than jobs
    ring_off = _up(256 + jobs * 2 * ring_depth * 4)
    gath_off = _up(ring_off + ring_lanes * (ring_depth * 128 * 256 + min(ring_depth, 16) * 128 * 128) * 2)
    gath = sum((s + 63) // 64 for s in seq_lens) * 64 * 1152
    lse_off = _up(gath_off + gath)
    rows = slots * total_q * heads
    return _up(lse_off + rows * 4) + rows * 128 * 4


def test_workspace_size_follows_plan(lib):
    # 1 request, C=256 in chunks of 128 plus the extend: the three ranges share
    # offset 0 and are contiguous, so they fold into one piece (no partial slots).
    # (pairs of a job: max(1, ceil(producer CTAs / 2)) + ceil(query tiles / 2), producer CTAs = min(4, ceil(tiles / 2)))
    n = _ws(lib, [320], [0, 64], 8, chunk=128)
    assert n == fused_layout(1, 8, 0, 64, [320], ring_depth=4, max_tiles=3, min_pairs=2)
    # segments: 4 documents of 64 (4 offsets) + extend = 5 pieces, 5 partial slots
    segs = [[0, 64 * d, 64, 64 * d] for d in range(4)]
    assert _ws(lib, [258], [0, 2], 1, segs=segs, chunk=64) == fused_layout(5, 1, 5, 2, [258], ring_depth=4,
                                                                          max_tiles=1, min_pairs=2)
    # a long context is cut into pieces of at most max(chunk, 16384) keys:
    # 16384 + 16384 + 7232 + 100; 3 pairs a job -> 25 lanes
    assert _ws(lib, [40000 + 100], [0, 100], 2, chunk=4096) == fused_layout(3, 2, 3, 100, [40100], max_tiles=128,
                                                                            min_pairs=3)
    # 8192 + 2048 keys in one piece: 80 tiles, 2 + 8 pairs a job -> 7 lanes of 128 slots
    assert _ws(lib, [10240], [0, 2048], 2, chunk=4096) == fused_layout(1, 2, 0, 2048, [10240], max_tiles=80,
                                                                       min_pairs=10)
    # 16384 cached + 4096 new keys in two pieces: 2 + 16 pairs a job -> 4 lanes
    assert _ws(lib, [20480], [0, 4096], 2, chunk=16384) == fused_layout(2, 2, 2, 4096, [20480], max_tiles=128,
                                                                        min_pairs=18)
    # 1000 keys: 8 tiles -> lanes of 8 slots
    assert _ws(lib, [1000], [0, 100], 3, chunk=512) == fused_layout(1, 3, 0, 100, [1000], ring_depth=8,
                                                                    max_tiles=8, min_pairs=3)


def test_min_workspace_size(lib):
    """The smallest workspace: two ring lanes of 4 tiles, flags of one piece's jobs."""
    sl, k1 = _lib.i32_host([258])
    cq, k2 = _lib.i32_host([0, 2])
    segs = [[0, 64 * d, 64, 64 * d] for d in range(4)]
    sp, ns, k3 = _lib.segments_host(segs)
    n = lib.mla_prefill_min_workspace_size(1, sl, cq, 3, sp, ns, 64, 3)
    assert n == fused_layout(1, 3, 5, 2, [258], ring_depth=4, ring_lanes=2)
    assert n < _ws(lib, [258], [0, 2], 3, segs=segs, chunk=64)
    assert lib.mla_prefill_min_workspace_size(1, sl, cq, 3, sp, ns, 100, 3) == 0    # chunk not a multiple of 64


@pytest.mark.parametrize("bad", [
    dict(chunk=100),                 # not a multiple of 64 -> unsupported
    dict(H=129),                     # more heads than supported
    dict(cu=[1, 64]),                # cu_q[0] != 0
    dict(seq=[10], cu=[0, 64]),      # extend longer than sequence
    dict(segs=[[0, 200, 100, 0]]),   # segment past the context
    dict(segs=[[0, 0, 64, 0], [0, 32, 64, 0]]),  # overlapping segments
    dict(parts=0),
])
def test_planner_rejects(lib, bad):
    args = dict(seq=[320], cu=[0, 64], H=8, segs=None, chunk=128, parts=3)
    args.update(bad)
    assert _ws(lib, args["seq"], args["cu"], args["H"], args["segs"], args["chunk"], args["parts"]) == 0


def test_prefill_host_validation_without_gpu(lib):
    """Invalid calls return a status before any CUDA call is made."""
    sl, k1 = _lib.i32_host([320])
    cq, k2 = _lib.i32_host([0, 64])
    dummy = ctypes.c_void_p(4096)
    def call(chunk=128, H=8, ws=None, ws_bytes=0, kv_dtype=0, theta=10000.0):
        return lib.mla_prefill_ctx(dummy, dummy, dummy, kv_dtype, 1.0, 8, dummy, 8, sl, cq, 1, H, None, 0, chunk,
                                   dummy, 0.07, theta, 3, dummy, 0, dummy, ws, ws_bytes, None)
    assert call(chunk=100) == _lib.MLA_ERR_UNSUPPORTED
    assert call(H=200) == _lib.MLA_ERR_UNSUPPORTED
    assert call(kv_dtype=7) == _lib.MLA_ERR_INVALID_ARG
    assert call(theta=0.5) == _lib.MLA_ERR_INVALID_ARG
    assert call(ws=None, ws_bytes=0) == _lib.MLA_ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p(4096 + 8), ws_bytes=1 << 30) == _lib.MLA_ERR_WORKSPACE  # misaligned


def test_other_entry_points_validate(lib):
    d = ctypes.c_void_p(4096)
    assert lib.mla_merge_states(d, d, d, d, d, d, 10, 6, None) == _lib.MLA_ERR_INVALID_ARG   # d_v % 4
    assert lib.mla_merge_states(d, d, d, d, d, d, 0, 128, None) == _lib.MLA_OK               # nothing to do
    assert lib.mla_rope_relocate(d, d, 0, 10000.0, d, 4, 2, 192, 130, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_rope_relocate(d, d, 0, 10000.0, d, 4, 2, 192, 136, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_gather_latent(d, 0, 1.0, 4, d, 2, 100, 64, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_gather_latent(d, 1, 0.0, 4, d, 2, 0, 64, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_get_device_error(None, None) == _lib.MLA_ERR_INVALID_ARG
    # block store: bad dtype, negative count, null or misaligned pointers; n = 0 launches nothing
    assert lib.mla_block_hash(d, 2, 4, d, 3, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_hash(d, 0, 4, d, -1, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_hash(None, 0, 4, d, 3, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_hash(d, 0, 4, d, 3, ctypes.c_void_p(4100), None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_hash(d, 0, 4, d, 0, d, None, None) == _lib.MLA_OK
    assert lib.mla_block_compare(d, 0, 0, d, d, 3, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_compare(d, 0, 4, d, None, 3, d, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_block_compare(d, 1, 4, d, d, 0, d, None, None) == _lib.MLA_OK


def _abs_layout(blocks, rows, slots=1, header=256):
    """Absorbed-path workspace: header, gathered rows, qlat, `slots` key splits of latent states and lse."""
    want = header + blocks * 64 * 1152
    want = (want + 255) // 256 * 256 + rows * 512 * 2
    want = (want + 255) // 256 * 256 + slots * rows * 512 * 4
    want = (want + 255) // 256 * 256 + slots * rows * 4
    return (want + 255) // 256 * 256


def test_absorbed_entry_validates_and_sizes(lib):
    # 1036 cached + 64 new tokens: every row sees >= 1024 keys, so the whole
    # request takes the absorbed path; the workspace leads with an empty
    # up-projected part (its 256-byte header, flags of one 8-head piece of 4-slot lanes)
    sl, cq = (ctypes.c_int32 * 1)(1100), (ctypes.c_int32 * 2)(0, 64)
    n = lib.mla_prefill_absorbed_workspace_size(1, sl, cq, 8, None, 0, 128, 3)
    fused_part = 256 + 8 * 2 * 4 * 4
    assert any(n == fused_part + _abs_layout(18, 64 * 8, k) for k in range(1, 5))   # the keys cut in 1-4 splits
    assert lib.mla_prefill_absorbed_workspace_size(1, sl, cq, 8, None, 0, 100, 3) == 0   # chunk not a multiple of 64
    # 256 cached tokens: rows see fewer than 1024 keys, so the request takes the
    # up-projected path (exact scores) and the absorbed part is empty
    sl2 = (ctypes.c_int32 * 1)(320)
    assert lib.mla_prefill_absorbed_workspace_size(1, sl2, cq, 8, None, 0, 128, 3) > _ws(lib, [320], [0, 64], 8, chunk=128)


def test_absorbed_plan_joins_chunk_pieces_and_spreads_single_rows(lib):
    """The absorbed planner's choices, seen through its workspace (one latent
    state slot per key split): a short extend over 32K cached tokens in 16K
    chunks plans one uncut key range (32 items of 256 rows fill the GPU's
    clusters in one wave, so no merge); one new token (a single item of 128
    rows) is cut into many key splits so that it spreads over the GPU."""
    blocks = (32768 + 64 + 63) // 64
    sl, cq = (ctypes.c_int32 * 1)(32768 + 64), (ctypes.c_int32 * 2)(0, 64)
    n = lib.mla_prefill_absorbed_workspace_size(1, sl, cq, 128, None, 0, 16384, 3)
    assert _abs_layout(blocks, 64 * 128, 1) < n < _abs_layout(blocks, 64 * 128, 2)
    sl1, cq1 = (ctypes.c_int32 * 1)(32768 + 1), (ctypes.c_int32 * 2)(0, 1)
    n1 = lib.mla_prefill_absorbed_workspace_size(1, sl1, cq1, 128, None, 0, 16384, 3)
    assert n1 > _abs_layout((32768 + 1 + 63) // 64, 128, 16)


def test_fp8_score_and_reuse_workspaces(lib):
    """Host-side sizing of the FP8-score absorbed path and of head-split reuse."""
    sl, cq = (ctypes.c_int32 * 1)(1100), (ctypes.c_int32 * 2)(0, 64)
    fp8 = lib.mla_prefill_absorbed_fp8_workspace_size(1, sl, cq, 8, None, 0, 128, 3)
    rows = 64 * 8
    extra = (rows * 512 + 255) // 256 * 256 + (rows * 4 + 255) // 256 * 256
    # E4M3 qlat and its row scales (the FP8 rows are read from the cache in place)
    assert any(fp8 == _abs_layout(18, rows, k) + extra for k in range(1, 5))

    sl, cq = (ctypes.c_int32 * 1)(320), (ctypes.c_int32 * 2)(0, 64)
    g = (ctypes.c_int32 * 2)(1, 5)
    none = lib.mla_prefill_reuse_workspace_size(1, sl, cq, 8, None, 0, 128, 3, g, 0, None)
    two = lib.mla_prefill_reuse_workspace_size(1, sl, cq, 8, None, 0, 128, 3, g, 2, None)
    prot = (ctypes.c_uint8 * 64)(*([1] * 8 + [0] * 56))
    both = lib.mla_prefill_reuse_workspace_size(1, sl, cq, 8, None, 0, 128, 3, g, 2, prot)
    assert 0 < none < two < both
    bad = (ctypes.c_int32 * 1)(8)       # head outside [0, 8)
    assert lib.mla_prefill_reuse_workspace_size(1, sl, cq, 8, None, 0, 128, 3, bad, 1, None) == 0


def test_fp8_score_entry_needs_fp8_cache(lib):
    d = ctypes.c_void_p(4096)
    sl, cq = (ctypes.c_int32 * 1)(320), (ctypes.c_int32 * 2)(0, 64)
    st = lib.mla_prefill_ctx_absorbed_fp8(d, d, d, 0, 1.0, 8, d, 8, sl, cq, 1, 8, None, 0, 128, d, 0.07, 10000.0, 3,
                                          d, 0, d, d, 1 << 30, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED
