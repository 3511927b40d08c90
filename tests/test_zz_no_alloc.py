"""mla_prefill_ctx_noalloc: the prefill entry point for callers that cannot
allocate device memory (a framework that owns every device byte through its
own pool, or a caller in the middle of a graph capture).  It must give the
same result as mla_prefill_ctx with a caller-provided workspace, on two calls
in a row (its fixed scratch keeps the previous call's contents), and refuse a
problem that does not fit its fixed scratch before launching anything.

This file sorts last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest

from mla_prefix_cache_gb300 import workload as W

from test_gpu_parity import assert_close, visible_keys

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc(L, dw, wl, out, lse):
    from mla_prefix_cache_gb300 import _lib
    from mla_prefix_cache_gb300.api import _dev, _stream_ptr, kv_dtype_code
    sl, k1 = _lib.i32_host(wl.seq_lens)
    cq, k2 = _lib.i32_host(wl.cu_q)
    sp, ns, k3 = _lib.segments_host(wl.segments)
    return L.mla_prefill_ctx_noalloc(
        _dev(dw.q, "q"), _dev(dw.q_pos, "q_pos"), _dev(dw.kv_cache, "kv_cache"), kv_dtype_code(dw.kv_cache),
        float(wl.kv_scale), int(dw.kv_cache.shape[0]), _dev(dw.block_table, "block_table"),
        int(dw.block_table.shape[1]), sl, cq, wl.num_reqs, wl.num_heads, sp, ns, wl.chunk,
        _dev(dw.kv_b_proj, "kv_b_proj"), float(wl.softmax_scale), float(wl.rope_theta), 3,
        _dev(out, "out"), 0, _dev(lse, "lse"), _stream_ptr(None))


@pytest.mark.parametrize("wl", [
    W.tiny(),
    W.make_workload("docs", 8, [128], [70], chunk=64, seed=40, doc_len=64),   # partial states + merge
    W.make_workload("h128", 128, [300], [70], chunk=128, seed=42),            # DeepSeek head count
], ids=["tiny", "segments", "h128"])
def test_noalloc_matches_workspace_entry_point(wl):
    from mla_prefix_cache_gb300 import _lib, api
    L = _lib.load()
    dw = api.DeviceWorkload(wl)
    ref_out, ref_lse = dw.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = ref_out.cpu().numpy(), ref_lse.cpu().numpy()
    nvis = visible_keys(wl)
    for _ in range(2):                      # the second call finds the first call's scratch contents
        out = torch.full((wl.total_q, wl.num_heads, 128), float("nan"), device="cuda")
        lse = torch.full((wl.total_q, wl.num_heads), float("nan"), device="cuda")
        assert _noalloc(L, dw, wl, out, lse) == _lib.MLA_OK
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, nvis)


def test_noalloc_rejects_problems_beyond_its_scratch():
    from mla_prefix_cache_gb300 import _lib, api
    L = _lib.load()
    wl = W.make_workload("big", 2, [40000], [1], seed=41)   # 46 MB of gathered rows alone
    assert api.prefill_min_workspace_size(wl.seq_lens, wl.cu_q, 2, None, wl.chunk) > _lib.NOALLOC_SCRATCH_BYTES
    dw = api.DeviceWorkload(wl)
    out = torch.zeros((1, 2, 128), device="cuda")
    lse = torch.zeros((1, 2), device="cuda")
    n0 = api.launch_count()
    assert _noalloc(L, dw, wl, out, lse) == _lib.MLA_ERR_TOO_LARGE
    assert api.launch_count() == n0


def test_noalloc_without_queries_launches_nothing():
    """A call with no query rows is valid and does nothing, as for mla_prefill_ctx."""
    from mla_prefix_cache_gb300 import _lib, api
    L = _lib.load()
    wl = W.make_workload("none", 2, [128], [0], seed=43)
    dw = api.DeviceWorkload(wl)
    out = torch.zeros((1, 2, 128), device="cuda")
    lse = torch.zeros((1, 2), device="cuda")
    n0 = api.launch_count()
    assert _noalloc(L, dw, wl, out, lse) == _lib.MLA_OK
    assert api.launch_count() == n0
