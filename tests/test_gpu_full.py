"""Full-size parity on the four large workloads, in the launch configuration the
bench times: the GPU computes every (row, head); the CPU oracle recomputes a
sample of rows (first and last of every request, every query-tile boundary,
random rows) for 8 heads spread over the role queue, and properties that hold
at any size are checked on the whole output."""
import numpy as np
import pytest

from mla_prefix_cache_gb300 import workload as W
from oracle import mla_oracle as O

from test_gpu_parity import assert_close, visible_keys

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def sample_rows(wl, rng, n_random=24):
    """First and last row of every request, both rows at every 128-row query
    tile boundary (a consumer CTA's tile; pairs of tiles are a consumer
    pair's), and random rows."""
    cu = wl.cu_q
    rows = set()
    for r in range(wl.num_reqs):
        a, b = int(cu[r]), int(cu[r + 1])
        rows.update((a, a + 1, b - 1))
        for x in range(a + 128, b, 128):
            rows.update((x - 1, x))
    rows.update(rng.integers(0, wl.total_q, size=n_random).tolist())
    return np.array(sorted(x for x in rows if 0 <= x < wl.total_q))


# heads spread over the role queue: the first and last ones, the producers'
# lookahead boundary (heads 0-2), and the middle of the queue
SAMPLED_HEADS = [0, 1, 2, 63, 64, 125, 126, 127]


@pytest.mark.parametrize("name", ["v3_8k", "batched", "fp8_128k", "reloc_256k"])
def test_full_size_sampled(name):
    from mla_prefix_cache_gb300 import api
    wl = W.by_name(name)
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run()
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 0
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(100)
    rows = sample_rows(wl, rng)
    heads = SAMPLED_HEADS
    ref_out, ref_lse = O.mla_prefill(**O.workload_args(wl), rows=rows, heads=heads)
    got_out = out[torch.from_numpy(rows).cuda()][:, heads].cpu().numpy()
    got_lse = lse[torch.from_numpy(rows).cuda()][:, heads].cpu().numpy()
    assert_close(got_out, got_lse, ref_out, ref_lse, visible_keys(wl)[rows])
    # every row sees its whole context, so lse >= the log of a positive sum everywhere;
    # the mean output over all rows/heads stays near zero for zero-mean values
    assert float(out.abs().max()) < 1.0


def test_absorbed_short_extend_full_size():
    """The absorbed path on the short-extend workload the bench times (128
    heads, 32K cached + 64 new tokens), sampled rows against the oracle, every
    row against the up-projected path."""
    from mla_prefix_cache_gb300 import api
    wl = W.by_name("short_ext_32k")
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run(absorbed=True)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 0
    assert bool(torch.isfinite(out).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(101)
    rows = np.array([0, 1, 17, 40, 62, 63])
    heads = [0, int(rng.integers(1, wl.num_heads - 1)), wl.num_heads - 1]
    ref_out, ref_lse = O.mla_prefill(**O.workload_args(wl), rows=rows, heads=heads)
    got_out = out[torch.from_numpy(rows).cuda()][:, heads].cpu().numpy()
    got_lse = lse[torch.from_numpy(rows).cuda()][:, heads].cpu().numpy()
    assert_close(got_out, got_lse, ref_out, ref_lse, visible_keys(wl)[rows])
    o2, l2 = dw.run()
    torch.cuda.synchronize()
    assert float((out - o2).abs().max()) <= 2e-2
    assert float((lse - l2).abs().max()) <= 1e-3
