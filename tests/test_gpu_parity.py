"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Tolerances (bf16 inputs, fp32 accumulation), on every row: out max abs
<= 2e-2 and mean abs <= 2e-3, lse within 1e-3, plus a stricter internal gate
of relative RMS error <= 1e-2 on out.  Gather and block-table indexing are
bit-exact.

lse and key count: the tensor cores take bf16 operands, so a score built
from the up-projected K_nope rounded to bf16 carries about 1.4e-3 (one sigma,
unit-variance scores) of rounding; lse averages that over the visible keys.
Rows that see fewer than 1024 keys in all (the small edge cases, down to a
single key) therefore take exact scores in the kernel (K_nope as bf16 plus
its bf16 residual) and are held to the same 1e-3 as every other row.
"""
import math

import numpy as np
import pytest

from mla_prefix_cache_gb300 import workload as W
from oracle import mla_oracle as O

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OUT_MAX, OUT_MEAN, LSE_MAX, REL_RMS = 2e-2, 2e-3, 1e-3, 1e-2


@pytest.fixture(scope="module")
def api():
    from mla_prefix_cache_gb300 import api as A
    from mla_prefix_cache_gb300 import _lib
    _lib.load()
    return A


def visible_keys(wl, parts=3):
    """Number of keys each query row attends to."""
    n = np.zeros(wl.total_q, dtype=np.int64)
    cu = wl.cu_q
    for r in range(wl.num_reqs):
        E, C = int(wl.ext_lens[r]), int(wl.ctx_lens[r])
        ctx = C if wl.segments is None else int(sum(s[2] for s in wl.segments if s[0] == r))
        n[cu[r]:cu[r + 1]] = (ctx if parts & 1 else 0) + (np.arange(1, E + 1) if parts & 2 else 0)
    return n


def assert_close(out, lse, ref_out, ref_lse, nvis=None):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    ref_out = np.asarray(ref_out, dtype=np.float64)
    ref_lse = np.asarray(ref_lse, dtype=np.float64)
    assert np.isfinite(out).all(), "non-finite output"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), "empty rows differ"
    err = np.abs(out - ref_out)
    assert err.max() <= OUT_MAX, f"max abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN, f"mean abs {err.mean():.3e}"
    if fin.any():
        le = np.abs(lse - ref_lse)
        bad = fin & (le > LSE_MAX)
        where = np.argwhere(bad)[:3].tolist()
        seen = [int(np.asarray(nvis)[w[0]]) for w in where] if nvis is not None else None
        assert not bad.any(), f"lse err {le[fin].max():.3e} (tol {LSE_MAX:.0e} at {where}, visible keys {seen})"
    den = math.sqrt(float((ref_out ** 2).mean())) or 1.0
    rel = math.sqrt(float((err ** 2).mean())) / den
    assert rel <= REL_RMS, f"rel rms {rel:.3e}"


def run_and_compare(api, wl, parts=3, out_dtype=None, rows=None, heads=None, **kw):
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run(parts=parts, out_dtype=out_dtype or torch.float32, **kw)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 0
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    ref_out, ref_lse = O.mla_prefill(**O.workload_args(wl), parts=parts, rows=rows, heads=heads)
    nvis = visible_keys(wl, parts)
    if rows is not None:
        out, lse, nvis = out[rows], lse[rows], nvis[rows]
    if heads is not None:
        out, lse = out[:, heads], lse[:, heads]
    assert_close(out, lse, ref_out, ref_lse, nvis)
    return out, lse


# ---------------------------------------------------------------- gather

def test_gather_bf16_bit_exact(api):
    wl = W.make_workload("g", 1, [200, 300], [5, 37], seed=21)
    dw = api.DeviceWorkload(wl)
    r = 1
    got = api.gather_latent(dw.kv_cache, dw.block_table[r], 3, 330).cpu().view(torch.int16).numpy().view(np.uint16)
    t = np.arange(3, 333)
    exp = wl.kv_cache[wl.block_table[r][t // 64], t % 64]
    assert np.array_equal(got, exp)


def test_gather_many_tiles_bit_exact(api):
    # 20000 rows from an unaligned start: 313 tiles of 64 rows, more than the
    # two resident CTAs per SM take in one round, and a ragged last tile
    wl = W.make_workload("gm", 1, [20100], [1], seed=26)
    dw = api.DeviceWorkload(wl)
    got = api.gather_latent(dw.kv_cache, dw.block_table[0], 37, 20000).cpu().view(torch.int16).numpy().view(np.uint16)
    t = np.arange(37, 20037)
    assert np.array_equal(got, wl.kv_cache[wl.block_table[0][t // 64], t % 64])


def test_gather_fp8_dequant_bit_exact(api):
    wl = W.make_workload("g8", 1, [130], [70], kv_dtype="fp8_e4m3", seed=22)
    dw = api.DeviceWorkload(wl)
    got = api.gather_latent(dw.kv_cache, dw.block_table[0], 0, 200, kv_scale=wl.kv_scale)
    got = got.cpu().view(torch.int16).numpy().view(np.uint16)
    t = np.arange(200)
    raw = wl.kv_cache[wl.block_table[0][t // 64], t % 64]
    lat = O.e4m3_to_float(raw[:, :512]).astype(np.float32) * np.float32(wl.kv_scale)
    assert np.array_equal(got[:, :512], W.f32_to_bf16_bits(lat))
    assert np.array_equal(got[:, 512:], np.ascontiguousarray(raw[:, 512:]).view(np.uint16))


def test_gather_bad_block_reports_error(api):
    wl = W.make_workload("gb", 1, [128], [1], seed=23)
    dw = api.DeviceWorkload(wl)
    table = dw.block_table[0].clone()
    table[1] = 10_000                     # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.gather_latent(dw.kv_cache, table, 0, 129, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    g = got.cpu().float().numpy()
    assert (g[64:128] == 0).all() and np.isfinite(g[:64]).all()


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("rows,d_v", [(1000, 128), (1001, 128), (3, 128), (333, 64)])
def test_merge_states_matches_oracle(api, rows, d_v):
    rng = np.random.default_rng(24)
    oa, ob = rng.standard_normal((rows, d_v)).astype(np.float32), rng.standard_normal((rows, d_v)).astype(np.float32)
    la, lb = (rng.standard_normal(rows) * 20).astype(np.float32), (rng.standard_normal(rows) * 20).astype(np.float32)
    la[::7] = -np.inf
    lb[::11] = -np.inf
    ref_o, ref_l = O.merge_attn_states(oa.astype(np.float64), la.astype(np.float64),
                                       ob.astype(np.float64), lb.astype(np.float64))
    t = [torch.from_numpy(x).cuda() for x in (oa, la, ob, lb)]
    o, l = api.merge_states(*t)
    np.testing.assert_allclose(o.cpu().numpy(), ref_o, atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(l.cpu().numpy(), ref_l, atol=1e-5, rtol=1e-6)
    # in place into the first state
    api.merge_states(t[0], t[1], t[2], t[3], out=t[0], lse=t[1])
    np.testing.assert_allclose(t[0].cpu().numpy(), ref_o, atol=1e-5, rtol=1e-5)
    np.testing.assert_allclose(t[1].cpu().numpy(), ref_l, atol=1e-5, rtol=1e-6)


# ---------------------------------------------------------------- rope

@pytest.mark.parametrize("T,H,inplace", [(300, 3, False), (77, 5, True), (64, 128, True)])
def test_rope_relocate_matches_oracle(api, T, H, inplace):
    rng = np.random.default_rng(25)
    x = W.f32_to_bf16_bits(rng.standard_normal((T, H, 192), dtype=np.float32))
    pos = (rng.integers(0, 300000, size=T)).astype(np.int32)
    off = 16384 * 7
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = api.rope_relocate(xt, torch.from_numpy(pos).cuda(), off, 10000.0, y=xt if inplace else None)
    y = y.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y[..., :128], x[..., :128])
    ref = O.rope_rotate(O.bf16_to_float(x[..., 128:], np.float64), (pos.astype(np.int64) - off)[:, None], 1e4,
                        np.float64)
    got = O.bf16_to_float(y[..., 128:], np.float64)
    assert np.abs(got - ref).max() <= 2.0 ** -7 * np.abs(ref).max()
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6).mean() > 0.999


# ---------------------------------------------------------------- prefill

def test_prefill_tiny(api):
    run_and_compare(api, W.tiny())


@pytest.mark.parametrize("case", [
    dict(H=4, ctx=[300], ext=[200], chunk=128),                       # ragged kv and q tails
    dict(H=2, ctx=[0], ext=[130], chunk=64),                          # no context
    dict(H=3, ctx=[64, 0, 777], ext=[1, 64, 129], chunk=256),         # ragged batch
    dict(H=2, ctx=[513], ext=[77], chunk=192, kv="fp8_e4m3"),         # FP8 cache
    dict(H=2, ctx=[256], ext=[40], chunk=64, doc=64),                 # relocated documents
    dict(H=2, ctx=[256], ext=[160], chunk=64, doc=64),                # documents, a whole tile of partial states
    dict(H=128, ctx=[200], ext=[130], chunk=128),                     # full head count
])
def test_prefill_small(api, case):
    wl = W.make_workload("s", case["H"], case["ctx"], case["ext"], chunk=case["chunk"],
                         kv_dtype=case.get("kv", "bf16"), doc_len=case.get("doc"), seed=30)
    run_and_compare(api, wl)


@pytest.mark.parametrize("parts", [1, 2])
def test_prefill_parts(api, parts):
    wl = W.make_workload("p", 2, [260], [150], chunk=128, seed=31)
    run_and_compare(api, wl, parts=parts)


@pytest.mark.parametrize("ext", [70, 200], ids=["partial_tile", "whole_and_partial_tiles"])
def test_prefill_bf16_out(api, ext):
    """bf16 output: whole 128-row tiles go out by TMA, partial ones by thread stores."""
    wl = W.make_workload("b", 2, [190], [ext], chunk=128, seed=32)
    run_and_compare(api, wl, out_dtype=torch.bfloat16)


def test_prefill_bad_block_reports_error(api):
    wl = W.make_workload("e", 2, [256], [16], chunk=128, seed=33)
    dw = api.DeviceWorkload(wl)
    dw.block_table[0, 1] = -5
    out, lse = dw.run()
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 3    # MLA_ERR_BAD_BLOCK_ID
    assert torch.isfinite(out).all()
    assert api.device_error(api.prefill.last_workspace) == 0    # cleared by the read


def test_prefill_empty_context_segments(api):
    # segments given but none for the request -> empty context; extend only
    wl = W.make_workload("z", 1, [128], [20], chunk=64, seed=34)
    dw = api.DeviceWorkload(wl)
    out, lse = api.prefill(dw.q, dw.q_pos, dw.kv_cache, dw.block_table, wl.seq_lens, wl.cu_q, dw.kv_b_proj,
                           chunk=64, softmax_scale=wl.softmax_scale, segments=np.zeros((0, 4), np.int64))
    ref = O.mla_prefill(**O.workload_args(wl), parts=2)
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), *ref, visible_keys(wl, 2))


def test_prefill_small_workspace_runs_in_several_launches(api):
    """The smallest workspace the call accepts: two ring lanes of 4 tiles and
    the ring flags of one piece (of two here, where both round up to the same
    256 bytes).  The call splits its pieces over several launches and must
    give the same result; a smaller one is refused."""
    from mla_prefix_cache_gb300 import _lib
    wl = W.make_workload("sw", 4, [192], [70], chunk=64, seed=35, doc_len=64)   # 3 documents + extend = 4 pieces
    dw = api.DeviceWorkload(wl)
    n_min = api.prefill_min_workspace_size(wl.seq_lens, wl.cu_q, 4, wl.segments, wl.chunk)
    assert n_min < api.prefill_workspace_size(wl.seq_lens, wl.cu_q, 4, wl.segments, wl.chunk)
    small = torch.empty(n_min, dtype=torch.uint8, device="cuda")
    n0 = api.launch_count()
    out, lse = dw.run(workspace=small)
    torch.cuda.synchronize()
    assert api.launch_count() - n0 >= 4          # the gather, two fused launches or more, the merge
    ref = O.mla_prefill(**O.workload_args(wl))
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), *ref, visible_keys(wl))
    with pytest.raises(_lib.MLAError):
        dw.run(workspace=torch.empty(n_min - 256, dtype=torch.uint8, device="cuda"))


@pytest.mark.parametrize("depth", [4, 8])
def test_prefill_shallow_ring_wraps(api, depth, monkeypatch):
    """K/V rings shallower than a piece: producers reuse ring slots once every
    consumer has released them (single releases at depth 4, batched at 8)."""
    monkeypatch.setenv("MLA_RING_DEPTH", str(depth))
    wl = W.make_workload("ring", 2, [1500, 600], [300, 200], chunk=2048, seed=36)   # 15 and 7 tiles
    run_and_compare(api, wl)


@pytest.mark.parametrize("knobs", [
    {"MLA_PRODUCER_LOOKAHEAD": "1"},
    {"MLA_PRODUCER_LOOKAHEAD": "5", "MLA_PRODUCERS": "2"},
    {"MLA_PRODUCERS": "8", "MLA_RING_DEPTH": "8"},
    {"MLA_RING_LANES": "3"},                                  # every job waits for the lane's job 3 before it
    {"MLA_RING_LANES": "2", "MLA_PRODUCER_LOOKAHEAD": "1", "MLA_RING_DEPTH": "4"},   # the fewest lanes
], ids=["lookahead1", "lookahead5_one_producer", "four_producers_shallow", "three_lanes", "two_shallow_lanes"])
def test_prefill_queue_knobs(api, knobs, monkeypatch):
    """The role queue's tuning knobs (producer count, lookahead, ring depth, ring lanes)
    change the schedule, never the result."""
    for k, v in knobs.items():
        monkeypatch.setenv(k, v)
    wl = W.make_workload("q", 6, [700, 300], [260, 130], chunk=256, seed=37)
    run_and_compare(api, wl)


def test_prefill_wait_runs_out_and_reports_timeout(api, monkeypatch):
    """Failure detection without a fault: the one job's producers are withheld
    (a test hook of the library), so its consumers' bounded waits for ready
    tiles run out after the shortened limit; the kernel records
    MLA_ERR_TIMEOUT, frees its tensor memory and returns, and the next call on
    the same device and workspace is correct.  One head, one piece: no K/V
    load or MMA is ever issued, only the Q loads, which complete."""
    wl = W.make_workload("to", 1, [300], [200], chunk=128, seed=38)
    dw = api.DeviceWorkload(wl)
    ws = torch.empty(api.prefill_workspace_size(wl.seq_lens, wl.cu_q, 1, None, wl.chunk), dtype=torch.uint8,
                     device="cuda")
    monkeypatch.setenv("MLA_WAIT_LIMIT_US", "2000")
    monkeypatch.setenv("MLA_TEST_WITHHOLD_JOB", "0")
    dw.run(workspace=ws)
    torch.cuda.synchronize()
    assert api.device_error(ws) == 6                 # MLA_ERR_TIMEOUT
    assert api.device_error(ws) == 0                 # cleared by the read
    monkeypatch.delenv("MLA_TEST_WITHHOLD_JOB")
    monkeypatch.delenv("MLA_WAIT_LIMIT_US")
    out, lse = dw.run(workspace=ws)
    torch.cuda.synchronize()
    assert api.device_error(ws) == 0
    ref = O.mla_prefill(**O.workload_args(wl))
    assert_close(out.cpu().numpy(), lse.cpu().numpy(), *ref, visible_keys(wl))


@pytest.mark.parametrize("case", [
    dict(H=4, ctx=[700], ext=[300], chunk=256, doc=None),     # 3 query tiles: one full pair, one half pair
    dict(H=2, ctx=[256], ext=[200], chunk=64, doc=64),        # relocated documents, partial states + merge
], ids=["ragged", "docs"])
def test_prefill_small_grid(api, case, monkeypatch):
    """Four CTA pairs take every role of the queue in turn: a role only ever
    waits on roles dequeued before it, so any grid finishes."""
    monkeypatch.setenv("MLA_FUSED_GRID", "8")
    wl = W.make_workload("grid", case["H"], case["ctx"], case["ext"], chunk=case["chunk"], seed=31,
                         doc_len=case["doc"])
    run_and_compare(api, wl)


# ---------------------------------------------------------------- absorbed (latent-space) path

# The absorbed path takes the requests whose rows all see >= 1024 keys; the
# others (few keys: exact scores) go through the up-projected kernel in the
# same call.  Contexts of >= 1023 tokens keep these cases on the latent kernel.
ABSORBED_CASES = [
    dict(H=4, ctx=[1100], ext=[20], chunk=128),                       # ragged kv tail, one row tile
    dict(H=2, ctx=[0], ext=[130], chunk=64),                          # no context, causal only (up-projected)
    dict(H=3, ctx=[1088, 0, 1777], ext=[1, 64, 29], chunk=256),       # ragged batch, one request up-projected
    dict(H=2, ctx=[1537], ext=[77], chunk=192, kv="fp8_e4m3"),        # FP8 cache
    dict(H=2, ctx=[1280], ext=[40], chunk=64, doc=64),                # 20 relocated documents
    dict(H=128, ctx=[1200], ext=[3], chunk=128),                      # full head count, 3 row tiles
]


def test_absorbed_tiny(api):
    """The tiny workload's rows see 257-320 keys: the absorbed entry point
    takes them through the up-projected kernel (exact scores)."""
    run_and_compare(api, W.tiny(), absorbed=True)


@pytest.mark.parametrize("split", [None, "64", "192"], ids=["auto", "split64", "split192"])
@pytest.mark.parametrize("case", ABSORBED_CASES, ids=["ragged", "noctx", "batch", "fp8", "docs", "h128"])
def test_absorbed_small(api, case, split, monkeypatch):
    """Same workloads as the up-projected path; MLA_ABS_SPLIT_KEYS forces key
    splits (several partial states per row, projected then merged)."""
    if split is not None:
        monkeypatch.setenv("MLA_ABS_SPLIT_KEYS", split)
    wl = W.make_workload("a", case["H"], case["ctx"], case["ext"], chunk=case["chunk"],
                         kv_dtype=case.get("kv", "bf16"), doc_len=case.get("doc"), seed=40)
    run_and_compare(api, wl, absorbed=True)


@pytest.mark.parametrize("parts", [1, 2])
def test_absorbed_parts(api, parts):
    wl = W.make_workload("ap", 2, [1060], [50], chunk=128, seed=41)
    run_and_compare(api, wl, parts=parts, absorbed=True)


def test_absorbed_bf16_out(api):
    wl = W.make_workload("ab", 2, [1090], [70], chunk=128, seed=42)
    run_and_compare(api, wl, out_dtype=torch.bfloat16, absorbed=True)


def test_absorbed_matches_fused_path(api):
    """Both entry points compute the same function: their outputs agree to the
    rounding of their different bf16 operands."""
    wl = W.make_workload("am", 8, [1500], [33], chunk=256, seed=43)
    dw = api.DeviceWorkload(wl)
    o1, l1 = dw.run()
    o2, l2 = dw.run(absorbed=True)
    torch.cuda.synchronize()
    assert (o1 - o2).abs().max().item() <= OUT_MAX
    assert (l1 - l2).abs().max().item() <= LSE_MAX


def test_absorbed_long_context_sampled(api):
    """128 heads, 16K cached tokens (FP8) and 64 new ones: the bench's
    short-extend shape at a quarter of its context, checked on sampled rows."""
    wl = W.make_workload("al", 128, [16384], [64], chunk=8192, kv_dtype="fp8_e4m3", seed=44)
    rows = np.array([0, 1, 31, 62, 63])
    run_and_compare(api, wl, rows=rows, heads=np.arange(0, 128, 9), absorbed=True)


@pytest.mark.parametrize("kv,mode,block", [("bf16", True, 1), ("bf16", True, 17), ("fp8_e4m3", "fp8", 1),
                                           ("fp8_e4m3", "fp8", 17)],
                         ids=["middle", "last", "fp8_scores_middle", "fp8_scores_last"])
def test_absorbed_bad_block_and_workspace(api, kv, mode, block):
    """A bad block id in the middle of a request or in its last block (read in
    place by the score side, from a copy by the P c side of a BF16 cache)
    reaches the error word, and the rows it stands for read as zeros, so the
    output stays finite."""
    from mla_prefix_cache_gb300 import _lib
    wl = W.make_workload("ae", 2, [1100], [16], chunk=128, kv_dtype=kv, seed=45)   # 1116 tokens: blocks 0-17
    dw = api.DeviceWorkload(wl)
    dw.block_table[0, block] = -5
    out, lse = dw.run(absorbed=mode)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 3    # MLA_ERR_BAD_BLOCK_ID
    assert torch.isfinite(out).all()
    with pytest.raises(_lib.MLAError):
        dw.run(absorbed=mode, workspace=torch.empty(4096, dtype=torch.uint8, device="cuda"))


# ---------------------------------------------------------------- content-addressed block store

def _pool(kv):
    return W.make_workload("bs", 2, [900, 333], [40, 7], chunk=128, kv_dtype=kv, seed=50)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_block_hash_bit_exact(api, kv):
    from oracle import block_store as BS
    wl = _pool(kv)
    dw = api.DeviceWorkload(wl)
    nb = wl.kv_cache.shape[0]
    ids = np.concatenate([np.arange(nb), np.random.default_rng(51).integers(0, nb, size=37)]).astype(np.int32)
    got = api.block_hash(dw.kv_cache, torch.from_numpy(ids).cuda()).cpu().numpy().view(np.uint64)
    want = np.array([BS.block_hash(wl.kv_cache, int(b)) for b in ids], dtype=np.uint64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_block_compare_and_bad_ids(api, kv):
    wl = _pool(kv)
    dw = api.DeviceWorkload(wl)
    nb = wl.kv_cache.shape[0]
    dw.kv_cache[5] = dw.kv_cache[2]          # planted equal content
    dw.kv_cache[9] = dw.kv_cache[2]
    dw.kv_cache[9].view(torch.uint8).view(-1)[-1] ^= 1   # same but the very last byte
    a = torch.tensor([2, 5, 2, 0, 3, 2, -1, 1], dtype=torch.int32, device="cuda")
    b = torch.tensor([5, 2, 9, 0, 4, 2, 1, nb], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    eq = api.block_compare(dw.kv_cache, a, b, dev_error=err).cpu().tolist()
    assert eq == [1, 1, 0, 1, 0, 1, -1, -1]
    assert int(err.item()) & 1
    err.zero_()
    h = api.block_hash(dw.kv_cache, torch.tensor([2, 5, 9, nb + 3], dtype=torch.int32, device="cuda"), dev_error=err)
    h = h.cpu().tolist()
    assert h[0] == h[1] != h[2] and h[3] == 0 and int(err.item()) & 1


def test_seal_protocol_on_gpu_matches_oracle(api):
    """The page's seal protocol driven by the two GPU calls (hash, then byte
    comparison on a hash match) gives the oracle's holders and collision
    count; 3-bit hashes make distinct blocks collide."""
    from oracle import block_store as BS
    wl = _pool("bf16")
    dw = api.DeviceWorkload(wl)
    for dst, src in ((7, 1), (12, 1), (20, 4)):
        dw.kv_cache[dst] = dw.kv_cache[src]
    cache_np = dw.kv_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    nb = cache_np.shape[0]
    ids = torch.arange(nb, dtype=torch.int32, device="cuda")
    keys = (api.block_hash(dw.kv_cache, ids).cpu().numpy().view(np.uint64) & np.uint64(7)).tolist()
    table, holders, coll = {}, [], 0
    for c in range(nb):
        same = table.get(keys[c], [])
        if same:
            eq = api.block_compare(dw.kv_cache, torch.tensor(same, dtype=torch.int32, device="cuda"),
                                   torch.full((len(same),), c, dtype=torch.int32, device="cuda")).cpu().tolist()
            hit = [b for b, e in zip(same, eq) if e == 1]
            if hit:
                holders.append(hit[0])
                continue
            coll += 1
        table.setdefault(keys[c], []).append(c)
        holders.append(c)
    want_holders, want_coll = BS.seal_all(cache_np, range(nb), hash_bits=3)
    assert holders == want_holders and coll == want_coll and coll > 0
    assert holders[7] == 1 and holders[12] == 1 and holders[20] == 4


# ---------------------------------------------------------------- head-split reuse (Global heads, protected rows)

REUSE_CASES = [
    dict(H=6, ctx=[300, 77], ext=[140, 9], chunk=128, glob=[1, 4], prot=[0, 5, 77, 139, 140, 148]),
    dict(H=4, ctx=[256], ext=[200], chunk=64, doc=64, glob=[3], prot=list(range(0, 200, 7))),
    dict(H=3, ctx=[513], ext=[77], chunk=192, kv="fp8_e4m3", glob=[], prot=[1, 2, 76]),
    dict(H=128, ctx=[300], ext=[130], chunk=128, glob=list(range(0, 128, 8)), prot=[0, 64, 127, 128, 129]),
    dict(H=5, ctx=[200], ext=[50], chunk=128, glob=[0, 1, 2, 3, 4], prot=[]),          # every head Global
    dict(H=5, ctx=[200], ext=[50], chunk=128, glob=[], prot=[]),                       # all from the artifact
    # protected rows that take the absorbed path (at most 208 a request, each seeing 1024 keys or more)
    dict(H=8, ctx=[1100, 2048], ext=[90, 40], chunk=512, glob=[2, 5], prot=[0, 7, 50, 89, 90, 95, 129]),
    dict(H=6, ctx=[1536], ext=[64], chunk=256, doc=512, glob=[0], prot=[1, 2, 30, 63]),
    dict(H=4, ctx=[1200], ext=[33], chunk=256, kv="fp8_e4m3", glob=[3], prot=list(range(0, 33, 4))),
]


@pytest.mark.parametrize("case", REUSE_CASES, ids=["batch", "docs", "fp8", "h128", "all_global", "all_artifact",
                                                   "absorbed_batch", "absorbed_docs", "absorbed_fp8"])
def test_prefill_reuse_matches_oracle(api, case, monkeypatch):
    """Each case through the call's own choice for its protected rows, and,
    where that is the absorbed path (at most 208 protected rows a request,
    each seeing 1024 keys or more), again with the up-projected path forced
    (MLA_REUSE_ABSORBED=0): both meet the oracle, and the two routes launch
    different kernels."""
    from oracle import head_reuse as R
    wl = W.make_workload("ru", case["H"], case["ctx"], case["ext"], chunk=case["chunk"],
                         kv_dtype=case.get("kv", "bf16"), doc_len=case.get("doc"), seed=70)
    dw = api.DeviceWorkload(wl)
    rng = np.random.default_rng(71)
    art_out = rng.standard_normal((wl.total_q, wl.num_heads, 128)).astype(np.float32)
    art_lse = rng.standard_normal((wl.total_q, wl.num_heads)).astype(np.float32)
    ref_out, ref_lse = R.prefill_reuse(O.workload_args(wl), case["glob"], case["prot"], art_out, art_lse)
    m = R.reuse_mask(wl.total_q, wl.num_heads, case["glob"], case["prot"])
    nvis = np.broadcast_to(visible_keys(wl)[:, None], m.shape)[m]
    protected_absorbed = min(case["ctx"]) + 1 >= 1024 and bool(case["prot"]) and len(case["glob"]) < case["H"]
    launches = []
    for forced_fused in ([False, True] if protected_absorbed else [False]):
        if forced_fused:
            monkeypatch.setenv("MLA_REUSE_ABSORBED", "0")
        n0 = api.launch_count()
        out, lse = api.prefill_reuse(dw.q, dw.q_pos, dw.kv_cache, dw.block_table, wl.seq_lens, wl.cu_q,
                                     dw.kv_b_proj, torch.from_numpy(art_out).cuda(), torch.from_numpy(art_lse).cuda(),
                                     global_heads=case["glob"], protected_rows=case["prot"], chunk=wl.chunk,
                                     softmax_scale=wl.softmax_scale, kv_scale=wl.kv_scale, segments=wl.segments)
        torch.cuda.synchronize()
        launches.append(api.launch_count() - n0)
        assert api.device_error(api.prefill_reuse.last_workspace) == 0
        out, lse = out.cpu().numpy(), lse.cpu().numpy()
        # reused entries are copied bit for bit; recomputed ones meet the attention tolerances
        assert np.array_equal(out[~m], art_out[~m]) and np.array_equal(lse[~m], art_lse[~m])
        if m.any():
            assert_close(out[m][:, None], lse[m][:, None], ref_out[m][:, None], ref_lse[m][:, None], nvis)
    if protected_absorbed:
        assert launches[0] != launches[1]


def test_prefill_reuse_reports_bad_blocks(api):
    wl = W.make_workload("rb", 2, [256], [16], chunk=128, seed=72)
    dw = api.DeviceWorkload(wl)
    dw.block_table[0, 1] = -5
    z = torch.zeros((wl.total_q, 2, 128), dtype=torch.float32, device="cuda")
    zl = torch.zeros((wl.total_q, 2), dtype=torch.float32, device="cuda")
    api.prefill_reuse(dw.q, dw.q_pos, dw.kv_cache, dw.block_table, wl.seq_lens, wl.cu_q, dw.kv_b_proj, z, zl,
                      global_heads=[1], protected_rows=[3], chunk=128, softmax_scale=wl.softmax_scale)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill_reuse.last_workspace) == 3


# ---------------------------------------------------------------- edge cases of the extra entry points

@pytest.mark.parametrize("case", [
    dict(H=1, ctx=[1100], ext=[45], chunk=128),                # one head
    dict(H=4, ctx=[0], ext=[1], chunk=64),                     # a single query with no context: itself only
    dict(H=3, ctx=[100, 1088, 0], ext=[0, 5, 0], chunk=64),    # requests without queries in the batch
])
@pytest.mark.parametrize("absorbed", [False, True], ids=["fused", "absorbed"])
def test_prefill_degenerate_shapes(api, case, absorbed):
    wl = W.make_workload("dg", case["H"], case["ctx"], case["ext"], chunk=case["chunk"], seed=80)
    run_and_compare(api, wl, absorbed=absorbed)


def test_absorbed_many_splits(api, monkeypatch):
    """64-key splits of a 2K context: 33 partial states per row, merged in latent space."""
    monkeypatch.setenv("MLA_ABS_SPLIT_KEYS", "64")
    wl = W.make_workload("as", 4, [2048], [6], chunk=512, seed=81)
    run_and_compare(api, wl, absorbed=True)


@pytest.mark.parametrize("mode", ["all_protected", "one_head", "bf16_out"])
def test_prefill_reuse_edges(api, mode):
    from oracle import head_reuse as R
    H = 1 if mode == "one_head" else 3
    wl = W.make_workload("re", H, [190, 64], [30, 0], chunk=64, seed=82)
    dw = api.DeviceWorkload(wl)
    rng = np.random.default_rng(83)
    art_out = rng.standard_normal((wl.total_q, H, 128)).astype(np.float32)
    art_lse = rng.standard_normal((wl.total_q, H)).astype(np.float32)
    glob = [] if mode != "bf16_out" else [2]
    prot = list(range(wl.total_q)) if mode == "all_protected" else [0, 29]
    out, lse = api.prefill_reuse(dw.q, dw.q_pos, dw.kv_cache, dw.block_table, wl.seq_lens, wl.cu_q, dw.kv_b_proj,
                                 torch.from_numpy(art_out).cuda(), torch.from_numpy(art_lse).cuda(),
                                 global_heads=glob, protected_rows=prot, chunk=wl.chunk,
                                 softmax_scale=wl.softmax_scale,
                                 out_dtype=torch.bfloat16 if mode == "bf16_out" else torch.float32)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    ref_out, ref_lse = R.prefill_reuse(O.workload_args(wl), glob, prot, art_out, art_lse)
    m = R.reuse_mask(wl.total_q, H, glob, prot)
    if mode == "bf16_out":
        bf = torch.from_numpy(art_out[~m]).bfloat16().float().numpy()
        assert np.array_equal(out[~m], bf) and np.array_equal(lse[~m], art_lse[~m])
    else:
        assert np.array_equal(out[~m], art_out[~m]) and np.array_equal(lse[~m], art_lse[~m])
    nvis = np.broadcast_to(visible_keys(wl)[:, None], m.shape)[m]
    assert_close(out[m][:, None], lse[m][:, None], ref_out[m][:, None], ref_lse[m][:, None], nvis)
    if mode == "all_protected":   # every row recomputed: plain attention
        po, pl = O.mla_prefill(**O.workload_args(wl))
        assert_close(out, lse, po, pl, visible_keys(wl))


def test_block_store_empty_calls(api):
    wl = _pool("fp8_e4m3")
    dw = api.DeviceWorkload(wl)
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    n0 = api.launch_count()
    assert api.block_hash(dw.kv_cache, e).numel() == 0
    assert api.block_compare(dw.kv_cache, e, e).numel() == 0
    assert api.launch_count() == n0


# ---------------------------------------------------------------- absorbed path with E4M3 scores (FP8 caches)

def assert_close_fp8_scores(out, lse, ref_out, ref_lse, nvis):
    """Tolerances of mla_prefill_ctx_absorbed_fp8, derived from its one extra
    rounding: qlat to E4M3, a relative error up to 2^-4 (RMS ~0.024) on each
    of its 512 components.  With unit-variance inputs a scaled logit's latent
    part has std ~ sqrt(512 * 0.25) / sqrt(192) ~ 0.8, so each logit carries
    ~0.02 of noise.  That noise is shared by every key of a row, because the
    rounded qlat is, and the softmax-weighted mean of the keys leans towards
    qlat (by scale * qlat for unit-variance keys).  So lse moves by
    ~scale^2 * sum_c dqlat_c qlat_c, RMS ~1e-3 whatever the key count (held
    to 5e-3), plus the per-key part ~0.02 / sqrt(n) (held to 0.1 / sqrt(n)).
    A row seeing few keys takes single-logit noise on its output, RMS
    ~0.02 * |v - out| / sqrt(n) ~ 0.03 / sqrt(n): held per row to 2e-2 +
    0.2 / sqrt(n) (max) and, averaged over the rows, to 2e-3 + 0.05 / sqrt(n)
    (mean).  Relative RMS 5e-2 over all.  A CPU emulation of the E4M3
    rounding reproduces the measured errors."""
    out, lse = np.asarray(out, np.float64), np.asarray(lse, np.float64)
    ref_out, ref_lse = np.asarray(ref_out, np.float64), np.asarray(ref_lse, np.float64)
    assert np.isfinite(out).all()
    nv = np.broadcast_to(np.asarray(nvis, np.float64).reshape(-1, 1), ref_lse.shape)
    err = np.abs(out - ref_out)
    row_max = err.max(axis=-1)
    assert (row_max <= 2e-2 + 0.2 / np.sqrt(nv)).all(), f"max abs {row_max.max():.3e}"
    mean_tol = float((OUT_MEAN + 0.05 / np.sqrt(nv)).mean())
    assert err.mean() <= mean_tol, f"mean abs {err.mean():.3e} (tol {mean_tol:.2e})"
    le = np.abs(lse - ref_lse)
    assert (le <= 5e-3 + 0.1 / np.sqrt(nv)).all(), f"lse err {le.max():.3e}"
    rel = math.sqrt(float((err ** 2).mean())) / (math.sqrt(float((ref_out ** 2).mean())) or 1.0)
    assert rel <= 5e-2, f"rel rms {rel:.3e}"


@pytest.mark.parametrize("case", [
    dict(H=4, ctx=[513], ext=[20], chunk=192),
    dict(H=3, ctx=[64, 0, 777], ext=[1, 64, 29], chunk=256),
    dict(H=2, ctx=[256], ext=[40], chunk=64, doc=64),
    dict(H=128, ctx=[300], ext=[3], chunk=128),
], ids=["ragged", "batch", "docs", "h128"])
def test_absorbed_fp8_scores(api, case):
    wl = W.make_workload("af", case["H"], case["ctx"], case["ext"], chunk=case["chunk"], kv_dtype="fp8_e4m3",
                         doc_len=case.get("doc"), seed=90)
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run(absorbed="fp8")
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 0
    ref_out, ref_lse = O.mla_prefill(**O.workload_args(wl))
    assert_close_fp8_scores(out.cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, visible_keys(wl))


def test_absorbed_fp8_scores_long_context_sampled(api):
    wl = W.make_workload("afl", 128, [16384], [64], chunk=8192, kv_dtype="fp8_e4m3", seed=91)
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run(absorbed="fp8")
    torch.cuda.synchronize()
    rows, heads = np.array([0, 31, 63]), np.arange(0, 128, 11)
    ref_out, ref_lse = O.mla_prefill(**O.workload_args(wl), rows=rows, heads=heads)
    assert_close_fp8_scores(out.cpu().numpy()[rows][:, heads], lse.cpu().numpy()[rows][:, heads], ref_out, ref_lse,
                            visible_keys(wl)[rows])


def test_absorbed_fp8_scores_needs_fp8_cache(api):
    from mla_prefix_cache_gb300 import _lib
    wl = W.make_workload("afb", 2, [128], [4], chunk=64, seed=92)
    with pytest.raises(_lib.MLAError):
        api.DeviceWorkload(wl).run(absorbed="fp8")


# ---------------------------------------------------------------- per-request dispatch

@pytest.mark.parametrize("case", [
    dict(H=4, ctx=[1300, 500, 1064, 0, 1200], ext=[5, 300, 64, 129, 1], chunk=128),   # both paths, interleaved
    dict(H=3, ctx=[256, 1280], ext=[200, 40], chunk=64, doc=64),                     # relocated documents
    dict(H=2, ctx=[1537, 64], ext=[160, 7], chunk=192, kv="fp8_e4m3"),              # FP8 cache
    dict(H=4, ctx=[1300], ext=[20], chunk=128),                                      # absorbed only
    dict(H=4, ctx=[300], ext=[200], chunk=128),                                      # up-projected only
    dict(H=2, ctx=[1200, 1100], ext=[208, 209], chunk=128),                          # either side of the threshold
    dict(H=2, ctx=[1022, 1023], ext=[8, 8], chunk=128),                              # either side of 1024 keys
], ids=["mixed", "docs", "fp8", "short_only", "long_only", "threshold", "few_keys"])
def test_prefill_auto_matches_oracle(api, case):
    wl = W.make_workload("au", case["H"], case["ctx"], case["ext"], chunk=case["chunk"],
                         kv_dtype=case.get("kv", "bf16"), doc_len=case.get("doc"), seed=95)
    run_and_compare(api, wl, absorbed="auto")


def test_prefill_auto_reports_bad_blocks_of_either_path(api):
    wl = W.make_workload("ab2", 2, [1100, 256], [16, 200], chunk=128, seed=96)
    for req in (0, 1):                 # request 0: absorbed path, request 1: up-projected
        dw = api.DeviceWorkload(wl)
        dw.block_table[req, 1] = -5
        dw.run(absorbed="auto")
        torch.cuda.synchronize()
        assert api.device_error(api.prefill.last_workspace) == 3


# ---------------------------------------------------------------- FP8 up-projection (E4M3 kv_b_proj)

def _pow2_scale(amax):
    """The power of two >= amax / 448: e4m3 values times it are exact bf16."""
    return float(2.0 ** math.ceil(math.log2(amax / 448.0)))


def test_kv_b_proj_e4m3_bit_exact(api):
    """The device quantizer against the host encoder: absmax exact, codes
    bit-exact (round to nearest even, saturation at 448 included: the scale is
    absmax / 448, so the largest weights land on or next to 448)."""
    wl = W.make_workload("q8", 8, [64], [1], seed=60)
    dw = api.DeviceWorkload(wl)
    w = (wl.kv_b_proj.astype(np.uint32) << 16).view(np.float32)
    amax = float(np.abs(w).max())
    assert api.kv_b_proj_absmax(dw.kv_b_proj) == amax
    scale = float(np.float32(amax / 448.0))
    got = api.kv_b_proj_to_e4m3(dw.kv_b_proj, scale).cpu().numpy()
    assert got.shape == (8 * 256, 512)
    assert np.array_equal(got, W.kv_b_proj_e4m3_t(wl.kv_b_proj, scale))


FP8W_CASES = [
    dict(H=4, ctx=[513], ext=[200], chunk=192),                 # ragged kv and q tails, rows with few keys
    dict(H=3, ctx=[1100, 0, 1777], ext=[1, 64, 129], chunk=256),   # ragged batch
    dict(H=2, ctx=[1280], ext=[40], chunk=64, doc=64),          # relocated documents, partial states + merge
    dict(H=128, ctx=[1200], ext=[130], chunk=128),              # full head count
]


@pytest.mark.parametrize("case", FP8W_CASES, ids=["ragged", "batch", "docs", "h128"])
def test_prefill_fp8w_matches_oracle(api, case):
    """mla_prefill_ctx_fp8w computes mla_prefill_ctx with kv_b_proj replaced by
    its E4M3 rounding: against the oracle on those weights it is held to the
    same bars as mla_prefill_ctx (a power-of-two scale makes the rounded
    weights exact bf16, so the oracle takes them unchanged).  Against the
    oracle on the unrounded weights it moves by the weights' rounding
    (checked loosely: relative RMS of out <= 0.1, lse within 0.15)."""
    wl = W.make_workload("w8", case["H"], case["ctx"], case["ext"], chunk=case["chunk"], kv_dtype="fp8_e4m3",
                         doc_len=case.get("doc"), seed=61)
    w = (wl.kv_b_proj.astype(np.uint32) << 16).view(np.float32)
    scale = _pow2_scale(float(np.abs(w).max()))
    codes = W.kv_b_proj_e4m3_t(wl.kv_b_proj, scale)
    w_q = W.f32_to_bf16_bits(np.ascontiguousarray(O.e4m3_to_float(codes).T) * np.float32(scale))
    dw = api.DeviceWorkload(wl)
    out, lse = dw.run(kv_b_proj_e4m3=torch.from_numpy(codes).cuda(), w_scale=scale)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    args = O.workload_args(wl)
    args["kv_b_proj"] = w_q
    ref_out, ref_lse = O.mla_prefill(**args)
    assert_close(out, lse, ref_out, ref_lse, visible_keys(wl))
    raw_out, raw_lse = O.mla_prefill(**O.workload_args(wl))
    rel = math.sqrt(float(((out - raw_out) ** 2).mean())) / math.sqrt(float((raw_out ** 2).mean()))
    assert rel <= 0.1 and float(np.abs(lse - raw_lse).max()) <= 0.15


def test_prefill_fp8w_reports_bad_block_and_needs_fp8_cache(api):
    from mla_prefix_cache_gb300 import _lib
    wl = W.make_workload("w8e", 2, [256], [16], chunk=128, kv_dtype="fp8_e4m3", seed=62)
    dw = api.DeviceWorkload(wl)
    codes = torch.from_numpy(W.kv_b_proj_e4m3_t(wl.kv_b_proj, 1.0 / 1024)).cuda()
    dw.block_table[0, 1] = -5
    out, lse = dw.run(kv_b_proj_e4m3=codes, w_scale=1.0 / 1024)
    torch.cuda.synchronize()
    assert api.device_error(api.prefill.last_workspace) == 3    # MLA_ERR_BAD_BLOCK_ID
    assert torch.isfinite(out).all()
    wb = W.make_workload("w8b", 2, [256], [16], chunk=128, seed=62)
    with pytest.raises(_lib.MLAError):
        api.DeviceWorkload(wb).run(kv_b_proj_e4m3=codes, w_scale=1.0 / 1024)
