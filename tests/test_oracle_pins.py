"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
against something other than the oracle itself (closed forms, invariants,
library cross-checks, brute force on tiny inputs, worked fixtures)."""
import math
import os

import numpy as np
import pytest

from oracle import brute
from oracle import mla_oracle as O
from mla_prefix_cache_gb300 import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


# ---------------------------------------------------------------- row widths

def test_row_width_576_elements():
    # Packed row [c_kv 512 | k_rope 64] (MLA cache note, section 5.2).
    assert O.D_C + O.D_R == 576 == O.ROW
    assert O.ROW_BYTES_BF16 == 1152
    assert O.ROW_BYTES_FP8 == 640
    wl = W.make_workload("w", 1, [64], [1], seed=5)
    x = O.gather_latent(wl.kv_cache, wl.kv_dtype, 1.0, wl.block_table[0], [0, 5], np.float32)
    assert x.shape == (2, 576)


def test_kv_accounting_table_reproduces():
    for ctx, col, val, unit, rep in _rows("kv_cache_accounting.txt"):
        g = O.kv_cache_gib(int(ctx))
        got = g["ratio_bf16"] if col == "ratio" else g[col]
        if unit == "TB":
            got = got / 1000.0
        printed = float(val)
        ndig = len(val.split(".")[1])
        if rep == "1":
            assert round(got, ndig) == pytest.approx(printed), (ctx, col, got)
        else:
            # recorded inconsistency: the printed cell does not follow from 1152/640 B rows
            assert round(got, ndig) != pytest.approx(printed), (ctx, col, got)


# ---------------------------------------------------------------- FP8 decode

def test_e4m3_all_codes_match_library():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_float(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert sorted(np.nonzero(nan)[0].tolist()) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan], lib[~nan])
    assert np.nanmax(ours) == 448.0 and ours[1] == 2.0 ** -9
    for c in range(256):
        b = brute._e4m3(c)
        assert (math.isnan(b) and nan[c]) or b == ours[c]


# ---------------------------------------------------------------- merge

def test_merge_closed_form_fixture():
    for oa, la, ob, lb, o, l in _rows("merge_cases.txt"):
        got_o, got_l = O.merge_attn_states(np.array([[float(oa)]]), np.array([float(la)]),
                                           np.array([[float(ob)]]), np.array([float(lb)]))
        assert got_o[0, 0] == pytest.approx(float(o), abs=1e-12)
        if float(l) == -math.inf:
            assert got_l[0] == -math.inf
        else:
            assert got_l[0] == pytest.approx(float(l), abs=1e-12)


def _rand_state(rng, n=17, d=8):
    return rng.standard_normal((n, d)), rng.standard_normal(n) * 3


def test_merge_algebra():
    rng = np.random.default_rng(0)
    a, b, c = (_rand_state(rng) for _ in range(3))
    ab = O.merge_attn_states(*a, *b)
    ba = O.merge_attn_states(*b, *a)
    np.testing.assert_allclose(ab[0], ba[0], atol=1e-12)
    np.testing.assert_allclose(ab[1], ba[1], atol=1e-12)
    l1 = O.merge_attn_states(*ab, *c)
    r1 = O.merge_attn_states(*a, *O.merge_attn_states(*b, *c))
    np.testing.assert_allclose(l1[0], r1[0], atol=1e-12)
    np.testing.assert_allclose(l1[1], r1[1], atol=1e-12)
    ident = (np.zeros_like(a[0]), np.full(a[1].shape, -np.inf))
    e = O.merge_attn_states(*ident, *a)
    np.testing.assert_array_equal(e[0], a[0])
    np.testing.assert_allclose(e[1], a[1], atol=0)


def test_merge_of_partition_equals_union_attention():
    rng = np.random.default_rng(1)
    m, n = 9, 40
    qn, qr = rng.standard_normal((m, 128)), rng.standard_normal((m, 64))
    kn, kr, v = rng.standard_normal((n, 128)), rng.standard_normal((n, 64)), rng.standard_normal((n, 128))
    full = O.attention(qn, qr, kn, kr, v, 0.1)
    for cut in (1, 13, 39):
        a = O.attention(qn, qr, kn[:cut], kr[:cut], v[:cut], 0.1)
        b = O.attention(qn, qr, kn[cut:], kr[cut:], v[cut:], 0.1)
        mo, ml = O.merge_attn_states(*a, *b)
        np.testing.assert_allclose(mo, full[0], atol=1e-12)
        np.testing.assert_allclose(ml, full[1], atol=1e-12)


# ---------------------------------------------------------------- attention core

def test_attention_special_cases():
    rng = np.random.default_rng(2)
    qn, qr = rng.standard_normal((3, 128)), rng.standard_normal((3, 64))
    kn, kr, v = rng.standard_normal((1, 128)), rng.standard_normal((1, 64)), rng.standard_normal((1, 128))
    out, lse = O.attention(qn, qr, kn, kr, v, 0.3)
    np.testing.assert_allclose(out, np.repeat(v, 3, 0), atol=1e-14)
    s = 0.3 * np.array([np.dot(qn[i], kn[0]) + np.dot(qr[i], kr[0]) for i in range(3)])
    np.testing.assert_allclose(lse, s, atol=1e-12)
    n = 37
    kn, kr, v = rng.standard_normal((n, 128)), rng.standard_normal((n, 64)), rng.standard_normal((n, 128))
    out, lse = O.attention(np.zeros((2, 128)), np.zeros((2, 64)), kn, kr, v, 0.3)
    np.testing.assert_allclose(out, np.repeat(v.mean(0, keepdims=True), 2, 0), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(n), atol=1e-13)
    # empty key set -> identity state
    out, lse = O.attention(qn, qr, kn[:0], kr[:0], v[:0], 0.3)
    assert (out == 0).all() and (lse == -np.inf).all()


def test_causal_diagonal_included():
    # Zero queries make every visible key equally likely: query i of the extend
    # sees C + i + 1 keys (all context plus extend tokens 0..i).
    wl = W.make_workload("c", 2, [70], [5], seed=3)
    wl.q[:] = 0
    args = O.workload_args(wl)
    out, lse = O.mla_prefill(**args, dtype=np.float64)
    np.testing.assert_allclose(lse[:, 0], np.log(70 + np.arange(1, 6)), atol=1e-12)
    x = O.gather_latent(wl.kv_cache, "bf16", 1.0, wl.block_table[0], np.arange(75), np.float64)
    _, v = O.up_project(x[:, :512], O.bf16_to_float(wl.kv_b_proj, np.float64), 1, 2)
    for i in range(5):
        np.testing.assert_allclose(out[i, 1], v[:71 + i].mean(0), atol=1e-12)


# ---------------------------------------------------------------- up-projection

def test_up_projection_absorbed_equals_materialised():
    rng = np.random.default_rng(4)
    H = 3
    w = rng.standard_normal((512, H * 256)) / math.sqrt(512)
    c = rng.standard_normal((11, 512))
    qn = rng.standard_normal((5, 128))
    for h in range(H):
        kn, v = O.up_project(c, w, h, H)
        assert kn.shape == (11, 128) and v.shape == (11, 128)
        wk = w[:, h * 128:(h + 1) * 128]
        absorbed = (qn @ wk.T) @ c.T            # q . W_UK^T then dot with latents
        np.testing.assert_allclose(absorbed, qn @ kn.T, rtol=1e-12, atol=1e-11)
        # V columns start after all heads' K columns
        np.testing.assert_allclose(v, c @ w[:, H * 128 + h * 128: H * 128 + (h + 1) * 128], atol=0)


# ---------------------------------------------------------------- RoPE

def _rotate_complex(x, pos, theta):
    z = x[..., 0::2] + 1j * x[..., 1::2]
    k = np.arange(32)
    z = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * theta ** (-2.0 * k / 64.0))
    y = np.empty_like(x)
    y[..., 0::2], y[..., 1::2] = z.real, z.imag
    return y


def test_rope_matches_complex_multiplication_and_invariants():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 64))
    pos = np.array([0, 1, 7, 4095, 262144 + 17, -300])
    y = O.rope_rotate(x, pos, 10000.0, np.float64)
    np.testing.assert_allclose(y, _rotate_complex(x, pos, 10000.0), atol=1e-12)
    np.testing.assert_array_equal(O.rope_rotate(x, 0, 10000.0, np.float64), x)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    a, b, o = 1000, 37, 555
    qa = O.rope_rotate(x[0], a, 1e4, np.float64)
    kb = O.rope_rotate(x[1], b, 1e4, np.float64)
    qa2 = O.rope_rotate(x[0], a - o, 1e4, np.float64)
    kb2 = O.rope_rotate(x[1], b - o, 1e4, np.float64)
    assert np.dot(qa, kb) == pytest.approx(np.dot(qa2, kb2), abs=1e-11)


def test_relocation_equals_true_position_attention():
    """Documents cached with k_rope at canonical positions 0..L-1 and attended
    with query-side relocation (rotate q by p - o_d, merge per-document states)
    equal attention over keys rotated at their true positions o_d + j."""
    rng = np.random.default_rng(6)
    L, ndoc, m, theta = 64, 3, 8, 10000.0
    p = ndoc * L + np.arange(m)                         # queries after the documents
    qn, qr = rng.standard_normal((m, 128)), rng.standard_normal((m, 64))
    kn = rng.standard_normal((ndoc * L, 128))
    v = rng.standard_normal((ndoc * L, 128))
    raw = rng.standard_normal((ndoc * L, 64))
    j = np.tile(np.arange(L), ndoc)
    off = np.repeat(np.arange(ndoc) * L, L)
    kr_canon = _rotate_complex(raw, j, theta)
    kr_true = _rotate_complex(raw, off + j, theta)
    full = O.attention(qn, O.rope_rotate(qr, p, theta), kn, kr_true, v, 0.07)
    state = (np.zeros((m, 128)), np.full(m, -np.inf))
    for d in range(ndoc):
        sl = slice(d * L, (d + 1) * L)
        part = O.attention(qn, O.rope_rotate(qr, p - d * L, theta), kn[sl], kr_canon[sl], v[sl], 0.07)
        state = O.merge_attn_states(*state, *part)
    np.testing.assert_allclose(state[0], full[0], atol=1e-10)
    np.testing.assert_allclose(state[1], full[1], atol=1e-10)


# ---------------------------------------------------------------- gather

def test_gather_index_fixture():
    rows = _rows("gather_case.txt")
    table = np.array([3, 0, 2], dtype=np.int32)
    nb = 4
    cache = np.zeros((nb, 64, 576), dtype=np.uint16)
    for b in range(nb):
        for s in range(64):
            cache[b, s, :] = W.f32_to_bf16_bits(np.full(576, b * 64 + s, np.float32))
    toks = [int(r[0]) for r in rows]
    x = O.gather_latent(cache, "bf16", 1.0, table, toks, np.float64)
    for (t, pb, sl), xr in zip(rows, x):
        assert (xr == int(pb) * 64 + int(sl)).all()
    with pytest.raises(IndexError):
        O.gather_latent(cache, "bf16", 1.0, np.array([0, -1]), [64], np.float64)


def test_fp8_gather_layout():
    wl = W.make_workload("f", 1, [64], [8], kv_dtype="fp8_e4m3", seed=7)
    x = O.gather_latent(wl.kv_cache, wl.kv_dtype, wl.kv_scale, wl.block_table[0], np.arange(72), np.float64)
    raw = wl.kv_cache[wl.block_table[0][1], 3]
    assert x[67, 0] == O.e4m3_to_float(raw[0]) * wl.kv_scale
    kr = int(raw[512]) | (int(raw[513]) << 8)
    assert x[67, 512] == O.bf16_to_float(np.array([kr], np.uint16), np.float64)[0]
    assert np.isfinite(x).all()


# ---------------------------------------------------------------- chunked == unchunked

@pytest.mark.parametrize("chunk", [64, 100, 128, 1000])
def test_chunk_loop_equals_unchunked(chunk):
    wl = W.make_workload("ch", 2, [300, 64], [17, 9], seed=8)
    args = O.workload_args(wl)
    ref = O.mla_prefill(**args, dtype=np.float64)
    got = O.mla_prefill_chunked(**args, chunk=chunk, dtype=np.float64)
    np.testing.assert_allclose(got[0], ref[0], atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], atol=1e-12)


def test_chunk_loop_with_segments_equals_unchunked():
    wl = W.make_workload("seg", 2, [192], [7], seed=9, doc_len=64, q_pos_base=[192])
    args = O.workload_args(wl)
    ref = O.mla_prefill(**args, dtype=np.float64)
    got = O.mla_prefill_chunked(**args, chunk=64, dtype=np.float64)
    np.testing.assert_allclose(got[0], ref[0], atol=1e-12)
    np.testing.assert_allclose(got[1], ref[1], atol=1e-12)


def test_parts_merge_to_whole():
    wl = W.make_workload("pm", 2, [130], [20], seed=10)
    args = O.workload_args(wl)
    whole = O.mla_prefill(**args, dtype=np.float64)
    ctx = O.mla_prefill(**args, parts=1, dtype=np.float64)
    ext = O.mla_prefill(**args, parts=2, dtype=np.float64)
    mo, ml = O.merge_attn_states(*ctx, *ext)
    np.testing.assert_allclose(mo, whole[0], atol=1e-12)
    np.testing.assert_allclose(ml, whole[1], atol=1e-12)


def test_sampled_rows_heads_equal_full():
    wl = W.make_workload("s", 3, [100, 200], [10, 6], seed=11)
    args = O.workload_args(wl)
    full = O.mla_prefill(**args)
    rows, heads = [0, 9, 10, 15], [2, 0]
    sub = O.mla_prefill(**args, rows=rows, heads=heads)
    np.testing.assert_array_equal(sub[0], full[0][rows][:, heads])
    np.testing.assert_array_equal(sub[1], full[1][rows][:, heads])


# ---------------------------------------------------------------- brute force

def _brute_compare(wl, rows, heads, atol_out, atol_lse, dtype):
    args = O.workload_args(wl)
    vec = O.mla_prefill(**args, rows=rows, heads=heads, dtype=dtype)
    bf = brute.prefill(**args, heads=heads, rows=rows)
    for ri, i in enumerate(rows):
        for hi, h in enumerate(heads):
            o, l = bf[(i, h)]
            np.testing.assert_allclose(vec[0][ri, hi], np.array(o), atol=atol_out, rtol=0)
            assert abs(vec[1][ri, hi] - l) <= atol_lse


def test_brute_force_bf16_ragged():
    wl = W.make_workload("b", 2, [70], [4], seed=12)
    _brute_compare(wl, [0, 3], [0, 1], 1e-12, 1e-12, np.float64)
    _brute_compare(wl, [0, 3], [0, 1], 2e-5, 2e-5, np.float32)


def test_brute_force_fp8():
    wl = W.make_workload("b8", 1, [64], [3], kv_dtype="fp8_e4m3", seed=13)
    _brute_compare(wl, [0, 2], [0], 1e-12, 1e-12, np.float64)


def test_brute_force_segments_relocated():
    wl = W.make_workload("bs", 1, [128], [2], seed=14, doc_len=64)
    _brute_compare(wl, [0, 1], [0], 1e-12, 1e-12, np.float64)
