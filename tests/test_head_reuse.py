"""Pins of the head-split reuse oracle (oracle/head_reuse.py): reduction to
plain attention, pass-through of the artifact, replacement (not double
counting) of protected rows, and the RedKnot page's printed head-row
ceilings."""
import os

import numpy as np
import pytest

from mla_prefix_cache_gb300 import workload as W
from oracle import head_reuse as R
from oracle import mla_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def small():
    wl = W.make_workload("r", 6, [192, 128], [40, 17], chunk=64, seed=60, doc_len=64)
    args = O.workload_args(wl)
    rng = np.random.default_rng(61)
    art_out = rng.standard_normal((wl.total_q, 6, 128)).astype(np.float32)
    art_lse = rng.standard_normal((wl.total_q, 6)).astype(np.float32)
    return wl, args, art_out, art_lse


def test_all_heads_global_is_plain_attention():
    wl, args, ao, al = small()
    o, l = R.prefill_reuse(args, range(6), [], ao, al)
    ro, rl = O.mla_prefill(**args)
    assert np.array_equal(o, ro) and np.array_equal(l, rl)


def test_no_online_work_returns_the_artifact():
    wl, args, ao, al = small()
    o, l = R.prefill_reuse(args, [], [], ao, al)
    assert np.array_equal(o, ao) and np.array_equal(l, al)


def test_protected_rows_are_replaced_not_accumulated():
    wl, args, ao, al = small()
    g, p = [1, 4], [0, 3, 41, 56]
    o1, l1 = R.prefill_reuse(args, g, p, ao, al)
    m = R.reuse_mask(wl.total_q, 6, g, p)
    ao2, al2 = ao.copy(), al.copy()
    ao2[m] += 5.0                 # artifact values under recomputed entries do not matter
    al2[m] -= 3.0
    o2, l2 = R.prefill_reuse(args, g, p, ao2, al2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    full_o, full_l = O.mla_prefill(**args)
    assert np.allclose(o1[m], full_o[m], atol=1e-6) and np.allclose(l1[m], full_l[m], atol=1e-6)
    assert np.array_equal(o1[~m], ao[~m]) and np.array_equal(l1[~m], al[~m])


def test_printed_head_row_ceilings():
    with open(os.path.join(HERE, "golden", "redknot_ceilings.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for name, ff, nr, fb, loc, glo, pct in rows:
        c = R.head_row_ceiling(int(nr), int(ff) + int(nr) + int(fb), int(loc), int(glo))
        assert round(100 * c, 2) == pytest.approx(float(pct)), name


def test_reused_fraction_counts_entries():
    assert R.reused_fraction(100, 64, range(8), []) == pytest.approx(56 / 64)
    assert R.reused_fraction(100, 64, range(8), range(10)) == pytest.approx(0.9 * 56 / 64)
