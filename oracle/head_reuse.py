"""CPU oracle of head-split reuse with protected-row replacement.  Test
infrastructure only.

Source: "RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4
Long-Context Serving".
- Section 2: Local and Global heads are disjoint roles over the logical
  heads of one packed latent stream.  Local contributions are retained
  offline (MLA-Off); the Global heads and the protected Local token rows are
  recomputed online (MLA-Online).  Cached Local values of protected rows are
  replaced, not double counted.
- Section 3.A: the structural logical head-row ceiling.

Reading (one attention layer): the offline artifact gives, for every query
row t and head h, a state (art_out[t, h], art_lse[t, h]).  The layer's result
is the plain attention state of mla_oracle.mla_prefill where h is Global or
row t is protected, and the artifact everywhere else.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np

from . import mla_oracle as O


def reuse_mask(num_rows: int, num_heads: int, global_heads: Sequence[int], protected_rows: Sequence[int]) -> np.ndarray:
    """True where (row, head) is recomputed online."""
    m = np.zeros((num_rows, num_heads), dtype=bool)
    m[:, list(global_heads)] = True
    m[list(protected_rows), :] = True
    return m


def prefill_reuse(args: dict, global_heads: Sequence[int], protected_rows: Sequence[int], art_out: np.ndarray,
                  art_lse: np.ndarray, dtype=np.float32):
    """args: keyword arguments of mla_oracle.mla_prefill (see workload_args).
    Returns (out [T_q, H, 128], lse [T_q, H])."""
    T_q, H = art_lse.shape
    out = np.array(art_out, dtype=dtype, copy=True)
    lse = np.array(art_lse, dtype=dtype, copy=True)
    g = sorted(set(int(h) for h in global_heads))
    p = sorted(set(int(t) for t in protected_rows))
    if g:
        o, l = O.mla_prefill(**args, heads=g, dtype=dtype)
        out[:, g], lse[:, g] = o, l
    local = [h for h in range(H) if h not in set(g)]
    if p and local:
        o, l = O.mla_prefill(**args, heads=local, rows=p, dtype=dtype)
        out[np.ix_(p, local)], lse[np.ix_(p, local)] = o, l
    return out, lse


def head_row_ceiling(reusable_layers: int, total_layers: int, local_heads: int, global_heads: int) -> float:
    """Fraction of logical (layer, head, row) entries that reuse can skip: the
    reusable layers' share times the Local heads' share."""
    return reusable_layers / total_layers * local_heads / (local_heads + global_heads)


def reused_fraction(num_rows: int, num_heads: int, global_heads: Sequence[int], protected_rows: Sequence[int]) -> float:
    """Fraction of one layer's (row, head) entries served from the artifact."""
    return 1.0 - float(reuse_mask(num_rows, num_heads, global_heads, protected_rows).mean())
