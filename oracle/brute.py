"""Scalar fp64 brute force for tiny inputs.  Test infrastructure only.

Every sum is an exactly rounded ``math.fsum`` over fp64 products, and every
step is an explicit loop over single tokens, heads and queries, with no masks,
no matrix products and no vectorised softmax.  It exists to pin the vectorised
oracle (``mla_oracle``) on inputs small enough for pure Python.

Definitions followed (web pages, by title and section):
"DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析" section 4.4 (gather,
kv_b_proj up-projection with K columns first then V columns, concat of the
broadcast k_rope, attention with lse) and section 5.2 (row layout);
"RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4 Long-Context
Serving" section 2 (query-side RoPE relocation per document segment).
"""
from __future__ import annotations

import math
import struct

import numpy as np

D_C, D_R, D_NOPE, D_V, BLOCK = 512, 64, 128, 128, 64


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def _e4m3(code: int) -> float:
    code = int(code)
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m, -9)          # m/8 * 2^-6
    return s * math.ldexp(8 + m, e - 10)      # (1 + m/8) * 2^(e-7)


def row(kv_cache, kv_dtype, kv_scale, table_row, t):
    """Decoded 576 values of logical token t."""
    b = int(table_row[t // BLOCK])
    raw = kv_cache[b, t % BLOCK]
    if kv_dtype == "bf16":
        return [_bf16(v) for v in raw.tolist()]
    vals = [_e4m3(v) * float(kv_scale) for v in raw[:D_C].tolist()]
    kb = raw[D_C:].tolist()
    vals += [_bf16(kb[2 * i] | (kb[2 * i + 1] << 8)) for i in range(D_R)]
    return vals


def rotate(pair_vals, delta, theta):
    """Interleaved pairs rotated by delta * theta^(-2k/64), per pair."""
    out = list(pair_vals)
    for k in range(D_R // 2):
        a = delta * theta ** (-(2.0 * k) / D_R)
        c, s = math.cos(a), math.sin(a)
        x0, x1 = pair_vals[2 * k], pair_vals[2 * k + 1]
        out[2 * k] = x0 * c - x1 * s
        out[2 * k + 1] = x0 * s + x1 * c
    return out


def prefill(q, q_pos, kv_cache, kv_dtype, kv_scale, block_table, ctx_lens, ext_lens, kv_b_proj,
            softmax_scale, rope_theta, segments=None, heads=None, rows=None):
    """Returns {(row, head): (out[128] list, lse float)} for the requested pairs."""
    T_q, H, _ = q.shape
    cu = [0]
    for e in ext_lens:
        cu.append(cu[-1] + int(e))
    heads = range(H) if heads is None else heads
    rows = range(T_q) if rows is None else rows
    W = [[_bf16(v) for v in r] for r in np.asarray(kv_b_proj).tolist()]
    res = {}
    kv_memo = {}
    for i in rows:
        r = max(k for k in range(len(ext_lens)) if cu[k] <= i and cu[k + 1] > i)
        C = int(ctx_lens[r])
        tok = C + (i - cu[r])
        # key set: (token, rope offset)
        keys = []
        segs = None
        if segments is not None:
            segs = [(int(s[1]), int(s[2]), int(s[3])) for s in np.asarray(segments).reshape(-1, 4) if int(s[0]) == r]
        else:
            segs = [(0, C, 0)]
        for start, n, off in segs:
            keys += [(t, off) for t in range(start, start + n)]
        keys += [(t, 0) for t in range(C, tok + 1)]
        rows_cache = {t: row(kv_cache, kv_dtype, kv_scale, block_table[r], t) for t, _ in keys}
        for h in heads:
            qv = [_bf16(v) for v in q[i, h].tolist()]
            qn, qr = qv[:D_NOPE], qv[D_NOPE:]
            scores, vals = [], []
            for t, off in keys:
                x = rows_cache[t]
                c, kr = x[:D_C], x[D_C:]
                if (r, t, h) not in kv_memo:
                    kv_memo[(r, t, h)] = (
                        [math.fsum(c[j] * W[j][h * D_NOPE + d] for j in range(D_C)) for d in range(D_NOPE)],
                        [math.fsum(c[j] * W[j][H * D_NOPE + h * D_V + d] for j in range(D_C)) for d in range(D_V)])
                kn, v = kv_memo[(r, t, h)]
                qrr = rotate(qr, int(q_pos[i]) - off, rope_theta)
                s = softmax_scale * (math.fsum(qn[d] * kn[d] for d in range(D_NOPE))
                                     + math.fsum(qrr[d] * kr[d] for d in range(D_R)))
                scores.append(s)
                vals.append(v)
            if not scores:
                res[(i, h)] = ([0.0] * D_V, -math.inf)
                continue
            m = max(scores)
            e = [math.exp(s - m) for s in scores]
            z = math.fsum(e)
            o = [math.fsum(e[k] * vals[k][d] for k in range(len(e))) / z for d in range(D_V)]
            res[(i, h)] = (o, m + math.log(z))
    return res
