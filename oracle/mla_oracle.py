"""Vectorised CPU oracle (numpy) for MLA chunked prefill.  Test infrastructure only.

The method reaches exactly (up to rounding order) a result with a plain
definition: attention of each query over the up-projected keys/values of every
visible cached token.  So the oracle materialises K/V per head and runs
*unchunked* full-softmax attention; ``mla_prefill_chunked`` additionally follows
the pages' chunk loop literally so the two can be checked against each other.

Sources (web pages, cited by title and section):

* [MLA-PC] "DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析":
  section 4.2 (two-stage prefill: context and extend each give (output, lse)),
  section 4.3 (merge_attn_states), section 4.4 (_compute_prefill_context chunk
  loop: gather, kv_b_proj up-projection, concat of broadcast k_rope,
  flash attention, merge), section 5.2 (packed 576-element row), section 2.2
  (FP8 cache; body missing from the extraction).
* [Tessera] "PagedAttention assumed MHA. DeepSeek-V4 says that assumption is
  broken": "What MLA changes about KV cache accounting" (DeepSeek-V3 geometry,
  latent 512, RoPE 64), "Block size is not a tuning knob here" (64-token blocks).
* [RedKnot] "RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4
  Long-Context Serving": section 2, "Online position restoration and merge"
  (query-side RoPE relocation into a document's canonical frame, segment merge).

Readings where the pages are silent (each also listed in the design notes):
natural-log lse with the softmax scale inside it; merged lse = max + ln(wa+wb);
identity state (out=0, lse=-inf); kv_b_proj columns = all heads' K_nope blocks
then all heads' V blocks, head-major; RoPE on interleaved pairs (2k, 2k+1) with
inverse frequency theta^(-2k/64) and angles from the integer position delta in
fp64; the context stage is unmasked and the extend stage causal with the
diagonal included; extend rows are read from the cache like context rows; FP8
rows are 512 E4M3FN codes times a per-tensor fp32 scale followed by 64 bf16
k_rope values.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

# Geometry: [Tessera] "What MLA changes about KV cache accounting" (latent 512,
# RoPE 64, head dim 128) and [MLA-PC] section 4.4 (d_nope = d_v = 128).
D_C = 512
D_R = 64
D_NOPE = 128
D_V = 128
D_QK = D_NOPE + D_R
BLOCK = 64                  # [Tessera] "Block size is not a tuning knob here"
ROW = D_C + D_R             # [MLA-PC] section 5.2: [c_kv 0..511 | k_rope 0..63]
ROW_BYTES_BF16 = 2 * ROW    # 1152
ROW_BYTES_FP8 = D_C + 2 * D_R  # 512 e4m3 codes + 64 bf16 values = 640

KV_BF16 = "bf16"
KV_FP8 = "fp8_e4m3"


# ---------------------------------------------------------------------------
# Storage decoding
# ---------------------------------------------------------------------------

def bf16_to_float(bits: np.ndarray, dtype=np.float32) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float: the upper half of an IEEE fp32."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(dtype)


def e4m3_to_float(codes: np.ndarray) -> np.ndarray:
    """OCP 8-bit E4M3FN code -> float64.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 gives
    subnormals m/8 * 2^-6; no infinities; S.1111.111 is NaN; largest finite
    value 448.  ([MLA-PC] section 2.2 names FP8 for the MLA cache; the format is
    the OCP E4M3 definition.)
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, val)


# ---------------------------------------------------------------------------
# Step 1: gather ([MLA-PC] section 4.4 step 1, section 5.2 row layout)
# ---------------------------------------------------------------------------

def gather_latent(kv_cache: np.ndarray, kv_dtype: str, kv_scale: float,
                  block_table_row: np.ndarray, tokens: Sequence[int],
                  dtype=np.float32) -> np.ndarray:
    """Rows of logical tokens ``tokens`` of one request, decoded to float [n, 576].

    Token t lives in physical block ``block_table_row[t // 64]`` at slot
    ``t % 64``.  BF16 rows decode exactly; FP8 rows give ``e4m3(code) * kv_scale``
    for the 512 latent values and the 64 bf16 k_rope values unchanged.
    """
    t = np.asarray(tokens, dtype=np.int64)
    blk = np.asarray(block_table_row, dtype=np.int64)[t // BLOCK]
    if (blk < 0).any() or (blk >= kv_cache.shape[0]).any():
        raise IndexError("block table entry out of range")
    raw = kv_cache[blk, t % BLOCK]
    if kv_dtype == KV_BF16:
        assert raw.shape[-1] == ROW
        return bf16_to_float(raw, dtype)
    if kv_dtype == KV_FP8:
        assert raw.shape[-1] == ROW_BYTES_FP8
        out = np.empty((t.shape[0], ROW), dtype=dtype)
        out[:, :D_C] = (e4m3_to_float(raw[:, :D_C]) * float(kv_scale)).astype(dtype)
        kr_bits = np.ascontiguousarray(raw[:, D_C:]).view(np.uint16)
        out[:, D_C:] = bf16_to_float(kr_bits, dtype)
        return out
    raise ValueError(kv_dtype)


# ---------------------------------------------------------------------------
# Step 2: up-projection ([MLA-PC] section 4.4 step 2)
# ---------------------------------------------------------------------------

def head_columns(h: int, num_heads: int) -> Tuple[slice, slice]:
    """Columns of kv_b_proj [512, H*(128+128)] holding head h's K_nope and V:
    the first H*128 columns are K_nope (head-major), the rest V (head-major)."""
    return (slice(h * D_NOPE, (h + 1) * D_NOPE),
            slice(num_heads * D_NOPE + h * D_V, num_heads * D_NOPE + (h + 1) * D_V))


def up_project(c_kv: np.ndarray, w: np.ndarray, h: int, num_heads: int):
    """K_nope_h = c_kv @ W[:, K cols of h];  V_h = c_kv @ W[:, V cols of h]."""
    ck, cv = head_columns(h, num_heads)
    return c_kv @ w[:, ck], c_kv @ w[:, cv]


# ---------------------------------------------------------------------------
# Query-side RoPE relocation ([RedKnot] section 2, "Online position
# restoration and merge")
# ---------------------------------------------------------------------------

def rope_inv_freq(theta: float) -> np.ndarray:
    """Inverse frequencies theta^(-2k/64), k = 0..31, in fp64."""
    return float(theta) ** (-np.arange(0, D_R, 2, dtype=np.float64) / D_R)


def rope_rotate(x: np.ndarray, delta, theta: float, dtype=None) -> np.ndarray:
    """Rotate each interleaved pair (x[2k], x[2k+1]) of the last axis (64 wide) by
    angle ``delta * theta^(-2k/64)``.  ``delta`` is an integer position (array
    broadcastable to x.shape[:-1]); the angle is formed in fp64 from it."""
    dtype = x.dtype if dtype is None else dtype
    xd = x.astype(np.float64)
    ang = np.asarray(delta, dtype=np.float64)[..., None] * rope_inv_freq(theta)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = xd[..., 0::2], xd[..., 1::2]
    y = np.empty_like(xd)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y.astype(dtype)


# ---------------------------------------------------------------------------
# Steps 3-4: concat + attention with (out, lse) ([MLA-PC] section 4.4 steps 3-4)
# ---------------------------------------------------------------------------

def softmax_attend(s: np.ndarray, v: np.ndarray):
    """Full softmax over the key axis of a score block s [m, n] (-inf = masked).

    out = sum_t softmax(s)_t v_t,  lse = ln sum_t exp(s_t).  A row with no
    visible key gives out = 0, lse = -inf (the merge identity)."""
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf, dtype=s.dtype)
    finite = np.isfinite(m)
    msafe = np.where(finite, m, 0).astype(s.dtype)
    p = np.exp(s - msafe[:, None])
    l = p.sum(axis=1)
    out = np.zeros((s.shape[0], v.shape[1]), dtype=s.dtype)
    if finite.any():
        out[finite] = (p[finite] @ v) / l[finite, None]
    lse = np.full(s.shape[0], -np.inf, dtype=s.dtype)
    lse[finite] = msafe[finite] + np.log(l[finite])
    return out, lse


def attention(qn, qr, kn, kr, v, scale, mask=None):
    """One score group: s = scale*(qn.kn + qr.kr) (k_rope broadcast to every head),
    masked where ``mask`` is False, then full softmax."""
    s = (qn @ kn.T + qr @ kr.T) * np.asarray(scale, dtype=qn.dtype)
    if mask is not None:
        s = np.where(mask, s, -np.inf).astype(qn.dtype)
    return softmax_attend(s, v)


# ---------------------------------------------------------------------------
# Step 5: merge ([MLA-PC] section 4.3)
# ---------------------------------------------------------------------------

def merge_attn_states(out_a, lse_a, out_b, lse_b):
    """LSE-weighted average of two partial states.

    m = max(lse_a, lse_b); wa = e^(lse_a - m); wb = e^(lse_b - m);
    out = (wa out_a + wb out_b) / (wa + wb); lse = m + ln(wa + wb).
    Two empty states (both lse = -inf) merge to (0, -inf)."""
    lse_a = np.asarray(lse_a)
    lse_b = np.asarray(lse_b)
    m = np.maximum(lse_a, lse_b)
    empty = ~np.isfinite(m)
    msafe = np.where(empty, 0, m)
    wa = np.where(np.isfinite(lse_a), np.exp(lse_a - msafe), 0)
    wb = np.where(np.isfinite(lse_b), np.exp(lse_b - msafe), 0)
    den = np.where(empty, 1, wa + wb)
    out = (wa[..., None] * out_a + wb[..., None] * out_b) / den[..., None]
    out = np.where(empty[..., None], 0, out)
    lse = np.where(empty, -np.inf, msafe + np.log(den))
    return out.astype(np.result_type(out_a, out_b)), lse.astype(np.result_type(lse_a, lse_b))


# ---------------------------------------------------------------------------
# The whole path
# ---------------------------------------------------------------------------

def key_groups(ctx_len: int, ext_len: int, req: int, segments, parts: int):
    """Key groups of one request as (first token, count, rope_offset, causal).

    Context keys: the request's segments (default: one segment [0, C_r) with
    offset 0).  Extend keys: tokens C_r .. C_r+E_r-1, offset 0, causal."""
    groups = []
    if parts & 1:
        segs = None
        if segments is not None:
            segs = [tuple(int(v) for v in s[1:]) for s in np.asarray(segments).reshape(-1, 4) if int(s[0]) == req]
        if not segs:
            segs = [(0, ctx_len, 0)] if segments is None else []
        for start, n, off in segs:
            groups.append((start, n, off, False))
    if parts & 2:
        groups.append((ctx_len, ext_len, 0, True))
    return groups


def mla_prefill(q, q_pos, kv_cache, kv_dtype, kv_scale, block_table, ctx_lens, ext_lens,
                kv_b_proj, softmax_scale, rope_theta, segments=None, parts=3,
                dtype=np.float32, heads: Optional[Sequence[int]] = None,
                rows: Optional[Sequence[int]] = None, q_block: int = 256):
    """Unchunked MLA prefill for every (query row, head) requested.

    q [T_q, H, 192] bf16 bits ([q_nope | q_rope], q_rope unrotated); q_pos [T_q];
    kv_b_proj [512, H*256] bf16 bits.  For query i of request r at position p and
    head h, the key set is the request's context segments plus (causally) its
    extend tokens C_r + j, j <= i.  Keys of a group with rope offset o are scored
    with q_rope rotated by (p - o).  Returns out [n_rows, n_heads, 128] and
    lse [n_rows, n_heads] in ``dtype`` (rows/heads default to all)."""
    q = np.asarray(q)
    T_q, H, _ = q.shape
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    ext_lens = np.asarray(ext_lens, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(ext_lens)])
    heads = list(range(H)) if heads is None else [int(h) for h in heads]
    rows = np.arange(T_q) if rows is None else np.asarray(rows, dtype=np.int64)
    w = bf16_to_float(kv_b_proj, dtype)
    out = np.zeros((rows.shape[0], len(heads), D_V), dtype=dtype)
    lse = np.full((rows.shape[0], len(heads)), -np.inf, dtype=dtype)
    row_req = np.searchsorted(cu, rows, side="right") - 1

    for r in range(ctx_lens.shape[0]):
        sel = np.nonzero(row_req == r)[0]
        if sel.size == 0:
            continue
        C, E = int(ctx_lens[r]), int(ext_lens[r])
        groups = key_groups(C, E, r, segments, parts)
        toks = np.concatenate([np.arange(g[0], g[0] + g[1]) for g in groups]) if groups else np.zeros(0, np.int64)
        x = gather_latent(kv_cache, kv_dtype, kv_scale, block_table[r], toks, dtype)
        c_kv, k_rope = x[:, :D_C], x[:, D_C:]
        for hi, h in enumerate(heads):
            kn, v = up_project(c_kv, w, h, H)
            for b0 in range(0, sel.size, q_block):
                bsel = sel[b0:b0 + q_block]
                qrows = rows[bsel]
                qh = bf16_to_float(q[qrows, h], dtype)
                qn, qr = qh[:, :D_NOPE], qh[:, D_NOPE:]
                pos = np.asarray(q_pos, dtype=np.int64)[qrows]
                qtok = C + (qrows - cu[r])          # token index of each query
                s_parts, col = [], 0
                for start, n, off, causal in groups:
                    ks = slice(col, col + n)
                    qrr = rope_rotate(qr, pos - off, rope_theta, dtype)
                    s = (qn @ kn[ks].T + qrr @ k_rope[ks].T) * np.asarray(softmax_scale, dtype=dtype)
                    if causal:
                        ktok = np.arange(start, start + n)
                        s = np.where(ktok[None, :] <= qtok[:, None], s, -np.inf).astype(dtype)
                    s_parts.append(s)
                    col += n
                s_all = np.concatenate(s_parts, axis=1) if s_parts else np.zeros((bsel.size, 0), dtype)
                o, l = softmax_attend(s_all, v)
                out[bsel, hi] = o
                lse[bsel, hi] = l
    return out, lse


def mla_prefill_chunked(q, q_pos, kv_cache, kv_dtype, kv_scale, block_table, ctx_lens, ext_lens,
                        kv_b_proj, softmax_scale, rope_theta, chunk, segments=None,
                        dtype=np.float64):
    """The pages' two-stage algorithm, step by step ([MLA-PC] sections 4.2-4.4).

    For each request: the context key range of every segment is cut into chunks
    of ``chunk`` tokens; for each chunk: gather the rows, up-project through
    kv_b_proj, concatenate the broadcast k_rope, attend (out, lse), and merge
    into the running context state, which starts at the identity (0, -inf).
    The extend stage attends causally over the new tokens, and the two stages
    are merged.  Returns out [T_q, H, 128], lse [T_q, H]."""
    q = np.asarray(q)
    T_q, H, _ = q.shape
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    ext_lens = np.asarray(ext_lens, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(ext_lens)])
    w = bf16_to_float(kv_b_proj, dtype)
    out = np.zeros((T_q, H, D_V), dtype=dtype)
    lse = np.full((T_q, H), -np.inf, dtype=dtype)
    for r in range(ctx_lens.shape[0]):
        C, E = int(ctx_lens[r]), int(ext_lens[r])
        if E == 0:
            continue
        qr_rows = np.arange(cu[r], cu[r + 1])
        qall = bf16_to_float(q[qr_rows], dtype)            # [E, H, 192]
        pos = np.asarray(q_pos, dtype=np.int64)[qr_rows]
        qtok = C + np.arange(E)
        for h in range(H):
            qn, qr = qall[:, h, :D_NOPE], qall[:, h, D_NOPE:]
            ctx_out = np.zeros((E, D_V), dtype=dtype)
            ctx_lse = np.full(E, -np.inf, dtype=dtype)
            for start, n, off, _ in key_groups(C, E, r, segments, 1):
                for c0 in range(start, start + n, chunk):
                    toks = np.arange(c0, min(c0 + chunk, start + n))
                    x = gather_latent(kv_cache, kv_dtype, kv_scale, block_table[r], toks, dtype)
                    kn, v = up_project(x[:, :D_C], w, h, H)
                    qrr = rope_rotate(qr, pos - off, rope_theta, dtype)
                    c_out, c_lse = attention(qn, qrr, kn, x[:, D_C:], v, softmax_scale)
                    ctx_out, ctx_lse = merge_attn_states(ctx_out, ctx_lse, c_out, c_lse)
            toks = np.arange(C, C + E)
            x = gather_latent(kv_cache, kv_dtype, kv_scale, block_table[r], toks, dtype)
            kn, v = up_project(x[:, :D_C], w, h, H)
            qrr = rope_rotate(qr, pos, rope_theta, dtype)
            mask = toks[None, :] <= qtok[:, None]
            e_out, e_lse = attention(qn, qrr, kn, x[:, D_C:], v, softmax_scale, mask)
            o, l = merge_attn_states(ctx_out, ctx_lse, e_out, e_lse)
            out[qr_rows, h] = o
            lse[qr_rows, h] = l
    return out, lse


def workload_args(wl) -> dict:
    """Keyword arguments of ``mla_prefill`` taken from a workload-like object
    (attribute access only; no import of the object's module)."""
    return dict(q=wl.q, q_pos=wl.q_pos, kv_cache=wl.kv_cache, kv_dtype=wl.kv_dtype,
                kv_scale=wl.kv_scale, block_table=wl.block_table, ctx_lens=wl.ctx_lens,
                ext_lens=wl.ext_lens, kv_b_proj=wl.kv_b_proj, softmax_scale=wl.softmax_scale,
                rope_theta=wl.rope_theta, segments=wl.segments)


def kv_cache_gib(context: int, layers: int = 61, heads: int = 128, head_dim: int = 128,
                 latent: int = D_C, rope: int = D_R) -> dict:
    """Per-layer-stack KV bytes for DeepSeek-V3 geometry ([Tessera] table in
    "What MLA changes about KV cache accounting"), in GiB."""
    mha = 2 * heads * head_dim * 2 * layers * context
    mla_bf16 = (latent + rope) * 2 * layers * context
    mla_fp8 = (latent + 2 * rope) * layers * context
    g = float(2 ** 30)
    return {"mha_bf16": mha / g, "mla_bf16": mla_bf16 / g, "mla_fp8": mla_fp8 / g,
            "ratio_bf16": mha / mla_bf16}
