"""Seeded synthetic inputs for MLA chunked prefill over a paged packed-latent cache.

This module only *constructs inputs*: random draws, rounding of those draws to the
storage formats, block-pool layout and NaN sentinels.  It holds none of the
method's arithmetic (no gather, up-projection, rotation, attention or merge), so
both the CPU oracle and the CUDA path can be fed from it without sharing code.

Storage formats (DeepSeek MLA cache note, section 5.2: one interleaved row
``[c_kv 0..511 | k_rope 0..63]`` = 576 elements per token; Tessera notes,
"Block size is not a tuning knob here": 64-token blocks):

* BF16 cache: ``uint16`` array ``[num_blocks, 64, 576]`` holding bfloat16 bit
  patterns.
* FP8 cache: ``uint8`` array ``[num_blocks, 64, 640]``; bytes 0..511 are OCP
  E4M3FN codes of ``c_kv / kv_scale`` and bytes 512..639 are the 64 ``k_rope``
  values as little-endian bfloat16.

Every bfloat16 tensor is carried as ``uint16`` bit patterns (numpy has no
bfloat16); the consumer reinterprets the bytes.

Recipe (one seeded ``numpy.random.Generator(PCG64(seed))`` per workload):
q, c_kv and k_rope are N(0,1) in fp32 rounded to bf16 (round-to-nearest-even);
kv_b_proj is N(0,1)/sqrt(512) rounded to bf16.  Cached k_rope is drawn directly
as N(0,1): a rotation of an isotropic Gaussian pair is again isotropic Gaussian,
so "stored already rotated at its (true or canonical) position" has the same
distribution.  Blocks come from a pool of sum(ceil(seq_len/64)) blocks plus 10 %
spare under a random physical permutation; spare blocks and tail slots past
``seq_len`` hold NaN so any stray read poisons the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

D_C = 512        # latent width
D_R = 64         # RoPE width
D_NOPE = 128     # no-RoPE key width per head
D_V = 128        # value width per head
D_QK = D_NOPE + D_R
BLOCK = 64       # tokens per cache block
ROW_BF16 = D_C + D_R           # elements per packed BF16 row
ROW_FP8_BYTES = D_C + 2 * D_R  # 512 e4m3 bytes + 64 bf16 k_rope

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)

KV_BF16 = "bf16"
KV_FP8 = "fp8_e4m3"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest-even), returning uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def kv_b_proj_e4m3_t(kv_b_proj: np.ndarray, w_scale: float) -> np.ndarray:
    """E4M3 codes of a bf16 kv_b_proj [512, H*256] (bit patterns) divided by
    w_scale, saturated to +-448 and rounded to nearest even by the library
    encoder, transposed to [H*256, 512] (the layout the FP8 up-projection
    reads)."""
    import torch  # library e4m3 encoder (CPU); only used to build inputs
    w = (np.ascontiguousarray(kv_b_proj).astype(np.uint32) << 16).view(np.float32)
    x = np.clip(w / np.float32(w_scale), np.float32(-448.0), np.float32(448.0)).astype(np.float32)
    codes = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return np.ascontiguousarray(codes.T)


@dataclasses.dataclass
class Workload:
    """All inputs of one prefill call (host copies)."""

    name: str
    num_heads: int
    ctx_lens: np.ndarray          # int32 [B]   C_r
    ext_lens: np.ndarray          # int32 [B]   E_r
    q: np.ndarray                 # uint16 [T_q, H, 192] bf16 bits, q_rope unrotated
    q_pos: np.ndarray             # int32 [T_q] true positions
    kv_dtype: str                 # "bf16" | "fp8_e4m3"
    kv_cache: np.ndarray          # uint16 [NB,64,576] or uint8 [NB,64,640]
    kv_scale: float
    block_table: np.ndarray       # int32 [B, max_blocks], -1 where unused
    kv_b_proj: np.ndarray         # uint16 [512, H*256] bf16 bits
    segments: Optional[np.ndarray]  # int64 [S, 4] (req, start, len, rope_offset) or None
    chunk: int
    softmax_scale: float
    rope_theta: float
    seed: int

    @property
    def num_reqs(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def seq_lens(self) -> np.ndarray:
        return (self.ctx_lens + self.ext_lens).astype(np.int32)

    @property
    def cu_q(self) -> np.ndarray:
        cu = np.zeros(self.num_reqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.ext_lens)
        return cu

    @property
    def total_q(self) -> int:
        return int(self.ext_lens.sum())

    @property
    def num_blocks(self) -> int:
        return int(self.kv_cache.shape[0])

    def algorithmic_flops(self) -> float:
        """Up-projection once per (token, head) plus attention over exactly the
        unmasked (query, key) pairs; dense K/V materialisation is never counted."""
        H = self.num_heads
        up = 2.0 * D_C * (D_NOPE + D_V) * H
        att = 2.0 * (D_QK + D_V) * H
        f = 0.0
        for c, e in zip(self.ctx_lens.tolist(), self.ext_lens.tolist()):
            f += (c + e) * up + e * c * att + e * (e + 1) / 2.0 * att
        return f

    def visible_pairs(self) -> float:
        """(query, key) pairs the attention covers, per head."""
        f = 0.0
        for c, e in zip(self.ctx_lens.tolist(), self.ext_lens.tolist()):
            f += e * c + e * (e + 1) / 2.0
        return f

    def absorbed_attention_flops(self) -> float:
        """Tensor-core work of the latent-space attention: per (query, key, head)
        a 576-wide score and a 512-wide P c product."""
        return 2.0 * (D_C + D_R + D_C) * self.num_heads * self.visible_pairs()

    def nbytes_inputs(self) -> int:
        return int(self.q.nbytes + self.kv_cache.nbytes + self.kv_b_proj.nbytes
                   + self.block_table.nbytes + self.q_pos.nbytes)


def _alloc_blocks(rng: np.random.Generator, seq_lens: Sequence[int]):
    need = [int(math.ceil(s / BLOCK)) for s in seq_lens]
    total = sum(need)
    pool = total + int(math.ceil(0.10 * total))
    perm = rng.permutation(pool).astype(np.int32)
    max_blocks = max(need) if need else 0
    table = np.full((len(seq_lens), max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(need):
        table[r, :n] = perm[off:off + n]
        off += n
    return table, pool


def make_workload(name: str, num_heads: int, ctx_lens: Sequence[int], ext_lens: Sequence[int],
                  *, kv_dtype: str = KV_BF16, chunk: int = 128, seed: int = 0,
                  doc_len: Optional[int] = None, rope_theta: float = 10000.0,
                  softmax_scale: Optional[float] = None, q_pos_base: Optional[Sequence[int]] = None
                  ) -> Workload:
    """Build one seeded workload.

    ``doc_len`` (relocated multi-document case): each request's context is cut into
    documents of ``doc_len`` tokens; document d becomes a segment
    ``(req, d*doc_len, doc_len, rope_offset=d*doc_len)`` whose k_rope is cached at
    canonical positions 0..doc_len-1.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(ctx_lens, dtype=np.int32)
    ext = np.asarray(ext_lens, dtype=np.int32)
    B = ctx.shape[0]
    H = int(num_heads)
    seq = ctx + ext
    T_q = int(ext.sum())

    table, pool = _alloc_blocks(rng, seq.tolist())

    q = f32_to_bf16_bits(rng.standard_normal((T_q, H, D_QK), dtype=np.float32))
    w = rng.standard_normal((D_C, H * (D_NOPE + D_V)), dtype=np.float32) / np.float32(math.sqrt(D_C))
    kv_b_proj = f32_to_bf16_bits(w)

    # Latent rows in logical (request, token) order, then scattered into the pool.
    valid = np.zeros((pool, BLOCK), dtype=bool)
    for r in range(B):
        nb = int(math.ceil(seq[r] / BLOCK))
        for lb in range(nb):
            n = min(BLOCK, int(seq[r]) - lb * BLOCK)
            valid[table[r, lb], :n] = True
    n_valid = int(valid.sum())
    ckv = rng.standard_normal((n_valid, D_C), dtype=np.float32)
    krope = f32_to_bf16_bits(rng.standard_normal((n_valid, D_R), dtype=np.float32))

    if kv_dtype == KV_BF16:
        cache = np.full((pool, BLOCK, ROW_BF16), BF16_NAN, dtype=np.uint16)
        rows = np.empty((n_valid, ROW_BF16), dtype=np.uint16)
        rows[:, :D_C] = f32_to_bf16_bits(ckv)
        rows[:, D_C:] = krope
        cache[valid] = rows
        kv_scale = 1.0
    elif kv_dtype == KV_FP8:
        import torch  # library e4m3 encoder (CPU); only used to build inputs
        amax = float(np.abs(ckv).max()) if n_valid else 1.0
        kv_scale = float(np.float32(amax / 448.0))
        codes = torch.from_numpy(ckv / np.float32(kv_scale)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        cache = np.empty((pool, BLOCK, ROW_FP8_BYTES), dtype=np.uint8)
        cache[:, :, :D_C] = E4M3_NAN
        kr_bytes = np.full((pool, BLOCK, D_R), BF16_NAN, dtype=np.uint16)
        kr_bytes[valid] = krope
        cache[:, :, D_C:] = kr_bytes.view(np.uint8).reshape(pool, BLOCK, 2 * D_R)
        cache[valid, :D_C] = codes
    else:
        raise ValueError(f"unknown kv_dtype {kv_dtype!r}")

    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(ext)
    q_pos = np.empty(T_q, dtype=np.int32)
    for r in range(B):
        base = int(ctx[r]) if q_pos_base is None else int(q_pos_base[r])
        q_pos[cu[r]:cu[r + 1]] = base + np.arange(int(ext[r]), dtype=np.int32)

    segments = None
    if doc_len is not None:
        segs: List[List[int]] = []
        for r in range(B):
            assert ctx[r] % doc_len == 0
            for d in range(int(ctx[r]) // doc_len):
                segs.append([r, d * doc_len, doc_len, d * doc_len])
        segments = np.asarray(segs, dtype=np.int64).reshape(-1, 4)

    scale = float(1.0 / math.sqrt(D_QK)) if softmax_scale is None else float(softmax_scale)
    return Workload(name=name, num_heads=H, ctx_lens=ctx, ext_lens=ext, q=q, q_pos=q_pos,
                    kv_dtype=kv_dtype, kv_cache=cache, kv_scale=kv_scale, block_table=table,
                    kv_b_proj=kv_b_proj, segments=segments, chunk=int(chunk),
                    softmax_scale=scale, rope_theta=float(rope_theta), seed=int(seed))


# ---------------------------------------------------------------------------
# The five workloads the bench and the full-size parity tests use.
# ---------------------------------------------------------------------------

def tiny() -> Workload:
    """1 request, 8 heads, 256 cached tokens in 4 shuffled blocks + 64 extend, chunk 128."""
    return make_workload("tiny", 8, [256], [64], chunk=128, seed=0)


def v3_8k() -> Workload:
    """DeepSeek-V3 geometry single layer: 128 heads, 8K context + 2K extend, chunk 4K."""
    return make_workload("v3_8k", 128, [8192], [2048], chunk=4096, seed=1)


def batched() -> Workload:
    """8 requests, 128 heads, context U{1K..32K step 64}, extend U{512..4K}, chunk 8K."""
    rng = np.random.Generator(np.random.PCG64(2))
    ctx = (rng.integers(1024 // 64, 32768 // 64 + 1, size=8) * 64).tolist()
    ext = rng.integers(512, 4096 + 1, size=8).tolist()
    return make_workload("batched", 128, ctx, ext, chunk=8192, seed=2)


def fp8_128k() -> Workload:
    """1 request, 128 heads, 128K FP8-e4m3 context (per-tensor scale) + 4K extend, chunk 16K."""
    return make_workload("fp8_128k", 128, [131072], [4096], kv_dtype=KV_FP8, chunk=16384, seed=3)


def reloc_256k() -> Workload:
    """16 documents x 16K cached at canonical positions, 4K extend at true offsets."""
    return make_workload("reloc_256k", 128, [262144], [4096], chunk=16384, seed=4, doc_len=16384)


def short_ext_32k() -> Workload:
    """A short extend for the absorbed (latent-space) path: 128 heads, 32K
    cached tokens + 64 new ones, chunk 16K, BF16."""
    return make_workload("short_ext_32k", 128, [32768], [64], chunk=16384, seed=5)


def short_ext_fp8_128k() -> Workload:
    """A short extend on the long FP8 cache: 128 heads, 128K FP8-e4m3 cached
    tokens + 64 new ones, chunk 16K."""
    return make_workload("short_ext_fp8_128k", 128, [131072], [64], kv_dtype=KV_FP8, chunk=16384, seed=6)


def mixed_32k() -> Workload:
    """A mixed serving batch, 128 heads, BF16: 4 requests with 32K cached +
    1024 new tokens and 12 short ones with 16K cached + 1 to 64 new tokens,
    chunk 16K."""
    ctx = [32768] * 4 + [16384] * 12
    ext = [1024] * 4 + [1, 4, 16, 64] * 3
    return make_workload("mixed_32k", 128, ctx, ext, chunk=16384, seed=7)


def long_16k() -> Workload:
    """A long-piece profiling case: 128 heads, 16K cached + 4K new tokens, chunk 16K, BF16 (two pieces of the
    long configurations' shape, small enough for a full ncu capture)."""
    return make_workload("long_16k", 128, [16384], [4096], chunk=16384, seed=8)


CONFIGS = {
    "tiny": tiny,
    "v3_8k": v3_8k,
    "batched": batched,
    "fp8_128k": fp8_128k,
    "reloc_256k": reloc_256k,
    "short_ext_32k": short_ext_32k,
    "short_ext_fp8_128k": short_ext_fp8_128k,
    "mixed_32k": mixed_32k,
    "long_16k": long_16k,
}


def by_name(name: str) -> Workload:
    return CONFIGS[name]()
