"""CPU oracle for the content-addressed block store's GPU steps.  Test
infrastructure only.

Source: "PagedAttention assumed MHA. DeepSeek-V4 says that assumption is
broken", sections "Position independence beats prefix matching" (hash a
block's latents when it is sealed, look the hash up, share the block on a
match) and "The finding: content-addressed dedup needs byte verification"
(on a hash match compare the bytes; if they differ, install the candidate as
a fresh block and count a dedup collision).

Reading: the page's hash is xxh3, a fast non-cryptographic 64-bit hash; the
scheme needs only some such hash, since byte verification makes sharing exact
whatever the hash.  This library defines its own, from a published mixer so
that the GPU can reduce a block in any order:

    h(block) = mix(n XOR sum_i mix(w_i + (i + 1) * GAMMA))      (mod 2^64)

where w_0..w_{n-1} are the block's bytes read as little-endian 64-bit words,
GAMMA = 0x9e3779b97f4a7c15 and mix is the SplitMix64 output function (Steele,
Lea and Flood, "Fast splittable pseudorandom number generators", 2014, with
the multipliers of Stafford's "mix13"):

    z ^= z >> 30; z *= 0xbf58476d1ce4e5b9; z ^= z >> 27; z *= 0x94d049bb133111eb; z ^= z >> 31.

Addition mod 2^64 is associative and commutative, so every reduction order
gives the same bits; the (i + 1) * GAMMA term makes the hash depend on where
each word sits.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 values (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def block_words(kv_cache: np.ndarray, block: int) -> np.ndarray:
    """The bytes of one 64-token cache block (as stored: bf16 rows of 576 or
    640-byte FP8 rows) as little-endian 64-bit words."""
    raw = np.ascontiguousarray(kv_cache[block]).view(np.uint8).reshape(-1)
    return raw.view("<u8")


def block_hash(kv_cache: np.ndarray, block: int) -> int:
    """h(block) as defined in the module docstring."""
    w = block_words(kv_cache, block)
    n = w.shape[0]
    idx = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        terms = mix(w + idx * GAMMA)
        acc = np.uint64(0)
        for t in np.array_split(terms, 16):     # wrapping sum
            acc = acc + np.sum(t, dtype=np.uint64)
    return int(mix(np.uint64(n) ^ acc))


def blocks_equal(kv_cache: np.ndarray, a: int, b: int) -> bool:
    return bool(np.array_equal(np.asarray(kv_cache[a]).view(np.uint8), np.asarray(kv_cache[b]).view(np.uint8)))


class SealStore:
    """The page's seal protocol over one cache pool, in order of the calls:
    look the candidate's hash up; on a match byte-compare it with every block
    installed under that hash; share the first equal one, else install the
    candidate and, if the hash did match, count a collision.

    ``hash_bits`` keeps only the low bits of the hash, so that tests can make
    distinct blocks collide."""

    def __init__(self, hash_bits: int = 64):
        self.mask = (1 << hash_bits) - 1
        self.table: Dict[int, List[int]] = {}
        self.collisions = 0

    def seal(self, kv_cache: np.ndarray, block: int, h: Optional[int] = None) -> int:
        """Returns the block that now holds the candidate's content: an
        installed block with the same bytes, or the candidate itself."""
        key = (block_hash(kv_cache, block) if h is None else int(h)) & self.mask
        same = self.table.get(key)
        if same:
            for b in same:
                if blocks_equal(kv_cache, b, block):
                    return b
            self.collisions += 1
            same.append(block)
            return block
        self.table[key] = [block]
        return block


def seal_all(kv_cache: np.ndarray, blocks: Sequence[int], hash_bits: int = 64) -> Tuple[List[int], int]:
    """Seal the blocks in order; returns (holder of each block, collisions)."""
    st = SealStore(hash_bits)
    return [st.seal(kv_cache, int(b)) for b in blocks], st.collisions
