"""Pins of the block-store oracle (oracle/block_store.py): the content hash
of a sealed 64-token block and the seal protocol of "PagedAttention assumed
MHA. DeepSeek-V4 says that assumption is broken" (hash, look up, byte-verify,
share or install fresh and count a collision)."""
import os

import numpy as np
import pytest

from mla_prefix_cache_gb300 import workload as W
from oracle import block_store as B

HERE = os.path.dirname(os.path.abspath(__file__))
M64 = (1 << 64) - 1


def golden_splitmix():
    with open(os.path.join(HERE, "golden", "splitmix64.txt")) as f:
        return [int(x, 16) for x in (ln.strip() for ln in f) if x and not x.startswith("#")]


def splitmix64(n):
    """The published generator, sequentially: state += gamma; output mix(state)."""
    out, state = [], 0
    for _ in range(n):
        state = (state + int(B.GAMMA)) & M64
        out.append(int(B.mix(np.uint64(state))))
    return out


def test_mix_matches_published_splitmix64_outputs():
    assert splitmix64(3) == golden_splitmix()


def test_mix_is_a_bijection():
    """Invert each step (xorshift by s: z ^= z >> s ^ z >> 2s ...; odd
    multipliers: their inverse mod 2^64) and recover random inputs."""
    def unshift(z, s):
        r = z
        for _ in range(64 // s):
            r = z ^ (r >> s)
        return r & M64
    inv1, inv2 = pow(int(B._M1), -1, 1 << 64), pow(int(B._M2), -1, 1 << 64)
    rng = np.random.default_rng(0)
    for x in rng.integers(0, 2**63, size=200, dtype=np.int64).astype(np.uint64).tolist() + [0, M64]:
        z = int(B.mix(np.uint64(x)))
        z = unshift(z, 31)
        z = (z * inv2) & M64
        z = unshift(z, 27)
        z = (z * inv1) & M64
        z = unshift(z, 30)
        assert z == x


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_zero_block_hash_is_splitmix_sum(kv):
    """A block of zero words hashes to mix(n XOR sum of the first n outputs of
    SplitMix64), n = 9216 (bf16 rows) or 5120 (FP8 rows) words."""
    shape = (2, 64, 576) if kv == "bf16" else (2, 64, 640)
    cache = np.zeros(shape, dtype=np.uint16 if kv == "bf16" else np.uint8)
    n = cache[0].nbytes // 8
    s = sum(splitmix64(n)) & M64
    assert B.block_hash(cache, 1) == int(B.mix(np.uint64(n ^ s)))


def test_hash_sees_every_byte_and_position():
    rng = np.random.default_rng(1)
    cache = rng.integers(0, 65536, size=(3, 64, 576), dtype=np.uint16)
    h0 = B.block_hash(cache, 0)
    raw = cache.view(np.uint8).reshape(3, -1)
    for pos in [0, 1, 7, 8, raw.shape[1] - 1] + rng.integers(0, raw.shape[1], size=300).tolist():
        c = cache.copy()
        c.view(np.uint8).reshape(3, -1)[0, pos] ^= np.uint8(1 << int(rng.integers(0, 8)))
        assert B.block_hash(c, 0) != h0
    c = cache.copy()
    w = c.view(np.uint8).reshape(3, -1)[0].view("<u8")
    w[[3, 500]] = w[[500, 3]]                 # same words, other places
    assert w[3] != w[500] and B.block_hash(c, 0) != h0
    cache[2] = cache[0]                       # same content in another block
    assert B.block_hash(cache, 2) == h0


def test_seal_shares_equal_blocks_and_installs_distinct_ones():
    rng = np.random.default_rng(2)
    cache = rng.integers(0, 65536, size=(8, 64, 576), dtype=np.uint16)
    cache[5] = cache[1]
    cache[7] = cache[1]
    cache[6] = cache[3]
    holder, coll = B.seal_all(cache, range(8))
    assert holder == [0, 1, 2, 3, 4, 1, 3, 1]
    assert coll == 0


def test_seal_counts_collisions_with_truncated_hashes():
    """With 3-bit hashes distinct blocks collide; each candidate that matches
    a hash but no installed bytes is installed and counted (brute force)."""
    rng = np.random.default_rng(3)
    cache = rng.integers(0, 65536, size=(40, 64, 576), dtype=np.uint16)
    for a, b in ((10, 2), (20, 2), (33, 15)):
        cache[a] = cache[b]
    holder, coll = B.seal_all(cache, range(40), hash_bits=3)
    hashes = [B.block_hash(cache, i) & 7 for i in range(40)]
    want_holder, want_coll, installed = [], 0, []
    for i in range(40):
        eq = [j for j in installed if np.array_equal(cache[j], cache[i])]
        if eq:
            want_holder.append(eq[0])
            continue
        if any(hashes[j] == hashes[i] for j in installed):
            want_coll += 1
        installed.append(i)
        want_holder.append(i)
    assert holder == want_holder and coll == want_coll and coll > 0


def test_workload_cache_blocks_hash_distinctly():
    wl = W.tiny()
    hs = [B.block_hash(wl.kv_cache, b) for b in range(wl.kv_cache.shape[0])]
    assert len(set(hs)) == len(hs)
