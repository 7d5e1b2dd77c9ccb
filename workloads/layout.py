"""Physical block layouts of the seeded workloads, as a block allocator
lays them out.

A workload's block tables are the ones the host block allocator produces
for this sequence of requests ("vLLM 0.5 深度解析" §2.1: a pool of physical
blocks and a free list, ceil(n / block_size) blocks per request, popped from
the free list; "vLLM 0.7.2深度解析" §2.1: a shared prefix is one set of
physical blocks referenced by every sequence that shares it):

  * the pool's free list is the block ids 0..NB-1 shuffled by Fisher-Yates
    (Durstenfeld's form: i from NB-1 down to 1, j = x_i mod (i + 1), swap
    ids i and j) with x the outputs of SplitMix64 (Steele, Lea and Flood,
    2014) seeded with the workload seed; a request pops blocks from the end
    of the list;
  * without a shared prefix, sequence b = 0, 1, ... requests its
    ceil(L_b / bs) blocks in turn;
  * with a shared prefix of P tokens (a multiple of bs), one request of P
    tokens comes first; each sequence is a fork of it (one more reference to
    each prefix block) that then appends its L_b - P private tokens (the
    prefix ends on a block boundary, so no copy-on-write); finally the prefix
    request itself is freed, which leaves every prefix block referenced once
    per sequence.

Only the order of block ids comes from here; nothing of the attention
arithmetic. SplitMix64 and the shuffle are written from their published
definitions; the test suite checks that the tables equal those of the
library's allocator and of its reference model under the same requests.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, n: int) -> np.ndarray:
    """The first n outputs of SplitMix64 seeded with `seed` (uint64; the
    arithmetic wraps modulo 2^64)."""
    k = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def shuffled_free_list(num_blocks: int, seed: int) -> list[int]:
    """Block ids 0..num_blocks-1 after the seeded Fisher-Yates shuffle, in
    free-list order (requests pop from the end)."""
    ids = list(range(num_blocks))
    if num_blocks < 2:
        return ids
    x = splitmix64(seed, num_blocks - 1)
    divisors = np.arange(num_blocks, 1, -1, dtype=np.uint64)  # i + 1 for i = NB-1 .. 1
    js = (x % divisors).astype(np.int64)
    for k, i in enumerate(range(num_blocks - 1, 0, -1)):
        j = int(js[k])
        ids[i], ids[j] = ids[j], ids[i]
    return ids


def allocation_order(num_blocks: int, seed: int) -> np.ndarray:
    """Block ids in the order successive requests receive them."""
    return np.asarray(shuffled_free_list(num_blocks, seed)[::-1], dtype=np.int64)


def block_tables(lens: np.ndarray, block_size: int, shared_prefix: int, num_blocks: int,
                 max_blocks: int, seed: int) -> np.ndarray:
    """int32 [B, max_blocks] tables (-1 past each sequence's blocks) for the
    requests described in the module docstring."""
    bs = block_size
    lens = np.asarray(lens, dtype=np.int64)
    B = lens.shape[0]
    order = allocation_order(num_blocks, seed)
    shared = shared_prefix // bs
    nblk = -(-lens // bs)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    cursor = shared
    for b in range(B):
        if lens[b] <= 0:
            continue
        tables[b, :shared] = order[:shared]
        n_priv = int(nblk[b]) - shared
        tables[b, shared:shared + n_priv] = order[cursor:cursor + n_priv]
        cursor += n_priv
    return tables
