"""Pins for the allocator model (the oracle of the host block allocator).

SplitMix64 is pinned to its published reference outputs; the rest is pinned by
invariants that any correct ref-counted block pool satisfies, checked after
every step of long random operation sequences.
"""
import random

import pytest

from oracle.alloc_model import BlockAllocatorModel, OutOfBlocks, SplitMix64, block_key, fnv1a64


def test_splitmix64_reference_outputs():
    # reference sequence for seed 1234567 (as published with the algorithm's
    # public-domain C reference and Java's SplittableRandom tests)
    r = SplitMix64(1234567)
    assert [r.next() for _ in range(3)] == [6457827717110365317, 3203168211198807973,
                                            9817491932198370423]
    r0 = SplitMix64(0)
    assert r0.next() == 0xE220A8397B1DCDAF


def test_initial_free_list_is_a_seeded_permutation():
    a = BlockAllocatorModel(1000, 16, seed=3)
    b = BlockAllocatorModel(1000, 16, seed=3)
    c = BlockAllocatorModel(1000, 16, seed=4)
    assert sorted(a.free) == list(range(1000))
    assert a.free == b.free and a.free != c.free
    assert a.free != list(range(1000))


def check_invariants(m: BlockAllocatorModel):
    counts = [0] * m.num_blocks
    for s in m.seqs.values():
        assert len(s["blocks"]) == -(-s["len"] // m.block_size)
        for blk in s["blocks"]:
            if blk >= 0:
                counts[blk] += 1
    # every reference held by a live sequence is counted exactly once
    assert counts == m.ref
    live = {i for i in range(m.num_blocks) if m.ref[i] > 0}
    free, pend = set(m.free), set(m.pending)
    assert len(free) == len(m.free) and len(pend) == len(m.pending)
    # free, pending and live blocks partition the pool
    assert not (free & pend) and not (free & live) and not (pend & live)
    assert free | pend | live == set(range(m.num_blocks))


def test_random_operation_sequences_keep_invariants():
    rnd = random.Random(42)
    for trial in range(20):
        bs = rnd.choice([1, 4, 16, 32])
        m = BlockAllocatorModel(rnd.randint(0, 120), bs, seed=trial)
        for _ in range(400):
            op = rnd.random()
            sids = list(m.seqs)
            snapshot = (list(m.free), list(m.pending), list(m.ref),
                        {k: (list(v["blocks"]), v["len"]) for k, v in m.seqs.items()})
            try:
                if op < 0.3 or not sids:
                    n = rnd.randint(0, 5 * bs)
                    before = m.num_free()
                    sid = m.add(n)
                    assert m.num_free() == before - (-(-n // bs))
                    assert all(m.refcount(b) == 1 for b in m.table(sid))
                elif op < 0.45:
                    src = rnd.choice(sids)
                    sid = m.fork(src)
                    assert m.table(sid) == m.table(src)
                elif op < 0.75:
                    sid = rnd.choice(sids)
                    old_tab, old_len = m.table(sid), m.seq_len(sid)
                    shared_last = bool(old_tab) and m.refcount(old_tab[-1]) > 1
                    n = rnd.randint(0, 3 * bs)
                    src, dst = m.append(sid, n)
                    new_tab = m.table(sid)
                    if n > 0 and old_len % bs != 0 and shared_last and old_tab[-1] >= 0:
                        assert src == old_tab[-1] and dst == new_tab[len(old_tab) - 1]
                        assert new_tab[:len(old_tab) - 1] == old_tab[:-1]
                    else:
                        assert (src, dst) == (-1, -1)
                        assert new_tab[:len(old_tab)] == old_tab
                elif op < 0.85:
                    m.free_seq(rnd.choice(sids))
                elif op < 0.95:
                    sid = rnd.choice(sids)
                    W = rnd.randint(1, 4 * bs)
                    before = m.table(sid)
                    n = m.trim_window(sid, W)
                    after = m.table(sid)
                    first_live = max(0, m.seq_len(sid) - W) // bs
                    assert all(b == -1 for b in after[:first_live])
                    assert after[first_live:] == before[first_live:]
                    assert n == sum(1 for b in before[:first_live] if b >= 0)
                else:
                    m.reclaim()
                    assert m.num_pending() == 0
            except OutOfBlocks:
                # rejected operations leave the state unchanged
                assert snapshot == (list(m.free), list(m.pending), list(m.ref),
                                    {k: (list(v["blocks"]), v["len"])
                                     for k, v in m.seqs.items()})
            check_invariants(m)


def test_exhaustion_rejects_and_deferred_reclaim():
    m = BlockAllocatorModel(4, 16, seed=1)
    a = m.add(64)
    with pytest.raises(OutOfBlocks):
        m.add(1)
    m.free_seq(a)
    assert m.num_free() == 0 and m.num_pending() == 4
    with pytest.raises(OutOfBlocks):
        m.add(1)       # freed blocks are not reusable before reclaim
    assert m.reclaim() == 4
    b = m.add(17)
    assert len(m.table(b)) == 2


def test_shared_prefix_fork_and_copy_on_write():
    m = BlockAllocatorModel(64, 16, seed=2)
    p = m.add(40)                    # 3 blocks, last one partial
    forks = [m.fork(p) for _ in range(5)]
    assert all(m.refcount(b) == 6 for b in m.table(p))
    src, dst = m.append(forks[0], 1)
    assert src == m.table(p)[-1] and m.refcount(src) == 5 and m.refcount(dst) == 1
    assert m.table(forks[0])[:2] == m.table(p)[:2]
    # a full last block needs no copy
    q = m.add(32)
    f = m.fork(q)
    assert m.append(f, 5) == (-1, -1)
    assert m.table(f)[:2] == m.table(q)


def test_trim_window_releases_only_blocks_before_the_window():
    m = BlockAllocatorModel(32, 16, seed=5)
    p = m.add(64)                       # 4 full blocks, shared below
    f = m.fork(p)
    m.append(f, 40)                     # f: 104 tokens, 7 blocks
    before = m.table(f)
    assert m.trim_window(f, 50) == 3    # window [54, 104) starts in block 3
    assert m.table(f)[:3] == [-1, -1, -1] and m.table(f)[3:] == before[3:]
    assert all(m.refcount(b) == 1 for b in before[:3])   # still held by p
    assert m.num_pending() == 0
    m.free_seq(p)
    assert m.num_pending() == 3         # blocks 0..2; block 3 is still held by f
    assert m.refcount(before[3]) == 1
    assert m.trim_window(f, 50) == 0    # idempotent
    g = m.fork(f)
    assert m.table(g)[:3] == [-1, -1, -1]


def test_fnv1a64_reference_values():
    # published FNV-1a 64-bit test vectors
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_prefix_cache_reuses_full_blocks_of_the_longest_cached_prefix():
    bs = 16
    m = BlockAllocatorModel(64, bs, seed=9)
    prompt = list(range(100, 140))                # 40 tokens: 2 full blocks + 8
    a, ca = m.add_cached(prompt)
    assert ca == 0
    b, cb = m.add_cached(prompt + [7, 8, 9])
    assert cb == 32 and m.table(b)[:2] == m.table(a)[:2]
    assert m.table(b)[2] != m.table(a)[2]           # partial blocks are never shared
    assert all(m.refcount(x) == 2 for x in m.table(a)[:2])
    c, cc = m.add_cached(prompt[:16] + [0] * 24)    # differs in block 1
    assert cc == 16 and m.table(c)[0] == m.table(a)[0] and m.table(c)[1] != m.table(a)[1]
    # keys chain: block 1 of a different first block is a different key
    assert block_key(block_key(0, prompt[:16]), prompt[16:32]) != \
        block_key(block_key(0, [0] * 16), prompt[16:32])
    check_invariants(m)
    # a cached block waiting for reclaim is taken back out of the pending list
    for sid in (a, b, c):
        m.free_seq(sid)
    assert m.num_pending() > 0
    d, cd = m.add_cached(prompt)
    assert cd == 32 and all(m.refcount(x) == 1 for x in m.table(d)[:2])
    check_invariants(m)
    # reclaim drops the cache entries of the blocks it frees
    m.free_seq(d)
    m.reclaim()
    e, ce = m.add_cached(prompt)
    assert ce == 0 and not set(m.cache.values()) - set(m.table(e))
    check_invariants(m)


def test_prefix_cache_random_sequences_keep_invariants():
    rnd = random.Random(7)
    bs = 4
    m = BlockAllocatorModel(200, bs, seed=3)
    prompts = [[rnd.randrange(5) for _ in range(rnd.randint(0, 40))] for _ in range(6)]
    for step in range(500):
        op = rnd.random()
        sids = sorted(m.seqs)
        try:
            if op < 0.5 or not sids:
                p = list(rnd.choice(prompts))
                p += [rnd.randrange(5) for _ in range(rnd.randint(0, 10))]
                sid, c = m.add_cached(p)
                assert c % bs == 0 and c <= len(p)
            elif op < 0.8:
                m.free_seq(rnd.choice(sids))
            elif op < 0.9:
                m.append(rnd.choice(sids), rnd.randint(1, 9))
            else:
                m.reclaim()
        except OutOfBlocks:
            pass
        check_invariants(m)
        for key, b in m.cache.items():
            assert m.cached[b][0] == key and (m.ref[b] > 0 or b in m.pending)
