"""Plain Python model of the host block allocator (test infrastructure only).

It is the oracle for the C++ allocator exported by the library. Both are
written from the same description, and neither is derived from the other:
  * "vLLM 0.5 深度解析" §2.1: a pool of physical blocks and a free list; a
    request of n tokens takes ceil(n / block_size) blocks, popped from the free
    list; the request's block table lists them in logical order.
  * "vLLM 0.7.2深度解析" §2.1: logical blocks of several sequences may point at
    one physical block (K/V only), and blocks are reclaimed by reference count,
    deferred rather than synchronous.
  * "vLLM 0.7.2深度解析" §5.3: the pool size is a hard cap; a request beyond it
    is rejected, not queued.

Behaviour fixed by this model (the pages leave it open):
  * The initial free list is 0..NB-1 shuffled by Fisher-Yates (Durstenfeld:
    i from NB-1 down to 1, j = next() mod (i + 1), swap) driven by SplitMix64
    seeded with ``seed``. Allocation pops from the end of the free list.
  * ``free`` drops one reference per block; a block whose count reaches zero
    waits in a pending list until ``reclaim`` appends the pending blocks, in
    order, to the free list.
  * ``append`` to a sequence whose last block is partial and shared first
    copies that block (copy-on-write): a fresh block replaces it in this
    sequence only, and the (source, destination) pair is reported so the caller
    can copy the cached rows.
  * Every operation is all-or-nothing: if the free list cannot cover it,
    ``OutOfBlocks`` is raised and the state is unchanged.
  * ``add_cached`` (prefix caching: "vLLM 0.7.2深度解析" §2.1 and §5.2,
    "vLLM 0.5 深度解析" §4.4) allocates a sequence for a list of token ids and
    reuses cached full blocks for its longest cached prefix. Full block i is
    keyed by h_i = FNV-1a-64(le64(h_{i-1}) || le32 tokens of block i), with
    h_{-1} = 0; a hit also needs the stored token ids to be equal. Cached
    blocks are live or waiting in the pending list (a hit there takes the
    block back out of it); ``reclaim`` drops the cache entries of the blocks it
    returns to the free list. New full blocks are registered if their key is
    not yet cached; partial blocks never are.
  * ``trim_window`` ("vLLM 0.7.2深度解析" §2.3: blocks known to lie outside a
    sliding window are skipped for allocation and loading) releases the
    blocks of a sequence that lie wholly before its window start
    ``max(0, len - window)``: each drops one reference and its table entry
    becomes -1 (never read by a windowed decode). Released entries stay -1;
    fork copies them as -1, free skips them.
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1


class OutOfBlocks(Exception):
    pass


class SplitMix64:
    """SplitMix64 (Steele, Lea, Flood 2014; Vigna's public-domain reference)."""

    def __init__(self, seed: int):
        self.state = seed & MASK64

    def next(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & MASK64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        return z ^ (z >> 31)


FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3


def fnv1a64(data: bytes, h: int = FNV64_OFFSET) -> int:
    """FNV-1a, 64-bit (Fowler, Noll, Vo): per byte, xor then multiply."""
    for byte in data:
        h ^= byte
        h = (h * FNV64_PRIME) & MASK64
    return h


def block_key(prev: int, tokens) -> int:
    data = prev.to_bytes(8, "little") + b"".join(
        (int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, block_size: int, seed: int):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool")
        self.num_blocks = num_blocks
        self.block_size = block_size
        ids = list(range(num_blocks))
        rng = SplitMix64(seed)
        for i in range(num_blocks - 1, 0, -1):
            j = rng.next() % (i + 1)
            ids[i], ids[j] = ids[j], ids[i]
        self.free = ids
        self.pending: list[int] = []
        self.ref = [0] * num_blocks
        self.seqs: dict[int, dict] = {}
        self.next_id = 0
        self.cache: dict[int, int] = {}              # key -> block
        self.cached: dict[int, tuple] = {}           # block -> (key, token ids)

    def _blocks_for(self, n_tokens: int) -> int:
        return (n_tokens + self.block_size - 1) // self.block_size

    def _pop(self) -> int:
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def add(self, n_tokens: int) -> int:
        if n_tokens < 0:
            raise ValueError("negative length")
        need = self._blocks_for(n_tokens)
        if need > len(self.free):
            raise OutOfBlocks()
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"blocks": [self._pop() for _ in range(need)], "len": n_tokens}
        return sid

    def fork(self, src: int) -> int:
        s = self.seqs[src]
        for b in s["blocks"]:
            if b >= 0:
                self.ref[b] += 1
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"blocks": list(s["blocks"]), "len": s["len"]}
        return sid

    def append(self, sid: int, n_tokens: int):
        """Grows a sequence; returns (cow_src, cow_dst) or (-1, -1)."""
        if n_tokens < 0:
            raise ValueError("negative length")
        s = self.seqs[sid]
        if n_tokens == 0:
            return (-1, -1)
        partial = s["len"] % self.block_size != 0
        cow = partial and self.ref[s["blocks"][-1]] > 1
        extra = self._blocks_for(s["len"] + n_tokens) - len(s["blocks"])
        if extra + (1 if cow else 0) > len(self.free):
            raise OutOfBlocks()
        pair = (-1, -1)
        if cow:
            old = s["blocks"][-1]
            new = self._pop()
            self.ref[old] -= 1
            s["blocks"][-1] = new
            pair = (old, new)
        for _ in range(extra):
            s["blocks"].append(self._pop())
        s["len"] += n_tokens
        return pair

    def free_seq(self, sid: int) -> None:
        s = self.seqs.pop(sid)
        for b in s["blocks"]:
            if b < 0:
                continue
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.pending.append(b)

    def trim_window(self, sid: int, window: int) -> int:
        """Releases the blocks wholly before the window; returns how many."""
        if window <= 0:
            return 0
        s = self.seqs[sid]
        first_live = max(0, s["len"] - window) // self.block_size
        n = 0
        for i in range(min(first_live, len(s["blocks"]))):
            b = s["blocks"][i]
            if b < 0:
                continue
            s["blocks"][i] = -1
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.pending.append(b)
            n += 1
        return n

    def add_cached(self, tokens) -> tuple[int, int]:
        """New sequence for `tokens`; returns (sequence id, cached tokens)."""
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        bs = self.block_size
        nblk = -(-n // bs)
        nfull = n // bs
        keys, reuse, prev, matching = [], [], 0, True
        for i in range(nfull):
            blk_tokens = tuple(tokens[i * bs:(i + 1) * bs])
            key = block_key(prev, blk_tokens)
            keys.append(key)
            prev = key
            if matching:
                b = self.cache.get(key)
                if b is not None and self.cached[b][1] == blk_tokens:
                    reuse.append(b)
                else:
                    matching = False
        if nblk - len(reuse) > len(self.free):
            raise OutOfBlocks()
        blocks = []
        for b in reuse:
            if self.ref[b] == 0:
                self.pending.remove(b)
            self.ref[b] += 1
            blocks.append(b)
        for i in range(len(reuse), nblk):
            b = self._pop()
            blocks.append(b)
            if i < nfull and keys[i] not in self.cache:
                self.cache[keys[i]] = b
                self.cached[b] = (keys[i], tuple(tokens[i * bs:(i + 1) * bs]))
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = {"blocks": blocks, "len": n}
        return sid, len(reuse) * bs

    def reclaim(self) -> int:
        n = len(self.pending)
        for b in self.pending:
            entry = self.cached.pop(b, None)
            if entry is not None:
                del self.cache[entry[0]]
        self.free.extend(self.pending)
        self.pending = []
        return n

    def table(self, sid: int) -> list[int]:
        return list(self.seqs[sid]["blocks"])

    def seq_len(self, sid: int) -> int:
        return self.seqs[sid]["len"]

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def num_free(self) -> int:
        return len(self.free)

    def num_pending(self) -> int:
        return len(self.pending)
