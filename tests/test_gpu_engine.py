"""An engine-shaped flow through the library, checked step by step against
the oracle: requests sharing a system prompt are admitted with the
allocator's prefix cache, their uncached prompt tokens are prefilled in
chunks (write path + pa_prefill_chunk), then they decode a few tokens
(append + write path + pa_decode); a request admitted after others finish
reuses the cached prefix blocks.

K/V rows are a seeded function of (token id, position), so equal prefixes
give equal rows, as a model's would. The oracle keeps its own copy of the
caches, written by its own write path from the same rows.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import have_gpu
from pa_testutil import CHUNK_REL_TOL, assert_close, out_f64

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

NB, BS, HKV, G, D = 256, 16, 2, 4, 128
HQ = HKV * G
VOCAB, MAXPOS = 50, 512
CHUNK = 32


class Model:
    """Seeded K/V rows per (token, position) and queries per (request, position)."""

    def __init__(self, seed):
        g = torch.Generator().manual_seed(seed)
        self.ek = torch.randn(VOCAB, HKV, D, generator=g)
        self.ev = torch.randn(VOCAB, HKV, D, generator=g)
        self.pk = 0.5 * torch.randn(MAXPOS, HKV, D, generator=g)
        self.pv = 0.5 * torch.randn(MAXPOS, HKV, D, generator=g)
        self.g = g

    def kv(self, tokens, positions):
        t = torch.as_tensor(tokens, dtype=torch.long)
        p = torch.as_tensor(positions, dtype=torch.long)
        return ((self.ek[t] + self.pk[p]).to(torch.bfloat16),
                (self.ev[t] + self.pv[p]).to(torch.bfloat16))

    def q(self, n):
        return torch.randn(n, HQ, D, generator=self.g).to(torch.bfloat16)


class Caches:
    """The device caches and the oracle's own host copy, kept in step."""

    def __init__(self, pa):
        shape = (NB, HKV, BS, D)
        self.pa = pa
        self.kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        self.kr = self.kc.cpu().view(torch.int16).numpy().view(np.uint16).copy()
        self.vr = self.vc.cpu().view(torch.int16).numpy().view(np.uint16).copy()

    def write(self, k, v, slots):
        s = torch.as_tensor(slots, dtype=torch.int64)
        oracle.reshape_and_cache(k, v, self.kr, self.vr, s.numpy(), "bf16", "bf16", 1.0, 1.0)
        self.pa.reshape_and_cache(k.cuda(), v.cuda(), self.kc, self.vc, s.cuda())


def slots_of(table, positions):
    return [table[p // BS] * BS + p % BS for p in positions]


def test_prefix_cached_chunked_prefill_then_decode(pa_lib):
    pa = pa_lib
    rng = np.random.default_rng(11)
    model = Model(12)
    caches = Caches(pa)
    alloc = pa.BlockAllocator(NB, BS, seed=13)
    system = list(rng.integers(0, VOCAB, 3 * BS))             # three full shared blocks
    prompts = [system + list(rng.integers(0, VOCAB, n)) for n in (21, 70, 5)]
    scale = D ** -0.5
    kw = dict(num_kv_heads=HKV, scale=scale, block_size=BS)

    def check(out, q4, lens, tables, what):
        ref = oracle.decode_multi(q4, caches.kr, caches.vr, tables, np.asarray(lens, np.int32),
                                  num_kv_heads=HKV, scale=scale, block_size=BS,
                                  q_dtype="bf16", cache_dtype="bf16")
        assert_close(out_f64(out), ref, what=what, rel=CHUNK_REL_TOL)

    def admit(tokens):
        seq, n_cached = alloc.add_cached(tokens)
        table = alloc.table(seq)
        done = n_cached
        while done < len(tokens):                     # chunked prefill of the rest
            T = min(CHUNK, len(tokens) - done)
            pos = list(range(done, done + T))
            k, v = model.kv(tokens[done:done + T], pos)
            caches.write(k, v, slots_of(table, pos))
            q4 = model.q(T).unsqueeze(0)
            bt = np.full((1, len(table) + 1), -1, np.int32)
            bt[0, :len(table)] = table
            out = pa.prefill_chunk(q4.cuda(), caches.kc, caches.vc, torch.from_numpy(bt).cuda(),
                                   torch.tensor([done + T], dtype=torch.int32, device="cuda"),
                                   **kw)
            torch.cuda.synchronize()
            check(out, q4, [done + T], bt, f"prefill {seq} [{done}, {done + T})")
            done += T
        return seq, n_cached

    seqs = []
    for i, p in enumerate(prompts):
        seq, n_cached = admit(p)
        assert n_cached == (0 if i == 0 else 3 * BS)   # the system prompt is cached after the first
        seqs.append(seq)
    toks = {s: list(p) for s, p in zip(seqs, prompts)}

    for step in range(3):                              # batched decode steps
        new_k, new_v, slots = [], [], []
        for s in seqs:
            src, dst = alloc.append(s, 1)
            assert (src, dst) == (-1, -1)              # last blocks are private: no copy
            L = alloc.seq_len(s)
            t = int(rng.integers(0, VOCAB))
            toks[s].append(t)
            k, v = model.kv([t], [L - 1])
            new_k.append(k)
            new_v.append(v)
            slots += slots_of(alloc.table(s), [L - 1])
        caches.write(torch.cat(new_k), torch.cat(new_v), slots)
        tables, lens = alloc.fill_tables(seqs, 16)
        q = model.q(len(seqs))
        out = pa.decode(q.cuda(), caches.kc, caches.vc, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(lens).cuda(), **kw)
        torch.cuda.synchronize()
        check(out.unsqueeze(1), q.unsqueeze(1), lens, tables, f"decode step {step}")

    # the first two finish; once their blocks are reclaimed a new request
    # finds the system prompt still cached through the third
    for s in seqs[:2]:
        alloc.free(s)
    torch.cuda.synchronize()
    alloc.reclaim()
    seq, n_cached = admit(system + list(rng.integers(0, VOCAB, 40)))
    assert n_cached == 3 * BS
    assert all(alloc.refcount(b) == 2 for b in alloc.table(seq)[:3])
    assert pa.check_device_error() == 0
