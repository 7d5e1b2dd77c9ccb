"""Structure of the seeded workloads: layouts, sharing, poisoning, determinism."""
import numpy as np
import pytest
import torch

from workloads import CONFIGS, generate
from workloads.configs import Spec
from workloads.gen import draw_seq_lens


def _small_prefix_window_spec(**kw):
    base = dict(name="pw_small", batch=6, num_q_heads=4, num_kv_heads=2, head_dim=16,
                block_size=16, dtype="bf16", window=40, shared_prefix=32,
                len_dist=("uniform", 1, 90), seed=77)
    base.update(kw)
    return Spec(**base)


def test_named_configs_match_their_descriptions():
    c = CONFIGS
    assert (c["tiny"].batch, c["tiny"].num_q_heads, c["tiny"].num_kv_heads, c["tiny"].head_dim,
            c["tiny"].block_size, c["tiny"].dtype, c["tiny"].pool_blocks) == \
        (4, 8, 2, 64, 16, "f16", 64)
    assert c["tiny"].softmax_scale == 1 / 8
    assert (c["llama8b"].batch, c["llama8b"].group, c["llama8b"].head_dim) == (64, 4, 128)
    assert (c["long_skew"].batch, c["long_skew"].group, c["long_skew"].block_size) == (8, 8, 32)
    assert c["prefix_window"].window == 4096 and c["prefix_window"].shared_prefix == 2048
    assert c["fp8"].kv_fp8 and c["fp8"].batch == 256
    seeds = [s.seed for s in c.values()]
    assert seeds == [267001, 267002, 267003, 267004, 267005, 267006, 267007, 267008]
    assert c["verify4_llama8b"].num_queries == 4 and c["prefill_chunk512"].num_queries == 512
    assert all(c[n].num_queries == 1 for n in ("tiny", "llama8b", "long_skew", "prefix_window",
                                               "fp8"))


def test_length_distributions():
    rng = np.random.default_rng(0)
    L = draw_seq_lens(CONFIGS["long_skew"], rng)
    assert L[0] == 131072 and ((L[1:] >= 256) & (L[1:] <= 2048)).all()
    L = draw_seq_lens(CONFIGS["fp8"], np.random.default_rng(1))
    assert ((L >= 1024) & (L <= 8192)).all() and 2500 < L.mean() < 4500
    L = draw_seq_lens(CONFIGS["prefix_window"], np.random.default_rng(2))
    assert ((L >= 2048 + 128) & (L <= 2048 + 30000)).all()


def test_tiny_layout_and_poison():
    w = generate(CONFIGS["tiny"])
    assert w.num_blocks == 64 and w.max_blocks == 13
    used = w.block_tables[w.block_tables >= 0]
    assert len(np.unique(used)) == len(used)                # private blocks only
    for b, L in enumerate(w.seq_lens):
        n = -(-int(L) // 16)
        assert (w.block_tables[b, :n] >= 0).all() and (w.block_tables[b, n:] == -1).all()
    kc = w.key_cache
    for b, L in enumerate(w.seq_lens):
        L = int(L)
        for p in range(L):
            row = kc[w.block_tables[b, p // 16], :, p % 16, :]
            assert torch.isnan(row).all() == (p == L - 1)    # new token not written yet
        last = w.block_tables[b, (L - 1) // 16]
        assert torch.isnan(kc[last, :, (L - 1) % 16 + 1:, :]).all()  # tail of the last block
    unused = np.setdiff1d(np.arange(64), used)
    assert torch.isnan(kc[torch.as_tensor(unused)]).all()


def test_shared_prefix_and_window_poison():
    s = _small_prefix_window_spec()
    w = generate(s)
    t = w.block_tables
    assert (t[:, :2] == t[0, :2]).all()                      # prefix blocks shared by all
    priv = t[:, 2:][t[:, 2:] >= 0]
    assert len(np.unique(priv)) == len(priv)
    kc = w.key_cache
    starts = np.maximum(0, w.seq_lens.astype(np.int64) - 40)
    for b, L in enumerate(w.seq_lens):
        for p in range(int(L)):
            row = kc[t[b, p // 16], :, p % 16, :]
            read_by_someone = any(
                starts[c] <= p < w.seq_lens[c] and (p < 32 or c == b) for c in range(s.batch))
            want_nan = (not read_by_someone) or p == L - 1
            assert bool(torch.isnan(row).all()) == want_nan, (b, p)


def test_generation_is_deterministic_and_seeded():
    s = _small_prefix_window_spec()
    a, b = generate(s), generate(s)
    c = generate(s.with_(seed=78))
    assert np.array_equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q, b.q) and torch.equal(a.k_new, b.k_new)
    assert not np.array_equal(a.block_tables, c.block_tables) or not torch.equal(a.q, c.q)


def test_fp8_workload_scales_and_history():
    s = _small_prefix_window_spec(kv_fp8=True, window=0)
    w = generate(s)
    assert w.key_cache is None and w.k_hist is not None
    assert w.k_hist.shape[0] == w.slot_hist.shape[0]
    assert len(torch.unique(w.slot_hist)) == w.slot_hist.shape[0]
    allk = torch.cat([w.k_hist, w.k_new]).float()
    assert w.k_scale == float(allk.abs().amax() / 448.0)
    kc, vc = w.empty_fp8_cache()
    assert kc.dtype == torch.uint8 and (kc == 0x7F).all()


def test_chunk_workload_new_rows_and_union_range():
    T, W = 5, 24
    s = _small_prefix_window_spec(num_queries=T, window=W, shared_prefix=0,
                                  seq_lens=(3, 40, 17, 0, 64, 5), seed=78)
    w = generate(s)
    assert tuple(w.q.shape) == (6, T, 4, 16)
    assert tuple(w.k_new.shape) == (6 * T, 2, 16) and w.slot_new.shape == (6 * T,)
    slots = w.slot_new.numpy()
    for b, L in enumerate(w.seq_lens):
        L = int(L)
        for t in range(T):
            p = L - T + t
            want = -1 if p < 0 else int(w.block_tables[b, p // 16]) * 16 + p % 16
            assert slots[b * T + t] == want
        # the union of the queries' windows starts at the first query's start
        assert w.starts[b] == max(0, L - T + 1 - W)
    # every new slot is poisoned until the write path fills it
    kc = w.key_cache.permute(0, 2, 1, 3).reshape(-1, 2, 16)
    live = slots >= 0
    assert torch.isnan(kc[torch.from_numpy(slots[live])].float()).all()
    # positions read by some query but before the chunk hold history values
    b, L = 4, 64
    p = L - T - 1
    slot = int(w.block_tables[b, p // 16]) * 16 + p % 16
    assert not torch.isnan(kc[slot].float()).any()


# ---- layouts come from allocator requests

def test_layout_splitmix64_published_outputs():
    from workloads.layout import splitmix64
    # Vigna's reference implementation seeded with 1234567 (its first outputs
    # as listed with the public-domain source), and seed 0
    x = splitmix64(1234567, 5)
    assert [int(v) for v in x] == [6457827717110365317, 3203168211198807973,
                                   9817491932198370423, 4593380528125082431,
                                   16408922859458223821]
    assert int(splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


def _model_tables(spec, lens, NB, MB):
    """The same requests on the allocator's reference model (oracle side)."""
    from oracle.alloc_model import BlockAllocatorModel
    m = BlockAllocatorModel(NB, spec.block_size, spec.seed)
    P = spec.shared_prefix
    if P:
        root = m.add(P)
        seqs = []
        for L in lens:
            sq = m.fork(root)
            assert m.append(sq, int(L) - P) == (-1, -1)   # block-aligned prefix: no copy
            seqs.append(sq)
        m.free_seq(root)
    else:
        seqs = [m.add(int(L)) for L in lens]
    t = np.full((len(lens), MB), -1, np.int32)
    for b, sq in enumerate(seqs):
        blocks = m.table(sq)
        t[b, :len(blocks)] = blocks
    return t, m, seqs


def _library_tables(spec, lens, NB, MB):
    """The same requests on the library's C++ allocator (product side)."""
    import paged_kv_cache_267_gb300 as pa
    a = pa.BlockAllocator(NB, spec.block_size, seed=spec.seed)
    P = spec.shared_prefix
    if P:
        root = a.add(P)
        seqs = []
        for L in lens:
            sq = a.fork(root)
            assert a.append(sq, int(L) - P) == (-1, -1)
            seqs.append(sq)
        a.free(root)
    else:
        seqs = [a.add(int(L)) for L in lens]
    t = np.full((len(lens), MB), -1, np.int32)
    for b, sq in enumerate(seqs):
        blocks = a.table(sq)
        t[b, :len(blocks)] = blocks
    return t, a, seqs


@pytest.mark.parametrize("name", list(CONFIGS))
def test_named_layouts_are_the_allocators_tables(name):
    """Every named workload's tables equal those of the allocator model and of
    the library's allocator under the same requests (prefix configs: one
    prefix request forked per sequence, then freed)."""
    from workloads.gen import layout
    s = CONFIGS[name]
    lens, tables, NB, MB = layout(s)
    model_t, m, seqs = _model_tables(s, lens, NB, MB)
    assert np.array_equal(tables, model_t)
    lib_t, a, lseqs = _library_tables(s, lens, NB, MB)
    assert np.array_equal(tables, lib_t)
    if s.shared_prefix:
        # each prefix block referenced once per sequence, in both allocators
        for blk in tables[0, :s.shared_prefix // s.block_size]:
            assert m.refcount(int(blk)) == s.batch
            assert a.refcount(int(blk)) == s.batch
    used = tables[tables >= 0]
    assert len(np.unique(used)) == len(used) or s.shared_prefix
