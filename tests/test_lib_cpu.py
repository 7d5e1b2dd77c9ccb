"""CPU checks of libpa: it builds, loads, exports every symbol include/pa.h
declares, rejects bad arguments on the host before touching a device, and its
host block allocator agrees exactly with the allocator model."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle.alloc_model import BlockAllocatorModel, OutOfBlocks


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported(pa_lib):
    names = declared_functions()
    assert len(names) >= 20
    L = ctypes.CDLL(pa_lib.build.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_version_and_launch_count(pa_lib):
    assert pa_lib.version() == 10000
    assert pa_lib.launch_count() >= 0


def _desc(pa, dtype, shape, data=0x1000):
    d = pa.PaTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    st = 1
    for i in reversed(range(len(shape))):
        d.shape[i] = shape[i]
        d.strides[i] = st
        st *= shape[i]
    return d


def test_host_validation_rejects_bad_arguments_without_a_device(pa_lib):
    pa = pa_lib
    L = pa.lib()
    B, Hq, Hkv, D, NB, bs, MB = 2, 8, 2, 128, 10, 16, 4
    base = 0x10000000

    def call(q=None, out=None, kc=None, vc=None, bt=None, sl=None, hkv=Hkv, bsz=bs, kv=0,
             ks=1.0, vs=1.0):
        q = q or _desc(pa, pa.PA_BF16, (B, Hq, D), base)
        out = out or _desc(pa, pa.PA_BF16, (B, Hq, D), base + 0x100000)
        kc = kc or _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x200000)
        vc = vc or _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x400000)
        bt = bt or _desc(pa, pa.PA_I32, (B, MB), base + 0x600000)
        sl = sl or _desc(pa, pa.PA_I32, (B,), base + 0x700000)
        args = [ctypes.byref(x) for x in (out, q, kc, vc, bt, sl)]
        return L.pa_decode(*args, hkv, 0.1, bsz, 0, kv, ks, vs, None)

    assert call(hkv=3) == -1                                      # num_kv_heads mismatch
    assert call(bsz=32) == -1                                     # block_size mismatch
    assert call(q=_desc(pa, pa.PA_BF16, (B, 12, D), base),
                out=_desc(pa, pa.PA_BF16, (B, 12, D), base + 0x100000),
                kc=_desc(pa, pa.PA_BF16, (NB, 5, bs, D), base + 0x200000),
                vc=_desc(pa, pa.PA_BF16, (NB, 5, bs, D), base + 0x400000), hkv=5) == -1
    assert call(q=_desc(pa, pa.PA_BF16, (B, 40, D), base),
                out=_desc(pa, pa.PA_BF16, (B, 40, D), base + 0x100000)) == -2   # G = 20
    assert call(q=_desc(pa, pa.PA_BF16, (B, Hq, 96), base),
                out=_desc(pa, pa.PA_BF16, (B, Hq, 96), base + 0x100000),
                kc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, 96), base + 0x200000),
                vc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, 96), base + 0x400000)) == -2
    assert call(out=_desc(pa, pa.PA_BF16, (B, Hq, D), base)) == -1    # out aliases q
    assert call(kv=2) == -1                                        # cache not e4m3
    assert call(kc=_desc(pa, pa.PA_FP8_E4M3, (NB, Hkv, bs, D), base + 0x200000),
                vc=_desc(pa, pa.PA_FP8_E4M3, (NB, Hkv, bs, D), base + 0x400000), kv=2,
                ks=0.0) == -1                                      # bad scale
    assert call(kc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x200002)) == -3  # misaligned
    bad_bs = _desc(pa, pa.PA_BF16, (NB, Hkv, 24, D), base + 0x200000)
    assert call(kc=bad_bs, vc=_desc(pa, pa.PA_BF16, (NB, Hkv, 24, D), base + 0x400000),
                bsz=24) == -2
    assert call(bt=_desc(pa, pa.PA_I64, (B, MB), base + 0x600000)) == -1
    assert L.pa_decode(None, None, None, None, None, None, 2, 0.1, 16, 0, 0, 1.0, 1.0, None) == -1
    assert "null" in pa.last_error()
    # write path
    k = _desc(pa, pa.PA_F16, (4, Hkv, D), base)
    v = _desc(pa, pa.PA_F16, (4, Hkv, D), base + 0x10000)
    kc = _desc(pa, pa.PA_F16, (NB, Hkv, bs, D), base + 0x200000)
    vc = _desc(pa, pa.PA_F16, (NB, Hkv, bs, D), base + 0x400000)
    sm = _desc(pa, pa.PA_I32, (4,), base + 0x600000)
    assert L.pa_reshape_and_cache(*[ctypes.byref(x) for x in (k, v, kc, vc, sm)], 0, 1.0, 1.0,
                                  None) == -1                      # slot_mapping must be int64
    sm64 = _desc(pa, pa.PA_I64, (4,), base + 0x600000)
    assert L.pa_reshape_and_cache(*[ctypes.byref(x) for x in (k, v, kc, vc, sm64)], 2, 1.0, 1.0,
                                  None) == -1                      # fp8 requested, f16 cache
    assert pa.lib().pa_set_decode_tuning(-1, 0, 0, 0) == -1
    assert pa.lib().pa_set_decode_tuning(0, 0, 0, -2) == -1
    assert pa.lib().pa_set_decode_tuning(0, 0, 1001, 0) == -1
    assert pa.lib().pa_profile_events(ctypes.c_void_p(1), None) == -1


def test_empty_inputs_with_zero_strides_are_accepted(pa_lib):
    """A write of zero rows and a decode of an empty batch are no-ops, whatever
    strides the empty tensors carry (torch gives some empty views stride 0):
    both return before touching a device."""
    pa = pa_lib
    L = pa.lib()
    Hkv, Hq, D, NB, bs, MB = 2, 8, 128, 10, 16, 4
    base = 0x10000000

    def zero_strides(d):
        for i in range(d.ndim):
            d.strides[i] = 0
        return d

    k = zero_strides(_desc(pa, pa.PA_BF16, (0, Hkv, D), base))
    v = zero_strides(_desc(pa, pa.PA_BF16, (0, Hkv, D), base + 0x10000))
    kc = _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x200000)
    vc = _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x400000)
    sm = zero_strides(_desc(pa, pa.PA_I64, (0,), base + 0x600000))
    assert L.pa_reshape_and_cache(*[ctypes.byref(x) for x in (k, v, kc, vc, sm)], 0, 1.0, 1.0,
                                  None) == 0, pa.last_error()
    q = zero_strides(_desc(pa, pa.PA_BF16, (0, Hq, D), base))
    out = zero_strides(_desc(pa, pa.PA_BF16, (0, Hq, D), base + 0x100000))
    bt = zero_strides(_desc(pa, pa.PA_I32, (0, MB), base + 0x600000))
    sl = zero_strides(_desc(pa, pa.PA_I32, (0,), base + 0x700000))
    args = [ctypes.byref(x) for x in (out, q, kc, vc, bt, sl)]
    assert L.pa_decode(*args, Hkv, 0.1, bs, 0, 0, 1.0, 1.0, None) == 0, pa.last_error()
    # a non-empty tensor with a wrong stride is still rejected
    sm_bad = _desc(pa, pa.PA_I64, (3,), base + 0x600000)
    sm_bad.strides[0] = 2
    k3 = _desc(pa, pa.PA_BF16, (3, Hkv, D), base)
    v3 = _desc(pa, pa.PA_BF16, (3, Hkv, D), base + 0x10000)
    assert L.pa_reshape_and_cache(*[ctypes.byref(x) for x in (k3, v3, kc, vc, sm_bad)], 0, 1.0,
                                  1.0, None) == -3


EXTREMES = [0, 1, 2, 3, 7, 16, 24, 64, 128, 256, 1024, 4096, 4097, 2**31 - 1, 2**31, 2**40,
            2**53 + 1, 2**62, 2**63 - 1]


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="host-only: descriptors point at made-up addresses")
def test_validation_survives_mutated_descriptors(pa_lib):
    """Valid-looking argument sets with one to three fields set to extreme or
    wrong values (extents and strides up to 2^63 - 1, bad dtypes and ranks,
    misaligned or null data, bad head counts, block sizes and scales): every
    entry point returns a documented status without crashing, and succeeds
    only for calls with nothing to do (no device work is possible here)."""
    pa = pa_lib
    L = pa.lib()
    rnd = random.Random(2671)
    base = 0x10000000
    codes = {0, -1, -2, -3, -4, -6}

    def fresh(entry):
        B, T, Hq, Hkv, D, NB, bs, MB = 2, 3, 8, 2, 128, 10, 16, 4
        if entry == "reshape":
            return dict(k=_desc(pa, pa.PA_BF16, (5, Hkv, D), base),
                        v=_desc(pa, pa.PA_BF16, (5, Hkv, D), base + 0x100000),
                        kc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x200000),
                        vc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x400000),
                        sm=_desc(pa, pa.PA_I64, (5,), base + 0x600000)), \
                dict(kv=0, ks=1.0, vs=1.0)
        qs = (B, T, Hq, D) if entry == "chunk" else (B, Hq, D)
        return dict(out=_desc(pa, pa.PA_BF16, qs, base + 0x100000),
                    q=_desc(pa, pa.PA_BF16, qs, base),
                    kc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x200000),
                    vc=_desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 0x400000),
                    bt=_desc(pa, pa.PA_I32, (B, MB), base + 0x600000),
                    sl=_desc(pa, pa.PA_I32, (B,), base + 0x700000)), \
            dict(hkv=Hkv, scale=0.1, bs=bs, window=0, kv=0, ks=1.0, vs=1.0)

    def mutate(ts, sc):
        name = rnd.choice(sorted(ts) + ["scalar"])
        if name == "scalar":
            key = rnd.choice(sorted(sc))
            if key in ("scale", "ks", "vs"):
                sc[key] = rnd.choice([0.0, -1.0, float("nan"), float("inf"), 1e38])
            else:
                sc[key] = rnd.choice([-(2**31), -16, -1, 0, 1, 2, 5, 16, 17, 1024, 2048, 2**31 - 1])
            return
        d = ts[name]
        what = rnd.choice(["shape", "stride", "dtype", "ndim", "data"])
        i = rnd.randrange(min(max(d.ndim, 1), len(d.shape)))
        if what == "shape":
            d.shape[i] = rnd.choice(EXTREMES + [-1])
        elif what == "stride":
            d.strides[i] = rnd.choice(EXTREMES + [-1])
        elif what == "dtype":
            d.dtype = rnd.choice([pa.PA_F16, pa.PA_BF16, pa.PA_FP8_E4M3, pa.PA_I32, pa.PA_I64, 9, -1])
        elif what == "ndim":
            d.ndim = rnd.choice([0, 1, 2, 3, 4, 5, -1])
        else:
            d.data = rnd.choice([None, base + 3, base + 8, 2**64 - 16])

    for it in range(4000):
        entry = rnd.choice(["decode", "noalloc", "chunk", "reshape"])
        ts, sc = fresh(entry)
        for _ in range(rnd.randint(1, 3)):
            mutate(ts, sc)
        if entry == "reshape":
            args = [ctypes.byref(ts[n]) for n in ("k", "v", "kc", "vc", "sm")]
            st = L.pa_reshape_and_cache(*args, sc["kv"], sc["ks"], sc["vs"], None)
            nothing = ts["k"].ndim == 3 and (ts["k"].shape[0] == 0 or ts["k"].shape[1] == 0)
        else:
            fn = {"decode": L.pa_decode, "noalloc": L.pa_decode_noalloc,
                  "chunk": L.pa_prefill_chunk}[entry]
            args = [ctypes.byref(ts[n]) for n in ("out", "q", "kc", "vc", "bt", "sl")]
            st = fn(*args, sc["hkv"], sc["scale"], sc["bs"], sc["window"], sc["kv"], sc["ks"],
                    sc["vs"], None)
            nothing = ts["q"].ndim >= 1 and ts["q"].shape[0] == 0
        assert st in codes, (it, entry, st, pa.last_error())
        assert st != 0 or nothing, (it, entry, "succeeded with work to do")


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="host-only: descriptors point at made-up addresses")
@pytest.mark.parametrize("name", ["tiny", "llama8b", "long_skew", "prefix_window", "fp8",
                                  "verify4_llama8b", "prefill_chunk512", "prefill_chunk512_fp8"])
def test_named_workload_shapes_pass_host_validation(name, pa_lib):
    """The argument sets of every named workload, with a pool of 1.2x the
    blocks of all sequences at the longest length, pass host validation: with
    no device here, each call stops at the device query (PA_ERR_CUDA), not at
    a size or layout check. Guards the validation's limits against rejecting
    the shapes the library is built for."""
    from workloads.configs import CONFIGS
    pa = pa_lib
    L = pa.lib()
    s = CONFIGS[name]
    longest = max([s.max_len or 0, s.len_dist[2], *s.long_seqs])
    MB = -(-longest // s.block_size) + 2
    NB = int(1.2 * s.batch * MB) + 1
    B, T, Hq, Hkv, D, bs = s.batch, s.num_queries, s.num_q_heads, s.num_kv_heads, s.head_dim, \
        s.block_size
    cdt = pa.PA_FP8_E4M3 if s.kv_fp8 else pa.PA_BF16
    kv = 2 if s.kv_fp8 else 0
    qs = (B, T, Hq, D) if T > 1 else (B, Hq, D)
    at = iter(range(1, 100))
    addr = lambda: next(at) << 40
    ts = [_desc(pa, pa.PA_BF16, qs, addr()), _desc(pa, pa.PA_BF16, qs, addr()),
          _desc(pa, cdt, (NB, Hkv, bs, D), addr()), _desc(pa, cdt, (NB, Hkv, bs, D), addr()),
          _desc(pa, pa.PA_I32, (B, MB), addr()), _desc(pa, pa.PA_I32, (B,), addr())]
    fn = L.pa_prefill_chunk if T > 1 else L.pa_decode
    st = fn(*[ctypes.byref(t) for t in ts], Hkv, D ** -0.5, bs, s.window, kv, 0.01, 0.01, None)
    assert st == -4, pa.last_error()
    rows = B * T
    k = _desc(pa, pa.PA_BF16, (rows, Hkv, D), addr())
    v = _desc(pa, pa.PA_BF16, (rows, Hkv, D), addr())
    sm = _desc(pa, pa.PA_I64, (rows,), addr())
    st = L.pa_reshape_and_cache(*[ctypes.byref(x) for x in (k, v, ts[2], ts[3], sm)], kv, 0.01,
                                0.01, None)
    assert st == -4, pa.last_error()
    n = ctypes.c_size_t(0)
    st = (L.pa_prefill_chunk_workspace_size(B, T, Hq, Hkv, D, ctypes.byref(n)) if T > 1
          else L.pa_decode_workspace_size(B, Hq, Hkv, D, ctypes.byref(n)))
    assert st == -4, pa.last_error()


def _model_vs_lib(pa, seed):
    rnd = random.Random(seed)
    bs = rnd.choice([1, 8, 16, 32])
    nb = rnd.randint(0, 150)
    m = BlockAllocatorModel(nb, bs, seed=seed * 7 + 1)
    a = pa.BlockAllocator(nb, bs, seed=seed * 7 + 1)
    for _ in range(500):
        op = rnd.random()
        sids = sorted(m.seqs)
        if op < 0.3 or not sids:
            n = rnd.randint(0, 4 * bs)
            try:
                sm = m.add(n)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    a.add(n)
                continue
            assert a.add(n) == sm
        elif op < 0.45:
            src = rnd.choice(sids)
            assert a.fork(src) == m.fork(src)
        elif op < 0.75:
            sid, n = rnd.choice(sids), rnd.randint(0, 3 * bs)
            try:
                pm = m.append(sid, n)
            except OutOfBlocks:
                with pytest.raises(pa.OutOfBlocks):
                    a.append(sid, n)
                continue
            assert a.append(sid, n) == pm
        elif op < 0.85:
            sid = rnd.choice(sids)
            m.free_seq(sid)
            a.free(sid)
        elif op < 0.95:
            sid, W = rnd.choice(sids), rnd.randint(-1, 4 * bs)
            assert a.trim_window(sid, W) == m.trim_window(sid, W)
        else:
            assert a.reclaim() == m.reclaim()
        for sid in m.seqs:
            assert a.table(sid) == m.table(sid)
            assert a.seq_len(sid) == m.seq_len(sid)
        assert [a.refcount(b) for b in range(nb)] == m.ref
        assert a.num_free() == m.num_free() and a.num_pending() == m.num_pending()
    if m.seqs:
        ids = sorted(m.seqs)
        mb = max(len(m.table(s)) for s in ids) + 2
        tables, lens = a.fill_tables(ids, mb)
        for i, s in enumerate(ids):
            t = m.table(s)
            assert list(tables[i, :len(t)]) == t and (tables[i, len(t):] == -1).all()
            assert lens[i] == m.seq_len(s)


@pytest.mark.parametrize("seed", range(12))
def test_allocator_matches_model_exactly(seed, pa_lib):
    _model_vs_lib(pa_lib, seed)


def test_allocator_errors(pa_lib):
    a = pa_lib.BlockAllocator(4, 16, seed=0)
    with pytest.raises(pa_lib.PAError) as e:
        a.free(99)
    assert e.value.status == -7
    assert a.refcount(-1) == -1 and a.refcount(4) == -1
    s = a.add(64)
    with pytest.raises(pa_lib.OutOfBlocks):
        a.add(1)
    with pytest.raises(pa_lib.PAError):
        a.fill_tables([s], 2)        # table wider than the matrix
    t, lens = a.fill_tables([s], 4)
    assert sorted(t[0]) == [0, 1, 2, 3] and lens[0] == 64
    # lengths near the int64 limit: no overflow in the block count or the
    # appended length, and no state change
    b = pa_lib.BlockAllocator(4, 16, seed=0)
    with pytest.raises(pa_lib.OutOfBlocks):
        b.add(2**63 - 1)
    s2 = b.add(5)
    with pytest.raises(pa_lib.PAError) as e:
        b.append(s2, 2**63 - 3)
    assert e.value.status == -1
    assert b.seq_len(s2) == 5 and b.num_free() == 3


@pytest.mark.parametrize("seed", range(6))
def test_allocator_prefix_cache_matches_model_exactly(seed, pa_lib):
    rnd = random.Random(100 + seed)
    bs = rnd.choice([1, 4, 16])
    nb = rnd.randint(20, 200)
    m = BlockAllocatorModel(nb, bs, seed=seed)
    a = pa_lib.BlockAllocator(nb, bs, seed=seed)
    prompts = [[rnd.randrange(4) for _ in range(rnd.randint(0, 6 * bs))] for _ in range(5)]
    for _ in range(400):
        op = rnd.random()
        sids = sorted(m.seqs)
        if op < 0.45 or not sids:
            p = list(rnd.choice(prompts)) + [rnd.randrange(4) for _ in range(rnd.randint(0, 2 * bs))]
            try:
                want = m.add_cached(p)
            except OutOfBlocks:
                with pytest.raises(pa_lib.OutOfBlocks):
                    a.add_cached(p)
                continue
            assert a.add_cached(p) == want
        elif op < 0.7:
            sid = rnd.choice(sids)
            m.free_seq(sid)
            a.free(sid)
        elif op < 0.8:
            sid, n = rnd.choice(sids), rnd.randint(1, 2 * bs)
            try:
                want = m.append(sid, n)
            except OutOfBlocks:
                with pytest.raises(pa_lib.OutOfBlocks):
                    a.append(sid, n)
                continue
            assert a.append(sid, n) == want
        elif op < 0.9:
            sid, W = rnd.choice(sids), rnd.randint(1, 3 * bs)
            assert a.trim_window(sid, W) == m.trim_window(sid, W)
        else:
            assert a.reclaim() == m.reclaim()
        for sid in m.seqs:
            assert a.table(sid) == m.table(sid)
        assert [a.refcount(b) for b in range(nb)] == m.ref
        assert a.num_free() == m.num_free() and a.num_pending() == m.num_pending()


def test_prefill_chunk_host_validation(pa_lib):
    pa = pa_lib
    L = pa.lib()
    B, T, Hq, Hkv, D, NB, bs, MB = 2, 3, 8, 2, 128, 10, 16, 4
    base = 0x10000000

    def call(q_shape=(B, T, Hq, D), out_shape=None, sl=None):
        far = 1 << 40                                         # disjoint fake address ranges
        q = _desc(pa, pa.PA_BF16, q_shape, base)
        out = _desc(pa, pa.PA_BF16, out_shape or q_shape, base + far)
        kc = _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 2 * far)
        vc = _desc(pa, pa.PA_BF16, (NB, Hkv, bs, D), base + 3 * far)
        bt = _desc(pa, pa.PA_I32, (q_shape[0], MB), base + 4 * far)
        sl = sl or _desc(pa, pa.PA_I32, (q_shape[0],), base + 5 * far)
        args = [ctypes.byref(x) for x in (out, q, kc, vc, bt, sl)]
        return L.pa_prefill_chunk(*args, Hkv, 0.1, bs, 0, 0, 1.0, 1.0, None)

    assert call(q_shape=(B, Hq, D)) == -1                      # q must be [B, T, Hq, D]
    assert call(out_shape=(B, T + 1, Hq, D)) == -1             # out shape != q shape
    assert call(q_shape=(B, 0, Hq, D)) == -2                   # T = 0
    assert call(q_shape=(B, 4097, Hq, D)) == -2                # T beyond the chunk limit
    assert call(q_shape=(B, T, 9, D)) == -1                    # Hq not a multiple of Hkv
    assert call(q_shape=(4096, 128, Hq, D)) == -2              # merge counters exceeded
    assert "too large" in pa.last_error()
    n = ctypes.c_size_t(0)
    assert L.pa_prefill_chunk_workspace_size(4, 0, Hq, Hkv, D, ctypes.byref(n)) == -2


def test_bounded_wait_selftest_validates_its_arguments(pa_lib):
    # rejected on the host, before any device call (status PA_ERR_INVALID_ARG)
    L = pa_lib.lib()
    for limit_us in (0, 1_000_001, 2**32 - 1):
        assert L.pa_selftest_bounded_wait(limit_us, None, None) == -1
        assert "limit_us" in pa_lib.last_error()
    assert L.pa_selftest_bounded_wait(1000, 0x10000004, None) == -1  # not 8-byte aligned
    assert "aligned" in pa_lib.last_error()
