"""GPU parity of the chunked-query path (pa_prefill_chunk) against the fp64
oracle's causal multi-query decode, through the C ABI.

Each case writes the chunk's B * T new K/V rows with the write path, then
attends every sequence's T queries causally over the paged cache; the write
must match the oracle bit for bit and the outputs within max-abs
1e-2 + 2^-8 |ref| (bf16 rounding of large outputs of short spans) and
mean-abs 1e-3. The cases cover one and several column groups (T * G above
16, with padding columns), GQA groups 1 to 16, head dims 64 to 256, block
sizes 16 and 32, sliding windows, FP8 caches, sequences shorter than the
chunk (rows of zeros for queries before the sequence) and empty sequences.
"""
import numpy as np
import pytest
import torch

from conftest import have_gpu
from workloads.configs import Spec
from pa_testutil import CHUNK_REL_TOL, assert_caches_equal, assert_close, out_f64, run_chunk

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

SMALL_LENS = (0, 1, 2, 3, 7, 16, 17, 31, 33, 64, 100, 129, 250, 300, 5, 48)

CASES = [
    # T, Hq, Hkv, D, bs, W, dtype, fp8
    (2, 8, 2, 128, 16, 0, "bf16", False),     # 8 columns: one n-tile
    (4, 8, 2, 128, 16, 0, "bf16", False),     # 16 columns: two n-tiles
    (5, 8, 2, 128, 16, 0, "f16", False),      # 20 columns: two groups, padding
    (3, 16, 2, 64, 32, 40, "f16", False),     # 24 columns, window, bs 32
    (16, 16, 2, 128, 16, 100, "bf16", False), # 128 columns: eight groups
    (7, 2, 2, 256, 16, 0, "bf16", False),     # G = 1: 7 columns, D = 256
    (3, 32, 2, 128, 16, 0, "bf16", False),    # G = 16: three groups
    (4, 8, 2, 128, 16, 0, "bf16", True),      # FP8 cache, bf16 q
    (6, 4, 2, 256, 32, 50, "f16", True),      # FP8 cache, f16 q, window
]


def _spec(T, Hq, Hkv, D, bs, W, dt, fp8, lens=SMALL_LENS, seed=2671, **kw):
    return Spec(f"chunk_T{T}", batch=len(lens), num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                block_size=bs, dtype=dt, kv_fp8=fp8, window=W, seq_lens=tuple(lens),
                max_len=max(lens) + 2 * bs, num_queries=T, pool_factor=1.3, seed=seed, **kw)


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_G{c[1] // c[2]}_D{c[3]}_bs{c[4]}_W{c[5]}_{c[6]}"
                                              f"{'_fp8' if c[7] else ''}" for c in CASES])
def test_chunk_parity(case, pa_lib):
    sides = run_chunk(_spec(*case))
    assert_caches_equal(sides, "chunk write path")
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=str(case), rel=CHUNK_REL_TOL)
    T = case[0]
    for b, L in enumerate(sides.w.seq_lens):
        for t in range(T):
            if L - T + t < 0:            # query before the sequence: zeros
                assert (got[b, t] == 0).all()
    assert pa_lib.check_device_error() == 0


def test_single_query_chunk_equals_decode_bit_for_bit(pa_lib):
    spec = _spec(1, 32, 8, 128, 16, 0, "bf16", False, lens=tuple(range(1, 400, 13)))
    pa_lib.set_decode_tuning(pool_permille=-1)     # fixed summation order
    try:
        a = run_chunk(spec).out
        b = run_chunk(spec, use_chunk_entry=False).out
    finally:
        pa_lib.set_decode_tuning()
    assert torch.equal(a.squeeze(1), b)


@pytest.mark.parametrize("tuning", [(8, 1, 500, 1), (0, 1, 1000, 1), (3, 2, -1, 0)])
def test_chunk_under_tuning_layouts(tuning, pa_lib):
    """Few CTAs, one-tile pieces and all-pool splits: many partials per pair,
    several merge groups per column."""
    pa_lib.set_decode_tuning(*tuning)
    try:
        sides = run_chunk(_spec(5, 8, 2, 128, 16, 30, "bf16", False,
                                lens=(900, 3, 0, 2000, 64, 17, 1500, 5), seed=2672))
    finally:
        pa_lib.set_decode_tuning()
    assert_close(out_f64(sides.out), sides.ref, what=f"tuning {tuning}", rel=CHUNK_REL_TOL)
    assert pa_lib.check_device_error() == 0


def _sample_triples(rng, B, T, Hq, n):
    return np.stack([rng.integers(0, B, n), rng.integers(0, T, n), rng.integers(0, Hq, n)], 1)


@pytest.mark.parametrize("name,T,lens,W", [
    ("verify_llama8b", 4, ("uniform", 512, 4096), 0),     # 4 drafted tokens per sequence
    ("prefill_chunk512", 512, ("uniform", 512, 8192), 0), # chunked prefill
    ("prefill_chunk256_window", 256, ("uniform", 256, 12000), 4096),
])
def test_chunk_workloads_sampled(name, T, lens, W, pa_lib):
    B = 64 if T <= 4 else 8
    spec = Spec(name, batch=B, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                dtype="bf16", window=W, len_dist=lens, num_queries=T, pool_factor=1.2,
                seed=2673 + T)
    rng = np.random.default_rng(5)
    tr = _sample_triples(rng, B, T, 32, 512)
    sides = run_chunk(spec, triples=tr)
    assert pa_lib.check_device_error() == 0
    assert_caches_equal(sides, name)
    got = out_f64(sides.out)
    assert np.isfinite(got).all()
    assert_close(got[tuple(tr.T)], sides.ref[tuple(tr.T)], what=name, rel=CHUNK_REL_TOL)


FORCED = [
    # T, Hq, Hkv, D, bs, W, dtype, fp8, lens
    (1, 8, 2, 128, 16, 0, "bf16", False, SMALL_LENS),          # 4 rows of 128: padding
    (33, 8, 2, 128, 16, 0, "bf16", False, SMALL_LENS),         # 132 rows: a second tile of 4
    (40, 32, 8, 128, 16, 100, "bf16", False, SMALL_LENS),      # window cuts tiles, G = 4
    (64, 16, 2, 128, 32, 0, "f16", False, (0, 1, 63, 64, 65, 700, 129, 3000)),  # bs 32, L < T
    (7, 32, 2, 128, 16, 24, "f16", False, (5, 6, 7, 8, 40, 300)),  # G = 16, short window
    (128, 8, 8, 128, 16, 0, "bf16", False, (128, 127, 1000, 2047)),  # G = 1
    (48, 16, 4, 128, 64, 0, "bf16", False, (0, 47, 48, 49, 300, 1000)),  # bs 64
    (40, 16, 4, 128, 128, 70, "f16", True, (5, 40, 41, 129, 500, 2000)),  # bs 128, e4m3, window
    (20, 8, 2, 128, 16, 30, "bf16", True, SMALL_LENS),        # e4m3, one row tile (80 rows)
    (40, 32, 8, 128, 16, 100, "bf16", True, SMALL_LENS),       # e4m3 cache, window
    (64, 16, 2, 128, 32, 0, "f16", True, (0, 1, 63, 64, 65, 700, 129, 3000)),  # e4m3, f16 q
]


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
@pytest.mark.parametrize("case", FORCED, ids=[f"T{c[0]}_G{c[1] // c[2]}_bs{c[4]}_W{c[5]}_{c[6]}"
                                                f"{'_fp8' if c[7] else ''}" for c in FORCED])
def test_chunk_kernels_forced(case, path, pa_lib):
    """Each chunk kernel, forced, against the oracle on the same inputs."""
    *shape, lens = case
    pa_lib.set_prefill_path(path)
    try:
        sides = run_chunk(_spec(*shape, lens=lens, seed=2690 + path))
    finally:
        pa_lib.set_prefill_path(0)
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=f"{case[:7]} path {path}", rel=CHUNK_REL_TOL)
    if path == 2:   # no atomics or dynamic split: a rerun is bit-identical
        import paged_kv_cache_267_gb300 as pa
        s = sides.w.spec
        pa_lib.set_prefill_path(path)
        try:
            q4 = sides.w.q if sides.w.q.dim() == 4 else sides.w.q.unsqueeze(1)
            again = pa.prefill_chunk(q4, sides.kc, sides.vc,
                                     torch.from_numpy(sides.w.block_tables).cuda(),
                                     torch.from_numpy(sides.w.seq_lens).cuda(),
                                     num_kv_heads=s.num_kv_heads, scale=s.softmax_scale,
                                     block_size=s.block_size, window=s.window,
                                     kv_dtype="fp8" if s.kv_fp8 else "auto",
                                     k_scale=sides.w.k_scale, v_scale=sides.w.v_scale)
        finally:
            pa_lib.set_prefill_path(0)
        assert torch.equal(again.view(torch.int16), sides.out.view(torch.int16))
    T = case[0]
    for b, L in enumerate(sides.w.seq_lens):
        for t in range(T):
            if L - T + t < 0:
                assert (got[b, t] == 0).all()
    assert pa_lib.check_device_error() == 0


@pytest.mark.parametrize("B", [60, 300], ids=["ranked", "index_order"])
def test_tensor_memory_chunk_large_batch(B, pa_lib):
    """The tensor-memory kernel hands its units out heaviest first when the
    batch has at most 64 sequences (ranked by every CTA, equal weights
    by index) and in sequence order beyond that: both against the oracle, on
    batches of few distinct lengths (many equal weights), some shorter than
    the chunk (their early queries attend to nothing)."""
    rng = np.random.default_rng(B)
    lens = tuple(int(x) for x in rng.choice([1, 7, 40, 100, 100, 100, 180], size=B))
    pa_lib.set_prefill_path(2)
    try:
        sides = run_chunk(_spec(8, 32, 8, 128, 16, 0, "bf16", False, lens=lens, seed=2700 + B))
    finally:
        pa_lib.set_prefill_path(0)
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=f"B{B}", rel=CHUNK_REL_TOL)
    for b, L in enumerate(sides.w.seq_lens):
        for t in range(8):
            if L - 8 + t < 0:
                assert (got[b, t] == 0).all()
    assert pa_lib.check_device_error() == 0


SCALES = [
    # scale, cache: a negative scale (the tensor-memory kernel flips Q's sign
    # to take the row max on raw scores), zero (uniform weights; masked
    # scores must still give exactly zero), and a large one (scores spread
    # over about +-30 log2 units: many reference-max moves and O rescales)
    (-0.0884, "bf16"), (0.0, "bf16"), (1.0, "bf16"), (-0.0884, "fp8"), (1.0, "fp8"),
]


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
@pytest.mark.parametrize("scale,cache", SCALES, ids=[f"s{c[0]}_{c[1]}" for c in SCALES])
def test_chunk_softmax_scale_range(scale, cache, path, pa_lib):
    """Both chunk kernels against the oracle for softmax scales other than
    1/sqrt(D), with a window and a tile boundary inside the chunk."""
    fp8 = cache == "fp8"
    spec = _spec(40, 32, 8, 128, 16, 100, "bf16", fp8, lens=(0, 39, 40, 41, 200, 300, 129, 77),
                 seed=2700 + path, scale=scale)
    pa_lib.set_prefill_path(path)
    try:
        sides = run_chunk(spec)
    finally:
        pa_lib.set_prefill_path(0)
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=f"scale {scale} {cache} path {path}", rel=CHUNK_REL_TOL)
    assert pa_lib.check_device_error() == 0


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
def test_chunk_bad_block_id_and_long_seq_are_flagged_not_faulted(path, pa_lib):
    """Device-side data errors in a chunk call: a block id outside the pool and
    a length beyond the table set their error bits; the kernels substitute a
    safe block / clamp the length instead of reading out of bounds."""
    import paged_kv_cache_267_gb300 as pa
    from workloads import generate
    w = generate(_spec(40, 8, 2, 128, 16, 0, "bf16", False, lens=(120, 300, 77)), device="cuda")
    s = w.spec
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    kw = dict(num_kv_heads=2, scale=s.softmax_scale, block_size=16)
    assert pa_lib.check_device_error() == 0
    pa_lib.set_prefill_path(path)
    try:
        for bad in (w.num_blocks + 5, -3):
            bt_bad = bt.clone()
            bt_bad[1, 2] = bad
            pa.prefill_chunk(w.q, w.key_cache, w.value_cache, bt_bad, sl, **kw)
            assert pa_lib.check_device_error() & pa_lib.DEVERR_BLOCK_ID
            assert pa_lib.check_device_error() == 0
        sl_bad = sl.clone()
        sl_bad[0] = w.max_blocks * 16 + 9
        pa.prefill_chunk(w.q, w.key_cache, w.value_cache, bt, sl_bad, **kw)
        assert pa_lib.check_device_error() & pa_lib.DEVERR_SEQ_LEN
    finally:
        pa_lib.set_prefill_path(0)


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
def test_chunk_step_replays_from_a_cuda_graph(path, pa_lib):
    """The chunk step (write path + pa_prefill_chunk) captured in one CUDA
    graph and replayed gives the eager result (the persistent kernel with the
    dynamic pool off, the tensor-memory kernel as it is: both repeat bit for
    bit)."""
    import paged_kv_cache_267_gb300 as pa
    from workloads import generate
    w = generate(_spec(48, 8, 2, 128, 16, 0, "bf16", False, lens=(300, 60, 1000)), device="cuda")
    s = w.spec
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    kw = dict(num_kv_heads=2, scale=s.softmax_scale, block_size=16)
    out = torch.empty_like(w.q)
    stream = torch.cuda.Stream()
    pa_lib.set_prefill_path(path)
    pa_lib.set_decode_tuning(pool_permille=-1)
    try:
        def step():
            pa.reshape_and_cache(w.k_new, w.v_new, w.key_cache, w.value_cache, w.slot_new)
            pa.prefill_chunk(w.q, w.key_cache, w.value_cache, bt, sl, out=out, **kw)
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        eager = out.clone()
        out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    finally:
        pa_lib.set_prefill_path(0)
        pa_lib.set_decode_tuning()
    assert pa_lib.check_device_error() == 0


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
def test_maximum_chunk(path, pa_lib):
    """T = 4096 queries (the library's limit) on one sequence of 4200
    positions: 16384 (query, head) rows per KV head; sampled rows against the
    oracle."""
    spec = _spec(4096, 8, 2, 128, 16, 0, "bf16", False, lens=(4200,), seed=2701)
    rng = np.random.default_rng(9)
    tr = np.stack([np.zeros(256, np.int64), rng.integers(0, 4096, 256), rng.integers(0, 8, 256)], 1)
    pa_lib.set_prefill_path(path)
    try:
        sides = run_chunk(spec, triples=tr)
    finally:
        pa_lib.set_prefill_path(0)
    assert pa_lib.check_device_error() == 0
    idx = tuple(tr.T)
    got = out_f64(sides.out)
    assert np.isfinite(got).all()
    assert_close(got[idx], sides.ref[idx], what=f"T=4096 path {path}", rel=CHUNK_REL_TOL)


@pytest.mark.parametrize("T,fp8", [(5, False), (3, True)], ids=["T5_bf16", "T3_fp8"])
def test_chunk_half_warp_merge_with_padded_groups(T, fp8, pa_lib):
    # 64 sequences x 8 KV heads x two column groups of 16 (T * G = 20 or 12
    # columns, the rest padding) = 16384 or 8192 merge columns, more than the
    # merge grid's warps: narrow columns take half a warp each, padding
    # columns none
    rng = np.random.default_rng(7000 + T)
    lens = tuple(int(x) for x in rng.integers(T, 600, size=64))
    sides = run_chunk(_spec(T, 32, 8, 128, 16, 0, "bf16", fp8, lens=lens, seed=7100 + T))
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=f"half-warp merge T={T}", rel=CHUNK_REL_TOL)
    assert pa_lib.check_device_error() == 0
