"""Seeded random shapes through the decode and both chunk kernels, against
the oracle: GQA groups 1 to 16, 1 to 8 KV heads, block sizes 16 to 1024,
windows from one position up, 16-bit and e4m3 caches, f16 and bf16 queries,
ragged lengths with empty sequences and sequences shorter than the chunk, and
(decode) the worker layouts of the tuning knobs. Each case draws its own
generator from (seed, case index), so a failure names a reproducible case.

Outputs are compared on sampled (sequence, [query,] head) rows; the write
path over the whole cache, bit for bit. A window of one position makes every
output one V row, held to a single rounding (see the window-one edge test);
every other case to the decode bar (chunks: plus 2^-8 |ref|).
"""
import numpy as np
import pytest
import torch

from conftest import have_gpu
from pa_testutil import (CHUNK_REL_TOL, MAX_ABS_TOL, MEAN_ABS_TOL, assert_caches_equal,
                         out_f64, run_both, run_chunk)
from workloads.configs import Spec

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

SEED = 26717
TUNINGS = [(), (8, 1, 500, 1), (0, 1, 1000, 1), (3, 2, -1, 0), (152, 4, 200, 8)]


def _one_rounding(got, ref, dtype):
    u, floor = (2.0 ** -8, 0.0) if dtype == "bf16" else (2.0 ** -11, 2.0 ** -25)
    excess = np.abs(got - ref) - (u * np.abs(ref) * (1 + 1e-4) + floor)
    assert excess.max() <= 0, f"exceeds one rounding by {excess.max():.3e}"


def _chunk_case(i):
    rng = np.random.default_rng([SEED, 1, i])
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    bs = int(rng.choice([16, 32, 64, 128, 256, 1024]))
    T = int(rng.choice([1, 2, 3, 7, 16, 31, 33, 64, 100, 128, 129, 200, 257, 400]))
    fp8 = bool(rng.random() < 0.5)
    dt = str(rng.choice(["bf16", "f16"]))
    W = int(rng.choice([0, 0, 0, 1, 17, 64, 128, 130, 500]))
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.integers(0, 3000, B)]
    lens[int(rng.integers(0, B))] = int(rng.choice([0, 1, max(T - 1, 0), T, T + 1, 128, 129]))
    if max(lens) == 0:
        lens[0] = 1   # an empty pool is rejected: any length would need a block
    spec = Spec(f"random_chunk{i}", batch=B, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                head_dim=128, block_size=bs, dtype=dt, kv_fp8=fp8, window=W,
                seq_lens=tuple(lens), max_len=max(lens) + 2 * bs, num_queries=T,
                pool_factor=1.3, seed=int(rng.integers(0, 1 << 30)))
    triples = np.stack([rng.integers(0, B, 64), rng.integers(0, T, 64),
                        rng.integers(0, G * Hkv, 64)], 1)
    return spec, triples


def _decode_case(i):
    rng = np.random.default_rng([SEED, 2, i])
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    fp8 = bool(rng.random() < 0.4)
    D = int(rng.choice([128, 256] if fp8 else [64, 128, 256]))
    bs = int(rng.choice([16, 32, 64, 128, 256, 1024]))
    dt = str(rng.choice(["bf16", "f16"]))
    W = int(rng.choice([0, 0, 0, 1, 17, 100, 1000]))
    B = int(rng.integers(1, 40))
    lens = [int(x) for x in rng.integers(0, 6000, B)]
    if rng.random() < 0.3:
        lens[0] = int(rng.integers(20000, 60000))
    cap = 40_000_000 // (Hkv * D)   # keeps the oracle's write path to seconds
    while sum(lens) > cap:
        lens = [x // 2 for x in lens]
    if max(lens) == 0:
        lens[0] = 1
    tuning = TUNINGS[int(rng.integers(0, len(TUNINGS)))]
    spec = Spec(f"random_decode{i}", batch=B, num_q_heads=G * Hkv, num_kv_heads=Hkv,
                head_dim=D, block_size=bs, dtype=dt, kv_fp8=fp8, window=W,
                seq_lens=tuple(lens), max_len=max(lens) + 2 * bs, pool_factor=1.3,
                seed=int(rng.integers(0, 1 << 30)))
    pairs = np.stack([rng.integers(0, B, 48), rng.integers(0, G * Hkv, 48)], 1)
    return spec, pairs, tuning


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
@pytest.mark.parametrize("i", range(24))
def test_random_chunk_shapes(i, path, pa_lib):
    spec, triples = _chunk_case(i)
    pa_lib.set_prefill_path(path)
    try:
        sides = run_chunk(spec, triples=triples)
    finally:
        pa_lib.set_prefill_path(0)
    assert pa_lib.check_device_error() == 0
    assert_caches_equal(sides, spec.name)
    got = out_f64(sides.out)
    assert np.isfinite(got).all()
    idx = tuple(triples.T)
    if spec.window == 1:
        _one_rounding(got[idx], sides.ref[idx], spec.dtype)
    else:
        err = np.abs(got[idx] - sides.ref[idx])
        excess = err - (MAX_ABS_TOL + CHUNK_REL_TOL * np.abs(sides.ref[idx]))
        assert excess.max() <= 0, f"{spec}: bound exceeded by {excess.max():.3e}"
        assert err.mean() <= MEAN_ABS_TOL
    for b, L in enumerate(sides.w.seq_lens):   # queries before the sequence: zeros
        t_first = max(0, spec.num_queries - int(L))
        assert (got[b, :t_first] == 0).all()


@pytest.mark.parametrize("i", range(24))
def test_random_decode_shapes(i, pa_lib):
    spec, pairs, tuning = _decode_case(i)
    pa_lib.set_decode_tuning(*tuning)
    try:
        sides = run_both(spec, pairs=pairs)
    finally:
        pa_lib.set_decode_tuning()
    assert pa_lib.check_device_error() == 0
    assert_caches_equal(sides, spec.name)
    got = out_f64(sides.out)
    assert np.isfinite(got).all()
    idx = tuple(pairs.T)
    if spec.window == 1:
        _one_rounding(got[idx], sides.ref[idx], spec.dtype)
    else:
        err = np.abs(got[idx] - sides.ref[idx])
        assert err.max() <= MAX_ABS_TOL, f"{spec}, tuning {tuning}: max {err.max():.3e}"
        assert err.mean() <= MEAN_ABS_TOL, f"{spec}, tuning {tuning}: mean {err.mean():.3e}"
    for b, L in enumerate(sides.w.seq_lens):
        if L == 0:
            assert (got[b] == 0).all()
