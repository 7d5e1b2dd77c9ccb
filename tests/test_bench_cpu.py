"""bench.py's CPU-baseline sample on a small chunk workload (no GPU): the
sample fits its budget by taking whole sequences while they fit, else evenly
spaced query positions of one sequence; the bytes it reports are the step's
algorithmic bytes scaled to the rows computed."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import Spec, generate  # noqa: E402


def _chunk_workload():
    spec = Spec("bench_sample", batch=3, num_q_heads=8, num_kv_heads=2, head_dim=64,
                block_size=16, dtype="bf16", seq_lens=(40, 100, 75), max_len=112,
                num_queries=12, pool_factor=1.3, seed=991)
    w = generate(spec, device="cpu")
    kc, vc = bench.host_caches(w, w.key_cache, w.value_cache)
    return w, kc, vc


def test_whole_sequences_when_they_fit():
    w, kc, vc = _chunk_workload()
    seqs, queries = bench.bounded_sample(w, kc, vc, budget_s=60.0)
    assert queries is None and seqs == [0, 1, 2]


def test_query_positions_when_a_sequence_does_not_fit(monkeypatch):
    w, kc, vc = _chunk_workload()
    seqs, queries = bench.bounded_sample(w, kc, vc, budget_s=1e-9)
    assert seqs == [0] and queries == [(w.spec.num_queries - 1) // 2]  # one row, the middle
    # with the probe timed at 1 s per row, a 4.5 s budget takes 4 evenly spaced
    # rows of sequence 0, first and last included
    monkeypatch.setattr(bench, "oracle_baseline",
                        lambda *a, **k: {"seconds_per_sample": 1.0})
    seqs, queries = bench.bounded_sample(w, kc, vc, budget_s=4.5)
    assert seqs == [0] and queries == [0, 4, 7, 11]


def test_sample_bytes_scale_with_the_rows_computed():
    w, kc, vc = _chunk_workload()
    s = w.spec
    full = bench.oracle_baseline(w, kc, vc, 0.0, seq_subset=[1])
    part = bench.oracle_baseline(w, kc, vc, 0.0, seq_subset=[1], queries=[0, 5, 11])
    # bytes = K/V of the read range x share of queries + q and out of the rows
    L, st = int(w.seq_lens[1]), int(w.starts[1])
    kv = (L - st) * s.num_kv_heads * 2 * s.head_dim * 2
    rows = lambda nq: nq * s.num_q_heads * s.head_dim * 2 * 2
    assert np.isclose(full["value"] * full["seconds_per_sample"] * 1e9, kv + rows(12))
    assert np.isclose(part["value"] * part["seconds_per_sample"] * 1e9, kv * 3 / 12 + rows(3))
    assert "3 of 12 queries" in part["sample"]
