"""Decode with crafted score sequences that drive the online softmax's
reference max (the scaled dot-product attention of "vLLM 0.5 深度解析" §2.3,
computed block by block with a running max and sum).

The decode kernel moves a column's reference max only when a score exceeds
it by more than 8 (log2 units); other tiles compute P against the reference
as it is, so P may reach 2^8. Random inputs rarely move the reference after a
segment's first tile, so these tests build scores that do: q = (c, 0, ..., 0)
and K rows (k_p, 0, ..., 0), with k_p chosen so that the log2-domain score of
position p follows a pattern:
  climb       +1 per token (the reference moves on every tile),
  slow_climb  +0.03 per token (it moves every ~17 tiles; P up to 2^8 between),
  jump        -40, then +60 for three tokens, then 0 (a jump of 100 and a long
              tail of negligible P),
  sawtooth    0 and 7.5 in runs of 40 tokens (never moves after the first
              tile; P up to 2^7.5).
Each runs with the grid cut to two CTAs (long segments per warp) and with
the default grid, on 16-bit and e4m3 caches, against the fp64 oracle; and as
chunks of 8 causal queries on both chunk kernels (the persistent one, whose
columns start from a finite floor, and the tensor-memory one, whose rows keep
a reference max of their own with the same rule).
"""
import numpy as np
import pytest
import torch

from conftest import have_gpu
from pa_testutil import CHUNK_REL_TOL, assert_close, out_f64, run_both, run_chunk
from workloads import CONFIGS

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

LOG2E = 1.4426950408889634
QV = 16.0  # q's one non-zero element

PATTERNS = {
    "climb": lambda p, L: 1.0 * p,
    "slow_climb": lambda p, L: 0.03 * p,
    "jump": lambda p, L: np.where(p < L // 2, -40.0, np.where(p < L // 2 + 3, 60.0, 0.0)),
    "sawtooth": lambda p, L: 7.5 * ((p // 40) % 2),
}


def _mutator(pattern):
    f = PATTERNS[pattern]

    def mutate(w):
        s = w.spec
        bs = s.block_size
        per_unit = s.softmax_scale * LOG2E * QV  # log2-domain score per unit of k[0]
        w.q.zero_()
        w.q[..., 0] = QV
        slots, vals = [], []
        for b in range(s.batch):
            L, st = int(w.seq_lens[b]), int(w.starts[b])
            pos = np.arange(st, L)
            slots.append(w.block_tables[b, pos // bs].astype(np.int64) * bs + pos % bs)
            vals.append(np.asarray(f(pos, L), dtype=np.float64) / per_unit)
        slots, vals = np.concatenate(slots), np.concatenate(vals)
        by_slot = dict(zip(slots.tolist(), vals.tolist()))
        dev, dt = w.q.device, w.q.dtype

        def rows(slot_list):
            r = torch.zeros((len(slot_list), s.num_kv_heads, s.head_dim), dtype=torch.float32)
            r[:, :, 0] = torch.tensor([by_slot[int(x)] for x in slot_list], dtype=torch.float32)[:, None]
            return r.to(dev).to(dt)

        new_slots = w.slot_new.cpu().numpy()
        w.k_new.copy_(rows(new_slots))
        if s.kv_fp8:
            w.k_hist.copy_(rows(w.slot_hist.cpu().numpy()))
            # the scale that maps the largest |k| onto the e4m3 maximum
            amax = float(max(w.k_hist.abs().amax().float().item(),
                             w.k_new.abs().amax().float().item()))
            w.k_scale = amax / 448.0 if amax > 0 else 1.0
        else:
            hist = np.setdiff1d(slots, new_slots)
            kc = w.key_cache.permute(0, 2, 1, 3)  # [NB, bs, Hkv, D] view
            ht = torch.as_tensor(hist, device=dev)
            kc[ht // bs, ht % bs] = rows(hist)
    return mutate


@pytest.mark.parametrize("grid", ["two_ctas", "default"])
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("pattern", list(PATTERNS))
def test_reference_max_under_crafted_score_growth(pattern, fp8, grid, pa_lib):
    spec = CONFIGS["llama8b"].with_(name=f"growth_{pattern}", batch=3,
                                    seq_lens=(700, 2048, 333), kv_fp8=fp8,
                                    seed=700 + list(PATTERNS).index(pattern))
    if grid == "two_ctas":
        pa_lib.set_decode_tuning(max_ctas=2)
    try:
        sides = run_both(spec, mutate=_mutator(pattern))
    finally:
        pa_lib.set_decode_tuning()
    got = out_f64(sides.out)
    assert_close(got, sides.ref, what=f"{pattern} {grid} {'e4m3' if fp8 else 'bf16'}")
    assert pa_lib.check_device_error() == 0


@pytest.mark.parametrize("path", [1, 2], ids=["persistent", "tensor_memory"])
@pytest.mark.parametrize("fp8", [False, True], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("pattern", list(PATTERNS))
def test_chunk_reference_max_under_crafted_score_growth(pattern, fp8, path, pa_lib):
    spec = CONFIGS["llama8b"].with_(name=f"chunk_growth_{pattern}", batch=3, num_queries=8,
                                    seq_lens=(700, 2048, 333), kv_fp8=fp8,
                                    seed=720 + list(PATTERNS).index(pattern))
    pa_lib.set_prefill_path(path)
    if path == 1:
        pa_lib.set_decode_tuning(max_ctas=2)
    try:
        sides = run_chunk(spec, mutate=_mutator(pattern))
    finally:
        pa_lib.set_decode_tuning()
        pa_lib.set_prefill_path(0)
    assert_close(out_f64(sides.out), sides.ref, rel=CHUNK_REL_TOL,
                 what=f"chunk {pattern} path {path} {'e4m3' if fp8 else 'bf16'}")
    assert pa_lib.check_device_error() == 0
