"""The allocation-free decode entry point (pa_decode_noalloc).

It serves callers that cannot allocate device memory while decoding, such as
code running inside a memory pool that owns the whole GPU, or a runtime whose
allocator must not be re-entered from inside a step. Its scratch is one
32 MiB array built into the library and shared by every call.

Checked here, through the C ABI:
  * its output matches the fp64 oracle (computed on host copies of the
    generator's inputs) and the ordinary pa_decode on the same inputs, on two
    calls in a row that share the built-in array;
  * on each named decode workload it either runs and matches the oracle on
    sampled (sequence, q head) rows and pa_decode everywhere, or refuses the
    step with PA_ERR_WORKSPACE and a message naming more bytes than the array
    holds;
  * it refuses a step whose scratch exceeds the array.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import re

import numpy as np
import pytest
import torch

from conftest import have_gpu
from pa_testutil import assert_close, out_f64, run_both
from workloads import CONFIGS, generate
from workloads.configs import Spec

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

SCRATCH_BYTES = 32 << 20   # size of the library's built-in array


def _spec(**kw):
    base = dict(name="noalloc", batch=12, num_q_heads=16, num_kv_heads=4, head_dim=128,
                block_size=16, dtype="bf16", seq_lens=(0, 1, 17, 300, 2048, 5000, 64, 999,
                                                        33, 4096, 15, 700),
                pool_factor=1.3, seed=31337)
    base.update(kw)
    if "seq_lens" in kw:
        base["batch"] = len(kw["seq_lens"])
    return Spec(**base)


def _noalloc_twice(pa_lib, sides, pairs=None, what=""):
    """Two pa_decode_noalloc calls in a row on the caches the write path
    filled; each must match the oracle (on `pairs`, or every row) and
    pa_decode's output (every row)."""
    w, s = sides.w, sides.w.spec
    kv = "fp8" if s.kv_fp8 else "auto"
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    kw = dict(num_kv_heads=s.num_kv_heads, scale=s.softmax_scale, block_size=s.block_size,
              window=s.window, kv_dtype=kv, k_scale=w.k_scale, v_scale=w.v_scale)
    ref_decode = out_f64(sides.out)
    for call in range(2):  # the second call finds the first one's contents in the array
        out = torch.full_like(w.q, float("nan"))
        pa_lib.decode_noalloc(w.q, sides.kc, sides.vc, bt, sl, out=out, **kw)
        torch.cuda.synchronize()
        got = out_f64(out)
        assert_close(got, sides.ref, pairs=pairs, what=f"{what} call {call}: noalloc vs oracle")
        assert_close(got, ref_decode, what=f"{what} call {call}: noalloc vs pa_decode")
        # L == 0 rows are exact zeros
        for b, L in enumerate(w.seq_lens):
            if L == 0:
                assert (out[b] == 0).all()
    assert pa_lib.check_device_error() == 0


@pytest.mark.parametrize("case", [dict(), dict(window=700, block_size=32, num_q_heads=32,
                                                num_kv_heads=8),
                                  dict(kv_fp8=True, dtype="f16", window=300)],
                         ids=["bf16", "bf16_window_bs32_g4", "fp8_f16_window"])
def test_noalloc_matches_oracle_and_decode_on_consecutive_calls(case, pa_lib):
    sides = run_both(_spec(**case))
    _noalloc_twice(pa_lib, sides, what=str(case))


def _sample_pairs(spec, n_seqs=8):
    """Oracle rows for a named workload: every row when the batch is small,
    else all q heads of evenly spaced sequences, the first and last included
    (skewed batches put their long sequences first)."""
    if spec.batch <= n_seqs:
        return None
    seqs = sorted({int(round(i)) for i in np.linspace(0, spec.batch - 1, n_seqs)})
    return [(b, h) for b in seqs for h in range(spec.num_q_heads)]


@pytest.mark.parametrize("name", ["tiny", "llama8b", "long_skew", "prefix_window", "fp8"])
def test_noalloc_on_named_workloads(name, pa_lib):
    s = CONFIGS[name]
    pairs = _sample_pairs(s)
    sides = run_both(s, pairs=pairs)
    try:
        _noalloc_twice(pa_lib, sides, pairs=pairs, what=name)
    except pa_lib.PAError as e:
        assert e.status == -6, str(e)
        need = int(re.search(r"needs (\d+) bytes", str(e)).group(1))
        assert need > SCRATCH_BYTES, str(e)
        print(f"{name}: refused, needs {need} bytes of scratch")
        return
    print(f"{name}: runs in the built-in scratch")


def test_noalloc_rejects_steps_beyond_its_scratch(pa_lib):
    # G = 16 with head_dim 256 (16.5 KB per partial slot) on 16 sequences of
    # 3000 tokens: enough tiles to keep the decode grid at its full size,
    # whose worker slots alone need more than 32 MiB
    w = generate(_spec(num_q_heads=16, num_kv_heads=1, head_dim=256, seq_lens=(3000,) * 16),
                 device="cuda")
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    out = torch.empty_like(w.q)
    with pytest.raises(pa_lib.PAError) as e:
        pa_lib.decode_noalloc(w.q, w.key_cache, w.value_cache, bt, sl, out=out, num_kv_heads=1,
                              scale=w.spec.softmax_scale, block_size=16)
    assert e.value.status == -6
    need = int(re.search(r"needs (\d+) bytes", str(e.value)).group(1))
    assert need > SCRATCH_BYTES
