"""The allocation-free decode entry point (pa_decode_noalloc).

It serves callers that cannot allocate device memory while decoding, such as
code running inside a memory pool that owns the whole GPU. Its output must
match the ordinary pa_decode on the same inputs, on consecutive calls that
share its built-in scratch array, and it must refuse steps that do not fit in
that array. This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from conftest import have_gpu
from pa_testutil import assert_close, out_f64
from workloads import generate
from workloads.configs import Spec

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]


def _inputs(**kw):
    base = dict(name="noalloc", batch=12, num_q_heads=16, num_kv_heads=4, head_dim=128,
                block_size=16, dtype="bf16", seq_lens=(0, 1, 17, 300, 2048, 5000, 64, 999,
                                                        33, 4096, 15, 700),
                pool_factor=1.3, new_tokens=False, seed=31337)
    base.update(kw)
    if "seq_lens" in kw:
        base["batch"] = len(kw["seq_lens"])
    w = generate(Spec(**base), device="cuda")
    bt = torch.from_numpy(w.block_tables).cuda()
    sl = torch.from_numpy(w.seq_lens).cuda()
    return w, bt, sl


def test_noalloc_matches_decode_on_consecutive_calls(pa_lib):
    results = []
    for case in (dict(), dict(window=700, block_size=32, num_q_heads=32, num_kv_heads=8)):
        w, bt, sl = _inputs(**case)
        s = w.spec
        kw = dict(num_kv_heads=s.num_kv_heads, scale=s.softmax_scale, block_size=s.block_size,
                  window=s.window)
        ref = pa_lib.decode(w.q, w.key_cache, w.value_cache, bt, sl, **kw)
        for _ in range(2):  # two calls in a row share the scratch array
            out = torch.full_like(w.q, float("nan"))
            pa_lib.decode_noalloc(w.q, w.key_cache, w.value_cache, bt, sl, out=out, **kw)
            torch.cuda.synchronize()
            assert_close(out_f64(out), out_f64(ref), what=f"noalloc vs decode {case}")
            results.append(out)
        assert pa_lib.check_device_error() == 0
    assert len(results) == 4


def test_noalloc_rejects_steps_beyond_its_scratch(pa_lib):
    # G = 16 with head_dim 256 needs far more partial storage than 32 MiB
    w, bt, sl = _inputs(num_q_heads=16, num_kv_heads=1, head_dim=256, seq_lens=(100, 3000))
    out = torch.empty_like(w.q)
    with pytest.raises(pa_lib.PAError) as e:
        pa_lib.decode_noalloc(w.q, w.key_cache, w.value_cache, bt, sl, out=out, num_kv_heads=1,
                              scale=w.spec.softmax_scale, block_size=16)
    assert e.value.status == -6
    assert "needs" in str(e.value) and "bytes" in str(e.value)
