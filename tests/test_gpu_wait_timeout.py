"""Bounded waits made to run out on purpose (pa_selftest_bounded_wait).

Every wait in the library's kernels gives up after a limit of device wall
time, records PA_DEVERR_TIMEOUT and lets the kernel return. The self-test
kernel runs the same bounded-wait code on an mbarrier phase that nothing
completes and on a device word that nothing writes; checked here, through
the C ABI:
  * both waits give up after the limit (and not much later), the error word
    carries PA_DEVERR_TIMEOUT, and reading it clears it;
  * the context stays usable: a decode step launched afterwards matches the
    fp64 oracle and leaves the error word clear;
  * on a side stream, with no duration output, the bit still arrives.
Nothing here faults, traps or hangs the GPU: the waits end by themselves.
"""
import pytest
import torch

from conftest import have_gpu
from pa_testutil import assert_close, out_f64, run_both
from workloads import CONFIGS

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not have_gpu(), reason="needs a GPU")]

PA_DEVERR_TIMEOUT = 8


@pytest.mark.parametrize("limit_us", [50, 2000])
def test_unsatisfiable_waits_give_up_after_their_limit(limit_us, pa_lib):
    assert pa_lib.check_device_error() == 0
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    pa_lib.selftest_bounded_wait(limit_us, elapsed)
    assert pa_lib.check_device_error() == PA_DEVERR_TIMEOUT
    assert pa_lib.check_device_error() == 0  # the read cleared it
    for what, ns in zip(("mbarrier phase", "device flag"), elapsed.cpu().tolist()):
        # gave up no earlier than the limit, and within 20 ms of it
        assert limit_us * 1000 <= ns < limit_us * 1000 + 20_000_000, (what, ns)


def test_context_usable_after_the_waits_gave_up(pa_lib):
    pa_lib.selftest_bounded_wait(1000)
    assert pa_lib.check_device_error() == PA_DEVERR_TIMEOUT
    sides = run_both(CONFIGS["llama8b"].with_(name="after_timeout", batch=6,
                                              seq_lens=(1, 17, 300, 2048, 999, 64)))
    assert_close(out_f64(sides.out), sides.ref, what="decode after the self-test")
    assert pa_lib.check_device_error() == 0


def test_side_stream_without_duration_output(pa_lib):
    s = torch.cuda.Stream()
    pa_lib.selftest_bounded_wait(100, None, s)
    assert pa_lib.check_device_error(s) == PA_DEVERR_TIMEOUT
    assert pa_lib.check_device_error(s) == 0
