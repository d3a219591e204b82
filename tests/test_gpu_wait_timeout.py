"""Bounded device waits run out, report, and leave the GPU usable.

Every wait in the kernels (mbarrier phases, the fused step's grid barrier,
the in-launch merge's counter polls) gives up after a time limit, records
bit 4 in the device error word and leaves.  Here a one-thread self-test kernel
of the library waits, with those same bounded waits, on an mbarrier that
never receives its arrival (no copy is in flight on it) and on a counter that
nothing increments, under a 2 ms limit.  Nothing else runs meanwhile, so the
timeout cannot strand an asynchronous copy, and the wait cannot hang: it ends
at its limit.
"""
import time

import pytest
import torch

import paged_kv_cache_185_gb300 as wllm
from paged_kv_cache_185_gb300 import workloads
from tests.gpu_common import assert_attention_close, gpu_step, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_cache_185_gb300 import build
    build.build()
    wllm.load_library()
    yield
    assert wllm.device_errors() == 0


def test_bounded_waits_give_up_and_report():
    assert wllm.device_errors() == 0
    t0 = time.perf_counter()
    wllm.selftest_wait_timeout(2_000_000)  # synchronises; raises unless both waits reported a timeout
    assert time.perf_counter() - t0 < 10.0
    assert wllm.device_errors() == 16, "bit 4: a bounded wait timed out"
    assert wllm.device_errors() == 0, "reading the word clears it"


def test_decode_after_a_timeout_is_correct():
    """The self-test leaves the persistent scheduler's claim counter set, as a
    launch that gave up would; wllm_device_errors() must restore it, or the
    next decode would skip units."""
    wllm.selftest_wait_timeout(1_000_000)
    assert wllm.device_errors() == 16
    case = workloads.custom_case("after_timeout", lens=[3000, 1, 700, 4100, 64], num_q_heads=28,
                                 num_kv_heads=4, head_dim=128, block_size=16, dtype=torch.bfloat16, seed=71)
    got, _, _ = gpu_step(case)
    ref, _, _ = oracle_step(case)
    assert_attention_close(got, ref, case.dtype, "decode after a timed-out wait")


def test_selftest_rejects_bad_limits():
    for limit in (0, 2_000_000_000):
        with pytest.raises(wllm.WllmError) as e:
            wllm.selftest_wait_timeout(limit)
        assert e.value.status == 1
