"""Bounded device waits reach their limit on purpose, without a fault.

Every wait of the verify kernels is bounded; past its limit the kernel
records KDA_STATUS_TMA_TIMEOUT and returns.  kda_selftest_bounded_wait runs the
same wait helpers against an mbarrier that nothing arrives at (a flag that
nothing sets), so the limit is reached; these tests check the status the
host reads, the time the wait took (a limit, not a hang), the abort flag that
ends the pipelined kernel's waits early, and that the context still runs a
verify that matches the oracle afterwards.
"""
import time

import pytest
import torch

import oracle
from linear_attention_speculative_gb300 import workloads as wk
from parity_util import assert_parity, run_kernel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from linear_attention_speculative_gb300 import kda
    kda.lib()


def _timed(mode, limit_ns):
    from linear_attention_speculative_gb300 import kda
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    status, mask = kda.selftest_bounded_wait(mode, limit_ns)
    return status, mask, time.perf_counter() - t0


def test_one_item_wait_gives_up_at_its_limit():
    from linear_attention_speculative_gb300 import kda
    status, mask, dt = _timed(0, 20_000_000)  # 20 ms
    assert status == kda.STATUS_TMA_TIMEOUT and mask == 1
    assert 0.015 < dt < 1.5, dt


def test_abort_flag_ends_the_pipelined_wait_early():
    from linear_attention_speculative_gb300 import kda
    status, mask, dt = _timed(1, 20_000_000)
    assert status == kda.STATUS_TMA_TIMEOUT and mask == 3  # both waits gave up
    assert dt < 1.0, dt  # the flag, not the pipelined wait's own 2 s limit, ended it


def test_pipelined_wait_gives_up_at_its_own_limit():
    from linear_attention_speculative_gb300 import kda
    status, mask, dt = _timed(2, 0)
    assert status == kda.STATUS_TMA_TIMEOUT and mask == 2
    assert 1.9 < dt < 4.0, dt


def test_cluster_roll_time_out_path_ends():
    # every CTA of the cluster arrives on the cluster barrier before its own
    # wait, so the wait on the cluster barrier after giving up ends at once
    from linear_attention_speculative_gb300 import kda
    status, mask, dt = _timed(3, 20_000_000)
    assert status == kda.STATUS_TMA_TIMEOUT and mask == 4
    assert 0.015 < dt < 1.5, dt


def test_context_still_runs_a_verify_afterwards():
    _timed(0, 1_000_000)
    wl = wk.custom(3, 4, 2, 4, 128, 128, seed=61)
    inp = wk.make_inputs(wl)
    ref = oracle.verify(inp, wl.gate)
    out, cs = run_kernel(inp, wl.gate)
    assert_parity(out, cs, ref)
