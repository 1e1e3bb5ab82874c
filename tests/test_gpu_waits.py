"""Failure detection without a GPU fault: every pipeline wait of the decode
kernel is bounded, and a wait that gives up returns an error status while
the context stays usable.

The wait is made to run out on a barrier that nothing completes (the
library's self-test runs the kernel's own wait routine with a short limit);
no fault, trap or hang is involved.
"""

import pytest

from gpu_common import (assert_parity, device_inputs, gpu_out_f64, gpu_step, host_copy,
                        oracle_step, status)
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


@pytest.mark.parametrize("limit_ms", [2, 50])
def test_wait_on_a_barrier_nothing_completes_gives_up(nsv, limit_ms):
    limit = limit_ms * 1000000
    gave_up, waited = nsv.selftest_bounded_wait(limit)
    assert gave_up == 1
    assert limit <= waited < limit + 500000000, waited


def test_context_stays_usable_after_a_wait_gives_up(nsv):
    gave_up, _ = nsv.selftest_bounded_wait(10000000)
    assert gave_up == 1
    # the self-test leaves the device status word alone
    assert status() == (0, 0)
    wl = W.custom("after_timeout", 91, rows=4, heads=8, kv_heads=2, head_dim=128,
                  block_size=16, max_blocks=40, dtype="bf16", lens=[5, 600, 0, 33],
                  free_frac=0.2, query_len=2)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))
