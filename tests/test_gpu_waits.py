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
    # the wait that gave up raised the timeout bit, as a decode kernel's would
    assert status() == (nsv.DEV_TIMEOUT, 0)
    assert status() == (0, 0)
    wl = W.custom("after_timeout", 91, rows=4, heads=8, kv_heads=2, head_dim=128,
                  block_size=16, max_blocks=40, dtype="bf16", lens=[5, 600, 0, 33],
                  free_frac=0.2, query_len=2)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))


def test_a_timeout_reaches_the_caller_without_a_device_synchronise(nsv):
    """nsv_status_async copies the status word into caller memory on the
    stream: a pinned host word (read after the stream is synchronised) and a
    device word both carry the timeout bit of a wait that gave up, and the
    clear that follows leaves the next copy at zero."""
    import torch
    stream = torch.cuda.current_stream()
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    dev = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    gave_up, _ = nsv.selftest_bounded_wait(2000000)
    assert gave_up == 1
    nsv.status_async(dev[0:1], clear=False)
    nsv.status_async(host, clear=True)
    nsv.status_async(dev[1:2], clear=False)
    stream.synchronize()
    assert int(host[0]) == nsv.DEV_TIMEOUT
    assert dev.cpu().tolist() == [nsv.DEV_TIMEOUT, 0]
    assert status() == (0, 0)


def test_a_flagged_length_reaches_the_caller_without_a_device_synchronise(nsv):
    """A context length beyond the table's width is read as an empty row and
    flagged; nsv_status_async hands the flag to the caller on the stream."""
    import torch
    wl = W.custom("bad_len", 93, rows=3, heads=4, kv_heads=4, head_dim=64, block_size=16,
                  max_blocks=4, dtype="f32", lens=[10, 64, 3], free_frac=0.2)
    inp = device_inputs(wl)
    inp["context_lens"][1] = 65  # one past max_blocks * 16
    out = gpu_step(wl, inp)
    host = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    nsv.status_async(host, clear=True)
    torch.cuda.current_stream().synchronize()
    assert int(host[0]) == nsv.DEV_BAD_CTX
    assert torch.all(out[1] == 0)
    assert status()[0] == 0
