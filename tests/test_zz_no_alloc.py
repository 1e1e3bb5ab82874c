"""The allocation-free decode entry point, nsv_paged_decode_noalloc.

Some callers may not allocate device memory at all: an engine that owns the
whole device through its own arena, a plugin hook that only gets pre-bound
buffers, a serving loop that cannot afford the device-wide synchronisation
an allocation can bring.  This entry point serves them by taking the split
path's scratch from a fixed buffer compiled into the library.  These tests
call it through the C ABI and hold it to the existing entry point
(nsv_paged_decode_ws with a caller-owned workspace) within the parity
tolerance, on two calls in a row with different inputs, so that whatever the
first call leaves in the shared buffer cannot leak into the second.

The file is named to be collected last: a run that stops at its first
failure has then already run every other test.
"""

import ctypes

import numpy as np
import pytest

from gpu_common import assert_parity, device_inputs, gpu_out_f64, gpu_read
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 4 << 20  # NSV_NOALLOC_SCRATCH_BYTES in include/nsv.h


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


def _noalloc_call(nsv, wl, inp, out):
    """One call of the new entry point through the C ABI (ctypes)."""
    import torch
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    rc = nsv._lib.nsv_paged_decode_noalloc(
        ctypes.byref(shape), inp["q"].data_ptr(), inp["k_pool"].data_ptr(),
        inp["v_pool"].data_ptr(), inp["block_tables"].data_ptr(),
        inp["context_lens"].data_ptr(), ctypes.c_float(wl.scale), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc


@pytest.mark.parametrize("make", [
    W.uniform_f32,
    lambda: W.custom("noalloc_bf16", 31, rows=10, heads=8, kv_heads=8, head_dim=128,
                     block_size=16, max_blocks=66, dtype="bf16",
                     lens=[1, 0, 17, 256, 1000, 333, 16, 15, 1024, 47], free_frac=0.2),
    lambda: W.custom("noalloc_gqa", 32, rows=10, heads=8, kv_heads=4, head_dim=128,
                     block_size=16, max_blocks=66, dtype="bf16",
                     lens=[1, 0, 17, 256, 1000, 333, 16, 15, 1024, 47], free_frac=0.2),
], ids=["uniform_f32", "ragged_bf16_10rows", "gqa_bf16_tensor_cores"])
def test_noalloc_matches_existing_entry_point_on_two_calls(nsv, make):
    import torch
    wl = make()
    for value_seed in (501, 502):
        inp = device_inputs(wl, value_seed=value_seed)
        shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
        plan = nsv.plan_split(shape)
        assert 0 < plan.workspace_bytes <= SCRATCH_LIMIT, \
            "the case must use scratch memory and fit the static buffer"
        want = gpu_read(wl, inp, plan=plan)          # existing entry point
        got = torch.full_like(inp["q"], float("nan"))
        assert _noalloc_call(nsv, wl, inp, got) == 0
        st, _ = nsv.device_status(clear=True)
        assert st == 0
        assert_parity(wl.dtype, gpu_out_f64(got), gpu_out_f64(want))


def test_noalloc_refuses_shapes_beyond_its_buffer(nsv):
    """A shape whose plan needs more scratch than the fixed buffer is refused
    before anything is launched.  The tensors are real and every row is empty,
    so even a launch could not read or write out of bounds."""
    import torch
    # 16 query heads per KV head: 8 KV heads per CTA carry 128 query vectors,
    # whose partial states make the scratch larger than the buffer.
    rows, heads, kv_heads, head_dim, max_blocks = 256, 128, 8, 128, 512
    q = torch.zeros((rows, heads, head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    pool = torch.zeros((2, kv_heads, 16, head_dim), dtype=torch.bfloat16, device="cuda")
    tables = torch.full((rows, max_blocks), -1, dtype=torch.int32, device="cuda")
    ctx = torch.zeros((rows,), dtype=torch.int32, device="cuda")
    shape = nsv.shape_of(q, pool, tables)
    need = nsv.plan_split(shape).workspace_bytes
    if need <= SCRATCH_LIMIT:
        pytest.skip("no shape of this size needs more than the fixed buffer")
    rc = nsv._lib.nsv_paged_decode_noalloc(
        ctypes.byref(shape), q.data_ptr(), pool.data_ptr(), pool.data_ptr(),
        tables.data_ptr(), ctx.data_ptr(), ctypes.c_float(1.0), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == -8, "a shape needing more scratch than the buffer must get NSV_ERR_WORKSPACE"
