"""The allocation-free decode entry point, nsv_paged_decode_noalloc.

Some callers may not allocate device memory at all: an engine that owns the
whole device through its own arena, a plugin hook that only gets pre-bound
buffers, a serving loop that cannot afford the device-wide synchronisation
an allocation can bring.  This entry point serves them by taking the split
path's scratch from a fixed buffer compiled into the library.  These tests
call it through the C ABI and hold it to the existing entry point
(nsv_paged_decode_ws with a caller-owned workspace and the same default
plan): the same kernel on the same plan must give the same bits.  They do so
on two calls in a row with different inputs, so that whatever the first call
leaves in the shared buffer cannot leak into the second, and check one call
against the oracle directly.

The file is named to be collected last: a run that stops at its first
failure has then already run every other test.
"""

import ctypes

import pytest

from gpu_common import assert_parity, device_inputs, gpu_out_f64, gpu_read, host_copy, oracle_read
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


def _noalloc_raw(nsv, wl, inp, out):
    """One call of the entry point through the raw C ABI (ctypes)."""
    import torch
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    rc = nsv._lib.nsv_paged_decode_noalloc(
        ctypes.byref(shape), inp["q"].data_ptr(), inp["k_pool"].data_ptr(),
        inp["v_pool"].data_ptr(), inp["block_tables"].data_ptr(),
        inp["context_lens"].data_ptr(), ctypes.c_float(wl.scale), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc


def _noalloc_binding(nsv, wl, inp, out):
    """The same call through the Python binding's marshalling."""
    import torch
    nsv.paged_decode_noalloc(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                             inp["context_lens"], wl.scale, out)
    torch.cuda.synchronize()
    return 0


CASES = [
    W.uniform_f32,
    lambda: W.custom("noalloc_bf16", 31, rows=10, heads=8, kv_heads=8, head_dim=128,
                     block_size=16, max_blocks=66, dtype="bf16",
                     lens=[1, 0, 17, 256, 1000, 333, 16, 15, 1024, 47], free_frac=0.2),
    lambda: W.custom("noalloc_gqa", 32, rows=10, heads=8, kv_heads=4, head_dim=128,
                     block_size=16, max_blocks=66, dtype="bf16",
                     lens=[1, 0, 17, 256, 1000, 333, 16, 15, 1024, 47], free_frac=0.2),
]
IDS = ["uniform_f32", "ragged_bf16_10rows", "gqa_bf16_tensor_cores"]


@pytest.mark.parametrize("make", CASES, ids=IDS)
def test_noalloc_matches_existing_entry_point_on_two_calls(nsv, make):
    import torch
    wl = make()
    # the first call through the raw C ABI, the second through the binding
    for value_seed, call in ((501, _noalloc_raw), (502, _noalloc_binding)):
        inp = device_inputs(wl, value_seed=value_seed)
        shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
        plan = nsv.plan_split(shape)
        assert 0 < plan.workspace_bytes <= SCRATCH_LIMIT, \
            "the case must use scratch memory and fit the static buffer"
        want = gpu_read(wl, inp, plan=plan)          # existing entry point, same plan
        got = torch.full_like(inp["q"], float("nan"))
        assert call(nsv, wl, inp, got) == 0
        st, _ = nsv.device_status(clear=True)
        assert st == 0
        assert torch.equal(got, want), "same kernel, same plan: the bits must agree"


@pytest.mark.parametrize("make", CASES[1:2], ids=IDS[1:2])
def test_noalloc_matches_the_oracle(nsv, make):
    import torch
    wl = make()
    inp = device_inputs(wl, value_seed=503)
    host = host_copy(inp)
    got = torch.full_like(inp["q"], float("nan"))
    assert _noalloc_raw(nsv, wl, inp, got) == 0
    assert nsv.device_status(clear=True)[0] == 0
    assert_parity(wl.dtype, gpu_out_f64(got), oracle_read(wl, host))


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
    assert need > SCRATCH_LIMIT, "the refusal case must need more than the buffer (%d)" % need
    rc = nsv._lib.nsv_paged_decode_noalloc(
        ctypes.byref(shape), q.data_ptr(), pool.data_ptr(), pool.data_ptr(),
        tables.data_ptr(), ctx.data_ptr(), ctypes.c_float(1.0), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == -8, "a shape needing more scratch than the buffer must get NSV_ERR_WORKSPACE"
    with pytest.raises(nsv.NsvError):
        nsv.paged_decode_noalloc(q, pool, pool, tables, ctx, 1.0, out)
