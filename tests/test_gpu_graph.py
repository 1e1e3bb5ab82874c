"""The serving step under CUDA-graph capture (Day 55: a graph recorded over
an all-padding warm batch computes real steps, because every argument it
holds is a window on storage the real steps write through).

The plan depends on the shape alone and the caller-workspace path neither
allocates nor synchronises, so one captured step can be replayed over any
batch of that shape written into the same buffers.
"""

import numpy as np
import pytest

from gpu_common import assert_parity, gpu_out_f64, oracle_read, oracle_step
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _batches(heads, kv_heads):
    base = dict(rows=6, heads=heads, kv_heads=kv_heads, head_dim=128, block_size=16,
                max_blocks=70, dtype="bf16", num_blocks=400)
    a = W.custom("graph_a", 41, lens=[100, 1, 0, 1100, 333, 17], **base)
    b = W.custom("graph_b", 42, lens=[5, 900, 64, 0, 2, 1024], **base)
    return base, a, b


@pytest.mark.parametrize("heads,kv_heads,consumer", [(8, 8, 1), (16, 4, 2), (16, 4, 4)])
def test_graph_recorded_on_padding_replays_real_steps(heads, kv_heads, consumer):
    """The CUDA-core and tensor-core consumers, and the TMEM form; the tensor
    forms hold their TMA tensor maps (over the pool, which the graph's replays
    keep) in the captured launch."""
    import torch
    from paged_kv_decode_nsv_gb300 import nsv
    base, wa, wb = _batches(heads, kv_heads)
    R, H, D, NB = base["rows"], base["heads"], base["head_dim"], base["num_blocks"]
    HKV = base["kv_heads"]
    dev = "cuda"
    # persistent buffers: the pool (the cache) and the step's inputs
    _, kp, vp, _, _ = W.device_values(wa, dev, value_seed=7)
    q = torch.zeros((R, H, D), dtype=torch.bfloat16, device=dev)
    kn = torch.zeros((R, HKV, D), dtype=torch.bfloat16, device=dev)
    vn = torch.zeros_like(kn)
    slots = torch.full((R,), NB * 16, dtype=torch.int64, device=dev)     # all to the sink
    tables = torch.full((R, base["max_blocks"]), -1, dtype=torch.int32, device=dev)
    ctx = torch.zeros((R,), dtype=torch.int32, device=dev)                # all padding
    out = torch.full((R, H, D), 3.0, dtype=torch.bfloat16, device=dev)
    shape = nsv.shape_of(q, kp, tables)
    # the default plan for the first two; the TMEM form is chosen explicitly
    plan = nsv.plan_split(shape) if consumer < 4 else nsv.plan_custom(shape, consumer=consumer)
    assert plan.consumer == consumer
    ws = nsv.workspace_for(plan)
    scale = wa.scale

    def step():
        nsv.decode_step(q, kn, vn, slots, kp, vp, tables, ctx, scale, out, workspace=ws,
                        plan=plan)

    k0, v0 = kp.clone(), vp.clone()
    step()                                     # first call on the device: set-up, uncaptured
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0, "a warm batch reads nothing"
    assert torch.equal(kp[:-1], k0[:-1]) and torch.equal(vp[:-1], v0[:-1])

    for wl, seed in ((wa, 101), (wb, 102)):
        hq, hkp, hvp, hkn, hvn = W.host_values(wl, value_seed=seed)
        host = dict(q=hq, k_pool=W.to_numpy(kp), v_pool=W.to_numpy(vp), k_new=hkn, v_new=hvn)
        for t, a in ((q, hq), (kn, hkn), (vn, hvn)):
            t.copy_(torch.from_numpy(a).view(torch.bfloat16))
        slots.copy_(torch.from_numpy(wl.write_slots))
        tables.copy_(torch.from_numpy(wl.block_tables))
        ctx.copy_(torch.from_numpy(wl.context_lens))
        g.replay()
        torch.cuda.synchronize()
        st, _ = nsv.device_status(clear=True)
        assert st == 0
        assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))


@pytest.mark.parametrize("heads,kv_heads,consumer", [(8, 8, 1), (16, 4, 4)])
def test_graph_of_the_read_alone_replays_real_batches(heads, kv_heads, consumer):
    """The read alone on a caller workspace (nsv_paged_decode_ws) under
    capture: its counter-zeroing kernel and the read launched dependent on it
    are recorded over an all-padding batch and replayed over two real ones,
    each checked against the oracle's read."""
    import torch
    from paged_kv_decode_nsv_gb300 import nsv
    base, wa, wb = _batches(heads, kv_heads)
    R, H, D = base["rows"], base["heads"], base["head_dim"]
    dev = "cuda"
    _, kp, vp, _, _ = W.device_values(wa, dev, value_seed=9)
    q = torch.zeros((R, H, D), dtype=torch.bfloat16, device=dev)
    tables = torch.full((R, base["max_blocks"]), -1, dtype=torch.int32, device=dev)
    ctx = torch.zeros((R,), dtype=torch.int32, device=dev)                # all padding
    out = torch.full((R, H, D), 3.0, dtype=torch.bfloat16, device=dev)
    shape = nsv.shape_of(q, kp, tables)
    plan = nsv.plan_split(shape) if consumer < 4 else nsv.plan_custom(shape, consumer=consumer)
    assert plan.consumer == consumer
    ws = nsv.workspace_for(plan)
    scale = wa.scale

    def read():
        nsv.paged_decode_ws(q, kp, vp, tables, ctx, scale, out, workspace=ws, plan=plan)

    read()                                     # first call on the device: set-up, uncaptured
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            read()
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0, "a warm batch reads nothing"
    for wl, seed in ((wa, 201), (wb, 202)):
        hq, _, _, _, _ = W.host_values(wl, value_seed=seed)
        host = dict(q=hq, k_pool=W.to_numpy(kp), v_pool=W.to_numpy(vp))
        q.copy_(torch.from_numpy(hq).view(torch.bfloat16))
        tables.copy_(torch.from_numpy(wl.block_tables))
        ctx.copy_(torch.from_numpy(wl.context_lens))
        g.replay()
        torch.cuda.synchronize()
        st, _ = nsv.device_status(clear=True)
        assert st == 0
        assert_parity("bf16", gpu_out_f64(out), oracle_read(wl, host))


def test_library_workspace_refuses_to_grow_under_capture():
    """nsv_paged_decode's library-owned workspace cannot grow inside a capture:
    the call returns NSV_ERR_CAPTURE and launches nothing.  Every row is empty
    and every tensor real, so a launch could not touch memory out of bounds."""
    import ctypes
    import torch
    from paged_kv_decode_nsv_gb300 import nsv
    # 16 query heads per KV head: the largest default workspace of any shape
    # the other tests use, so the library's buffer must grow here
    rows, heads, kv_heads, head_dim, max_blocks = 512, 128, 8, 128, 1024
    q = torch.zeros((rows, heads, head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    pool = torch.zeros((2, kv_heads, 16, head_dim), dtype=torch.bfloat16, device="cuda")
    tables = torch.full((rows, max_blocks), -1, dtype=torch.int32, device="cuda")
    ctx = torch.zeros((rows,), dtype=torch.int32, device="cuda")
    shape = nsv.shape_of(q, pool, tables)
    if nsv.plan_split(shape).workspace_bytes == 0:
        pytest.skip("the default plan of this shape needs no workspace")
    small = torch.zeros(1, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    codes = []
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            small.add_(1.0)
            codes.append(nsv._lib.nsv_paged_decode(
                ctypes.byref(shape), q.data_ptr(), pool.data_ptr(), pool.data_ptr(),
                tables.data_ptr(), ctx.data_ptr(), ctypes.c_float(1.0), out.data_ptr(),
                ctypes.c_void_p(s.cuda_stream)))
    torch.cuda.synchronize()
    assert codes == [-6], "growing the library workspace inside a capture must be refused"
