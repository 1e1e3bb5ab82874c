"""Parity at the documented limits and degenerate shapes."""

import numpy as np
import pytest

import oracle
from gpu_common import (assert_parity, default_plan, device_inputs, gpu_out_f64, gpu_step,
                        host_copy, oracle_step, oracle_step_sampled, status)
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


def test_largest_batch(nsv):
    """8192 rows (the row-table limit): the plan gives up a stage to fit the
    per-CTA row tables; sampled rows against the oracle."""
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 97, size=8192)
    wl = W.custom("rows8192", 81, rows=8192, heads=8, kv_heads=8, head_dim=128,
                  block_size=16, max_blocks=8, dtype="bf16", lens=lens)
    inp = device_inputs(wl)
    plan = default_plan(inp)
    assert plan.smem_bytes <= 227 * 1024
    rows = [0, 1, 4095, 8191] + list(map(int, rng.choice(8192, 8, replace=False)))
    ref = oracle_step_sampled(wl, inp, rows)
    out = gpu_step(wl, inp, plan=plan)
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)
    assert_parity("bf16", gpu_out_f64(out)[rows], ref)
    zero = np.nonzero(wl.context_lens == 0)[0]
    assert np.all(gpu_out_f64(out)[zero] == 0.0)


def test_one_very_long_row(nsv):
    """One 131,072-token row among short ones: it is cut over every CTA and
    merged from about 150 pieces."""
    lens = [131072, 5, 0, 300]
    wl = W.custom("longrow", 82, rows=4, heads=8, kv_heads=8, head_dim=128, block_size=16,
                  max_blocks=8192, dtype="bf16", lens=lens)
    inp = device_inputs(wl)
    ref = oracle_step_sampled(wl, inp, [0, 1, 3])
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out)[[0, 1, 3]], ref)


@pytest.mark.parametrize("qlen,heads,kv_heads", [(32, 8, 8), (15, 4, 4), (2, 16, 1)])
def test_query_len_limits(nsv, qlen, heads, kv_heads):
    lens = [qlen, 3 * qlen + 1, 0, 700, 1]
    wl = W.custom("qlen_limit", 83, rows=len(lens), heads=heads, kv_heads=kv_heads,
                  head_dim=128, block_size=16, max_blocks=48, dtype="bf16", lens=lens,
                  free_frac=0.2, query_len=qlen)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))


def test_empty_batch(nsv):
    import torch
    q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((2, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    tables = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    ctx = torch.zeros((0,), dtype=torch.int32, device="cuda")
    slots = torch.zeros((0,), dtype=torch.int64, device="cuda")
    new = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    nsv.decode_step(q, new, new, slots, pool, pool, tables, ctx, 1.0, out)
    nsv.paged_decode(q, pool, pool, tables, ctx, 1.0, out)
    torch.cuda.synchronize()
    assert status()[0] == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_head_dim_64_grouped_multi_query(nsv, dtype):
    lens = [3, 257, 0, 1024, 40]
    wl = W.custom("d64", 84, rows=len(lens), heads=16, kv_heads=4, head_dim=64, block_size=16,
                  max_blocks=70, dtype=dtype, lens=lens, free_frac=0.2, query_len=3)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity(dtype, gpu_out_f64(out), oracle_step(wl, host))


def _occupancy_shapes():
    base = dict(rows=256, head_dim=128, max_blocks=512, num_blocks=70000)
    for dt in (0, 1):
        for heads, kv, ql in [(32, 32, 1), (32, 8, 1), (32, 32, 4), (32, 8, 8), (128, 8, 1),
                              (16, 16, 17), (8, 8, 3), (64, 8, 8), (64, 1, 1)]:
            for d in (64, 128):
                yield dict(base, num_heads=heads, num_kv_heads=kv, query_len=ql, dtype=dt,
                           head_dim=d)


def test_every_plan_is_resident_in_one_wave(nsv):
    """The planner sizes the persistent grid to num_sms x ctas_per_sm; the
    device's occupancy calculator must agree that that many CTAs of the
    plan's kernel fit on one SM at once, for every consumer form it offers."""
    checked = 0
    for kw in _occupancy_shapes():
        shape = nsv.make_shape(**kw)
        for extra in (dict(), dict(consumer=1), dict(consumer=2), dict(consumer=3), dict(consumer=4),
                      dict(consumer=1, vectors_per_warp=4), dict(kv_heads_per_cta=1),
                      dict(kv_heads_per_cta=2, ctas_per_sm=2)):
            try:
                plan = nsv.plan_custom(shape, **extra)
            except nsv.NsvError:
                continue          # not offered for this shape
            resident = nsv.plan_resident_ctas(shape, plan)
            # The calculator answers one CTA per SM for a kernel that
            # allocates tensor memory; the TMEM form's plans hold to its
            # columns instead (two CTAs of 256 columns run side by side).
            want = 1 if plan.consumer == nsv.CONSUMER_TENSOR_TMEM else plan.ctas_per_sm
            assert resident >= want, (kw, extra, plan.as_dict(), resident)
            checked += 1
    assert checked > 100
