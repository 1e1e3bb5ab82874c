"""The tensor-core consumer (bf16 mma.sync over TMA-staged, 128-byte-swizzled
K/V tiles) against the oracle: grouped query heads and several query tokens
per row, both head dims, every plan shape the planner allows, the slot-table
gather, and rows whose early query tokens see no position.

Two forms: the block's tokens as the MMA rows and the query vectors as its
columns, 8 per warp (NSV_CONSUMER_TENSOR, the default up to 8 vectors per
KV head); or the vectors as the rows, 16 per warp
(NSV_CONSUMER_TENSOR_VECTOR_ROWS, the default beyond); or tcgen05.mma into
tensor memory with 128 MMA rows shared by 4 KV heads of up to 32 vectors or
2 of up to 64 (NSV_CONSUMER_TENSOR_TMEM), a stage holding up to 4 blocks of a
row.  Every test runs all three, up to
64 vectors per KV head; the TMEM form skips shapes whose KV heads do not
split into its groups."""

import numpy as np
import pytest

import oracle
from gpu_common import (assert_parity, device_inputs, gpu_out_f64, gpu_read, gpu_step,
                        host_copy, oracle_read, oracle_step, status)
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LENS = [40, 513, 0, 2048, 77, 1, 15, 16, 17, 300]


@pytest.fixture(params=[2, 3, 4], ids=["tokens_as_rows", "vectors_as_rows", "tmem"])
def form(request):
    return request.param


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


def _case(heads, kv_heads, qlen, head_dim, lens=LENS, seed=5, free_frac=0.3):
    return W.custom("tc", seed, rows=len(lens), heads=heads, kv_heads=kv_heads,
                    head_dim=head_dim, block_size=16, max_blocks=140, dtype="bf16", lens=lens,
                    free_frac=free_frac, query_len=qlen)


def _plan(nsv, inp, **kw):
    return nsv.plan_custom(nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"]), **kw)


@pytest.mark.parametrize("heads,kv_heads,qlen,head_dim", [
    (32, 8, 1, 128),    # 4 query heads per KV head
    (16, 1, 1, 128),    # 16: a full MMA tile, one KV head
    (8, 8, 2, 128),     # 2 query tokens
    (8, 8, 3, 64),      # odd vector count, head_dim 64
    (12, 3, 4, 64),     # 4 heads x 4 tokens = 16
    (32, 32, 4, 128),   # 32 KV heads in groups of 8
    (6, 2, 5, 128),     # 3 heads x 5 tokens = 15
    (32, 8, 8, 128),    # 4 heads x 8 tokens = 32: two warps per KV head
    (16, 4, 5, 64),     # 20
    (8, 8, 17, 128),    # 17: an odd count, the second warp runs one vector
    (16, 2, 3, 128),    # 24
    (64, 8, 8, 128),    # 8 heads x 8 tokens = 64: four warps per KV head
    (32, 4, 5, 64),     # 40
    (64, 1, 1, 128),    # 64 query heads on one KV head
])
def test_tensor_consumer_against_the_oracle(nsv, form, heads, kv_heads, qlen, head_dim):
    wl = _case(heads, kv_heads, qlen, head_dim)
    inp = device_inputs(wl)
    host = host_copy(inp)
    plan = _plan(nsv, inp, consumer=form)
    assert plan.consumer == form
    out = gpu_step(wl, inp, plan=plan)
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)
    assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))


@pytest.mark.parametrize("kw", [
    dict(grid=1),                            # one CTA walks every unit
    dict(grid=3),
    dict(grid=5000),                         # more CTAs than units
    dict(stages=2, grid=9),
    dict(stages=6, kv_heads_per_cta=2),
    dict(kv_heads_per_cta=1),
    dict(kv_heads_per_cta=2, ctas_per_sm=2),
    dict(kv_heads_per_cta=8, ctas_per_sm=1, grid=100),
])
@pytest.mark.parametrize("qlen", [2, 3, 6])   # 8, 12 and 24 vectors per KV head
def test_tensor_consumer_plans(nsv, form, kw, qlen):
    wl = _case(32, 8, qlen, 128, seed=7)
    inp = device_inputs(wl)
    host = host_copy(inp)
    try:
        plan = _plan(nsv, inp, consumer=form, **kw)
    except nsv.NsvError as e:   # too many consumer warps, or CTAs per SM, for this shape
        assert e.code == -5 and ("kv_heads_per_cta" in kw or "ctas_per_sm" in kw)
        assert qlen >= 3 or form == nsv.CONSUMER_TENSOR_TMEM  # its group size is fixed
        pytest.skip("plan does not fit this shape")
    out = gpu_read(wl, inp, plan=plan)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_read(wl, host))


@pytest.mark.parametrize("qlen", [2, 4, 7])   # 8, 16 and 28 vectors per KV head
def test_both_consumers_agree_with_the_oracle(nsv, form, qlen):
    """The same inputs through the CUDA-core and the tensor-core consumer."""
    wl = _case(16, 4, qlen, 128, seed=9)
    inp = device_inputs(wl)
    host = host_copy(inp)
    ref = oracle_read(wl, host)
    errs = {}
    for c in (nsv.CONSUMER_CUDA, form):
        out = gpu_read(wl, inp, plan=_plan(nsv, inp, consumer=c))
        assert status()[0] == 0
        errs[c] = assert_parity("bf16", gpu_out_f64(out), ref)
    # P rounded to bf16 costs the tensor path a little, never an order of magnitude
    assert errs[form] <= max(10 * errs[nsv.CONSUMER_CUDA], 1e-2)


@pytest.mark.parametrize("heads,kv_heads,qlen", [(8, 2, 4), (4, 2, 4), (8, 2, 8),
                                                 (8, 2, 16), (16, 4, 4), (32, 8, 8)])
# 16, 8, 32, 64, 16, 32 vectors
def test_early_query_tokens_that_see_nothing(nsv, form, heads, kv_heads, qlen):
    """query_len n over rows shorter than n: query token j sees
    ctx - n + 1 + j positions, none when that is not positive (output 0)."""
    lens = [1, 2, 3, 4, 5, 0, 33]
    wl = _case(heads, kv_heads, qlen, 128, lens=lens, seed=13)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp, plan=_plan(nsv, inp, consumer=form))
    assert status()[0] == 0
    got = gpu_out_f64(out)
    ref = oracle_step(wl, host)
    assert_parity("bf16", got, ref)
    for r, c in enumerate(lens):
        assert np.all(got[r, :max(0, qlen - c)] == 0)      # tokens that see nothing
        assert c == 0 or np.any(got[r, qlen - min(c, qlen):] != 0)
    assert np.all(got[5] == 0)


@pytest.mark.parametrize("heads,kv_heads,head_dim", [(16, 4, 128), (16, 2, 128), (8, 4, 64),
                                                     (32, 2, 128)])   # 8, 16, 4, 32 vectors
def test_tensor_consumer_slot_gather(nsv, form, heads, kv_heads, head_dim):
    """Tokens scattered one by one over the pool: the producer warp gathers
    them into the swizzled layout the MMA reads."""
    import torch
    wl = _case(heads, kv_heads, 2, head_dim, seed=17, free_frac=1.5)
    inp = device_inputs(wl)
    host = host_copy(inp)
    rng = np.random.default_rng(21)
    pool_slots = (wl.num_blocks + 1) * 16
    width = wl.max_blocks * 16
    table = np.zeros((wl.rows, width), dtype=np.int64)
    for r in range(wl.rows):
        table[r] = rng.choice(pool_slots - 16, size=width, replace=False)
    # about half the blocks keep one aligned run: the bulk path beside the gather
    for r in range(wl.rows):
        for b in range(0, wl.max_blocks, 2):
            base = int(rng.integers(0, wl.num_blocks)) * 16
            table[r, b * 16:(b + 1) * 16] = base + np.arange(16)
    table = np.ascontiguousarray(table)
    out = torch.empty_like(inp["q"])
    plan = _plan(nsv, inp, consumer=form)
    nsv.paged_decode_slots(inp["q"], inp["k_pool"], inp["v_pool"],
                           torch.from_numpy(table).cuda(), inp["context_lens"], wl.scale, out,
                           workspace=nsv.workspace_for(plan), plan=plan,
                           max_blocks=wl.max_blocks)
    torch.cuda.synchronize()
    assert status()[0] == 0
    ref = oracle.paged_decode_slots(host["q"], host["k_pool"], host["v_pool"], table, width,
                                    wl.context_lens, wl.scale)
    assert_parity("bf16", gpu_out_f64(out), ref)


@pytest.mark.parametrize("consumer", [3, 4], ids=["vectors_as_rows", "tmem"])
def test_tensor_forms_ignore_poisoned_padding(nsv, consumer):
    """NaN in every pool slot no row addresses (past a row's length inside
    its last block, and all unused blocks) and garbage in the table's padding
    give the same bits as the clean run: masked scores and zeroed V rows keep
    NaN out of the MMAs (32 vectors per KV head)."""
    import torch
    wl = _case(32, 8, 8, 128, lens=[3, 16, 200, 1, 0, 999, 513, 40], seed=23, free_frac=0.5)
    inp = device_inputs(wl)
    host = host_copy(inp)
    plan = _plan(nsv, inp, consumer=consumer)
    clean = gpu_read(wl, inp, plan=plan).clone()
    used = np.zeros((wl.num_blocks + 1, 16), dtype=bool)
    for r, c in enumerate(wl.context_lens):
        for t in range(int(c)):
            used[wl.block_tables[r, t // 16], t % 16] = True
    mask = torch.from_numpy(~used).cuda()[:, None, :, None]
    nan = torch.tensor(float("nan"), dtype=inp["k_pool"].dtype, device="cuda")
    inp["k_pool"] = torch.where(mask, nan, inp["k_pool"])
    inp["v_pool"] = torch.where(mask, nan, inp["v_pool"])
    bt = wl.block_tables.copy()
    bt[bt < 0] = 2 ** 30
    inp["block_tables"] = torch.from_numpy(bt).cuda()
    poisoned = gpu_read(wl, inp, plan=plan)
    assert status()[0] == 0
    assert torch.equal(poisoned, clean)
    assert_parity("bf16", gpu_out_f64(poisoned), oracle_read(wl, host))


@pytest.mark.parametrize("consumer", [3, 4], ids=["vectors_as_rows", "tmem"])
def test_tensor_forms_skip_a_bad_block_mid_row(nsv, consumer):
    """A walked block id outside the pool in the middle of a row: that stage
    carries no data, the status flags it, and every other row stays exact."""
    import torch
    wl = _case(32, 8, 8, 128, lens=[40, 600, 300, 17], seed=29)
    inp = device_inputs(wl)
    host = host_copy(inp)
    ref = oracle_read(wl, host)
    bt = wl.block_tables.copy()
    bt[1, 5] = wl.num_blocks + 5
    inp["block_tables"] = torch.from_numpy(bt).cuda()
    status()
    out = gpu_out_f64(gpu_read(wl, inp, plan=_plan(nsv, inp, consumer=consumer)))
    st, _ = status()
    assert st & nsv.DEV_BAD_BLOCK
    keep = [0, 2, 3]
    assert_parity("bf16", out[keep], ref[keep])


@pytest.mark.parametrize("grid", [0, 7], ids=["grid_default", "grid_7"])
@pytest.mark.parametrize("blocks,stages", [(1, 2), (1, 5), (2, 3), (2, 4), (3, 2), (3, 3),
                                           (4, 2)])
@pytest.mark.parametrize("heads,kv_heads,qlen,head_dim", [
    (64, 8, 8, 128),    # 64 vectors per KV head, groups of 2
    (32, 8, 5, 128),    # 20 vectors
    (64, 1, 1, 128),    # one KV head: a group of 1
    (32, 8, 8, 64),     # head_dim 64, groups of 4
    (20, 5, 5, 64),     # 5 KV heads: groups of 1
])
def test_tmem_stage_sizes(nsv, grid, blocks, stages, heads, kv_heads, qlen, head_dim):
    """The TMEM form with every stage size (1 to 4 consecutive blocks of a
    row per stage, fewer where a segment ends) and several ring depths,
    against the oracle.  The lengths end mid-block, on block and on stage
    boundaries; a grid of 7 CTAs also cuts rows between CTAs, so pieces start
    and end inside a stage's reach."""
    wl = _case(heads, kv_heads, qlen, head_dim, seed=31)
    inp = device_inputs(wl)
    host = host_copy(inp)
    try:
        plan = _plan(nsv, inp, consumer=nsv.CONSUMER_TENSOR_TMEM, blocks_per_stage=blocks,
                     stages=stages, grid=grid)
    except nsv.NsvError as e:   # the stage does not fit shared or tensor memory
        assert e.code == -5
        pytest.skip("stage size does not fit this shape")
    assert plan.blocks_per_stage == blocks and plan.stages == stages
    out = gpu_read(wl, inp, plan=plan)
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)
    assert_parity("bf16", gpu_out_f64(out), oracle_read(wl, host))
