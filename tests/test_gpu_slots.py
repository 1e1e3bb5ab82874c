"""The decode read through a per-token slot table (Day 51's SlotTable) on
the GPU, against the oracle and against the block-table read."""

import numpy as np
import pytest

import oracle
from gpu_common import (assert_parity, default_plan, device_inputs, gpu_out_f64, gpu_read,
                        host_copy, status)
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


def slots_from_tables(bt, B=16):
    R, MB = bt.shape
    t = np.arange(MB * B)
    blk = bt[:, t // B].astype(np.int64)
    return np.ascontiguousarray(np.where(blk >= 0, blk * B + t % B, -1), dtype=np.int64)


def read_slots(nsv, wl, inp, table, plan=None, width=None):
    import torch
    out = torch.empty_like(inp["q"])
    if plan is None:
        plan = default_plan(inp)
    ws = nsv.workspace_for(plan)
    nsv.paged_decode_slots(inp["q"], inp["k_pool"], inp["v_pool"], table, inp["context_lens"],
                           wl.scale, out, workspace=ws, plan=plan, max_blocks=wl.max_blocks)
    torch.cuda.synchronize()
    return out


def _case(name, lens, dtype="bf16", query_len=1, heads=8, kv_heads=8, free_frac=0.3):
    return W.custom(name, 71, rows=len(lens), heads=heads, kv_heads=kv_heads, head_dim=128,
                    block_size=16, max_blocks=70, dtype=dtype, lens=lens, free_frac=free_frac,
                    query_len=query_len)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_table_from_block_tables_reads_the_same_bits(nsv, dtype):
    import torch
    wl = _case("slots_same", [1, 0, 300, 1024, 17, 999], dtype=dtype)
    inp = device_inputs(wl)
    plan = default_plan(inp)
    base = gpu_read(wl, inp, plan=plan).clone()
    table = torch.from_numpy(slots_from_tables(wl.block_tables)).cuda()
    got = read_slots(nsv, wl, inp, table, plan=plan)
    assert status()[0] == 0
    assert torch.equal(got, base)
    # the same table as a window of a wider, persistent buffer (row stride 4096)
    wide = torch.full((wl.rows, 4096), -7, dtype=torch.int64, device="cuda")
    wide[:, :table.shape[1]] = table
    got2 = read_slots(nsv, wl, inp, wide[:, :table.shape[1]], plan=plan)
    assert status()[0] == 0
    assert torch.equal(got2, base)


def _scatter_tokens(wl, seed, shuffle_frac=1.0):
    """A slot table whose tokens sit at arbitrary slots of the pool: each
    row's positions take distinct slots; a fraction of the rows keeps the
    block-table layout, the rest is shuffled token by token."""
    rng = np.random.default_rng(seed)
    B = wl.block_size
    base = slots_from_tables(wl.block_tables, B)
    free = rng.permutation(wl.num_blocks * B)
    table = np.ascontiguousarray(base)
    off = 0
    for r, c in enumerate(wl.context_lens):
        c = int(c)
        if c == 0 or rng.random() > shuffle_frac:
            continue
        table[r, :c] = free[off:off + c]
        off += c
    return table


@pytest.mark.parametrize("qlen,frac,dtype", [(1, 1.0, "bf16"), (1, 0.5, "f32"),
                                              (4, 1.0, "bf16"), (2, 0.5, "bf16")])
def test_scattered_tokens_against_the_oracle(nsv, qlen, frac, dtype):
    import torch
    lens = [qlen, 0, 300, 1024, 17, 999, 64]
    wl = _case("slots_scattered", lens, dtype=dtype, query_len=qlen, free_frac=1.5)
    inp = device_inputs(wl)
    host = host_copy(inp)
    table_np = _scatter_tokens(wl, 5 + qlen, frac)
    # the oracle gathers its whole rectangle: make every padding entry legal
    table_np = np.ascontiguousarray(np.where(table_np >= 0, table_np, 0))
    out = read_slots(nsv, wl, inp, torch.from_numpy(table_np).cuda())
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)
    ref = oracle.paged_decode_slots(host["q"], host["k_pool"], host["v_pool"], table_np,
                                    table_np.shape[1], wl.context_lens, wl.scale)
    assert_parity(dtype, gpu_out_f64(out), ref)


def test_gqa_through_scattered_slots(nsv):
    import torch
    wl = _case("slots_gqa", [40, 513, 0, 1100], heads=32, kv_heads=8, free_frac=1.5)
    inp = device_inputs(wl)
    host = host_copy(inp)
    table_np = _scatter_tokens(wl, 9, 0.6)
    table_np = np.ascontiguousarray(np.where(table_np >= 0, table_np, 0))
    out = read_slots(nsv, wl, inp, torch.from_numpy(table_np).cuda())
    assert status()[0] == 0
    ref = oracle.paged_decode_slots(host["q"], host["k_pool"], host["v_pool"], table_np,
                                    table_np.shape[1], wl.context_lens, wl.scale)
    assert_parity("bf16", gpu_out_f64(out), ref)


def test_slots_past_the_length_are_never_read(nsv):
    """NaN everywhere no row addresses and garbage slots past each row's
    length leave every output bit unchanged, in both gather paths."""
    import torch
    wl = _case("slots_poison", [3, 16, 200, 1, 0, 999], free_frac=1.5)
    inp = device_inputs(wl)
    table_np = _scatter_tokens(wl, 13, 0.5)
    table = torch.from_numpy(table_np).cuda()
    clean = read_slots(nsv, wl, inp, table).clone()
    B = 16
    used = np.zeros((wl.num_blocks + 1) * B, dtype=bool)
    for r, c in enumerate(wl.context_lens):
        used[table_np[r, :int(c)]] = True
    mask = torch.from_numpy(~used.reshape(-1, B)).cuda()[:, None, :, None]
    nan = torch.tensor(float("nan"), dtype=inp["k_pool"].dtype, device="cuda")
    inp["k_pool"] = torch.where(mask, nan, inp["k_pool"])
    inp["v_pool"] = torch.where(mask, nan, inp["v_pool"])
    t2 = table_np.copy()
    for r, c in enumerate(wl.context_lens):
        t2[r, int(c):] = 2 ** 40
    got = read_slots(nsv, wl, inp, torch.from_numpy(t2).cuda())
    assert status()[0] == 0
    assert torch.equal(got, clean)


def test_bad_slots_are_flagged_and_skipped(nsv):
    import torch
    wl = _case("slots_bad", [40, 100, 7, 300], dtype="f32")
    inp = device_inputs(wl)
    host = host_copy(inp)
    table_np = slots_from_tables(wl.block_tables)
    table_np = np.ascontiguousarray(np.where(table_np >= 0, table_np, 0))
    ref = oracle.paged_decode_slots(host["q"], host["k_pool"], host["v_pool"], table_np,
                                    table_np.shape[1], wl.context_lens, wl.scale)
    status()
    bad = table_np.copy()
    bad[2, 3] = (wl.num_blocks + 1) * 16 + 5     # row 2: one slot past the pool
    bad[1, 0] = (wl.num_blocks + 9) * 16         # row 1: a whole run past the pool
    out = gpu_out_f64(read_slots(nsv, wl, inp, torch.from_numpy(bad).cuda()))
    st, _ = status()
    assert st & nsv.DEV_BAD_BLOCK
    assert_parity("f32", out[[0, 3]], ref[[0, 3]])


def test_headline_through_a_slot_table_reads_the_same_bits(nsv):
    """The full headline batch: a slot table built from its block tables,
    read in the benchmark's plan, gives the block-table read's bits."""
    import torch
    wl = W.headline_bf16()
    inp = device_inputs(wl)
    plan = default_plan(inp)
    base = gpu_read(wl, inp, plan=plan).clone()
    table = torch.from_numpy(slots_from_tables(wl.block_tables)).cuda()
    got = read_slots(nsv, wl, inp, table, plan=plan)
    st, walked = status()
    assert st == 0 and walked == 2 * oracle.walked_tiles(wl.context_lens, 16)
    assert torch.equal(got, base)
