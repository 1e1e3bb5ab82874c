"""GPU parity: the CUDA path through the C ABI against the oracle.

Every comparison here feeds both sides the same seeded inputs; expected
values come only from the oracle (or, for bit-level invariants, from a second
run of the GPU path on relabelled or poisoned inputs).
"""

import numpy as np
import pytest

import oracle
from gpu_common import (assert_parity, default_plan, device_inputs, gpu_out_f64, gpu_read,
                        gpu_step, host_copy, oracle_read, oracle_step, oracle_step_sampled,
                        status)
from paged_kv_decode_nsv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nsv():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_kv_decode_nsv_gb300 import nsv as mod
    mod.device_status(clear=True)
    return mod


@pytest.fixture(autouse=True)
def _clean_status(nsv):
    yield
    import torch
    torch.cuda.empty_cache()


def _custom(name, lens, dtype="bf16", heads=8, kv_heads=8, head_dim=128, max_blocks=None,
            seed=7, free_frac=0.25):
    lens = np.asarray(lens)
    mb = max_blocks or max(1, int(max((int(c) + 15) // 16 for c in lens)) + 2)
    return W.custom(name, seed, rows=len(lens), heads=heads, kv_heads=kv_heads,
                    head_dim=head_dim, block_size=16, max_blocks=mb, dtype=dtype, lens=lens,
                    free_frac=free_frac)


# ---------------------------------------------------------------------------
# the KV append


@pytest.mark.parametrize("name", ["tiny_f32", "uniform_f32", "manyrow_bf16"])
def test_kv_write_bit_exact(nsv, name):
    wl = W.WORKLOADS[name]()
    inp = device_inputs(wl)
    host = host_copy(inp)
    nsv.kv_write(inp["k_new"], inp["v_new"], inp["write_slots"], inp["k_pool"], inp["v_pool"])
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    oracle.kv_write(host["k_new"], host["v_new"], wl.write_slots, kp, vp)
    gk, gv = W.to_numpy(inp["k_pool"]), W.to_numpy(inp["v_pool"])
    # the sink block's contents are unspecified when several pad rows name it
    assert np.array_equal(gk[:-1], kp[:-1]) and np.array_equal(gv[:-1], vp[:-1])
    st, _ = status()
    assert st == 0


# ---------------------------------------------------------------------------
# the full step (append + read) on the named workloads


@pytest.mark.parametrize("name", ["tiny_f32", "uniform_f32", "ragged_bf16", "manyrow_bf16"])
def test_step_parity_full(nsv, name):
    wl = W.WORKLOADS[name]()
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    st, walked = status()
    assert st == 0
    assert walked == oracle.walked_tiles(wl.context_lens, 16)
    ref = oracle_step(wl, host)
    assert_parity(wl.dtype, gpu_out_f64(out), ref)


def test_manyrow_interleaved_pads(nsv):
    wl = W.manyrow_bf16(interleave_pads=True)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    got = gpu_out_f64(out)
    pads = np.nonzero(wl.context_lens == 0)[0]
    assert len(pads) == 16 and np.all(got[pads] == 0.0)
    rows = list(pads[:4]) + [int(np.argmax(wl.context_lens))] + list(range(0, 256, 37))
    ref = oracle_step(wl, host, rows=rows)
    assert_parity(wl.dtype, got[rows], ref)


def test_headline_sampled_in_bench_configuration(nsv):
    """Full-size headline batch, the default plan the benchmark times,
    sampled rows (longest, shortest, first, last and a few more)."""
    wl = W.headline_bf16()
    inp = device_inputs(wl)
    ctx = wl.context_lens
    rng = np.random.default_rng(99)
    rows = sorted({int(np.argmax(ctx)), int(np.argmin(ctx)), 0, wl.rows - 1,
                   *map(int, rng.choice(wl.rows, 4, replace=False))})
    ref = oracle_step_sampled(wl, inp, rows)
    plan = default_plan(inp)
    out = gpu_step(wl, inp, plan=plan)
    st, walked = status()
    assert st == 0
    assert walked == oracle.walked_tiles(ctx, 16)
    assert_parity(wl.dtype, gpu_out_f64(out)[rows], ref)


# ---------------------------------------------------------------------------
# plans: every mode and knob gives the oracle's answer


MEDIUM_LENS = [1, 0, 17, 256, 1000, 333, 16, 15, 1024, 47]


@pytest.mark.parametrize("kw", [
    dict(),
    dict(grid=1),                            # one CTA walks every unit
    dict(grid=3),
    dict(grid=7, stages=2),
    dict(grid=5000),                         # more CTAs than units: empty ranges
    dict(stages=2),
    dict(stages=6, kv_heads_per_cta=2),
    dict(kv_heads_per_cta=1),
    dict(kv_heads_per_cta=2, ctas_per_sm=2),
    dict(kv_heads_per_cta=4, ctas_per_sm=1, grid=100),
    dict(kv_heads_per_cta=1, ctas_per_sm=4),  # four small CTAs per SM
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_plan_variants(nsv, kw, dtype):
    wl = _custom("medium", MEDIUM_LENS, dtype=dtype)
    inp = device_inputs(wl)
    host = host_copy(inp)
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    plan = nsv.plan_custom(shape, **kw)
    out = gpu_read(wl, inp, plan=plan)
    assert status()[0] == 0
    assert_parity(dtype, gpu_out_f64(out), oracle_read(wl, host))


@pytest.mark.parametrize("kw", [
    dict(kv_heads_per_cta=1, ctas_per_sm=8),
    dict(kv_heads_per_cta=1, ctas_per_sm=7, stages=2),
    dict(kv_heads_per_cta=2, ctas_per_sm=3),
    dict(consumer=2, kv_heads_per_cta=1, ctas_per_sm=6),
])
def test_many_small_ctas_per_sm(nsv, kw):
    """Plans with up to 8 resident CTAs per SM (small stages, one or two KV
    heads per CTA) read as the oracle does; with 2 query heads per KV head
    the tensor-core consumer is covered too."""
    wl = _custom("many_ctas", MEDIUM_LENS, heads=16 if kw.get("consumer") else 8)
    inp = device_inputs(wl)
    host = host_copy(inp)
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    plan = nsv.plan_custom(shape, **kw)
    assert plan.ctas_per_sm == kw["ctas_per_sm"]
    out = gpu_read(wl, inp, plan=plan)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_read(wl, host))


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 64), ("f32", 64), ("f32", 128)])
def test_head_dims_and_dtypes(nsv, dtype, head_dim):
    wl = _custom("dims", [5, 300, 0, 129, 700], dtype=dtype, head_dim=head_dim, heads=4,
                 kv_heads=4, seed=3)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    assert status()[0] == 0
    assert_parity(dtype, gpu_out_f64(out), oracle_step(wl, host))


@pytest.mark.parametrize("qw", [0, 1, 4])
@pytest.mark.parametrize("heads,kv_heads,dtype", [(32, 8, "bf16"), (16, 1, "bf16"),
                                                   (8, 4, "f32"), (12, 3, "bf16")])
def test_grouped_kv_heads(nsv, heads, kv_heads, dtype, qw):
    G = heads // kv_heads
    if qw and (G % qw or G // qw > (16 if qw <= 2 else 8)):
        pytest.skip("this group size cannot give %d vectors per warp" % qw)
    wl = _custom("gqa", [40, 513, 0, 2048, 77, 1], dtype=dtype, heads=heads,
                 kv_heads=kv_heads, seed=11)
    inp = device_inputs(wl)
    host = host_copy(inp)
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    out = gpu_step(wl, inp, plan=nsv.plan_custom(shape, vectors_per_warp=qw))
    assert status()[0] == 0
    assert_parity(dtype, gpu_out_f64(out), oracle_step(wl, host))


# ---------------------------------------------------------------------------
# invariants fixed by the pages


def test_poisoned_padding_is_never_read(nsv):
    """NaN in every slot no row addresses and garbage in the table's padding
    give the same bits as the clean run (Day 59: the load does not happen)."""
    import torch
    wl = _custom("poison", [3, 16, 200, 1, 0, 999], dtype="bf16", seed=5, free_frac=0.5)
    inp = device_inputs(wl)
    host = host_copy(inp)
    clean = gpu_read(wl, inp).clone()
    B = 16
    used = np.zeros((wl.num_blocks + 1, B), dtype=bool)
    for r, c in enumerate(wl.context_lens):
        for t in range(int(c)):
            used[wl.block_tables[r, t // B], t % B] = True
    mask = torch.from_numpy(~used).cuda()[:, None, :, None]
    nan = torch.tensor(float("nan"), dtype=inp["k_pool"].dtype, device="cuda")
    inp["k_pool"] = torch.where(mask, nan, inp["k_pool"])
    inp["v_pool"] = torch.where(mask, nan, inp["v_pool"])
    bt = wl.block_tables.copy()
    bt[bt < 0] = 2 ** 30
    inp["block_tables"] = torch.from_numpy(bt).cuda()
    poisoned = gpu_read(wl, inp)
    assert status()[0] == 0, "padding past a row's length must not even be range-checked"
    assert torch.equal(poisoned, clean)
    assert_parity("bf16", gpu_out_f64(poisoned), oracle_read(wl, host))


def test_warm_batch_of_padding_touches_nothing(nsv):
    """Day 55: an all-padding batch (ctx 0, writes to the sink) computes
    zeros and leaves every non-sink pool byte unchanged."""
    import torch
    wl = _custom("warm", [0] * 12, dtype="bf16", seed=9)
    wl.num_blocks = 64
    wl.block_tables[:] = -1
    wl.write_slots[:] = wl.sink_slot
    inp = device_inputs(wl)
    before_k, before_v = inp["k_pool"].clone(), inp["v_pool"].clone()
    out = torch.full_like(inp["q"], 7.0)
    gpu_step(wl, inp, out=out)
    st, walked = status()
    assert st == 0 and walked == 0
    assert torch.count_nonzero(out).item() == 0
    assert torch.equal(inp["k_pool"][:-1], before_k[:-1])
    assert torch.equal(inp["v_pool"][:-1], before_v[:-1])


def test_block_relabelling_is_bit_exact(nsv):
    import torch
    wl = _custom("perm", [700, 31, 0, 1500, 256], dtype="f32", seed=13)
    inp = device_inputs(wl)
    plan = default_plan(inp)
    base = gpu_read(wl, inp, plan=plan).clone()
    rng = np.random.default_rng(1)
    nb = wl.num_blocks
    perm = np.arange(nb + 1)
    perm[:nb] = rng.permutation(nb)
    pt = torch.from_numpy(perm).cuda()
    k2, v2 = torch.empty_like(inp["k_pool"]), torch.empty_like(inp["v_pool"])
    k2[pt] = inp["k_pool"]
    v2[pt] = inp["v_pool"]
    bt = np.where(wl.block_tables >= 0, perm[np.maximum(wl.block_tables, 0)], -1)
    inp2 = dict(inp, k_pool=k2, v_pool=v2,
                block_tables=torch.from_numpy(bt.astype(np.int32)).cuda())
    got = gpu_read(wl, inp2, plan=plan)
    assert torch.equal(got, base)


def test_repeat_runs_are_bit_identical(nsv):
    import torch
    wl = W.ragged_bf16()
    inp = device_inputs(wl)
    a = gpu_read(wl, inp).clone()
    b = gpu_read(wl, inp)
    assert torch.equal(a, b)


def test_library_workspace_matches_caller_workspace(nsv):
    import torch
    wl = _custom("libws", [900, 5, 2000, 0], dtype="bf16", seed=17)
    inp = device_inputs(wl)
    a = gpu_read(wl, inp).clone()
    b = torch.empty_like(inp["q"])
    nsv.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                     inp["context_lens"], wl.scale, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_walk_count_matches_host_accounting(nsv):
    """Day 59, "What I learned" 5: the tiles the kernel walks and the host's
    count of them must meet."""
    wl = W.WORKLOADS["ragged_bf16"]()
    inp = device_inputs(wl)
    status()
    for kw in (dict(), dict(grid=5), dict(grid=999, kv_heads_per_cta=1)):
        shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
        gpu_read(wl, inp, plan=nsv.plan_custom(shape, **kw))
        st, walked = status()
        assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)


# ---------------------------------------------------------------------------
# refusals: bad device-side values are flagged and skipped, never read


def test_device_side_refusals(nsv):
    import torch
    wl = _custom("bad", [40, 100, 7, 300], dtype="f32", seed=19)
    inp = device_inputs(wl)
    host = host_copy(inp)
    ref = oracle_read(wl, host)
    status()
    # a context length past the width: the row reads as empty and is flagged
    ctx = wl.context_lens.copy()
    ctx[1] = wl.width + 1
    inp_bad = dict(inp, context_lens=torch.from_numpy(ctx).cuda())
    out = gpu_out_f64(gpu_read(wl, inp_bad))
    st, _ = status()
    assert st & nsv.DEV_BAD_CTX
    assert np.all(out[1] == 0.0)
    keep = [0, 2, 3]
    assert_parity("f32", out[keep], ref[keep])
    # a walked block id outside the pool: skipped and flagged
    bt = wl.block_tables.copy()
    bt[2, 0] = wl.num_blocks + 5
    inp_bad = dict(inp, block_tables=torch.from_numpy(bt).cuda())
    out = gpu_out_f64(gpu_read(wl, inp_bad))
    st, _ = status()
    assert st & nsv.DEV_BAD_BLOCK
    assert_parity("f32", out[[0, 1, 3]], ref[[0, 1, 3]])
    # a write slot outside the pool array: not written, flagged
    slots = wl.write_slots.copy()
    slots[0] = (wl.num_blocks + 1) * 16
    kb = inp["k_pool"].clone()
    nsv.kv_write(inp["k_new"][:1], inp["v_new"][:1], torch.from_numpy(slots[:1]).cuda(),
                 inp["k_pool"], inp["v_pool"])
    st, _ = status()
    assert st & nsv.DEV_BAD_SLOT
    assert torch.equal(kb, inp["k_pool"])


def test_host_side_refusals(nsv):
    import torch
    wl = _custom("abi", [40, 100], dtype="bf16", seed=23)
    inp = device_inputs(wl)
    out = torch.empty_like(inp["q"])
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    plan = nsv.plan_custom(shape, grid=40)
    assert plan.workspace_bytes > 256
    with pytest.raises(nsv.NsvError) as e:
        nsv.paged_decode_ws(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                            inp["context_lens"], wl.scale, out, workspace=None, plan=plan)
    assert e.value.code == -8
    small = torch.empty(plan.workspace_bytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(nsv.NsvError) as e:
        nsv.paged_decode_ws(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                            inp["context_lens"], wl.scale, out, workspace=small, plan=plan)
    assert e.value.code == -8
    plan.grid += 1 if plan.grid < 100 else -1
    plan.smem_bytes += 16                      # no longer a plan the planner made
    with pytest.raises(nsv.NsvError) as e:
        nsv.paged_decode_ws(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                            inp["context_lens"], wl.scale, out,
                            workspace=nsv.workspace_for(plan), plan=plan)
    assert e.value.code == -5
    odd = torch.empty(out.numel() * 2 + 8, dtype=torch.uint8, device="cuda")[8:]
    odd = odd.view(torch.bfloat16).view(out.shape)
    with pytest.raises(nsv.NsvError) as e:
        nsv.paged_decode(inp["q"], inp["k_pool"], inp["v_pool"], inp["block_tables"],
                         inp["context_lens"], wl.scale, odd)
    assert e.value.code == -4


def test_refused_step_launches_nothing(nsv):
    """nsv_decode_step checks the read's arguments before launching the
    append: a step whose read is refused leaves the pool untouched."""
    import torch
    wl = _custom("step_refused", [40, 100], dtype="bf16", seed=29)
    inp = device_inputs(wl)
    k0, v0 = inp["k_pool"].clone(), inp["v_pool"].clone()
    out = torch.empty_like(inp["q"])
    odd = torch.empty(out.numel() * 2 + 8, dtype=torch.uint8, device="cuda")[8:]
    odd = odd.view(torch.bfloat16).view(out.shape)          # misaligned output
    with pytest.raises(nsv.NsvError) as e:
        nsv.decode_step(inp["q"], inp["k_new"], inp["v_new"], inp["write_slots"],
                        inp["k_pool"], inp["v_pool"], inp["block_tables"], inp["context_lens"],
                        wl.scale, odd)
    assert e.value.code == -4
    torch.cuda.synchronize()
    assert torch.equal(inp["k_pool"], k0) and torch.equal(inp["v_pool"], v0)
    assert status()[0] == 0


# ---------------------------------------------------------------------------
# several query tokens per row (causal among themselves) and grouped heads:
# a consumer warp serves up to 4 query vectors from one K/V tile


@pytest.mark.parametrize("qlen,heads,kv_heads,dtype,head_dim", [
    (2, 8, 8, "bf16", 128), (3, 8, 8, "f32", 128), (4, 8, 8, "bf16", 128),
    (4, 32, 8, "bf16", 128), (2, 16, 4, "f32", 64), (8, 8, 2, "bf16", 64),
    (5, 4, 4, "bf16", 128), (4, 4, 1, "f32", 128),
])
def test_multi_query_step(nsv, qlen, heads, kv_heads, dtype, head_dim):
    lens = [qlen, 100, 0, 1030, 17, 2 * qlen + 1, 1]   # the last row is shorter than qlen
    wl = W.custom("mq", 51 + qlen, rows=len(lens), heads=heads, kv_heads=kv_heads,
                  head_dim=head_dim, block_size=16, max_blocks=70, dtype=dtype, lens=lens,
                  free_frac=0.2, query_len=qlen)
    inp = device_inputs(wl)
    host = host_copy(inp)
    out = gpu_step(wl, inp)
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(wl.context_lens, 16)
    ref = oracle_step(wl, host)
    assert ref.shape == (len(lens), qlen, heads, head_dim)
    assert_parity(dtype, gpu_out_f64(out), ref)


@pytest.mark.parametrize("kw", [dict(grid=1), dict(grid=5000), dict(stages=2, grid=9),
                                dict(kv_heads_per_cta=1), dict(vectors_per_warp=4),
                                dict(vectors_per_warp=1), dict(vectors_per_warp=4, grid=7),
                                dict(vectors_per_warp=2, kv_heads_per_cta=8)])
def test_multi_query_plans(nsv, kw):
    wl = W.custom("mq_plans", 61, rows=5, heads=8, kv_heads=8, head_dim=128, block_size=16,
                  max_blocks=70, dtype="bf16", lens=[4, 700, 0, 1100, 33], free_frac=0.2,
                  query_len=4)
    inp = device_inputs(wl)
    host = host_copy(inp)
    shape = nsv.shape_of(inp["q"], inp["k_pool"], inp["block_tables"])
    plan = nsv.plan_custom(shape, **kw)
    out = gpu_step(wl, inp, plan=plan)
    assert status()[0] == 0
    assert_parity("bf16", gpu_out_f64(out), oracle_step(wl, host))


@pytest.mark.parametrize("name", ["headline_spec4_bf16", "headline_gqa4_bf16",
                                  "headline_gqa8_spec8_bf16", "headline_mqa8_bf16"])
def test_headline_variants_sampled(nsv, name):
    """Full-size headline batches with 4 query tokens per row, with 4 query
    heads per KV head, with both grouped heads and speculative tokens (64
    query vectors per KV head, tcgen05), and with 8 query heads on a single
    KV head (six small CTAs per SM), in the benchmark's default plan; sampled
    rows."""
    wl = W.WORKLOADS[name]()
    inp = device_inputs(wl)
    ctx = wl.context_lens
    rows = sorted({int(np.argmax(ctx)), int(np.argmin(ctx)), 0, wl.rows - 1, 77, 130})
    ref = oracle_step_sampled(wl, inp, rows)
    out = gpu_step(wl, inp, plan=default_plan(inp))
    st, walked = status()
    assert st == 0 and walked == oracle.walked_tiles(ctx, 16)
    assert_parity(wl.dtype, gpu_out_f64(out)[rows], ref)
