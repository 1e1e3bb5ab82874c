"""The seeded input generators follow the recipe they state (workloads.py's
docstring): the named lengths, one block-table run per row dealt from a
permutation of the pool, -1 padding, write slots at each row's last
positions (the sink for a padded row), reproducible draws, and bf16 values
rounded to nearest even.  Every parity test compares the two sides on these
inputs, so they are pinned here on the CPU.
"""

import numpy as np
import pytest
import torch

from paged_kv_decode_nsv_gb300 import workloads as W

NAMES = sorted(W.WORKLOADS)


def _nblocks(wl):
    return (wl.context_lens.astype(np.int64) + wl.block_size - 1) // wl.block_size


@pytest.mark.parametrize("name", NAMES)
def test_tables_are_one_run_per_row_from_a_permutation(name):
    wl = W.WORKLOADS[name]()
    nb = _nblocks(wl)
    bt = wl.block_tables
    assert bt.shape == (wl.rows, wl.max_blocks) and bt.dtype == np.int32
    assert (nb <= wl.max_blocks).all()
    used = []
    for r in range(wl.rows):
        run = bt[r, :nb[r]]
        assert ((run >= 0) & (run < wl.num_blocks)).all()
        assert (bt[r, nb[r]:] == -1).all()
        used.extend(run.tolist())
    # every block is some row's, once: the rows never share a block
    assert len(used) == len(set(used)) == int(nb.sum()) <= wl.num_blocks
    # and the blocks are scattered (dealt from a permutation, not in order)
    if len(used) > 64:
        assert np.mean(np.diff(np.asarray(used)) == 1) < 0.1


@pytest.mark.parametrize("name", NAMES)
def test_write_slots_are_each_rows_last_positions(name):
    wl = W.WORKLOADS[name]()
    B, ql = wl.block_size, wl.query_len
    ws = np.asarray(wl.write_slots).reshape(wl.rows, ql)
    sink = wl.num_blocks * B
    assert wl.sink_slot == sink
    for r in range(wl.rows):
        for j in range(ql):
            t = int(wl.context_lens[r]) - ql + j
            want = sink if t < 0 else int(wl.block_tables[r, t // B]) * B + t % B
            assert int(ws[r, j]) == want, (r, j)


@pytest.mark.parametrize("name", NAMES)
def test_generators_are_reproducible(name):
    a, b = W.WORKLOADS[name](), W.WORKLOADS[name]()
    assert np.array_equal(a.context_lens, b.context_lens)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(np.asarray(a.write_slots), np.asarray(b.write_slots))
    assert a.num_blocks == b.num_blocks and a.scale == b.scale


def test_named_lengths_and_pools():
    t = W.tiny_f32()
    assert t.context_lens.tolist() == [16, 40, 100, 257, 0] and t.num_blocks == 64
    assert t.scale == 1.0 / 8.0 and t.dtype == "f32" and t.head_dim == 64
    u = W.uniform_f32()
    assert (u.context_lens == 2048).all() and u.rows == 8 and u.num_blocks == 2048
    assert int(_nblocks(u).sum()) == 1024   # half the pool
    rg = W.ragged_bf16()
    lens = rg.context_lens
    assert lens[0] == 8192 and ((lens[1:] >= 128) & (lens[1:] < 2048)).all()
    assert rg.num_blocks == int(_nblocks(rg).sum())
    for name in ("manyrow_bf16", "manyrow_gqa4_bf16", "manyrow_gqa8_spec8_bf16",
                 "manyrow_gqa16_bf16"):
        m = W.WORKLOADS[name]()
        lens = m.context_lens
        assert m.rows == 256 and lens[0] == 2048
        assert ((lens[1:240] >= 128) & (lens[1:240] < 2048)).all() and (lens[240:] == 0).all()
        need = int(_nblocks(m).sum())
        assert m.num_blocks == int(np.ceil(need * 1.1))
    for name in ("headline_bf16", "headline_gqa4_bf16", "headline_spec4_bf16",
                 "headline_gqa8_spec8_bf16", "headline_mqa8_bf16"):
        h = W.WORKLOADS[name]()
        lens = h.context_lens
        assert h.rows == 256 and h.head_dim == 128 and h.max_blocks == 512
        assert ((lens >= 512) & (lens <= 8192)).all()
        assert h.num_blocks == int(_nblocks(h).sum())
    # the headline batch's lengths are the same draw in every variant of it
    base = W.headline_bf16().context_lens
    for name in ("headline_gqa4_bf16", "headline_spec4_bf16", "headline_gqa8_spec8_bf16",
                 "headline_mqa8_bf16"):
        assert np.array_equal(W.WORKLOADS[name]().context_lens, base)


def test_host_values_are_seeded_normals():
    wl = W.tiny_f32()
    q, kp, vp, kn, vn = W.host_values(wl)
    q2, kp2, _, _, _ = W.host_values(wl)
    assert np.array_equal(q, q2) and np.array_equal(kp, kp2)
    assert q.shape == tuple(wl.q_shape) and kp.shape == tuple(wl.pool_shape)
    assert kn.shape == tuple(wl.new_shape) and vn.shape == tuple(wl.new_shape)
    x = np.concatenate([a.ravel() for a in (q, kp, vp)])
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1.0) < 0.05
    other = W.host_values(wl, value_seed=12345)[0]
    assert not np.array_equal(q, other)


def test_bf16_rounding_is_round_to_nearest_even():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(4096).astype(np.float32) * np.float32(3.0)
    # exact ties and values next to them: the rounding bit pattern 0x8000
    # below the kept half, with an even and an odd kept part
    base = rng.integers(0x3F800000, 0x40800000, size=256, dtype=np.uint32) & np.uint32(0xFFFF0000)
    ties = np.concatenate([base | np.uint32(0x8000), (base | np.uint32(0x10000)) | np.uint32(0x8000),
                           base | np.uint32(0x7FFF), base | np.uint32(0x8001)])
    x = np.concatenate([x, ties.view(np.float32)])
    ours = W.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(W.bf16_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())
