"""Seeded synthetic decode batches shaped like the nanoserve pages' workloads.

This module only builds inputs: context lengths, block tables, write slots
and N(0, 1) values.  It holds none of the decode read's arithmetic, imports
neither the CUDA binding nor the oracle, and is shared by the tests, the
benchmark and the smoke check so that both sides of every comparison see the
same seeded numbers.

Recipe (the same for every workload):
  * lengths: per workload, below.  A row's context length already counts the
    token this step appends (its write slot is the row's last real entry,
    nanoserve Day 51, "What I learned" item 2).
  * blocks: row r needs cdiv(ctx_r, block_size) blocks.  A seeded permutation
    of the pool's blocks is dealt out to the rows in order, so every row's
    blocks are scattered over the pool.  Block-table entries past a row's
    last block are -1 (Day 59, "Why it matters": the padding may be -1).
  * write slots: a real row writes the slot of its position ctx - 1; a padded
    row (ctx 0) writes the sink slot num_blocks * block_size, one past the
    pool the allocator hands out (Day 55, "Why it matters").
  * values: q, K, V, k_new, v_new ~ N(0, 1), drawn in fp32 and rounded to
    bf16 (round to nearest even) for bf16 workloads.  Small pools are drawn on
    the host with numpy; large pools are drawn on the device with torch's
    seeded CUDA generator (host draws of 10^9-10^10 values would take minutes).

The five named workloads:
  tiny_f32      4 rows + 1 padded row, 4 heads, head_dim 64, block 16,
                64-block pool, lengths {16, 40, 100, 257, 0}, scale 1/8.
  uniform_f32   8 rows, 32 heads, head_dim 128, every length 2048,
                2048-block pool (half used).
  ragged_bf16   32 rows, 32 heads, head_dim 128, width 8192; row 0 is 8192
                long, the rest floor(log-uniform[128, 2048]); pool = the sum.
  manyrow_bf16  256 rows, 32 heads, head_dim 128, width 2048; row 0 is 2048
                long, rows 1..239 log-uniform[128, 2048], the last 16 rows
                padded; pool = what the rows need + 10% free.
  headline_bf16 256 rows, 32 heads, head_dim 128, width 8192, lengths
                uniform integers in [512, 8192]; pool = the sum.
  headline_gqa4_bf16  the same with 8 KV heads shared by 32 query heads.
"""

from dataclasses import dataclass, field
import math

import numpy as np

# Pool elements above which values are drawn on the device, not the host.
HOST_DRAW_LIMIT = 64 * 1024 * 1024


@dataclass
class Workload:
    name: str
    rows: int
    heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    max_blocks: int
    num_blocks: int            # blocks the allocator hands out (sink excluded)
    dtype: str                 # "f32" or "bf16"
    scale: float
    seed: int
    context_lens: np.ndarray = field(repr=False)   # [rows] int32
    block_tables: np.ndarray = field(repr=False)   # [rows, max_blocks] int32
    write_slots: np.ndarray = field(repr=False)    # [rows] (or [rows, query_len]) int64
    query_len: int = 1                              # query tokens per row

    @property
    def width(self):
        return self.max_blocks * self.block_size

    @property
    def sink_slot(self):
        return self.num_blocks * self.block_size

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def pool_shape(self):
        return (self.num_blocks + 1, self.kv_heads, self.block_size, self.head_dim)

    @property
    def pool_elems(self):
        return math.prod(self.pool_shape)

    @property
    def total_tokens(self):
        return int(self.context_lens.astype(np.int64).sum())

    def kv_bytes_read(self):
        """Unique K and V bytes the read needs: sum(ctx) * kv_heads * head_dim * 2 * elem."""
        return self.total_tokens * self.kv_heads * self.head_dim * 2 * self.elem_bytes

    def q_out_bytes(self):
        return 2 * self.rows * self.query_len * self.heads * self.head_dim * self.elem_bytes

    def append_bytes(self):
        """The append reads k_new, v_new and writes the same bytes into the pool."""
        return (2 * 2 * self.rows * self.query_len * self.kv_heads * self.head_dim *
                self.elem_bytes)

    @property
    def q_shape(self):
        if self.query_len == 1:
            return (self.rows, self.heads, self.head_dim)
        return (self.rows, self.query_len, self.heads, self.head_dim)

    @property
    def new_shape(self):
        if self.query_len == 1:
            return (self.rows, self.kv_heads, self.head_dim)
        return (self.rows, self.query_len, self.kv_heads, self.head_dim)

    def read_bytes(self):
        """Algorithmic bytes of one decode read (KV + q + out)."""
        return self.kv_bytes_read() + self.q_out_bytes()

    def step_bytes(self):
        """Algorithmic bytes of one serving step (append + read)."""
        return self.read_bytes() + self.append_bytes()


def bf16_bits(x):
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite x)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = u >> 16
    r &= 1
    r += 0x7FFF
    r += u          # finite inputs stay below 2^32 - 2^16, so no wrap-around
    r >>= 16
    return r.astype(np.uint16)


def bf16_to_f32(bits):
    """bf16 bit patterns -> fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _tables(rng, lens, block_size, num_blocks, max_blocks, query_len=1):
    """Deal a seeded permutation of the pool's blocks out to the rows."""
    nb = [(int(c) + block_size - 1) // block_size for c in lens]
    need = sum(nb)
    if need > num_blocks:
        raise ValueError("pool of %d blocks cannot hold %d" % (num_blocks, need))
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(nb):
        if n > max_blocks:
            raise ValueError("row %d needs %d blocks > max_blocks %d" % (r, n, max_blocks))
        bt[r, :n] = perm[off:off + n]
        off += n
    # the step's new tokens are each row's last query_len positions
    ws = np.empty((len(lens), query_len), dtype=np.int64)
    for r, c in enumerate(lens):
        for j in range(query_len):
            t = int(c) - query_len + j
            if t < 0:
                ws[r, j] = num_blocks * block_size
            else:
                ws[r, j] = int(bt[r, t // block_size]) * block_size + t % block_size
    return bt, (ws[:, 0].copy() if query_len == 1 else ws)


def _make(name, seed, rows, heads, kv_heads, head_dim, block_size, max_blocks,
          dtype, lens, num_blocks=None, free_frac=0.0, scale=None, rng=None, query_len=1):
    rng = rng if rng is not None else np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    need = int(sum((int(c) + block_size - 1) // block_size for c in lens))
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(need * (1.0 + free_frac))))
    bt, ws = _tables(rng, lens, block_size, num_blocks, max_blocks, query_len)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Workload(name=name, rows=rows, heads=heads, kv_heads=kv_heads,
                    head_dim=head_dim, block_size=block_size, max_blocks=max_blocks,
                    num_blocks=num_blocks, dtype=dtype, scale=scale, seed=seed,
                    context_lens=lens, block_tables=bt, write_slots=ws, query_len=query_len)


def _log_uniform(rng, n, lo, hi):
    return np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))).astype(np.int64)


def tiny_f32(seed=0):
    return _make("tiny_f32", seed, rows=5, heads=4, kv_heads=4, head_dim=64,
                 block_size=16, max_blocks=17, dtype="f32",
                 lens=[16, 40, 100, 257, 0], num_blocks=64, scale=1.0 / 8.0)


def uniform_f32(seed=1):
    return _make("uniform_f32", seed, rows=8, heads=32, kv_heads=32, head_dim=128,
                 block_size=16, max_blocks=128, dtype="f32",
                 lens=[2048] * 8, num_blocks=2048)


def ragged_bf16(seed=2):
    rng = np.random.default_rng(seed)
    lens = np.concatenate([[8192], _log_uniform(rng, 31, 128, 2048)])
    return _make("ragged_bf16", seed, rows=32, heads=32, kv_heads=32, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng)


def manyrow_bf16(seed=3, interleave_pads=False):
    rng = np.random.default_rng(seed)
    real = np.concatenate([[2048], _log_uniform(rng, 239, 128, 2048)])
    lens = np.concatenate([real, np.zeros(16, dtype=np.int64)])
    if interleave_pads:
        lens = lens[rng.permutation(256)]
    return _make("manyrow_bf16" + ("_interleaved" if interleave_pads else ""), seed,
                 rows=256, heads=32, kv_heads=32, head_dim=128, block_size=16,
                 max_blocks=128, dtype="bf16", lens=lens, free_frac=0.10, rng=rng)


def headline_bf16(seed=4):
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=256, endpoint=True)
    return _make("headline_bf16", seed, rows=256, heads=32, kv_heads=32, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng)


def headline_gqa4_bf16(seed=4):
    """The headline batch with grouped-query attention: 32 query heads share
    8 KV heads (4 per group); same lengths and pool recipe."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=256, endpoint=True)
    return _make("headline_gqa4_bf16", seed, rows=256, heads=32, kv_heads=8, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng)


def headline_spec4_bf16(seed=4):
    """The headline batch verifying 4 speculative tokens per row: 4 query
    tokens per row and head, causal among themselves; same lengths (which
    count the 4 new tokens) and pool recipe."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=256, endpoint=True)
    return _make("headline_spec4_bf16", seed, rows=256, heads=32, kv_heads=32, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng, query_len=4)


def headline_gqa8_spec8_bf16(seed=4):
    """The headline batch with both: 64 query heads share 8 KV heads (8 per
    group) and each row verifies 8 speculative tokens, so 64 query vectors
    read every K/V tile; same lengths (which count the 8 new tokens) and pool
    recipe."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=256, endpoint=True)
    return _make("headline_gqa8_spec8_bf16", seed, rows=256, heads=64, kv_heads=8, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng, query_len=8)


def manyrow_gqa8_spec8_bf16(seed=3):
    """The many-row batch with 64 query vectors per KV tile (64 query heads
    over 8 KV heads, 8 query tokens): a 0.7 GB case for a full ncu capture."""
    rng = np.random.default_rng(seed)
    real = np.concatenate([[2048], _log_uniform(rng, 239, 128, 2048)])
    lens = np.concatenate([real, np.zeros(16, dtype=np.int64)])
    return _make("manyrow_gqa8_spec8_bf16", seed, rows=256, heads=64, kv_heads=8, head_dim=128,
                 block_size=16, max_blocks=128, dtype="bf16", lens=lens, free_frac=0.10, rng=rng,
                 query_len=8)


def manyrow_gqa4_bf16(seed=3):
    """The many-row batch with 8 KV heads shared by 32 query heads: a 0.7 GB
    grouped-query case small enough for a full ncu capture."""
    rng = np.random.default_rng(seed)
    real = np.concatenate([[2048], _log_uniform(rng, 239, 128, 2048)])
    lens = np.concatenate([real, np.zeros(16, dtype=np.int64)])
    return _make("manyrow_gqa4_bf16", seed, rows=256, heads=32, kv_heads=8, head_dim=128,
                 block_size=16, max_blocks=128, dtype="bf16", lens=lens, free_frac=0.10, rng=rng)


def manyrow_gqa16_bf16(seed=3):
    """The many-row batch with 16 query vectors per KV head: 64 query heads
    share 4 KV heads.  The default plan
    runs it with the vectors as the MMA rows (mma.sync), so it is the capture
    case of that form; 0.35 GB per read."""
    rng = np.random.default_rng(seed)
    real = np.concatenate([[2048], _log_uniform(rng, 239, 128, 2048)])
    lens = np.concatenate([real, np.zeros(16, dtype=np.int64)])
    return _make("manyrow_gqa16_bf16", seed, rows=256, heads=64, kv_heads=4, head_dim=128,
                 block_size=16, max_blocks=128, dtype="bf16", lens=lens, free_frac=0.10, rng=rng)


def headline_mqa8_bf16(seed=4):
    """The headline batch as one tensor-parallel shard of a grouped-query
    model: 8 query heads share the shard's single KV head; same lengths and
    pool recipe.  Its stages are small (one KV head of one block, 8 KiB), so
    the read is bound by how many consumer warps an SM keeps resident."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(512, 8192, size=256, endpoint=True)
    return _make("headline_mqa8_bf16", seed, rows=256, heads=8, kv_heads=1, head_dim=128,
                 block_size=16, max_blocks=512, dtype="bf16", lens=lens, rng=rng)


WORKLOADS = {
    "tiny_f32": tiny_f32,
    "uniform_f32": uniform_f32,
    "ragged_bf16": ragged_bf16,
    "manyrow_bf16": manyrow_bf16,
    "headline_bf16": headline_bf16,
    "headline_gqa4_bf16": headline_gqa4_bf16,
    "headline_spec4_bf16": headline_spec4_bf16,
    "manyrow_gqa4_bf16": manyrow_gqa4_bf16,
    "headline_gqa8_spec8_bf16": headline_gqa8_spec8_bf16,
    "manyrow_gqa8_spec8_bf16": manyrow_gqa8_spec8_bf16,
    "headline_mqa8_bf16": headline_mqa8_bf16,
    "manyrow_gqa16_bf16": manyrow_gqa16_bf16,
}


def custom(name, seed, rows, heads, kv_heads, head_dim, block_size, max_blocks,
           dtype, lens, num_blocks=None, free_frac=0.0, scale=None, query_len=1):
    """A workload with given lengths (used for edge cases and small sweeps)."""
    return _make(name, seed, rows=rows, heads=heads, kv_heads=kv_heads,
                 head_dim=head_dim, block_size=block_size, max_blocks=max_blocks,
                 dtype=dtype, lens=lens, num_blocks=num_blocks,
                 free_frac=free_frac, scale=scale, query_len=query_len)


def spread_lengths(rows, width, spread):
    """Length mixes of the Day-59 streambench table ("spread" column).

    uniform   every row at the full width
    2x        rows alternate between the width and half of it
    long tail in each group of 8 rows, one row at the width, seven at width/8
    """
    if spread == "uniform":
        return np.full(rows, width, dtype=np.int32)
    if spread == "2x":
        return np.array([width if r % 2 == 0 else width // 2 for r in range(rows)], dtype=np.int32)
    if spread == "long tail":
        return np.array([width if r % 8 == 0 else width // 8 for r in range(rows)], dtype=np.int32)
    raise ValueError("unknown spread %r" % spread)


# ---------------------------------------------------------------------------
# values


def _host_normal(rng, shape, dtype):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return x if dtype == "f32" else bf16_bits(x)


def host_values(wl, value_seed=None):
    """q, k_pool, v_pool, k_new, v_new as numpy arrays (fp32 or bf16 bits)."""
    rng = np.random.default_rng(wl.seed + 1000 if value_seed is None else value_seed)
    q = _host_normal(rng, wl.q_shape, wl.dtype)
    k_pool = _host_normal(rng, wl.pool_shape, wl.dtype)
    v_pool = _host_normal(rng, wl.pool_shape, wl.dtype)
    k_new = _host_normal(rng, wl.new_shape, wl.dtype)
    v_new = _host_normal(rng, wl.new_shape, wl.dtype)
    return q, k_pool, v_pool, k_new, v_new


def device_values(wl, device, value_seed=None):
    """q, k_pool, v_pool, k_new, v_new as torch tensors on `device`.

    Pools above HOST_DRAW_LIMIT elements are drawn with torch's seeded
    generator on that device, in slabs; smaller ones come from host_values.
    bf16 tensors are torch.bfloat16.
    """
    import torch
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    if wl.pool_elems <= HOST_DRAW_LIMIT:
        arrs = host_values(wl, value_seed)
        out = []
        for a in arrs:
            t = torch.from_numpy(np.ascontiguousarray(a))
            if wl.dtype == "bf16":
                t = t.view(torch.int16).view(torch.bfloat16)
            out.append(t.to(device))
        return tuple(out)
    seed = wl.seed + 1000 if value_seed is None else value_seed
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    def draw(shape):
        t = torch.empty(shape, dtype=tdt, device=device)
        flat = t.view(-1)
        slab = 1 << 28
        for s in range(0, flat.numel(), slab):
            n = min(slab, flat.numel() - s)
            flat[s:s + n].copy_(torch.randn(n, generator=g, device=device, dtype=torch.float32))
        return t

    q = draw(wl.q_shape)
    k_pool = draw(wl.pool_shape)
    v_pool = draw(wl.pool_shape)
    k_new = draw(wl.new_shape)
    v_new = draw(wl.new_shape)
    return q, k_pool, v_pool, k_new, v_new


def to_numpy(t):
    """A torch tensor (fp32 or bf16, any device) -> numpy fp32 / bf16 bits."""
    import torch
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def compact_rows(wl, rows):
    """Block tables for `rows` renumbered onto a compact pool of their blocks.

    Returns (blocks, tables, slots): `blocks` lists the original block ids the
    rows use (in first-use order), `tables` is [len(rows), max_blocks] int32
    indexing into that list (padding -1), and `slots` is the rows' write slots
    renumbered the same way (a sink write maps to the compact pool's sink).
    Renumbering physical blocks is a relabelling the read must be invariant
    to, which is what lets a few sampled rows of a full-size batch be checked
    on a small host copy of the pool.
    """
    rows = list(rows)
    B = wl.block_size
    order, index = [], {}
    tables = np.full((len(rows), wl.max_blocks), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        n = (int(wl.context_lens[r]) + B - 1) // B
        for j in range(n):
            b = int(wl.block_tables[r, j])
            if b not in index:
                index[b] = len(order)
                order.append(b)
            tables[i, j] = index[b]
    nb = len(order)
    src = np.asarray(wl.write_slots)[rows]
    slots = np.empty(src.shape, dtype=np.int64)
    for i, s in np.ndenumerate(src):
        s = int(s)
        if s // B == wl.num_blocks:
            slots[i] = nb * B + s % B
        else:
            slots[i] = index[s // B] * B + s % B
    return np.asarray(order, dtype=np.int64), tables, slots
