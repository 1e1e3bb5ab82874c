"""Pins that tie the oracle to something other than itself.

Each ``pin_*`` function takes a loaded ``oracle.Oracle`` and raises
AssertionError when the oracle disagrees with what the nanoserve pages or the
mathematics fix:

  * brute force: an explicit per-key loop in Python over the row's real
    positions only (no rectangle, no mask), on tiny inputs, fp32 and bf16,
    with and without grouped KV heads;
  * closed forms: one key returns its value exactly; two keys return the
    logistic mix of their values; a constant V returns V; scale 0 returns the
    arithmetic mean of the row's values;
  * invariants: a row with context 0 gives zeros; relabelling physical blocks
    leaves every output bit unchanged; the value of a padding entry does not
    matter; NaN in a slot the rectangle gathers reaches the oracle's output
    (Day 59, "Why it matters": the reference reads the padding, then masks);
  * refusals on out-of-range inputs;
  * the KV append as a bytewise scatter;
  * the tile accounting and score-rectangle sizes printed in the Day-59
    streambench table (tests/golden/day59_streambench.txt).

``ALL_PINS`` is run against the real oracle by test_oracle_pins.py and against
deliberately broken copies of it by test_oracle_mutants.py.
"""

import math
import os

import numpy as np

from oracle import OracleRefusal
from paged_kv_decode_nsv_gb300 import workloads as wlmod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "day59_streambench.txt")


# ---------------------------------------------------------------------------
# small inputs


def _values(rng, shape, dtype):
    x = rng.standard_normal(size=shape).astype(np.float32)
    return x if dtype == "f32" else wlmod.bf16_bits(x)


def _f64(a):
    if a.dtype == np.uint16:
        return wlmod.bf16_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


def small_case(seed, dtype="f32", rows=None, heads=None, kv_heads=None,
               head_dim=None, block_size=None, lens=None, spare=3):
    """A tiny batch: random shapes unless given, blocks scattered, -1 padding."""
    rng = np.random.default_rng(seed)
    R = rows if rows is not None else int(rng.integers(1, 6))
    Hkv = kv_heads if kv_heads is not None else int(rng.choice([1, 2]))
    H = heads if heads is not None else Hkv * int(rng.choice([1, 2]))
    D = head_dim if head_dim is not None else int(rng.choice([8, 16]))
    B = block_size if block_size is not None else int(rng.choice([4, 16]))
    if lens is None:
        lens = rng.integers(0, 41, size=R)
        if R >= 2:
            lens[0] = B * 2          # block-exact length
            lens[-1] = 0             # a padded row
    lens = np.asarray(lens, dtype=np.int32)
    R = len(lens)
    nb = [(int(c) + B - 1) // B for c in lens]
    MB = max(1, max(nb) + 1)
    NB = sum(nb) + spare
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((R, MB), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(nb):
        bt[r, :n] = perm[off:off + n]
        off += n
    q = _values(rng, (R, H, D), dtype)
    k = _values(rng, (NB + 1, Hkv, B, D), dtype)
    v = _values(rng, (NB + 1, Hkv, B, D), dtype)
    scale = 1.0 / math.sqrt(D)
    return dict(q=q, k=k, v=v, bt=bt, ctx=lens, scale=scale, B=B, NB=NB)


def brute_force(q, k, v, bt, ctx, scale, B):
    """Per-key loop over the positions each query sees; fp64; no rectangle,
    no mask.  q is [R, H, D] (one query per row) or [R, NQ, H, D] (query
    token j of NQ sees the row's first ctx - NQ + 1 + j positions)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    single = q.ndim == 3
    if single:
        q = q[:, None]
    R, NQ, H, D = q.shape
    Hkv = k.shape[1]
    group = H // Hkv
    out = np.zeros((R, NQ, H, D))
    for r in range(R):
        for j in range(NQ):
            c = int(ctx[r]) - (NQ - 1 - j)
            for h in range(H):
                if c <= 0:
                    continue
                g = h // group
                keys, vals = [], []
                for t in range(c):
                    blk = int(bt[r, t // B])
                    keys.append(k[blk, g, t % B])
                    vals.append(v[blk, g, t % B])
                scores = [scale * math.fsum(q[r, j, h, d] * kk[d] for d in range(D))
                          for kk in keys]
                mx = max(scores)
                w = [math.exp(s - mx) for s in scores]
                z = math.fsum(w)
                for d in range(D):
                    out[r, j, h, d] = math.fsum(w[t] / z * vals[t][d] for t in range(c))
    return out[:, 0] if single else out


def _decode(orc, cs, **over):
    kw = dict(cs)
    kw.update(over)
    return orc.paged_decode(kw["q"], kw["k"], kw["v"], kw["bt"], kw["ctx"], kw["scale"])


# ---------------------------------------------------------------------------
# pins


def pin_brute_force(orc):
    for seed in range(8):
        for dtype in ("f32", "bf16"):
            cs = small_case(100 + seed, dtype)
            got = _decode(orc, cs)
            ref = brute_force(cs["q"], cs["k"], cs["v"], cs["bt"], cs["ctx"], cs["scale"], cs["B"])
            err = float(np.max(np.abs(got - ref))) if got.size else 0.0
            assert err <= 1e-12, "seed %d %s: oracle vs brute force %.3g" % (seed, dtype, err)


def pin_gqa_brute_force(orc):
    # 4 query heads per KV head, and every query head on a single KV head
    for seed, heads, kv_heads in ((7, 8, 2), (8, 8, 1)):
        cs = small_case(seed, "f32", rows=3, heads=heads, kv_heads=kv_heads, head_dim=8,
                        block_size=4, lens=[5, 13, 9])
        got = _decode(orc, cs)
        ref = brute_force(cs["q"], cs["k"], cs["v"], cs["bt"], cs["ctx"], cs["scale"], cs["B"])
        assert np.max(np.abs(got - ref)) <= 1e-12, (heads, kv_heads)


def _mq_case(seed, nq, dtype="f32", lens=None, heads=2, kv_heads=2):
    cs = small_case(seed, dtype, heads=heads, kv_heads=kv_heads, head_dim=8, block_size=4,
                    lens=lens)
    rng = np.random.default_rng(seed + 7)
    R, H, D = cs["q"].shape
    cs["q"] = _values(rng, (R, nq, H, D), dtype)
    return cs


def pin_multiquery_brute_force(orc):
    for seed, nq, dtype in ((30, 2, "f32"), (31, 3, "bf16"), (32, 4, "f32")):
        cs = _mq_case(seed, nq, dtype, lens=[1, 2, 5, 11, 0, 17], heads=4, kv_heads=2)
        got = _decode(orc, cs)
        ref = brute_force(cs["q"], cs["k"], cs["v"], cs["bt"], cs["ctx"], cs["scale"], cs["B"])
        assert got.shape == ref.shape
        assert np.max(np.abs(got - ref)) <= 1e-12, "multi-query oracle vs brute force"


def pin_multiquery_last_token_is_the_decode_read(orc):
    cs = _mq_case(33, 3, "bf16", lens=[7, 3, 20, 9])
    got = _decode(orc, cs)
    single = _decode(orc, cs, q=np.ascontiguousarray(cs["q"][:, -1]))
    assert np.array_equal(got[:, -1], single)


def pin_multiquery_first_token_sees_one_key(orc):
    nq = 3
    cs = _mq_case(34, nq, "f32", lens=[nq, nq, nq])
    got = _decode(orc, cs)
    v = _f64(cs["v"])
    for r in range(3):
        blk = int(cs["bt"][r, 0])
        for h in range(2):
            assert np.array_equal(got[r, 0, h], v[blk, h, 0]), "query 0 sees position 0 only"


def pin_multiquery_is_causal(orc):
    """Changing the value at position p leaves every query that cannot see p
    bit-identical and changes the ones that can."""
    nq = 4
    cs = _mq_case(35, nq, "f32", lens=[13])
    base = _decode(orc, cs)
    p = 13 - 2                     # seen by queries j with 13 - 3 + j > p, i.e. j >= 2
    v2 = cs["v"].copy()
    v2[int(cs["bt"][0, p // 4]), :, p % 4, :] += 1.0
    got = _decode(orc, cs, v=v2)
    assert np.array_equal(got[0, :2], base[0, :2])
    assert np.all(np.abs(got[0, 2:] - base[0, 2:]).max(axis=-1) > 0)


def pin_multiquery_short_row(orc):
    nq = 4
    cs = _mq_case(36, nq, "f32", lens=[2])
    got = _decode(orc, cs)
    assert np.all(got[0, :2] == 0.0), "queries that see no position output 0"
    assert np.any(got[0, 2:] != 0.0)


def _slots_from_tables(bt, B):
    """The slot table the reference builds from block tables: slot of
    position t = table[t / B] * B + t % B; padding entries stay negative."""
    R, MB = bt.shape
    t = np.arange(MB * B)
    blk = bt[:, t // B].astype(np.int64)
    return np.where(blk >= 0, blk * B + t % B, -1).astype(np.int64)


def brute_force_slots(q, k, v, slots, ctx, scale, B):
    """Per-key loop through a slot table; fp64; q [R, H, D]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    R, H, D = q.shape
    group = H // k.shape[1]
    out = np.zeros((R, H, D))
    for r in range(R):
        c = int(ctx[r])
        for h in range(H):
            if c == 0:
                continue
            g = h // group
            kk = [k[int(slots[r, t]) // B, g, int(slots[r, t]) % B] for t in range(c)]
            vv = [v[int(slots[r, t]) // B, g, int(slots[r, t]) % B] for t in range(c)]
            sc = [scale * math.fsum(q[r, h, d] * x[d] for d in range(D)) for x in kk]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            z = math.fsum(w)
            for d in range(D):
                out[r, h, d] = math.fsum(w[t] / z * vv[t][d] for t in range(c))
    return out


def pin_slots_equal_block_tables(orc):
    """A slot table built from the block tables reads what the block tables
    read, bit for bit (same gathered rectangle, same arithmetic)."""
    for dtype in ("f32", "bf16"):
        cs = small_case(40, dtype, rows=4, heads=4, kv_heads=2, head_dim=8, block_size=4,
                        lens=[3, 0, 14, 8])
        base = _decode(orc, cs)
        slots = _slots_from_tables(cs["bt"], cs["B"])
        got = orc.paged_decode_slots(cs["q"], cs["k"], cs["v"], slots, slots.shape[1],
                                     cs["ctx"], cs["scale"])
        assert np.array_equal(got, base)


def pin_slots_brute_force(orc):
    """Arbitrary per-token slots (not grouped into blocks) against a per-key
    loop; a wider table (row stride > width) is read only up to the width."""
    rng = np.random.default_rng(41)
    cs = small_case(41, "f32", rows=3, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[5, 9, 1], spare=6)
    nslots = cs["k"].shape[0] * 4
    width, stride = 12, 20
    slots = np.full((3, stride), 10 ** 9, dtype=np.int64)   # past the width: never read
    for r in range(3):
        slots[r, :width] = rng.choice(nslots, size=width, replace=False)
    got = orc.paged_decode_slots(cs["q"], cs["k"], cs["v"], slots, width, cs["ctx"],
                                 cs["scale"])
    ref = brute_force_slots(cs["q"], cs["k"], cs["v"], slots, cs["ctx"], cs["scale"], 4)
    assert np.max(np.abs(got - ref)) <= 1e-12


def pin_slots_rectangle_reads_padding(orc):
    """A -1 slot wraps onto the pool's last slot (the sink block's); NaN there
    reaches the oracle's output because the rectangle gathers its padding."""
    cs = small_case(43, "f32", rows=2, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[5, 6])
    slots = _slots_from_tables(cs["bt"], 4)
    assert np.all(slots[:, -1] == -1)
    clean = orc.paged_decode_slots(cs["q"], cs["k"], cs["v"], slots, slots.shape[1],
                                   cs["ctx"], cs["scale"])
    assert np.all(np.isfinite(clean))
    v = cs["v"].copy()
    v[-1, :, -1, :] = np.nan
    got = orc.paged_decode_slots(cs["q"], cs["k"], v, slots, slots.shape[1], cs["ctx"],
                                 cs["scale"])
    assert np.all(np.isnan(got))


def pin_slots_refusals(orc):
    cs = small_case(42, "f32", rows=2, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[3, 6])
    slots = _slots_from_tables(cs["bt"], 4)
    nslots = cs["k"].shape[0] * 4
    for bad in (nslots, -nslots - 1):
        s2 = slots.copy()
        s2[1, 2] = bad
        try:
            orc.paged_decode_slots(cs["q"], cs["k"], cs["v"], s2, s2.shape[1], cs["ctx"], 1.0)
        except OracleRefusal as e:
            assert e.code == -5
        else:
            raise AssertionError("slot %d must be refused" % bad)
    try:
        orc.paged_decode_slots(cs["q"], cs["k"], cs["v"], slots, slots.shape[1] + 1,
                               cs["ctx"], 1.0)
    except OracleRefusal as e:
        assert e.code == -3
    else:
        raise AssertionError("a width past the row stride must be refused")


def pin_single_key(orc):
    for dtype in ("f32", "bf16"):
        cs = small_case(11, dtype, rows=3, heads=2, kv_heads=2, head_dim=16, block_size=4,
                        lens=[1, 1, 1])
        got = _decode(orc, cs)
        v = _f64(cs["v"])
        for r in range(3):
            blk = int(cs["bt"][r, 0])
            for h in range(2):
                assert np.array_equal(got[r, h], v[blk, h, 0]), "one key must return its value"


def pin_two_keys_closed_form(orc):
    cs = small_case(12, "f32", rows=2, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[2, 2])
    got = _decode(orc, cs)
    q, k, v = _f64(cs["q"]), _f64(cs["k"]), _f64(cs["v"])
    for r in range(2):
        blk = int(cs["bt"][r, 0])
        for h in range(2):
            s0 = cs["scale"] * float(q[r, h] @ k[blk, h, 0])
            s1 = cs["scale"] * float(q[r, h] @ k[blk, h, 1])
            p0 = 1.0 / (1.0 + math.exp(s1 - s0))
            want = p0 * v[blk, h, 0] + (1.0 - p0) * v[blk, h, 1]
            assert np.max(np.abs(got[r, h] - want)) <= 1e-13


def pin_constant_v(orc):
    cs = small_case(13, "f32", rows=4, heads=4, kv_heads=2, head_dim=8, block_size=4,
                    lens=[3, 17, 30, 8])
    c = np.random.default_rng(5).standard_normal((2, 8)).astype(np.float32)
    v = np.empty_like(cs["v"])
    v[:] = c[None, :, None, :]
    got = _decode(orc, cs, v=v)
    for h in range(4):
        want = c[h // 2].astype(np.float64)
        assert np.max(np.abs(got[:, h] - want[None, :])) <= 1e-13, "constant V must return V"


def pin_scale_zero_is_mean(orc):
    cs = small_case(14, "bf16", rows=3, heads=2, kv_heads=1, head_dim=8, block_size=4,
                    lens=[7, 12, 1])
    got = _decode(orc, cs, scale=0.0)
    v = _f64(cs["v"])
    for r in range(3):
        c = int(cs["ctx"][r])
        rows = [v[int(cs["bt"][r, t // 4]), 0, t % 4] for t in range(c)]
        mean = np.mean(np.stack(rows), axis=0)
        for h in range(2):
            assert np.max(np.abs(got[r, h] - mean)) <= 1e-13, "scale 0 must give the mean of V"


def pin_ctx_zero(orc):
    cs = small_case(15, "f32", rows=3, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[0, 9, 0])
    got = _decode(orc, cs)
    assert np.all(got[0] == 0.0) and np.all(got[2] == 0.0)
    assert np.any(got[1] != 0.0)


def pin_permutation_invariance(orc):
    cs = small_case(16, "bf16", rows=4, heads=2, kv_heads=2, head_dim=16, block_size=4)
    base = _decode(orc, cs)
    NB1 = cs["k"].shape[0]
    rng = np.random.default_rng(3)
    perm = np.arange(NB1)
    perm[:NB1 - 1] = rng.permutation(NB1 - 1)     # keep the sink block in place
    k2 = np.empty_like(cs["k"])
    v2 = np.empty_like(cs["v"])
    k2[perm] = cs["k"]
    v2[perm] = cs["v"]
    bt2 = np.where(cs["bt"] >= 0, perm[np.maximum(cs["bt"], 0)], -1).astype(np.int32)
    got = _decode(orc, cs, k=k2, v=v2, bt=bt2)
    assert np.array_equal(got, base), "relabelling blocks must not change one bit"


def pin_padding_value_irrelevant(orc):
    cs = small_case(17, "f32", rows=3, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[5, 2, 11])
    base = _decode(orc, cs)
    bt2 = np.where(cs["bt"] >= 0, cs["bt"], 0).astype(np.int32)   # pad with block 0
    got = _decode(orc, cs, bt=bt2)
    assert np.array_equal(got, base)


def pin_rectangle_reads_padding(orc):
    """NaN in the block a -1 entry wraps to reaches the oracle's output."""
    cs = small_case(18, "f32", rows=2, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[5, 6])
    clean = _decode(orc, cs)
    assert np.all(np.isfinite(clean))
    v = cs["v"].copy()
    v[-1] = np.nan                     # the sink block: where -1 wraps to
    got = _decode(orc, cs, v=v)
    assert np.all(np.isnan(got)), "the rectangle read gathers its padding, so NaN must reach it"


def pin_refusals(orc):
    cs = small_case(19, "f32", rows=2, heads=2, kv_heads=2, head_dim=8, block_size=4,
                    lens=[5, 6])
    W = cs["bt"].shape[1] * 4
    for bad in ([W + 1, 6], [-1, 6]):
        try:
            _decode(orc, cs, ctx=np.array(bad, dtype=np.int32))
        except OracleRefusal as e:
            assert e.code == -5
        else:
            raise AssertionError("context length %r must be refused" % (bad,))
    NB1 = cs["k"].shape[0]
    for badblk in (NB1, -NB1 - 1):
        bt = cs["bt"].copy()
        bt[1, 0] = badblk
        try:
            _decode(orc, cs, bt=bt)
        except OracleRefusal as e:
            assert e.code == -5
        else:
            raise AssertionError("block id %d must be refused" % badblk)
    try:
        orc.paged_decode(np.zeros((2, 3, 8), np.float32), cs["k"], cs["v"], cs["bt"],
                         cs["ctx"], 1.0)
    except OracleRefusal as e:
        assert e.code == -3
    else:
        raise AssertionError("heads not a multiple of kv_heads must be refused")


def pin_kv_write(orc):
    for dtype in ("f32", "bf16"):
        rng = np.random.default_rng(20)
        NB, Hkv, B, D = 6, 2, 4, 8
        k = _values(rng, (NB + 1, Hkv, B, D), dtype)
        v = _values(rng, (NB + 1, Hkv, B, D), dtype)
        kn = _values(rng, (4, Hkv, D), dtype)
        vn = _values(rng, (4, Hkv, D), dtype)
        slots = np.array([5, 22, NB * B, NB * B + 3], dtype=np.int64)
        k2, v2 = k.copy(), v.copy()
        orc.kv_write(kn, vn, slots, k2, v2)
        kw, vw = k.copy(), v.copy()
        for r, s in enumerate(slots):
            kw[s // B, :, s % B, :] = kn[r]
            vw[s // B, :, s % B, :] = vn[r]
        assert np.array_equal(k2, kw) and np.array_equal(v2, vw)
        assert np.array_equal(k2[:NB], k[:NB]) is False   # something real was written
        k3, v3 = k.copy(), v.copy()
        try:
            orc.kv_write(kn, vn, np.array([5, (NB + 1) * B, 0, 1], np.int64), k3, v3)
        except OracleRefusal as e:
            assert e.code == -5
        else:
            raise AssertionError("a slot past the sink block must be refused")
        assert np.array_equal(k3, k) and np.array_equal(v3, v), "a refusal writes nothing"


def load_golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            r, w, spread, rect_mb, tile_mb, walked, rect = line.split()
            rows.append(dict(rows=int(r), width=int(w), spread=spread.replace("_", " "),
                             rect_mb=float(rect_mb), tile_mb=float(tile_mb),
                             walked=int(walked), rect_tiles=int(rect)))
    return rows


def pin_walk_table(orc):
    for g in load_golden():
        lens = wlmod.spread_lengths(g["rows"], g["width"], g["spread"])
        assert orc.walked_tiles(lens, 128) == g["walked"], g
        assert orc.rect_tiles(g["rows"], g["width"], 128) == g["rect_tiles"], g


def pin_walk_counts_tiles_touched(orc):
    """A walked tile is one that holds at least one real position (ragged lengths)."""
    rng = np.random.default_rng(21)
    for tile in (16, 128):
        lens = rng.integers(0, 5 * tile, size=40).astype(np.int32)
        lens[:4] = [0, 1, tile, tile + 1]
        touched = sum(1 for c in lens for start in range(0, 5 * tile, tile) if start < c)
        assert orc.walked_tiles(lens, tile) == touched
        assert orc.rect_tiles(len(lens), 5 * tile, tile) == 5 * len(lens)


def pin_score_bytes(orc):
    for g in load_golden():
        rect = orc.score_rect_bytes(g["rows"], 32, g["width"]) / 1e6
        tile = orc.score_tile_bytes(g["rows"], 32, 128) / 1e6
        assert round(rect, 1) == g["rect_mb"], (g, rect)
        assert round(tile, 2) == g["tile_mb"], (g, tile)


ALL_PINS = [
    pin_brute_force, pin_gqa_brute_force, pin_single_key, pin_two_keys_closed_form,
    pin_constant_v, pin_scale_zero_is_mean, pin_ctx_zero, pin_permutation_invariance,
    pin_padding_value_irrelevant, pin_rectangle_reads_padding, pin_refusals,
    pin_kv_write, pin_walk_table, pin_walk_counts_tiles_touched, pin_score_bytes,
    pin_multiquery_brute_force, pin_multiquery_last_token_is_the_decode_read,
    pin_multiquery_first_token_sees_one_key, pin_multiquery_is_causal, pin_multiquery_short_row,
    pin_slots_equal_block_tables, pin_slots_brute_force, pin_slots_rectangle_reads_padding,
    pin_slots_refusals,
]
