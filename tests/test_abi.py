"""The C-ABI library on the CPU: it loads, exports exactly what include/nsv.h
declares, plans deterministically, and refuses bad host-visible arguments
before touching any device (none of these calls needs a GPU)."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nsv.h")


@pytest.fixture(scope="module")
def nsv():
    from paged_kv_decode_nsv_gb300 import build
    build.build()
    from paged_kv_decode_nsv_gb300 import nsv as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"NSV_API\s+[\w\s\*]+?\b(nsv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("nsv_kv_write", "nsv_paged_decode", "nsv_plan_split"):
        assert required in names


def test_library_exports_every_declared_symbol(nsv):
    lib = ctypes.CDLL(nsv.lib_path())
    for name in declared_functions():
        assert hasattr(lib, name), "libnsv.so does not export %s" % name


def test_library_exports_nothing_else(nsv):
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", nsv.lib_path()], check=True,
                         capture_output=True, text=True).stdout
    funcs = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert funcs == set(declared_functions()), funcs ^ set(declared_functions())


def test_abi_version_and_strerror(nsv):
    assert nsv.abi_version() == nsv.ABI_VERSION == 102
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -10):
        assert nsv.strerror(code) and "unknown" not in nsv.strerror(code)
    assert "unknown" in nsv.strerror(-99)


def _cta_warps(nsv, consumer, consumer_warps, head_dim=128):
    """Warps of a planned CTA: the producer and the consumers, plus, with the
    vectors as the MMA rows at head_dim 128, an idle warp at each multiple of
    4 the consumers pass (none shares the producer's sub-partition)."""
    if consumer == nsv.CONSUMER_TENSOR_TMEM:
        return 10     # a producer, eight softmax warps and an MMA warp
    if consumer == nsv.CONSUMER_TENSOR_VECTOR_ROWS and head_dim == 128:
        return consumer_warps + 1 + (consumer_warps - 1) // 3
    return consumer_warps + 1


def _shape(nsv, **kw):
    d = dict(rows=256, num_heads=32, num_kv_heads=32, head_dim=128, max_blocks=512,
             num_blocks=70000, dtype=nsv.BF16, query_len=1)
    d.update(kw)
    return nsv.make_shape(**d)


def test_plan_headline_shape(nsv):
    p = nsv.plan_split(_shape(nsv), num_sms=152)
    assert p.kv_heads_per_cta == 8 and p.threads == 9 * 32
    assert p.stages == 3 and p.ctas_per_sm == 1 and p.grid == 152
    assert p.smem_bytes <= 227 * 1024
    slots = 152 * 2 * 8                      # two partials per CTA, 8 query heads
    counters = 256 * (32 // 8) * 4           # one per (row, head group)
    want = -(-counters // 256) * 256 + -(-slots * 8 // 256) * 256 + slots * 128 * 4
    assert p.workspace_bytes == want
    again = nsv.plan_split(_shape(nsv), num_sms=152)
    assert bytes(again) == bytes(p), "planning must be deterministic"


def test_plan_shapes_of_every_workload(nsv):
    from paged_kv_decode_nsv_gb300 import workloads as W
    for name, make in W.WORKLOADS.items():
        wl = make()
        shape = nsv.make_shape(wl.rows, wl.heads, wl.kv_heads, wl.head_dim, wl.max_blocks,
                               wl.num_blocks, nsv.F32 if wl.dtype == "f32" else nsv.BF16,
                               query_len=wl.query_len)
        p = nsv.plan_split(shape, num_sms=152)
        assert p.grid == 152 * p.ctas_per_sm
        assert p.smem_bytes <= 227 * 1024
        nvec = p.kv_heads_per_cta * (wl.heads // wl.kv_heads) * wl.query_len
        assert 0 < p.workspace_bytes < p.grid * 2 * nvec * (wl.head_dim * 4 + 8) + (1 << 16)
        assert wl.kv_heads % p.kv_heads_per_cta == 0
        vpk = (wl.heads // wl.kv_heads) * wl.query_len
        if p.consumer != nsv.CONSUMER_CUDA:  # one warp per 8 or per 16 vectors of a KV head
            wpk = -(-vpk // (8 if p.consumer == nsv.CONSUMER_TENSOR else 16))
            assert p.vectors_per_warp == 1
            assert p.threads // 32 == _cta_warps(nsv, p.consumer, p.kv_heads_per_cta * wpk,
                                                 wl.head_dim)
        else:
            assert p.consumer == nsv.CONSUMER_CUDA
            assert (p.threads // 32 - 1) * p.vectors_per_warp == nvec


@pytest.mark.parametrize("heads,kv_heads,qlen,qw,warps", [
    (32, 32, 1, 1, 8), (32, 8, 1, 2, 8), (32, 32, 4, 2, 8), (32, 32, 2, 2, 8),
    (32, 32, 3, 1, 3), (16, 1, 1, 2, 8), (32, 8, 8, 2, 16), (8, 8, 5, 1, 5),
])
def test_plan_query_vectors(nsv, heads, kv_heads, qlen, qw, warps):
    """On the CUDA cores a consumer warp serves two query vectors by default
    when the vectors per KV head (query heads per KV head x tokens) pair up,
    else one."""
    p = nsv.plan_custom(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen),
                        num_sms=152, consumer=nsv.CONSUMER_CUDA)
    assert p.consumer == nsv.CONSUMER_CUDA
    assert p.vectors_per_warp == qw
    assert p.threads == (warps + 1) * 32


@pytest.mark.parametrize("heads,kv_heads,qlen,head_dim,consumer,group,cps", [
    (32, 32, 1, 128, 1, 8, 1),   # 64 KiB stages: one CTA of 8 warps per SM
    (32, 8, 1, 128, 2, 8, 1),
    (1, 1, 1, 128, 1, 1, 8),     # one KV head: as many small CTAs as fit (2 stages)
    (2, 2, 1, 128, 1, 2, 5),
    (16, 4, 1, 128, 2, 2, 3),    # 3 CTAs of 2 warps beat 1 of 4
    (8, 2, 2, 64, 2, 2, 5),      # head_dim 64 tokens-as-rows warps fit 4 per sub-partition
    (8, 8, 1, 64, 1, 8, 2),      # 16 warps either way: the larger group
    (8, 1, 1, 128, 2, 1, 6),
])
def test_plan_keeps_consumer_warps_resident(nsv, heads, kv_heads, qlen, head_dim, consumer,
                                            group, cps):
    """The default group is the one whose plan keeps the most consumer warps
    resident per SM (counted up to 16), the larger on a tie, and the default
    CTAs per SM are as many as fit (up to 8)."""
    p = nsv.plan_split(_shape(nsv, rows=512, num_blocks=200000, num_heads=heads,
                              num_kv_heads=kv_heads, query_len=qlen, head_dim=head_dim),
                       num_sms=152)
    assert (p.consumer, p.kv_heads_per_cta, p.ctas_per_sm) == (consumer, group, cps)
    assert p.grid == 152 * cps


@pytest.mark.parametrize("heads,kv_heads,head_dim,stages,cps", [
    (1, 1, 128, 2, 8), (2, 2, 128, 2, 5),   # every KV head in one small-stage CTA
    (4, 4, 128, 3, 2),                      # 32 KiB stages keep 3
    (32, 32, 128, 3, 1),                    # a group of 8 out of 32 keeps 3
])
def test_cuda_core_small_stage_ring(nsv, heads, kv_heads, head_dim, stages, cps):
    """A CUDA-core CTA that streams every KV head in stages of at most 16 KiB
    takes a 2-stage ring where that fits more CTAs per SM."""
    p = nsv.plan_split(_shape(nsv, rows=512, num_blocks=200000, num_heads=heads,
                              num_kv_heads=kv_heads, head_dim=head_dim), num_sms=152)
    assert p.consumer == nsv.CONSUMER_CUDA
    assert (p.stages, p.ctas_per_sm) == (stages, cps)


@pytest.mark.parametrize("heads,kv_heads,qlen,dtype", [
    (32, 8, 17, 1), (128, 1, 1, 1), (64, 2, 3, 1),   # more than 64 vectors per KV head
    (32, 8, 9, 0), (68, 2, 1, 0),     # fp32 (CUDA cores): more than 32
    (32, 32, 17, 0),   # fp32: an odd count above 15 needs 17 warps
])
def test_plan_refuses_too_many_query_vectors(nsv, heads, kv_heads, qlen, dtype):
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_split(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen,
                              dtype=dtype), num_sms=152)
    assert e.value.code == -3


def test_odd_vector_counts_above_15_run_on_the_tensor_cores(nsv):
    # 32 KV heads split into the TMEM form's groups of 2 (17 vectors each; a
    # group's P.V output, group x head_dim columns, is one MMA wide)
    p = nsv.plan_split(_shape(nsv, query_len=17), num_sms=152)
    assert p.consumer == nsv.CONSUMER_TENSOR_TMEM and p.kv_heads_per_cta == 2
    # 5 KV heads split into no group of 2 or 4: two vectors-as-rows warps per KV head
    p = nsv.plan_split(_shape(nsv, num_heads=5, num_kv_heads=5, query_len=17), num_sms=152)
    assert p.consumer == nsv.CONSUMER_TENSOR_VECTOR_ROWS
    assert p.threads == _cta_warps(nsv, p.consumer, p.kv_heads_per_cta * 2) * 32


def _tmem_cols(head_dim, group, blocks):
    used = group * head_dim + 2 * blocks * group * 16 + head_dim // 2
    return next(c for c in (32, 64, 128, 256, 512) if used <= c)


@pytest.mark.parametrize("heads,kv_heads,qlen,head_dim,group,blocks,stages,cps", [
    (32, 8, 8, 128, 2, 3, 4, 1), (64, 8, 8, 128, 2, 3, 4, 1), (32, 8, 1, 128, 2, 3, 4, 1),
    (32, 8, 9, 128, 2, 3, 4, 1), (8, 8, 17, 128, 2, 3, 4, 1), (32, 8, 8, 64, 2, 4, 5, 1),
    (64, 8, 8, 64, 2, 4, 5, 1), (24, 6, 5, 128, 2, 3, 4, 1), (64, 1, 1, 128, 1, 4, 5, 1),
    (20, 5, 5, 64, 1, 4, 6, 1)])
def test_plan_tmem_form(nsv, heads, kv_heads, qlen, head_dim, group, blocks, stages, cps):
    """NSV_CONSUMER_TENSOR_TMEM: one 128-row MMA group per CTA (the largest of
    4, 2 or 1 KV heads that divides the KV heads, leaves each head rows for
    its vectors, keeps group x head_dim within one MMA's 256 columns and
    leaves tensor memory for stages of 3 blocks), a producer, eight softmax
    warps and an MMA warp, one CTA per SM; stages of 1 to 4 blocks: the
    largest that leaves a ring of 3, with the deepest ring (up to 6) that
    fits.  Tensor memory holds O, two score buffers and the query rows."""
    p = nsv.plan_custom(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen,
                               head_dim=head_dim),
                        num_sms=152, consumer=nsv.CONSUMER_TENSOR_TMEM)
    assert p.consumer == nsv.CONSUMER_TENSOR_TMEM and p.kv_heads_per_cta == group
    assert p.threads == 10 * 32 and p.vectors_per_warp == 1
    assert (p.blocks_per_stage, p.stages) == (blocks, stages)
    assert p.ctas_per_sm == cps and p.grid == 152 * cps
    assert p.smem_bytes <= 227 * 1024 and cps * (p.smem_bytes + 1024) <= 228 * 1024
    assert cps * _tmem_cols(head_dim, group, blocks) <= 512
    assert blocks * group * 16 <= 256 and group * head_dim <= 256


@pytest.mark.parametrize("qlen,warps", [(2, 1), (16, 1), (17, 2), (32, 2)])
def test_plan_vector_rows_form(nsv, qlen, warps):
    """NSV_CONSUMER_TENSOR_VECTOR_ROWS: one warp per 16 vectors of a KV head."""
    p = nsv.plan_custom(_shape(nsv, query_len=qlen), num_sms=152,
                        consumer=nsv.CONSUMER_TENSOR_VECTOR_ROWS)
    assert p.consumer == nsv.CONSUMER_TENSOR_VECTOR_ROWS
    assert p.threads == _cta_warps(nsv, p.consumer, p.kv_heads_per_cta * warps) * 32


@pytest.mark.parametrize("heads,kv_heads,qlen,dtype,consumer,hg,warps", [
    (32, 32, 1, "bf16", 1, 8, 8),    # one vector per KV head: CUDA cores
    (32, 8, 1, "bf16", 2, 8, 8),     # 4 query heads per KV head: tensor cores
    (32, 32, 4, "bf16", 2, 8, 8),    # 4 query tokens
    (32, 32, 3, "bf16", 2, 8, 8),
    (16, 1, 1, "bf16", 3, 1, 1),     # 16 vectors: one warp, vectors as the MMA rows
    (32, 8, 8, "bf16", 4, 2, 10),    # 32 vectors: tcgen05, 2 KV heads of 64 rows
    (32, 8, 5, "bf16", 4, 2, 10),    # 20 vectors
    (64, 8, 8, "bf16", 4, 2, 10),    # 64 vectors: 2 KV heads of 64 rows
    (24, 6, 5, "bf16", 4, 2, 10),    # 20 vectors, 6 KV heads: groups of 2 (64 rows each)
    (20, 5, 5, "bf16", 3, 1, 2),     # 20 vectors, 5 KV heads: no group of 2 or 4
    (32, 8, 1, "f32", 1, 4, 8),      # fp32 stays on the CUDA cores
])
def test_plan_consumer_choice(nsv, heads, kv_heads, qlen, dtype, consumer, hg, warps):
    """The default plan runs bf16 shapes with 2 or more query vectors per KV
    head on the tensor cores: up to 8 with the tokens as the MMA rows (one
    warp per KV head), 9 to 16 with the vectors as the rows (16 per warp),
    beyond with tcgen05 into tensor memory where the KV heads split into its
    groups (else the vectors as the rows)."""
    p = nsv.plan_split(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen,
                              dtype=nsv.BF16 if dtype == "bf16" else nsv.F32), num_sms=152)
    assert p.consumer == consumer and p.kv_heads_per_cta == hg
    assert p.threads == _cta_warps(nsv, consumer, warps) * 32
    if consumer != nsv.CONSUMER_CUDA:
        assert p.vectors_per_warp == 1
    assert (p.blocks_per_stage > 1) == (consumer == nsv.CONSUMER_TENSOR_TMEM)


@pytest.mark.parametrize("kw,ckw", [
    (dict(num_kv_heads=32), dict(consumer=2)),                      # 1 vector per KV head
    (dict(num_kv_heads=8, dtype=1), dict(consumer=2, vectors_per_warp=2)),
    (dict(num_kv_heads=8, dtype=0), dict(consumer=2)),              # fp32
    (dict(num_kv_heads=8), dict(consumer=5)),                       # no such consumer
    (dict(num_kv_heads=8, dtype=0), dict(consumer=4)),              # fp32
    (dict(num_heads=24, num_kv_heads=6), dict(consumer=4, kv_heads_per_cta=4)),  # 4 does not divide 6
    (dict(num_kv_heads=8, query_len=9), dict(consumer=4, kv_heads_per_cta=4)),   # 4 x 36 rows > 128
    (dict(num_kv_heads=8), dict(consumer=4, kv_heads_per_cta=8)),   # its group is 4 heads at most
    (dict(num_kv_heads=8, num_heads=64), dict(consumer=4, kv_heads_per_cta=4)),  # 4 x 128 > 256 columns
    (dict(num_kv_heads=8, num_heads=64), dict(consumer=4, blocks_per_stage=5)),  # at most 4 blocks
    (dict(num_kv_heads=8, num_heads=64, head_dim=64), dict(consumer=4, kv_heads_per_cta=4,
                                                          blocks_per_stage=3)),   # 640 TMEM columns
    (dict(num_kv_heads=8), dict(consumer=2, blocks_per_stage=2)),   # one block per stage
    (dict(num_kv_heads=8, num_heads=64), dict(consumer=4, ctas_per_sm=2)),  # one CTA per SM
    (dict(num_kv_heads=8, dtype=0), dict(consumer=3)),              # fp32
    (dict(num_kv_heads=8, num_blocks=(1 << 24)), dict(consumer=2)), # TMA row index overflows
])
def test_plan_tensor_consumer_refusals(nsv, kw, ckw):
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_custom(_shape(nsv, **kw), num_sms=152, **ckw)
    assert e.value.code == -5


def test_plan_tensor_consumer_needs_32bit_rows(nsv):
    """Where the pools have 2^31 or more 16-token tile rows the default plan
    keeps the CUDA-core consumer."""
    p = nsv.plan_split(_shape(nsv, num_kv_heads=8, num_blocks=(1 << 24)), num_sms=152)
    assert p.consumer == nsv.CONSUMER_CUDA
    p = nsv.plan_split(_shape(nsv, num_kv_heads=8, num_blocks=(1 << 24) - 2), num_sms=152)
    assert p.consumer == nsv.CONSUMER_TENSOR


def test_plan_four_vectors_per_warp_on_request(nsv):
    p = nsv.plan_custom(_shape(nsv, num_kv_heads=8), num_sms=152, vectors_per_warp=4)
    assert p.vectors_per_warp == 4 and p.threads == 9 * 32
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_custom(_shape(nsv, num_kv_heads=32, query_len=2), num_sms=152,
                        vectors_per_warp=4)
    assert e.value.code == -5


def test_plan_custom_choices(nsv):
    p = nsv.plan_custom(_shape(nsv), num_sms=152, kv_heads_per_cta=2, stages=5,
                        ctas_per_sm=2, grid=77)
    assert (p.kv_heads_per_cta, p.stages, p.ctas_per_sm, p.grid) == (2, 5, 2, 77)
    assert p.threads == 3 * 32


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), -10), (dict(head_dim=256), -10), (dict(dtype=7), -2),
    (dict(num_heads=30, num_kv_heads=8), -3), (dict(rows=-1), -3), (dict(rows=8193), -3),
    (dict(max_blocks=0), -3), (dict(num_blocks=0), -3),
    (dict(num_heads=130, num_kv_heads=2), -3),   # 65 query heads per KV head
    (dict(query_len=65), -3),
])
def test_shape_refusals(nsv, kw, code):
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_split(_shape(nsv, **kw), num_sms=152)
    assert e.value.code == code


def test_block_size_refusal(nsv):
    s = _shape(nsv)
    s.block_size = 32
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_split(s, num_sms=152)
    assert e.value.code == -10


@pytest.mark.parametrize("kw", [dict(kv_heads_per_cta=3), dict(stages=1), dict(stages=9),
                                dict(ctas_per_sm=9), dict(kv_heads_per_cta=8, ctas_per_sm=2),
                                dict(kv_heads_per_cta=32, stages=8),
                                dict(kv_heads_per_cta=8, stages=4), dict(grid=70000)])
def test_plan_custom_refusals(nsv, kw):
    with pytest.raises(nsv.NsvError) as e:
        nsv.plan_custom(_shape(nsv), num_sms=152, **kw)
    assert e.value.code == -5


def test_null_and_misaligned_pointers_refused_before_any_device_call(nsv):
    lib = nsv._lib
    s = _shape(nsv)
    fake = ctypes.c_void_p(0x100000)
    odd = ctypes.c_void_p(0x100008)
    args = [fake, fake, fake, fake, fake]
    rc = lib.nsv_paged_decode(ctypes.byref(s), None, *args[:4], 1.0, fake, None)
    assert rc == -1
    rc = lib.nsv_paged_decode(ctypes.byref(s), odd, fake, fake, fake, fake, 1.0, fake, None)
    assert rc == -4
    rc = lib.nsv_kv_write(ctypes.byref(s), fake, fake, ctypes.c_void_p(0x100004), fake, fake,
                          None)
    assert rc == -4
    rc = lib.nsv_kv_write(None, fake, fake, fake, fake, fake, None)
    assert rc == -1


def test_status_async_refuses_null_and_misaligned_destinations(nsv):
    lib = nsv._lib
    assert lib.nsv_status_async(None, 1, None) == -1
    assert lib.nsv_status_async(ctypes.c_void_p(0x100002), 1, None) == -4


def test_tampered_plan_refused_before_any_device_call(nsv):
    lib = nsv._lib
    s = _shape(nsv)
    p = nsv.plan_split(s, num_sms=152)
    p.smem_bytes += 16          # not what the planner made for these choices
    fake = ctypes.c_void_p(0x100000)
    rc = lib.nsv_paged_decode_ws(ctypes.byref(s), ctypes.byref(p), fake, fake, fake, fake, fake,
                                 1.0, fake, fake, 1 << 30, None)
    assert rc == -5


@pytest.mark.parametrize("limit", [0, 999, 2000000001])
def test_bounded_wait_selftest_refuses_limits_out_of_range(nsv, limit):
    """Checked on the host before any device call."""
    g, w = ctypes.c_int(0), ctypes.c_uint64(0)
    rc = nsv._lib.nsv_selftest_bounded_wait(limit, ctypes.byref(g), ctypes.byref(w), None)
    assert rc == -5


def test_bounded_wait_selftest_refuses_null_results(nsv):
    assert nsv._lib.nsv_selftest_bounded_wait(1000000, None, None, None) == -1


@pytest.mark.parametrize("kw,regs", [
    (dict(), 96), (dict(num_kv_heads=8), 168), (dict(num_kv_heads=8, query_len=8), 168),
    (dict(num_kv_heads=8, dtype=0), 96),    # fp32 grouped: 2 vectors per warp
])
def test_plan_fits_its_ctas_by_registers(nsv, kw, regs):
    """A plan's CTAs per SM fit the SM's registers at the variant's fixed
    register count: 4 sub-partitions of 16 K registers, each holding whole
    warps (allocated per warp in units of 256)."""
    p = nsv.plan_split(_shape(nsv, **kw), num_sms=152)
    warps = p.threads // 32
    per_warp = -(-regs * 32 // 256) * 256
    assert p.ctas_per_sm * warps <= 4 * (16384 // per_warp)


def test_cuda_core_plan_with_17_warps_takes_one_cta_per_sm(nsv):
    """16 consumer warps + the producer at 96 registers: one CTA per SM (two
    would need 34 warps' registers)."""
    p = nsv.plan_custom(_shape(nsv, num_kv_heads=8, query_len=8), num_sms=152,
                        consumer=nsv.CONSUMER_CUDA)
    assert p.threads == 17 * 32 and p.ctas_per_sm == 1 and p.grid == 152


def test_every_plan_round_trips(nsv):
    """A plan the planner makes, handed back with all its choices fixed (as
    nsv_paged_decode_ws checks a caller's plan), must come out identical:
    no choice the heuristic takes may be one the explicit path refuses."""
    base = dict(rows=256, max_blocks=512, num_blocks=70000)
    checked = 0
    for dtype in (nsv.F32, nsv.BF16):
        for heads, kv, ql in [(32, 32, 1), (32, 8, 1), (32, 32, 4), (32, 8, 8), (128, 8, 1),
                              (16, 16, 17), (8, 8, 3), (16, 1, 2), (8, 2, 16), (64, 8, 8),
                              (64, 1, 1), (32, 32, 64), (1, 1, 1), (2, 2, 1), (8, 1, 1),
                              (24, 6, 5), (20, 5, 5)]:
            for d in (64, 128):
                shape = nsv.make_shape(num_heads=heads, num_kv_heads=kv, query_len=ql,
                                       dtype=dtype, head_dim=d, **base)
                for extra in (dict(), dict(consumer=1), dict(consumer=2), dict(consumer=3),
                              dict(consumer=1, vectors_per_warp=4), dict(kv_heads_per_cta=1),
                              dict(kv_heads_per_cta=2, ctas_per_sm=2), dict(stages=2),
                              dict(consumer=4), dict(consumer=4, kv_heads_per_cta=1),
                              dict(consumer=4, blocks_per_stage=1),
                              dict(consumer=4, blocks_per_stage=2, stages=4),
                              dict(consumer=4, blocks_per_stage=4)):
                    try:
                        p = nsv.plan_custom(shape, num_sms=152, **extra)
                    except nsv.NsvError:
                        continue
                    q = nsv.plan_custom(shape, num_sms=p.num_sms,
                                        kv_heads_per_cta=p.kv_heads_per_cta, stages=p.stages,
                                        ctas_per_sm=p.ctas_per_sm, grid=p.grid,
                                        vectors_per_warp=p.vectors_per_warp,
                                        consumer=p.consumer,
                                        blocks_per_stage=p.blocks_per_stage)
                    assert bytes(q) == bytes(p), (heads, kv, ql, dtype, d, extra)
                    checked += 1
    assert checked > 150


@pytest.mark.parametrize("heads,kv_heads,qlen", [(64, 8, 8), (64, 1, 1), (32, 32, 64),
                                                 (32, 8, 10), (128, 2, 1)])
def test_bf16_takes_up_to_64_vectors_per_kv_head(nsv, heads, kv_heads, qlen):
    """Beyond 32 query vectors per KV head only the tensor cores serve the
    read: tcgen05 into tensor memory, 2 KV heads of 64 rows per MMA, or with
    an odd KV-head count the vectors as the rows, one warp per 16 of them."""
    p = nsv.plan_split(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen),
                       num_sms=152)
    vpk = heads // kv_heads * qlen
    assert vpk > 32
    if kv_heads % 2 == 0:
        assert p.consumer == nsv.CONSUMER_TENSOR_TMEM and p.kv_heads_per_cta == 2
        assert p.threads == 10 * 32
    else:
        assert p.consumer == nsv.CONSUMER_TENSOR_VECTOR_ROWS
        assert p.threads == _cta_warps(nsv, p.consumer, p.kv_heads_per_cta * -(-vpk // 16)) * 32


@pytest.mark.parametrize("heads,kv_heads,qlen,consumer", [
    (32, 8, 8, 3),    # head_dim 64, 32 vectors: the vectors as the MMA rows
    (16, 4, 5, 3),    # 20 vectors
    (64, 8, 8, 4),    # 64 vectors: tcgen05 into tensor memory
    (40, 4, 4, 4),    # 40 vectors
])
def test_plan_head_dim_64_tmem_rule(nsv, heads, kv_heads, qlen, consumer):
    """At head_dim 64 the TMEM form is the default only beyond 32 vectors per
    KV head: up to 32, its stages' fixed cost on half-size blocks left it
    behind the vectors-as-rows form."""
    p = nsv.plan_split(_shape(nsv, num_heads=heads, num_kv_heads=kv_heads, query_len=qlen,
                              head_dim=64), num_sms=152)
    assert p.consumer == consumer


def test_binding_refuses_to_load_without_the_library(tmp_path):
    """No fallback: a copy of the package without its built library cannot
    be imported as a binding, and bench.py's GPU arm exits non-zero."""
    import sys
    pkg = tmp_path / "paged_kv_decode_nsv_gb300"
    shutil.copytree(os.path.join(ROOT, "paged_kv_decode_nsv_gb300"), pkg,
                    ignore=shutil.ignore_patterns("_lib", "_build", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import paged_kv_decode_nsv_gb300.nsv"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libnsv.so is not built" in r.stderr
    shutil.copy(os.path.join(ROOT, "bench.py"), tmp_path / "bench.py")
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny_f32", "--steps", "1",
                        "--warmup", "3", "--cpu-seconds", "0"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0 and "libnsv.so is not built" in r.stderr
    assert not [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
