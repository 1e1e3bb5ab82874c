// Batched paged-attention decode read for sm_103a.
//
// What it computes (nanoserve Day 59, "the rectangle the read builds, and
// the tile that replaces it", "What I added today" and "What I learned"
// items 3-4): for every row and query head, softmax(scale * q.K^T) V over
// the row's own context_lens[row] positions, folded block by block with an
// online softmax (running max m, running denominator l, running weighted
// sum acc).  The row's blocks are found through its block table and only
// cdiv(ctx, block) of them are walked; nothing past a row's length is
// loaded, so table padding may be -1 and unwritten slots may hold NaN
// ("Why it matters", the masked-load paragraph).
//
// How it runs on GB300 (the design differs from the pages' (row, head) grid):
//  * A persistent grid of CTAs (SM count x resident CTAs).  The work is the
//    sequence of units (head group, row, block) -- a head group is
//    `heads_per_cta` KV heads with all their query heads -- laid end to end
//    over every row's cdiv(ctx, block) blocks.  CTA c takes the units
//    [c*U/G, (c+1)*U/G): every CTA streams the same number of blocks (stream-K
//    style), whatever the length mix.  Every CTA derives the sequence from
//    context_lens in shared memory, so the launch depends on shape alone.
//  * Warp 0 is the producer.  Per block it copies the head group's K tiles
//    and V tiles (each one contiguous run in the [block][kv_head][token][dim]
//    pool) into a ring of shared-memory stages guarded by mbarriers: two
//    cp.async.bulk copies for the CUDA-core consumer, 2-D TMA tiles with the
//    128-byte swizzle for the tensor-core one; plus the query vectors at each
//    segment's first stage.  The block ids of the next 32 units are loaded a
//    window ahead.  A slot-table block that is not one aligned run of slots
//    is gathered token by token by the producer warp instead.
//  * Warps 1..N are consumers.  On the CUDA cores (fp32, or one query
//    vector per KV head) a warp serves 1, 2 or 4 query vectors of one KV
//    head: a lane owns 16 bytes of a key row; the score of each token of the
//    tile is reduced with a transposing butterfly (one shuffle per token
//    instead of five), the tile max with a plain butterfly, probabilities go
//    through shared memory to the lanes that own the value dims, and P.V
//    accumulates in fp32.  On the tensor cores (bf16, 2 to 64 query vectors
//    per KV head) the same two contractions run as mma.sync.m16n8k16: with
//    the block's 16 tokens as the MMA rows for up to 8 vectors, with the
//    vectors as the rows (16 per warp) beyond.
//  * A segment (a CTA's run of one row) that covers the whole row writes
//    `out` directly.  A row cut by CTA boundaries leaves one partial (m, l,
//    acc) per CTA it crosses -- at most two per CTA.  Each piece's CTA then
//    counts itself in the row's arrival counter, and the CTA that arrives
//    last merges the pieces (flash-decoding style) and writes `out`.  Nobody
//    waits for anybody: the last arrival finds every partial already
//    written.  Empty rows get their zero output from the consumers up front.
// Every wait is bounded; a wait that gives up sets NSV_DEV_TIMEOUT and the
// kernel returns.  Bad lengths and block ids are skipped and flagged.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "nsv_common.cuh"

namespace nsv {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s
// Slack of the tensor consumer's lazily raised running max, in log2 units.
constexpr float kRescaleSlack = 8.f;
// Tensor-core consumer forms (the kernel's MMA template argument; 0: CUDA cores).
constexpr int kMmaVectorRows = kFormVectorRows;  // query vectors as the MMA rows (M = 16)
constexpr int kMmaTokenRows = kFormTokenRows;    // the block's tokens as the MMA rows (M = 16)
constexpr int kMmaCols = 8;        // query vectors per warp with tokens as rows
constexpr int kMmaTmem = kFormTmem;               // tcgen05.mma, accumulators in tensor memory

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// Add `bytes` to the transaction count the current phase of `bar` waits
// for (no arrival): the TMEM form arms a stage block by block and arrives
// once when the stage is complete.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Whether the phase of `bar` with the given parity has completed, without
// waiting.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete; false if
// it has not after limit_ns.  The first try is inline (the common case: the
// phase is already complete); the bounded loop is out of line.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            unsigned long long limit_ns) {
  const unsigned long long t0 = global_ns();
  while (true) {
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, kWaitLimitNs);
}

// Self-test of the bounded wait: one thread waits, with limit_ns, for a
// phase of a fresh mbarrier that nothing completes.  result[0] = 1 when the
// wait gave up, result[1] = the nanoseconds it waited; a wait that gave up
// sets NSV_DEV_TIMEOUT in *status, as the decode kernel's waits do.
__global__ void bounded_wait_probe(unsigned long long limit_ns, unsigned long long* result,
                                   uint32_t* status) {
  __shared__ __align__(8) unsigned long long bar_word;
  if (threadIdx.x != 0) return;
  const uint32_t bar = smem_u32(&bar_word);
  mbar_init(bar, 1);
  fence_mbar_init();
  const unsigned long long t0 = global_ns();
  const bool completed = mbar_wait_slow(bar, 0, limit_ns);
  result[1] = global_ns() - t0;
  result[0] = completed ? 0ull : 1ull;
  if (!completed) atomicOr(status, (uint32_t)NSV_DEV_TIMEOUT);
}

// Programmatic dependent launch: wait until the grid this launch depends on
// (the step's append) has completed and its writes are visible.  Returns at
// once when the launch has no such dependency.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Prefetch `bytes` (a multiple of 16) at a 16-byte aligned global address
// into L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One 2-D TMA tile load global -> this CTA's shared memory (the tensor map's
// box, with its swizzle), completing on `bar`.  x is the innermost coordinate.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

// The same with a 4-D tensor map (coordinates x innermost, y, z, w).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            int w, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(pol)
      : "memory");
}

// The same with a 3-D tensor map (coordinates x innermost, y, z).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

// Four 8x8 bf16 matrices from shared memory (row addresses from lanes 8i..8i+7).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// The same, each matrix transposed.
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, bf16, row) * B(16x8, bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The transpose of an 8x8 b16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of 16-byte chunk `dc` (dims 8*dc .. 8*dc+7) of row r of a K
// or V tile set staged by 128-byte-swizzled TMA loads: the dims are split in
// 64-dim halves of half_bytes each, a row of a half is 128 bytes, and chunk c
// of row r sits at position c ^ (r % 8).
// Byte offset of 16-byte chunk dc of token row r in the TMEM form's K
// layout: rows in groups of 8, each group's 64-dim halves one 1024-byte
// atom after the other ([group][half][8 rows][128 bytes], 128-byte swizzle).
template <int D>
__device__ __forceinline__ uint32_t swz_grouped(int r, int dc) {
  return (uint32_t)(r >> 3) * (D / 64) * 1024u + (uint32_t)(dc >> 3) * 1024u +
         (uint32_t)(r & 7) * 128u + ((uint32_t)((dc & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t swz(int r, int dc, uint32_t half_bytes) {
  return (uint32_t)(dc >> 3) * half_bytes + (uint32_t)r * 128u +
         ((uint32_t)((dc & 7) ^ (r & 7)) << 4);
}

// ---------------------------------------------------------------------------
// element traits: a lane loads 16 bytes = kDpl elements and widens to fp32

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kDpl = 4;
  __device__ __forceinline__ static void widen(const uint4& r, float (&x)[4]) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  }
  __device__ __forceinline__ static uint4 narrow(const float (&x)[4]) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kDpl = 8;
  // bf16 is the upper half of an fp32: widening is a shift or a mask.
  __device__ __forceinline__ static void widen(const uint4& r, float (&x)[8]) {
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
    x[4] = __uint_as_float(r.z << 16);
    x[5] = __uint_as_float(r.z & 0xffff0000u);
    x[6] = __uint_as_float(r.w << 16);
    x[7] = __uint_as_float(r.w & 0xffff0000u);
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint4 narrow(const float (&x)[8]) {
    return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]),
                      pack2(x[6], x[7]));
  }
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Two fp32 fused multiply-adds in one instruction (sm_100+ packed f32x2):
// (d0, d1) = (a0 * b0 + d0, a1 * b1 + d1), each rounded as fmaf would.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Validated context length (a bad one is read as 0 and flagged).
__device__ __forceinline__ int checked_ctx(const DecodeParams& p, int r) {
  int c = p.context_lens[r];
  const int limit = p.slots ? min(p.max_blocks * kBlock, p.slot_cols) : p.max_blocks * kBlock;
  if (c < 0 || c > limit) {
    atomicOr(p.status, (uint32_t)NSV_DEV_BAD_CTX);
    c = 0;
  }
  return c;
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor of a tcgen05.mma operand: start address,
// leading- and stride-dimension byte offsets (16-byte units), the fixed
// version field, and the swizzle mode.  For a K-major operand with the
// 128-byte swizzle the stride offset is the step between 8-row groups (the
// leading one is unused); for an MN-major one the stride offset steps 8 rows
// of K and the leading one steps 64 elements of M or N; without swizzle
// (8x16-byte core matrices) the leading offset steps K and the stride
// offset steps 8 rows.
constexpr uint32_t kUmmaSwizzleNone = 0, kUmmaSwizzle128 = 2;
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)swizzle << 61);
}
// Instruction descriptor of a kind::f16 MMA: fp32 accumulator, bf16 A and B,
// A K-major, B K-major or MN-major, N / 8 and M / 16.
__device__ __forceinline__ uint32_t umma_idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// D (tensor memory) = A.B (+ D when `accumulate`): one MMA, executed by a
// whole warp (uniform control flow, so the descriptors can stay
// warp-uniform) with only the `lead` lane issuing.
__device__ __forceinline__ void umma_bf16_warp(uint32_t d_tmem, uint64_t a, uint64_t b,
                                               uint32_t idesc, bool accumulate, bool lead) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %4, 0;\n\tsetp.ne.u32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u), "r"(lead ? 1u : 0u)
      : "memory");
}
// The same with the A operand in tensor memory (`a_tmem`: its rows in the
// lanes, two bf16 of a row's K to a 32-bit column).
__device__ __forceinline__ void umma_bf16_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                                  uint32_t idesc, bool accumulate, bool lead) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %4, 0;\n\tsetp.ne.u32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u), "r"(lead ? 1u : 0u)
      : "memory");
}
// One arrive on `bar` once every MMA the `lead` lane issued so far is
// complete (executed by the whole warp).
__device__ __forceinline__ void umma_commit_warp(uint32_t bar, bool lead) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar),
      "r"(lead ? 1u : 0u)
      : "memory");
}
// 2^x by the special-function unit (ex2.approx: relative error about
// 2^-22, +0 for -inf), for the TMEM form's probabilities, which are rounded
// to bf16 right after.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// 8, 16 or 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Block id of a unit under slot-table addressing: the block's `nval` slots
// must be one aligned, contiguous run (as a table built from block tables
// always is); otherwise kTokenWise, and the block is gathered per token.
constexpr int kTokenWise = -2;

__device__ __forceinline__ int slot_block(const int64_t* sp, int nval) {
  const long long s0 = sp[0];
  bool run = (s0 % kBlock) == 0;
#pragma unroll 4
  for (int i = 1; i < kBlock; ++i)
    if (i < nval) run = run && (sp[i] == s0 + i);
  if (!run) return kTokenWise;
  const long long b = s0 / kBlock;  // may be out of range: flagged by the caller
  return (b < 0 || b > 0x7fffffffll) ? -1 : (int)b;
}

// Barrier over the consumer warps only (the producer never joins it).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// CTA whose unit range [c*U/G, (c+1)*U/G) holds unit u (the last such c
// when empty ranges share a start).
__device__ __forceinline__ int cta_of(long long u, long long U, int G) {
  long long c = ((u + 1) * G + U - 1) / U - 1;
  return (int)(c < G - 1 ? c : G - 1);
}

// A consumer warp has written its partials of a cut row (the row's pieces
// lie on CTAs c0..c1).  Count this CTA's piece once it is published; the CTA
// whose piece arrives last merges every piece, each of its warps for its own
// query vectors [v0, v0 + nv).  Nobody waits for another CTA: the last
// arrival finds every partial already written.  kLanes: lanes per query
// vector in the merge (32 / kLanes vectors at a time); kChunk: pieces whose
// loads are in flight together.
template <typename T, int D, int kLanes, int kChunk>
__device__ __forceinline__ void finish_cut_row(const DecodeParams& p, int row, int kv0,
                                               const int* s_prefix, int N, long long U, int nhg,
                                               int nvec, int v0, int nv, int ncw, int cw,
                                               int lane, volatile int* s_merge) {
  const int G = p.group, NQ = p.query_len, HG = p.heads_per_cta;
  const int vpk = G * NQ;
  __threadfence();
  consumer_sync(ncw * 32);
  const int hg = kv0 / HG;
  const int pr = s_prefix[row], nb = s_prefix[row + 1] - pr;
  const long long u0 = (long long)hg * N + pr, u1 = u0 + nb;
  const int c0 = cta_of(u0, U, gridDim.x), c1 = cta_of(u1 - 1, U, gridDim.x);
  // (The counters are written by the step's append; this comes after the
  // piece's stages, so after the producer's wait for the append.)
  if (cw == 0 && lane == 0) {
    int pieces = c1 - c0 + 1;
    if (U < gridDim.x) {  // some CTAs have no units and wrote nothing
      pieces = 0;
      for (int c = c0; c <= c1; ++c)
        pieces += ((long long)(c + 1) * U / gridDim.x != (long long)c * U / gridDim.x);
    }
    int* cnt = p.ws_cnt + (size_t)row * nhg + hg;
    const int before = atomicAdd(cnt, 1);
    const bool last = before == pieces - 1;
    if (last) *cnt = 0;  // every piece has arrived: nobody touches it again
    *s_merge = last ? 1 : 0;
  }
  consumer_sync(ncw * 32);
  if (!*s_merge) return;
  __threadfence();
  // 32 / kLpv vectors at a time, kLpv lanes each; lane dq of a vector owns
  // the 4-dim groups dq, dq + kLpv, dq + 2 kLpv, ... (dims 4(f kLpv + dq) ..
  // + 3 for f = 0 .. kF4 - 1), so that one load instruction's lanes read a
  // vector's partial in whole sectors.  Every load of a step is independent
  // of the others, so merging a batch of vectors costs about 1 + ns/kChunk
  // L2 round trips (the partials were just written by other CTAs: read
  // through L2).
  constexpr int kLpv = kLanes < D / 4 ? kLanes : D / 4;
  constexpr int kDl = D / kLpv;
  constexpr int kF4 = kDl / 4;
  const int ns = c1 - c0 + 1;
  const int qh0 = kv0 * G;
  const int j = lane / kLpv, dq = lane % kLpv;
  // slot of the k-th CTA's piece, or -1 for a CTA with no units
  auto slot_of = [&](int kk) {
    const int c = c0 + kk;
    const long long sc = (long long)c * U / gridDim.x;
    if ((long long)(c + 1) * U / gridDim.x == sc) return -1;
    return c * 2 + ((c == c0 && sc < u0) ? 1 : 0);
  };
  // the first kLpv pieces' slots, one per lane of a vector's group; later
  // pieces (a row cut into many) are found again where they are needed
  const int sl_own = dq < ns ? slot_of(dq) : -1;
  const int g0 = lane & ~(kLpv - 1);
  auto slot_k = [&](int kk) {  // kk is warp-uniform
    const int sl = __shfl_sync(kFull, sl_own, g0 + (kk & (kLpv - 1)));
    return kk < kLpv ? sl : slot_of(kk);
  };
  for (int k0 = 0; k0 < nv; k0 += 32 / kLpv) {
    const bool vok = k0 + j < nv;
    const int vv = v0 + (vok ? k0 + j : 0);
    // the pieces' combined max and denominator: the vector's lanes take
    // every eighth piece, then fold their (max, sum) pairs together
    float M = -INFINITY, Ls = 0.f;
    for (int kk = dq; kk < ns; kk += kLpv) {
      const int sl = kk < kLpv ? sl_own : slot_of(kk);
      if (sl < 0) continue;
      const float2 ml = __ldcg(&p.ws_ml[(size_t)sl * nvec + vv]);
      if (ml.x == -INFINITY) continue;
      const float mn = fmaxf(M, ml.x);
      Ls = Ls * exp2f(M - mn) + ml.y * exp2f(ml.x - mn);
      M = mn;
    }
#pragma unroll
    for (int o2 = 1; o2 < kLpv; o2 <<= 1) {
      const float Mo = __shfl_xor_sync(kFull, M, o2), Lo = __shfl_xor_sync(kFull, Ls, o2);
      const float mn = fmaxf(M, Mo);
      if (mn != -INFINITY) {
        Ls = (M == -INFINITY ? 0.f : Ls * exp2f(M - mn)) + (Mo == -INFINITY ? 0.f : Lo * exp2f(Mo - mn));
        M = mn;
      }
    }
    float a[kDl];
#pragma unroll
    for (int e = 0; e < kDl; ++e) a[e] = 0.f;
    for (int kk0 = 0; kk0 < ns; kk0 += kChunk) {
      float2 ml[kChunk];
      float4 v[kChunk][kF4];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const int sl = kk0 + u < ns ? slot_k(kk0 + u) : -1;
        const size_t idx = (size_t)(sl < 0 ? 0 : sl) * nvec + vv;
        ml[u] = sl < 0 ? make_float2(-INFINITY, 0.f) : __ldcg(&p.ws_ml[idx]);
        const float4* src = reinterpret_cast<const float4*>(p.ws_acc + idx * D) + dq;
#pragma unroll
        for (int f = 0; f < kF4; ++f)
          v[u][f] = sl < 0 ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldcg(src + f * kLpv);
      }
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const float w = ml[u].x == -INFINITY ? 0.f : exp2f(ml[u].x - M);
#pragma unroll
        for (int f = 0; f < kF4; ++f) {
          a[4 * f] = fmaf(w, v[u][f].x, a[4 * f]);
          a[4 * f + 1] = fmaf(w, v[u][f].y, a[4 * f + 1]);
          a[4 * f + 2] = fmaf(w, v[u][f].z, a[4 * f + 2]);
          a[4 * f + 3] = fmaf(w, v[u][f].w, a[4 * f + 3]);
        }
      }
    }
    if (!vok) continue;
    const int kvl = vv / vpk, rem = vv - kvl * vpk;
    const int qh = qh0 + kvl * G + rem / NQ, jq = rem % NQ;
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    T* o = static_cast<T*>(p.out) + (((size_t)row * NQ + jq) * p.heads + qh) * D + 4 * dq;
#pragma unroll
    for (int f = 0; f < kF4; ++f) {
      T* of = o + 4 * f * kLpv;
      if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(of) = make_float4(a[4 * f] * inv, a[4 * f + 1] * inv,
                                                     a[4 * f + 2] * inv, a[4 * f + 3] * inv);
      } else {
        *reinterpret_cast<uint2*>(of) = make_uint2(pack_bf16(a[4 * f] * inv, a[4 * f + 1] * inv),
                                                   pack_bf16(a[4 * f + 2] * inv, a[4 * f + 3] * inv));
      }
    }
  }
}

// finish_cut_row for the TMEM form, out of line: it runs once per piece of a
// cut row, and inlined into the softmax warps' stage loop its registers
// pushed that loop's working set into local memory.
template <typename T, int D, int kLanes, int kChunk>
__device__ __noinline__ void finish_cut_row_call(const DecodeParams& p, int row, int kv0,
                                                 const int* s_prefix, int N, long long U,
                                                 int nhg, int nvec, int v0, int nv, int ncw,
                                                 int cw, int lane, volatile int* s_merge) {
  finish_cut_row<T, D, kLanes, kChunk>(p, row, kv0, s_prefix, N, U, nhg, nvec, v0, nv, ncw, cw,
                                       lane, s_merge);
}

// Tensor-core consumer (bf16) with the query vectors as the MMA rows: a KV
// head's query vectors (the group's query heads of that KV head times the
// query tokens, 2 to 64 of them, by default 9 and more) are the rows of
// mma.sync.m16n8k16 (bf16 inputs, fp32 accumulate), 16 rows per warp, so
// one to four warps per KV head read the same K/V tile.  Each warp zeroes
// the tile's empty V rows itself (they all write the same zeros).  Per
// 16-token block: S = Q.K^T from the K tile staged by
// swizzled TMA loads and read with ldmatrix, the online softmax on the score
// fragments, then O += P.V with P (bf16) taken straight from the score
// fragments and V read with ldmatrix.trans.  Fragment layout of m16n8k16:
// lane = 4*g + t4 holds rows g and g+8, columns 2*t4 and 2*t4+1.
template <int D>
__device__ __forceinline__ void consume_mma(const DecodeParams& p, unsigned char* smem,
                                            const SmemLayout& L, const int4* s_meta,
                                            uint32_t bars, const int* s_prefix,
                                            volatile int* s_abort, int N, long long U, int nhg,
                                            int nvec, int ncw, int warp, int lane) {
  using T = __nv_bfloat16;
  constexpr int kKs = D / 16;  // k-steps of the score MMA
  constexpr int kNd = D / 8;   // n-tiles of the P.V MMA
  const int G = p.group, NQ = p.query_len, HG = p.heads_per_cta, S = p.stages;
  if (warp > ncw) return;
  const int cw = warp - 1;
  const int vpk = G * NQ;               // query vectors per KV head (<= 32)
  const int wpk = ncw / HG;             // warps per KV head: one per 16 vectors
  const int kvl = cw / wpk;             // this warp's KV head within the group
  const int v0w = (cw - kvl * wpk) * kMmaRows;  // its first vector of that KV head
  const int nvw = min(kMmaRows, vpk - v0w);     // and how many it runs (<= 16)
  const int vbase = kvl * vpk + v0w;
  const int g = lane >> 2, t4 = lane & 3;
  const int hq = HG * G;
  const uint32_t half_bytes = (uint32_t)HG * kBlock * 128;
  volatile int* s_merge = s_abort + 1;

  // rows g and g + 8 of the MMA: their query head within the group and token
  int rqh[2], rjq[2];
  bool rok[2];
#pragma unroll
  for (int rh = 0; rh < 2; ++rh) {
    const int r = g + 8 * rh;
    rok[rh] = r < nvw;
    const int rr = v0w + (rok[rh] ? r : 0);
    rqh[rh] = kvl * G + rr / NQ;
    rjq[rh] = rr % NQ;
  }

  // Empty rows see nothing: zeros for all their (token, head) vectors.
  constexpr int kChunks = D * 2 / 16;
  for (int r = blockIdx.x; r < p.rows; r += gridDim.x) {
    if (s_prefix[r + 1] != s_prefix[r]) continue;
    for (int vh = cw; vh < NQ * p.heads; vh += ncw)
      for (int c = lane; c < kChunks; c += 32)
        reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)r * NQ * p.heads + vh) * D)[c] =
            make_uint4(0u, 0u, 0u, 0u);
  }

  uint32_t qa[kKs][4];
  float o[kNd][4], m[2], l[2];
#pragma unroll
  for (int ks = 0; ks < kKs; ++ks) qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
#pragma unroll
  for (int nd = 0; nd < kNd; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  m[0] = m[1] = -INFINITY;
  l[0] = l[1] = 0.f;

  for (uint32_t n = 0;; ++n) {
    const uint32_t s = n % S;
    if (!mbar_wait(bars + 8 * s, (n / S) & 1)) {
      if (lane == 0) atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
      *s_abort = 1;
      return;
    }
    const int4 meta = s_meta[s];
    const int flags = meta.w;
    if (flags & kEnd) break;
    unsigned char* st = smem + s * L.stage_bytes;
    const uint32_t kbase = smem_u32(st), vbase_s = kbase + L.kv_bytes;
    const int tmask = meta.y & 0xffff;
    const int qh0 = (flags >> 16) * G;

    if (flags & kFirst) {
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int nd = 0; nd < kNd; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
      if (flags & kHasQ) {
        // q ring: after the S stages; this form has one slot
        constexpr int qslot = 0;
        const unsigned char* qs = smem + (size_t)S * L.stage_bytes;
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
#pragma unroll
          for (int rh = 0; rh < 2; ++rh) {
            const unsigned char* row =
                qs + ((size_t)(rjq[rh] * hq + rqh[rh]) * D + ks * 16 + t4 * 2) * sizeof(T);
            qa[ks][rh] = rok[rh] ? *reinterpret_cast<const uint32_t*>(row) : 0u;
            qa[ks][2 + rh] = rok[rh] ? *reinterpret_cast<const uint32_t*>(row + 16) : 0u;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (2 * S + qslot));  // the q slot is free
      }
    }

    if (flags & kData) {
      const int rem = flags & 0xff;
      const int nvalid = min(kBlock, rem);
      // V rows that hold no data (past the row's length, or tokens the
      // producer did not gather) become zeros: P is 0 there, but 0 * NaN is not.
      if (nvalid < kBlock || tmask != 0xffff) {
        for (int c = lane; c < kBlock * kChunks; c += 32) {
          const int t = c / kChunks, dc = c - t * kChunks;
          if (!(t < nvalid && ((tmask >> t) & 1)))
            *reinterpret_cast<uint4*>(st + L.kv_bytes + swz(kvl * kBlock + t, dc, half_bytes)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // scores: 2 n-tiles of 8 tokens, kKs k-steps of 16 dims
      float sc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      {
        const int mi = lane >> 3, i = lane & 7;
        const int r = kvl * kBlock + (mi >> 1) * 8 + i;
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz(r, ks * 2 + (mi & 1), half_bytes), b0, b1, b2, b3);
          mma_bf16(sc[0], qa[ks], b0, b1);
          mma_bf16(sc[1], qa[ks], b2, b3);
        }
      }
      // Online softmax per row (a row's 16 scores sit on 4 lanes).  The
      // running max is raised lazily: only when a block's max exceeds it by
      // more than kRescaleSlack (log2 units) are l and O rescaled, so most
      // blocks skip the rescale and the probabilities stay <= 2^kRescaleSlack.
      // Any reference max gives the same softmax; l and O always refer to m.
      // A block every row sees in full needs no masks: rows past the vector
      // count have zero queries, finite scores, and are never written.
      const bool dense = nvalid == kBlock && tmask == 0xffff && rem - (NQ - 1) >= kBlock;
      uint32_t pa[4];
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = sc[e >> 1][rh * 2 + (e & 1)] * p.qscale;
        if (!dense) {
          const int nv = rem - (NQ - 1 - rjq[rh]);  // positions this row's query sees
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = (e >> 1) * 8 + t4 * 2 + (e & 1);
            if (!(rok[rh] && tok < nv && ((tmask >> tok) & 1))) x[e] = -INFINITY;
          }
        }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        if (mx > m[rh] + kRescaleSlack) {  // also the first finite max (m = -inf)
          const float alpha = exp2f(m[rh] - mx);
          m[rh] = mx;
          l[rh] *= alpha;
#pragma unroll
          for (int nd = 0; nd < kNd; ++nd) {
            o[nd][rh * 2] *= alpha;
            o[nd][rh * 2 + 1] *= alpha;
          }
        }
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = (dense || x[e] != -INFINITY) ? exp2f(x[e] - m[rh]) : 0.f;
          l[rh] += pv[e];
        }
        pa[rh] = pack_bf16(pv[0], pv[1]);      // row rh*8 + g, tokens 2*t4, 2*t4+1
        pa[2 + rh] = pack_bf16(pv[2], pv[3]);  // the same row, tokens 8 + 2*t4, ...
      }
      // O += P.V: n-tiles of 8 dims, V read transposed
      {
        const int mi = lane >> 3, i = lane & 7;
        const int r = kvl * kBlock + (mi & 1) * 8 + i;
#pragma unroll
        for (int nd = 0; nd < kNd; nd += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase_s + swz(r, nd + (mi >> 1), half_bytes), b0, b1, b2, b3);
          mma_bf16(o[nd], pa, b0, b1);
          mma_bf16(o[nd + 1], pa, b2, b3);
        }
      }
    }

    if (flags & kLast) {
      const int row = meta.x;
      float lt[2];
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        lt[rh] = l[rh];
        lt[rh] += __shfl_xor_sync(kFull, lt[rh], 1);
        lt[rh] += __shfl_xor_sync(kFull, lt[rh], 2);
      }
      if (flags & kFinal) {
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          if (!rok[rh]) continue;
          const float inv = lt[rh] > 0.f ? 1.f / lt[rh] : 0.f;
          T* out = static_cast<T*>(p.out) +
                   (((size_t)row * NQ + rjq[rh]) * p.heads + qh0 + rqh[rh]) * D + t4 * 2;
#pragma unroll
          for (int nd = 0; nd < kNd; ++nd)
            *reinterpret_cast<uint32_t*>(out + nd * 8) =
                pack_bf16(o[nd][rh * 2] * inv, o[nd][rh * 2 + 1] * inv);
        }
      } else {
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
          if (!rok[rh]) continue;
          const size_t slot = (size_t)meta.z * nvec + vbase + g + 8 * rh;
          float* a = p.ws_acc + slot * D + t4 * 2;
#pragma unroll
          for (int nd = 0; nd < kNd; ++nd)
            *reinterpret_cast<float2*>(a + nd * 8) = make_float2(o[nd][rh * 2], o[nd][rh * 2 + 1]);
          if (t4 == 0) p.ws_ml[slot] = make_float2(m[rh], lt[rh]);
        }
        finish_cut_row<T, D, 8, 2>(p, row, flags >> 16, s_prefix, N, U, nhg, nvec, vbase, nvw,
                                   ncw, cw, lane, s_merge);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
}

// The TMEM form (bf16) on the 5th-generation tensor cores: tcgen05.mma from
// shared-memory operands into tensor-memory accumulators.  The MMA has 128
// rows: the group's KV heads take R = 128 / group rows each (their query
// vectors, zero rows past them).  A stage holds up to `blocks_per_stage`
// consecutive blocks of one segment, so one scores MMA per 16 dims covers
// all of them (N = blocks x group x 16 tokens) and each row keeps its own
// head's 16 columns of every block.  The P.V product of a block is one MMA
// of N = group x head_dim: every row's probabilities (for its own head's
// tokens) times every head's V of the block, of which each row keeps its own
// head's columns.  Roles:
//   * an MMA warp (one lane issues) runs S = Q.K^T for stage n + 1 while the
//     softmax warps work on stage n (two score buffers in tensor memory, two
//     probability buffers in shared memory), then O += P.V for stage n once
//     they hand P over, committed to the stage's empty barrier;
//   * four softmax warps, one per TMEM lane quadrant: thread r owns row r
//     (its online-softmax state in registers), reads its head's 16 scores of
//     each block with tcgen05.ld and writes its probabilities (bf16) into P.
// Shared-memory operands: Q (128 x D, 128-byte swizzle, K-major) copied
// from global memory by the softmax warps; K as staged by TMA, the stage's
// token rows (block, head, token) in order within each 64-dim half
// (K-major); P in 8x16-byte core matrices, 16 tokens per block; V as
// staged, block by block, each block's 64-dim chunks (half, head) 2 KiB
// apart (MN-major).  Tensor memory: O in columns [0, group x D), the chunk
// (half h, head k) at columns (h x group + k) x 64; then two score buffers
// of blocks x group x 16 columns.
// Barriers beyond the ring's: scores ready [2], probabilities handed over
// [2], a piece's O complete, every MMA drained, query rows ready.  (A stage's
// empty barrier, which its P.V's commit completes, also tells the softmax
// warps that this P.V is done.)
struct TmemBars {
  uint32_t base;
  __device__ uint32_t scores(uint32_t b) const { return base + 8 * b; }
  __device__ uint32_t handed(uint32_t b) const { return base + 16 + 8 * b; }
  __device__ uint32_t out() const { return base + 32; }
  __device__ uint32_t drained() const { return base + 40; }
  __device__ uint32_t qready() const { return base + 48; }
};
constexpr int kTmemBars = 7;

// Token mask of block b of a TMEM stage (its second metadata word).
__device__ __forceinline__ int tmem_block_mask(const int4& mm, int b) {
  return ((b < 2 ? mm.x : mm.y) >> (16 * (b & 1))) & 0xffff;
}

// The MMA warp.  The d-th stage with data has its scores in buffer d & 1,
// stage n's probabilities are in buffer n & 1; every barrier completes once
// per use and never runs more than one phase ahead of a wait on it, so
// parity waits suffice.
template <int D>
__device__ __forceinline__ bool tmem_mma_warp(const DecodeParams& p, unsigned char* smem,
                                              const SmemLayout& L, const int4* s_meta,
                                              uint32_t bars, uint32_t tmem, int lane) {
  const int HG = p.heads_per_cta, S = p.stages, NB = p.blocks_per_stage;
  const int ntok = NB * HG * kBlock;               // a full stage's token rows
  // K: the stage's token rows in groups of 8, a group's 64-dim halves one
  // 1024-byte atom apart: within a half, groups are D / 64 atoms apart
  constexpr uint32_t kGroupBytes = (uint32_t)(D / 64) * 1024u;
  const uint32_t k_area = (uint32_t)NB * L.kv_bytes;
  const TmemBars tb{bars + 8 * (2 * S + (int)L.q_slots)};
  const bool lead = lane == 0;
  const uint32_t stage0 = smem_u32(smem);
  const uint32_t pb_s = smem_u32(smem + L.off_pbuf);
  const uint32_t pbuf_bytes = (uint32_t)(kTmemRows * NB * kBlock * 2);
  const int pch = NB * 2;  // 16-byte chunks of a P row
  // the query rows in tensor memory after the score buffers: 16 dims of K
  // are 8 columns
  const uint32_t q_col = (uint32_t)(HG * D + 2 * ntok);
  // descriptors are linear in the start address: a base plus an offset
  const uint64_t dk0 = umma_desc(0u, 16, kGroupBytes, kUmmaSwizzle128);
  const uint64_t dp0 = umma_desc(pb_s, 128, (uint32_t)pch * 128, kUmmaSwizzleNone);
  // V, MN-major: the leading offset steps the block's 64-dim chunks (half,
  // head), 2 KiB apart; the stride offset steps 8 tokens
  const uint64_t dv0 = umma_desc(0u, 2048, 1024, kUmmaSwizzle128);
  const uint32_t idesc_o = umma_idesc_bf16(kTmemRows, HG * D, true);
  const uint32_t s_col = (uint32_t)(HG * D);  // the score buffers follow O

  uint32_t nd = 0;  // stages with data whose scores were issued
  auto issue_scores = [&](uint32_t stage, int nb) {
    tc_fence_after();
    const uint32_t st_s = stage0 + stage * L.stage_bytes;
    const uint32_t sb = tmem + s_col + (nd & 1) * (uint32_t)ntok;
    const uint32_t idesc_s = umma_idesc_bf16(kTmemRows, nb * HG * kBlock, false);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      // 16 dims: K's 64-dim half ks / 4, 32 bytes into its 128-byte rows
      const uint32_t koff = st_s + (uint32_t)(ks >> 2) * 1024u + (uint32_t)(ks & 3) * 32;
      umma_bf16_ts_warp(sb, tmem + q_col + (uint32_t)ks * 8, dk0 + (koff >> 4), idesc_s, ks > 0,
                        lead);
    }
    umma_commit_warp(tb.scores(nd & 1), lead);
    ++nd;
  };

  uint32_t nq = 0;  // query-row hand-overs waited for
  bool fresh = true;
  // stage 0
  if (!mbar_wait(bars, 0)) return false;
  int4 meta = s_meta[0];
  int nb = s_meta[1].z;
  // every stage that brings query rows has them handed over (even one with
  // no data), so the hand-over barrier's phases match the waits
  if (!(meta.w & kEnd)) {
    if (meta.w & kHasQ) {
      if (!mbar_wait(tb.qready(), nq & 1)) return false;
      ++nq;
    }
    if (meta.w & kData) issue_scores(0, nb);
  }
  uint32_t s = 0, ph = 0;
  for (uint32_t n = 0;; ++n) {
    const int flags = meta.w;
    if (flags & kEnd) break;
    const uint32_t s1 = (s + 1 == (uint32_t)S) ? 0u : s + 1;
    const uint32_t ph1 = (s + 1 == (uint32_t)S) ? ph ^ 1u : ph;
    // Wait (bounded) for stage n's probabilities.  Meanwhile, as soon as
    // stage n + 1 is in and needs no new query rows, its scores go to the
    // tensor core ahead of this stage's P.V.  (A phase that one lane sees
    // complete is complete for all: the tests are made warp-uniform.)
    bool have_next = false, scored1 = false;
    int4 meta1 = make_int4(0, 0, 0, 0);
    int nb1 = 0;
    {
      const uint32_t hbar = tb.handed(n & 1), hph = (n >> 1) & 1;
      const unsigned long long t0 = global_ns();
      for (uint32_t spin = 0;; ++spin) {
        if (!have_next && __any_sync(kFull, mbar_test_wait(bars + 8 * s1, ph1))) {
          have_next = true;
          meta1 = s_meta[2 * s1];
          nb1 = s_meta[2 * s1 + 1].z;
          if ((meta1.w & kData) && !(meta1.w & kEnd) && !(meta1.w & kHasQ)) {
            issue_scores(s1, nb1);
            scored1 = true;
          }
        }
        if (__any_sync(kFull, mbar_test_wait(hbar, hph))) break;
        if ((spin & 63) == 63 && __any_sync(kFull, global_ns() - t0 > kWaitLimitNs)) return false;
      }
    }
    tc_fence_after();
    if (flags & kFirst) fresh = true;
    if (flags & kData) {
      const uint32_t vb = stage0 + s * L.stage_bytes + k_area;
      const uint32_t pb = (n & 1) * pbuf_bytes;
      for (int b = 0; b < nb; ++b)  // one MMA of K = 16 tokens per block
        umma_bf16_warp(tmem, dp0 + ((pb + (uint32_t)b * 256) >> 4),
                       dv0 + ((vb + (uint32_t)b * L.kv_bytes) >> 4), idesc_o, !fresh || b > 0,
                       lead);
      fresh = false;
      umma_commit_warp(bars + 8 * (S + s), lead);  // the stage is free once P.V has read it
    } else if (lead) {
      mbar_arrive(bars + 8 * (S + s));
    }
    if (flags & kLast) umma_commit_warp(tb.out(), lead);
    // stage n + 1
    if (!have_next) {
      if (!mbar_wait(bars + 8 * s1, ph1)) return false;
      meta1 = s_meta[2 * s1];
      nb1 = s_meta[2 * s1 + 1].z;
    }
    if (!scored1 && !(meta1.w & kEnd)) {
      if (meta1.w & kHasQ) {
        if (!mbar_wait(tb.qready(), nq & 1)) return false;
        ++nq;
      }
      if (meta1.w & kData) issue_scores(s1, nb1);
    }
    meta = meta1;
    nb = nb1;
    s = s1;
    ph = ph1;
  }
  return true;
}

// The eight softmax warps of the TMEM form (warps 1-8; warp w reaches TMEM
// lanes 32 (w % 4) .. + 31, so warps w and w + 4 share a quadrant).  Thread
// r of either warp of a pair owns MMA row r: the pair splits each stage's
// blocks (the first warp takes the first half), exchanges the rows' maxima
// through shared memory, keeps the same running max and rescale decisions,
// and splits the output columns for the rescale and the epilogue; each warp
// keeps its own part of the running sum.  The query rows of a piece come
// straight from global memory into tensor memory (the form keeps no q ring;
// the producer prefetches them into L2 when it opens the piece's first
// stage, and the softmax warps stage them during the previous piece's
// epilogue when that piece's last stage names it).
template <int D>
__device__ __forceinline__ void consume_tmem(const DecodeParams& p, unsigned char* smem,
                                             const SmemLayout& L, const int4* s_meta,
                                             uint32_t bars, const int* s_prefix,
                                             volatile int* s_abort, int N, long long U, int nhg,
                                             int nvec, int warp, int lane, uint32_t tmem) {
  using T = __nv_bfloat16;
  constexpr int kNcw = kTmemWarps;
  constexpr int kPieces = D / 64;           // 32-column pieces of a row's O each warp owns
  const int G = p.group, NQ = p.query_len, HG = p.heads_per_cta, S = p.stages;
  const int NB = p.blocks_per_stage;
  const int vpk = G * NQ;
  const int R = kTmemRows / HG;             // rows per KV head of the group
  const int cw = warp - 1;
  const int q4 = warp & 3;                  // the TMEM lane quadrant this warp reaches
  const int hf = cw >> 2;                   // which half of the pair
  const int r = q4 * 32 + lane;             // this thread's MMA row
  const int kvl = r / R, v = r - kvl * R;   // its KV head within the group, its vector
  const bool rok = v < vpk;
  const int qhl = kvl * G + (rok ? v / NQ : 0);  // query head within the group
  const int jq = rok ? v % NQ : 0;               // query token
  const int ntok = NB * HG * kBlock;
  const int pch = NB * 2;                   // 16-byte chunks of a P row
  const uint32_t pbuf_bytes = (uint32_t)(kTmemRows * NB * kBlock * 2);
  const uint32_t k_area = (uint32_t)NB * L.kv_bytes;
  const uint32_t vhalf = (uint32_t)HG * kBlock * 128;  // a block's V: one 64-dim half
  volatile int* s_merge = s_abort + 1;
  const TmemBars tb{bars + 8 * (2 * S + (int)L.q_slots)};
  unsigned char* const pb = smem + L.off_pbuf;     // P: two buffers of 128 x NB*16
  // the pairs' exchanges: maxima [stage parity][half][row], sums [piece parity][half][row]
  float* const s_xmax = reinterpret_cast<float*>(pb + 2 * pbuf_bytes);
  float* const s_xl = s_xmax + 4 * kTmemRows;
  const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
  const uint32_t t_o = tmem + lane_base;
  const uint32_t s_col = (uint32_t)(HG * D);
  // this warp's 32-column pieces of the row's O: piece c covers the row's
  // own columns [32c, 32c + 32), i.e. chunk (c / 2, kvl) at offset c % 2
  auto o_col = [&](int c) { return (uint32_t)(((c >> 1) * HG + kvl) * 64 + (c & 1) * 32); };
  const int pc0 = hf * kPieces;
  auto pair_sync = [&]() {
    asm volatile("bar.sync %0, 64;" ::"r"(3 + q4) : "memory");
  };

  // Empty rows see nothing: zeros for all their (token, head) vectors.
  constexpr int kChunks = D * 2 / 16;
  for (int rr = blockIdx.x; rr < p.rows; rr += gridDim.x) {
    if (s_prefix[rr + 1] != s_prefix[rr]) continue;
    for (int vh = cw; vh < NQ * p.heads; vh += kNcw)
      for (int c = lane; c < kChunks; c += 32)
        reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)rr * NQ * p.heads + vh) * D)[c] =
            make_uint4(0u, 0u, 0u, 0u);
  }
  // this row's P: block b's tokens in 16-byte chunks 2b and 2b + 1
  unsigned char* const prow = pb + (r >> 3) * (pch * 128) + (r & 7) * 16;

  // A segment's query vector of this row -> lane r of the Q operand in
  // tensor memory, two dims to a column (as they lie in memory); each warp
  // of the pair copies half of the dims.  Every scores MMA that read the
  // previous query rows is complete (each was waited for below).
  auto stage_q = [&](int qrow, int qkv0) {
    const uint4* src = reinterpret_cast<const uint4*>(
                           static_cast<const T*>(p.q) +
                           (((size_t)qrow * NQ + jq) * p.heads + qkv0 * G + qhl) * D) +
                       hf * (D / 16);
    constexpr int kWords = D / 4;  // this warp's columns: D / 2 dims
    uint32_t w[kWords];
#pragma unroll
    for (int c = 0; c < kWords / 4; ++c) {
      const uint4 v4 = rok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      w[4 * c] = v4.x;
      w[4 * c + 1] = v4.y;
      w[4 * c + 2] = v4.z;
      w[4 * c + 3] = v4.w;
    }
    const uint32_t qt = tmem + lane_base + s_col + 2u * (uint32_t)ntok + (uint32_t)(hf * kWords);
    if constexpr (kWords == 32) {
      tmem_st32(qt, w);
    } else {
      tmem_st16(qt, w);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tb.qready());
  };
  // whether the next segment's query rows are already in place: a
  // segment's last stage stages them (once its own scores are done), so
  // the next segment's first scores can run during this one's epilogue
  bool q_staged = false;

  float m = -INFINITY, l = 0.f;  // l: this warp's part of the running sum
  bool fresh = true;   // no P.V yet in this piece: O holds nothing of it
  uint32_t pv_s = 0, pv_ph = 0;  // stage and phase of the last P.V handed over
  uint32_t npv = 0;    // P.V products handed over so far (all pieces); also
                       // the count of stages with data, whose scores
                       // alternate between two buffers
  uint32_t nout = 0;   // pieces finished
  bool failed = false;
  uint32_t s = 0, ph = 0;
  for (uint32_t n = 0;; ++n, s = (s + 1 == (uint32_t)S) ? (ph ^= 1u, 0u) : s + 1) {
    if (!mbar_wait(bars + 8 * s, ph)) {
      failed = true;
      break;
    }
    const int4 meta = s_meta[2 * s];
    const int4 mm = s_meta[2 * s + 1];
    const int flags = meta.w;
    if (flags & kEnd) break;
    const int nb = mm.z;
    unsigned char* st = smem + s * L.stage_bytes;
    const int qh0 = (flags >> 16) * G;
    const uint32_t b = n & 1;

    if (flags & kFirst) {
      m = -INFINITY;
      l = 0.f;
      fresh = true;
      if (flags & kHasQ) {
        if (!q_staged) stage_q(meta.x, flags >> 16);
        q_staged = false;
      }
    }

    if (flags & kData) {
      const int rem0 = flags & 0xff;  // the row's positions from the stage's first block on
      // V rows that hold no data become zeros (P is 0 there, but 0 * NaN is
      // not); the MMA warp reads V only after the hand-over below.
#pragma unroll
      for (int bb = 0; bb < kTmemMaxBlocks; ++bb) {
        if (bb >= nb) break;
        const int mask = tmem_block_mask(mm, bb);
        const int nvalid = min(kBlock, rem0 - bb * kBlock);
        if (nvalid < kBlock || mask != 0xffff) {
          unsigned char* vblk = st + k_area + bb * L.kv_bytes;
          for (int c = cw * 32 + lane; c < HG * kBlock * kChunks; c += kNcw * 32) {
            const int tr = c / kChunks, dc = c - tr * kChunks;
            const int t = tr % kBlock;
            if (!(t < nvalid && ((mask >> t) & 1)))
              *reinterpret_cast<uint4*>(vblk + swz(tr, dc, vhalf)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (!mbar_wait(tb.scores(npv & 1), (npv >> 1) & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      // This warp's share of the stage: blocks [b0, b0 + nw), at most two
      // (the first warp of the pair takes the first half, rounded up).
      // Their raw scores are read from tensor memory once, by two loads that
      // are always issued (past the warp's share they read the stage's last
      // block again), so that the registers they fill are always defined.
      const int lo_n = (nb + 1) >> 1;
      const int b0 = hf ? lo_n : 0;
      const int nw = hf ? nb - lo_n : lo_n;
      const uint32_t sbase = tmem + lane_base + s_col + (npv & 1) * (uint32_t)ntok;
      const float qs = p.qscale;
      uint32_t sr[2][16];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        tmem_ld16(sbase + (uint32_t)((min(b0 + i, nb - 1) * HG + kvl) * kBlock), sr[i]);
      tmem_wait_ld();
      // Whether block b0 + i is seen in full by every query token of every
      // row (warp-uniform): then it needs no per-token masks.  Rows past the
      // vector count (zero queries) may then compute finite garbage: their
      // state is never written anywhere.
      auto dense = [&](int i) {
        const int bb = b0 + i;
        return tmem_block_mask(mm, bb) == 0xffff && rem0 - bb * kBlock - (NQ - 1) >= kBlock;
      };
      // the tokens of block b0 + i this row's query sees (bit t: token t)
      auto visible = [&](int i) {
        const int bb = b0 + i;
        const int nv = rem0 - bb * kBlock - (NQ - 1 - jq);
        const int upto = nv <= 0 ? 0 : nv >= kBlock ? 0xffff : (1 << nv) - 1;
        return rok ? tmem_block_mask(mm, bb) & upto : 0;
      };
      float mx = -INFINITY;  // this warp's maximum of the scaled scores
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (i >= nw) break;
        if (dense(i)) {
          // the maximum of scale * s is scale times the largest s (the
          // smallest for a negative scale)
          float a8[8];
          if (qs >= 0.f) {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              a8[t] = fmaxf(__uint_as_float(sr[i][t]), __uint_as_float(sr[i][t + 8]));
#pragma unroll
            for (int t = 0; t < 4; ++t) a8[t] = fmaxf(a8[t], a8[t + 4]);
            mx = fmaxf(mx, fmaxf(fmaxf(a8[0], a8[2]), fmaxf(a8[1], a8[3])) * qs);
          } else {
#pragma unroll
            for (int t = 0; t < 8; ++t)
              a8[t] = fminf(__uint_as_float(sr[i][t]), __uint_as_float(sr[i][t + 8]));
#pragma unroll
            for (int t = 0; t < 4; ++t) a8[t] = fminf(a8[t], a8[t + 4]);
            mx = fmaxf(mx, fminf(fminf(a8[0], a8[2]), fminf(a8[1], a8[3])) * qs);
          }
        } else {
          const int vis = visible(i);
#pragma unroll
          for (int t = 0; t < kBlock; ++t)
            if ((vis >> t) & 1) mx = fmaxf(mx, __uint_as_float(sr[i][t]) * qs);
        }
      }
      // the pair's maximum over the whole stage
      float* xm = s_xmax + (npv & 1) * (2 * kTmemRows);
      xm[hf * kTmemRows + r] = mx;
      pair_sync();
      mx = fmaxf(xm[r], xm[kTmemRows + r]);
      // Online softmax; the running max is raised lazily (by more than
      // kRescaleSlack), as in the other tensor forms.  Both warps of the pair
      // see the same maximum and take the same decisions.
      float alpha = 1.f;
      const bool raise = mx > m + kRescaleSlack;  // also the first finite max (m = -inf)
      if (raise) {
        alpha = exp2f(m - mx);
        m = mx;
        l *= alpha;
      }
      if (!fresh && __any_sync(kFull, raise)) {
        // O holds earlier blocks of the piece: once the last P.V handed over
        // is complete (its commit completes that stage's empty barrier),
        // rescale this warp's columns of its rows (1 where the max did not move)
        if (!mbar_wait(bars + 8 * (S + pv_s), pv_ph)) {
          failed = true;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2 * kPieces; ++c) {
          const uint32_t col = o_col(pc0 + (c >> 1)) + (uint32_t)(c & 1) * 16;
          uint32_t o[16];
          tmem_ld16(t_o + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st16(t_o + col, o);
        }
        tmem_wait_st();
      }
      // probabilities 2^(scale * s - m), rounded to bf16 into P (none while
      // the row has seen no position: m = -inf)
      {
        const bool live = m != -INFINITY;
        unsigned char* pr = prow + b * pbuf_bytes;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= nw) break;
          float pv[16];
#pragma unroll
          for (int t = 0; t < kBlock; t += 2) {
            pv[t] = -m;
            pv[t + 1] = -m;
            fma2(pv[t], pv[t + 1], __uint_as_float(sr[i][t]), __uint_as_float(sr[i][t + 1]), qs,
                 qs);
          }
          if (dense(i) && live) {
#pragma unroll
            for (int t = 0; t < kBlock; ++t) pv[t] = ex2_approx(pv[t]);
          } else {
            const int vis = live ? visible(i) : 0;
#pragma unroll
            for (int t = 0; t < kBlock; ++t) pv[t] = ((vis >> t) & 1) ? ex2_approx(pv[t]) : 0.f;
          }
          float s8[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) s8[t] = pv[t] + pv[t + 8];
#pragma unroll
          for (int t = 0; t < 4; ++t) s8[t] += s8[t + 4];
          l += (s8[0] + s8[2]) + (s8[1] + s8[3]);
          uint32_t pk[8];
#pragma unroll
          for (int t2 = 0; t2 < 8; ++t2) pk[t2] = pack_bf16(pv[2 * t2], pv[2 * t2 + 1]);
          const int kc = 2 * (b0 + i);
          *reinterpret_cast<uint4*>(pr + kc * 128) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(pr + (kc + 1) * 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      fence_proxy_async_smem();
      ++npv;
      pv_s = s;
      pv_ph = ph;
      fresh = false;
    }
    // hand the stage over: P (and zeroed V rows, rescaled O) are in place, or
    // the stage had no data and its metadata has been read
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(tb.handed(b));

    if (flags & kLast) {
      if (meta.y > 0) {  // the next segment's query rows, while P.V runs
        stage_q(meta.y - 1, mm.w);
        q_staged = true;
      }
      const int row = meta.x;
      // the piece's last P.V is complete
      if (!mbar_wait(tb.out(), nout & 1)) {
        failed = true;
        break;
      }
      tc_fence_after();
      // the row's whole running sum: both warps' parts
      float* xl = s_xl + (nout & 1) * (2 * kTmemRows);
      xl[hf * kTmemRows + r] = l;
      pair_sync();
      const float lt = xl[r] + xl[kTmemRows + r];
      ++nout;
      if (flags & kFinal) {
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        T* out = static_cast<T*>(p.out) + (((size_t)row * NQ + jq) * p.heads + qh0 + qhl) * D;
#pragma unroll
        for (int c = 0; c < kPieces; ++c) {
          uint32_t o[32];
          if (!fresh) {
            tmem_ld32(t_o + o_col(pc0 + c), o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (rok) {
#pragma unroll
            for (int j = 0; j < 32; j += 8)
              *reinterpret_cast<uint4*>(out + (pc0 + c) * 32 + j) = make_uint4(
                  pack_bf16(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                  pack_bf16(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                  pack_bf16(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                  pack_bf16(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
          }
        }
      } else {
        const size_t slot = (size_t)meta.z * nvec + (size_t)(kvl * vpk + v);
#pragma unroll
        for (int c = 0; c < kPieces; ++c) {
          uint32_t o[32];
          if (!fresh) {
            tmem_ld32(t_o + o_col(pc0 + c), o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (rok) {
            float* a = p.ws_acc + slot * D + (pc0 + c) * 32;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(a + j) =
                  make_float4(__uint_as_float(o[j]), __uint_as_float(o[j + 1]),
                              __uint_as_float(o[j + 2]), __uint_as_float(o[j + 3]));
          }
        }
        if (rok && hf == 0) p.ws_ml[slot] = make_float2(m, lt);
        // this quadrant's rows are vectors [vw, vw + 32) of one KV head; the
        // pair merges 16 of them each
        const int vw = q4 * 32 - kvl * R;
        const int nvq = max(0, min(32, vpk - vw));
        const int nvw = max(0, min(16, nvq - hf * 16));
        finish_cut_row_call<T, D, 8, 4>(p, row, flags >> 16, s_prefix, N, U, nhg, nvec,
                                  kvl * vpk + vw + hf * 16, nvw, kNcw, cw, lane, s_merge);
      }
      tc_fence_before();
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
    *s_abort = 1;
  }
}

// Tensor-core consumer with the block's 16 tokens as the MMA rows (bf16): a
// KV head's query vectors (2 to 64) are the MMA columns, 8 per warp, so one
// to eight warps per KV head read the same K/V tile.  Each warp zeroes the
// tile's empty V rows itself (they all write the same zeros).  Per block:
// S^T = K.Q^T (M = 16 tokens, N = 8 vectors, K = head_dim), the online
// softmax down the columns of S^T, then O^T += V^T.P^T (M = head_dim, N = 8
// vectors, K = 16 tokens).  The probabilities go from the S^T accumulators
// to the P^T operand with one movmatrix transpose per 8 tokens.  Against
// vectors as the rows this takes half the MMAs and half the accumulators.
// Fragment layout of m16n8k16: lane = 4*g + t4 holds rows g and g+8,
// columns 2*t4 and 2*t4+1 of C; column g of B.
template <int D>
__device__ __forceinline__ void consume_mma_t(const DecodeParams& p, unsigned char* smem,
                                              const SmemLayout& L, const int4* s_meta,
                                              uint32_t bars, const int* s_prefix,
                                              volatile int* s_abort, int N, long long U,
                                              int nhg, int nvec, int ncw, int warp, int lane) {
  using T = __nv_bfloat16;
  constexpr int kKs = D / 16;  // k-steps of S^T, and m-tiles of O^T
  const int G = p.group, NQ = p.query_len, HG = p.heads_per_cta, S = p.stages;
  if (warp > ncw) return;
  const int cw = warp - 1;
  const int vpk = G * NQ;               // query vectors per KV head (<= 32)
  const int wpk = ncw / HG;             // warps per KV head: one per 8 vectors
  const int kvl = cw / wpk;             // this warp's KV head within the group
  const int v0w = (cw - kvl * wpk) * kMmaCols;  // its first vector of that KV head
  const int nvw = min(kMmaCols, vpk - v0w);     // and how many it runs (<= 8)
  const int vbase = kvl * vpk + v0w;
  const int g = lane >> 2, t4 = lane & 3;
  const int hq = HG * G;
  const uint32_t half_bytes = (uint32_t)HG * kBlock * 128;
  volatile int* s_merge = s_abort + 1;

  // B-operand column g: the query vector this lane loads.  Accumulator
  // columns 2*t4 + c (c = 0, 1): the vectors whose softmax state it keeps.
  const bool gok = g < nvw;
  const int gv = v0w + (gok ? g : 0);
  const int gqh = kvl * G + gv / NQ, gjq = gv % NQ;
  bool cok[2];
  int cqh[2], cjq[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int v = 2 * t4 + c;
    cok[c] = v < nvw;
    const int vv = v0w + (cok[c] ? v : 0);
    cqh[c] = kvl * G + vv / NQ;
    cjq[c] = vv % NQ;
  }

  // Empty rows see nothing: zeros for all their (token, head) vectors.
  constexpr int kChunks = D * 2 / 16;
  for (int r = blockIdx.x; r < p.rows; r += gridDim.x) {
    if (s_prefix[r + 1] != s_prefix[r]) continue;
    for (int vh = cw; vh < NQ * p.heads; vh += ncw)
      for (int c = lane; c < kChunks; c += 32)
        reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)r * NQ * p.heads + vh) * D)[c] =
            make_uint4(0u, 0u, 0u, 0u);
  }

  uint32_t qb[kKs][2];
  float o[kKs][4], m[2], l[2];
#pragma unroll
  for (int ks = 0; ks < kKs; ++ks) qb[ks][0] = qb[ks][1] = 0u;
#pragma unroll
  for (int mt = 0; mt < kKs; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  m[0] = m[1] = -INFINITY;
  l[0] = l[1] = 0.f;
  const int mi = lane >> 3, i8 = lane & 7;  // ldmatrix: matrix and row this lane addresses

  for (uint32_t n = 0;; ++n) {
    const uint32_t s = n % S;
    if (!mbar_wait(bars + 8 * s, (n / S) & 1)) {
      if (lane == 0) atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
      *s_abort = 1;
      return;
    }
    const int4 meta = s_meta[s];
    const int flags = meta.w;
    if (flags & kEnd) break;
    unsigned char* st = smem + s * L.stage_bytes;
    const uint32_t kbase = smem_u32(st), vbase_s = kbase + L.kv_bytes;
    const int tmask = meta.y & 0xffff;
    const int qh0 = (flags >> 16) * G;

    if (flags & kFirst) {
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < kKs; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      if (flags & kHasQ) {
        // q ring: after the S stages, slots of the CTA's query vectors
        const int qslot = meta.y >> 16;
        const unsigned char* row =
            smem + (size_t)S * L.stage_bytes +
            (size_t)qslot * align_up((uint32_t)nvec * D * sizeof(T), 128) +
            ((size_t)(gjq * hq + gqh) * D + t4 * 2) * sizeof(T);
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
          qb[ks][0] = gok ? *reinterpret_cast<const uint32_t*>(row + ks * 32) : 0u;
          qb[ks][1] = gok ? *reinterpret_cast<const uint32_t*>(row + ks * 32 + 16) : 0u;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (2 * S + qslot));  // the q slot is free
      }
    }

    if (flags & kData) {
      const int rem = flags & 0xff;
      const int nvalid = min(kBlock, rem);
      // V rows that hold no data (past the row's length, or tokens the
      // producer did not gather) become zeros: P is 0 there, but 0 * NaN is not.
      if (nvalid < kBlock || tmask != 0xffff) {
        for (int c = lane; c < kBlock * kChunks; c += 32) {
          const int t = c / kChunks, dc = c - t * kChunks;
          if (!(t < nvalid && ((tmask >> t) & 1)))
            *reinterpret_cast<uint4*>(st + L.kv_bytes + swz(kvl * kBlock + t, dc, half_bytes)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // S^T: two accumulation chains (even and odd k-steps) for latency
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int r = kvl * kBlock + (mi & 1) * 8 + i8;
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
          uint32_t a[4];
          ldsm_x4(kbase + swz(r, ks * 2 + (mi >> 1), half_bytes), a[0], a[1], a[2], a[3]);
          mma_bf16((ks & 1) ? sb : sa, a, qb[ks][0], qb[ks][1]);
        }
      }
      // Online softmax down each column (a vector's 16 scores: tokens g and
      // g + 8 on the 8 lanes of equal t4), with the lazily raised running max
      // of the other tensor form; full blocks need no masks.
      const bool dense = nvalid == kBlock && tmask == 0xffff && rem - (NQ - 1) >= kBlock;
      float pr[2][2];  // [column c][token g, token g + 8]
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float x0 = (sa[c] + sb[c]) * p.qscale;
        float x1 = (sa[2 + c] + sb[2 + c]) * p.qscale;
        if (!dense) {
          const int nv = rem - (NQ - 1 - cjq[c]);  // positions this vector's query sees
          if (!(cok[c] && g < nv && ((tmask >> g) & 1))) x0 = -INFINITY;
          if (!(cok[c] && g + 8 < nv && ((tmask >> (g + 8)) & 1))) x1 = -INFINITY;
        }
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        if (mx > m[c] + kRescaleSlack) {  // also the first finite max (m = -inf)
          const float alpha = exp2f(m[c] - mx);
          m[c] = mx;
          l[c] *= alpha;
#pragma unroll
          for (int mt = 0; mt < kKs; ++mt) {
            o[mt][c] *= alpha;
            o[mt][2 + c] *= alpha;
          }
        }
        pr[c][0] = (dense || x0 != -INFINITY) ? exp2f(x0 - m[c]) : 0.f;
        pr[c][1] = (dense || x1 != -INFINITY) ? exp2f(x1 - m[c]) : 0.f;
        l[c] += pr[c][0] + pr[c][1];
      }
      // P^T operand: the 8x8 blocks [token][vector] of tokens 0-7 and 8-15,
      // transposed to [vector][token] pairs.
      const uint32_t b0 = movm_trans(pack_bf16(pr[0][0], pr[1][0]));
      const uint32_t b1 = movm_trans(pack_bf16(pr[0][1], pr[1][1]));
      // O^T += V^T.P^T: m-tiles of 16 dims, V read transposed
      {
        const int r = kvl * kBlock + (mi >> 1) * 8 + i8;
#pragma unroll
        for (int mt = 0; mt < kKs; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(vbase_s + swz(r, mt * 2 + (mi & 1), half_bytes), a[0], a[1], a[2], a[3]);
          mma_bf16(o[mt], a, b0, b1);
        }
      }
    }

    if (flags & kLast) {
      const int row = meta.x;
      float lt[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        lt[c] = l[c];
        lt[c] += __shfl_xor_sync(kFull, lt[c], 4);
        lt[c] += __shfl_xor_sync(kFull, lt[c], 8);
        lt[c] += __shfl_xor_sync(kFull, lt[c], 16);
      }
      if (flags & kFinal) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!cok[c]) continue;
          const float inv = lt[c] > 0.f ? 1.f / lt[c] : 0.f;
          T* out = static_cast<T*>(p.out) +
                   (((size_t)row * NQ + cjq[c]) * p.heads + qh0 + cqh[c]) * D + g;
#pragma unroll
          for (int mt = 0; mt < kKs; ++mt) {
            out[mt * 16] = __float2bfloat16_rn(o[mt][c] * inv);
            out[mt * 16 + 8] = __float2bfloat16_rn(o[mt][2 + c] * inv);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!cok[c]) continue;
          const size_t slot = (size_t)meta.z * nvec + vbase + 2 * t4 + c;
          float* a = p.ws_acc + slot * D + g;
#pragma unroll
          for (int mt = 0; mt < kKs; ++mt) {
            a[mt * 16] = o[mt][c];
            a[mt * 16 + 8] = o[mt][2 + c];
          }
          if (g == 0) p.ws_ml[slot] = make_float2(m[c], lt[c]);
        }
        finish_cut_row<T, D, 8, 2>(p, row, flags >> 16, s_prefix, N, U, nhg, nvec, vbase, nvw,
                                   ncw, cw, lane, s_merge);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
}

template <typename T, int D, int QW, int MMA>
// The TMEM form launches kTmemWarps + 2 warps, but declares one more in its
// launch bound: on GB300 the code generated for that bound read the 64-vector
// batches 2.5 % faster than for the exact count, in repeated same-box A/B
// runs (and a bound of two more was 2 % slower).  The register cap is the
// same 168 either way.
__global__ void __launch_bounds__(MMA == kMmaTmem ? (kTmemWarps + 3) * 32
                                  : consumers_off_producer(MMA, D) ? kMaxThreadsOffProducer
                                  : MMA ? kMaxThreadsMulti
                                      : (QW <= 2 ? kMaxThreads : kMaxThreadsMulti))
    __maxnreg__(decode_regs(MMA == kMmaTokenRows    ? kConsumerTensor
                            : MMA == kMmaVectorRows ? kConsumerTensorVectorRows
                            : MMA == kMmaTmem       ? kConsumerTensorTmem
                                                    : kConsumerCuda, QW, D))
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using E = Elem<T>;
  constexpr int kDpl = E::kDpl;           // dims per lane per 16-byte load
  constexpr int kLpt = D / kDpl;          // lanes per token row
  constexpr int kTpi = 32 / kLpt;         // tokens per warp-wide load
  constexpr int kNp = kBlock / kTpi;      // loads (partials) per tile per lane
  constexpr int kDup = kLpt / kNp;        // lanes holding the same token's score
  static_assert(kLpt * kDpl == D && kLpt <= 32 && kNp >= 4 && kNp <= kLpt, "tile shape");
  static_assert(kDup * kNp == kLpt && kNp % 4 == 0, "butterfly shape");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned base (the layout's total carries the slack)
  unsigned char* const smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int G = p.group;
  const int NQ = p.query_len;
  const int HG = p.heads_per_cta;
  const int nvec = HG * G * NQ;          // query vectors per CTA
  // consumer warps: per KV head one per 8 vectors (tokens as MMA rows) or
  // one per 16 (vectors as MMA rows); QW vectors per warp on the CUDA cores
  const int ncw = MMA == kMmaTokenRows    ? HG * ((G * NQ + kMmaCols - 1) / kMmaCols)
                  : MMA == kMmaVectorRows ? HG * ((G * NQ + kMmaRows - 1) / kMmaRows)
                  : MMA == kMmaTmem       ? kTmemWarps
                                          : nvec / QW;
  const int S = p.stages;
  const int NBS = MMA == kMmaTmem ? p.blocks_per_stage : 1;  // blocks per stage
  const SmemLayout L = make_layout((int)sizeof(T), D, HG, nvec, S, p.rows, MMA, QW, NBS);

  int4* s_meta = reinterpret_cast<int4*>(smem + L.off_meta);
  const uint32_t bars = smem_u32(smem + L.off_bars);  // full[s] at +8s, empty[s] at +8(S+s)
  float* s_pbuf = reinterpret_cast<float*>(smem + L.off_pbuf);
  int* s_ctx = reinterpret_cast<int*>(smem + L.off_ctx);
  int* s_prefix = reinterpret_cast<int*>(smem + L.off_prefix);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.off_flag);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // the TMEM form's tensor-memory columns and their base address
  const uint32_t tmem_ncols = MMA == kMmaTmem ? (uint32_t)tmem_cols(D, HG, NBS) : 0u;
  uint32_t* const s_tmem = reinterpret_cast<uint32_t*>(smem + L.off_flag + 8);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);  // full: the producer's arrive + tx bytes
      // empty: one arrive per consumer warp (the TMEM form: one commit of
      // the MMAs that read the stage)
      mbar_init(bars + 8 * (S + s), MMA == kMmaTmem ? 1 : ncw);
    }
    for (int j = 0; j < (int)L.q_slots; ++j)
      mbar_init(bars + 8 * (2 * S + j), ncw);  // qfree: every consumer warp has read it
    if (MMA == kMmaTmem) {
      // scores ready [2], probabilities handed over [2] (one arrive per
      // softmax warp), a piece's O complete, all MMAs drained, query rows
      // ready (per softmax warp)
      const uint32_t tb = bars + 8 * (2 * S + (int)L.q_slots);
      const uint32_t counts[kTmemBars] = {1, 1, kTmemWarps, kTmemWarps, 1, 1, kTmemWarps};
      for (int j = 0; j < kTmemBars; ++j) mbar_init(tb + 8 * j, counts[j]);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  if (MMA == kMmaTmem && warp == 1) tmem_alloc(smem_u32(s_tmem), tmem_ncols);
  // Row table: validated lengths and block counts (prefix computed below).
  for (int r = tid; r < p.rows; r += blockDim.x) {
    const int c = checked_ctx(p, r);
    s_ctx[r] = c;
    s_prefix[r + 1] = cdiv(c, kBlock);
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of block counts into prefix[1..rows]
    const int per = (p.rows + 31) / 32;
    const int lo = min(p.rows, lane * per), hi = min(p.rows, lo + per);
    int sum = 0;
    for (int r = lo; r < hi; ++r) sum += s_prefix[r + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int r = lo; r < hi; ++r) {
      run += s_prefix[r + 1];
      s_prefix[r + 1] = run;
    }
    if (lane == 0) s_prefix[0] = 0;
  }
  if (MMA == kMmaTmem) tc_fence_before();
  __syncthreads();
  if (MMA == kMmaTmem) tc_fence_after();

  const int nhg = p.kv_heads / HG;
  const int N = s_prefix[p.rows];                 // blocks per head group
  const long long U = (long long)N * nhg;         // units
  const long long beg = (long long)blockIdx.x * U / gridDim.x;
  const long long end = ((long long)blockIdx.x + 1) * U / gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol = evict_first_policy();
    const size_t tile_elems = (size_t)kBlock * D;
    const size_t block_elems = (size_t)p.kv_heads * tile_elems;
    const T* kp = static_cast<const T*>(p.k_pool);
    const T* vp = static_cast<const T*>(p.v_pool);
    const T* qp = static_cast<const T*>(p.q);
    const uint32_t q_slice = L.q_bytes / NQ;   // one query token's heads of the group
    const uint32_t half_bytes = (uint32_t)HG * kBlock * 128;  // swizzled 64-dim half
    const int slot0 = blockIdx.x * 2;
    unsigned long long walked = 0;
    uint32_t n = 0;   // fills issued (meaningful in lane 0)
    uint32_t qnext = 0;   // q slot of the next query load (lane 0)
    uint32_t qphase = 0;  // laps of the q ring completed
    bool ok = true;

    // Unit u (this lane's): its row, its block within the row, its stage
    // flags and its block id.
    auto unit_at = [&](long long u, int& row, int& blk, int& flags, int& phys) {
      const int hg = (int)(u / N);
      const int rb = (int)(u - (long long)hg * N);
      int lo = 0, hi = p.rows - 1;  // last row r with prefix[r] <= rb
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_prefix[mid] <= rb) lo = mid; else hi = mid - 1;
      }
      const int j = rb - s_prefix[lo];
      const int nb = s_prefix[lo + 1] - s_prefix[lo];
      const long long rs = (long long)hg * N + s_prefix[lo];  // the row's first unit
      // low byte: positions of the row from this block on (clipped at 255)
      int f = min(255, s_ctx[lo] - j * kBlock) | ((hg * HG) << 16);
      if (u == beg || j == 0) f |= kFirst | kHasQ;
      if (u == end - 1 || j == nb - 1) f |= kLast;
      if (rs >= beg && rs + nb <= end) f |= kFinal;
      if (rs > beg) f |= kSlot1;
      row = lo;
      blk = j;
      flags = f;
      if (p.slots)
        phys = slot_block(p.slots + (size_t)lo * p.slot_stride + (size_t)j * kBlock,
                          min(kBlock, s_ctx[lo] - j * kBlock));
      else
        phys = p.block_tables[(size_t)lo * p.max_blocks + j];
    };

    // Wait (lane 0) until the next stage is free.
    auto wait_free = [&]() -> bool {
      if (*s_abort) return false;  // a consumer gave up waiting
      if (n >= (uint32_t)S)
        return mbar_wait(bars + 8 * (S + n % S), ((n / S) - 1) & 1);
      return true;
    };
    // Wait (lane 0) until the next q slot is free: every consumer warp has
    // read the query vectors loaded into it q_slots loads ago.
    auto wait_q = [&]() -> bool {
      if (qphase > 0) return mbar_wait(bars + 8 * (2 * S + qnext), (qphase - 1) & 1);
      return true;
    };
    // Publish the next stage (lane 0): write its metadata, arm its barrier
    // and start its copies (K/V unless the warp gathered them already, q on
    // a segment's first stage, into the next q slot).
    auto publish = [&](int row, int flags, int phys, int mask) {
      const uint32_t s = n % S;
      const uint32_t full = bars + 8 * s;
      const int kv0 = flags >> 16;
      const int qh0 = kv0 * G;
      const uint32_t qslot = qnext;
      s_meta[s] = make_int4(row, mask | (int)(qslot << 16), slot0 + ((flags & kSlot1) ? 1 : 0),
                            flags);
      uint32_t bytes = 0;
      if ((flags & kData) && !(flags & kGathered)) bytes += 2 * L.kv_bytes;
      const bool ring_q = MMA != kMmaTmem && (flags & kHasQ);  // the TMEM form reads q itself
      if (ring_q) bytes += L.q_bytes;
      if (bytes == 0) {
        mbar_arrive(full);
      } else {
        mbar_arrive_tx(full, bytes);
        const uint32_t base = smem_u32(smem + s * L.stage_bytes);
        if ((flags & kData) && !(flags & kGathered)) {
          if constexpr (MMA) {
            // 64-dim halves of the group's [HG * block, D] tile rows, swizzled
            const int y = (phys * p.kv_heads + kv0) * kBlock;
#pragma unroll
            for (int h2 = 0; h2 < D / 64; ++h2) {
              tma_load_2d(base + h2 * half_bytes, &p.tmap_k, h2 * 64, y, full, pol);
              tma_load_2d(base + L.kv_bytes + h2 * half_bytes, &p.tmap_v, h2 * 64, y, full, pol);
            }
          } else {
            const size_t off = (size_t)phys * block_elems + (size_t)kv0 * tile_elems;
            bulk_g2s(base, kp + off, L.kv_bytes, full, pol);
            bulk_g2s(base + L.kv_bytes, vp + off, L.kv_bytes, full, pol);
          }
        }
        if (ring_q) {
          const uint32_t qbase = smem_u32(smem + L.off_q + qslot * L.q_slot_bytes);
          for (int jq = 0; jq < NQ; ++jq)
            bulk_g2s(qbase + jq * q_slice, qp + (((size_t)row * NQ + jq) * p.heads + qh0) * D,
                     q_slice, full, pol);
        }
      }
      if (ring_q) {
        if (++qnext == L.q_slots) {
          qnext = 0;
          ++qphase;
        }
      }
      ++n;
    };
    auto emit = [&](int row, int flags, int phys) -> bool {
      if (!wait_free()) return false;
      if (MMA != kMmaTmem && (flags & kHasQ) && !wait_q()) return false;
      publish(row, flags, phys, 0xffff);
      return true;
    };

    // The TMEM form packs up to NBS consecutive blocks of one segment into a
    // stage and fills a stage in one pass: every lane issues the copies of
    // its own unit of the window, lane 0 arms the stage's full barrier once
    // with their bytes and publishes the stage (metadata, one arrival) when
    // it is full or its segment ends.
    // The open stage's bookkeeping is warp-uniform (every lane keeps the
    // same copy, so a chunk of a window needs no broadcasts): whether a
    // stage is open, its blocks so far and their token masks, whether any
    // holds data or was gathered, its row and its first block's flags.
    int t_open = 0, t_nb = 0, t_row = 0, t_flags = 0, t_mask01 = 0, t_mask23 = 0;
    bool t_data = false, t_gath = false;
    const uint32_t t_vhalf = (uint32_t)HG * kBlock * 128;       // a block's V half
    const uint32_t t_karea = (uint32_t)NBS * L.kv_bytes;
    // A stage that ends a segment also names the next segment's row and
    // head group (row + 1 in its first metadata word's y, 0 when this CTA
    // has none), so the consumers can stage that segment's query rows early.
    auto tmem_close = [&](int last_flags, int next_row1, int next_flags) {
      if (lane == 0) {  // every lane keeps the bookkeeping; lane 0 publishes
        const uint32_t s = n % S;
        int f = t_flags | (last_flags & kLast);
        if (t_data) f |= kData;
        if (t_gath) f |= kGathered;
        const bool nx = (f & kLast) && next_row1 > 0;
        s_meta[2 * s] = make_int4(t_row, nx ? next_row1 : 0, slot0 + ((f & kSlot1) ? 1 : 0), f);
        s_meta[2 * s + 1] = make_int4(t_mask01, t_mask23, t_nb, nx ? next_flags >> 16 : 0);
        mbar_arrive(bars + 8 * s);
      }
      ++n;
      t_open = 0;
    };
    auto add_mask = [&](int bj, int mj) {
      if (bj < 2)
        t_mask01 |= mj << (16 * bj);
      else
        t_mask23 |= mj << (16 * (bj - 2));
      if (mj) t_data = true;
    };
    // The warp gathers unit (row, blk) token by token (slot mode, a block
    // whose slots are not one aligned run) into block b of stage slot s, in
    // the layout the copies write; returns the mask of tokens gathered.
    auto tmem_gather = [&](uint32_t s, int b, int row, int blk, int flags) -> int {
      unsigned char* stg = smem + (size_t)s * L.stage_bytes;
      const int64_t* sp = p.slots + (size_t)row * p.slot_stride + (size_t)blk * kBlock;
      const int nval = min(kBlock, flags & 0xff);
      const long long my = lane < nval ? sp[lane] : -1;
      const bool in_pool = lane < nval && my >= 0 && my < p.pool_blocks * kBlock;
      if (lane < nval && !in_pool) atomicOr(p.status, (uint32_t)NSV_DEV_BAD_BLOCK);
      const int mask = (int)(__ballot_sync(kFull, in_pool) & 0xffffu);
      const int kv0 = flags >> 16;
      constexpr int kVpr = D * (int)sizeof(T) / 16;  // 16-byte vectors per token row
      const int items = kBlock * HG * 2 * kVpr;
      for (int it = lane; it < items; it += 32) {
        const int vv = it % kVpr;
        int rest = it / kVpr;
        const int h = rest % HG;
        rest /= HG;
        const int which = rest & 1;  // 0: K, 1: V
        const int t = rest >> 1;
        if (!((mask >> t) & 1)) continue;
        const long long sl = sp[t];
        const T* src = (which ? vp : kp) +
                       (((size_t)(sl / kBlock) * p.kv_heads + kv0 + h) * kBlock + sl % kBlock) * D;
        const uint32_t dst = which ? t_karea + (uint32_t)b * L.kv_bytes +
                                         swz(h * kBlock + t, vv, t_vhalf)
                                   : swz_grouped<D>((b * HG + h) * kBlock + t, vv);
        *reinterpret_cast<uint4*>(stg + dst) = *(reinterpret_cast<const uint4*>(src) + vv);
      }
      fence_proxy_async_smem();
      __syncwarp();
      return mask;
    };
    // One window of units (lane j holds unit w0 + j, nwin of them valid);
    // x_row1 / x_flags: the row + 1 and flags of the unit after the window
    // (x_row1 = 0: none in this CTA's range).
    auto tmem_window = [&](int nwin, int u_row, int u_blk, int u_flags, int u_phys, int x_row1,
                           int x_flags) -> bool {
      const bool act = lane < nwin;
      const bool tokw = act && u_phys == kTokenWise;
      const bool valid = act && !tokw && u_phys >= 0 && (long long)u_phys < p.pool_blocks;
      if (act && !tokw && !valid) atomicOr(p.status, (uint32_t)NSV_DEV_BAD_BLOCK);
      const unsigned wk = __ballot_sync(kFull, (valid || tokw) && (u_flags >> 16) == 0);
      if (lane == 0) walked += (unsigned long long)__popc(wk);
      const unsigned vmw = __ballot_sync(kFull, valid);  // units copied
      const unsigned gmw = __ballot_sync(kFull, tokw);   // units gathered token by token
      // this unit's index within its segment, modulo the stage size: the
      // blocks before the window of a segment that continues into it are
      // the open stage's (a closed stage holds NBS blocks)
      const unsigned fm = __ballot_sync(kFull, act && (u_flags & kFirst));
      const unsigned upto = fm & (0xffffffffu >> (31 - lane));  // firsts at lanes <= this one
      const int k = upto ? lane - (31 - __clz((int)upto)) : t_nb + lane;
      const bool ends = act && ((k % NBS) == NBS - 1 || (u_flags & kLast));
      const unsigned em = __ballot_sync(kFull, ends);
      int pos = 0;
      while (pos < nwin) {
        const unsigned rest = em & (0xffffffffu << pos);
        const int e = rest ? __ffs((int)rest) - 1 : nwin - 1;
        if (!t_open) {
          const int row0 = __shfl_sync(kFull, u_row, pos);
          const int flags0 = __shfl_sync(kFull, u_flags, pos);
          bool ok2 = true;
          if (lane == 0) ok2 = wait_free();
          if (!__shfl_sync(kFull, ok2, 0)) return false;
          t_open = 1;
          t_nb = 0;
          t_row = row0;
          t_flags = flags0 & ~(kLast | kData | kGathered);
          t_mask01 = t_mask23 = 0;
          t_data = t_gath = false;
          if (flags0 & kHasQ) {
            // the piece's query rows, which the softmax warps load when it
            // starts: into L2 now, a few stages ahead of them (a lane per
            // query token)
            const int qh0 = (flags0 >> 16) * G;
            for (int jq = lane; jq < NQ; jq += 32)
              prefetch_l2(qp + (((size_t)row0 * NQ + jq) * p.heads + qh0) * D,
                          (uint32_t)(HG * G * D * sizeof(T)));
          }
        }
        const uint32_t s = n % S;
        const int nb0 = t_nb;
        const bool mine = lane >= pos && lane <= e;
        const int bl = nb0 + lane - pos;  // this unit's block within the stage
        const unsigned cm = (0xffffffffu >> (31 - e)) & (0xffffffffu << pos);  // lanes pos..e
        const unsigned vm = vmw & cm, gm = gmw & cm;
        // copies: each lane its own unit's (K: one box of both 64-dim
        // halves, V: one box of both halves)
        const uint32_t full = bars + 8 * s;
        if (lane == 0 && vm) mbar_expect_tx(full, (uint32_t)__popc(vm) * 2u * L.kv_bytes);
        if (mine && valid) {
          const uint32_t base = smem_u32(smem + (size_t)s * L.stage_bytes);
          const int y = (u_phys * p.kv_heads + (u_flags >> 16)) * kBlock;
          tma_load_4d(base + (uint32_t)bl * L.kv_bytes, &p.tmap_k, 0, 0, 0, y >> 3, full, pol);
          tma_load_3d(base + t_karea + (uint32_t)bl * L.kv_bytes, &p.tmap_v, 0, y, 0, full,
                      pol);
        }
        if (gm == 0) {
          // a copied block has all its tokens (the consumers mask the
          // positions past the row's end); a block out of the pool none
          for (int j = 0; j <= e - pos; ++j) add_mask(nb0 + j, ((vm >> (pos + j)) & 1) ? 0xffff : 0);
        } else {
          // gathered units, one at a time with the whole warp
          int mymask = (mine && valid) ? 0xffff : 0;
          for (unsigned g2 = gm; g2; g2 &= g2 - 1) {
            const int g = __ffs((int)g2) - 1;
            const int msk = tmem_gather(s, nb0 + g - pos, __shfl_sync(kFull, u_row, g),
                                        __shfl_sync(kFull, u_blk, g),
                                        __shfl_sync(kFull, u_flags, g));
            if (lane == g) mymask = msk;
          }
          for (int j = pos; j <= e; ++j) add_mask(nb0 + j - pos, __shfl_sync(kFull, mymask, j));
          t_gath = true;
        }
        t_nb = nb0 + e - pos + 1;
        if (rest) {  // full, or the segment ends here
          const int src = (e + 1) & 31;
          const int flags_e = __shfl_sync(kFull, u_flags, e);
          const int r1 = __shfl_sync(kFull, u_row, src) + 1, f1 = __shfl_sync(kFull, u_flags, src);
          const bool in_win = e + 1 < nwin;
          tmem_close(flags_e, in_win ? r1 : x_row1, in_win ? f1 : x_flags);
        }
        pos = e + 1;
      }
      return true;
    };
    // Slot mode, a block whose slots are not one aligned run: the whole warp
    // gathers the block's tokens (every head of the group, K and V) into the
    // next stage with 16-byte loads and stores, then lane 0 publishes it with
    // the mask of tokens whose slot lies in the pool.
    const long long pool_slots = p.pool_blocks * kBlock;
    auto gather = [&](int row, int blk, int flags) -> bool {
      bool ok2 = true;
      if (lane == 0) ok2 = wait_free() && (MMA == kMmaTmem || !(flags & kHasQ) || wait_q());
      ok2 = __shfl_sync(kFull, ok2, 0);
      if (!ok2) return false;
      const uint32_t s = __shfl_sync(kFull, n, 0) % S;
      unsigned char* stg = smem + (size_t)s * L.stage_bytes;
      const int64_t* sp = p.slots + (size_t)row * p.slot_stride + (size_t)blk * kBlock;
      const int nval = min(kBlock, flags & 0xff);
      const long long my = lane < nval ? sp[lane] : -1;
      const bool in_pool = lane < nval && my >= 0 && my < pool_slots;
      if (lane < nval && !in_pool) atomicOr(p.status, (uint32_t)NSV_DEV_BAD_BLOCK);
      const int mask = (int)(__ballot_sync(kFull, in_pool) & 0xffffu);
      const int kv0 = flags >> 16;
      constexpr int kVpr = D * (int)sizeof(T) / 16;  // 16-byte vectors per token row
      const int items = kBlock * HG * 2 * kVpr;
      for (int it = lane; it < items; it += 32) {
        const int v = it % kVpr;
        int rest = it / kVpr;
        const int h = rest % HG;
        rest /= HG;
        const int which = rest & 1;  // 0: K, 1: V
        const int t = rest >> 1;
        if (!((mask >> t) & 1)) continue;
        const long long sl = sp[t];
        const T* src = (which ? vp : kp) +
                       (((size_t)(sl / kBlock) * p.kv_heads + kv0 + h) * kBlock + sl % kBlock) * D;
        const uint32_t dst = MMA ? swz(h * kBlock + t, v, half_bytes)
                                 : (uint32_t)((((size_t)h * kBlock + t) * D) * sizeof(T) + v * 16);
        *reinterpret_cast<uint4*>(stg + which * L.kv_bytes + dst) =
            *(reinterpret_cast<const uint4*>(src) + v);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) publish(row, flags | kData | kGathered, 0, mask);
      return true;
    };

    long long w0 = beg;
    int c_row = 0, c_blk = 0, c_flags = 0, c_phys = -1;
    if (w0 + lane < end) unit_at(w0 + lane, c_row, c_blk, c_flags, c_phys);
    // Everything so far read only the step's inputs (lengths, block tables
    // or slots).  The pools and the arrival counters may still be being
    // written by the step's append: wait for it before the first copy.
    // Only this warp waits.  The consumer warps are ordered after it
    // because everything they read or write that the append writes comes
    // after data this warp copied following the wait: K/V through the
    // stages' full barriers, and the arrival counters, which a consumer
    // touches only in finish_cut_row, after its piece's last stage arrived.
    // (griddepcontrol.wait makes the prerequisite grid's writes visible to
    // the whole dependent grid.)  A consumer path that touched the pools or
    // the counters before its first stage would have to wait as well.
    griddep_wait();
    while (w0 < end && ok) {
      // Prefetch the next window's units while this one is issued.
      const long long nw0 = w0 + 32;
      int n_row = 0, n_blk = 0, n_flags = 0, n_phys = -1;
      if (nw0 + lane < end) unit_at(nw0 + lane, n_row, n_blk, n_flags, n_phys);
      const int nwin = (int)min(32ll, end - w0);
      if constexpr (MMA == kMmaTmem) {
        // the unit after this window, if this CTA has one
        const int x_row = __shfl_sync(kFull, n_row, 0), x_flags = __shfl_sync(kFull, n_flags, 0);
        ok = tmem_window(nwin, c_row, c_blk, c_flags, c_phys, nw0 < end ? x_row + 1 : 0, x_flags);
      }
      for (int jj = 0; MMA != kMmaTmem && jj < nwin && ok; ++jj) {
        const int row = __shfl_sync(kFull, c_row, jj);
        int flags = __shfl_sync(kFull, c_flags, jj);
        const int phys = __shfl_sync(kFull, c_phys, jj);
        const int blk = __shfl_sync(kFull, c_blk, jj);
        if (phys == kTokenWise) {
          if ((flags >> 16) == 0) ++walked;
          ok = gather(row, blk, flags);
          continue;
        }
        if (phys >= 0 && (long long)phys < p.pool_blocks) {
          flags |= kData;
          if ((flags >> 16) == 0) ++walked;
        } else if (lane == 0) {
          atomicOr(p.status, (uint32_t)NSV_DEV_BAD_BLOCK);
        }
        if (lane == 0) ok = emit(row, flags, phys);
        ok = __shfl_sync(kFull, ok, 0);
      }
      w0 = nw0;
      c_row = n_row;
      c_blk = n_blk;
      c_flags = n_flags;
      c_phys = n_phys;
    }
    if (lane == 0) {
      if constexpr (MMA == kMmaTmem) {
        // every segment ended with its last unit, which closed its stage
        if (ok) ok = wait_free();
        if (ok) {
          const uint32_t s = n % S;
          s_meta[2 * s] = make_int4(0, 0, 0, kEnd);
          s_meta[2 * s + 1] = make_int4(0, 0, 0, 0);
          mbar_arrive(bars + 8 * s);
          ++n;
        }
      } else {
        if (ok) ok = emit(0, kEnd, 0);
      }
      if (!ok) {
        atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
        *s_abort = 1;
        // Let copies already issued land before the CTA can exit: wait
        // (bounded) for the last phase armed on every stage.
        for (uint32_t k = (n > (uint32_t)S ? n - S : 0); k < n; ++k)
          (void)mbar_wait(bars + 8 * (k % S), (k / S) & 1);
      }
      if (walked) atomicAdd(p.walked, walked);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  if constexpr (MMA == kMmaTmem) {
    if (warp > kTmemWarps + 1) return;
    const uint32_t tmem = *s_tmem;
    const TmemBars tb{bars + 8 * (2 * S + (int)L.q_slots)};
    if (warp == kTmemWarps + 1) {
      // the MMA warp; on a timeout the softmax warps time out too
      if (!tmem_mma_warp<D>(p, smem, L, s_meta, bars, tmem, lane)) {
        if (lane == 0) atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
        *s_abort = 1;
      }
      umma_commit_warp(tb.drained(), lane == 0);  // arrives once every MMA it issued is done
    } else {
      consume_tmem<D>(p, smem, L, s_meta, bars, s_prefix, s_abort, N, U, nhg, nvec, warp, lane,
                      tmem);
    }
    // Free the tensor memory once every role is done with it and the
    // tensor core has finished every MMA (bounded wait on the last commit).
    tc_fence_before();
    asm volatile("bar.sync 2, %0;" ::"r"((kTmemWarps + 1) * 32) : "memory");
    tc_fence_after();
    if (warp == 1) {
      (void)mbar_wait(tb.drained(), 0);
      tc_fence_after();
      tmem_dealloc(tmem, tmem_ncols);
    }
    return;
  }
  if constexpr (consumers_off_producer(MMA, D)) {
    // Off the producer's sub-partition: warps 4, 8, ... idle; the others
    // are consumers 1, 2, 3, 4 (warp 5), ... in order.
    if ((warp & 3) == 0) return;
    consume_mma<D>(p, smem, L, s_meta, bars, s_prefix, s_abort, N, U, nhg, nvec, ncw,
                   warp - (warp >> 2), lane);
    return;
  } else if constexpr (MMA == kMmaVectorRows) {
    consume_mma<D>(p, smem, L, s_meta, bars, s_prefix, s_abort, N, U, nhg, nvec, ncw, warp, lane);
    return;
  } else if constexpr (MMA == kMmaTokenRows) {
    consume_mma_t<D>(p, smem, L, s_meta, bars, s_prefix, s_abort, N, U, nhg, nvec, ncw, warp,
                     lane);
    return;
  } else {
  // A consumer warp serves QW query vectors that read the same KV head: the
  // group's query heads of that KV head and the row's query tokens, so each
  // K/V tile is loaded and widened once for all of them.  Vector v of the CTA
  // is (KV head v / (G*NQ), query head (v / NQ) % G, query token v % NQ).
  if (warp > ncw) return;
  const int cw = warp - 1;
  const int vpk = G * NQ;
  const int v0 = cw * QW;
  const int kvl = v0 / vpk;           // KV head within the group
  const int sub = lane % kLpt;        // which 16-byte slice of a token row
  const int grp = lane / kLpt;        // which token of a warp-wide load
  const int tok = (sub / kDup) * kTpi + grp;  // token whose score this lane ends with
  const int hq = HG * G;              // query heads per group
  float* pbuf = s_pbuf + (size_t)v0 * kBlock;
  volatile int* s_merge = s_abort + 1;

  int qhl[QW], jq[QW];                // query head within the group, query token
#pragma unroll
  for (int k = 0; k < QW; ++k) {
    const int rem = v0 + k - kvl * vpk;
    qhl[k] = kvl * G + rem / NQ;
    jq[k] = rem % NQ;
  }

  // Empty rows see nothing: their output is zero.  CTA c writes the empty
  // rows c, c + G, ...; its consumer warps share the (token, head) vectors.
  for (int r = blockIdx.x; r < p.rows; r += gridDim.x) {
    if (s_prefix[r + 1] != s_prefix[r]) continue;
    for (int vh = cw; vh < NQ * p.heads; vh += ncw)
      if (lane < kLpt)
        *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + ((size_t)r * NQ * p.heads + vh) * D +
                                  sub * kDpl) = make_uint4(0u, 0u, 0u, 0u);
  }

  float qv[QW][kDpl], acc[QW][kDpl], m[QW], l[QW];
#pragma unroll
  for (int k = 0; k < QW; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.f;
#pragma unroll
    for (int e = 0; e < kDpl; ++e) { qv[k][e] = 0.f; acc[k][e] = 0.f; }
  }

  for (uint32_t n = 0;; ++n) {
    const uint32_t s = n % S;
    if (!mbar_wait(bars + 8 * s, (n / S) & 1)) {
      if (lane == 0) atomicOr(p.status, (uint32_t)NSV_DEV_TIMEOUT);
      *s_abort = 1;
      return;
    }
    const int4 meta = s_meta[s];
    const int flags = meta.w;
    if (flags & kEnd) break;
    const unsigned char* st = smem + s * L.stage_bytes;
    const int tmask = meta.y & 0xffff;     // tokens of the block that hold data
    const int qh0 = (flags >> 16) * G;     // the group's first query head

    if (flags & kFirst) {
      // q ring slot of this segment (always slot 0 with 2 or 4 vectors per warp)
      const int qslot = fixed_q_slot(kFormCuda, QW) ? 0 : (meta.y >> 16);
      const unsigned char* qs = smem + L.off_q + qslot * L.q_slot_bytes;
#pragma unroll
      for (int k = 0; k < QW; ++k) {
        m[k] = -INFINITY;
        l[k] = 0.f;
#pragma unroll
        for (int e = 0; e < kDpl; ++e) acc[k][e] = 0.f;
        if (flags & kHasQ) {
          const uint4 raw = *reinterpret_cast<const uint4*>(
              qs + (((size_t)jq[k] * hq + qhl[k]) * D + sub * kDpl) * sizeof(T));
          E::widen(raw, qv[k]);
#pragma unroll
          for (int e = 0; e < kDpl; ++e) qv[k][e] *= p.qscale;
        }
      }
      if (flags & kHasQ) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (2 * S + qslot));  // the q slot is free
      }
    }

    if (flags & kData) {
      const int rem = flags & 0xff;             // the row's positions from this block on
      const int nvalid = min(kBlock, rem);      // what the last query token sees
      const unsigned char* kt = st + (size_t)kvl * kBlock * D * sizeof(T);
      const unsigned char* vt = kt + L.kv_bytes;
      // scores: partial dot products of this lane's 16-byte slice, one
      // widening of the key slice for all QW vectors
      float part[QW][kNp];
#pragma unroll
      for (int i = 0; i < kNp; ++i) {
        const int t = i * kTpi + grp;
        const uint4 raw =
            *reinterpret_cast<const uint4*>(kt + ((size_t)t * D + sub * kDpl) * sizeof(T));
        float kk[kDpl];
        E::widen(raw, kk);
#pragma unroll
        for (int k = 0; k < QW; ++k) {
          float a0 = 0.f, a1 = 0.f;  // even and odd dims, two FMAs per instruction
#pragma unroll
          for (int e = 0; e < kDpl; e += 2) fma2(a0, a1, qv[k][e], qv[k][e + 1], kk[e], kk[e + 1]);
          part[k][i] = a0 + a1;
        }
      }
#pragma unroll
      for (int k = 0; k < QW; ++k) {
        // transposing butterfly: afterwards this lane holds token `tok`'s sum
#pragma unroll
        for (int stp = 0, cnt = kNp; cnt > 1; ++stp, cnt >>= 1) {
          const int o = kLpt >> (stp + 1);
          const bool upper = (sub & o) != 0;
          const int half = cnt >> 1;
#pragma unroll
          for (int j = 0; j < half; ++j) {
            const float send = upper ? part[k][j] : part[k][j + half];
            const float keep = upper ? part[k][j + half] : part[k][j];
            part[k][j] = keep + __shfl_xor_sync(kFull, send, o);
          }
        }
        float sc = part[k][0];
#pragma unroll
        for (int o = kDup >> 1; o >= 1; o >>= 1) sc += __shfl_xor_sync(kFull, sc, o);
        // this vector sees the row's positions before ctx - (NQ - 1 - jq)
        const int nv = rem - (NQ - 1 - jq[k]);
        sc = (tok < nv && ((tmask >> tok) & 1)) ? sc : -INFINITY;
        float mx = sc;
#pragma unroll
        for (int o = kDup; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
        if (mx > m[k]) {  // warp-uniform
          const float alpha = exp2f(m[k] - mx);
          l[k] *= alpha;
#pragma unroll
          for (int e = 0; e < kDpl; ++e) acc[k][e] *= alpha;
          m[k] = mx;
        }
        const float pr = (sc == -INFINITY) ? 0.f : exp2f(sc - m[k]);
        if ((sub % kDup) == 0) pbuf[k * kBlock + grp * kNp + sub / kDup] = pr;
      }
      __syncwarp();
      float pv[QW][kNp];
#pragma unroll
      for (int k = 0; k < QW; ++k) {
#pragma unroll
        for (int i = 0; i < kNp; i += 4) {
          const float4 f = *reinterpret_cast<const float4*>(pbuf + k * kBlock + grp * kNp + i);
          pv[k][i] = f.x; pv[k][i + 1] = f.y; pv[k][i + 2] = f.z; pv[k][i + 3] = f.w;
        }
      }
#pragma unroll
      for (int i = 0; i < kNp; ++i) {
        const int t = i * kTpi + grp;
        if (t < nvalid && ((tmask >> t) & 1)) {  // never touch values past the row's length
          const uint4 raw =
              *reinterpret_cast<const uint4*>(vt + ((size_t)t * D + sub * kDpl) * sizeof(T));
          float v[kDpl];
          E::widen(raw, v);
#pragma unroll
          for (int k = 0; k < QW; ++k) {
#pragma unroll
            for (int e = 0; e < kDpl; e += 2)
              fma2(acc[k][e], acc[k][e + 1], pv[k][i], pv[k][i], v[e], v[e + 1]);
            l[k] += pv[k][i];
          }
        }
      }
    }

    if (flags & kLast) {
      const int row = meta.x;
      float lt[QW], at[QW][kDpl];
#pragma unroll
      for (int k = 0; k < QW; ++k) {
        lt[k] = l[k];
#pragma unroll
        for (int e = 0; e < kDpl; ++e) at[k][e] = acc[k][e];
#pragma unroll
        for (int o = kLpt; o < 32; o <<= 1) {
          lt[k] += __shfl_xor_sync(kFull, lt[k], o);
#pragma unroll
          for (int e = 0; e < kDpl; ++e) at[k][e] += __shfl_xor_sync(kFull, at[k][e], o);
        }
      }
      if (flags & kFinal) {
#pragma unroll
        for (int k = 0; k < QW; ++k) {
          if (lane < kLpt) {
            const float inv = lt[k] > 0.f ? 1.f / lt[k] : 0.f;
#pragma unroll
            for (int e = 0; e < kDpl; ++e) at[k][e] *= inv;
            T* o = static_cast<T*>(p.out) +
                   (((size_t)row * NQ + jq[k]) * p.heads + qh0 + qhl[k]) * D + sub * kDpl;
            *reinterpret_cast<uint4*>(o) = E::narrow(at[k]);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < QW; ++k) {
          const size_t slot = (size_t)meta.z * nvec + v0 + k;
          if (lane < kLpt) {
            float* a = p.ws_acc + slot * D + sub * kDpl;
#pragma unroll
            for (int e = 0; e < kDpl; e += 4)
              *reinterpret_cast<float4*>(a + e) =
                  make_float4(at[k][e], at[k][e + 1], at[k][e + 2], at[k][e + 3]);
          }
          if (lane == 0) p.ws_ml[slot] = make_float2(m[k], lt[k]);
        }
        finish_cut_row<T, D, 32 / QW, 2>(p, row, flags >> 16, s_prefix, N, U, nhg, nvec, v0,
                                              QW, ncw, cw, lane, s_merge);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
  }  // CUDA-core consumer
}

template <typename T, int D, int QW, int MMA>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(decode_kernel<T, D, QW, MMA>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

template <typename T, int D>
cudaError_t set_attrs() {
  cudaError_t e;
  if ((e = set_attr<T, D, 1, 0>()) != cudaSuccess) return e;
  if ((e = set_attr<T, D, 2, 0>()) != cudaSuccess) return e;
  if ((e = set_attr<T, D, 4, 0>()) != cudaSuccess) return e;
  if constexpr (sizeof(T) == 2) {
    if ((e = set_attr<T, D, 1, kMmaVectorRows>()) != cudaSuccess) return e;
    if ((e = set_attr<T, D, 1, kMmaTmem>()) != cudaSuccess) return e;
    return set_attr<T, D, 1, kMmaTokenRows>();
  }
  return cudaSuccess;
}

// One launch; `pdl` lets it start while the previous kernel on the stream
// (the step's append) is still running (programmatic stream serialization;
// the kernel waits for it before touching what it writes).
cudaError_t launch_one(void (*kernel)(const DecodeParams), const DecodeParams& p, int grid,
                       int threads, int smem, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename T, int D>
cudaError_t launch_typed(const DecodeParams& p, int qw, int consumer, int grid, int threads,
                         int smem, cudaStream_t stream, bool pdl) {
  if constexpr (sizeof(T) == 2) {
    if (consumer == kConsumerTensor)
      return launch_one(decode_kernel<T, D, 1, kMmaTokenRows>, p, grid, threads, smem, stream,
                        pdl);
    if (consumer == kConsumerTensorVectorRows)
      return launch_one(decode_kernel<T, D, 1, kMmaVectorRows>, p, grid, threads, smem, stream,
                        pdl);
    if (consumer == kConsumerTensorTmem)
      return launch_one(decode_kernel<T, D, 1, kMmaTmem>, p, grid, threads, smem, stream, pdl);
  }
  if (qw == 4) return launch_one(decode_kernel<T, D, 4, 0>, p, grid, threads, smem, stream, pdl);
  if (qw == 2) return launch_one(decode_kernel<T, D, 2, 0>, p, grid, threads, smem, stream, pdl);
  return launch_one(decode_kernel<T, D, 1, 0>, p, grid, threads, smem, stream, pdl);
}

template <typename T, int D>
cudaError_t occupancy_typed(int qw, int consumer, int threads, int smem, int* ctas) {
  const void* fn;
  if constexpr (sizeof(T) == 2) {
    if (consumer == kConsumerTensor)
      fn = reinterpret_cast<const void*>(decode_kernel<T, D, 1, kMmaTokenRows>);
    else if (consumer == kConsumerTensorVectorRows)
      fn = reinterpret_cast<const void*>(decode_kernel<T, D, 1, kMmaVectorRows>);
    else if (consumer == kConsumerTensorTmem)
      fn = reinterpret_cast<const void*>(decode_kernel<T, D, 1, kMmaTmem>);
    else
      fn = qw == 4   ? reinterpret_cast<const void*>(decode_kernel<T, D, 4, 0>)
           : qw == 2 ? reinterpret_cast<const void*>(decode_kernel<T, D, 2, 0>)
                     : reinterpret_cast<const void*>(decode_kernel<T, D, 1, 0>);
  } else {
    fn = qw == 4   ? reinterpret_cast<const void*>(decode_kernel<T, D, 4, 0>)
         : qw == 2 ? reinterpret_cast<const void*>(decode_kernel<T, D, 2, 0>)
                   : reinterpret_cast<const void*>(decode_kernel<T, D, 1, 0>);
  }
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, fn, threads, (size_t)smem);
}

}  // namespace

cudaError_t decode_occupancy(int dtype, int head_dim, int qw, int consumer, int threads,
                             int smem, int* ctas) {
  if (dtype == NSV_F32)
    return head_dim == 64 ? occupancy_typed<float, 64>(qw, consumer, threads, smem, ctas)
                          : occupancy_typed<float, 128>(qw, consumer, threads, smem, ctas);
  return head_dim == 64 ? occupancy_typed<__nv_bfloat16, 64>(qw, consumer, threads, smem, ctas)
                        : occupancy_typed<__nv_bfloat16, 128>(qw, consumer, threads, smem, ctas);
}

cudaError_t launch_wait_probe(unsigned long long limit_ns, unsigned long long* result,
                              uint32_t* status, cudaStream_t stream) {
  bounded_wait_probe<<<1, 32, 0, stream>>>(limit_ns, result, status);
  return cudaGetLastError();
}

cudaError_t prepare_decode_kernels() {
  cudaError_t e;
  if ((e = set_attrs<float, 64>()) != cudaSuccess) return e;
  if ((e = set_attrs<float, 128>()) != cudaSuccess) return e;
  if ((e = set_attrs<__nv_bfloat16, 64>()) != cudaSuccess) return e;
  return set_attrs<__nv_bfloat16, 128>();
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int qw, int consumer,
                          int grid, int threads, int smem, cudaStream_t stream, bool pdl) {
  if (dtype == NSV_F32)
    return head_dim == 64
               ? launch_typed<float, 64>(p, qw, consumer, grid, threads, smem, stream, pdl)
               : launch_typed<float, 128>(p, qw, consumer, grid, threads, smem, stream, pdl);
  return head_dim == 64
             ? launch_typed<__nv_bfloat16, 64>(p, qw, consumer, grid, threads, smem, stream, pdl)
             : launch_typed<__nv_bfloat16, 128>(p, qw, consumer, grid, threads, smem, stream,
                                                pdl);
}

}  // namespace nsv
