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
//  * A persistent grid of CTAs (SM count x resident CTAs).  Work items are
//    (row, split, head group): a head group is `heads_per_cta` KV heads with
//    all their query heads, a split is `chunk_blocks` consecutive blocks of
//    the row.  Every CTA builds the same compacted item list from
//    context_lens in shared memory (no host read of the lengths, so the plan
//    depends on shape alone) and takes items blockIdx.x, +gridDim.x, ...
//  * Warp 0 is the producer.  Per block it issues two cp.async.bulk copies
//    (the head group's K tiles and V tiles are each one contiguous run in the
//    [block][kv_head][token][dim] pool) into a ring of shared-memory stages
//    guarded by mbarriers, plus the query vectors on an item's first stage.
//    Block ids of the next window are prefetched a window ahead.
//  * Warps 1..N are consumers, one per query head.  A lane owns 16 bytes of
//    a key row; the score of each token of the tile is reduced with a
//    transposing butterfly (one shuffle per token instead of five), the
//    tile max with a plain butterfly, probabilities go through shared memory
//    to the lanes that own the value dims, and P.V accumulates in fp32.
//  * An item that covers its row's whole length writes `out` directly;
//    otherwise it writes its (m, l, acc) partial and a combine kernel merges
//    the row's partials (flash-decoding style).
//  * No tensor cores: one query per head makes each tile a GEMV.
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

// Wait for the phase of `bar` with the given parity to complete; false if
// it has not after kWaitLimitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
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

// Validated context length (a bad one is read as 0 and flagged).
__device__ __forceinline__ int checked_ctx(const DecodeParams& p, int r) {
  int c = p.context_lens[r];
  if (c < 0 || c > p.max_blocks * kBlock) {
    atomicOr(p.status, (uint32_t)NSV_DEV_BAD_CTX);
    c = 0;
  }
  return c;
}

// Work items of a row: its splits (at least one, so an empty row still gets
// an item that writes its zero output).
__device__ __forceinline__ int row_splits(int ctx, int chunk_blocks) {
  int nb = cdiv(ctx, kBlock);
  int s = cdiv(nb, chunk_blocks);
  return s > 0 ? s : 1;
}

struct Item {
  int row, hg, split, ctx, b0, b1;  // blocks [b0, b1) of the row
  bool final_;                      // the row has one split
};

__device__ __forceinline__ Item item_at(int it, int nhg, const int* s_prefix, const int* s_ctx,
                                        int rows, int chunk_blocks) {
  Item I;
  const int rs = it / nhg;
  I.hg = it - rs * nhg;
  // largest row r with prefix[r] <= rs (prefix is strictly increasing)
  int lo = 0, hi = rows - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= rs) lo = mid; else hi = mid - 1;
  }
  I.row = lo;
  I.split = rs - s_prefix[lo];
  I.ctx = s_ctx[lo];
  const int nb = cdiv(I.ctx, kBlock);
  I.b0 = I.split * chunk_blocks;
  I.b1 = min(nb, I.b0 + chunk_blocks);
  if (I.b1 < I.b0) I.b1 = I.b0;
  I.final_ = (s_prefix[lo + 1] - s_prefix[lo]) == 1;
  return I;
}

template <typename T, int D>
__global__ void __launch_bounds__(kMaxThreads, 1) decode_kernel(const DecodeParams p) {
  using E = Elem<T>;
  constexpr int kDpl = E::kDpl;           // dims per lane per 16-byte load
  constexpr int kLpt = D / kDpl;          // lanes per token row
  constexpr int kTpi = 32 / kLpt;         // tokens per warp-wide load
  constexpr int kNp = kBlock / kTpi;      // loads (partials) per tile per lane
  constexpr int kDup = kLpt / kNp;        // lanes holding the same token's score
  static_assert(kLpt * kDpl == D && kLpt <= 32 && kNp >= 4 && kNp <= kLpt, "tile shape");
  static_assert(kDup * kNp == kLpt && kNp % 4 == 0, "butterfly shape");

  extern __shared__ __align__(128) unsigned char smem[];
  const int G = p.group;
  const int HG = p.heads_per_cta;
  const int ncw = HG * G;
  const int S = p.stages;
  const SmemLayout L = make_layout((int)sizeof(T), D, HG, G, S, p.rows);

  int4* s_meta = reinterpret_cast<int4*>(smem + L.off_meta);
  const uint32_t bars = smem_u32(smem + L.off_bars);  // full[s] at +8s, empty[s] at +8(S+s)
  float* s_pbuf = reinterpret_cast<float*>(smem + L.off_pbuf);
  int* s_ctx = reinterpret_cast<int*>(smem + L.off_ctx);
  int* s_prefix = reinterpret_cast<int*>(smem + L.off_prefix);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.off_flag);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8 * s, 1);              // full: the producer's arrive + tx bytes
      mbar_init(bars + 8 * (S + s), ncw);      // empty: one arrive per consumer warp
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // Row table: validated lengths and split counts (prefix computed below).
  for (int r = tid; r < p.rows; r += blockDim.x) {
    const int c = checked_ctx(p, r);
    s_ctx[r] = c;
    s_prefix[r + 1] = row_splits(c, p.chunk_blocks);
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of split counts into prefix[1..rows]
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
  __syncthreads();

  const int nhg = p.kv_heads / HG;
  const int total = s_prefix[p.rows] * nhg;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    const uint64_t pol = evict_first_policy();
    const size_t tile_elems = (size_t)kBlock * D;
    const size_t block_elems = (size_t)p.kv_heads * tile_elems;
    const T* kp = static_cast<const T*>(p.k_pool);
    const T* vp = static_cast<const T*>(p.v_pool);
    const T* qp = static_cast<const T*>(p.q);
    unsigned long long walked = 0;
    uint32_t n = 0;  // fills issued (meaningful in lane 0)
    bool ok = true;

    // Emit one stage (lane 0 only): wait for it to be free, write its
    // metadata, arm its barrier and start its copies.
    auto emit = [&](int row, int qh0, int split, int flags, int phys) -> bool {
      const uint32_t s = n % S;
      const uint32_t full = bars + 8 * s, empty = bars + 8 * (S + s);
      if (*s_abort) return false;  // a consumer gave up waiting
      if (n >= (uint32_t)S) {
        if (!mbar_wait(empty, ((n / S) - 1) & 1)) return false;
      }
      s_meta[s] = make_int4(row, qh0, split, flags);
      uint32_t bytes = 0;
      if (flags & kData) bytes += 2 * L.kv_bytes;
      if (flags & kHasQ) bytes += L.q_bytes;
      if (bytes == 0) {
        mbar_arrive(full);
      } else {
        mbar_arrive_tx(full, bytes);
        const uint32_t base = smem_u32(smem + s * L.stage_bytes);
        if (flags & kData) {
          const size_t off = (size_t)phys * block_elems + (size_t)(flags >> 16) * tile_elems;
          bulk_g2s(base, kp + off, L.kv_bytes, full, pol);
          bulk_g2s(base + L.kv_bytes, vp + off, L.kv_bytes, full, pol);
        }
        if (flags & kHasQ) {
          bulk_g2s(base + 2 * L.kv_bytes, qp + ((size_t)row * p.heads + qh0) * D, L.q_bytes,
                   full, pol);
        }
      }
      ++n;
      return true;
    };

    int it = blockIdx.x;
    Item cur{};
    int w0 = 0;
    int cur_id = -1;
    if (it < total) {
      cur = item_at(it, nhg, s_prefix, s_ctx, p.rows, p.chunk_blocks);
      w0 = cur.b0;
      if (w0 + lane < cur.b1) cur_id = p.block_tables[(size_t)cur.row * p.max_blocks + w0 + lane];
    }
    while (it < total && ok) {
      // Locate the next window (32 blocks) and prefetch its block ids.
      int nit = it, nw0 = w0 + 32;
      Item nxt = cur;
      if (nw0 >= cur.b1) {
        nit = it + gridDim.x;
        if (nit < total) {
          nxt = item_at(nit, nhg, s_prefix, s_ctx, p.rows, p.chunk_blocks);
          nw0 = nxt.b0;
        }
      }
      int nxt_id = -1;
      if (nit < total && nw0 + lane < nxt.b1)
        nxt_id = p.block_tables[(size_t)nxt.row * p.max_blocks + nw0 + lane];

      const int qh0 = cur.hg * HG * G;
      const int fin = cur.final_ ? kFinal : 0;
      const int kv0 = cur.hg * HG;
      const int nwin = min(32, cur.b1 - w0);
      if (nwin <= 0) {
        // An empty row: one stage with no data that makes its output zero.
        if (lane == 0) ok = emit(cur.row, qh0, cur.split, kFirst | kLast | fin, 0);
        ok = __shfl_sync(kFull, ok, 0);
      }
      for (int jj = 0; jj < nwin && ok; ++jj) {
        const int phys = __shfl_sync(kFull, cur_id, jj);
        const int j = w0 + jj;
        const int nvalid = min(kBlock, cur.ctx - j * kBlock);
        int flags = nvalid | fin | (kv0 << 16);
        if (j == cur.b0) flags |= kFirst | kHasQ;
        if (j == cur.b1 - 1) flags |= kLast;
        if (phys >= 0 && (long long)phys < p.pool_blocks) {
          flags |= kData;
          if (cur.hg == 0) ++walked;
        } else if (lane == 0) {
          atomicOr(p.status, (uint32_t)NSV_DEV_BAD_BLOCK);
        }
        if (lane == 0) ok = emit(cur.row, qh0, cur.split, flags, phys);
        ok = __shfl_sync(kFull, ok, 0);
      }
      it = nit;
      w0 = nw0;
      cur = nxt;
      cur_id = nxt_id;
    }
    if (lane == 0) {
      if (ok) ok = emit(0, 0, 0, kEnd, 0);
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
  if (warp > ncw) return;
  const int cw = warp - 1;            // query head within the CTA's group
  const int kvl = cw / G;             // KV head within the CTA's group
  const int sub = lane % kLpt;        // which 16-byte slice of a token row
  const int grp = lane / kLpt;        // which token of a warp-wide load
  const int tok = (sub / kDup) * kTpi + grp;  // token whose score this lane ends with
  float* pbuf = s_pbuf + cw * kBlock;

  float qv[kDpl], acc[kDpl];
  float m = -INFINITY, l = 0.f;
#pragma unroll
  for (int e = 0; e < kDpl; ++e) { qv[e] = 0.f; acc[e] = 0.f; }

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

    if (flags & kFirst) {
      m = -INFINITY;
      l = 0.f;
#pragma unroll
      for (int e = 0; e < kDpl; ++e) acc[e] = 0.f;
      if (flags & kHasQ) {
        const uint4 raw = *reinterpret_cast<const uint4*>(st + 2 * L.kv_bytes +
                                                          ((size_t)cw * D + sub * kDpl) * sizeof(T));
        E::widen(raw, qv);
#pragma unroll
        for (int e = 0; e < kDpl; ++e) qv[e] *= p.qscale;
      }
    }

    if (flags & kData) {
      const int nvalid = flags & 0xff;
      const unsigned char* kt = st + (size_t)kvl * kBlock * D * sizeof(T);
      const unsigned char* vt = kt + L.kv_bytes;
      // scores: partial dot products of this lane's 16-byte slice
      float part[kNp];
#pragma unroll
      for (int i = 0; i < kNp; ++i) {
        const int t = i * kTpi + grp;
        const uint4 raw =
            *reinterpret_cast<const uint4*>(kt + ((size_t)t * D + sub * kDpl) * sizeof(T));
        float k[kDpl];
        E::widen(raw, k);
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < kDpl; ++e) a = fmaf(qv[e], k[e], a);
        part[i] = a;
      }
      // transposing butterfly: afterwards this lane holds token `tok`'s sum
#pragma unroll
      for (int stp = 0, cnt = kNp; cnt > 1; ++stp, cnt >>= 1) {
        const int o = kLpt >> (stp + 1);
        const bool upper = (sub & o) != 0;
        const int half = cnt >> 1;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = upper ? part[j] : part[j + half];
          const float keep = upper ? part[j + half] : part[j];
          part[j] = keep + __shfl_xor_sync(kFull, send, o);
        }
      }
      float sc = part[0];
#pragma unroll
      for (int o = kDup >> 1; o >= 1; o >>= 1) sc += __shfl_xor_sync(kFull, sc, o);
      sc = (tok < nvalid) ? sc : -INFINITY;
      float mx = sc;
#pragma unroll
      for (int o = kDup; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (mx > m) {  // warp-uniform
        const float alpha = exp2f(m - mx);
        l *= alpha;
#pragma unroll
        for (int e = 0; e < kDpl; ++e) acc[e] *= alpha;
        m = mx;
      }
      const float pr = exp2f(sc - m);
      if ((sub % kDup) == 0) pbuf[grp * kNp + sub / kDup] = pr;
      __syncwarp();
      float pv[kNp];
#pragma unroll
      for (int i = 0; i < kNp; i += 4) {
        const float4 f = *reinterpret_cast<const float4*>(pbuf + grp * kNp + i);
        pv[i] = f.x; pv[i + 1] = f.y; pv[i + 2] = f.z; pv[i + 3] = f.w;
      }
#pragma unroll
      for (int i = 0; i < kNp; ++i) {
        const int t = i * kTpi + grp;
        if (t < nvalid) {  // never touch values past the row's length
          const uint4 raw =
              *reinterpret_cast<const uint4*>(vt + ((size_t)t * D + sub * kDpl) * sizeof(T));
          float v[kDpl];
          E::widen(raw, v);
#pragma unroll
          for (int e = 0; e < kDpl; ++e) acc[e] = fmaf(pv[i], v[e], acc[e]);
          l += pv[i];
        }
      }
    }

    if (flags & kLast) {
      float lt = l;
      float at[kDpl];
#pragma unroll
      for (int e = 0; e < kDpl; ++e) at[e] = acc[e];
#pragma unroll
      for (int o = kLpt; o < 32; o <<= 1) {
        lt += __shfl_xor_sync(kFull, lt, o);
#pragma unroll
        for (int e = 0; e < kDpl; ++e) at[e] += __shfl_xor_sync(kFull, at[e], o);
      }
      const int row = meta.x, qh = meta.y + cw, split = meta.z;
      if (flags & kFinal) {
        if (lane < kLpt) {
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
          for (int e = 0; e < kDpl; ++e) at[e] *= inv;
          T* o = static_cast<T*>(p.out) + ((size_t)row * p.heads + qh) * D + sub * kDpl;
          *reinterpret_cast<uint4*>(o) = E::narrow(at);
        }
      } else {
        const size_t slot = ((size_t)row * p.heads + qh) * p.max_splits + split;
        if (lane < kLpt) {
          float* a = p.ws_acc + slot * D + sub * kDpl;
#pragma unroll
          for (int e = 0; e < kDpl; e += 4)
            *reinterpret_cast<float4*>(a + e) = make_float4(at[e], at[e + 1], at[e + 2], at[e + 3]);
        }
        if (lane == 0) p.ws_ml[slot] = make_float2(m, lt);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (S + s));
  }
}

// Merge the partial softmax states of rows that were split.  One warp per
// (row, query head); rows with a single split were finished by the decode
// kernel and are skipped.
template <typename T, int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
  constexpr int kPer = D / 32;  // dims per lane
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.rows * p.heads) return;
  const int row = gw / p.heads;
  int c = p.context_lens[row];
  if (c < 0 || c > p.max_blocks * kBlock) c = 0;  // flagged by the decode kernel
  const int nsplit = cdiv(cdiv(c, kBlock), p.chunk_blocks);
  if (nsplit <= 1) return;
  const size_t base = (size_t)gw * p.max_splits;
  float M = -INFINITY;
  for (int i = lane; i < nsplit; i += 32) M = fmaxf(M, p.ws_ml[base + i].x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float Lsum = 0.f;
  float a[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) a[e] = 0.f;
  for (int i = 0; i < nsplit; ++i) {
    const float2 ml = p.ws_ml[base + i];
    const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - M);
    Lsum = fmaf(w, ml.y, Lsum);
    const float* src = p.ws_acc + (base + i) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; ++e) a[e] = fmaf(w, src[e], a[e]);
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  T* o = static_cast<T*>(p.out) + (size_t)gw * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    if constexpr (sizeof(T) == 4) {
      o[e] = a[e] * inv;
    } else {
      o[e] = __float2bfloat16_rn(a[e] * inv);
    }
  }
}

template <typename T, int D>
cudaError_t set_attrs() {
  return cudaFuncSetAttribute(decode_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              227 * 1024);
}

}  // namespace

cudaError_t prepare_decode_kernels() {
  cudaError_t e;
  if ((e = set_attrs<float, 64>()) != cudaSuccess) return e;
  if ((e = set_attrs<float, 128>()) != cudaSuccess) return e;
  if ((e = set_attrs<__nv_bfloat16, 64>()) != cudaSuccess) return e;
  return set_attrs<__nv_bfloat16, 128>();
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int grid, int threads,
                          int smem, cudaStream_t stream) {
  if (dtype == NSV_F32) {
    if (head_dim == 64)
      decode_kernel<float, 64><<<grid, threads, smem, stream>>>(p);
    else
      decode_kernel<float, 128><<<grid, threads, smem, stream>>>(p);
  } else {
    if (head_dim == 64)
      decode_kernel<__nv_bfloat16, 64><<<grid, threads, smem, stream>>>(p);
    else
      decode_kernel<__nv_bfloat16, 128><<<grid, threads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, int dtype, int head_dim, cudaStream_t stream) {
  const long long warps = (long long)p.rows * p.heads;
  if (warps == 0) return cudaSuccess;
  const int wpb = 8;
  const int grid = (int)((warps + wpb - 1) / wpb);
  if (dtype == NSV_F32) {
    if (head_dim == 64)
      combine_kernel<float, 64><<<grid, wpb * 32, 0, stream>>>(p);
    else
      combine_kernel<float, 128><<<grid, wpb * 32, 0, stream>>>(p);
  } else {
    if (head_dim == 64)
      combine_kernel<__nv_bfloat16, 64><<<grid, wpb * 32, 0, stream>>>(p);
    else
      combine_kernel<__nv_bfloat16, 128><<<grid, wpb * 32, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace nsv
