// Host side of the C ABI declared in include/nsv.h: argument checks, the
// shape-only launch planner, per-device state (the device status word and
// the library-owned workspace) and the entry points.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "nsv_common.cuh"

namespace nsv {

// Sticky device status (NSV_DEV_* bits) and the walked-block counter.
__device__ uint32_t g_status;
__device__ unsigned long long g_walked;
// Result of the bounded-wait self-test: gave up (0/1), nanoseconds waited.
__device__ unsigned long long g_probe[2];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSmemPerSm = 228 * 1024;     // shared memory per SM on sm_103
constexpr int kSmemPerCta = 227 * 1024;    // opt-in maximum per CTA
constexpr int kSmemReserved = 1024;        // per-CTA system reservation
constexpr int kThreadsPerSm = 2048;
constexpr int kMaxCtasPerSm = 8;        // resident CTAs per SM a plan may ask for
constexpr int kEnoughWarpsPerSm = 16;   // consumer warps per SM that keep HBM busy

struct DeviceState {
  bool ready = false;
  void* ctx = nullptr;  // the CUDA context the addresses below belong to
  uint32_t* status = nullptr;
  unsigned long long* walked = nullptr;
  int num_sms = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// so that the library needs no link against libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail() {
  (void)cudaGetLastError();  // do not leave a stale error for the next caller
  return NSV_ERR_CUDA;
}

// cuCtxGetCurrent, reached like cuTensorMapEncodeTiled below (loaded once).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn g_ctx_current = nullptr;
std::once_flag g_ctx_once;

}  // namespace

void* current_cuda_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    else
      (void)cudaGetLastError();
  });
  CUcontext c = nullptr;
  if (!g_ctx_current || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
  return reinterpret_cast<void*>(c);
}

namespace {

// Per-device set-up on first use: symbol addresses of the status words,
// kernel attributes, SM count.  Needs the device current.  Done again when
// a different context is current on the device than the one the addresses
// were taken in (the old one was destroyed, by cudaDeviceReset for one): its
// workspace went with it and is dropped, not freed.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_fail();
  if (dev < 0 || dev >= kMaxDevices) return NSV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ready) {
    void* now = current_cuda_context();
    if (now != nullptr && now != d.ctx) {
      d.ready = false;
      d.ws = nullptr;
      d.ws_bytes = 0;
    }
  }
  if (!d.ready) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status) != cudaSuccess)
      return cuda_fail();
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.walked), g_walked) != cudaSuccess)
      return cuda_fail();
    if (prepare_decode_kernels() != cudaSuccess) return cuda_fail();
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_fail();
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return cuda_fail();
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ctx = current_cuda_context();  // bound by the runtime calls above
    d.ready = true;
  }
  *out = &d;
  return NSV_OK;
}

int elem_bytes(int dtype) { return dtype == NSV_F32 ? 4 : 2; }

int query_len(const nsv_shape* s) { return s->query_len > 0 ? s->query_len : 1; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const nsv_shape* s) {
  if (!s) return NSV_ERR_NULLPTR;
  if (s->dtype != NSV_F32 && s->dtype != NSV_BF16) return NSV_ERR_DTYPE;
  if (s->query_len < 0 || s->query_len > kMaxVectorsPerKvHead) return NSV_ERR_SHAPE;
  if (s->rows < 0 || s->rows > kMaxRows) return NSV_ERR_SHAPE;
  if (s->num_heads < 1 || s->num_kv_heads < 1 || s->num_heads % s->num_kv_heads != 0)
    return NSV_ERR_SHAPE;
  if ((s->num_heads / s->num_kv_heads) * (s->query_len > 0 ? s->query_len : 1) >
      kMaxVectorsPerKvHead)
    return NSV_ERR_SHAPE;
  if (s->head_dim != 64 && s->head_dim != 128) return NSV_ERR_UNSUPPORTED;
  if (s->block_size != kBlock) return NSV_ERR_UNSUPPORTED;
  if (s->max_blocks < 1 || (int64_t)s->max_blocks * s->block_size >= (int64_t(1) << 31))
    return NSV_ERR_SHAPE;
  if (s->num_blocks < 1 || s->num_blocks > (int64_t(1) << 31) - 2) return NSV_ERR_SHAPE;
  return NSV_OK;
}

// Rows of the [block][kv_head][token] pool seen as one 2-D tensor of
// head_dim-wide rows, the tensor consumer's TMA view; its row coordinate is
// a signed 32-bit value.
bool tensor_rows_fit(const nsv_shape* s) {
  return (s->num_blocks + 1) * (int64_t)s->num_kv_heads * kBlock < (int64_t(1) << 31);
}

// The TMEM form's sizes: its group, blocks per stage, ring and CTAs per SM.
// One CTA per SM: its eight softmax warps, MMA warp and producer take most
// of the register file, and a group of two KV heads at head_dim 128 takes
// all 512 tensor-memory columns.
int plan_tmem(const nsv_shape* s, int vpk, int* hg, int* bps, int* stages, int* cps) {
  const int D = s->head_dim;
  const int rows = s->rows > 0 ? s->rows : 1;
  if (*hg <= 0)
    *hg = tmem_group(s->num_kv_heads, vpk, D);
  else if (!tmem_group_ok(*hg, s->num_kv_heads, vpk, D))
    return NSV_ERR_RANGE;
  if (*bps > 0 && !tmem_blocks_ok(D, *hg, *bps)) return NSV_ERR_RANGE;
  if (*stages > 0 && (*stages < 2 || *stages > 8)) return NSV_ERR_RANGE;
  if (*cps > 1) return NSV_ERR_RANGE;
  const int nvec = *hg * vpk;
  auto fits = [&](int b, int st) {
    return make_layout(2, D, *hg, nvec, st, rows, kFormTmem, 1, b).total <=
           (uint32_t)kSmemPerCta;
  };
  // By default the largest stage (up to 4 blocks) that still leaves a ring
  // of 3, with the deepest ring (up to 6) that fits; else 2 stages.
  const int b_hi = *bps > 0 ? *bps : kTmemMaxBlocks, b_lo = *bps > 0 ? *bps : 1;
  for (int min_st : {3, 2}) {
    for (int b = b_hi; b >= b_lo; --b) {
      if (!tmem_blocks_ok(D, *hg, b)) continue;
      int st = 0;
      if (*stages > 0) {
        st = fits(b, *stages) ? *stages : 0;
      } else {
        for (int k = 2; k <= 6; ++k)
          if (fits(b, k)) st = k;
        if (st < min_st) st = 0;
      }
      if (st) {
        *bps = b;
        *stages = st;
        *cps = 1;
        return NSV_OK;
      }
    }
    if (*stages > 0) break;  // min_st does not apply to a fixed ring
  }
  return NSV_ERR_RANGE;
}

int make_plan(const nsv_shape* s, int num_sms, int hg, int stages, int cps, int grid, int qw,
              int consumer, int bps, nsv_plan* p) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (!p) return NSV_ERR_NULLPTR;
  if (num_sms <= 0) {
    DeviceState* d = nullptr;
    if ((rc = device_state(&d)) != NSV_OK) return rc;
    num_sms = d->num_sms;
  }
  const int elem = elem_bytes(s->dtype);
  const int G = s->num_heads / s->num_kv_heads;
  const int vpk = G * query_len(s);                // query vectors per KV head
  const bool tensor_ok = s->dtype == NSV_BF16 && vpk >= 2 && vpk <= kMaxVectorsPerKvHead &&
                         tensor_rows_fit(s);
  if (consumer == NSV_CONSUMER_AUTO) {
    // The tensor cores pay off once several query vectors share a K/V tile,
    // where the CUDA cores repeat the work per vector.  Up to 8 vectors the
    // tokens are the MMA rows (one warp per KV head); 9 to 16, the vectors
    // (16 per warp), which measured faster than 8 per warp with tokens as
    // rows; beyond, tcgen05 into tensor memory when the KV heads split into
    // its groups (at head_dim 128, 17-64 vectors: 1.0-1.9x the
    // vectors-as-rows form's speed), except at head_dim 64 up to 32 vectors,
    // where a stage's fixed cost weighs on its half-size blocks and the
    // vectors as the rows measured faster (32 vectors on 8 KV heads: 400
    // against 498 us).
    consumer = !(tensor_ok && qw <= 0) ? kConsumerCuda
               : vpk <= 8              ? kConsumerTensor
               : (vpk > kMmaRows && tmem_group(s->num_kv_heads, vpk, s->head_dim) >= 2 &&
                  !(s->head_dim == 64 && vpk <= 32))
                   ? kConsumerTensorTmem
                   : kConsumerTensorVectorRows;
  } else if (consumer == kConsumerTensor || consumer == kConsumerTensorVectorRows ||
             consumer == kConsumerTensorTmem) {
    if (!tensor_ok || qw > 1) return NSV_ERR_RANGE;
  } else if (consumer != kConsumerCuda) {
    return NSV_ERR_RANGE;
  }
  const bool tensor = consumer != kConsumerCuda;
  if (tensor) {
    qw = 1;  // unused: a warp runs 8 or 16 of its KV head's vectors on the MMAs
  } else if (qw <= 0) {
    // Two vectors per warp when they pair up: one widening of each tile
    // serves both, and their registers still let 16 warps run per SM (two
    // CTAs), which measured faster than four vectors on 8 warps.
    qw = vpk % 2 == 0 ? 2 : 1;
    if (vpk / qw > max_consumer_warps(qw)) return NSV_ERR_SHAPE;
  } else if ((qw != 1 && qw != 2 && qw != 4) || vpk % qw != 0 ||
             vpk / qw > max_consumer_warps(qw)) {
    return NSV_ERR_RANGE;
  }
  // consumer warps per KV head: on the tensor cores one per 8 vectors
  // (tokens as the MMA rows) or one per 16 (vectors as the rows)
  const int wpk = consumer == kConsumerTensor            ? (vpk + 7) / 8
                  : consumer == kConsumerTensorVectorRows ? (vpk + kMmaRows - 1) / kMmaRows
                                                          : vpk / qw;
  const int max_warps = tensor ? kMaxConsumerWarpsMulti : max_consumer_warps(qw);
  const int tile = kBlock * s->head_dim * elem;
  const bool tmem_form = consumer == kConsumerTensorTmem;
  if (!tmem_form && bps > 1) return NSV_ERR_RANGE;  // one block per stage
  if (tmem_form) {
    // one 128-row MMA group per CTA (4, 2 or 1 KV heads, each with 128 /
    // group rows for its vectors), stages of up to 4 blocks
    if ((rc = plan_tmem(s, vpk, &hg, &bps, &stages, &cps)) != NSV_OK) return rc;
  } else if (hg <= 0) {
    // Among 1 and the KV-head groups whose K+V stage stays within 64 KiB and
    // whose query vectors fill at most 8 consumer warps, the one whose plan keeps
    // the most consumer warps resident per SM, counted up to 16, the larger
    // group on a tie (big bulk copies, few CTAs).  A consumer warp's chain of
    // dependent steps per tile, not the bytes in flight, bounds one CTA's
    // rate once its stages are small: a deeper ring leaves the read time
    // unchanged, more warps per SM shorten it until HBM is the bound, which
    // 12 to 16 reach.
    int best_warps = 0;
    nsv_plan best{};
    int best_rc = NSV_ERR_RANGE;
    for (int c : {8, 4, 2, 1}) {
      if (c > 1 && (s->num_kv_heads % c != 0 || c * wpk > 8 || 2 * c * tile > 64 * 1024))
        continue;
      nsv_plan cand;
      const int rc_c = make_plan(s, num_sms, c, stages, cps, grid, qw, consumer, 1, &cand);
      if (rc_c != NSV_OK) {
        if (best_warps == 0) best_rc = rc_c;
        continue;
      }
      const int warps = std::min(cand.ctas_per_sm * c * wpk, kEnoughWarpsPerSm);
      if (warps > best_warps) {
        best_warps = warps;
        best = cand;
      }
    }
    if (best_warps == 0) return best_rc;
    *p = best;
    return NSV_OK;
  } else if (s->num_kv_heads % hg != 0 || hg * wpk > max_warps) {
    return NSV_ERR_RANGE;
  }
  if (!tmem_form) bps = 1;
  const int nvec = hg * vpk;
  const int rows_for_layout = s->rows > 0 ? s->rows : 1;
  const bool auto_stages = stages <= 0 && !tmem_form;
  if (auto_stages) stages = 3;
  if (stages < 2 || stages > 8) return NSV_ERR_RANGE;
  const int form = form_of(consumer);
  SmemLayout L =
      make_layout(elem, s->head_dim, hg, nvec, stages, rows_for_layout, form, qw, bps);
  while (auto_stages && L.total > (uint32_t)kSmemPerCta && stages > 2) {
    --stages;
    L = make_layout(elem, s->head_dim, hg, nvec, stages, rows_for_layout, form, qw, bps);
  }
  if (L.total > (uint32_t)kSmemPerCta) return NSV_ERR_RANGE;
  const int threads =
      (tmem_form ? kTmemWarps + 2 : cta_warps(form_of(consumer), s->head_dim, hg * wpk)) * 32;
  int fit = kSmemPerSm / (int)(L.total + kSmemReserved);
  // CTAs one SM holds by threads and by registers (each kernel variant's
  // register count is fixed at compile time)
  const int regs = decode_regs(consumer, qw, s->head_dim);
  int fit_threads = std::min(kThreadsPerSm / threads, ctas_by_registers(threads, regs));
  // The TMEM form's CTAs also share the SM's 512 tensor-memory columns.
  // (The device's occupancy calculator answers one CTA per SM for a kernel
  // that allocates tensor memory, however few columns it takes; two CTAs of
  // 256 columns do run side by side: an earlier one-block-per-stage version
  // of the form read 64 vectors per KV head in 929 us with two per SM
  // against 1540 us with one, on GB300.)
  if (tmem_form) fit_threads = std::min(fit_threads, 512 / tmem_cols(s->head_dim, hg, bps));
  if (fit_threads < 1) return NSV_ERR_RANGE;  // one CTA would not fit the register file
  if (!tensor && auto_stages && cps <= 0 && stages == 3 && hg == s->num_kv_heads &&
      2 * hg * tile <= 16 * 1024) {
    // CUDA-core consumer whose CTA streams every KV head (one or two of
    // them) in stages of at most 16 KiB: where shared memory alone holds the
    // CTAs per SM below what registers allow and their consumer warps stay
    // under 16, a 2-stage ring that fits more CTAs reads faster (one KV head
    // of one query head: 7 CTAs of 3 stages 222 us, 8 of 2 stages 206 us on
    // GB300).  The tensor-core forms lost 4-14 % with 2 stages, so they keep
    // 3, and so do shapes with more KV heads, whose larger groups were not
    // measured against it.
    const int warps_cta = threads / 32 - 1;
    const int now = std::min({fit, fit_threads, kMaxCtasPerSm});
    const SmemLayout L2 =
        make_layout(elem, s->head_dim, hg, nvec, 2, rows_for_layout, form, qw, 1);
    const int fit2 = kSmemPerSm / (int)(L2.total + kSmemReserved);
    if (now * warps_cta < kEnoughWarpsPerSm &&
        std::min({fit2, fit_threads, kMaxCtasPerSm}) > now) {
      stages = 2;
      L = L2;
      fit = fit2;
    }
  }
  if (tensor && !tmem_form && auto_stages && cps <= 0 && std::min(fit, fit_threads) < 2) {
    // One CTA per SM either way: spend the rest of its shared memory on a
    // deeper ring (up to 6 stages), which keeps more bytes in flight for
    // the consumers that would otherwise wait on HBM latency.
    while (stages < 6) {
      const SmemLayout L2 =
          make_layout(elem, s->head_dim, hg, nvec, stages + 1, rows_for_layout, form, qw, 1);
      if (L2.total > (uint32_t)kSmemPerCta) break;
      ++stages;
      L = L2;
    }
    fit = kSmemPerSm / (int)(L.total + kSmemReserved);
  }
  if (cps <= 0) {
    // As many as fit: up to 8, or 2 for the TMEM form (measured no further)
    cps = std::min(fit, tmem_form ? 2 : kMaxCtasPerSm);
    if (cps > fit_threads) cps = fit_threads;
    if (cps < 1) cps = 1;
  } else if (cps > kMaxCtasPerSm || cps > fit || cps > fit_threads) {
    return NSV_ERR_RANGE;
  }
  if (grid <= 0) {
    grid = num_sms * cps;
  } else if (grid > (1 << 16)) {
    return NSV_ERR_RANGE;
  }
  const WsLayout W =
      make_ws_layout(rows_for_layout, s->num_kv_heads / hg, grid, nvec, s->head_dim);
  memset(p, 0, sizeof(*p));
  p->kv_heads_per_cta = hg;
  p->stages = stages;
  p->ctas_per_sm = cps;
  p->grid = grid;
  p->threads = threads;
  p->smem_bytes = (int)L.total;
  p->num_sms = num_sms;
  p->vectors_per_warp = qw;
  p->consumer = consumer;
  p->blocks_per_stage = bps;
  p->workspace_bytes = (int64_t)W.total;
  return NSV_OK;
}

// A caller's plan must be exactly what the planner makes from its choices.
int check_plan(const nsv_shape* s, const nsv_plan* given, nsv_plan* use) {
  int rc = make_plan(s, given->num_sms, given->kv_heads_per_cta, given->stages,
                     given->ctas_per_sm, given->grid, given->vectors_per_warp,
                     given->consumer, given->blocks_per_stage, use);
  if (rc) return rc;
  if (memcmp(use, given, sizeof(nsv_plan)) != 0) return NSV_ERR_RANGE;
  return NSV_OK;
}

// Checks the append's arguments and fills its launch parameters (no launch).
int kv_write_prepare(const nsv_shape* s, const void* k_new, const void* v_new,
                     const int64_t* write_slots, void* k_pool, void* v_pool, KvWriteParams* p) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (s->rows == 0) return NSV_OK;  // an empty batch: nothing to write
  if (!k_new || !v_new || !write_slots || !k_pool || !v_pool) return NSV_ERR_NULLPTR;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(write_slots) & 7u))
    return NSV_ERR_ALIGN;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d)) != NSV_OK) return rc;
  p->k_new = k_new;
  p->v_new = v_new;
  p->write_slots = write_slots;
  p->k_pool = k_pool;
  p->v_pool = v_pool;
  p->status = d->status;
  p->pool_slots = (s->num_blocks + 1) * (long long)s->block_size;
  p->rows = s->rows * query_len(s);  // every new token of every row
  p->kv_heads = s->num_kv_heads;
  p->vec_per_head = s->head_dim * elem_bytes(s->dtype) / 16;
  p->block_size = s->block_size;
  p->zero_words = nullptr;
  p->zero_count = 0;
  return NSV_OK;
}

// The read through either addressing form: block_tables (slots null) or a
// slot table `slots` with `slot_cols` readable columns per row and row
// stride `slot_stride` (block_tables null).  With `append` (the fused step)
// the append is launched right before the read, after every check has
// passed, and zeroes the read's arrival counters itself.
int decode_impl(const nsv_shape* s, const nsv_plan* plan_in, const void* q, const void* k_pool,
                const void* v_pool, const int32_t* block_tables, const int64_t* slots,
                int64_t slot_cols, int64_t slot_stride, const int32_t* context_lens,
                float scale, void* out, void* ws, size_t ws_bytes, bool library_ws,
                cudaStream_t stream, KvWriteParams* append = nullptr) {
  int rc = check_shape(s);
  if (rc) return rc;
  if (s->rows == 0) return NSV_OK;  // an empty batch: nothing to read
  if (!q || !k_pool || !v_pool || !(block_tables || slots) || !context_lens || !out)
    return NSV_ERR_NULLPTR;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(slots) & 7u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return NSV_ERR_ALIGN;
  if (slots && (slot_cols < 1 || slot_cols > (int64_t)s->max_blocks * s->block_size ||
                slot_stride < slot_cols))
    return NSV_ERR_SHAPE;
  nsv_plan plan;
  if (plan_in) {
    if ((rc = check_plan(s, plan_in, &plan)) != NSV_OK) return rc;
  }
  DeviceState* d = nullptr;
  if ((rc = device_state(&d)) != NSV_OK) return rc;
  if (!plan_in) {
    if ((rc = make_plan(s, d->num_sms, 0, 0, 0, 0, 0, 0, 0, &plan)) != NSV_OK) return rc;
  }
  if (s->rows == 0) return NSV_OK;
  if (library_ws) {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((size_t)plan.workspace_bytes > d->ws_bytes) {
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return cuda_fail();
      if (cs != cudaStreamCaptureStatusNone) return NSV_ERR_CAPTURE;
      if (d->ws) {
        if (cudaFree(d->ws) != cudaSuccess) return cuda_fail();
        d->ws = nullptr;
        d->ws_bytes = 0;
      }
      if (cudaMalloc(&d->ws, (size_t)plan.workspace_bytes) != cudaSuccess) return cuda_fail();
      d->ws_bytes = (size_t)plan.workspace_bytes;
    }
    ws = d->ws;
    ws_bytes = d->ws_bytes;
  }
  if (!ws || ws_bytes < (size_t)plan.workspace_bytes ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return NSV_ERR_WORKSPACE;
  const int nvec = plan.kv_heads_per_cta * (s->num_heads / s->num_kv_heads) * query_len(s);
  const WsLayout W = make_ws_layout(s->rows, s->num_kv_heads / plan.kv_heads_per_cta, plan.grid,
                                    nvec, s->head_dim);
  char* wsb = static_cast<char*>(ws);
  DecodeParams p;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_tables = block_tables;
  p.slots = slots;
  p.slot_stride = slots ? slot_stride : 0;
  p.slot_cols = slots ? (int)slot_cols : 0;
  p.context_lens = context_lens;
  p.out = out;
  p.ws_cnt = reinterpret_cast<int32_t*>(wsb);
  p.ws_ml = reinterpret_cast<float2*>(wsb + W.off_ml);
  p.ws_acc = reinterpret_cast<float*>(wsb + W.off_acc);
  p.status = d->status;
  p.walked = d->walked;
  p.pool_blocks = s->num_blocks + 1;
  p.rows = s->rows;
  p.heads = s->num_heads;
  p.kv_heads = s->num_kv_heads;
  p.max_blocks = s->max_blocks;
  p.heads_per_cta = plan.kv_heads_per_cta;
  p.group = s->num_heads / s->num_kv_heads;
  p.query_len = query_len(s);
  p.stages = plan.stages;
  p.blocks_per_stage = plan.blocks_per_stage;
  p.qscale = scale * 1.4426950408889634f;  // log2(e): the kernels use exp2
  memset(&p.tmap_k, 0, sizeof(p.tmap_k));
  memset(&p.tmap_v, 0, sizeof(p.tmap_v));
  if (plan.consumer != kConsumerCuda) {
    // The pools as [(num_blocks+1)*kv_heads*16 rows][head_dim] bf16; a box is
    // 64 dims (128 bytes, the swizzle span) by the head group's 16-token tiles.
    const cuuint64_t rows = (cuuint64_t)(s->num_blocks + 1) * s->num_kv_heads * kBlock;
    const cuuint64_t dims[2] = {(cuuint64_t)s->head_dim, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)s->head_dim * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)(plan.kv_heads_per_cta * kBlock)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (plan.consumer == kConsumerTensorTmem) {
      // K for the TMEM form: the rows seen as [64 dims][8 rows][64-dim
      // halves][groups of 8 rows], so that one box lands a block's tiles as
      // [group][half][8 rows][128 bytes], the layout whose groups the scores
      // MMA steps through at one stride across all blocks of a stage.
      const cuuint64_t dims4[4] = {64u, 8u, (cuuint64_t)(s->head_dim / 64), rows / 8};
      const cuuint64_t strides4[3] = {(cuuint64_t)s->head_dim * 2, 128u,
                                      (cuuint64_t)s->head_dim * 2 * 8};
      const cuuint32_t box4[4] = {64u, 8u, (cuuint32_t)(s->head_dim / 64),
                                  (cuuint32_t)(plan.kv_heads_per_cta * kBlock / 8)};
      const cuuint32_t estr4[4] = {1u, 1u, 1u, 1u};
      if (g_encode(&p.tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(k_pool),
                   dims4, strides4, box4, estr4, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return NSV_ERR_CUDA;
    } else if (g_encode(&p.tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(k_pool),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      return NSV_ERR_CUDA;
    }
    if (plan.consumer == kConsumerTensorTmem) {
      // V for the TMEM form: the same rows seen as [64 dims][rows][64-dim
      // halves], so that one box (64 dims x the group's 16-token tiles x
      // both halves) lands a block as [half][head][token][128 bytes].
      const cuuint64_t dims3[3] = {64u, rows, (cuuint64_t)(s->head_dim / 64)};
      const cuuint64_t strides3[2] = {(cuuint64_t)s->head_dim * 2, 128u};
      const cuuint32_t box3[3] = {64u, (cuuint32_t)(plan.kv_heads_per_cta * kBlock),
                                  (cuuint32_t)(s->head_dim / 64)};
      if (g_encode(&p.tmap_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v_pool),
                   dims3, strides3, box3, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return NSV_ERR_CUDA;
    } else if (g_encode(&p.tmap_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v_pool),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      return NSV_ERR_CUDA;
    }
  }
  // The arrival counters of cut rows start every call at zero: zeroed by
  // the step's append launch, or, for the read alone, by the same kernel
  // with no rows to append.
  KvWriteParams zero;
  if (!append) {
    memset(&zero, 0, sizeof zero);
    append = &zero;
  }
  append->zero_words = reinterpret_cast<int32_t*>(wsb);
  append->zero_count = (int)(W.cnt_bytes / 4);
  if (launch_kv_write(*append, stream) != cudaSuccess) return cuda_fail();
  // The read may start while that kernel runs (programmatic dependent
  // launch): it reads only the step's inputs until the kernel has completed.
  if (launch_decode(p, s->dtype, s->head_dim, plan.vectors_per_warp, plan.consumer, plan.grid,
                    plan.threads, plan.smem_bytes, stream, true) != cudaSuccess)
    return cuda_fail();
  return NSV_OK;
}

}  // namespace
}  // namespace nsv

using namespace nsv;

extern "C" {

NSV_API int nsv_abi_version(void) { return NSV_ABI_VERSION; }

NSV_API const char* nsv_strerror(int code) {
  switch (code) {
    case NSV_OK: return "success";
    case NSV_ERR_NULLPTR: return "a required pointer is NULL";
    case NSV_ERR_DTYPE: return "dtype must be NSV_F32 or NSV_BF16";
    case NSV_ERR_SHAPE: return "a size is outside its documented range";
    case NSV_ERR_ALIGN: return "a data pointer is not 16-byte aligned";
    case NSV_ERR_RANGE: return "a plan field does not fit the shape";
    case NSV_ERR_CAPTURE: return "the library workspace would have to grow during stream capture";
    case NSV_ERR_CUDA: return "a CUDA runtime call failed";
    case NSV_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than the plan needs";
    case NSV_ERR_UNSUPPORTED: return "head_dim must be 64 or 128 and block_size 16";
    default: return "unknown nsv error code";
  }
}

NSV_API int nsv_plan_split(const nsv_shape* shape, int num_sms, nsv_plan* plan) {
  return make_plan(shape, num_sms, 0, 0, 0, 0, 0, 0, 0, plan);
}

NSV_API int nsv_plan_custom(const nsv_shape* shape, int num_sms, int kv_heads_per_cta,
                            int stages, int ctas_per_sm, int grid, int vectors_per_warp,
                            int consumer, int blocks_per_stage, nsv_plan* plan) {
  return make_plan(shape, num_sms, kv_heads_per_cta, stages, ctas_per_sm, grid,
                   vectors_per_warp, consumer, blocks_per_stage, plan);
}

NSV_API int nsv_plan_resident_ctas(const nsv_shape* shape, const nsv_plan* plan,
                                   int* ctas_per_sm) {
  if (!ctas_per_sm) return NSV_ERR_NULLPTR;
  if (!plan) return NSV_ERR_NULLPTR;
  nsv_plan use;
  int rc = check_plan(shape, plan, &use);
  if (rc) return rc;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d)) != NSV_OK) return rc;
  int n = 0;
  if (decode_occupancy(shape->dtype, shape->head_dim, use.vectors_per_warp, use.consumer,
                       use.threads, use.smem_bytes, &n) != cudaSuccess)
    return cuda_fail();
  *ctas_per_sm = n;
  return NSV_OK;
}

NSV_API int nsv_kv_write(const nsv_shape* s, const void* k_new, const void* v_new,
                         const int64_t* write_slots, void* k_pool, void* v_pool,
                         cudaStream_t stream) {
  KvWriteParams p;
  int rc = kv_write_prepare(s, k_new, v_new, write_slots, k_pool, v_pool, &p);
  if (rc) return rc;
  if (s->rows == 0) return NSV_OK;  // an empty batch: nothing to write
  if (launch_kv_write(p, stream) != cudaSuccess) return cuda_fail();
  return NSV_OK;
}

NSV_API int nsv_paged_decode(const nsv_shape* shape, const void* q, const void* k_pool,
                             const void* v_pool, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, void* out,
                             cudaStream_t stream) {
  return decode_impl(shape, nullptr, q, k_pool, v_pool, block_tables, nullptr, 0, 0,
                     context_lens, scale, out, nullptr, 0, true, stream);
}

NSV_API int nsv_paged_decode_ws(const nsv_shape* shape, const nsv_plan* plan, const void* q,
                                const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, void* out, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  return decode_impl(shape, plan, q, k_pool, v_pool, block_tables, nullptr, 0, 0, context_lens,
                     scale, out, workspace, workspace_bytes, false, stream);
}

NSV_API int nsv_decode_step(const nsv_shape* shape, const nsv_plan* plan, const void* q,
                            const void* k_new, const void* v_new, const int64_t* write_slots,
                            void* k_pool, void* v_pool, const int32_t* block_tables,
                            const int32_t* context_lens, float scale, void* out,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  KvWriteParams append;
  int rc = kv_write_prepare(shape, k_new, v_new, write_slots, k_pool, v_pool, &append);
  if (rc) return rc;
  const bool lib_ws = workspace == nullptr && workspace_bytes == 0;
  // Checks both halves before launching either: the append and the read
  // are launched back to back by decode_impl, or neither is.
  return decode_impl(shape, plan, q, k_pool, v_pool, block_tables, nullptr, 0, 0, context_lens,
                     scale, out, workspace, workspace_bytes, lib_ws, stream, &append);
}

NSV_API int nsv_paged_decode_slots(const nsv_shape* shape, const nsv_plan* plan, const void* q,
                                   const void* k_pool, const void* v_pool,
                                   const int64_t* slot_table, int64_t slot_cols,
                                   int64_t slot_row_stride, const int32_t* context_lens,
                                   float scale, void* out, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream) {
  if (!slot_table) return NSV_ERR_NULLPTR;
  const bool lib_ws = workspace == nullptr && workspace_bytes == 0;
  return decode_impl(shape, plan, q, k_pool, v_pool, nullptr, slot_table, slot_cols,
                     slot_row_stride, context_lens, scale, out, workspace, workspace_bytes,
                     lib_ws, stream);
}

NSV_API int nsv_selftest_bounded_wait(uint64_t limit_ns, int* gave_up, uint64_t* waited_ns,
                                      cudaStream_t stream) {
  if (!gave_up || !waited_ns) return NSV_ERR_NULLPTR;
  if (limit_ns < 1000 || limit_ns > 2000000000ull) return NSV_ERR_RANGE;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  unsigned long long* res = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&res), g_probe) != cudaSuccess)
    return cuda_fail();
  if (cudaMemsetAsync(res, 0xff, sizeof(g_probe), stream) != cudaSuccess) return cuda_fail();
  if (launch_wait_probe(limit_ns, res, d->status, stream) != cudaSuccess) return cuda_fail();
  unsigned long long h[2] = {0, 0};
  if (cudaMemcpyAsync(h, res, sizeof h, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return cuda_fail();
  if (cudaStreamSynchronize(stream) != cudaSuccess) return cuda_fail();
  *gave_up = h[0] == 1ull ? 1 : 0;
  *waited_ns = (uint64_t)h[1];
  return NSV_OK;
}

NSV_API int nsv_status_async(uint32_t* dst, int clear, cudaStream_t stream) {
  if (!dst) return NSV_ERR_NULLPTR;
  if (reinterpret_cast<uintptr_t>(dst) & 3u) return NSV_ERR_ALIGN;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (cudaMemcpyAsync(dst, d->status, sizeof(uint32_t), cudaMemcpyDefault, stream) !=
      cudaSuccess)
    return cuda_fail();
  if (clear && cudaMemsetAsync(d->status, 0, sizeof(uint32_t), stream) != cudaSuccess)
    return cuda_fail();
  return NSV_OK;
}

NSV_API int nsv_device_status(uint32_t* status, uint64_t* blocks_walked, int clear) {
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail();
  uint32_t st = 0;
  unsigned long long w = 0;
  if (cudaMemcpy(&st, d->status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail();
  if (cudaMemcpy(&w, d->walked, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
    return cuda_fail();
  if (status) *status = st;
  if (blocks_walked) *blocks_walked = (uint64_t)w;
  if (clear) {
    if (cudaMemset(d->status, 0, sizeof st) != cudaSuccess) return cuda_fail();
    if (cudaMemset(d->walked, 0, sizeof w) != cudaSuccess) return cuda_fail();
    if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail();
  }
  return NSV_OK;
}

}  // extern "C"
