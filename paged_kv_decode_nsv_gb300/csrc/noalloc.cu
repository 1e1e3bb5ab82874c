// nsv_paged_decode_noalloc: the decode read for callers that must not
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits or unwelcome.
// Examples are an engine that owns every byte of the device through its own
// pre-sized arena and treats any outside allocation as a budget violation;
// plugin hooks that are handed only pre-bound buffers at enqueue time; and
// callers that cannot tolerate the device-wide synchronisation a
// cudaMalloc/cudaFree pair can cause in the middle of a serving loop.  The
// split (flash-decoding) path needs scratch for its partial softmax states;
// this entry point takes that scratch from a fixed buffer compiled into the
// library instead of from the caller or from cudaMalloc.
//
// The buffer is a file-scope __device__ array, so every GPU that loads the
// library holds NSV_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use the array's name as a device pointer; its device
// address is looked up with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and cached, and looked up again
// if a different CUDA context has become current on the device since.
//
// All calls on one device share the buffer.  Its first part holds the read's
// arrival counters (one per row and KV-head group), which must be zero when
// the kernel starts: nsv_paged_decode_ws clears them on the caller's
// stream before every launch, with a small kernel of its own (no
// allocation).  Everything
// else in it (the partial softmax states of rows cut between CTAs) each call
// writes before it reads it.  So a caller never clears the buffer, whatever
// an earlier call left there; but calls whose kernels overlap on the GPU
// (different streams, no ordering between them) race on it.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "nsv_common.cuh"

namespace {

constexpr size_t kScratchBytes = NSV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

void* g_scratch_addr[kMaxDevices];
void* g_scratch_ctx[kMaxDevices];  // the context each address belongs to
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return NSV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return NSV_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] != nullptr) {
    void* now = nsv::current_cuda_context();
    if (now != nullptr && now != g_scratch_ctx[dev]) g_scratch_addr[dev] = nullptr;
  }
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return NSV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = nsv::current_cuda_context();
  }
  *out = g_scratch_addr[dev];
  return NSV_OK;
}

}  // namespace

extern "C" NSV_API int nsv_paged_decode_noalloc(const nsv_shape* shape, const void* q,
                                                const void* k_pool, const void* v_pool,
                                                const int32_t* block_tables,
                                                const int32_t* context_lens, float scale,
                                                void* out, cudaStream_t stream) {
  nsv_plan plan;
  int rc = nsv_plan_split(shape, 0, &plan);
  if (rc != NSV_OK) return rc;
  if (shape->rows == 0) return NSV_OK;  // an empty batch: nothing to read
  if (plan.workspace_bytes > (int64_t)kScratchBytes) return NSV_ERR_WORKSPACE;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (plan.workspace_bytes > 0) {
    if ((rc = scratch_address(&scratch)) != NSV_OK) return rc;
    scratch_bytes = kScratchBytes;
  }
  return nsv_paged_decode_ws(shape, &plan, q, k_pool, v_pool, block_tables, context_lens, scale,
                             out, scratch, scratch_bytes, stream);
}
