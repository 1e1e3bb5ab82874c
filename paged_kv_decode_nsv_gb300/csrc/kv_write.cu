// KV append for sm_103a: every row's new key and value land at its write
// slot (nanoserve Day 55, "the capture list moved to startup, and the dummy
// batch was all padding", "Why it matters": the write is one indexed write
// over the padded batch, and a padded row's slot is the sink slot).
//
// One thread moves one 16-byte vector of K and the same vector of V.  The
// new rows are read contiguously; each (row, KV head) lands as one
// contiguous head_dim run inside its (block, head) tile of the
// [block][kv_head][token][dim] pool, so every write is a whole number of
// 32-byte sectors.  A slot outside the pool array is skipped and flagged;
// nothing here can write out of bounds.  When the append and the read form
// one step, the same launch also zeroes the read's arrival counters, which
// saves the step a separate memset.

#include <cuda_runtime.h>
#include <stdint.h>

#include "nsv_common.cuh"

namespace nsv {
namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(const KvWriteParams p) {
  // The step's read may be scheduled now: it waits for this grid's writes
  // itself (a no-op when nothing depends on this launch).
  asm volatile("griddepcontrol.launch_dependents;");
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < p.zero_count) p.zero_words[i] = 0;
  const long long per_row = (long long)p.kv_heads * p.vec_per_head;
  if (i >= (long long)p.rows * per_row) return;
  const int r = (int)(i / per_row);
  const int rem = (int)(i - (long long)r * per_row);
  const int g = rem / p.vec_per_head;
  const int v = rem - g * p.vec_per_head;
  const long long slot = p.write_slots[r];
  if (slot < 0 || slot >= p.pool_slots) {
    if (rem == 0) atomicOr(p.status, (uint32_t)NSV_DEV_BAD_SLOT);
    return;
  }
  const long long blk = slot / p.block_size, off = slot - blk * p.block_size;
  // vectors: a (block, head) tile is block_size * vec_per_head vectors
  const size_t dst = ((size_t)(blk * p.kv_heads + g) * p.block_size + off) * p.vec_per_head + v;
  const uint4 kv = static_cast<const uint4*>(p.k_new)[i];
  const uint4 vv = static_cast<const uint4*>(p.v_new)[i];
  static_cast<uint4*>(p.k_pool)[dst] = kv;
  static_cast<uint4*>(p.v_pool)[dst] = vv;
}

}  // namespace

cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t stream) {
  long long n = (long long)p.rows * p.kv_heads * p.vec_per_head;
  if (p.zero_count > n) n = p.zero_count;
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const long long grid = (n + threads - 1) / threads;
  kv_write_kernel<<<(unsigned)grid, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace nsv
