// Internal declarations shared by the library's translation units: kernel
// parameter blocks, the shared-memory layout of the decode kernel (computed
// identically on host and device), and the launchers each .cu file exports.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nsv.h"

namespace nsv {

// The kernels are built for this block size (the pages' 16-token blocks).
constexpr int kBlock = 16;
// Largest number of consumer warps one decode CTA runs: 16 when each warp
// serves one or two query vectors, 8 when it serves 4 (their registers).
constexpr int kMaxConsumerWarps = 16;
constexpr int kMaxConsumerWarpsMulti = 8;
__host__ __device__ constexpr int max_consumer_warps(int qw) {
  return qw <= 2 ? kMaxConsumerWarps : kMaxConsumerWarpsMulti;
}
// Largest number of query vectors (query heads x query tokens) that share
// one KV head: 64 on the tensor cores (4 warps of 16 MMA rows), 32 on the
// CUDA cores (16 warps of 2).
constexpr int kMaxVectorsPerKvHead = 64;
// Rows of the tensor-core MMA (m16n8k16): 16 query vectors per warp when the
// vectors are the rows.
constexpr int kMmaRows = 16;
enum : int {
  kConsumerCuda = 1,
  kConsumerTensor = 2,
  kConsumerTensorVectorRows = 3,
  kConsumerTensorTmem = 4
};
constexpr int kMaxThreads = (kMaxConsumerWarps + 1) * 32;
constexpr int kMaxThreadsMulti = (kMaxConsumerWarpsMulti + 1) * 32;

// Registers per thread of each decode-kernel variant, fixed at compile time
// (__maxnreg__) so that the planner can size the grid to the CTAs that are
// really resident: CUDA-core consumer with 1 or 2 vectors per warp (96: a
// 17-warp CTA fits, 5 warps of it per sub-partition, and two 9-warp CTAs
// do), the two mma.sync forms at head_dim 64 (what they use without
// spilling: 112 with tokens as rows, 128 with vectors as rows, which lets
// 4 warps share a sub-partition instead of 3), and every other variant
// (4 vectors per warp, the mma.sync forms at head_dim 128, the TMEM form).
constexpr int kRegsNarrow = 96;
constexpr int kRegsWide = 168;
constexpr int kRegsTmem = 168;
constexpr int kRegsTokenRows64 = 112;
constexpr int kRegsVectorRows64 = 128;
__host__ __device__ constexpr int decode_regs(int consumer, int qw, int head_dim) {
  return consumer == kConsumerTensorTmem                      ? kRegsTmem
         : (consumer == kConsumerCuda && qw <= 2)             ? kRegsNarrow
         : (consumer == kConsumerTensor && head_dim == 64)    ? kRegsTokenRows64
         : (consumer == kConsumerTensorVectorRows && head_dim == 64) ? kRegsVectorRows64
                                                              : kRegsWide;
}
// CTAs of `threads` threads at `regs` registers each that one SM's
// registers hold: 4 sub-partitions of 16 K registers, each holding whole
// warps (allocated in units of 256 registers).
__host__ __device__ constexpr int ctas_by_registers(int threads, int regs) {
  return 4 * (16384 / (((regs * 32 + 255) / 256) * 256)) / ((threads + 31) / 32);
}
// Largest batch the decode kernel's per-CTA row tables hold.
constexpr int kMaxRows = 8192;

// Stage flags written by the producer warp for the consumers.  The low 8
// bits of a stage's flag word carry the row's positions from the block on
// (clipped at 255) and bits 16 and up the first KV head of the head group.
enum : int {
  kFirst = 1 << 8,   // first block of a segment: reset the softmax state
  kLast = 1 << 9,    // last block of a segment: write out or the partial
  kFinal = 1 << 10,  // the segment is the whole row: write `out`
  kData = 1 << 11,   // the stage holds a K and a V tile
  kHasQ = 1 << 12,   // the stage holds the group's query vectors
  kEnd = 1 << 13,    // no more work: consumers exit
  kSlot1 = 1 << 14,  // a partial segment that is not the CTA's first one
  kGathered = 1 << 15,  // the K/V tiles were gathered token by token by the
                        // producer warp (slot-table addressing)
};

// Workspace of one decode read (all offsets 256-byte aligned):
//   cnt     int32 [rows][head groups]  pieces of a cut row that have
//           finished; zeroed on the stream before every launch
//   ml      float2 [grid][2][nvec]  (running max, denominator) of partials
//   acc     float [grid][2][nvec][head_dim]
// where nvec = query vectors per CTA.  Each CTA has at most two partial
// segments: the row its range starts inside of and the row it ends inside of.
struct WsLayout {
  uint64_t cnt_bytes, off_ml, off_acc, total;
};

__host__ __device__ inline WsLayout make_ws_layout(int rows, int head_groups, int grid,
                                                   int nvec, int head_dim) {
  WsLayout W;
  const uint64_t slots = (uint64_t)grid * 2 * nvec;
  W.cnt_bytes = (uint64_t)rows * head_groups * 4;
  W.off_ml = (W.cnt_bytes + 255) / 256 * 256;
  W.off_acc = W.off_ml + (slots * 8 + 255) / 256 * 256;
  W.total = W.off_acc + slots * head_dim * 4;
  return W;
}

struct DecodeParams {
  // K and V pools as 2-D tensors [(num_blocks+1) * kv_heads * block, head_dim]
  // for the tensor-core consumer's swizzled TMA loads (unused otherwise).
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;  // block-table addressing (null in slot mode)
  const int64_t* slots;         // slot-table addressing (null in block mode)
  long long slot_stride;        // row stride of the slot table, in entries
  int slot_cols;                // readable columns of each slot-table row
  const int32_t* context_lens;
  void* out;
  int32_t* ws_cnt;     // workspace arrival counters (zero at launch)
  float2* ws_ml;       // workspace partial (m, l)
  float* ws_acc;       // workspace partial acc
  uint32_t* status;    // device status word
  unsigned long long* walked;  // (row, block) pairs walked
  long long pool_blocks;       // num_blocks + 1
  int rows, heads, kv_heads, max_blocks;
  int heads_per_cta;  // KV heads per CTA
  int group;          // query heads per KV head
  int query_len;      // query tokens per row
  int stages;
  int blocks_per_stage;  // blocks a stage holds (the TMEM form; 1 otherwise)
  float qscale;       // scale * log2(e)
};

struct KvWriteParams {
  const void* k_new;
  const void* v_new;
  const int64_t* write_slots;
  void* k_pool;
  void* v_pool;
  uint32_t* status;
  long long pool_slots;  // (num_blocks + 1) * block_size
  int rows, kv_heads, vec_per_head;  // 16-byte vectors per (row, head)
  int block_size;
  // Words set to zero on the way (the decode read's arrival counters when
  // the append and the read form one step), or none.
  int32_t* zero_words;
  int zero_count;
};

// Shared-memory carve-up of one decode CTA.
struct SmemLayout {
  uint32_t kv_bytes;     // one K (or V) tile set: heads_per_cta * block * D * elem
  uint32_t q_bytes;      // the CTA's query vectors
  uint32_t stage_bytes;  // K + V, rounded to 1024
  uint32_t q_slots;      // ring of query-vector slots (one per segment in flight)
  uint32_t q_slot_bytes; // q_bytes rounded to 128
  uint32_t off_q;        // the q ring
  uint32_t off_meta;     // int4 per stage
  uint32_t off_bars;     // full[stages], empty[stages], qfree[q_slots] mbarriers
  uint32_t off_pbuf;     // per query vector: block-size floats
  uint32_t off_ctx;      // rows ints (validated context lengths)
  uint32_t off_prefix;   // rows + 1 ints (work-item prefix sums)
  uint32_t off_flag;     // abort flag, then the merge flag
  uint32_t total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) {
  return (x + a - 1) / a * a;
}

// Consumer form of a decode-kernel variant (its MMA template argument).
enum : int { kFormCuda = 0, kFormVectorRows = 1, kFormTokenRows = 2, kFormTmem = 3 };
__host__ __device__ constexpr int form_of(int consumer) {
  return consumer == kConsumerTensor            ? kFormTokenRows
         : consumer == kConsumerTensorVectorRows ? kFormVectorRows
         : consumer == kConsumerTensorTmem       ? kFormTmem
                                                 : kFormCuda;
}

// The TMEM form (tcgen05.mma, accumulators in tensor memory).  Its MMA has
// 128 rows: each KV head of the CTA's group takes 128 / group of them (its
// query vectors, the rest zero).  A stage holds up to `blocks` consecutive
// blocks of one segment, and one scores MMA per 16 dims covers all of them
// (N = blocks x group x 16 tokens; each row uses its own head's columns).
// The P.V MMA of a block is one instruction with N = group x head_dim: every
// row's probabilities times every head's V, of which a row keeps its own
// head's columns.  Eight softmax warps, two per TMEM lane quadrant: a pair
// shares its quadrant's 32 rows (a thread owns one row) and splits each
// stage's blocks.
constexpr int kTmemWarps = 8;
constexpr int kTmemRows = 128;
constexpr int kTmemMaxBlocks = 4;  // blocks one stage holds at most
// Whether `group` KV heads of `vpk` query vectors each can share the MMA:
// 1, 2 or 4 heads dividing the KV heads, 128 / group rows for each head's
// vectors, and a P.V product (group x head_dim columns) one MMA wide.
__host__ __device__ constexpr bool tmem_group_ok(int group, int kv_heads, int vpk,
                                                 int head_dim) {
  return (group == 1 || group == 2 || group == 4) && kv_heads % group == 0 &&
         group * vpk <= kTmemRows && group * head_dim <= 256;
}
// Whether a stage of `blocks` blocks fits the form: its scores MMA at most
// 256 columns wide and all its columns within the SM's 512.
__host__ __device__ constexpr bool tmem_blocks_ok(int head_dim, int group, int blocks);
// The default group: the largest of 4, 2 and 1 that fits with stages of at
// least 3 blocks (a stage's fixed cost is what bounds the form; see the
// planner), else the largest that fits.
__host__ __device__ constexpr int tmem_group(int kv_heads, int vpk, int head_dim) {
  return (tmem_group_ok(4, kv_heads, vpk, head_dim) && tmem_blocks_ok(head_dim, 4, 3))   ? 4
         : (tmem_group_ok(2, kv_heads, vpk, head_dim) && tmem_blocks_ok(head_dim, 2, 3)) ? 2
         : tmem_group_ok(4, kv_heads, vpk, head_dim)                                     ? 4
         : tmem_group_ok(2, kv_heads, vpk, head_dim)                                     ? 2
                                                                                         : 1;
}
// Tensor-memory columns the form uses: the output accumulator (group x
// head_dim), two score buffers (blocks x group x 16 each) and the query rows
// (head_dim bf16, two to a column), the scores MMA's A operand.
__host__ __device__ constexpr int tmem_cols_used(int head_dim, int group, int blocks) {
  return group * head_dim + 2 * blocks * group * kBlock + head_dim / 2;
}
// What a CTA allocates: that, rounded up to a power of two (at least 32).
__host__ __device__ constexpr int tmem_cols(int head_dim, int group, int blocks) {
  return tmem_cols_used(head_dim, group, blocks) <= 32    ? 32
         : tmem_cols_used(head_dim, group, blocks) <= 64  ? 64
         : tmem_cols_used(head_dim, group, blocks) <= 128 ? 128
         : tmem_cols_used(head_dim, group, blocks) <= 256 ? 256
                                                          : 512;
}
// Whether a stage of `blocks` blocks fits the form: its scores MMA at most
// 256 columns wide and all its columns within the SM's 512.
__host__ __device__ constexpr bool tmem_blocks_ok(int head_dim, int group, int blocks) {
  return blocks >= 1 && blocks <= kTmemMaxBlocks && blocks * group * kBlock <= 256 &&
         tmem_cols_used(head_dim, group, blocks) <= 512;
}

// Whether a variant keeps its consumer warps off the producer's SM
// sub-partition.  Warp w runs on sub-partition w % 4; in such a variant warps
// 4, 8, ... are launched idle and return at once, and the consumers take the
// other warps in order.  With the vectors as the MMA rows at head_dim 128,
// consumer warps beside the producer measured about a quarter slower per
// stage than the rest, and as every stage waits for its slowest consumer they
// set the pace (20-64 vectors per KV head: 5-6 % faster without them); at
// head_dim 64 and with the tokens as the rows the three-consumer
// sub-partitions this leaves cost more than it saves.
__host__ __device__ constexpr bool consumers_off_producer(int form, int head_dim) {
  return form == kFormVectorRows && head_dim == 128;
}
// Warps of a decode CTA: the producer, the consumers and any idle warps.
__host__ __device__ constexpr int cta_warps(int form, int head_dim, int consumer_warps) {
  return consumers_off_producer(form, head_dim) ? consumer_warps + 1 + (consumer_warps - 1) / 3
                                                : consumer_warps + 1;
}
constexpr int kMaxThreadsOffProducer = cta_warps(kFormVectorRows, 128, kMaxConsumerWarpsMulti) * 32;

// Whether a variant reads its query vectors from one fixed q slot: the
// vectors-as-rows form (whose query vectors are nearly always large) and the
// CUDA-core consumer with 2 or 4 vectors per warp.  A slot index known at
// compile time keeps their register allocations free of spills.
__host__ __device__ constexpr bool fixed_q_slot(int form, int qw) {
  return form == kFormVectorRows || form == kFormTmem || (form == kFormCuda && qw >= 2);
}

// Query-vector slots of the q ring: one per stage while the query vectors
// of a head group are small (a slot is then never waited for: a segment's
// slot is reused only after the stage that read it was released); one when
// they are large, which leaves the shared memory to the K/V stages at the
// price of a wait for segments shorter than the ring of stages, and one for
// the variants that read a fixed slot.
__host__ __device__ inline int q_slots_for(uint32_t q_bytes, int stages, int form, int qw) {
  if (form == kFormTmem) return 0;  // it reads its query rows from global memory
  return (!fixed_q_slot(form, qw) && q_bytes <= 8192u) ? stages : 1;
}

// The CUDA-core consumer also keeps per-vector probability buffers (the
// tensor-core forms hold probabilities in registers).  `blocks` is the
// blocks a stage holds (1 outside the TMEM form).
__host__ __device__ inline SmemLayout make_layout(int elem, int head_dim, int heads_per_cta,
                                                  int nvec, int stages, int rows, int form,
                                                  int qw, int blocks) {
  SmemLayout L;
  L.kv_bytes = (uint32_t)(heads_per_cta * kBlock * head_dim * elem);
  L.q_bytes = (uint32_t)(nvec * head_dim * elem);
  // Stages start on 1024-byte boundaries: 128-byte-swizzled TMA writes
  // need it (the kernel aligns the dynamic shared memory base itself).
  L.stage_bytes = align_up(2 * (uint32_t)blocks * L.kv_bytes, 1024);
  L.q_slots = (uint32_t)q_slots_for(L.q_bytes, stages, form, qw);
  L.q_slot_bytes = align_up(L.q_bytes, 128);
  L.off_q = (uint32_t)stages * L.stage_bytes;
  uint32_t off = L.off_q + L.q_slots * L.q_slot_bytes;
  L.off_meta = off;
  // an int4 per stage; the TMEM form adds one for its blocks' token masks
  off += (uint32_t)stages * (form == kFormTmem ? 32 : 16);
  L.off_bars = align_up(off, 8);
  // mbarriers: full[stages], empty[stages], qfree[q_slots]; the TMEM form
  // adds seven (scores ready [2], handed over [2], output ready, drained,
  // query rows ready)
  off = L.off_bars + (uint32_t)(2 * stages + (int)L.q_slots + (form == kFormTmem ? 7 : 0)) * 8;
  if (form == kFormTmem) {
    // its shared-memory MMA operand: two probability buffers (128 x a
    // stage's tokens of one head each; the query rows live in tensor
    // memory); then the softmax warp pairs' exchange of row maxima (two
    // stages x two warps x 128 rows) and of row sums (two pieces x two warps
    // x 128 rows)
    L.off_pbuf = align_up(off, 1024);
    off = L.off_pbuf + 2u * (uint32_t)(kTmemRows * blocks * kBlock * 2) +
          (4u + 4u) * kTmemRows * 4u;
  } else {
    L.off_pbuf = align_up(off, 16);
    off = L.off_pbuf + (form == kFormCuda ? (uint32_t)(nvec * kBlock * 4) : 0u);
  }
  L.off_ctx = off;
  off += (uint32_t)rows * 4;
  L.off_prefix = off;
  off += (uint32_t)(rows + 1) * 4;
  L.off_flag = align_up(off, 4);
  off = L.off_flag + 16;  // abort flag, merge flag, tensor-memory address
  L.total = align_up(off, 128) + 1024;  // + slack to align the base to 1024
  return L;
}

// Launchers (return the launch's cudaError_t).
cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int qw, int consumer,
                          int grid, int threads, int smem, cudaStream_t stream, bool pdl);
cudaError_t launch_kv_write(const KvWriteParams& p, cudaStream_t stream);
// One-time per-device attribute set-up of the decode kernels.
cudaError_t prepare_decode_kernels();
// CTAs of the plan's kernel variant that one SM of the current device holds
// (cudaOccupancyMaxActiveBlocksPerMultiprocessor).
cudaError_t decode_occupancy(int dtype, int head_dim, int qw, int consumer, int threads,
                             int smem, int* ctas);
// The bounded-wait self-test kernel (result: device [gave_up, waited_ns]);
// a wait that gives up also sets NSV_DEV_TIMEOUT in *status.
cudaError_t launch_wait_probe(unsigned long long limit_ns, unsigned long long* result,
                              uint32_t* status, cudaStream_t stream);
// The CUDA context current on the calling thread (null when there is none or
// it cannot be read): per-device state is keyed on it.
void* current_cuda_context();

}  // namespace nsv
