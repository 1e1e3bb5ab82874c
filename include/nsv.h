/*
 * nsv.h -- C ABI of the GB300 (sm_103a) batched paged-attention decode read
 * and KV append.
 *
 * The operation, as the nanoserve daily log defines it:
 *
 *   KV append (nanoserve Day 55, "the capture list moved to startup, and the
 *   dummy batch was all padding", section "Why it matters"): the step's new
 *   key and value of every row land at the row's write slot, as one indexed
 *   write over the padded batch.  A padded row's write slot is the sink slot,
 *   "one past the pool the allocator hands out": a legal address that no
 *   block table can name.
 *
 *   Decode read (nanoserve Day 59, "the rectangle the read builds, and the
 *   tile that replaces it", sections "What I added today" and "What I
 *   learned" items 3-4): one query token per row and per query head attends
 *   over that row's own context_lens[row] keys and values.  Position t of a
 *   row lives in pool block block_tables[row][t / block_size] at offset
 *   t % block_size (block-id addressing, Day 51, "the read rectangle stopped
 *   being built", section "Why it matters").  The read walks
 *   cdiv(ctx, block_size) blocks of the row, never the rest of the table,
 *   and folds them with an online softmax (running max, running denominator,
 *   running weighted sum of V).  Output = softmax(scale * q.K^T) V over the
 *   row's positions; a row with context length 0 attends over nothing and
 *   its output is 0.
 *
 * Ownership: every pointer passed in is owned by the caller; the library
 * never frees, retains or reallocates caller memory.  Device pointers must
 * be device memory of the current CUDA device.  All calls are asynchronous
 * on the given stream unless stated otherwise.
 *
 * Per-device state: on its first call on a device the library looks up the
 * device addresses of its status word and scratch buffers and sets kernel
 * attributes; it redoes this when it finds a different CUDA context current
 * on that device (after cudaDeviceReset, say).  The library-owned workspace
 * of the old context is dropped with it, not freed (its context is gone).
 *
 * Layouts (all C-contiguous, no strides; element type from nsv_shape.dtype):
 *   q, out          [rows][query_len][num_heads][head_dim]
 *   k_pool, v_pool  [num_blocks + 1][num_kv_heads][block_size][head_dim]
 *                   the last block (index num_blocks) is the sink block;
 *                   flat slot s is (block s / block_size, offset
 *                   s % block_size); the sink slot is num_blocks*block_size.
 *   k_new, v_new    [rows][query_len][num_kv_heads][head_dim]
 *   write_slots     [rows][query_len] int64
 *   block_tables    [rows][max_blocks] int32; entries at or past
 *                   cdiv(context_lens[r], block_size) are never read and may
 *                   hold anything (-1 by convention)
 *   context_lens    [rows] int32
 * Query head h reads KV head h / (num_heads / num_kv_heads).
 *
 * Several query tokens per row (query_len > 1, e.g. verifying speculative
 * tokens): the step appends query_len tokens per row and query token j of a
 * row of length ctx (which counts them) sits at position ctx - query_len + j
 * and sees the positions t < ctx - query_len + 1 + j.  This is the multi-
 * token form of the streaming loop that Day 59 "What I learned" item 3
 * describes (the single-sequence kernel's [n_q, d] accumulators), read as
 * causal among the step's new tokens; a query that sees no position outputs
 * 0.  query_len 1 is the decode read.
 * Every data pointer must be 16-byte aligned.
 *
 * Errors: every entry point returns NSV_OK (0) or a negative NSV_ERR_* code
 * after checking its host-visible arguments; nothing is launched when an
 * error is returned.  A batch of 0 rows is a valid no-op (its data pointers
 * may be NULL).  Values that live in device memory (context lengths,
 * block ids, write slots) are checked by the kernels themselves: a bad value
 * never causes an out-of-bounds access; the offending row, block or write is
 * skipped and a bit is set in the device status word (nsv_device_status).
 * No kernel traps.
 */
#ifndef NSV_H
#define NSV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define NSV_API __attribute__((visibility("default")))
#else
#define NSV_API
#endif

/* Element types of q, out, pools and new K/V (one type for all of them). */
enum { NSV_F32 = 0, NSV_BF16 = 1 };

/* Return codes. */
enum {
    NSV_OK = 0,
    NSV_ERR_NULLPTR = -1,     /* a required pointer is NULL */
    NSV_ERR_DTYPE = -2,       /* dtype is not NSV_F32 or NSV_BF16 */
    NSV_ERR_SHAPE = -3,       /* a size is out of its documented range */
    NSV_ERR_ALIGN = -4,       /* a data pointer is not 16-byte aligned */
    NSV_ERR_RANGE = -5,       /* a plan field is inconsistent with the shape */
    NSV_ERR_CAPTURE = -6,     /* the library workspace must grow while the
                                 stream is being captured */
    NSV_ERR_CUDA = -7,        /* a CUDA runtime call failed */
    NSV_ERR_WORKSPACE = -8,   /* workspace missing, misaligned or smaller than
                                 the plan needs */
    NSV_ERR_UNSUPPORTED = -10 /* head_dim or block_size the kernels lack */
};

/* Device status bits, sticky until cleared by nsv_device_status. */
enum {
    NSV_DEV_BAD_CTX = 1u,   /* context length outside [0, max_blocks*block_size];
                               the row was read as empty (output 0) */
    NSV_DEV_BAD_BLOCK = 2u, /* a walked block id outside [0, num_blocks], or a
                               read slot outside the pool; skipped */
    NSV_DEV_BAD_SLOT = 4u,  /* write slot outside [0, (num_blocks+1)*block_size);
                               that row's K/V was not written */
    NSV_DEV_TIMEOUT = 8u    /* an in-kernel wait gave up after its limit and the
                               kernel returned early; results are invalid */
};

/* Sizes of one decode batch.  Limits: 0 <= rows <= 8192; num_heads a
 * multiple of num_kv_heads; head_dim 64 or 128; block_size 16; 1 <=
 * max_blocks with max_blocks*block_size < 2^31; 1 <= num_blocks < 2^31 - 1;
 * query_len 0 or 1 (one query token per row) up to 64.  The query vectors
 * per KV head, query_len * num_heads/num_kv_heads, are at most 64 for bf16
 * (the tensor-core consumer) and at most 32 for fp32 (the CUDA-core
 * consumer; at most 15 when odd); beyond, the planner refuses with
 * NSV_ERR_SHAPE. */
typedef struct nsv_shape {
    int32_t rows;
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t max_blocks;   /* block-table row length; width = max_blocks*block_size */
    int64_t num_blocks;   /* blocks the allocator hands out; pools hold one more */
    int32_t dtype;        /* NSV_F32 or NSV_BF16 */
    int32_t query_len;    /* query tokens per row; 0 means 1 */
} nsv_shape;

/* Launch plan of the decode read.  A plan depends on the shape and the SM
 * count only, never on the values of context_lens, so one plan serves every
 * step of a given shape (and a captured graph of it).
 *
 * The read is split evenly over a persistent grid: the units (KV-head group,
 * row, block) of all rows are laid end to end and CTA c of `grid` takes the
 * units [c*U/grid, (c+1)*U/grid).  A row cut by CTA boundaries is finished by
 * the CTA that completes its last piece, which merges the partial softmax
 * states of all its pieces. */
typedef struct nsv_plan {
    int32_t kv_heads_per_cta; /* KV heads one CTA streams together (a head group) */
    int32_t stages;           /* shared-memory pipeline depth */
    int32_t ctas_per_sm;      /* resident CTAs per SM the grid is sized for */
    int32_t grid;             /* persistent CTAs launched */
    int32_t threads;          /* threads per CTA: a producer warp and the
                                 consumer warps; with the vectors as the MMA
                                 rows at head_dim 128 also idle warps 4, 8,
                                 ..., so that no consumer shares the
                                 producer's SM sub-partition */
    int32_t smem_bytes;       /* dynamic shared memory per CTA */
    int32_t num_sms;          /* SM count the plan was made for */
    int32_t vectors_per_warp; /* query vectors (query heads x query tokens
                                 that share a KV head) one consumer warp
                                 serves from each K/V tile: 1, 2 or 4
                                 (CUDA-core consumer; 1 for the tensor one) */
    int32_t consumer;         /* NSV_CONSUMER_CUDA, _TENSOR, _TENSOR_VECTOR_ROWS
                                 or _TENSOR_TMEM */
    int32_t blocks_per_stage; /* consecutive blocks of one row a stage holds:
                                 1 to 4 for NSV_CONSUMER_TENSOR_TMEM, else 1 */
    int64_t workspace_bytes;  /* device scratch the read needs */
} nsv_plan;

/* How a CTA's consumer warps fold a K/V tile into the softmax state.
 *  NSV_CONSUMER_CUDA:   fp32 FMAs on the CUDA cores; a warp serves
 *                       vectors_per_warp query vectors of one KV head.  Any
 *                       dtype and shape.
 *  NSV_CONSUMER_TENSOR: bf16 only.  A KV head's query vectors (query heads
 *                       of the group x query tokens, 2 to 64 of them) go
 *                       through 16x8x16 bf16 tensor-core MMAs with fp32
 *                       accumulation: scores against the block's keys, then
 *                       the weighted sum of its values, with the
 *                       probabilities rounded to bf16 for the second
 *                       product.  The block's 16 tokens are the MMA rows and
 *                       the vectors its columns, 8 per warp (one to four
 *                       warps per KV head).  K/V tiles arrive by 2-D TMA
 *                       with a 128-byte swizzle.  Needs
 *                       (num_blocks+1)*num_kv_heads*16 < 2^31.
 *  NSV_CONSUMER_TENSOR_VECTOR_ROWS: the same with the query vectors as the
 *                       MMA rows, 16 per warp (one to four warps per KV head).
 *  NSV_CONSUMER_TENSOR_TMEM: bf16 only, on the 5th-generation tensor cores
 *                       (tcgen05.mma with the accumulators in tensor
 *                       memory).  The MMA's 128 rows are the query vectors
 *                       of a group of 4, 2 or 1 KV heads (128 / group rows
 *                       each, zero past the vectors; group x head_dim at
 *                       most 256): kv_heads_per_cta is the group, which must
 *                       divide num_kv_heads; by default the largest that
 *                       fits.  A stage holds blocks_per_stage consecutive
 *                       blocks of one row (fewer at a segment's end), and
 *                       one scores MMA per 16 dims covers all of them.
 *                       One CTA per SM: a producer warp, eight softmax
 *                       warps (one thread per row, two warps per tensor-
 *                       memory lane quadrant) and an MMA warp that issues
 *                       the next stage's scores while the softmax warps
 *                       work; K and V tiles by one multi-dimensional TMA box
 *                       per block.  At head_dim 64 the default takes it
 *                       from 33 query vectors per KV head.
 * The default plan takes NSV_CONSUMER_TENSOR for bf16 shapes with 2 to 8
 * query vectors per KV head, NSV_CONSUMER_TENSOR_VECTOR_ROWS for 9 to 16,
 * NSV_CONSUMER_TENSOR_TMEM for 17 to 64 (33 to 64 at head_dim 64) when its
 * group can be 2 or 4 KV heads (NSV_CONSUMER_TENSOR_VECTOR_ROWS otherwise,
 * for example for an odd num_kv_heads), and the CUDA-core one otherwise.  Outside the TMEM form
 * the default kv_heads_per_cta is, among 1 and the groups whose K+V stage
 * is at most 64 KiB and whose vectors need at most 8 consumer warps, the
 * one whose plan keeps the most consumer warps resident per SM (counted up
 * to 16; the larger group on a tie), and the default ctas_per_sm is as many
 * as shared memory, threads and registers allow, up to 8 (1 for the TMEM
 * form, which takes the largest blocks_per_stage that leaves it a ring of
 * at least 3 stages, up to 6).  The default ring is 3 stages; a tensor-core CTA alone on its SM
 * deepens it to fill shared memory (up to 6), and a CUDA-core CTA that
 * streams all of one or two KV heads in stages of at most 16 KiB takes 2
 * where that fits more CTAs per SM. */
enum {
    NSV_CONSUMER_AUTO = 0,
    NSV_CONSUMER_CUDA = 1,
    NSV_CONSUMER_TENSOR = 2,
    NSV_CONSUMER_TENSOR_VECTOR_ROWS = 3,
    NSV_CONSUMER_TENSOR_TMEM = 4
};

/*
 * Plan the decode read for `shape` on a GPU with `num_sms` SMs (<= 0: the
 * current device's count).  Host-only apart from that optional device query;
 * deterministic; depends on the shape alone.  Returns NSV_OK or
 * NSV_ERR_{NULLPTR, DTYPE, SHAPE, UNSUPPORTED, CUDA}.
 *
 * Why the shape alone: the streamed read's saving over the rectangle is a
 * property of the width axis only, rows and heads cancelling out of it
 * (Day 59, "Why it matters", first paragraph), and a read that accumulates
 * tile by tile has no width to specialise on, so the shapes a server
 * presents are its batch sizes (Day 59, "What I learned" item 7).  A step
 * recorded into a CUDA graph is bound to what it was launched with, and it
 * is recorded on a batch whose rows are all padding (Day 55, "the capture
 * list moved to startup, and the dummy batch was all padding", "Why it
 * matters"): a plan chosen from the lengths would differ between that warm
 * batch and the real ones.  How the work is split (stream-K over a
 * persistent grid, with the pieces of a cut row merged flash-decoding
 * style) is this library's design; the pages' kernel runs one program per
 * (row, query head).
 */
NSV_API int nsv_plan_split(const nsv_shape *shape, int num_sms, nsv_plan *plan);

/*
 * The same planner with some choices fixed, for sweeps and tests (the pages
 * have no counterpart; every plan it returns is one the read runs
 * correctly).  Any argument <= 0 is chosen by the heuristic: kv_heads_per_cta (must divide num_kv_heads), stages (2..8),
 * ctas_per_sm (1..8), grid (persistent CTAs; default num_sms * ctas_per_sm)
 * vectors_per_warp (1, 2 or 4, dividing the query vectors per KV head;
 * at most 16 consumer warps for 1 or 2, 8 for 4; CUDA-core consumer only),
 * consumer (NSV_CONSUMER_*; AUTO picks as the default plan does) and
 * blocks_per_stage (1 to 4, NSV_CONSUMER_TENSOR_TMEM only; its scores
 * product is at most 256 tokens wide and its tensor-memory columns at most
 * 512).  Returns NSV_ERR_RANGE when a fixed choice does not fit the shape or
 * the shared-memory limit, or asks for the tensor consumer where it does not
 * apply.
 */
NSV_API int nsv_plan_custom(const nsv_shape *shape, int num_sms, int kv_heads_per_cta,
                            int stages, int ctas_per_sm, int grid, int vectors_per_warp,
                            int consumer, int blocks_per_stage, nsv_plan *plan);

/*
 * How many CTAs of `plan`'s kernel one SM of the current device holds at the
 * plan's threads and shared memory (the CUDA occupancy calculator on the
 * compiled kernel).  A plan's grid is sized as num_sms * ctas_per_sm on the
 * assumption that all of them are resident at once; this reports whether
 * the device agrees (*ctas_per_sm >= plan->ctas_per_sm).  `plan` must be one
 * the planner made for `shape`.  Returns NSV_ERR_{NULLPTR, RANGE, CUDA} or a
 * shape error.
 */
NSV_API int nsv_plan_resident_ctas(const nsv_shape *shape, const nsv_plan *plan,
                                   int *ctas_per_sm);

/*
 * KV append: for every row r (and each of its query_len new tokens j),
 * k_pool/v_pool at slot write_slots[r][j] receive k_new[r][j]/v_new[r][j]
 * (all KV heads), bit for bit.  Real rows' slots must be
 * distinct; any number of padded rows may name the sink slot, whose contents
 * are then unspecified.  Pool bytes at every other slot are untouched.
 * A slot outside [0, (num_blocks+1)*block_size) is skipped and sets
 * NSV_DEV_BAD_SLOT.  Uses shape.rows, query_len, num_kv_heads, head_dim,
 * block_size, num_blocks, dtype (num_heads and max_blocks must still be
 * valid).
 */
NSV_API int nsv_kv_write(const nsv_shape *shape, const void *k_new, const void *v_new,
                         const int64_t *write_slots, void *k_pool, void *v_pool,
                         cudaStream_t stream);

/*
 * Decode read with the default plan and a library-owned workspace (one per
 * device, grown with cudaMalloc on first need and kept until exit; returns
 * NSV_ERR_CAPTURE instead of growing it while `stream` is capturing, so make
 * one uncaptured call of each shape first).  Calls on different streams of
 * one device must not overlap when they share that workspace.
 * out[r][h] = softmax over the row's positions of scale * q[r][h].K, times V.
 */
NSV_API int nsv_paged_decode(const nsv_shape *shape, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *block_tables,
                             const int32_t *context_lens, float scale, void *out,
                             cudaStream_t stream);

/*
 * Decode read with an explicit plan (NULL: the default plan) and a
 * caller-owned device workspace of at least plan->workspace_bytes bytes
 * (256-byte aligned).  The workspace holds no state between calls; each
 * call clears the part that must start at zero on `stream` with a small
 * kernel of its own (the append kernel given no rows), and launches the
 * read programmatically dependent on it.  Two calls that overlap on the GPU
 * need two workspaces.  A plan passed in must be one nsv_plan_split/nsv_plan_custom
 * returned for this shape (NSV_ERR_RANGE otherwise).
 *
 * The workspace is the read's only intermediate in device memory: one
 * arrival counter per (row, KV-head group) and, per CTA, at most two partial
 * softmax states (running max, denominator, weighted sum of V) of the query
 * vectors it serves.  It stands where the gather read's [rows, heads, 1,
 * width] score rectangle stood (Day 59, "What I added today": 268.4 MB at
 * 256 rows, 32 heads and width 8192, against one tile and three
 * accumulators for the streamed read), and it is sized by the grid, not by
 * rows x width (1.27 MB at that shape).  A workspace at a fixed caller
 * address is what a captured step replays against (Day 55, "Why it
 * matters": a graph is bound to the addresses it was launched with).
 */
NSV_API int nsv_paged_decode_ws(const nsv_shape *shape, const nsv_plan *plan,
                                const void *q, const void *k_pool, const void *v_pool,
                                const int32_t *block_tables, const int32_t *context_lens,
                                float scale, void *out, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * One serving step: nsv_kv_write then the decode read on the same stream.
 * context_lens already count the appended token: the write slot is the
 * row's last real entry (Day 51, "the read rectangle stopped being built",
 * "What I learned" item 2), so the read must see what the append wrote, and
 * a padded row writes the sink slot and reads nothing (Day 55, "Why it
 * matters").  plan/workspace as in nsv_paged_decode_ws;
 * workspace NULL with workspace_bytes 0 uses the library-owned workspace.
 * Both halves' arguments are checked before either is launched: on an
 * error return nothing was launched.  The append's launch also zeroes the
 * read's arrival counters, so the step is two kernels and no memset.
 */
NSV_API int nsv_decode_step(const nsv_shape *shape, const nsv_plan *plan, const void *q,
                            const void *k_new, const void *v_new,
                            const int64_t *write_slots, void *k_pool, void *v_pool,
                            const int32_t *block_tables, const int32_t *context_lens,
                            float scale, void *out, void *workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/*
 * Decode read that allocates nothing, for callers that cannot call
 * cudaMalloc or hand the library scratch memory: engines that own all device
 * memory through a fixed arena, plugin hooks that only receive pre-bound
 * buffers, loops that must avoid the device-wide synchronisation an
 * allocation can cause.  The nanoserve pages have no counterpart; this is a
 * deployment convenience of this library.
 *
 * Same arguments, layouts and result as nsv_paged_decode (default plan).  The
 * split path's scratch comes from a buffer of NSV_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library holds
 * until exit; a shape whose plan needs more (plan.workspace_bytes) is
 * refused with NSV_ERR_WORKSPACE and nothing is launched.  The first call on
 * a device looks up the buffer's device address (cudaGetSymbolAddress, no
 * allocation); make that first call before any stream capture.  Calls share
 * the buffer: two calls whose kernels overlap on the GPU race on it.  The
 * caller never clears it: the part that must start at zero (the read's
 * arrival counters) is zeroed by each call on `stream` with a small kernel
 * of its own, and each call writes the rest before reading it.
 */
#define NSV_NOALLOC_SCRATCH_BYTES (4u << 20)

NSV_API int nsv_paged_decode_noalloc(const nsv_shape *shape, const void *q,
                                     const void *k_pool, const void *v_pool,
                                     const int32_t *block_tables,
                                     const int32_t *context_lens, float scale, void *out,
                                     cudaStream_t stream);

/*
 * Decode read through a per-token slot table instead of block tables
 * (nanoserve Day 51, "the read rectangle stopped being built", "What I added
 * today": the SlotTable, one [max_batch_size, max_model_len] int64 buffer of
 * flat slots, read as a window [rows, width] with the buffer's row stride).
 * Position t of row r lives at flat slot slot_table[r * slot_row_stride + t],
 * i.e. block slot / block_size, offset slot % block_size.  Only positions
 * t < context_lens[r] are read, and context_lens[r] <= slot_cols <=
 * min(slot_row_stride, max_blocks * block_size) (a longer row is read as
 * empty and flagged NSV_DEV_BAD_CTX).
 *
 * A block whose slots form one aligned run of consecutive slots (always so
 * for a table built from block tables) is moved with the same bulk copies as
 * the block-table read and gives the same bits; any other block is gathered
 * token by token.  A slot outside [0, (num_blocks+1)*block_size) is skipped
 * and sets NSV_DEV_BAD_BLOCK.  plan and workspace as in nsv_decode_step
 * (workspace NULL with workspace_bytes 0: the library-owned workspace).
 */
NSV_API int nsv_paged_decode_slots(const nsv_shape *shape, const nsv_plan *plan,
                                   const void *q, const void *k_pool, const void *v_pool,
                                   const int64_t *slot_table, int64_t slot_cols,
                                   int64_t slot_row_stride, const int32_t *context_lens,
                                   float scale, void *out, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/*
 * Self-test of the bounded wait (the pages have no counterpart; this checks
 * the library's own failure detection).  Every pipeline wait of the decode
 * kernel gives up after a limit (1 s) instead of spinning forever; a wait
 * that gives up sets NSV_DEV_TIMEOUT and the kernel returns, leaving the
 * context usable.  This call runs that same wait routine in a one-thread
 * kernel, with limit_ns (1 us .. 2 s), on an mbarrier phase that nothing
 * completes, so it must give up; when it does, it sets NSV_DEV_TIMEOUT in
 * the device status word exactly as a decode kernel's wait would, so the
 * whole signalling path (nsv_device_status, nsv_status_async) can be
 * checked without a fault.  Synchronous on `stream`; touches no caller
 * memory.  On NSV_OK, *gave_up is 1 when the wait gave up (the expected
 * outcome) and *waited_ns is how long it waited.  Returns
 * NSV_ERR_{NULLPTR, RANGE, CUDA}.
 */
NSV_API int nsv_selftest_bounded_wait(uint64_t limit_ns, int *gave_up, uint64_t *waited_ns,
                                      cudaStream_t stream);

/*
 * Synchronise the current device, then report its status word (NSV_DEV_*
 * bits raised since the last clear) and the number of (row, block) pairs the
 * decode kernels walked (each row's cdiv(ctx, block_size) blocks, counted
 * once per row, not per head).  Either output pointer may be NULL.  clear != 0
 * resets both.  Not for use inside stream capture.
 */
NSV_API int nsv_device_status(uint32_t *status, uint64_t *blocks_walked, int clear);

/*
 * The status word without a device-wide synchronisation, for a serving loop
 * that must learn of NSV_DEV_TIMEOUT or a flagged bad value before it uses a
 * step's output (the pages have no counterpart: Day 59, "What I added
 * today", has the kernel make every refusal the oracle makes, and this is
 * how a caller hears of one).  Enqueues on `stream` a 4-byte copy of the
 * current device's status word into `dst`, which is device memory or
 * page-locked host memory of at least 4 bytes, 4-byte aligned, owned by the
 * caller; with clear != 0 it then zeroes the status word, also on `stream`.
 * Nothing waits: `dst` holds the bits raised by all work ordered before the
 * copy once `stream` reaches it (for pinned host memory, after the caller
 * synchronises `stream` or an event recorded after this call).  The status
 * word is one per device and sticky: bits raised by work on other streams
 * show up too, and a clear can drop a bit that such work raises between the
 * copy and the clear.  Returns NSV_ERR_{NULLPTR, ALIGN, CUDA}.
 */
NSV_API int nsv_status_async(uint32_t *dst, int clear, cudaStream_t stream);

/* Static description of a return code. */
NSV_API const char *nsv_strerror(int code);

/* ABI version of this header (major * 100 + minor). */
NSV_API int nsv_abi_version(void);

#define NSV_ABI_VERSION 102

#ifdef __cplusplus
}
#endif

#endif /* NSV_H */
