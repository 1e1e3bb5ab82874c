/*
 * nsv_oracle.c -- the oracle for the batched paged-attention decode read and
 * the KV append.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, obviously correct CPU statement of what the hot
 * path computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference arm load it.  The product library never links,
 * loads or calls it, and it shares no code, header, table or helper with the
 * CUDA path.
 *
 * Source pages (nanoserve daily log):
 *   [Day 59] "the rectangle the read builds, and the tile that replaces it",
 *            sections "What I added today" and "Why it matters".
 *   [Day 55] "the capture list moved to startup, and the dummy batch was all
 *            padding", section "Why it matters" (padded rows, sink slot,
 *            the append as one indexed write over the padded batch).
 *   [Day 51] "the read rectangle stopped being built, and the length that
 *            could not be shared", sections "Why it matters" (block-id
 *            addressing: slot = block_id * block_size + offset) and
 *            "What I learned" item 2 (the write slot is the row's last real
 *            entry).
 *
 * What it computes, in the pages' terms:
 *   - oracle_paged_decode: the reference read.  For each selected row and
 *     query head it gathers the row's whole rectangle of keys and values
 *     (every one of the row's max_blocks block-table entries, padding
 *     included), scores every position of the rectangle, kills positions at
 *     or past the row's context length by selecting -inf, and takes a
 *     two-pass softmax and the probability-weighted sum of values, all in
 *     fp64.  Because it gathers before it masks, a padding entry must be a
 *     legal index; a negative entry wraps onto the end of the pool array the
 *     way a Python index does (Day 59, "Why it matters").
 *     With query_len = n > 1 (several query tokens per row, the multi-token
 *     form of the Day-22 single-sequence loop that Day 59 "What I learned"
 *     item 3 describes with [n_q, d] accumulators), query token j of a row
 *     of length ctx sits at position ctx - n + j and sees the positions
 *     t < ctx - n + 1 + j (causal within the step's new tokens); a query
 *     that sees no position outputs 0.  query_len 1 is the decode read.
 *   - oracle_paged_decode_slots: the same read through a per-token slot
 *     table instead of a block table (Day 51 "What I added today": the
 *     SlotTable window the reference read gathers through).
 *   - oracle_kv_write: pool[write_slots[r]] = new[r], one row at a time.
 *   - oracle_walked_tiles / oracle_rect_tiles: the tile accounting of the
 *     streamed read (tiles walked = sum over rows of cdiv(ctx, tile); the
 *     rectangle charges every row cdiv(width, tile) tiles) -- Day 59,
 *     "What I added today" (streamed_work) and "What I learned" item 4.
 *   - oracle_score_rect_bytes / oracle_score_tile_bytes: what one decode step
 *     holds as fp32 scores in the rectangle read ([rows, heads, 1, width])
 *     against the streamed read ([rows, heads, tile]) -- Day 59 table.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - a row with context length 0 attends over nothing; its output is 0.
 *   - the pool arrays hold num_blocks + 1 blocks; the last one is the sink
 *     block, so the sink slot is num_blocks * block_size ("one past the pool
 *     the allocator hands out").
 *   - pool layout [num_blocks + 1][kv_heads][block_size][head_dim]; query and
 *     output layout [rows][heads][head_dim]; query head h reads KV head
 *     h / (heads / kv_heads).
 *
 * Refusals (returned as negative codes, matching the product library's):
 *   -3  a shape argument is not positive, or heads % kv_heads != 0
 *   -5  a selected row's context length is outside [0, max_blocks*block_size],
 *       a block-table entry of a selected row is not a legal (wrapping)
 *       index into the num_blocks + 1 block array, a selected row index is
 *       out of range, or a write slot is outside [0, (num_blocks+1)*block_size)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_OK = 0, OR_ERR_SHAPE = -3, OR_ERR_RANGE = -5, OR_ERR_NOMEM = -9 };

/* Widen one stored element to fp64.  bf16 is the upper half of an IEEE fp32,
 * so the conversion is exact. */
static double widen(const void *base, int dtype, int64_t idx)
{
    if (dtype == OR_F32)
        return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int elem_bytes(int dtype)
{
    return dtype == OR_F32 ? 4 : 2;
}

/*
 * The reference read over a subset of rows, through either addressing form:
 * a block table [R][MB] (position t of row r in block table[r][t / B] at
 * offset t % B; W = MB * B) or a slot table (position t of row r at flat
 * slot slots[r * stride + t], slot s being block s / B, offset s % B; the
 * rectangle is the table's first W columns).
 *
 * NQ: query tokens per row (1 for the decode read).
 * rows / nrows: which rows to compute (rows == NULL means 0..R-1, nrows = R).
 * out: fp64 [nrows][NQ][H][D], row i of out belongs to batch row rows[i].
 * threads: OpenMP threads (<= 0 means the runtime default).
 */
static int read_rect(int64_t R, int64_t NQ, int64_t H, int64_t Hkv, int64_t D,
                     int64_t B, int64_t MB, int64_t W, int64_t NB, int dtype,
                     const void *q, const void *k_pool, const void *v_pool,
                     const int32_t *block_tables, const int64_t *slots,
                     int64_t stride, const int32_t *context_lens,
                     double scale, const int64_t *rows, int64_t nrows,
                     int threads, double *out)
{
    if (R < 0 || NQ <= 0 || H <= 0 || Hkv <= 0 || D <= 0 || B <= 0 ||
        W <= 0 || NB <= 0 || H % Hkv != 0 ||
        (dtype != OR_F32 && dtype != OR_BF16))
        return OR_ERR_SHAPE;
    if (slots == NULL && MB <= 0)
        return OR_ERR_SHAPE;
    if (slots != NULL && stride < W)
        return OR_ERR_SHAPE;
    if (rows == NULL)
        nrows = R;
    const int64_t pool_blocks = NB + 1; /* allocator's blocks + the sink */
    const int64_t group = H / Hkv;

    /* The oracle's own refusals, checked before any arithmetic: every entry
     * of the rectangle it gathers must be a legal (wrapping) index. */
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= R)
            return OR_ERR_RANGE;
        int64_t c = context_lens[r];
        if (c < 0 || c > W)
            return OR_ERR_RANGE;
        if (slots == NULL) {
            for (int64_t j = 0; j < MB; ++j) {
                int64_t b = block_tables[r * MB + j];
                if (b < -pool_blocks || b >= pool_blocks)
                    return OR_ERR_RANGE;
            }
        } else {
            for (int64_t t = 0; t < W; ++t) {
                int64_t e = slots[r * stride + t];
                if (e < -pool_blocks * B || e >= pool_blocks * B)
                    return OR_ERR_RANGE;
            }
        }
    }

    int failed = 0;
    const int64_t items = nrows * NQ * H;
#ifdef _OPENMP
    int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        /* Per-thread rectangle of one (row, KV head): [W][D] keys and values,
         * plus the [W] score row. */
        double *Krect = (double *)malloc(sizeof(double) * (size_t)(W * D));
        double *Vrect = (double *)malloc(sizeof(double) * (size_t)(W * D));
        double *s = (double *)malloc(sizeof(double) * (size_t)W);
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        if (!Krect || !Vrect || !s || !qv) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t it = 0; it < items; ++it) {
            if (failed)
                continue;
            int64_t i = it / (NQ * H), jq = (it / H) % NQ, h = it % H;
            int64_t r = rows ? rows[i] : i;
            int64_t g = h / group;
            /* positions this query sees: all of the row's for the last
             * query token, one fewer for each token before it */
            int64_t c = context_lens[r] - (NQ - 1 - jq);
            if (c < 0)
                c = 0;
            double *o = out + ((i * NQ + jq) * H + h) * D;

            /* 1. Gather the whole rectangle through the addressing. */
            for (int64_t t = 0; t < W; ++t) {
                int64_t base;
                if (slots == NULL) {
                    /* position t lives in block table[r][t / B], offset t % B */
                    int64_t b = block_tables[r * MB + t / B];
                    if (b < 0)
                        b += pool_blocks; /* a negative index wraps, as in Python */
                    base = ((b * Hkv + g) * B + t % B) * D;
                } else {
                    /* position t lives at flat slot slots[r][t] */
                    int64_t sl = slots[r * stride + t];
                    if (sl < 0)
                        sl += pool_blocks * B; /* wraps, as in Python */
                    base = (((sl / B) * Hkv + g) * B + sl % B) * D;
                }
                for (int64_t d = 0; d < D; ++d) {
                    Krect[t * D + d] = widen(k_pool, dtype, base + d);
                    Vrect[t * D + d] = widen(v_pool, dtype, base + d);
                }
            }
            for (int64_t d = 0; d < D; ++d)
                qv[d] = widen(q, dtype, ((r * NQ + jq) * H + h) * D + d);

            /* 2. Score every position of the rectangle. */
            for (int64_t t = 0; t < W; ++t) {
                double acc = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    acc += qv[d] * Krect[t * D + d];
                s[t] = scale * acc;
            }

            /* 3. Mask by length: positions at or past ctx become -inf. */
            for (int64_t t = 0; t < W; ++t)
                s[t] = (t < c) ? s[t] : -INFINITY;

            if (c == 0) { /* sees no position: output 0 */
                for (int64_t d = 0; d < D; ++d)
                    o[d] = 0.0;
                continue;
            }

            /* 4. Two-pass softmax over the rectangle. */
            double m = -INFINITY;
            for (int64_t t = 0; t < W; ++t)
                if (s[t] > m)
                    m = s[t];
            double z = 0.0;
            for (int64_t t = 0; t < W; ++t) {
                s[t] = exp(s[t] - m); /* exp(-inf) = 0 for masked positions */
                z += s[t];
            }
            for (int64_t t = 0; t < W; ++t)
                s[t] /= z;

            /* 5. Probability-weighted sum of values over the rectangle. */
            for (int64_t d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t t = 0; t < W; ++t)
                for (int64_t d = 0; d < D; ++d)
                    o[d] += s[t] * Vrect[t * D + d];
        }
        free(Krect);
        free(Vrect);
        free(s);
        free(qv);
    }
    return failed ? OR_ERR_NOMEM : OR_OK;
}

/* The read through block tables (the decode read of the Day-59 page). */
int oracle_paged_decode(int64_t R, int64_t NQ, int64_t H, int64_t Hkv,
                        int64_t D, int64_t B, int64_t MB, int64_t NB,
                        int dtype, const void *q, const void *k_pool,
                        const void *v_pool, const int32_t *block_tables,
                        const int32_t *context_lens, double scale,
                        const int64_t *rows, int64_t nrows, int threads,
                        double *out)
{
    return read_rect(R, NQ, H, Hkv, D, B, MB, MB * B, NB, dtype, q, k_pool,
                     v_pool, block_tables, NULL, 0, context_lens, scale, rows,
                     nrows, threads, out);
}

/* The read through a per-token slot table (nanoserve Day 51, "the read
 * rectangle stopped being built", "What I added today": the SlotTable's
 * [rows, width] window of flat slots, row stride `stride`, that the
 * reference read gathers through). */
int oracle_paged_decode_slots(int64_t R, int64_t NQ, int64_t H, int64_t Hkv,
                              int64_t D, int64_t B, int64_t W, int64_t stride,
                              int64_t NB, int dtype, const void *q,
                              const void *k_pool, const void *v_pool,
                              const int64_t *slots, const int32_t *context_lens,
                              double scale, const int64_t *rows, int64_t nrows,
                              int threads, double *out)
{
    if (slots == NULL)
        return OR_ERR_SHAPE;
    return read_rect(R, NQ, H, Hkv, D, B, 0, W, NB, dtype, q, k_pool, v_pool,
                     NULL, slots, stride, context_lens, scale, rows, nrows,
                     threads, out);
}

/*
 * The KV append: for every row, the row's new key and value land at its
 * write slot; every other pool element keeps its bytes.  Padded rows name the
 * sink slot.  The copy is bytewise, so it is exact for either element type.
 * All slots are checked before anything is written.
 */
int oracle_kv_write(int64_t R, int64_t Hkv, int64_t D, int64_t B, int64_t NB,
                    int dtype, const void *k_new, const void *v_new,
                    const int64_t *write_slots, void *k_pool, void *v_pool)
{
    if (R < 0 || Hkv <= 0 || D <= 0 || B <= 0 || NB <= 0 ||
        (dtype != OR_F32 && dtype != OR_BF16))
        return OR_ERR_SHAPE;
    const int64_t slots = (NB + 1) * B;
    for (int64_t r = 0; r < R; ++r)
        if (write_slots[r] < 0 || write_slots[r] >= slots)
            return OR_ERR_RANGE;
    const int es = elem_bytes(dtype);
    for (int64_t r = 0; r < R; ++r) {
        int64_t blk = write_slots[r] / B, off = write_slots[r] % B;
        for (int64_t g = 0; g < Hkv; ++g) {
            size_t dst = (size_t)(((blk * Hkv + g) * B + off) * D) * es;
            size_t src = (size_t)((r * Hkv + g) * D) * es;
            memcpy((char *)k_pool + dst, (const char *)k_new + src,
                   (size_t)D * es);
            memcpy((char *)v_pool + dst, (const char *)v_new + src,
                   (size_t)D * es);
        }
    }
    return OR_OK;
}

/* Tiles the streamed read walks: sum over rows of cdiv(ctx, tile). */
int64_t oracle_walked_tiles(const int32_t *context_lens, int64_t R,
                            int64_t tile)
{
    int64_t n = 0;
    for (int64_t r = 0; r < R; ++r)
        n += (context_lens[r] + tile - 1) / tile;
    return n;
}

/* Tiles the rectangle implies: every row is charged the full width. */
int64_t oracle_rect_tiles(int64_t R, int64_t width, int64_t tile)
{
    return R * ((width + tile - 1) / tile);
}

/* fp32 score bytes of the rectangle read, [rows, heads, 1, width]. */
int64_t oracle_score_rect_bytes(int64_t R, int64_t H, int64_t width)
{
    return R * H * width * 4;
}

/* fp32 score bytes the streamed read holds, one [tile] row per (row, head). */
int64_t oracle_score_tile_bytes(int64_t R, int64_t H, int64_t tile)
{
    return R * H * tile * 4;
}
