/*
 * kv_oracle.c -- plain, slow, single-threaded CPU oracle of the paged
 * KV-cache hot path (slot mapping, range slot mapping, KV write, block-table
 * gather, kernel-block expansion) and of its next steps (range expansion
 * into a block table, range-addressed gather, copy-on-write block copy).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg and reference arm may load this library.  It shares no code,
 * header or constant table with the CUDA library: every definition here is
 * written out again from the pages it cites.
 *
 * Sources (page title, section):
 *   [BT]  "Blocktabelle" (vLLM v0.25.1 walkthrough): Verantwortung,
 *         Entwurfsmotivation, Datenfluss (slot-mapping kernel signature and
 *         padding branch), Grenzen und Fehler.
 *   [VBM] "vLLM Block Table Management": Symbol Map, Deep Dive 1 (null block),
 *         Deep Dive 7 (worker materialisation, map_to_kernel_blocks),
 *         Deep Dive 8 (slot_mapping), PagedAttention Figure 6 walkthrough.
 *   [RNG] "Range-addressed KV cache blocks for the vLLM serving engine":
 *         The Innovation (paged and range formulas, PAD for positions outside
 *         every range), The Coordinate Approach (n(layer, block, token)),
 *         The Fork Implementation (256-range cap, fail closed).
 *
 * Conventions (readings where the pages are silent are marked READING):
 *   PAD id = -1 ([VBM] Deep Dive 8 stores PAD_SLOT_ID (-1)).
 *   Null block id = 0 ([VBM] Symbol Map: block 0, never cached or freed).
 *   Slot ids are int64, block tables int32 ([VBM] Deep Dive 8 "Remember").
 *   bf16 values are copied as raw 16-bit patterns: every output is an integer
 *   or copied bits, so results are exact.
 *
 * Parity status: every function is pinned by the tests to the pages' worked
 * examples, closed forms, brute force or invariants, except the
 * context-parallel filter (orc_slot_mapping_paged_cp): PARITY UNPINNED beyond
 * world size 1, its formula being cut off on the pages (a reading; pinned only
 * at world size 1 and by partition/distinctness properties).
 *
 * Error word bits (OR-ed into *err; identical meaning in the CUDA library):
 *   1 BAD_BLOCK, 2 BAD_SLOT, 4 BAD_POSITION, 8 BAD_RANGE, 16 NULL_WRITE,
 *   32 BAD_QSL, 64 OUT_OF_SPACE.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORC_PAD_SLOT (-1LL)
#define ORC_NULL_BLOCK 0
#define ORC_RANGE_CAP 256

enum {
    ORC_BAD_BLOCK = 1,
    ORC_BAD_SLOT = 2,
    ORC_BAD_POSITION = 4,
    ORC_BAD_RANGE = 8,
    ORC_NULL_WRITE = 16,
    ORC_BAD_QSL = 32,
    ORC_OUT_OF_SPACE = 64,
};

enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_EUNSUPPORTED = -2 };

/* --------------------------------------------------------------------- */
/* Coordinate map: [RNG] The Coordinate Approach,
 *   n(layer, block, token) = (layer * B + block) * T + token.
 * Row n of a [L, B, T, H, D] cache starts at element n * H * D.            */
int64_t orc_coord(int64_t layer, int64_t block, int64_t token, int64_t B, int64_t T)
{
    return (layer * B + block) * T + token;
}

/* --------------------------------------------------------------------- */
/* query_start_loc sanity: spans must be non-decreasing, start at or after
 * token 0 and end at or before num_tokens.  READING: a violation raises
 * BAD_QSL; slot values are only defined for non-decreasing spans.          */
static int32_t qsl_errors(const int32_t* qsl, int32_t R, int32_t N)
{
    int32_t e = 0;
    if (R <= 0) return 0;
    if (qsl[0] < 0 || qsl[R] > N) e |= ORC_BAD_QSL;
    for (int32_t r = 0; r < R; ++r)
        if (qsl[r] > qsl[r + 1]) e |= ORC_BAD_QSL;
    return e;
}

/* Paged slot of one position of request r.
 * [RNG] The Innovation: physical_block = block_table[req][position // block_size];
 * [VBM] Deep Dive 8: slot = block_number * block_size + offset.
 * READING: a position whose logical block lies past the table row, or whose
 * table entry is the null block, gets the PAD id ([BT] CUDA-graph padding:
 * null entries are skipped; [RNG] out-of-range positions get the pad id).
 * A negative position gets PAD and BAD_POSITION; an entry outside
 * [1, num_blocks) gets PAD and BAD_BLOCK.                                   */
static int64_t paged_slot(int64_t p, const int32_t* row, int32_t stride, int32_t T,
                          int64_t B, int32_t* err)
{
    if (p < 0) { *err |= ORC_BAD_POSITION; return ORC_PAD_SLOT; }
    int64_t lb = p / T;
    if (lb >= stride) return ORC_PAD_SLOT;
    int64_t b = row[lb];
    if (b == ORC_NULL_BLOCK) return ORC_PAD_SLOT;
    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }
    return b * T + p % T;
}

/* [BT] Datenfluss: one program per request walks the request's tokens
 * [qsl[r], qsl[r+1]); the last program fills [num_tokens, max_num_tokens)
 * with the pad id.  READING: tokens below num_tokens that no request span
 * covers are PAD as well.                                                   */
int orc_slot_mapping_paged(const int32_t* qsl, const int64_t* positions,
                           const int32_t* block_table, int32_t table_stride,
                           int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                           int32_t block_size, int64_t num_blocks,
                           int64_t* slot_mapping, int32_t* err)
{
    if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
        num_blocks < 1 || table_stride < 0)
        return ORC_EINVAL;
    int32_t e = 0;
    for (int32_t t = 0; t < max_num_tokens; ++t) slot_mapping[t] = ORC_PAD_SLOT;
    e |= qsl_errors(qsl, num_reqs, num_tokens);
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t lo = qsl[r] < 0 ? 0 : qsl[r];
        int32_t hi = qsl[r + 1] > num_tokens ? num_tokens : qsl[r + 1];
        const int32_t* row = block_table + (int64_t)r * table_stride;
        for (int32_t t = lo; t < hi; ++t)
            slot_mapping[t] = paged_slot(positions[t], row, table_stride, block_size, num_blocks, &e);
    }
    *err |= e;
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* Context-parallel filter of the paged slot mapping.  PARITY UNPINNED beyond
 * world size 1: [BT] Entwurfsmotivation names the three constants
 * (TOTAL_CP_WORLD_SIZE, TOTAL_CP_RANK, CP_KV_CACHE_INTERLEAVE_SIZE) and says
 * the kernel writes real slots only for the tokens of its own rank, PAD for
 * all others; [VBM] Symbol Map says DCP multiplies the block size of
 * attention groups; [BT] Grenzen und Fehler falls back to world size 1.  The
 * formula itself is cut off with the listing.  READING: a table entry names a
 * virtual block of block_size * W tokens; its tokens are dealt to the ranks
 * in interleave chunks of I tokens, round robin, so position p belongs to
 * rank (p / I) % W; on its rank, token p is element
 * ((p % (T*W)) / (I*W)) * I + p % I of the rank's physical block b, whose
 * slot is b * T + that element (T = block_size, T % I == 0).  With W = 1 this
 * is orc_slot_mapping_paged.                                                */
static int64_t paged_cp_slot(int64_t p, const int32_t* row, int32_t stride, int32_t T,
                             int64_t B, int32_t W, int32_t rank, int32_t I, int32_t* err)
{
    if (p < 0) { *err |= ORC_BAD_POSITION; return ORC_PAD_SLOT; }
    int64_t virt = (int64_t)T * W;
    if ((p / I) % W != rank) return ORC_PAD_SLOT;
    int64_t lb = p / virt;
    if (lb >= stride) return ORC_PAD_SLOT;
    int64_t b = row[lb];
    if (b == ORC_NULL_BLOCK) return ORC_PAD_SLOT;
    if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }
    int64_t v = p % virt;
    return b * T + (v / ((int64_t)I * W)) * I + p % I;
}

int orc_slot_mapping_paged_cp(const int32_t* qsl, const int64_t* positions,
                              const int32_t* block_table, int32_t table_stride,
                              int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                              int32_t block_size, int64_t num_blocks, int32_t cp_world_size,
                              int32_t cp_rank, int32_t cp_interleave, int64_t* slot_mapping,
                              int32_t* err)
{
    if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
        num_blocks < 1 || table_stride < 0 || cp_world_size < 1 || cp_rank < 0 ||
        cp_rank >= cp_world_size || cp_interleave < 1)
        return ORC_EINVAL;
    if (block_size % cp_interleave != 0) return ORC_EUNSUPPORTED;
    int32_t e = 0;
    for (int32_t t = 0; t < max_num_tokens; ++t) slot_mapping[t] = ORC_PAD_SLOT;
    e |= qsl_errors(qsl, num_reqs, num_tokens);
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t lo = qsl[r] < 0 ? 0 : qsl[r];
        int32_t hi = qsl[r + 1] > num_tokens ? num_tokens : qsl[r + 1];
        const int32_t* row = block_table + (int64_t)r * table_stride;
        for (int32_t t = lo; t < hi; ++t)
            slot_mapping[t] = paged_cp_slot(positions[t], row, table_stride, block_size,
                                            num_blocks, cp_world_size, cp_rank, cp_interleave, &e);
    }
    *err |= e;
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* Range descriptors: [RNG] The Innovation,
 *   physical_block = range_start + (position // block_size - range_cum),
 * where range_cum is the number of logical blocks the request's earlier
 * ranges cover (READING: ranges are listed in logical order, so range_cum of
 * range i is the sum of the lengths of ranges 0..i-1).  Positions outside
 * every range get the pad id.  READING: a descriptor row with more than
 * range_stride entries, or a negative count, is malformed (BAD_RANGE, every
 * token of the request PAD); a range of length <= 0 is malformed (BAD_RANGE)
 * and covers no logical block.                                              */
static int32_t range_row_errors(const int32_t* rlen, int32_t nr, int32_t range_stride)
{
    if (nr < 0 || nr > range_stride) return ORC_BAD_RANGE;
    for (int32_t i = 0; i < nr; ++i)
        if (rlen[i] <= 0) return ORC_BAD_RANGE;
    return 0;
}

static int64_t range_slot(int64_t p, const int32_t* rstart, const int32_t* rlen, int32_t nr,
                          int32_t range_stride, int32_t T, int64_t B, int32_t* err)
{
    if (p < 0) { *err |= ORC_BAD_POSITION; return ORC_PAD_SLOT; }
    if (nr < 0 || nr > range_stride) return ORC_PAD_SLOT;
    int64_t lb = p / T;
    int64_t range_cum = 0;
    for (int32_t i = 0; i < nr; ++i) {
        int64_t len = rlen[i] > 0 ? rlen[i] : 0;
        if (range_cum <= lb && lb < range_cum + len) {
            int64_t b = (int64_t)rstart[i] + (lb - range_cum);
            if (b == ORC_NULL_BLOCK) return ORC_PAD_SLOT;
            if (b < 0 || b >= B) { *err |= ORC_BAD_BLOCK; return ORC_PAD_SLOT; }
            return b * T + p % T;
        }
        range_cum += len;
    }
    return ORC_PAD_SLOT;
}

int orc_slot_mapping_range(const int32_t* qsl, const int64_t* positions,
                           const int32_t* range_start, const int32_t* range_len,
                           const int32_t* num_ranges, int32_t range_stride,
                           int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                           int32_t block_size, int64_t num_blocks,
                           int64_t* slot_mapping, int32_t* err)
{
    if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
        num_blocks < 1 || range_stride < 0)
        return ORC_EINVAL;
    /* [RNG] The Fork Implementation: range tables are capped at 256 ranges
     * per request and larger ones are rejected (fail closed). */
    if (range_stride > ORC_RANGE_CAP) return ORC_EUNSUPPORTED;
    int32_t e = 0;
    for (int32_t t = 0; t < max_num_tokens; ++t) slot_mapping[t] = ORC_PAD_SLOT;
    e |= qsl_errors(qsl, num_reqs, num_tokens);
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int32_t* rs = range_start + (int64_t)r * range_stride;
        const int32_t* rl = range_len + (int64_t)r * range_stride;
        e |= range_row_errors(rl, num_ranges[r], range_stride);
        int32_t lo = qsl[r] < 0 ? 0 : qsl[r];
        int32_t hi = qsl[r + 1] > num_tokens ? num_tokens : qsl[r + 1];
        for (int32_t t = lo; t < hi; ++t)
            slot_mapping[t] = range_slot(positions[t], rs, rl, num_ranges[r], range_stride,
                                         block_size, num_blocks, &e);
    }
    *err |= e;
    return ORC_OK;
}

/* Expansion of range descriptors into a block-table row: logical block
 * range_cum + j of range i is physical block range_start + j.  This is what
 * the range backend has to materialise for table-reading consumers ([RNG]
 * Status: the per-step block-table copy is redundant once the ranges hold the
 * layout; a range-expansion kernel can fill the table directly), and it is
 * the table for which [RNG] Benchmark Methodology states that both slot
 * mapping strategies agree.  Entries the ranges do not reach stay the null
 * block.  READING: a malformed row (count outside [0, range_stride]) is all
 * null with BAD_RANGE; a range of length <= 0 covers nothing and sets
 * BAD_RANGE; ranges reaching past table_stride are cut there with
 * OUT_OF_SPACE; an entry outside the int32 range is null with BAD_BLOCK.   */
int orc_table_from_ranges(const int32_t* range_start, const int32_t* range_len,
                          const int32_t* num_ranges, int32_t range_stride, int32_t num_reqs,
                          int32_t table_stride, int32_t* table, int32_t* err)
{
    if (num_reqs < 0 || range_stride < 0 || table_stride < 0) return ORC_EINVAL;
    if (range_stride > ORC_RANGE_CAP) return ORC_EUNSUPPORTED;
    int32_t e = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t* row = table + (int64_t)r * table_stride;
        for (int32_t c = 0; c < table_stride; ++c) row[c] = ORC_NULL_BLOCK;
        int32_t nr = num_ranges[r];
        if (nr < 0 || nr > range_stride) { e |= ORC_BAD_RANGE; continue; }
        int64_t range_cum = 0;
        for (int32_t i = 0; i < nr; ++i) {
            int64_t len = range_len[(int64_t)r * range_stride + i];
            if (len <= 0) { e |= ORC_BAD_RANGE; continue; }
            for (int64_t j = 0; j < len; ++j) {
                int64_t lb = range_cum + j;
                int64_t b = (int64_t)range_start[(int64_t)r * range_stride + i] + j;
                if (lb >= table_stride) { e |= ORC_OUT_OF_SPACE; break; }
                if (b < 0 || b > INT32_MAX) { e |= ORC_BAD_BLOCK; continue; }
                row[lb] = (int32_t)b;
            }
            range_cum += len;
        }
    }
    *err |= e;
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* KV write (the attention backend's cache write by slot; [BT] Verantwortung:
 * the kernels read and write KV directly through slot_mapping; [VBM] Deep
 * Dive 8: each token's KV is stored at exactly its slot).
 * READING: K and V are separate bf16 caches [L, B, T, H, D]; the new rows are
 * [L, N, H, D]; token t's row of layer l goes to cache row
 * n(l, slot / T, slot % T).  Negative slots (PAD) are skipped silently; a
 * slot inside the null block is skipped with NULL_WRITE (added guard: block 0
 * is never written); a slot at or past B * T is skipped with BAD_SLOT.
 * Returns the destination row, or -1 when the token is skipped.            */
static int64_t write_dest_row(int64_t s, int64_t layer, int64_t B, int32_t T, int32_t* err)
{
    if (s < 0) return -1;
    int64_t b = s / T;
    if (b == ORC_NULL_BLOCK) { *err |= ORC_NULL_WRITE; return -1; }
    if (b >= B) { *err |= ORC_BAD_SLOT; return -1; }
    return orc_coord(layer, b, s % T, B, T);
}

int orc_cache_write(const uint16_t* key, const uint16_t* value, uint16_t* k_cache,
                    uint16_t* v_cache, const int64_t* slot_mapping, int32_t num_tokens,
                    int32_t num_layers, int64_t num_blocks, int32_t block_size,
                    int32_t num_kv_heads, int32_t head_dim, int32_t* err)
{
    if (num_tokens < 0 || num_layers < 0 || num_blocks < 1 || block_size <= 0 ||
        num_kv_heads <= 0 || head_dim <= 0)
        return ORC_EINVAL;
    int64_t E = (int64_t)num_kv_heads * head_dim;
    int32_t e = 0;
    for (int32_t t = 0; t < num_tokens; ++t) {
        for (int32_t l = 0; l < num_layers; ++l) {
            int64_t n = write_dest_row(slot_mapping[t], l, num_blocks, block_size, &e);
            if (n < 0) continue;
            int64_t src = ((int64_t)l * num_tokens + t) * E;
            for (int64_t x = 0; x < E; ++x) {
                k_cache[n * E + x] = key[src + x];
                v_cache[n * E + x] = value[src + x];
            }
        }
    }
    *err |= e;
    return ORC_OK;
}

/* Destination rows of the write, one per (layer, token), -1 where skipped:
 * lets a test check sampled rows of a cache too large to copy to the host. */
int orc_write_rows(const int64_t* slot_mapping, int32_t num_tokens, int32_t num_layers,
                   int64_t num_blocks, int32_t block_size, int64_t* dest_rows, int32_t* err)
{
    if (num_tokens < 0 || num_layers < 0 || num_blocks < 1 || block_size <= 0) return ORC_EINVAL;
    int32_t e = 0;
    for (int32_t l = 0; l < num_layers; ++l)
        for (int32_t t = 0; t < num_tokens; ++t)
            dest_rows[(int64_t)l * num_tokens + t] =
                write_dest_row(slot_mapping[t], l, num_blocks, block_size, &e);
    *err |= e;
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* Read-path gather ([RNG] Block-table lookup per position: the attention
 * kernels resolve block_table[r][c] again on the read path; [VBM] Deep Dive 7:
 * the kernel reads block_table[row][col] to find a KV block).
 * READING: request r's positions [start_r, end_r) are packed into the output
 * in request order; output row o_r + (p - start_r) with o_r the sum of the
 * earlier requests' lengths.  A null table entry yields a zero row (the
 * "dummy zeroing" test of [RNG] Correctness Verification); an entry outside
 * [1, B) yields a zero row and BAD_BLOCK; a position whose logical block lies
 * past the table row yields a zero row and BAD_POSITION; a request with
 * start < 0 or end < start contributes no rows and sets BAD_POSITION; rows
 * at or past out_rows are not written and set OUT_OF_SPACE.
 * Source row of output row o: >= 0 cache row, -1 zero row, -2 not written. */
int orc_gather_rows(int32_t layer, int64_t num_blocks, int32_t block_size,
                    const int32_t* block_table, int32_t table_stride,
                    const int32_t* gather_start, const int32_t* gather_end, int32_t num_reqs,
                    int64_t out_rows, int64_t* src_rows, int32_t* err)
{
    if (layer < 0 || num_blocks < 1 || block_size <= 0 || table_stride < 0 || num_reqs < 0 ||
        out_rows < 0)
        return ORC_EINVAL;
    int32_t e = 0;
    for (int64_t o = 0; o < out_rows; ++o) src_rows[o] = -2;
    int64_t o_r = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t s0 = gather_start[r], s1 = gather_end[r];
        if (s0 < 0 || s1 < s0) { e |= ORC_BAD_POSITION; continue; }
        const int32_t* row = block_table + (int64_t)r * table_stride;
        for (int64_t p = s0; p < s1; ++p) {
            int64_t o = o_r + (p - s0);
            if (o >= out_rows) { e |= ORC_OUT_OF_SPACE; continue; }
            int64_t lb = p / block_size;
            if (lb >= table_stride) { e |= ORC_BAD_POSITION; src_rows[o] = -1; continue; }
            int64_t b = row[lb];
            if (b == ORC_NULL_BLOCK) { src_rows[o] = -1; continue; }
            if (b < 0 || b >= num_blocks) { e |= ORC_BAD_BLOCK; src_rows[o] = -1; continue; }
            src_rows[o] = orc_coord(layer, b, p % block_size, num_blocks, block_size);
        }
        o_r += s1 - s0;
    }
    *err |= e;
    return ORC_OK;
}

int orc_cache_gather(const uint16_t* k_cache, const uint16_t* v_cache, int32_t layer,
                     int32_t num_layers, int64_t num_blocks, int32_t block_size,
                     int32_t num_kv_heads, int32_t head_dim, const int32_t* block_table,
                     int32_t table_stride, const int32_t* gather_start,
                     const int32_t* gather_end, int32_t num_reqs, uint16_t* k_out,
                     uint16_t* v_out, int64_t out_rows, int64_t* scratch_src_rows,
                     int32_t* err)
{
    if (num_layers <= 0 || layer >= num_layers || num_kv_heads <= 0 || head_dim <= 0)
        return ORC_EINVAL;
    int rc = orc_gather_rows(layer, num_blocks, block_size, block_table, table_stride,
                             gather_start, gather_end, num_reqs, out_rows, scratch_src_rows, err);
    if (rc != ORC_OK) return rc;
    int64_t E = (int64_t)num_kv_heads * head_dim;
    for (int64_t o = 0; o < out_rows; ++o) {
        int64_t n = scratch_src_rows[o];
        if (n == -2) continue;
        for (int64_t x = 0; x < E; ++x) {
            k_out[o * E + x] = n >= 0 ? k_cache[n * E + x] : 0;
            v_out[o * E + x] = n >= 0 ? v_cache[n * E + x] : 0;
        }
    }
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* Range-addressed read path ([RNG] The Direction, milestone M7: range
 * arithmetic instead of block-table resolution in the read-path kernels;
 * Status: profile the gather against sequential range access).  Same output
 * as the table gather of section above, with the block of position p found
 * from the request's ranges: physical_block = range_start +
 * (p // block_size - range_cum) ([RNG] The Innovation).
 * READING: a position no range covers is a zero row (as a null table entry);
 * a malformed descriptor row gives zero rows for all its positions; BAD_RANGE
 * is set for every malformed row r < num_reqs; a resolved block 0 is a zero
 * row; a block outside [0, B) is a zero row with BAD_BLOCK; spans and
 * out_rows as in the table gather.  Source rows as orc_gather_rows.        */
int orc_gather_rows_range(int32_t layer, int64_t num_blocks, int32_t block_size,
                          const int32_t* range_start, const int32_t* range_len,
                          const int32_t* num_ranges, int32_t range_stride,
                          const int32_t* gather_start, const int32_t* gather_end, int32_t num_reqs,
                          int64_t out_rows, int64_t* src_rows, int32_t* err)
{
    if (layer < 0 || num_blocks < 1 || block_size <= 0 || range_stride < 0 || num_reqs < 0 ||
        out_rows < 0)
        return ORC_EINVAL;
    if (range_stride > ORC_RANGE_CAP) return ORC_EUNSUPPORTED;
    int32_t e = 0;
    for (int64_t o = 0; o < out_rows; ++o) src_rows[o] = -2;
    for (int32_t r = 0; r < num_reqs; ++r)
        e |= range_row_errors(range_len + (int64_t)r * range_stride, num_ranges[r], range_stride);
    int64_t o_r = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t s0 = gather_start[r], s1 = gather_end[r];
        if (s0 < 0 || s1 < s0) { e |= ORC_BAD_POSITION; continue; }
        const int32_t* rs = range_start + (int64_t)r * range_stride;
        const int32_t* rl = range_len + (int64_t)r * range_stride;
        int32_t nr = num_ranges[r];
        for (int64_t p = s0; p < s1; ++p) {
            int64_t o = o_r + (p - s0);
            if (o >= out_rows) { e |= ORC_OUT_OF_SPACE; continue; }
            src_rows[o] = -1;
            if (nr < 0 || nr > range_stride) continue;
            int64_t lb = p / block_size;
            int64_t range_cum = 0;
            for (int32_t i = 0; i < nr; ++i) {
                int64_t len = rl[i] > 0 ? rl[i] : 0;
                if (range_cum <= lb && lb < range_cum + len) {
                    int64_t b = (int64_t)rs[i] + (lb - range_cum);
                    if (b < 0 || b >= num_blocks) e |= ORC_BAD_BLOCK;
                    else if (b != ORC_NULL_BLOCK)
                        src_rows[o] = orc_coord(layer, b, p % block_size, num_blocks, block_size);
                    break;
                }
                range_cum += len;
            }
        }
        o_r += s1 - s0;
    }
    *err |= e;
    return ORC_OK;
}

/* Batched block copy for copy-on-write ([VBM] Deep Dive 3: when a writer
 * diverges from a shared block the manager allocates a fresh block and
 * queues KVCacheBlockCopy(src, dst) so that the worker copies the KV data
 * before the writer overwrites it).  READING: every layer's K and V block
 * dst becomes a copy of block src, pairs in order; src outside [1, B) is
 * skipped with BAD_BLOCK (block 0 holds no data); dst == 0 is skipped with
 * NULL_WRITE; dst outside [0, B) is skipped with BAD_BLOCK.                */
int orc_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, int32_t num_layers, int64_t num_blocks,
                    int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                    const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                    int32_t* err)
{
    if (num_layers < 0 || num_blocks < 1 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || num_pairs < 0)
        return ORC_EINVAL;
    int64_t E = (int64_t)num_kv_heads * head_dim;
    int32_t e = 0;
    if (num_layers == 0) return ORC_OK;  /* nothing to read, write or check */
    for (int32_t i = 0; i < num_pairs; ++i) {
        int64_t sb = src_blocks[i], db = dst_blocks[i];
        if (sb <= ORC_NULL_BLOCK || sb >= num_blocks) { e |= ORC_BAD_BLOCK; continue; }
        if (db == ORC_NULL_BLOCK) { e |= ORC_NULL_WRITE; continue; }
        if (db < 0 || db >= num_blocks) { e |= ORC_BAD_BLOCK; continue; }
        for (int32_t l = 0; l < num_layers; ++l)
            for (int32_t t = 0; t < block_size; ++t) {
                int64_t s = orc_coord(l, sb, t, num_blocks, block_size) * E;
                int64_t d = orc_coord(l, db, t, num_blocks, block_size) * E;
                for (int64_t x = 0; x < E; ++x) {
                    k_cache[d + x] = k_cache[s + x];
                    v_cache[d + x] = v_cache[s + x];
                }
            }
    }
    *err |= e;
    return ORC_OK;
}

/* --------------------------------------------------------------------- */
/* Kernel-block expansion ([BT] Entwurfsmotivation: map_to_kernel_blocks
 * unfolds one manager block into blocks_per_kv_block kernel blocks;
 * Grenzen und Fehler: block_size % kernel_block_size != 0 is rejected).
 * Manager block m covers kernel blocks m*k .. m*k+k-1, k = mbs / kbs.
 * READING: the null manager block expands to k null kernel blocks (so that
 * no kernel block of block 0 becomes writable); columns past mgr_stride * k
 * are null; an entry < 0, or one whose last kernel block overflows int32,
 * expands to null blocks and sets BAD_BLOCK.                                */
int orc_expand_kernel_blocks(const int32_t* mgr_table, int32_t num_reqs, int32_t mgr_stride,
                             int32_t mgr_block_size, int32_t kernel_block_size,
                             int32_t* kernel_table, int32_t kernel_stride, int32_t* err)
{
    if (num_reqs < 0 || mgr_stride < 0 || mgr_block_size <= 0 || kernel_block_size <= 0 ||
        kernel_stride < 0)
        return ORC_EINVAL;
    if (mgr_block_size % kernel_block_size != 0) return ORC_EUNSUPPORTED;
    int64_t k = mgr_block_size / kernel_block_size;
    if ((int64_t)kernel_stride < (int64_t)mgr_stride * k) return ORC_EINVAL;
    int32_t e = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int32_t* in = mgr_table + (int64_t)r * mgr_stride;
        int32_t* out = kernel_table + (int64_t)r * kernel_stride;
        for (int32_t c = 0; c < kernel_stride; ++c) out[c] = ORC_NULL_BLOCK;
        for (int32_t c = 0; c < mgr_stride; ++c) {
            int64_t m = in[c];
            if (m == ORC_NULL_BLOCK) continue;
            if (m < 0 || m * k + (k - 1) > INT32_MAX) { e |= ORC_BAD_BLOCK; continue; }
            for (int64_t j = 0; j < k; ++j) out[c * k + j] = (int32_t)(m * k + j);
        }
    }
    *err |= e;
    return ORC_OK;
}
