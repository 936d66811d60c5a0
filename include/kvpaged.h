/*
 * kvpaged.h -- C ABI of the GB300 paged KV-cache hot path (libkvpaged.so).
 *
 * Thirteen calls, each one kernel launch on the caller's stream:
 *   kv_slot_mapping_paged    token -> cache slot through a block table
 *   kv_slot_mapping_paged_cp the same, for one rank of context parallelism
 *   kv_slot_mapping_range    token -> cache slot through contiguous ranges
 *   kv_cache_write           scatter new K/V rows into the paged caches
 *   kv_slot_mapping_paged_write  slot mapping and KV write in one launch
 *   kv_slot_mapping_range_write  the same through contiguous ranges
 *   kv_cache_gather          gather a request's K/V through its block table
 *   kv_cache_gather_bulk     the same gather, moved by bulk (TMA) copies
 *   kv_expand_kernel_blocks  manager-size block table -> kernel-size blocks
 *   kv_table_from_ranges     range descriptors -> block table
 *   kv_cache_gather_range    the gather, with blocks found from ranges
 *   kv_copy_blocks           copy-on-write copy of whole blocks
 *   kv_copy_blocks_bulk      the same copies, moved by bulk (TMA) copies
 *
 * Sources (page title, section):
 *   [BT]  "Blocktabelle" (vLLM v0.25.1 walkthrough)
 *   [VBM] "vLLM Block Table Management" (PagedAttention, vLLM V1 block stack)
 *   [RNG] "Range-addressed KV cache blocks for the vLLM serving engine"
 *
 * Common rules for every call
 * ---------------------------
 * Memory.  Every array argument is a device pointer owned by the caller
 *   (for example a torch CUDA tensor).  The library allocates nothing, keeps
 *   no state between calls and never synchronises: each call validates its
 *   host-visible arguments, enqueues one kernel on `stream` and returns.
 *   Kernels are launched with programmatic dependent launch: one may be
 *   scheduled while the previous kernel on the stream is finishing, but it
 *   waits for that kernel to complete before its first memory access, so the
 *   results are those of plain stream order (also inside CUDA graphs).
 *   A pointer may be NULL only where the call reads nothing through it (for
 *   example `positions` when num_tokens == 0).
 * Layouts.  All arrays are dense, row-major, without padding between rows
 *   other than the stated strides.  Block tables are int32
 *   [rows, table_stride]: row r is request r, column j the physical block of
 *   logical block j ([BT] Verantwortung).  Slot ids are int64, PAD = -1, and
 *   block 0 is the null block ([VBM] Symbol Map; Deep Dive 8).  K and V are
 *   separate bf16 caches [num_layers, num_blocks, block_size, num_kv_heads,
 *   head_dim]; the row of (layer, block, token) is
 *   n = (layer * num_blocks + block) * block_size + token and holds
 *   num_kv_heads * head_dim contiguous elements ([RNG] The Coordinate
 *   Approach).  All offsets are computed in 64 bits.
 * Status.  The return value is a kv_status: KV_OK, or a negative code when a
 *   host-visible argument is invalid (nothing is launched then), or
 *   KV_ECUDA when the launch itself failed.
 * Error word.  Data errors that only the device can see (a bad block id in a
 *   table, a slot outside the cache, a malformed range row ...) never fault
 *   and never stop the kernel: the affected token or row is skipped or
 *   padded as documented per call, and the matching KV_ERR_* bit is OR-ed
 *   into *d_err (int32, device memory, caller-cleared; d_err may be NULL to
 *   ignore such errors).  Read it after the stream has reached the call.
 * Empty work (zero tokens, zero requests) is valid and returns KV_OK.
 */
#ifndef KVPAGED_H
#define KVPAGED_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* kv_stream_t;

enum kv_status {
    KV_OK = 0,
    KV_EINVAL = -1,        /* null/misaligned pointer, negative or inconsistent size */
    KV_EUNSUPPORTED = -2,  /* a configuration the pages reject (fail closed) */
    KV_ECUDA = -3          /* the kernel launch failed */
};

enum kv_error_bits {
    KV_ERR_BAD_BLOCK = 1,     /* table/range block id outside [0, num_blocks) */
    KV_ERR_BAD_SLOT = 2,      /* write slot at or past num_blocks * block_size */
    KV_ERR_BAD_POSITION = 4,  /* negative position, or gather span invalid / past the table */
    KV_ERR_BAD_RANGE = 8,     /* descriptor count outside [0, range_stride] or a range length <= 0 */
    KV_ERR_NULL_WRITE = 16,   /* write slot inside the null block 0 */
    KV_ERR_BAD_QSL = 32,      /* query_start_loc decreasing, negative, or past num_tokens */
    KV_ERR_OUT_OF_SPACE = 64, /* gather rows exceed out_rows, or ranges exceed a table row */
    KV_ERR_TIMEOUT = 128      /* an asynchronous bulk copy did not complete within the bounded
                                 wait (see "Bounded waits" below) */
};

/*
 * Bounded waits.  Only the two bulk-copy calls (kv_cache_gather_bulk,
 * kv_copy_blocks_bulk) wait on the copy engine, and every such wait gives up
 * after 1 s of GPU time (the global nanosecond timer) or 2^22 tries,
 * whichever comes first; a CTA that gave up waits once more, with the same
 * bound, for each of its own loads still in flight, then ends.  A healthy
 * copy completes in microseconds, so a timeout means the GPU is in trouble.
 * After a call has set KV_ERR_TIMEOUT:
 *   - its outputs are undefined: rows may be missing, partly written, or
 *     written after the kernel ended (a load still in flight when its CTA
 *     gave up), so do not use them;
 *   - treat later results on the same stream as suspect until the stream has
 *     been synchronised and checked for CUDA errors.
 * No wait in this library is unbounded.
 */

#define KV_PAD_SLOT_ID (-1)
#define KV_NULL_BLOCK_ID 0
#define KV_MAX_RANGES_PER_REQ 256   /* [RNG] The Fork Implementation: capped at 256 ranges */
#define KV_MAX_GATHER_REQS 4096     /* requests per kv_cache_gather(_range) call */
/* Largest max_num_tokens of one slot-mapping call (paged, range,
 * context-parallel, fused with the write): 2^31 - 65536, so that token indices
 * of a whole last tile stay in int32.  Larger values: KV_EINVAL. */
#define KV_MAX_TOKENS 2147418112

/*
 * kv_slot_mapping_paged -- per-token cache slot through the block table.
 *
 * Defined by [BT] Datenfluss (the slot-mapping kernel: block_index =
 * pos // block_size, block_number = block_table[req, block_index],
 * slot = block_number * block_size + pos % block_size; the last program pads
 * [num_tokens, max_num_tokens) with PAD) and [VBM] Deep Dive 8.
 *
 *   query_start_loc  int32 [num_reqs + 1]; request r owns tokens
 *                    [qsl[r], qsl[r+1]).  Must be non-decreasing.
 *   positions        int64 [num_tokens]; position of each token in its request.
 *   block_table      int32 [num_reqs, table_stride].
 *   slot_mapping     int64 [max_num_tokens], written entirely.
 *
 * For token t < num_tokens of request r with position p:
 *   p < 0                              -> PAD, KV_ERR_BAD_POSITION
 *   p / block_size >= table_stride     -> PAD
 *   b = block_table[r][p / block_size]:
 *     b == 0 (null block)              -> PAD  ([BT] CUDA-Graph-Padding: null rows are skipped)
 *     b < 0 or b >= num_blocks         -> PAD, KV_ERR_BAD_BLOCK
 *     otherwise                        -> b * block_size + p % block_size
 * Tokens in no request span, and tokens in [num_tokens, max_num_tokens), get
 * PAD.  A decreasing qsl, qsl[0] < 0 or qsl[num_reqs] > num_tokens sets
 * KV_ERR_BAD_QSL (slot values are then unspecified, but every store stays in
 * bounds).
 * Errors: KV_EINVAL for negative sizes, num_tokens > max_num_tokens,
 * max_num_tokens > KV_MAX_TOKENS, block_size <= 0, num_blocks < 1,
 * table_stride < 0, or a null/misaligned pointer that would be read.
 */
int kv_slot_mapping_paged(const int32_t* query_start_loc, const int64_t* positions,
                          const int32_t* block_table, int32_t table_stride, int32_t num_reqs,
                          int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                          int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                          kv_stream_t stream);

/*
 * kv_slot_mapping_paged_cp -- kv_slot_mapping_paged filtered for one rank of
 * decode/prefill context parallelism.
 *
 * [BT] Entwurfsmotivation: with TOTAL_CP_WORLD_SIZE, TOTAL_CP_RANK and
 * CP_KV_CACHE_INTERLEAVE_SIZE the slot-mapping kernel writes real slots only
 * for the tokens of its own rank and PAD for all others; [VBM] Symbol Map:
 * DCP multiplies the block size of attention groups.  The pages stop before
 * the formula; this library's reading (its parity is pinned only at world
 * size 1 and by the partition properties): a table entry b names a virtual
 * block of block_size * W tokens, dealt to the W ranks in chunks of I tokens,
 * round robin; position p belongs to rank (p / I) % W and, on that rank, is
 * element ((p % (block_size*W)) / (I*W)) * I + p % I of physical block b, so
 * its slot is b * block_size + that element.  Each rank thus holds
 * block_size tokens of every virtual block, every token lives on exactly one
 * rank, and W = 1 gives kv_slot_mapping_paged.  All other rules (PAD, null
 * entries, errors, tail) are those of kv_slot_mapping_paged, with the table
 * indexed by p / (block_size * W).
 *
 *   cp_world_size W >= 1, 0 <= cp_rank < W, cp_interleave I >= 1.
 * Errors: as kv_slot_mapping_paged; KV_EINVAL for the ranges above or
 * block_size * W beyond int32; KV_EUNSUPPORTED when I does not divide
 * block_size.
 */
int kv_slot_mapping_paged_cp(const int32_t* query_start_loc, const int64_t* positions,
                             const int32_t* block_table, int32_t table_stride, int32_t num_reqs,
                             int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                             int64_t num_blocks, int32_t cp_world_size, int32_t cp_rank,
                             int32_t cp_interleave, int64_t* slot_mapping, int32_t* d_err,
                             kv_stream_t stream);

/*
 * kv_slot_mapping_range -- per-token cache slot through contiguous ranges.
 *
 * Defined by [RNG] The Innovation: physical_block = range_start +
 * (pos // block_size - range_cum); positions outside every range get the
 * same PAD id as the paged call.  Descriptors are never loaded per position:
 * a lane reuses the range it resolved last, a warp of tokens of one request
 * reads 32 descriptors at once, and on large prefill batches a CTA stages
 * its tile's requests' first 32 descriptors in shared memory once.
 *
 *   range_start, range_len  int32 [num_reqs, range_stride]; request r's ranges
 *                           i < num_ranges[r] in logical order: range i holds
 *                           logical blocks [cum_i, cum_i + range_len[r][i])
 *                           with cum_i = sum of range_len[r][0..i-1], and
 *                           logical block cum_i + j is physical block
 *                           range_start[r][i] + j.
 *   num_ranges              int32 [num_reqs].
 *   other arguments         as kv_slot_mapping_paged.
 *
 * A logical block inside no range -> PAD.  The physical block b it resolves
 * to is checked like a table entry (0 -> PAD; outside [0, num_blocks) -> PAD
 * and KV_ERR_BAD_BLOCK).  A row with num_ranges[r] outside
 * [0, range_stride] sets KV_ERR_BAD_RANGE and all its tokens get PAD; a
 * range with length <= 0 sets KV_ERR_BAD_RANGE and covers no block.  Every
 * row r < num_reqs is validated, with or without tokens.
 * When block_table is the expansion of the ranges (and holds them all), the
 * two calls return identical slot_mapping and error words ([RNG] Benchmark
 * Methodology: both strategies produce identical slot ids).
 * Errors: as kv_slot_mapping_paged; range_stride > KV_MAX_RANGES_PER_REQ is
 * KV_EUNSUPPORTED ([RNG] The Fork Implementation: fail closed above 256).
 */
int kv_slot_mapping_range(const int32_t* query_start_loc, const int64_t* positions,
                          const int32_t* range_start, const int32_t* range_len,
                          const int32_t* num_ranges, int32_t range_stride, int32_t num_reqs,
                          int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                          int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                          kv_stream_t stream);

/*
 * kv_cache_write -- scatter each new token's K and V rows to its slot.
 *
 * The cache write by slot of [BT] Verantwortung (kernels read and write KV
 * directly through slot_mapping) and [VBM] Deep Dive 8; multi-layer
 * addressing by [RNG] The Coordinate Approach.
 *
 *   key, value        bf16 [num_layers, num_tokens, num_kv_heads, head_dim].
 *   k_cache, v_cache  bf16 [num_layers, num_blocks, block_size, num_kv_heads, head_dim].
 *   slot_mapping      int64 [num_tokens].
 *
 * For every token t and layer l with s = slot_mapping[t]:
 *   s < 0 (PAD)                 -> skipped
 *   s / block_size == 0         -> skipped, KV_ERR_NULL_WRITE (block 0 is never written)
 *   s >= num_blocks*block_size  -> skipped, KV_ERR_BAD_SLOT
 *   otherwise cache row (l * num_blocks + s / block_size) * block_size + s % block_size
 *   of k_cache (v_cache) receives key[l][t] (value[l][t]) bit for bit.
 * Two tokens with the same slot race: each 16-byte piece of the row comes
 * from one of them, not necessarily the same one for every piece.
 * Errors: KV_EINVAL for a null or non-16-byte-aligned K/V pointer, negative
 * sizes, num_blocks < 1, block_size <= 0, num_kv_heads <= 0 or head_dim <= 0;
 * KV_EUNSUPPORTED when num_kv_heads * head_dim * 2 is not a multiple of 16.
 */
int kv_cache_write(const void* key, const void* value, void* k_cache, void* v_cache,
                   const int64_t* slot_mapping, int32_t num_tokens, int32_t num_layers,
                   int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                   int32_t head_dim, int32_t* d_err, kv_stream_t stream);

/*
 * kv_slot_mapping_paged_write -- kv_slot_mapping_paged, then kv_cache_write on
 * the slots it produced, in one launch.
 *
 * The slot of [BT] Datenfluss and the write by slot of [BT] Verantwortung
 * and [VBM] Deep Dive 8 with no trip through memory in between: each token's
 * K and V rows go straight to the slot computed for it.
 *
 *   query_start_loc .. num_blocks, slot_mapping  as kv_slot_mapping_paged;
 *                     slot_mapping is still written in full (PAD tail
 *                     included), for the attention kernels that read it.
 *   key, value        bf16 [num_layers, num_tokens, num_kv_heads, head_dim].
 *   k_cache, v_cache  bf16 [num_layers, num_blocks, block_size, num_kv_heads, head_dim].
 *
 * Results (slot_mapping, cache bytes, error bits) are exactly those of the
 * two calls in sequence; since a slot produced here is never in block 0 nor
 * past the pool, the write half adds no error bit of its own.  Tokens given
 * the same slot (a table that repeats a block) race as in kv_cache_write.
 * Errors: the union of the two calls' argument checks.
 */
int kv_slot_mapping_paged_write(const int32_t* query_start_loc, const int64_t* positions,
                                const int32_t* block_table, int32_t table_stride,
                                int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                                int32_t block_size, int64_t num_blocks, const void* key,
                                const void* value, void* k_cache, void* v_cache,
                                int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                                int64_t* slot_mapping, int32_t* d_err, kv_stream_t stream);

/*
 * kv_slot_mapping_range_write -- kv_slot_mapping_range, then kv_cache_write on
 * the slots it produced, in one launch ([RNG] The Innovation for the block,
 * otherwise as kv_slot_mapping_paged_write).
 *
 *   range_start, range_len, num_ranges, range_stride  as kv_slot_mapping_range.
 *   other arguments   as kv_slot_mapping_paged_write.
 *
 * Results are exactly those of kv_slot_mapping_range followed by
 * kv_cache_write, including KV_ERR_BAD_RANGE for every malformed row
 * r < num_reqs.  Errors: as kv_slot_mapping_range and kv_cache_write.
 */
int kv_slot_mapping_range_write(const int32_t* query_start_loc, const int64_t* positions,
                                const int32_t* range_start, const int32_t* range_len,
                                const int32_t* num_ranges, int32_t range_stride,
                                int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                                int32_t block_size, int64_t num_blocks, const void* key,
                                const void* value, void* k_cache, void* v_cache,
                                int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                                int64_t* slot_mapping, int32_t* d_err, kv_stream_t stream);

/*
 * kv_cache_gather -- read each request's K/V through its block table into
 * contiguous buffers (the read-path resolution of [RNG] Block-table lookup
 * per position; [VBM] Deep Dive 7: the kernel reads block_table[row][col]).
 *
 *   k_cache, v_cache  bf16 caches as in kv_cache_write; `layer` selects the layer.
 *   block_table       int32 [num_reqs, table_stride].
 *   gather_start/end  int32 [num_reqs]; request r asks for positions [start, end).
 *   k_out, v_out      bf16 [out_rows, num_kv_heads, head_dim].
 *
 * Requests are packed in order: position p of request r goes to output row
 * o_r + (p - start_r), o_r = sum of the earlier requests' lengths.  Each row:
 *   table entry b = block_table[r][p / block_size]:
 *     p / block_size >= table_stride -> zero row, KV_ERR_BAD_POSITION
 *     b == 0 (null block)            -> zero row (padding and recycled blocks)
 *     b < 0 or b >= num_blocks       -> zero row, KV_ERR_BAD_BLOCK
 *     otherwise                      -> cache row (layer, b, p % block_size)
 * A request with start < 0 or end < start contributes no rows and sets
 * KV_ERR_BAD_POSITION.  Rows at or past out_rows are not written and set
 * KV_ERR_OUT_OF_SPACE.  Output rows past the total are left untouched.
 * Errors: KV_EINVAL as kv_cache_write, or layer outside [0, num_layers),
 * out_rows < 0; KV_EUNSUPPORTED for a row size not a multiple of 16 bytes or
 * num_reqs > KV_MAX_GATHER_REQS (split the batch).
 */
int kv_cache_gather(const void* k_cache, const void* v_cache, int32_t layer, int32_t num_layers,
                    int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                    int32_t head_dim, const int32_t* block_table, int32_t table_stride,
                    const int32_t* gather_start, const int32_t* gather_end, int32_t num_reqs,
                    void* k_out, void* v_out, int64_t out_rows, int32_t* d_err,
                    kv_stream_t stream);

/*
 * kv_cache_gather_bulk -- kv_cache_gather done by the bulk-copy engine.
 *
 * Same arguments, output, packing, zero-row rules and error bits as
 * kv_cache_gather.  The rows of one request inside one cache block are moved
 * as one asynchronous bulk copy (global -> shared -> global, cp.async.bulk,
 * at most 32 KiB per copy) issued by a single thread per CTA, two one-warp
 * CTAs per SM: the whole-block gather with TMA bulk copies.  It reaches the
 * same bandwidth as kv_cache_gather while occupying 64 threads per SM, which
 * leaves the SMs to concurrent kernels.  Every wait for a copy is bounded
 * (see "Bounded waits"): if one ever ran out, KV_ERR_TIMEOUT is set and the
 * call's outputs are undefined.
 * Errors: as kv_cache_gather; KV_EUNSUPPORTED for a row of more than 32 KiB
 * (num_kv_heads * head_dim * 2 > 32768) or num_reqs > 2048.
 */
int kv_cache_gather_bulk(const void* k_cache, const void* v_cache, int32_t layer,
                         int32_t num_layers, int64_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, const int32_t* block_table,
                         int32_t table_stride, const int32_t* gather_start,
                         const int32_t* gather_end, int32_t num_reqs, void* k_out, void* v_out,
                         int64_t out_rows, int32_t* d_err, kv_stream_t stream);

/*
 * kv_expand_kernel_blocks -- unfold manager blocks into kernel blocks.
 *
 * [BT] Entwurfsmotivation (map_to_kernel_blocks unfolds one manager block
 * into blocks_per_kv_block kernel blocks, e.g. manager 32 over kernel 16)
 * and Grenzen und Fehler (a kernel block size that does not divide the
 * manager block size is rejected).  With k = mgr_block_size /
 * kernel_block_size, manager entry m at column c becomes kernel entries
 * m*k + j at columns c*k + j, j < k; the null block 0 stays null (k zeros).
 * Columns at or past mgr_stride * k are set to 0.  An entry m < 0, or one
 * whose last kernel block would overflow int32, gives k null entries and
 * KV_ERR_BAD_BLOCK.
 *
 *   mgr_table     int32 [num_reqs, mgr_stride].
 *   kernel_table  int32 [num_reqs, kernel_stride], written entirely.
 * Errors: KV_EUNSUPPORTED when mgr_block_size % kernel_block_size != 0;
 * KV_EINVAL for block sizes <= 0, negative sizes, kernel_stride <
 * mgr_stride * k, or null pointers with work to do.
 */
int kv_expand_kernel_blocks(const int32_t* mgr_table, int32_t num_reqs, int32_t mgr_stride,
                            int32_t mgr_block_size, int32_t kernel_block_size,
                            int32_t* kernel_table, int32_t kernel_stride, int32_t* d_err,
                            kv_stream_t stream);

/*
 * kv_table_from_ranges -- materialise a block table from range descriptors.
 *
 * "Range-addressed KV cache blocks ...", Status: in range mode the staged
 * block table is copied to the kernels' table every step although the range
 * tables already hold the layout; a range-expansion kernel fills the table
 * directly.  Row r gets, in logical order, the blocks of request r's ranges:
 * logical block cum_i + j is range_start[r][i] + j (The Innovation).
 *
 *   range_start, range_len, num_ranges, range_stride  as kv_slot_mapping_range.
 *   block_table  int32 [num_reqs, table_stride], written entirely.
 *
 * Columns past the ranges are the null block 0.  A row with num_ranges[r]
 * outside [0, range_stride] is all null with KV_ERR_BAD_RANGE; a range with
 * length <= 0 covers nothing and sets KV_ERR_BAD_RANGE; ranges reaching past
 * table_stride are cut there with KV_ERR_OUT_OF_SPACE; an entry outside the
 * int32 range is null with KV_ERR_BAD_BLOCK.  kv_slot_mapping_paged on the
 * result equals kv_slot_mapping_range on the descriptors whenever no range is
 * cut.
 * Errors: KV_EINVAL for negative sizes or null/misaligned pointers with work
 * to do; KV_EUNSUPPORTED for range_stride > KV_MAX_RANGES_PER_REQ.
 */
int kv_table_from_ranges(const int32_t* range_start, const int32_t* range_len,
                         const int32_t* num_ranges, int32_t range_stride, int32_t num_reqs,
                         int32_t* block_table, int32_t table_stride, int32_t* d_err,
                         kv_stream_t stream);

/*
 * kv_cache_gather_range -- kv_cache_gather with the blocks found from range
 * descriptors instead of a block table (range arithmetic on the read path:
 * "Range-addressed KV cache blocks ...", The Direction, milestone M7, and the
 * planned comparison of the table gather against sequential range access in
 * Status).
 *
 * Arguments as kv_cache_gather, with (range_start, range_len, num_ranges,
 * range_stride) as in kv_slot_mapping_range in place of the table.  Output
 * rows, packing, spans, out_rows and the zero-row rules are those of
 * kv_cache_gather, where "table entry" reads "the block range arithmetic
 * gives": a logical block no range covers is a zero row (no error, like a
 * null entry); every row r < num_reqs with a malformed descriptor row sets
 * KV_ERR_BAD_RANGE and yields zero rows.  Equal to kv_cache_gather on the
 * table kv_table_from_ranges builds whenever every requested position lies
 * inside that table's stride.
 * Errors: as kv_cache_gather; range_stride > KV_MAX_RANGES_PER_REQ is
 * KV_EUNSUPPORTED.
 */
int kv_cache_gather_range(const void* k_cache, const void* v_cache, int32_t layer,
                          int32_t num_layers, int64_t num_blocks, int32_t block_size,
                          int32_t num_kv_heads, int32_t head_dim, const int32_t* range_start,
                          const int32_t* range_len, const int32_t* num_ranges,
                          int32_t range_stride, const int32_t* gather_start,
                          const int32_t* gather_end, int32_t num_reqs, void* k_out, void* v_out,
                          int64_t out_rows, int32_t* d_err, kv_stream_t stream);

/*
 * kv_copy_blocks -- batched whole-block copy for copy-on-write ("vLLM Block
 * Table Management", Deep Dive 3: KVCacheBlockCopy(src, dst) is queued so the
 * worker copies the KV data of a shared block into a fresh one before the
 * writer overwrites it).
 *
 *   k_cache, v_cache  bf16 [num_layers, num_blocks, block_size, kv_heads, head_dim],
 *                     read and written in place.
 *   src_blocks, dst_blocks  int32 [num_pairs].
 *
 * For every pair i and layer l, block dst_blocks[i] of K and of V becomes a
 * bit copy of block src_blocks[i].  A source outside [1, num_blocks) is
 * skipped with KV_ERR_BAD_BLOCK (block 0 holds no data); a destination 0 is
 * skipped with KV_ERR_NULL_WRITE; a destination outside [0, num_blocks) is
 * skipped with KV_ERR_BAD_BLOCK.  Destinations must be distinct and no
 * destination may be the source of another pair (as for freshly allocated
 * copy targets); otherwise copies race.  num_layers == 0 reads, writes and
 * checks nothing.
 * Errors: KV_EINVAL as kv_cache_write; KV_EUNSUPPORTED for a row size not a
 * multiple of 16 bytes.
 */
int kv_copy_blocks(void* k_cache, void* v_cache, int32_t num_layers, int64_t num_blocks,
                   int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                   const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                   int32_t* d_err, kv_stream_t stream);

/*
 * kv_copy_blocks_bulk -- kv_copy_blocks moved by the bulk-copy (TMA) engine.
 *
 * The same arguments, results, error bits and rules as kv_copy_blocks.  Each
 * K or V block of a (pair, layer) -- or each 32 KiB piece of a larger block --
 * goes global -> shared -> global with cp.async.bulk from one thread per
 * one-warp CTA, two CTAs per SM.  Every wait on the copy engine is bounded
 * (see "Bounded waits"): one that runs out sets KV_ERR_TIMEOUT, the kernel
 * ends normally, and the destination blocks are undefined.
 * Errors: as kv_copy_blocks; KV_ECUDA if the shared-memory size cannot be set.
 */
int kv_copy_blocks_bulk(void* k_cache, void* v_cache, int32_t num_layers, int64_t num_blocks,
                        int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                        const int32_t* src_blocks, const int32_t* dst_blocks,
                        int32_t num_pairs, int32_t* d_err, kv_stream_t stream);

/*
 * kv_diag_bounded_wait -- self-test of the bounded wait the bulk-copy gather
 * relies on.  No page defines it: it exists so the timeout path can be
 * exercised on a real GPU without faulting or hanging it.  One thread waits,
 * for at most spin_limit tries, on a shared-memory barrier that nothing will
 * complete; when the limit runs out it OR-s KV_ERR_TIMEOUT into *d_err and
 * the kernel ends normally, so the context stays usable.
 *   spin_limit  1 .. 2^20 tries.
 *   d_err       int32 device word (required).
 * Errors: KV_EINVAL for a limit out of range or a null/misaligned d_err.
 */
int kv_diag_bounded_wait(int32_t spin_limit, int32_t* d_err, kv_stream_t stream);

/* Human-readable name of a kv_status value (static string). */
const char* kv_status_string(int status);

/* ABI version of this header (bumped on any signature change). */
int kv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVPAGED_H */
