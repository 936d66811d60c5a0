// kv_slot_write.cu -- slot mapping and KV write in one launch.
//
// Sources: "Blocktabelle", Datenfluss (a token's slot from its request's
// block-table row) and Verantwortung (the KV write goes through the slot
// mapping); "Range-addressed KV cache blocks ...", The Innovation (the block
// from the request's range descriptors, PAD outside every range);
// "vLLM Block Table Management", Deep Dive 8 (each token's KV stored at
// exactly its slot).
//
// The result is kv_slot_mapping_paged (or kv_slot_mapping_range) followed by
// kv_cache_write on the slots it produced: the same slot mapping, the same
// cache bytes, the same error bits.  A slot produced here is never in the
// null block nor past the pool, so the write adds no error of its own.
//
// GPU shape.  At a decode step the two separate launches are two dependent
// latency chains (2 KiB moved per token).  Here one warp owns one token: while
// the CTA stages query_start_loc in shared memory, every warp already has its
// position and the first 2 KiB of its layer-0 K and V rows in flight (they do
// not depend on the slot).  The warp then resolves the block -- paged: one
// broadcast table load; range: the request's descriptors 32 at a time, one
// per lane, a warp scan for the range ends and a ballot for the range that
// holds the position -- lane 0 stores the slot, and the warp stores the rows
// of every layer (16-byte vectors, 2 KiB of K and of V per step).
#include "kv_slot_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;          // tokens per CTA
constexpr int kVecPerLane = 4;                 // 16-byte vectors per lane per chunk
constexpr int kChunkVecs = 32 * kVecPerLane;   // 2 KiB per K (and V) chunk
constexpr int kStageMax = 2048;                // query_start_loc entries staged per CTA

struct RowArgs {
  const uint4* key;    // [L, num_tokens, row_vecs]
  const uint4* value;
  uint4* k_cache;      // [L, B, T, row_vecs]
  uint4* v_cache;
  int32_t num_layers;
  int32_t row_vecs;
};

// Block of logical block lb of request r through the block table (kNull
// when the row has no entry there).  The lookup is split in two: prefetch()
// issues the loads of request r's row, resolve() consumes them, so the loads
// can be started before the request is known for sure.  Warp-uniform
// arguments.
struct PagedLookup {
  const int32_t* __restrict__ table;
  int32_t stride;
  static constexpr bool kRows = false;
  static constexpr bool kNeedsBlock = true;  // prefetch() reads the entry of lb
  struct Pre {
    int32_t entry;
  };
  __device__ __forceinline__ Pre prefetch(int r, int64_t lb) const {
    return Pre{lb < stride ? table[(int64_t)r * stride + lb] : kNull};
  }
  __device__ __forceinline__ int64_t resolve(const Pre& pre, int, int64_t) const {
    return pre.entry;
  }
};

// The same through range descriptors: range i covers logical blocks
// [cum_i, cum_i + len_i) from physical block start_i.  The prefetch is the
// row's descriptors 0..31 (one per lane) and its count; the rest of a row
// with more than 32 ranges is read 32 at a time while resolving.  Lengths
// below zero count as zero and a count outside [0, stride] resolves nothing
// (both are reported by the row sweep), as in the range slot map.
struct RangeLookup {
  const int32_t* __restrict__ start;
  const int32_t* __restrict__ len;
  const int32_t* __restrict__ count;
  int32_t stride;
  static constexpr bool kRows = true;
  static constexpr bool kNeedsBlock = false;  // prefetch() reads the row's head
  struct Pre {
    int32_t s, l, nr;
  };
  __device__ __forceinline__ Pre prefetch(int r, int64_t) const {
    const int lane = threadIdx.x & 31;
    Pre pre{0, 0, 0};
    if (lane < stride) {
      pre.s = start[(int64_t)r * stride + lane];
      pre.l = len[(int64_t)r * stride + lane];
    }
    pre.nr = count[r];
    return pre;
  }
  __device__ __forceinline__ int64_t resolve(const Pre& pre, int r, int64_t lb) const {
    const int lane = threadIdx.x & 31;
    const int32_t nr = pre.nr;
    if (nr < 0 || nr > stride) return kNull;
    const int32_t* rs = start + (int64_t)r * stride;
    const int32_t* rl = len + (int64_t)r * stride;
    int32_t s = pre.s, l = pre.l;
    int64_t cum = 0;
    for (int c0 = 0; c0 < nr; c0 += 32) {
      const int i = c0 + lane;
      if (c0 > 0 && i < nr) {
        s = rs[i];
        l = rl[i];
      }
      const int32_t li = i < nr ? max(l, 0) : 0;
      // a 32-bit scan while every length of the chunk is below 2^26 (the sum
      // of 32 of them then fits int32), else 64-bit: half the shuffles, and no
      // spill at 64 registers (ncu, decode batch: 5.49 -> 5.22 us)
      int64_t incl;
      if (__all_sync(kFull, li < (1 << 26)))
        incl = warp_inclusive_scan<int32_t>(li);
      else
        incl = warp_inclusive_scan<int64_t>((int64_t)li);
      const int64_t total = __shfl_sync(kFull, incl, 31);
      if (lb < cum + total) {
        // the first range whose end passes lb holds it (empty ranges hold nothing)
        const int j = __ffs(__ballot_sync(kFull, cum + incl > lb)) - 1;
        const int64_t end_j = cum + __shfl_sync(kFull, incl, j);
        const int32_t len_j = __shfl_sync(kFull, li, j);
        return (int64_t)__shfl_sync(kFull, s, j) + (lb - (end_j - len_j));
      }
      cum += total;
    }
    return kNull;
  }
};

// Unit u of token t's rows: layer u / per_layer, vectors from
// (u % per_layer) * kChunkVecs, 4 per lane.
__device__ __forceinline__ void load_unit(const RowArgs& w, const SlotArgs& a, int32_t t, int u,
                                          int per_layer, int lane, uint4 (&kr)[kVecPerLane],
                                          uint4 (&vr)[kVecPerLane]) {
  const int l = u / per_layer;
  const int c0 = (u - l * per_layer) * kChunkVecs;
  const int64_t i = ((int64_t)l * a.num_tokens + t) * w.row_vecs;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = c0 + j * 32 + lane;
    if (v < w.row_vecs) {
      kr[j] = ld_stream(w.key + i + v);
      vr[j] = ld_stream(w.value + i + v);
    }
  }
}

// Store unit u to the cache row of (layer, block b, offset off).
__device__ __forceinline__ void store_unit(const RowArgs& w, const SlotArgs& a, int64_t b,
                                           int64_t off, int u, int per_layer, int lane,
                                           const uint4 (&kr)[kVecPerLane],
                                           const uint4 (&vr)[kVecPerLane]) {
  const int l = u / per_layer;
  const int c0 = (u - l * per_layer) * kChunkVecs;
  const int64_t n = (((int64_t)l * a.num_blocks + b) * a.bs.size + off) * w.row_vecs;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const int v = c0 + j * 32 + lane;
    if (v < w.row_vecs) {
      st_stream(w.k_cache + n + v, kr[j]);
      st_stream(w.v_cache + n + v, vr[j]);
    }
  }
}

// At most 64 registers (4 CTAs per SM): the range form would otherwise take
// 78 and run 3 CTAs per SM, measured 1.8 % slower over 32 layers (335.7 vs
// 329.7 us).
template <class Lookup>
__global__ void __launch_bounds__(kThreads, 4)
slot_write_kernel(SlotArgs a, Lookup lk, RowArgs w, bool qsl_in_smem, bool vec4) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int32_t s_qsl[];
  const int lane = threadIdx.x & 31;
  const int32_t t = blockIdx.x * kWarps + (int32_t)(threadIdx.x >> 5);  // warp-uniform
  const bool live = t < a.num_tokens;
  // loads that do not depend on the slot: the position, the first chunk of
  // the token's layer-0 rows
  const int64_t p = live ? a.positions[t] : 0;
  uint4 kr[kVecPerLane], vr[kVecPerLane];
  if (live && w.num_layers > 0) {
    const uint4* ks = w.key + (int64_t)t * w.row_vecs;
    const uint4* vs = w.value + (int64_t)t * w.row_vecs;
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = j * 32 + lane;
      if (v < w.row_vecs) {
        kr[j] = ld_stream(ks + v);
        vr[j] = ld_stream(vs + v);
      }
    }
  }
  // A decode batch gives request t its token t (one token each): request t's
  // row is requested before query_start_loc says whose token t is, and used
  // if the lookup below confirms the guess.  A wrong guess (t inside a longer
  // request) only costs the unused loads.  The range row needs no position
  // and goes out at once; the table entry waits on the position and goes out
  // while query_start_loc is being staged.
  const bool guess = live && t < a.num_reqs;
  int64_t lb = 0, off = 0;
  typename Lookup::Pre g_pre{};
  if constexpr (!Lookup::kNeedsBlock) {
    if (guess) g_pre = lk.prefetch(t, 0);
  }
  uint32_t err = 0;
  // descriptor-row validation, one row per thread grid-wide (range form): the
  // first row is requested now and checked at the end
  RangeRowCheck first_row;
  if constexpr (Lookup::kRows) {
    unsigned r0, step;
    if (grid_first(a.num_reqs, r0, step))
      first_row.load(lk.count, lk.len, (int)r0, lk.stride, vec4);
  }
  const int32_t* q = stage_qsl<2>(a, s_qsl, qsl_in_smem, [&] {  // 2: 64 registers
    if (live && p >= 0) a.bs.divmod(p, lb, off);
    if constexpr (Lookup::kNeedsBlock) {
      if (guess && p >= 0) g_pre = lk.prefetch(t, lb);
    }
  });
  check_qsl(a, q, err);

  int64_t b = kNull, slot = kPad;
  if (live) {
    const int r = request_of_guess(q, a.num_reqs, t);
    if (r >= 0) {
      if (p < 0) {
        err |= KV_ERR_BAD_POSITION;
      } else {
        const typename Lookup::Pre pre = (guess && r == t) ? g_pre : lk.prefetch(r, lb);
        b = lk.resolve(pre, r, lb);
        slot = slot_of(b, off, a.bs.size, a.num_blocks, err);
      }
    }
  }
  if (lane == 0 && t < a.max_num_tokens) a.slot_mapping[t] = slot;

  if (slot >= 0) {  // warp-uniform
    // the token's rows as units (layer, 2 KiB chunk of K and of V); unit 0
    // is already in registers.  (Loading unit u+1 before storing unit u was
    // measured: +1 % on the paged form over 32 layers, but -33 % on the range
    // form at 97 registers per thread, so one unit stays in flight.)
    const int per_layer = (w.row_vecs + kChunkVecs - 1) / kChunkVecs;
    const int units = w.num_layers * per_layer;
    for (int u = 0; u < units; ++u) {
      if (u > 0) load_unit(w, a, t, u, per_layer, lane, kr, vr);
      store_unit(w, a, b, off, u, per_layer, lane, kr, vr);
    }
  }

  if constexpr (Lookup::kRows) {
    unsigned r, step;  // this thread's rows: the first was loaded above
    if (grid_first(a.num_reqs, r, step)) {
      if (first_row.malformed(lk.len, lk.stride)) err |= KV_ERR_BAD_RANGE;
      while (grid_next(a.num_reqs, r, step))
        if (range_row_malformed(lk.count, lk.len, (int)r, lk.stride)) err |= KV_ERR_BAD_RANGE;
    }
  }
  report(a.err, err);
}

// Checks of the write half (the same rules as kv_cache_write).
int check_rows(const void* key, const void* value, void* k_cache, void* v_cache,
               int32_t num_tokens, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
               int32_t* row_vecs) {
  if (num_layers < 0 || num_kv_heads <= 0 || head_dim <= 0) return KV_EINVAL;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return KV_EUNSUPPORTED;
  if ((int64_t)num_layers * num_tokens > 0) {
    if (key == nullptr || value == nullptr || k_cache == nullptr || v_cache == nullptr)
      return KV_EINVAL;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16))
      return KV_EINVAL;
  }
  *row_vecs = (int32_t)(row_bytes / 16);
  return KV_OK;
}

template <class Lookup>
int launch_slot_write(const int32_t* qsl, const int64_t* positions, const Lookup& lk,
                      bool vec4, int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
                      int32_t block_size, int64_t num_blocks, const void* key,
                      const void* value, void* k_cache, void* v_cache, int32_t num_layers,
                      int32_t row_vecs, int64_t* slot_mapping, int32_t* d_err,
                      kv_stream_t stream) {
  if (max_num_tokens == 0 && num_reqs == 0) return KV_OK;
  const int64_t ctas = ((int64_t)max_num_tokens + kWarps - 1) / kWarps;
  const int grid = (int)(ctas > 0 ? ctas : 1);
  const bool staged = num_reqs > 0 && num_reqs + 1 <= kStageMax;
  const size_t smem = staged ? sizeof(int32_t) * (num_reqs + 1) : 0;
  SlotArgs a{qsl, positions, num_reqs, num_tokens, max_num_tokens, BlockDiv::make(block_size),
             num_blocks, slot_mapping, d_err};
  RowArgs w{static_cast<const uint4*>(key), static_cast<const uint4*>(value),
            static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_layers, row_vecs};
  return launch_pdl(slot_write_kernel<Lookup>, grid, kThreads, smem, stream, a, lk, w, staged,
                    vec4);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_slot_mapping_paged_write(
    const int32_t* query_start_loc, const int64_t* positions, const int32_t* block_table,
    int32_t table_stride, int32_t num_reqs, int32_t num_tokens, int32_t max_num_tokens,
    int32_t block_size, int64_t num_blocks, const void* key, const void* value, void* k_cache,
    void* v_cache, int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
    int64_t* slot_mapping, int32_t* d_err, kv_stream_t stream) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  if (table_stride < 0) return KV_EINVAL;
  if (num_reqs > 0 && num_tokens > 0 && table_stride > 0 &&
      (block_table == nullptr || !aligned(block_table, 4)))
    return KV_EINVAL;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  int32_t row_vecs = 0;
  rc = check_rows(key, value, k_cache, v_cache, num_tokens, num_layers, num_kv_heads, head_dim,
                  &row_vecs);
  if (rc != KV_OK) return rc;
  return launch_slot_write(query_start_loc, positions, PagedLookup{block_table, table_stride},
                           false, num_reqs, num_tokens, max_num_tokens, block_size, num_blocks,
                           key, value, k_cache, v_cache, num_layers, row_vecs, slot_mapping,
                           d_err, stream);
}

extern "C" int kv_slot_mapping_range_write(
    const int32_t* query_start_loc, const int64_t* positions, const int32_t* range_start,
    const int32_t* range_len, const int32_t* num_ranges, int32_t range_stride, int32_t num_reqs,
    int32_t num_tokens, int32_t max_num_tokens, int32_t block_size, int64_t num_blocks,
    const void* key, const void* value, void* k_cache, void* v_cache, int32_t num_layers,
    int32_t num_kv_heads, int32_t head_dim, int64_t* slot_mapping, int32_t* d_err,
    kv_stream_t stream) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  rc = check_ranges(range_start, range_len, num_ranges, range_stride, num_reqs);
  if (rc != KV_OK) return rc;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  int32_t row_vecs = 0;
  rc = check_rows(key, value, k_cache, v_cache, num_tokens, num_layers, num_kv_heads, head_dim,
                  &row_vecs);
  if (rc != KV_OK) return rc;
  return launch_slot_write(query_start_loc, positions,
                           RangeLookup{range_start, range_len, num_ranges, range_stride},
                           rows_vec4(range_start, range_len, range_stride), num_reqs,
                           num_tokens, max_num_tokens, block_size, num_blocks, key, value,
                           k_cache, v_cache, num_layers, row_vecs, slot_mapping, d_err, stream);
}
