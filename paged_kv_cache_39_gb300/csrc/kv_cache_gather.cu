// kv_cache_gather.cu -- read each request's K/V rows through its block table
// into contiguous output buffers.
//
// Sources: "Range-addressed KV cache blocks ...", Block-table lookup per
// position (the attention kernels resolve the table again on the read path)
// and Status (the planned gather profile); "vLLM Block Table Management",
// Deep Dive 7 (the kernel reads block_table[row][col] to find a KV block);
// "Range-addressed ...", Correctness Verification ("dummy zeroing": null
// entries read as zero rows).
//
// GPU shape.  Every CTA first turns the requests' span lengths into packed
// output offsets with a block-wide scan in shared memory (a few hundred
// int32 pairs, L2-resident), so no second launch or scratch buffer is
// needed.  The output rows are then walked by warps in a grid-stride loop
// over a persistent grid: a warp takes 4 consecutive output rows, finds the
// request of the first by a binary search of the shared offsets, resolves
// the block of each row from the table (consecutive rows share a table
// entry, an L1 hit) and copies the 2 KiB K and V rows with 16-byte vector
// loads and stores, 4 KiB in flight per warp.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerLane = 4;
constexpr int kChunkVecs = 32 * kVecPerLane;
constexpr int kRowsPerWarp = 4;
// static shared memory of the two vector kernels (the per-warp scan totals);
// it counts against the 48 KiB a launch gets without opting in
constexpr size_t kGatherStaticSmem = sizeof(int64_t) * (kThreads / 32);

struct GatherArgs {
  const uint4* k_cache;
  const uint4* v_cache;
  int64_t layer_base;  // layer * num_blocks
  int64_t num_blocks;
  int32_t block_size, row_vecs;
  const int32_t* table;
  int32_t stride;
  const int32_t* g0;
  const int32_t* g1;
  int32_t num_reqs;
  uint4* k_out;
  uint4* v_out;
  int64_t out_rows;
  int32_t* err;
  cudaStream_t stream;
};

// Copy (or zero) one output row: src_row >= 0 copies that cache row.
__device__ __forceinline__ void move_row(const GatherArgs& a, int64_t src_row, int64_t o,
                                         int lane) {
  uint4* kd = a.k_out + o * a.row_vecs;
  uint4* vd = a.v_out + o * a.row_vecs;
  if (src_row < 0) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = lane; v < a.row_vecs; v += 32) {
      st_stream(kd + v, z);
      st_stream(vd + v, z);
    }
    return;
  }
  const uint4* ks = a.k_cache + src_row * a.row_vecs;
  const uint4* vs = a.v_cache + src_row * a.row_vecs;
  for (int c0 = 0; c0 < a.row_vecs; c0 += kChunkVecs) {
    uint4 kr[kVecPerLane], vr[kVecPerLane];
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = c0 + j * 32 + lane;
      if (v < a.row_vecs) {
        kr[j] = ld_stream(ks + v);
        vr[j] = ld_stream(vs + v);
      }
    }
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = c0 + j * 32 + lane;
      if (v < a.row_vecs) {
        st_stream(kd + v, kr[j]);
        st_stream(vd + v, vr[j]);
      }
    }
  }
}

// Packed output offsets: exclusive scan of the span lengths into s_off
// (int64 [R + 1]) and the span starts into s_start.  Span errors are
// returned by CTA 0 only so they are reported once.
__device__ __forceinline__ int64_t packed_offsets(const GatherArgs& a, int64_t* s_off,
                                                  int32_t* s_start, int64_t* s_warp_sum,
                                                  uint32_t& err) {
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int R = a.num_reqs;
  const int per = (R + kThreads - 1) / kThreads;
  const int r_lo = threadIdx.x * per;
  const int r_hi = min(R, r_lo + per);
  uint32_t span_err = 0;
  int64_t local = 0;
  for (int r = r_lo; r < r_hi; ++r) {
    const int32_t s0 = a.g0[r], s1 = a.g1[r];
    const bool ok = s0 >= 0 && s1 >= s0;
    if (!ok) span_err |= KV_ERR_BAD_POSITION;
    s_start[r] = s0;
    local += ok ? (int64_t)(s1 - s0) : 0;
  }
  const int64_t incl = warp_inclusive_scan<int64_t>(local);
  if (lane == 31) s_warp_sum[wid] = incl;
  __syncthreads();
  int64_t warp_base = 0;
  for (int w = 0; w < wid; ++w) warp_base += s_warp_sum[w];
  int64_t run = warp_base + incl - local;
  for (int r = r_lo; r < r_hi; ++r) {
    s_off[r] = run;
    const int32_t s0 = s_start[r], s1 = a.g1[r];
    run += (s0 >= 0 && s1 >= s0) ? (int64_t)(s1 - s0) : 0;
  }
  if (threadIdx.x == kThreads - 1) s_off[R] = run;
  __syncthreads();
  const int64_t total = s_off[R];
  if (blockIdx.x == 0) {
    err |= span_err;
    if (threadIdx.x == 0 && total > a.out_rows) err |= KV_ERR_OUT_OF_SPACE;
  }
  return total;
}

// Block of logical block lb of request r through the block table.
struct TableResolver {
  const int32_t* table;
  int32_t stride;
  // returns the physical block, 0 for a zero row; sets error bits
  __device__ __forceinline__ int64_t operator()(int r, int64_t lb, uint32_t& err) {
    if (lb >= stride) {
      err |= KV_ERR_BAD_POSITION;
      return kNull;
    }
    return table[(int64_t)r * stride + lb];
  }
};

// Block of logical block lb of request r through its range descriptors.  The
// warp keeps the last range it resolved (request, logical window, start):
// consecutive rows of a request fall in the same range, so a lookup -- one
// coalesced load of up to 32 descriptors, a warp scan and a ballot -- is
// needed only when a warp's rows cross into another range.  lb and r are
// warp-uniform here.
struct RangeResolver {
  const int32_t* rs;
  const int32_t* rl;
  const int32_t* nr;
  int32_t rstride;
  int cr = -1;             // cached request
  int64_t w_lo = 0, w_hi = 0, w_start = 0;  // cached window [w_lo, w_hi) -> w_start
  bool w_null = false;     // the cached window is covered by no range
  __device__ __forceinline__ int64_t operator()(int r, int64_t lb, uint32_t&) {
    if (r == cr && lb >= w_lo && lb < w_hi) return w_null ? kNull : w_start + (lb - w_lo);
    const int lane = threadIdx.x & 31;
    const int n = nr[r];
    cr = r;
    w_null = true;
    w_lo = 0;
    w_hi = INT64_MAX;
    if (n < 0 || n > rstride) return kNull;  // malformed row (flagged by the sweep)
    const int32_t* s_ = rs + (int64_t)r * rstride;
    const int32_t* l_ = rl + (int64_t)r * rstride;
    int64_t cum_base = 0;
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int i = c0 + lane;
      int32_t st = 0, len = 0;
      if (i < n) {
        st = s_[i];
        len = max(l_[i], 0);
      }
      const int64_t incl = warp_inclusive_scan<int64_t>((int64_t)len);
      const int64_t end = cum_base + incl;
      const unsigned hit = __ballot_sync(kFull, i < n && end > lb);
      if (hit != 0u) {
        const int j = __ffs(hit) - 1;
        const int64_t e = __shfl_sync(kFull, end, j);
        const int32_t ln = __shfl_sync(kFull, len, j);
        const int32_t sj = __shfl_sync(kFull, st, j);
        w_lo = e - ln;
        w_hi = e;
        w_start = sj;
        w_null = false;
        return w_start + (lb - w_lo);
      }
      cum_base += __shfl_sync(kFull, incl, 31);
    }
    w_lo = cum_base;  // past every range: zero rows from here on (w_null, w_hi set above)
    return kNull;
  }
};

template <typename Resolver>
__device__ __forceinline__ void gather_rows(const GatherArgs& a, const int64_t* s_off,
                                            const int32_t* s_start, int64_t rows,
                                            Resolver& resolve, uint32_t& err) {
  const int lane = threadIdx.x & 31;
  const int R = a.num_reqs;
  const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  for (int64_t o0 = warp0 * kRowsPerWarp; o0 < rows; o0 += nwarps * kRowsPerWarp) {
    int r = find_span64(s_off, R, o0);
    const int64_t o_end = o0 + kRowsPerWarp < rows ? o0 + kRowsPerWarp : rows;
    for (int64_t o = o0; o < o_end; ++o) {
      while (o >= s_off[r + 1]) ++r;  // skip to the request holding row o
      const int64_t p = (int64_t)s_start[r] + (o - s_off[r]);
      const int64_t lb = p / a.block_size;
      const int64_t b = resolve(r, lb, err);
      int64_t src = -1;
      if (b != kNull) {
        if (b < 0 || b >= a.num_blocks) err |= KV_ERR_BAD_BLOCK;
        else src = (a.layer_base + b) * a.block_size + (p - lb * a.block_size);
      }
      move_row(a, src, o, lane);
    }
  }
}

__global__ void __launch_bounds__(kThreads) cache_gather_kernel(GatherArgs a) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int64_t smem[];
  int64_t* s_off = smem;                                                 // [num_reqs + 1]
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + a.num_reqs + 1);  // [num_reqs]
  __shared__ int64_t s_warp_sum[kGatherStaticSmem / sizeof(int64_t)];
  uint32_t err = 0;
  const int64_t total = packed_offsets(a, s_off, s_start, s_warp_sum, err);
  const int64_t rows = total < a.out_rows ? total : a.out_rows;
  TableResolver res{a.table, a.stride};
  gather_rows(a, s_off, s_start, rows, res, err);
  report(a.err, err);
}

// Range-addressed read path ("Range-addressed KV cache blocks ...", The
// Direction, M7): the same output with no block table at all.
__global__ void __launch_bounds__(kThreads)
cache_gather_range_kernel(GatherArgs a, const int32_t* __restrict__ range_start,
                          const int32_t* __restrict__ range_len,
                          const int32_t* __restrict__ num_ranges, int32_t rstride) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ int64_t smem[];
  int64_t* s_off = smem;
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + a.num_reqs + 1);
  __shared__ int64_t s_warp_sum[kGatherStaticSmem / sizeof(int64_t)];
  uint32_t err = 0;
  // descriptor-row validation, every request, grid-wide
  {
    unsigned r, step;
    if (grid_first(a.num_reqs, r, step)) do {
        if (range_row_malformed(num_ranges, range_len, (int)r, rstride)) err |= KV_ERR_BAD_RANGE;
      } while (grid_next(a.num_reqs, r, step));
  }
  const int64_t total = packed_offsets(a, s_off, s_start, s_warp_sum, err);
  const int64_t rows = total < a.out_rows ? total : a.out_rows;
  RangeResolver res{range_start, range_len, num_ranges, rstride};
  gather_rows(a, s_off, s_start, rows, res, err);
  report(a.err, err);
}

// ---------------------------------------------------------------------------
// Whole-block bulk gather (kv_cache_gather_bulk).  The same output as
// cache_gather_kernel, moved by the bulk-copy engine: a CTA is one warp; lane 0 streams its share of
// "chunks" (the rows of one request inside one cache block, at most 32 KiB of
// K and as much of V) global -> shared -> global with cp.async.bulk.  Each
// chunk is two units (K, V); a unit's load completes on a shared mbarrier,
// its store is one bulk group.  Two stage buffers, one unit loaded ahead, two
// CTAs per SM: 64 KiB of loads in flight per SM with the stores draining
// behind them (the best of the shapes measured: more loads in flight per CTA
// starved the stores, fewer starved the loads).  It reaches the bandwidth of
// the vector kernel (within 1 %) while issuing from 64 threads per SM.
// Null or invalid blocks are written from a
// shared zero buffer.  The other 31 lanes compute the chunk descriptors (one
// table lookup each, 32 at a time) and the packed offsets.

constexpr int kBulkStages = 2;
constexpr int kBulkStageBytes = 32768;
constexpr int kBulkZeroBytes = 4096;
constexpr int kBulkCtasPerSm = 2;
constexpr int kBulkMaxReqs = 2048;
constexpr int kBulkHeader = 128;  // mbarriers

__host__ __device__ constexpr size_t bulk_smem_bytes(int num_reqs) {
  return kBulkHeader + kBulkZeroBytes + (size_t)kBulkStages * kBulkStageBytes +
         sizeof(int64_t) * 2 * (num_reqs + 1) + sizeof(int32_t) * num_reqs;
}

__global__ void __launch_bounds__(32) cache_gather_bulk_kernel(GatherArgs a, int32_t chunk_rows) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char bulk_smem[];
  const int R = a.num_reqs;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bulk_smem);
  unsigned char* zero = bulk_smem + kBulkHeader;
  unsigned char* stage = zero + kBulkZeroBytes;
  int64_t* s_off = reinterpret_cast<int64_t*>(stage + kBulkStages * kBulkStageBytes);  // rows
  int64_t* s_coff = s_off + (R + 1);                                               // chunks
  int32_t* s_start = reinterpret_cast<int32_t*>(s_coff + (R + 1));
  const int lane = threadIdx.x;
  const int64_t CH = chunk_rows;
  const int64_t row_bytes = (int64_t)a.row_vecs * 16;
  uint32_t err = 0;

  // packed row offsets and chunk offsets of every request
  {
    const int per = (R + 31) / 32;
    const int r_lo = lane * per, r_hi = min(R, r_lo + per);
    uint32_t span_err = 0;
    int64_t lrows = 0, lch = 0;
    for (int r = r_lo; r < r_hi; ++r) {
      const int32_t s0 = a.g0[r], s1 = a.g1[r];
      const bool ok = s0 >= 0 && s1 >= s0;
      if (!ok) span_err |= KV_ERR_BAD_POSITION;
      s_start[r] = s0;
      const int64_t n = ok ? (int64_t)(s1 - s0) : 0;
      lrows += n;
      lch += n > 0 ? (int64_t)(s1 - 1) / CH - (int64_t)s0 / CH + 1 : 0;
    }
    const int64_t incl_rows = warp_inclusive_scan<int64_t>(lrows);
    const int64_t incl_ch = warp_inclusive_scan<int64_t>(lch);
    int64_t run_rows = incl_rows - lrows, run_ch = incl_ch - lch;
    for (int r = r_lo; r < r_hi; ++r) {
      s_off[r] = run_rows;
      s_coff[r] = run_ch;
      const int32_t s0 = s_start[r], s1 = a.g1[r];
      const int64_t n = (s0 >= 0 && s1 >= s0) ? (int64_t)(s1 - s0) : 0;
      run_rows += n;
      run_ch += n > 0 ? (int64_t)(s1 - 1) / CH - (int64_t)s0 / CH + 1 : 0;
    }
    if (lane == 31) {
      s_off[R] = run_rows;
      s_coff[R] = run_ch;
    }
    if (blockIdx.x == 0) err |= span_err;
  }
  // zero source for null blocks, visible to the bulk-copy engine
  for (int i = lane; i < kBulkZeroBytes / 16; i += 32)
    reinterpret_cast<uint4*>(zero)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (lane == 0) {
    for (int st = 0; st < kBulkStages; ++st) mbar_init(&bars[st], 1);
    mbar_fence_init();
  }
  __syncwarp();
  const int64_t total_rows = s_off[R], total_ch = s_coff[R];
  if (blockIdx.x == 0 && lane == 0 && total_rows > a.out_rows) err |= KV_ERR_OUT_OF_SPACE;

  // this CTA's contiguous share of the chunks
  const int64_t per_cta = (total_ch + gridDim.x - 1) / gridDim.x;
  const int64_t c0 = (int64_t)blockIdx.x * per_cta;
  const int64_t c1 = c0 + per_cta < total_ch ? c0 + per_cta : total_ch;

  uint32_t phase_bits = 0, armed_bits = 0;
  bool failed = false;
  // the unit loaded last: its store is issued at the next unit
  int64_t p_src = 0, p_dst = 0;
  int32_t p_bytes = 0, p_kv = 0, p_stage = 0;
  bool have_prev = false;
  int64_t unit = 0;

  // finish the previous unit: wait for its load, store it, commit its group
  auto finish_prev = [&]() {
    const uint32_t bit = 1u << p_stage;
    if (p_src >= 0) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&bars[p_stage], (phase_bits >> p_stage) & 1u);
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) {
        failed = true;
        return;
      }
      phase_bits ^= bit;
      armed_bits &= ~bit;
    }
    if (lane == 0) {
      unsigned char* out = reinterpret_cast<unsigned char*>(p_kv ? a.v_out : a.k_out) + p_dst;
      if (p_src >= 0) {
        bulk_s2g(out, stage + (size_t)p_stage * kBulkStageBytes, (uint32_t)p_bytes);
      } else {
        for (int32_t off = 0; off < p_bytes; off += kBulkZeroBytes)
          bulk_s2g(out + off, zero, (uint32_t)min(kBulkZeroBytes, p_bytes - off));
      }
      bulk_commit();
    }
  };

  for (int64_t cb = c0; cb < c1 && !failed; cb += 32) {
    // lane q describes chunk cb + q
    int64_t src_row = -1, dst_row = 0, nrows = 0;
    const int64_t u = cb + lane;
    if (u < c1) {
      const int r = find_span64(s_coff, R, u);
      const int64_t k = u - s_coff[r];
      const int64_t g0 = s_start[r];
      const int64_t g1 = g0 + (s_off[r + 1] - s_off[r]);
      const int64_t P = (g0 / CH + k) * CH;
      const int64_t p0 = P > g0 ? P : g0;
      const int64_t p1 = P + CH < g1 ? P + CH : g1;
      dst_row = s_off[r] + (p0 - g0);
      nrows = p1 - p0;
      if (dst_row >= a.out_rows) nrows = 0;  // past out_rows: not written
      else if (dst_row + nrows > a.out_rows) nrows = a.out_rows - dst_row;
      if (nrows > 0) {
        const int64_t lb = p0 / a.block_size;  // a chunk never crosses a block
        if (lb >= a.stride) {
          err |= KV_ERR_BAD_POSITION;
        } else {
          const int64_t b = a.table[(int64_t)r * a.stride + lb];
          if (b != kNull) {
            if (b < 0 || b >= a.num_blocks) err |= KV_ERR_BAD_BLOCK;
            else src_row = (a.layer_base + b) * a.block_size + (p0 - lb * a.block_size);
          }
        }
      }
    }
    const int nq = (int)(c1 - cb < 32 ? c1 - cb : 32);
    for (int q = 0; q < nq && !failed; ++q) {
      const int64_t q_src = __shfl_sync(kFull, src_row, q);
      const int64_t q_dst = __shfl_sync(kFull, dst_row, q);
      const int64_t q_rows = __shfl_sync(kFull, nrows, q);
      if (q_rows == 0) continue;
      for (int kv = 0; kv < 2 && !failed; ++kv) {
        if (have_prev) finish_prev();
        if (failed) break;
        const int st = (int)(unit % kBulkStages);
        const int32_t bytes = (int32_t)(q_rows * row_bytes);
        if (q_src >= 0) {
          if (lane == 0) {
            // the stage's previous unit was stored one unit ago: its group must
            // have finished reading the stage (all but the latest group)
            if (unit >= kBulkStages) bulk_wait_read<kBulkStages - 1>();
            const unsigned char* src =
                reinterpret_cast<const unsigned char*>(kv ? a.v_cache : a.k_cache) +
                q_src * row_bytes;
            mbar_arrive_expect_tx(&bars[st], (uint32_t)bytes);
            bulk_g2s(stage + (size_t)st * kBulkStageBytes, src, (uint32_t)bytes, &bars[st]);
          }
          armed_bits |= 1u << st;
        }
        p_src = q_src >= 0 ? q_src * row_bytes : -1;
        p_dst = q_dst * row_bytes;
        p_bytes = bytes;
        p_kv = kv;
        p_stage = st;
        have_prev = true;
        ++unit;
      }
    }
  }
  if (have_prev && !failed) finish_prev();
  if (failed) {
    err |= KV_ERR_TIMEOUT;
    // bounded wait for this CTA's loads still in flight before its shared memory goes away
    if (lane == 0)
      for (int st = 0; st < kBulkStages; ++st)
        if ((armed_bits >> st) & 1u) mbar_wait_bounded(&bars[st], (phase_bits >> st) & 1u);
  }
  if (lane == 0) bulk_wait_all();
  report(a.err, err);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

static int gather_checks(const void* k_cache, const void* v_cache, int32_t layer,
                         int32_t num_layers, int64_t num_blocks, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, const int32_t* gather_start,
                         const int32_t* gather_end, int32_t num_reqs, void* k_out, void* v_out,
                         int64_t out_rows, int32_t* d_err) {
  if (num_layers <= 0 || layer < 0 || layer >= num_layers || num_blocks < 1 ||
      block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_reqs < 0 || out_rows < 0)
    return KV_EINVAL;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return KV_EUNSUPPORTED;
  if (num_reqs > KV_MAX_GATHER_REQS) return KV_EUNSUPPORTED;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (num_reqs == 0) return KV_OK;
  if (gather_start == nullptr || gather_end == nullptr || !aligned(gather_start, 4) ||
      !aligned(gather_end, 4))
    return KV_EINVAL;
  if (k_cache == nullptr || v_cache == nullptr || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KV_EINVAL;
  if (out_rows > 0 && (k_out == nullptr || v_out == nullptr || !aligned(k_out, 16) ||
                       !aligned(v_out, 16)))
    return KV_EINVAL;
  return KV_OK;
}

template <typename Kernel, typename... Extra>
static int launch_gather(Kernel kernel, const GatherArgs& a, Extra... extra) {
  const size_t smem = sizeof(int64_t) * (a.num_reqs + 1) + sizeof(int32_t) * a.num_reqs;
  const int64_t rows_per_cta = (kThreads / 32) * kRowsPerWarp;
  const int64_t ctas_needed = (a.out_rows + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = (int64_t)sm_count() * (2048 / kThreads);
  const int grid = (int)(ctas_needed < 1 ? 1 : (ctas_needed < cap ? ctas_needed : cap));
  if (smem + kGatherStaticSmem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return KV_ECUDA;
  return launch_pdl(kernel, grid, kThreads, smem, a.stream, a, extra...);
}

extern "C" int kv_cache_gather(const void* k_cache, const void* v_cache, int32_t layer,
                               int32_t num_layers, int64_t num_blocks, int32_t block_size,
                               int32_t num_kv_heads, int32_t head_dim,
                               const int32_t* block_table, int32_t table_stride,
                               const int32_t* gather_start, const int32_t* gather_end,
                               int32_t num_reqs, void* k_out, void* v_out, int64_t out_rows,
                               int32_t* d_err, kv_stream_t stream) {
  int rc = gather_checks(k_cache, v_cache, layer, num_layers, num_blocks, block_size,
                         num_kv_heads, head_dim, gather_start, gather_end, num_reqs, k_out,
                         v_out, out_rows, d_err);
  if (rc != KV_OK || num_reqs == 0) return rc;
  if (table_stride < 0) return KV_EINVAL;
  if (table_stride > 0 && (block_table == nullptr || !aligned(block_table, 4)))
    return KV_EINVAL;
  GatherArgs a{static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache),
               (int64_t)layer * num_blocks, num_blocks, block_size,
               num_kv_heads * head_dim * 2 / 16, block_table, table_stride, gather_start,
               gather_end, num_reqs, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out),
               out_rows, d_err, stream};
  return launch_gather(cache_gather_kernel, a);
}

extern "C" int kv_cache_gather_bulk(const void* k_cache, const void* v_cache, int32_t layer,
                                    int32_t num_layers, int64_t num_blocks, int32_t block_size,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    const int32_t* block_table, int32_t table_stride,
                                    const int32_t* gather_start, const int32_t* gather_end,
                                    int32_t num_reqs, void* k_out, void* v_out,
                                    int64_t out_rows, int32_t* d_err, kv_stream_t stream) {
  int rc = gather_checks(k_cache, v_cache, layer, num_layers, num_blocks, block_size,
                         num_kv_heads, head_dim, gather_start, gather_end, num_reqs, k_out,
                         v_out, out_rows, d_err);
  if (rc != KV_OK) return rc;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (row_bytes > kBulkStageBytes || num_reqs > kBulkMaxReqs) return KV_EUNSUPPORTED;
  if (num_reqs == 0) return KV_OK;
  if (table_stride < 0) return KV_EINVAL;
  if (table_stride > 0 && (block_table == nullptr || !aligned(block_table, 4)))
    return KV_EINVAL;
  GatherArgs a{static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache),
               (int64_t)layer * num_blocks, num_blocks, block_size,
               num_kv_heads * head_dim * 2 / 16, block_table, table_stride, gather_start,
               gather_end, num_reqs, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out),
               out_rows, d_err, stream};
  // a chunk is the rows of one request inside one block, at most one stage:
  // the largest divisor of block_size whose rows fit 32 KiB
  int32_t chunk_rows = (int32_t)(kBulkStageBytes / row_bytes);
  if (chunk_rows > block_size) chunk_rows = block_size;
  while (block_size % chunk_rows != 0) --chunk_rows;
  const size_t smem = bulk_smem_bytes(num_reqs);
  if (cudaFuncSetAttribute(cache_gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return KV_ECUDA;
  const int grid = sm_count() * kBulkCtasPerSm;
  return launch_pdl(cache_gather_bulk_kernel, grid, 32, smem, stream, a, chunk_rows);
}

extern "C" int kv_cache_gather_range(const void* k_cache, const void* v_cache, int32_t layer,
                                     int32_t num_layers, int64_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                     const int32_t* range_start, const int32_t* range_len,
                                     const int32_t* num_ranges, int32_t range_stride,
                                     const int32_t* gather_start, const int32_t* gather_end,
                                     int32_t num_reqs, void* k_out, void* v_out,
                                     int64_t out_rows, int32_t* d_err, kv_stream_t stream) {
  int rc = gather_checks(k_cache, v_cache, layer, num_layers, num_blocks, block_size,
                         num_kv_heads, head_dim, gather_start, gather_end, num_reqs, k_out,
                         v_out, out_rows, d_err);
  if (rc != KV_OK) return rc;
  if (range_stride < 0) return KV_EINVAL;
  if (range_stride > KV_MAX_RANGES_PER_REQ) return KV_EUNSUPPORTED;
  if (num_reqs == 0) return KV_OK;
  if (num_ranges == nullptr || !aligned(num_ranges, 4)) return KV_EINVAL;
  if (range_stride > 0 && (range_start == nullptr || range_len == nullptr ||
                           !aligned(range_start, 4) || !aligned(range_len, 4)))
    return KV_EINVAL;
  GatherArgs a{static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache),
               (int64_t)layer * num_blocks, num_blocks, block_size,
               num_kv_heads * head_dim * 2 / 16, nullptr, 0, gather_start, gather_end,
               num_reqs, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), out_rows,
               d_err, stream};
  return launch_gather(cache_gather_range_kernel, a, range_start, range_len, num_ranges,
                       range_stride);
}
