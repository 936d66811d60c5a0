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
  extern __shared__ int64_t smem[];
  int64_t* s_off = smem;                                                 // [num_reqs + 1]
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + a.num_reqs + 1);  // [num_reqs]
  __shared__ int64_t s_warp_sum[kThreads / 32];
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
  extern __shared__ int64_t smem[];
  int64_t* s_off = smem;
  int32_t* s_start = reinterpret_cast<int32_t*>(smem + a.num_reqs + 1);
  __shared__ int64_t s_warp_sum[kThreads / 32];
  uint32_t err = 0;
  // descriptor-row validation, every request, grid-wide
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < a.num_reqs;
       r += gridDim.x * blockDim.x)
    if (range_row_malformed(num_ranges, range_len, r, rstride)) err |= KV_ERR_BAD_RANGE;
  const int64_t total = packed_offsets(a, s_off, s_start, s_warp_sum, err);
  const int64_t rows = total < a.out_rows ? total : a.out_rows;
  RangeResolver res{range_start, range_len, num_ranges, rstride};
  gather_rows(a, s_off, s_start, rows, res, err);
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
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return KV_ECUDA;
  kernel<<<grid, kThreads, smem, a.stream>>>(a, extra...);
  return launch_status();
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
