// kv_range_table.cu -- fill a block table directly from range descriptors.
//
// Source: "Range-addressed KV cache blocks ...", Status: in range mode the
// staged block table is copied to the kernels' table every step although the
// range tables already hold the request layout; a range-expansion kernel can
// fill the kernels' table directly from the ranges.  Logical block
// range_cum + j of range i is physical block range_start + j (The
// Innovation).
//
// GPU shape.  A CTA owns a chunk of up to 2048 columns of one row (grid-stride
// over (row, chunk) pairs, so a few long rows still spread over the SMs).  The
// row's descriptors (at most 256, one per thread) are scanned into range ends
// in shared memory with a block-wide scan; then the CTA writes its columns
// with coalesced stores, each thread finding its column's range by a binary
// search of the shared ends.  Columns past the ranges are the null block.
// Row-level errors are reported by the CTA that owns the row's first chunk.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;  // >= KV_MAX_RANGES_PER_REQ: one descriptor per thread
constexpr int kColsPerCta = 2048;

__global__ void __launch_bounds__(kThreads)
table_from_ranges_kernel(const int32_t* __restrict__ range_start,
                         const int32_t* __restrict__ range_len,
                         const int32_t* __restrict__ num_ranges, int32_t rstride,
                         int32_t num_reqs, int32_t* __restrict__ table, int32_t tstride,
                         int32_t* err_word) {
  pdl_allow_next();
  pdl_wait();
  __shared__ int64_t s_cum[kThreads];   // first logical block of range i
  __shared__ int64_t s_end[kThreads];   // first logical block after range i
  __shared__ int32_t s_start[kThreads];
  __shared__ int64_t s_warp[kThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint32_t err = 0;
  const int chunks = (tstride + kColsPerCta - 1) / kColsPerCta;
  const int64_t units = (int64_t)num_reqs * (chunks > 0 ? chunks : 1);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int r = (int)(u / (chunks > 0 ? chunks : 1));
    const int chunk = (int)(u - (int64_t)r * (chunks > 0 ? chunks : 1));
    const bool first = chunk == 0;  // reports the row-level errors
    int nr = num_ranges[r];
    if (nr < 0 || nr > rstride) {
      if (tid == 0 && first) err |= KV_ERR_BAD_RANGE;
      nr = 0;
    }
    int32_t st = 0, len = 0;
    if (tid < nr) {
      st = range_start[(int64_t)r * rstride + tid];
      len = range_len[(int64_t)r * rstride + tid];
      if (len <= 0) {
        if (first) err |= KV_ERR_BAD_RANGE;
        len = 0;
      }
    }
    // block-wide inclusive scan of the lengths
    const int64_t incl_w = warp_inclusive_scan<int64_t>((int64_t)len);
    if (lane == 31) s_warp[wid] = incl_w;
    __syncthreads();
    int64_t base = 0;
    for (int w = 0; w < wid; ++w) base += s_warp[w];
    int64_t total = 0;
    for (int w = 0; w < kThreads / 32; ++w) total += s_warp[w];
    const int64_t incl = base + incl_w;
    if (tid < nr) {
      s_cum[tid] = incl - len;
      s_end[tid] = incl;
      s_start[tid] = st;
    }
    __syncthreads();
    if (tid == 0 && first && total > tstride) err |= KV_ERR_OUT_OF_SPACE;
    int32_t* row = table + (int64_t)r * tstride;
    const int c_end = min(tstride, (chunk + 1) * kColsPerCta);
    for (int c = chunk * kColsPerCta + tid; c < c_end; c += kThreads) {
      int32_t v = kNull;
      if (c < total) {
        // first range whose end lies past column c (zero-length ranges never qualify)
        int lo = 0, hi = nr - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (s_end[mid] > c) hi = mid; else lo = mid + 1;
        }
        const int64_t b = (int64_t)s_start[lo] + (c - s_cum[lo]);
        if (b < 0 || b > INT32_MAX) err |= KV_ERR_BAD_BLOCK;
        else v = (int32_t)b;
      }
      row[c] = v;
    }
    __syncthreads();  // shared arrays are rewritten for the next row
  }
  report(err_word, err);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_table_from_ranges(const int32_t* range_start, const int32_t* range_len,
                                    const int32_t* num_ranges, int32_t range_stride,
                                    int32_t num_reqs, int32_t* block_table,
                                    int32_t table_stride, int32_t* d_err, kv_stream_t stream) {
  if (num_reqs < 0 || range_stride < 0 || table_stride < 0) return KV_EINVAL;
  if (range_stride > KV_MAX_RANGES_PER_REQ) return KV_EUNSUPPORTED;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (num_reqs == 0) return KV_OK;
  if (num_ranges == nullptr || !aligned(num_ranges, 4)) return KV_EINVAL;
  if (range_stride > 0 && (range_start == nullptr || range_len == nullptr ||
                           !aligned(range_start, 4) || !aligned(range_len, 4)))
    return KV_EINVAL;
  if (table_stride > 0 && (block_table == nullptr || !aligned(block_table, 4))) return KV_EINVAL;
  const int64_t chunks = table_stride > 0 ? (table_stride + kColsPerCta - 1) / kColsPerCta : 1;
  const int64_t units = (int64_t)num_reqs * chunks;
  const int64_t cap = (int64_t)sm_count() * (2048 / kThreads);
  const int grid = (int)(units < cap ? units : cap);
  return launch_pdl(table_from_ranges_kernel, grid, kThreads, 0, stream, range_start, range_len,
                    num_ranges, range_stride, num_reqs, block_table, table_stride, d_err);
}
