// kv_expand.cu -- unfold a manager-block table into a kernel-block table.
//
// Source: "Blocktabelle", Entwurfsmotivation (map_to_kernel_blocks: one
// manager block of block_size tokens is blocks_per_kv_block kernel blocks,
// e.g. 32 over 16) and Grenzen und Fehler (a kernel block size that does not
// divide the manager block size is rejected).  The pages do this on the host
// before the table is copied to the GPU; here it is one pass over the output
// table on the device, so the expanded table never crosses PCIe/C2C.
//
// GPU shape.  One thread per group of 4 output columns (one 16-byte store
// when the row pitch allows it), grid-stride over [num_reqs, kernel_stride].
// The manager row is read through L1: k neighbouring outputs share one entry.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int32_t expand_one(const int32_t* __restrict__ row, int32_t q,
                                              int32_t mgr_stride, int32_t k, uint32_t& err) {
  const int32_t c = q / k;
  if (c >= mgr_stride) return kNull;
  const int64_t m = row[c];
  if (m == kNull) return kNull;
  const int64_t j = q - (int64_t)c * k;
  if (m < 0 || m * k + (k - 1) > INT32_MAX) { err |= KV_ERR_BAD_BLOCK; return kNull; }
  return (int32_t)(m * k + j);
}

template <bool kVec4>
__global__ void __launch_bounds__(kThreads)
expand_kernel(const int32_t* __restrict__ mgr, int32_t num_reqs, int32_t mgr_stride, int32_t k,
              int32_t* __restrict__ out, int32_t kernel_stride, int32_t* err_word) {
  pdl_allow_next();
  pdl_wait();
  uint32_t err = 0;
  const int32_t groups = (kernel_stride + 3) / 4;
  const int64_t total = (int64_t)num_reqs * groups;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * kThreads) {
    const int32_t r = (int32_t)(i / groups);
    const int32_t q0 = (int32_t)(i - (int64_t)r * groups) * 4;
    const int32_t* row = mgr + (int64_t)r * mgr_stride;
    int32_t* dst = out + (int64_t)r * kernel_stride + q0;
    if (kVec4) {
      int4 v;
      v.x = expand_one(row, q0 + 0, mgr_stride, k, err);
      v.y = expand_one(row, q0 + 1, mgr_stride, k, err);
      v.z = expand_one(row, q0 + 2, mgr_stride, k, err);
      v.w = expand_one(row, q0 + 3, mgr_stride, k, err);
      *reinterpret_cast<int4*>(dst) = v;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (q0 + j < kernel_stride) dst[j] = expand_one(row, q0 + j, mgr_stride, k, err);
    }
  }
  report(err_word, err);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_expand_kernel_blocks(const int32_t* mgr_table, int32_t num_reqs,
                                       int32_t mgr_stride, int32_t mgr_block_size,
                                       int32_t kernel_block_size, int32_t* kernel_table,
                                       int32_t kernel_stride, int32_t* d_err,
                                       kv_stream_t stream) {
  if (num_reqs < 0 || mgr_stride < 0 || mgr_block_size <= 0 || kernel_block_size <= 0 ||
      kernel_stride < 0)
    return KV_EINVAL;
  if (mgr_block_size % kernel_block_size != 0) return KV_EUNSUPPORTED;
  const int32_t k = mgr_block_size / kernel_block_size;
  if ((int64_t)kernel_stride < (int64_t)mgr_stride * k) return KV_EINVAL;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (num_reqs == 0 || kernel_stride == 0) return KV_OK;
  if (kernel_table == nullptr || !aligned(kernel_table, 4)) return KV_EINVAL;
  if (mgr_stride > 0 && (mgr_table == nullptr || !aligned(mgr_table, 4))) return KV_EINVAL;
  const bool vec4 = kernel_stride % 4 == 0 && aligned(kernel_table, 16);
  const int64_t groups = (int64_t)num_reqs * ((kernel_stride + 3) / 4);
  const int64_t ctas = (groups + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)sm_count() * (2048 / kThreads);
  const int grid = (int)(ctas < cap ? ctas : cap);
  return launch_pdl(vec4 ? expand_kernel<true> : expand_kernel<false>, grid, kThreads, 0, stream,
                    mgr_table, num_reqs, mgr_stride, k, kernel_table, kernel_stride, d_err);
}
