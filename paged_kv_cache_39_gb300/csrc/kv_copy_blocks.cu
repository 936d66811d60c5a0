// kv_copy_blocks.cu -- batched whole-block copy for copy-on-write.
//
// Source: "vLLM Block Table Management", Deep Dive 3: when a writer has to
// diverge from a shared block, the manager allocates a fresh block and queues
// KVCacheBlockCopy(src, dst) for the worker, which copies the KV data before
// the writer overwrites it; divergence costs one copy per diverging block.
//
// GPU shape.  Work units are runs of consecutive rows of one (pair, layer)
// block: one warp copies a K row and a V row at a time (16-byte vectors,
// 4 KiB in flight per warp), four rows per warp step on large batches (as in
// the KV write: a warp's rows leave back to back), one on small ones.  Both
// the source and the destination block (block_size x row_bytes, 32 KiB for
// 16 x 2 KiB) are read and written contiguously.  Persistent grid,
// grid-stride loop.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerLane = 4;
constexpr int kChunkVecs = 32 * kVecPerLane;

template <int kRowsPerWarp>  // consecutive rows of one (pair, layer) block per warp step
__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   int64_t num_blocks, int32_t block_size, int32_t num_layers,
                   int32_t row_vecs, const int32_t* __restrict__ src_blocks,
                   const int32_t* __restrict__ dst_blocks, int64_t num_pairs,
                   int32_t* err_word) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t groups = (block_size + kRowsPerWarp - 1) / kRowsPerWarp;  // per block
  const int64_t per_pair = (int64_t)num_layers * groups;
  const int64_t units = num_pairs * per_pair;
  uint32_t err = 0;
  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t pair = u / per_pair;
    const int64_t rem = u - pair * per_pair;
    const int64_t layer = rem / groups;
    const int64_t t0 = (rem - layer * groups) * kRowsPerWarp;
    const int64_t sb = src_blocks[pair], db = dst_blocks[pair];
    if (sb <= kNull || sb >= num_blocks) { err |= KV_ERR_BAD_BLOCK; continue; }
    if (db == kNull) { err |= KV_ERR_NULL_WRITE; continue; }
    if (db < 0 || db >= num_blocks) { err |= KV_ERR_BAD_BLOCK; continue; }
    const int nt = (int)(block_size - t0 < kRowsPerWarp ? block_size - t0 : kRowsPerWarp);
    for (int k = 0; k < nt; ++k) {
      const int64_t s_row = (layer * num_blocks + sb) * block_size + t0 + k;
      const int64_t d_row = (layer * num_blocks + db) * block_size + t0 + k;
      const uint4* ks = k_cache + s_row * row_vecs;
      const uint4* vs = v_cache + s_row * row_vecs;
      uint4* kd = k_cache + d_row * row_vecs;
      uint4* vd = v_cache + d_row * row_vecs;
      for (int c0 = 0; c0 < row_vecs; c0 += kChunkVecs) {
        uint4 kr[kVecPerLane], vr[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) {
          const int v = c0 + j * 32 + lane;
          if (v < row_vecs) {
            kr[j] = ks[v];  // plain loads: the same buffer is written (no .nc path)
            vr[j] = vs[v];
          }
        }
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) {
          const int v = c0 + j * 32 + lane;
          if (v < row_vecs) {
            st_stream(kd + v, kr[j]);
            st_stream(vd + v, vr[j]);
          }
        }
      }
    }
  }
  report(err_word, err);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_copy_blocks(void* k_cache, void* v_cache, int32_t num_layers,
                              int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, const int32_t* src_blocks,
                              const int32_t* dst_blocks, int32_t num_pairs, int32_t* d_err,
                              kv_stream_t stream) {
  if (num_layers < 0 || num_blocks < 1 || block_size <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_pairs < 0)
    return KV_EINVAL;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return KV_EUNSUPPORTED;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  const int64_t items = (int64_t)num_pairs * num_layers * block_size;
  if (items == 0) return KV_OK;
  if (k_cache == nullptr || v_cache == nullptr || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KV_EINVAL;
  if (src_blocks == nullptr || dst_blocks == nullptr || !aligned(src_blocks, 4) ||
      !aligned(dst_blocks, 4))
    return KV_EINVAL;
  // four rows per warp step on large batches (a block's rows are contiguous on
  // both sides), one row per warp when few rows leave warps idle
  const int64_t cap = (int64_t)sm_count() * (2048 / kThreads);
  const bool grouped = items >= cap * (kThreads / 32) * 4;
  const int rpw = grouped ? 4 : 1;
  const int64_t warps_needed =
      (int64_t)num_pairs * num_layers * ((block_size + rpw - 1) / rpw);
  const int64_t ctas_needed = (warps_needed * 32 + kThreads - 1) / kThreads;
  const int grid = (int)(ctas_needed < cap ? ctas_needed : cap);
  auto k4 = copy_blocks_kernel<4>;
  auto k1 = copy_blocks_kernel<1>;
  (grouped ? k4 : k1)<<<grid, kThreads, 0, stream>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks, block_size,
      num_layers, (int32_t)(row_bytes / 16), src_blocks, dst_blocks, num_pairs, d_err);
  return launch_status();
}
