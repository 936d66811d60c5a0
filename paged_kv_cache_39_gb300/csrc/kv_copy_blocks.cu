// kv_copy_blocks.cu -- batched whole-block copy for copy-on-write (vector
// and bulk-copy forms).
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
  pdl_allow_next();
  pdl_wait();
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

// ---------------------------------------------------------------------------
// Bulk-copy form (kv_copy_blocks_bulk): the same copies moved by the
// bulk-copy engine, whole blocks at a time.  A unit is one K or V block of one
// (pair, layer), or a 32 KiB piece of it when the block is larger; it goes
// global -> shared -> global with cp.async.bulk (the load completes on a
// shared mbarrier, the store is one bulk group).  A CTA is one warp: the 32
// lanes describe 32 consecutive units (source and destination offsets, one
// pair lookup each) and lane 0 issues them, two stage buffers with one unit
// loaded ahead, two CTAs per SM (the shape the bulk-copy gather measured
// best).  Every wait is bounded; a timeout sets KV_ERR_TIMEOUT.

constexpr int kBulkStages = 2;
constexpr int kBulkStageBytes = 32768;
constexpr int kBulkCtasPerSm = 2;
constexpr int kBulkHeader = 128;  // mbarriers
constexpr size_t kBulkSmem = kBulkHeader + (size_t)kBulkStages * kBulkStageBytes;

__global__ void __launch_bounds__(32)
copy_blocks_bulk_kernel(unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                        int64_t num_blocks, int32_t num_layers, int64_t block_bytes,
                        int32_t pieces, const int32_t* __restrict__ src_blocks,
                        const int32_t* __restrict__ dst_blocks, int64_t num_pairs,
                        int32_t* err_word) {
  pdl_allow_next();
  pdl_wait();
  extern __shared__ __align__(128) unsigned char copy_smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(copy_smem);
  unsigned char* stage = copy_smem + kBulkHeader;
  const int lane = threadIdx.x;
  uint32_t err = 0;
  if (lane == 0) {
    for (int st = 0; st < kBulkStages; ++st) mbar_init(&bars[st], 1);
    mbar_fence_init();
  }
  __syncwarp();

  // units in pair-major order: (pair, layer, K/V, piece)
  const int64_t per_pair = (int64_t)num_layers * 2 * pieces;
  const int64_t total = num_pairs * per_pair;
  const int64_t per_cta = (total + gridDim.x - 1) / gridDim.x;
  const int64_t u0 = (int64_t)blockIdx.x * per_cta;
  const int64_t u1 = u0 + per_cta < total ? u0 + per_cta : total;

  uint32_t phase_bits = 0, armed_bits = 0;
  bool failed = false;
  int64_t p_dst = 0;
  int32_t p_bytes = 0, p_kv = 0, p_stage = 0;
  bool have_prev = false;
  int64_t unit = 0;

  // finish the previous unit: wait for its load, store it, commit its group
  auto finish_prev = [&]() {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(&bars[p_stage], (phase_bits >> p_stage) & 1u);
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    if (!ok) {
      failed = true;
      return;
    }
    phase_bits ^= 1u << p_stage;
    armed_bits &= ~(1u << p_stage);
    if (lane == 0) {
      unsigned char* out = (p_kv ? v_cache : k_cache) + p_dst;
      bulk_s2g(out, stage + (size_t)p_stage * kBulkStageBytes, (uint32_t)p_bytes);
      bulk_commit();
    }
  };

  for (int64_t ub = u0; ub < u1 && !failed; ub += 32) {
    // lane q describes unit ub + q (-1: nothing to copy)
    int64_t src_off = -1, dst_off = 0;
    int32_t bytes = 0, kv = 0;
    const int64_t u = ub + lane;
    if (u < u1) {
      const int64_t pair = u / per_pair;
      int64_t rem = u - pair * per_pair;
      const int64_t layer = rem / (2 * pieces);
      rem -= layer * 2 * pieces;
      kv = (int32_t)(rem / pieces);
      const int64_t piece = rem - (int64_t)kv * pieces;
      const int64_t sb = src_blocks[pair], db = dst_blocks[pair];
      if (sb <= kNull || sb >= num_blocks) {
        err |= KV_ERR_BAD_BLOCK;
      } else if (db == kNull) {
        err |= KV_ERR_NULL_WRITE;
      } else if (db < 0 || db >= num_blocks) {
        err |= KV_ERR_BAD_BLOCK;
      } else {
        const int64_t p0 = piece * kBulkStageBytes;
        const int64_t left = block_bytes - p0;
        bytes = (int32_t)(left < kBulkStageBytes ? left : kBulkStageBytes);
        src_off = (layer * num_blocks + sb) * block_bytes + p0;
        dst_off = (layer * num_blocks + db) * block_bytes + p0;
      }
    }
    const int nq = (int)(u1 - ub < 32 ? u1 - ub : 32);
    for (int q = 0; q < nq && !failed; ++q) {
      const int64_t q_src = __shfl_sync(kFull, src_off, q);
      const int64_t q_dst = __shfl_sync(kFull, dst_off, q);
      const int32_t q_bytes = __shfl_sync(kFull, bytes, q);
      const int32_t q_kv = __shfl_sync(kFull, kv, q);
      if (q_src < 0) continue;
      if (have_prev) finish_prev();
      if (failed) break;
      const int st = (int)(unit % kBulkStages);
      if (lane == 0) {
        // the stage's previous unit was stored one unit ago: its group must
        // have finished reading the stage (all but the latest group)
        if (unit >= kBulkStages) bulk_wait_read<kBulkStages - 1>();
        mbar_arrive_expect_tx(&bars[st], (uint32_t)q_bytes);
        bulk_g2s(stage + (size_t)st * kBulkStageBytes, (q_kv ? v_cache : k_cache) + q_src,
                 (uint32_t)q_bytes, &bars[st]);
      }
      armed_bits |= 1u << st;
      p_dst = q_dst;
      p_bytes = q_bytes;
      p_kv = q_kv;
      p_stage = st;
      have_prev = true;
      ++unit;
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
  report(err_word, err);
}

// Argument checks shared by both entry points; sets *row_bytes.
int copy_checks(void* k_cache, void* v_cache, int32_t num_layers, int64_t num_blocks,
                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                int32_t* d_err, int64_t* row_bytes) {
  if (num_layers < 0 || num_blocks < 1 || block_size <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_pairs < 0)
    return KV_EINVAL;
  *row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (*row_bytes % 16 != 0 || *row_bytes / 16 > INT32_MAX) return KV_EUNSUPPORTED;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if ((int64_t)num_pairs * num_layers * block_size == 0) return KV_OK;
  if (k_cache == nullptr || v_cache == nullptr || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return KV_EINVAL;
  if (src_blocks == nullptr || dst_blocks == nullptr || !aligned(src_blocks, 4) ||
      !aligned(dst_blocks, 4))
    return KV_EINVAL;
  return KV_OK;
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_copy_blocks(void* k_cache, void* v_cache, int32_t num_layers,
                              int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, const int32_t* src_blocks,
                              const int32_t* dst_blocks, int32_t num_pairs, int32_t* d_err,
                              kv_stream_t stream) {
  int64_t row_bytes = 0;
  const int rc = copy_checks(k_cache, v_cache, num_layers, num_blocks, block_size, num_kv_heads,
                             head_dim, src_blocks, dst_blocks, num_pairs, d_err, &row_bytes);
  const int64_t items = (int64_t)num_pairs * num_layers * block_size;
  if (rc != KV_OK || items == 0) return rc;
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
  return launch_pdl(grouped ? k4 : k1, grid, kThreads, 0, stream, static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), num_blocks, block_size, num_layers,
                    (int32_t)(row_bytes / 16), src_blocks, dst_blocks, (int64_t)num_pairs,
                    d_err);
}

extern "C" int kv_copy_blocks_bulk(void* k_cache, void* v_cache, int32_t num_layers,
                                   int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                   int32_t head_dim, const int32_t* src_blocks,
                                   const int32_t* dst_blocks, int32_t num_pairs, int32_t* d_err,
                                   kv_stream_t stream) {
  int64_t row_bytes = 0;
  const int rc = copy_checks(k_cache, v_cache, num_layers, num_blocks, block_size, num_kv_heads,
                             head_dim, src_blocks, dst_blocks, num_pairs, d_err, &row_bytes);
  if (rc != KV_OK || (int64_t)num_pairs * num_layers * block_size == 0) return rc;
  const int64_t block_bytes = row_bytes * block_size;
  const int64_t pieces = (block_bytes + kBulkStageBytes - 1) / kBulkStageBytes;
  if (pieces > INT32_MAX) return KV_EUNSUPPORTED;
  if (cudaFuncSetAttribute(copy_blocks_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kBulkSmem) != cudaSuccess)
    return KV_ECUDA;
  const int grid = sm_count() * kBulkCtasPerSm;
  return launch_pdl(copy_blocks_bulk_kernel, grid, 32, kBulkSmem, stream,
                    static_cast<unsigned char*>(k_cache), static_cast<unsigned char*>(v_cache),
                    num_blocks, num_layers, block_bytes, (int32_t)pieces, src_blocks, dst_blocks,
                    (int64_t)num_pairs, d_err);
}
