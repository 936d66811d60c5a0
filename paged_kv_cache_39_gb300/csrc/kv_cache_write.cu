// kv_cache_write.cu -- scatter each new token's K and V rows into the paged
// caches at its slot, for every layer.
//
// Sources: "Blocktabelle", Verantwortung (the attention kernels write KV
// directly through slot_mapping); "vLLM Block Table Management", Deep Dive 8
// (each token's KV is stored at exactly its slot); "Range-addressed KV cache
// blocks ...", The Coordinate Approach (row n(layer, block, token) =
// (layer * B + block) * T + token, offset n * bytes_per_token).
//
// GPU shape.  A row is num_kv_heads * head_dim bf16 values (2 KiB for 8x128),
// contiguous in the input and in the cache, so one warp moves one (layer,
// token) row pair with 16-byte vector accesses: 32 lanes x 16 B = 512 B per
// instruction, fully coalesced on both sides.  Each lane keeps up to 4 K and
// 4 V vectors in flight (4 KiB per warp).  On large batches a warp step
// takes 4 consecutive tokens of one layer (their slots in one load, one lane
// each), so a warp writes the consecutive rows a prefill places in one block
// back to back (measured +5 % over one row per step); a small batch keeps one
// row per warp so its latency is one row's, and requests the row before the
// slot so that the slot and row loads share one round trip.
// Warps walk these groups in a grid-stride loop over a persistent grid sized
// to the SM count.  Everything is 64-bit addressed: a 32-layer cache passes
// 2^32 bytes.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;       // CTA size of the grouped form (large batches)
constexpr int kSmallThreads = 64;   // one row per warp: 2 warps per CTA, spread over more SMs
constexpr int kVecPerLane = 4;                 // 16-byte vectors per lane per chunk
constexpr int kChunkVecs = 32 * kVecPerLane;   // 2 KiB per K (and V) chunk


// The token's slot, read by every lane (one broadcast); issued in program
// order after the loads before it.
__device__ __forceinline__ int64_t ld_slot(const int64_t* p) {
  int64_t v;
  asm volatile("ld.global.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// Move one (layer, token) row pair to its slot (nothing for PAD or errors).
// With kLoadSlot the slot is read from *sp only once the row's first chunk
// has been requested: the K and V rows do not depend on the slot, so the two
// round trips overlap (a decode batch's write is one round trip, not two).
template <bool kLoadSlot>
__device__ __forceinline__ void write_row(const uint4* __restrict__ ks,
                                          const uint4* __restrict__ vs, int64_t s,
                                          const int64_t* sp, int64_t layer,
                                          uint4* __restrict__ k_cache,
                                          uint4* __restrict__ v_cache, int64_t num_blocks,
                                          int32_t block_size, int32_t row_vecs, int lane,
                                          uint32_t& err) {
  for (int c0 = 0; c0 < row_vecs; c0 += kChunkVecs) {
    uint4 kr[kVecPerLane], vr[kVecPerLane];
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
      const int v = c0 + j * 32 + lane;
      if (v < row_vecs) {
        kr[j] = ld_stream(ks + v);
        vr[j] = ld_stream(vs + v);
      }
    }
    if (kLoadSlot && c0 == 0) s = ld_slot(sp);
    if (s < 0) return;  // PAD: nothing to store (warp-uniform)
    const int64_t b = s / block_size;
    if (b == kNull) { err |= KV_ERR_NULL_WRITE; return; }
    if (b >= num_blocks) { err |= KV_ERR_BAD_SLOT; return; }
    const int64_t n = (layer * num_blocks + b) * block_size + (s - b * block_size);
    uint4* kd = k_cache + n * row_vecs;
    uint4* vd = v_cache + n * row_vecs;
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

template <int kRowsPerWarp>  // consecutive tokens of one layer per warp step
__global__ void __launch_bounds__(kThreads)
cache_write_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                   uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int64_t* __restrict__ slot_mapping, int32_t num_tokens,
                   int64_t items, int64_t num_blocks, int32_t block_size, int32_t row_vecs,
                   int32_t* err_word) {
  pdl_allow_next();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t groups = (num_tokens + kRowsPerWarp - 1) / kRowsPerWarp;  // per layer
  const int64_t units = groups * (items / num_tokens);
  uint32_t err = 0;
  for (int64_t u = warp0; u < units; u += nwarps) {
    const int64_t layer = u / groups;
    const int64_t t0 = (u - layer * groups) * kRowsPerWarp;
    if constexpr (kRowsPerWarp == 1) {
      const int64_t i = layer * num_tokens + t0;
      write_row<true>(key + i * row_vecs, value + i * row_vecs, 0, slot_mapping + t0, layer,
                      k_cache, v_cache, num_blocks, block_size, row_vecs, lane, err);
      continue;
    }
    const int nt = (int)(num_tokens - t0 < kRowsPerWarp ? num_tokens - t0 : kRowsPerWarp);
    // the slots of the group, one lane each, then shared by the warp
    const int64_t my_s = lane < nt ? slot_mapping[t0 + lane] : -1;
    for (int k = 0; k < nt; ++k) {
      const int64_t s = __shfl_sync(kFull, my_s, k);
      const int64_t i = layer * num_tokens + t0 + k;
      write_row<false>(key + i * row_vecs, value + i * row_vecs, s, nullptr, layer, k_cache,
                       v_cache, num_blocks, block_size, row_vecs, lane, err);
    }
  }
  report(err_word, err);
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_cache_write(const void* key, const void* value, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, int32_t num_tokens,
                              int32_t num_layers, int64_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim, int32_t* d_err,
                              kv_stream_t stream) {
  if (num_tokens < 0 || num_layers < 0 || num_blocks < 1 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return KV_EINVAL;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
  if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return KV_EUNSUPPORTED;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  const int64_t items = (int64_t)num_layers * num_tokens;
  if (items == 0) return KV_OK;
  if (key == nullptr || value == nullptr || k_cache == nullptr || v_cache == nullptr ||
      slot_mapping == nullptr)
    return KV_EINVAL;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
    return KV_EINVAL;
  const int32_t row_vecs = (int32_t)(row_bytes / 16);
  // Four rows per warp step once there are enough rows to keep every warp
  // slot busy several times over; a small batch (a decode step) spreads one
  // row per warp so that no warp serialises rows, two warps per CTA so that
  // the rows spread over 4x as many SMs (ncu, the 256-row decode write: 3.65
  // against 3.87 us with 8-warp CTAs).
  const bool grouped = items >= (int64_t)sm_count() * (2048 / 32) * 4;
  const int rpw = grouped ? 4 : 1;
  const int threads = grouped ? kThreads : kSmallThreads;
  const int64_t cap = (int64_t)sm_count() * (2048 / threads);
  const int64_t warps_needed = (int64_t)num_layers * ((num_tokens + rpw - 1) / rpw);
  const int64_t ctas_needed = (warps_needed * 32 + threads - 1) / threads;
  const int grid = (int)(ctas_needed < cap ? ctas_needed : cap);
  auto k4 = cache_write_kernel<4>;
  auto k1 = cache_write_kernel<1>;
  return launch_pdl(grouped ? k4 : k1, grid, threads, 0, stream,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping,
                    num_tokens, items, num_blocks, block_size, row_vecs, d_err);
}
