// kv_slot_mapping.cu -- token -> cache slot, through a block table ("paged")
// or through contiguous range descriptors ("range").
//
// Sources: "Blocktabelle", Datenfluss (the slot-mapping kernel: block index
// pos // block_size, table lookup, slot = block * block_size + offset, tail
// padded with PAD); "Range-addressed KV cache blocks ...", The Innovation
// (physical_block = range_start + (pos // block_size - range_cum), descriptor
// loaded once per position block, positions outside every range padded).
//
// GPU shape.  The pages' kernel runs one program per request and walks its
// tokens, which leaves a 128K-token request on one SM.  Here a CTA owns a
// fixed tile of 1024 consecutive tokens (4 per thread, coalesced), so the
// grid depends only on max_num_tokens (stable under CUDA-graph capture) and
// long prefills spread over every SM.  Each thread finds its request by a
// binary search of query_start_loc staged in shared memory.  The tail
// [num_tokens, max_num_tokens) is just more tiles that store PAD.
#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kThreads = 256;
constexpr int kTokPerThread = 4;
constexpr int kTile = kThreads * kTokPerThread;
constexpr int kQslSmemMax = 8192;  // int32 entries of query_start_loc staged in smem

struct SlotArgs {
  const int32_t* qsl;
  const int64_t* positions;
  int32_t num_reqs, num_tokens, max_num_tokens, block_size;
  int64_t num_blocks;
  int64_t* slot_mapping;
  int32_t* err;
};

// Stage query_start_loc in shared memory when it fits; validate it grid-wide.
__device__ __forceinline__ const int32_t* stage_qsl(const SlotArgs& a, int32_t* s_qsl,
                                                    bool staged, uint32_t& err) {
  const int n = a.num_reqs;
  if (staged) {
    for (int i = threadIdx.x; i <= n; i += blockDim.x) s_qsl[i] = a.qsl[i];
    __syncthreads();
  }
  const int32_t* q = staged ? s_qsl : a.qsl;
  if (n > 0) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
      if (q[i] > q[i + 1]) err |= KV_ERR_BAD_QSL;
    if (blockIdx.x == 0 && threadIdx.x == 0 && (q[0] < 0 || q[n] > a.num_tokens))
      err |= KV_ERR_BAD_QSL;
  }
  return q;
}

// Request owning token t (t < num_tokens), or -1 when no span covers it.
__device__ __forceinline__ int request_of(const int32_t* q, int n, int32_t t) {
  if (n <= 0) return -1;
  const int r = find_span(q, n, t);
  return (r >= 0 && t < q[r + 1]) ? r : -1;
}

// Final check of a resolved physical block and the slot it gives.
__device__ __forceinline__ int64_t slot_of(int64_t b, int64_t p, int32_t T, int64_t B,
                                           uint32_t& err) {
  if (b == kNull) return kPad;
  if (b < 0 || b >= B) { err |= KV_ERR_BAD_BLOCK; return kPad; }
  return b * T + p % T;
}

__global__ void __launch_bounds__(kThreads)
slot_mapping_paged_kernel(SlotArgs a, const int32_t* __restrict__ table, int32_t stride,
                          bool qsl_in_smem) {
  extern __shared__ int32_t s_qsl[];
  const int32_t base = blockIdx.x * kTile + threadIdx.x;
  // positions do not depend on the request: start their loads first
  int64_t p[kTokPerThread];
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    p[k] = t < a.num_tokens ? a.positions[t] : 0;
  }
  uint32_t err = 0;
  const int32_t* q = stage_qsl(a, s_qsl, qsl_in_smem, err);
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    if (t >= a.max_num_tokens) break;
    int64_t slot = kPad;
    if (t < a.num_tokens) {
      const int r = request_of(q, a.num_reqs, t);
      if (r >= 0) {
        if (p[k] < 0) {
          err |= KV_ERR_BAD_POSITION;
        } else {
          const int64_t lb = p[k] / a.block_size;
          if (lb < stride)
            slot = slot_of(table[(int64_t)r * stride + lb], p[k], a.block_size, a.num_blocks, err);
        }
      }
    }
    a.slot_mapping[t] = slot;
  }
  report(a.err, err);
}

// ---------------------------------------------------------------------------
// Range variant.  For a warp whose 32 tokens belong to one request (prefill,
// long context) the request's descriptors are read 32 at a time, one per
// lane; a warp scan turns the lengths into range ends, and each lane finds
// its range with a 5-step binary search over the lanes (shuffles).  The loop
// stops as soon as every lane is resolved, so the steady state of one range
// per request costs one descriptor load per 32 positions.  Warps that mix
// requests (decode batches) let each lane walk its own request's few ranges.
// Rows with a bad count or bad lengths are flagged by a separate grid-wide
// sweep over every request, so the error word does not depend on which
// descriptors the token loop happened to read.

// Warp path: all needing lanes share request r0.  The count and the first 32
// descriptors are requested together (`pre_s`, `pre_l`: descriptor `lane`,
// loaded before the count is known), so the steady state costs one round trip.
__device__ __forceinline__ void range_lookup_warp(const int32_t* __restrict__ rs,
                                                  const int32_t* __restrict__ rl, int nr,
                                                  int32_t pre_s, int32_t pre_l, bool need,
                                                  int64_t lb, int64_t& b_out, bool& found) {
  const int lane = threadIdx.x & 31;
  int64_t cum_base = 0;
  for (int c0 = 0; c0 < nr; c0 += 32) {
    const int i = c0 + lane;
    int32_t s = 0, len = 0;
    if (i < nr) {
      s = c0 == 0 ? pre_s : rs[i];
      len = max(c0 == 0 ? pre_l : rl[i], 0);
    }
    const int64_t incl = warp_inclusive_scan<int64_t>((int64_t)len);
    const int64_t total = __shfl_sync(kFull, incl, 31);
    const int64_t end = cum_base + incl;  // first logical block after range i
    // first lane j whose range ends past lb
    int lo = 0, hi = 31;
#pragma unroll
    for (int it = 0; it < 5; ++it) {
      const int mid = (lo + hi) >> 1;
      const int64_t v = __shfl_sync(kFull, end, mid);
      if (lo < hi) {
        if (v > lb) hi = mid; else lo = mid + 1;
      }
    }
    const int32_t sj = __shfl_sync(kFull, s, lo);
    const int64_t endj = __shfl_sync(kFull, end, lo);
    const int32_t lenj = __shfl_sync(kFull, len, lo);
    if (need && !found && lb < cum_base + total) {
      found = true;
      b_out = (int64_t)sj + (lb - (endj - lenj));
    }
    cum_base += total;
    if (!__any_sync(kFull, need && !found)) break;
  }
}

constexpr int kLanePrefetch = 4;  // descriptors a lane requests with the count

__global__ void __launch_bounds__(kThreads)
slot_mapping_range_kernel(SlotArgs a, const int32_t* __restrict__ range_start,
                          const int32_t* __restrict__ range_len,
                          const int32_t* __restrict__ num_ranges, int32_t rstride,
                          bool qsl_in_smem) {
  extern __shared__ int32_t s_qsl[];
  const int32_t base = blockIdx.x * kTile + threadIdx.x;
  const int lane = threadIdx.x & 31;
  int64_t p[kTokPerThread];
#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    p[k] = t < a.num_tokens ? a.positions[t] : 0;
  }
  uint32_t err = 0;
  const int32_t* q = stage_qsl(a, s_qsl, qsl_in_smem, err);

  // descriptor-row validation, every request, grid-wide
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < a.num_reqs;
       r += gridDim.x * blockDim.x) {
    const int nr = num_ranges[r];
    if (nr < 0 || nr > rstride) {
      err |= KV_ERR_BAD_RANGE;
    } else {
      const int32_t* rl = range_len + (int64_t)r * rstride;
      for (int i = 0; i < nr; ++i)
        if (rl[i] <= 0) { err |= KV_ERR_BAD_RANGE; break; }
    }
  }

#pragma unroll
  for (int k = 0; k < kTokPerThread; ++k) {
    const int32_t t = base + k * kThreads;
    // every lane of the warp reaches the shuffles below: no early exit here
    const int r = t < a.num_tokens ? request_of(q, a.num_reqs, t) : -1;
    bool need = false;
    if (r >= 0) {
      if (p[k] < 0) err |= KV_ERR_BAD_POSITION;
      else need = true;
    }
    const int64_t lb = need ? p[k] / a.block_size : 0;
    bool found = false;
    int64_t b = 0;
    const unsigned needers = __ballot_sync(kFull, need);
    if (needers != 0u) {
      const int r0 = __shfl_sync(kFull, r, __ffs(needers) - 1);
      if (__all_sync(kFull, !need || r == r0)) {
        const int32_t* rs0 = range_start + (int64_t)r0 * rstride;
        const int32_t* rl0 = range_len + (int64_t)r0 * rstride;
        int32_t pre_s = 0, pre_l = 0;
        if (lane < rstride) {
          pre_s = rs0[lane];
          pre_l = rl0[lane];
        }
        const int nr0 = num_ranges[r0];
        if (nr0 >= 0 && nr0 <= rstride)  // malformed rows: PAD (flagged by the sweep)
          range_lookup_warp(rs0, rl0, nr0, pre_s, pre_l, need, lb, b, found);
      } else if (need) {
        const int32_t* rs = range_start + (int64_t)r * rstride;
        const int32_t* rl = range_len + (int64_t)r * rstride;
        int32_t pre_s[kLanePrefetch], pre_l[kLanePrefetch];
#pragma unroll
        for (int i = 0; i < kLanePrefetch; ++i) {
          pre_s[i] = i < rstride ? rs[i] : 0;
          pre_l[i] = i < rstride ? rl[i] : 0;
        }
        const int nr = num_ranges[r];
        if (nr >= 0 && nr <= rstride) {
          int64_t cum = 0;
#pragma unroll
          for (int i = 0; i < kLanePrefetch; ++i) {
            if (!found && i < nr) {
              const int64_t len = max(pre_l[i], 0);
              if (lb < cum + len) {
                b = (int64_t)pre_s[i] + (lb - cum);
                found = true;
              }
              cum += len;
            }
          }
          for (int i = kLanePrefetch; !found && i < nr; ++i) {
            const int64_t len = max(rl[i], 0);
            if (lb < cum + len) {
              b = (int64_t)rs[i] + (lb - cum);
              found = true;
            }
            cum += len;
          }
        }
      }
    }
    if (t < a.max_num_tokens)
      a.slot_mapping[t] = found ? slot_of(b, p[k], a.block_size, a.num_blocks, err) : kPad;
  }
  report(a.err, err);
}

int check_common(const int32_t* qsl, const int64_t* positions, int32_t num_reqs,
                 int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                 int64_t num_blocks, const int64_t* slot_mapping) {
  if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens || block_size <= 0 ||
      num_blocks < 1)
    return KV_EINVAL;
  if (num_reqs > 0 && (qsl == nullptr || !aligned(qsl, 4))) return KV_EINVAL;
  if (num_tokens > 0 && (positions == nullptr || !aligned(positions, 8))) return KV_EINVAL;
  if (max_num_tokens > 0 && (slot_mapping == nullptr || !aligned(slot_mapping, 8)))
    return KV_EINVAL;
  return KV_OK;
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" int kv_slot_mapping_paged(const int32_t* query_start_loc, const int64_t* positions,
                                     const int32_t* block_table, int32_t table_stride,
                                     int32_t num_reqs, int32_t num_tokens,
                                     int32_t max_num_tokens, int32_t block_size,
                                     int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                                     kv_stream_t stream) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  if (table_stride < 0) return KV_EINVAL;
  if (num_reqs > 0 && num_tokens > 0 && table_stride > 0 &&
      (block_table == nullptr || !aligned(block_table, 4)))
    return KV_EINVAL;
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (max_num_tokens == 0 && num_reqs == 0) return KV_OK;
  const int grid = max(1, (max_num_tokens + kTile - 1) / kTile);
  const bool staged = num_reqs + 1 <= kQslSmemMax;
  const size_t smem = staged && num_reqs > 0 ? sizeof(int32_t) * (num_reqs + 1) : 0;
  SlotArgs a{query_start_loc, positions, num_reqs, num_tokens, max_num_tokens, block_size,
             num_blocks, slot_mapping, d_err};
  slot_mapping_paged_kernel<<<grid, kThreads, smem, stream>>>(a, block_table, table_stride,
                                                              staged && num_reqs > 0);
  return launch_status();
}

extern "C" int kv_slot_mapping_range(const int32_t* query_start_loc, const int64_t* positions,
                                     const int32_t* range_start, const int32_t* range_len,
                                     const int32_t* num_ranges, int32_t range_stride,
                                     int32_t num_reqs, int32_t num_tokens,
                                     int32_t max_num_tokens, int32_t block_size,
                                     int64_t num_blocks, int64_t* slot_mapping, int32_t* d_err,
                                     kv_stream_t stream) {
  int rc = check_common(query_start_loc, positions, num_reqs, num_tokens, max_num_tokens,
                        block_size, num_blocks, slot_mapping);
  if (rc != KV_OK) return rc;
  if (range_stride < 0) return KV_EINVAL;
  if (range_stride > KV_MAX_RANGES_PER_REQ) return KV_EUNSUPPORTED;
  if (num_reqs > 0) {
    if (num_ranges == nullptr || !aligned(num_ranges, 4)) return KV_EINVAL;
    if (range_stride > 0 && (range_start == nullptr || range_len == nullptr ||
                             !aligned(range_start, 4) || !aligned(range_len, 4)))
      return KV_EINVAL;
  }
  if (d_err != nullptr && !aligned(d_err, 4)) return KV_EINVAL;
  if (max_num_tokens == 0 && num_reqs == 0) return KV_OK;
  const int grid = max(1, (max_num_tokens + kTile - 1) / kTile);
  const bool staged = num_reqs + 1 <= kQslSmemMax;
  const size_t smem = staged && num_reqs > 0 ? sizeof(int32_t) * (num_reqs + 1) : 0;
  SlotArgs a{query_start_loc, positions, num_reqs, num_tokens, max_num_tokens, block_size,
             num_blocks, slot_mapping, d_err};
  slot_mapping_range_kernel<<<grid, kThreads, smem, stream>>>(
      a, range_start, range_len, num_ranges, range_stride, staged && num_reqs > 0);
  return launch_status();
}
