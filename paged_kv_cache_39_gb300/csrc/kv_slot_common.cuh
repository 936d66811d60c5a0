// kv_slot_common.cuh -- per-token request lookup and slot checks shared by
// the slot-mapping kernels and the fused slot-mapping + KV write kernels.
//
// Source: "Blocktabelle", Datenfluss: a request owns the tokens
// [query_start_loc[r], query_start_loc[r+1]); a token's slot is its
// physical block * block_size + the offset in the block, PAD when there is
// none.
#pragma once

#include "kv_common.cuh"

namespace kvp {
namespace {

constexpr int kQslSmemMax = 8192;  // int32 entries of query_start_loc staged in smem

struct SlotArgs {
  const int32_t* qsl;
  const int64_t* positions;
  int32_t num_reqs, num_tokens, max_num_tokens;
  BlockDiv bs;
  int64_t num_blocks;
  int64_t* slot_mapping;
  int32_t* err;
};

// Stage query_start_loc in shared memory when it fits.
// `overlap()` runs once the thread's staging loads are in flight and before
// the barrier: work that waits on other loads (a position) can then issue
// its own loads without holding the staging back.
// Up to kStageLoads entries per thread are requested before any is stored,
// so up to kStageLoads * blockDim entries arrive in one round trip (a
// 256-request batch has 257: with one load per thread before the store,
// thread 0's second load waited on its first, and the barrier on both).
template <int kStageLoads = 4, class Overlap>
__device__ __forceinline__ const int32_t* stage_qsl(const SlotArgs& a, int32_t* s_qsl,
                                                    bool staged, Overlap&& overlap) {
  const int n = a.num_reqs;
  if (staged) {
    const int i0 = threadIdx.x;
    int32_t v[kStageLoads];
#pragma unroll
    for (int u = 0; u < kStageLoads; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      v[u] = i <= n ? a.qsl[i] : 0;
    }
    overlap();
#pragma unroll
    for (int u = 0; u < kStageLoads; ++u) {
      const int i = i0 + u * (int)blockDim.x;
      if (i <= n) s_qsl[i] = v[u];
    }
    for (int i = i0 + kStageLoads * (int)blockDim.x; i <= n; i += blockDim.x) s_qsl[i] = a.qsl[i];
    __syncthreads();
  } else {
    overlap();
  }
  return staged ? s_qsl : a.qsl;
}

// Validate query_start_loc grid-wide (q: the staged or the global copy):
// non-decreasing, q[0] >= 0, q[num_reqs] <= num_tokens.
__device__ __forceinline__ void check_qsl(const SlotArgs& a, const int32_t* q, uint32_t& err) {
  const int n = a.num_reqs;
  unsigned i, step;
  if (grid_first(n, i, step)) do {
      if (q[i] > q[i + 1]) err |= KV_ERR_BAD_QSL;
    } while (grid_next(n, i, step));
  if (n > 0 && blockIdx.x == 0 && threadIdx.x == 0 && (q[0] < 0 || q[n] > a.num_tokens))
    err |= KV_ERR_BAD_QSL;
}

__device__ __forceinline__ const int32_t* stage_qsl(const SlotArgs& a, int32_t* s_qsl,
                                                    bool staged) {
  return stage_qsl<4>(a, s_qsl, staged, [] {});
}

// Request owning token t (t < num_tokens), or -1 when no span covers it.
__device__ __forceinline__ int request_of(const int32_t* q, int n, int32_t t) {
  if (n <= 0) return -1;
  const int r = find_span(q, n, t);
  return (r >= 0 && t < q[r + 1]) ? r : -1;
}

// Same, trying request t first: a decode batch gives request t its token t,
// and two reads of q (shared memory when staged) confirm it where the search
// takes about nine dependent ones.  Exact whenever query_start_loc is non-decreasing (spans
// are then disjoint); with a malformed one the slots are unspecified anyway.
__device__ __forceinline__ int request_of_guess(const int32_t* q, int n, int32_t t) {
  if (t < n && q[t] <= t && t < q[t + 1]) return t;
  return request_of(q, n, t);
}

// Same, trying the thread's previous request first: a thread's tokens are
// 256 apart, so inside a long prefill they keep falling in one span.  Two
// forms, each measured on the map that uses it at 1M positions: the paged
// map re-reads the span bounds from shared memory (32 registers, 8 CTAs per
// SM; keeping them in registers took it to 38 and 3.7 % slower), the range
// map keeps them in registers (4.6 % faster than re-reading).
__device__ __forceinline__ int request_of_cached(const int32_t* q, int n, int32_t t, int& last) {
  if (last >= 0 && t >= q[last] && t < q[last + 1]) return last;
  const int r = request_of(q, n, t);
  if (r >= 0) last = r;
  return r;
}

struct ReqSpan {
  int r = -1;
  int32_t lo = 0, hi = 0;  // the span [lo, hi) of request r (empty while r < 0)
};
__device__ __forceinline__ int request_of_cached(const int32_t* q, int n, int32_t t, ReqSpan& c) {
  if (t >= c.lo && t < c.hi) return c.r;
  const int r = request_of(q, n, t);
  if (r >= 0) {
    c.r = r;
    c.lo = q[r];
    c.hi = q[r + 1];
  }
  return r;
}

// Final check of a resolved physical block and the slot it gives (off is
// the position's offset inside its block).
__device__ __forceinline__ int64_t slot_of(int64_t b, int64_t off, int32_t T, int64_t B,
                                           uint32_t& err) {
  if (b == kNull) return kPad;
  if (b < 0 || b >= B) { err |= KV_ERR_BAD_BLOCK; return kPad; }
  return b * T + off;
}

// Host-side checks shared by every slot-mapping entry point.
int check_common(const int32_t* qsl, const int64_t* positions, int32_t num_reqs,
                 int32_t num_tokens, int32_t max_num_tokens, int32_t block_size,
                 int64_t num_blocks, const int64_t* slot_mapping) {
  if (num_reqs < 0 || num_tokens < 0 || max_num_tokens < num_tokens ||
      max_num_tokens > KV_MAX_TOKENS || block_size <= 0 || num_blocks < 1)
    return KV_EINVAL;
  if (num_reqs > 0 && (qsl == nullptr || !aligned(qsl, 4))) return KV_EINVAL;
  if (num_tokens > 0 && (positions == nullptr || !aligned(positions, 8))) return KV_EINVAL;
  if (max_num_tokens > 0 && (slot_mapping == nullptr || !aligned(slot_mapping, 8)))
    return KV_EINVAL;
  return KV_OK;
}

// Descriptor arrays of the range entry points: at most 256 ranges per request
// (more is refused, fail closed), int32 rows of range_stride entries.
int check_ranges(const int32_t* range_start, const int32_t* range_len, const int32_t* num_ranges,
                 int32_t range_stride, int32_t num_reqs) {
  if (range_stride < 0) return KV_EINVAL;
  if (range_stride > KV_MAX_RANGES_PER_REQ) return KV_EUNSUPPORTED;
  if (num_reqs > 0) {
    if (num_ranges == nullptr || !aligned(num_ranges, 4)) return KV_EINVAL;
    if (range_stride > 0 && (range_start == nullptr || range_len == nullptr ||
                             !aligned(range_start, 4) || !aligned(range_len, 4)))
      return KV_EINVAL;
  }
  return KV_OK;
}

// Rows start on 16-byte boundaries: a row's first four descriptors come in one load.
bool rows_vec4(const int32_t* range_start, const int32_t* range_len, int32_t range_stride) {
  return range_stride >= 4 && range_stride % 4 == 0 && aligned(range_start, 16) &&
         aligned(range_len, 16);
}

}  // namespace
}  // namespace kvp
