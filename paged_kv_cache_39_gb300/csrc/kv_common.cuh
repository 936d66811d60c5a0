// kv_common.cuh -- device helpers shared by the kvpaged kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvpaged.h"

namespace kvp {

constexpr int64_t kPad = KV_PAD_SLOT_ID;
constexpr int32_t kNull = KV_NULL_BLOCK_ID;
constexpr unsigned kFull = 0xffffffffu;

// Number of SMs of the current device, cached per device for grid sizing.
int sm_count();

// OR the error bits of a warp into *err with one atomic per warp.
__device__ __forceinline__ void report(int32_t* err, uint32_t bits) {
  const unsigned active = __activemask();
  const uint32_t all = __reduce_or_sync(active, bits);
  if (err != nullptr && all != 0u) {
    const int leader = __ffs(active) - 1;
    if ((int)(threadIdx.x & 31) == leader) atomicOr(err, (int32_t)all);
  }
}

// 16-byte read-only global load that does not allocate in L1: every K/V
// byte moved here is touched exactly once.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte global store that does not allocate in L1 (streaming output).
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};"
               :
               : "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Quotient and remainder of a non-negative position by the block size: a
// shift and a mask when the block size is a power of two (the usual 16 or
// 32), a 32-bit division when the position fits, else a 64-bit division.
struct BlockDiv {
  int32_t size;
  int32_t shift;  // log2(size) when size is a power of two, else -1

  static BlockDiv make(int32_t size) {
    int32_t sh = -1;
    if (size > 0 && (size & (size - 1)) == 0) {
      sh = 0;
      while ((1 << sh) != size) ++sh;
    }
    return BlockDiv{size, sh};
  }

  __device__ __forceinline__ void divmod(int64_t p, int64_t& q, int64_t& r) const {
    if (shift >= 0) {
      q = p >> shift;
      r = p & (size - 1);
    } else if (p <= 0x7fffffff) {
      const uint32_t pu = (uint32_t)p, qu = pu / (uint32_t)size;
      q = qu;
      r = pu - qu * (uint32_t)size;
    } else {
      q = p / size;
      r = p - q * size;
    }
  }
};

// Largest r in [0, n) with q[r] <= t, or -1: the request whose span starts
// at or before token t (q is a non-decreasing query_start_loc).
__device__ __forceinline__ int find_span(const int32_t* q, int n, int32_t t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (q[mid] <= t) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

// Same search over int64 prefix offsets.
__device__ __forceinline__ int find_span64(const int64_t* q, int n, int64_t t) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (q[mid] <= t) lo = mid + 1; else hi = mid;
  }
  return lo - 1;
}

// Validation of descriptor row r: malformed when its count lies outside
// [0, stride] or one of its first `count` lengths is <= 0.  load() requests
// the count and the first four lengths together (one round trip for the
// usual short rows) and malformed() consumes them, so a caller can issue the
// loads early and pay for them late.
struct RangeRowCheck {
  int r = -1;
  int32_t n = 0;
  int32_t l4[4] = {1, 1, 1, 1};

  __device__ __forceinline__ void load(const int32_t* __restrict__ num_ranges,
                                       const int32_t* __restrict__ range_len, int row,
                                       int32_t stride, bool vec4 = false) {
    r = row;
    const int32_t* rl = range_len + (int64_t)row * stride;
    if (vec4) {  // the caller checked: stride >= 4, rows 16-byte aligned
      const int4 v = *reinterpret_cast<const int4*>(rl);
      l4[0] = v.x;
      l4[1] = v.y;
      l4[2] = v.z;
      l4[3] = v.w;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) l4[i] = i < stride ? rl[i] : 1;
    }
    n = num_ranges[row];
  }
  __device__ __forceinline__ bool malformed(const int32_t* __restrict__ range_len,
                                            int32_t stride) const {
    if (n < 0 || n > stride) return true;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) bad |= (i < n && l4[i] <= 0);
    const int32_t* rl = range_len + (int64_t)r * stride;
    for (int i = 4; i < n && !bad; ++i) bad = rl[i] <= 0;
    return bad;
  }
};

__device__ __forceinline__ bool range_row_malformed(const int32_t* __restrict__ num_ranges,
                                                    const int32_t* __restrict__ range_len,
                                                    int r, int32_t stride) {
  RangeRowCheck c;
  c.load(num_ranges, range_len, r, stride);
  return c.malformed(range_len, stride);
}

template <typename T>
__device__ __forceinline__ T warp_inclusive_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const T n = __shfl_up_sync(kFull, v, d);
    if (lane >= d) v += n;
  }
  return v;
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (cp.async.bulk) and shared-memory mbarriers.
// Global->shared copies complete a transaction count on an mbarrier;
// shared->global copies are tracked in bulk groups per issuing thread.
// Every wait on an mbarrier in this library is bounded twice: by kSpinLimit
// tries and by kWaitLimitNs of wall time on the GPU's global nanosecond timer,
// whichever runs out first.  A try may suspend the thread for a
// hardware-defined interval, so the try count alone would not bound the time;
// the timer does (a healthy copy completes in microseconds).

constexpr long kSpinLimit = 1L << 22;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity; false when either limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long limit = kSpinLimit,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_ns();
  for (long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's most recent bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's generic-proxy shared-memory writes before later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Asynchronous 8-byte global -> shared copy (no register holds the value
// while it is in flight); cp_async_wait_all() makes this thread's copies
// complete and visible to it.
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Grid-stride walk of [0, n) (n <= INT32_MAX), this thread's share, safe for
// grids of more than 2^32 threads: the CTA's first index and the grid's
// thread count are formed as 64-bit products (one wide multiply each, no
// division); past the test the index is below n + blockDim, so the walk runs
// in 32 bits.  A grid that covers n walks once (step n), else its thread
// count is below n, and i + step is formed only while it stays below n.
//   unsigned i, step;
//   if (grid_first(n, i, step)) do { ... i ... } while (grid_next(n, i, step));
__device__ __forceinline__ bool grid_first(int n, unsigned& i, unsigned& step) {
  if (n <= 0) return false;
  const uint64_t base = (uint64_t)blockIdx.x * blockDim.x;
  if (base >= (uint64_t)n) return false;
  i = (unsigned)base + threadIdx.x;
  const uint64_t total = (uint64_t)gridDim.x * blockDim.x;
  step = total >= (uint64_t)n ? (unsigned)n : (unsigned)total;
  return i < (unsigned)n;
}
__device__ __forceinline__ bool grid_next(int n, unsigned& i, unsigned step) {
  if (i >= (unsigned)n - step) return false;
  i += step;
  return true;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ECUDA;
}

// Programmatic dependent launch.  A kernel launched through launch_pdl() may
// be scheduled while the previous kernel on the stream is still running; it
// lets its own successor be scheduled at once (pdl_allow_next), then waits
// for the previous grid to complete, its memory visible (pdl_wait), before
// its first global load or store.  Results are those of plain stream order;
// only the gap between dependent launches shrinks.  Both instructions are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_allow_next() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr = {};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    (void)cudaGetLastError();
    return KV_ECUDA;
  }
  return KV_OK;
}

}  // namespace kvp
