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

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? KV_OK : KV_ECUDA;
}

}  // namespace kvp
