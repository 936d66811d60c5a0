// kv_abi.cu -- status strings, ABI version and the per-device SM count.
#include <mutex>

#include "kv_common.cuh"

namespace kvp {

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace kvp

namespace kvp {
namespace {

// A wait that nothing will satisfy: an mbarrier expecting one arrival that
// never comes, waited on with the library's bounded wait.  It must give up
// after `limit` tries and report KV_ERR_TIMEOUT, leaving the context usable.
__global__ void bounded_wait_probe_kernel(int64_t limit, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_fence_init();
  if (!mbar_wait_bounded(&bar, 0u, limit)) atomicOr(err, KV_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kvp

extern "C" int kv_diag_bounded_wait(int32_t spin_limit, int32_t* d_err, kv_stream_t stream) {
  if (spin_limit < 1 || spin_limit > (1 << 20) || d_err == nullptr ||
      !kvp::aligned(d_err, 4))
    return KV_EINVAL;
  kvp::bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(spin_limit, d_err);
  return kvp::launch_status();
}

extern "C" const char* kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "KV_OK";
    case KV_EINVAL: return "KV_EINVAL: invalid argument";
    case KV_EUNSUPPORTED: return "KV_EUNSUPPORTED: configuration rejected (fail closed)";
    case KV_ECUDA: return "KV_ECUDA: kernel launch failed";
    default: return "unknown kv_status";
  }
}

extern "C" int kv_abi_version(void) { return 7; }
