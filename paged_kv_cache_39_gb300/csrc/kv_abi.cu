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

extern "C" const char* kv_status_string(int status) {
  switch (status) {
    case KV_OK: return "KV_OK";
    case KV_EINVAL: return "KV_EINVAL: invalid argument";
    case KV_EUNSUPPORTED: return "KV_EUNSUPPORTED: configuration rejected (fail closed)";
    case KV_ECUDA: return "KV_ECUDA: kernel launch failed";
    default: return "unknown kv_status";
  }
}

extern "C" int kv_abi_version(void) { return 4; }
