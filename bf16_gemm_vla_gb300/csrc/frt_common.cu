// Status strings, ABI version, device queries and the launch counter.
#include <atomic>
#include <mutex>

#include "frt_host.h"

namespace frt {

int sm_count() {
  static std::mutex mu;
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      counts[dev] = n;
  }
  return counts[dev];
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}  // namespace

void note_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

}  // namespace frt

extern "C" int frt_abi_version(void) { return 3; }

extern "C" unsigned long long frt_launch_count(void) { return frt::g_launches.load(); }

extern "C" const char* frt_status_string(frt_status s) {
  switch (s) {
    case FRT_OK: return "FRT_OK";
    case FRT_ERR_INVALID_ARG: return "FRT_ERR_INVALID_ARG";
    case FRT_ERR_UNSUPPORTED_SHAPE: return "FRT_ERR_UNSUPPORTED_SHAPE";
    case FRT_ERR_MISALIGNED: return "FRT_ERR_MISALIGNED";
    case FRT_ERR_WORKSPACE_TOO_SMALL: return "FRT_ERR_WORKSPACE_TOO_SMALL";
    case FRT_ERR_CUDA: return "FRT_ERR_CUDA";
    case FRT_ERR_TIMEOUT: return "FRT_ERR_TIMEOUT";
  }
  return "FRT_ERR_UNKNOWN";
}
