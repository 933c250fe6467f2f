// Status names, ABI version and per-device host caches of libtt.
#include <atomic>

#include "common.cuh"

namespace tt {
int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int sm_count() {
  static std::atomic<int> n_sm[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 1;
  int n = n_sm[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    n_sm[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}
}  // namespace tt

TT_API const char* tt_status_string(int code) {
  switch (code) {
    case TT_OK: return "TT_OK";
    case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG: bad pointer, size, stride, alignment or target id";
    case TT_ERR_INVALID_TREE: return "TT_ERR_INVALID_TREE: parent/length arrays are not a topological tree";
    case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED: head_dim or head grouping not covered";
    case TT_ERR_WORKSPACE: return "TT_ERR_WORKSPACE: workspace or interval capacity too small";
    case TT_ERR_CUDA: return "TT_ERR_CUDA: a CUDA runtime call failed";
    case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "unknown tt status";
  }
}

TT_API int tt_version(void) { return 203; }
