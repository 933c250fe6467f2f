// Status names and ABI version of libtt.
#include <stdlib.h>
#include <string.h>

#include "common.cuh"

namespace tt {
bool use_mma_kernels() {
  const char* v = getenv("TT_ATTN_IMPL");
  return v && strcmp(v, "mma") == 0;
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

TT_API int tt_version(void) { return 101; }
