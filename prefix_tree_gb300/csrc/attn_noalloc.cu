// Chunk-mode attention backward that allocates nothing.
//
// Some callers cannot allocate device memory when they make this call: code
// running on a runtime that owns every device allocation through its own
// pool, or code on a latency path where cudaMalloc's implicit device
// synchronisation is not acceptable. tt_tree_attn_chunk_bwd_noalloc therefore
// takes no workspace. Its per-row scratch (lse·log2 e and Σ dO·O of the
// chunk's query rows) lives in the file-scope device array below, which every
// GPU that loads the library holds until the process exits.
#include <mutex>

#include "attn.cuh"

namespace {
// 2 MiB: room for 2 · Hq · roundup(C, 128) floats with Hq · roundup(C, 128) <= 262144.
constexpr size_t kNoAllocScratchFloats = size_t(1) << 19;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[tt::kMaxDevices] = {};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached. The cache is not
// refreshed after cudaDeviceReset (the module, and so the array, may then be
// loaded at another address).
int noalloc_scratch(void** out) {
  const int dev = tt::current_device();
  if (dev < 0) return TT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return TT_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TT_OK;
}
}  // namespace

using namespace tt;

TT_API int tt_tree_attn_chunk_bwd_noalloc(const tt_bf16* q, int64_t C, int64_t s0, const tt_bf16* k_path,
                                          const tt_bf16* v_path, const tt_bf16* o, const float* lse, int64_t lse_ld,
                                          const tt_bf16* dO, tt_bf16* dq, float* dk_acc, float* dv_acc, int Hq,
                                          int Hkv, int d, float scale, int32_t* err, tt_stream_t stream) {
  if (Hq < 1 || Hkv < 1) return TT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (d != 64 && d != 128)) return TT_ERR_UNSUPPORTED;
  if (!q || !k_path || !v_path || !o || !lse || !dO || !dq || !dk_acc || !dv_acc || !err || C < 1 || s0 < 0 ||
      lse_ld < C || s0 + C > (int64_t)INT32_MAX - 128)
    return TT_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_path) || !aligned16(v_path) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk_acc) || !aligned16(dv_acc))
    return TT_ERR_INVALID_ARG;
  if (tc::bwd_ws_bytes(C, Hq) > kNoAllocScratchFloats * sizeof(float)) return TT_ERR_WORKSPACE;
  void* ws = nullptr;
  const int rc = noalloc_scratch(&ws);
  if (rc != TT_OK) return rc;
  // The pre-kernel of the backward rewrites every scratch entry this call
  // reads (padding rows included), so nothing needs clearing between calls.
  return tc::bwd_chunk(q, C, s0, k_path, v_path, nullptr, nullptr, o, lse, lse_ld, dO, dq, dk_acc, dv_acc, Hq, Hkv, d, scale,
                       ws, err, reinterpret_cast<cudaStream_t>(stream));
}
