// Internal helpers shared by the libtt CUDA sources (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tt.h"

namespace tt {

// First error wins: kernels record a device-detected error in the caller's word.
__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

static inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? TT_OK : TT_ERR_CUDA; }

#define TT_LAUNCH_CHECK()                                   \
  do {                                                      \
    cudaError_t e_ = cudaGetLastError();                    \
    if (e_ != cudaSuccess) return TT_ERR_CUDA;              \
  } while (0)

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side per-device caches (kernel attributes, SM counts, occupancy) are
// indexed by the current device's ordinal; devices at or beyond kMaxDevices
// are rejected with TT_ERR_CUDA.
constexpr int kMaxDevices = 64;
// Ordinal of the current device, or -1 if it cannot be read or is >= kMaxDevices.
int current_device();
// Multiprocessor count of the current device (cached per device; 1 if unknown).
int sm_count();

// loss = −Σ_t w_t·logp_t (weights NULL = ones) into one device double, fixed
// summation order (logprob.cu).
cudaError_t launch_weighted_loss(const float* logp, const float* weights, int64_t N, double* loss, cudaStream_t st);

// Brackets one kernel launch with CUDA events on its stream while launch
// timing is on (tt_kernel_timing); `cls` is a TT_KT_* kernel class.
class KtScope {
 public:
  KtScope(int cls, cudaStream_t st);
  ~KtScope();
  KtScope(const KtScope&) = delete;
  KtScope& operator=(const KtScope&) = delete;

 private:
  int slot_;
  cudaStream_t st_;
};

// ------------------------------------------------------------------ tree workspace
// Device workspace written by tt_tree_build and read by the attention calls.
// Header (int64): [0] magic, [1] N, [2] S, [3] valid flag, [4] B.
constexpr int64_t kTreeMagic = 0x7474726565777331LL;  // "ttreews1"
constexpr int kTile = 128;                           // schedule granularity (rows)

struct TreeWs {
  size_t hdr, send, blk_min, blk_max, fwd_cnt, fwd_order, bwd_cnt, bwd_order;
  // build-time scratch
  size_t child_ptr, child_idx, sub, dfs_seg, dfs_start, ivcnt, total;
};

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static inline TreeWs tree_ws_layout(int64_t S, int64_t N) {
  TreeWs w;
  const int64_t nT = (N + kTile - 1) / kTile;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, 256); return r; };
  w.hdr = take(8 * sizeof(int64_t));
  w.send = take(sizeof(int32_t) * nT * kTile);  // zero-padded to whole 128-key blocks
  w.blk_min = take(sizeof(int32_t) * nT);
  w.blk_max = take(sizeof(int32_t) * nT);
  w.fwd_cnt = take(sizeof(int32_t) * nT);
  w.fwd_order = take(sizeof(int32_t) * nT);
  w.bwd_cnt = take(sizeof(int32_t) * nT);
  w.bwd_order = take(sizeof(int32_t) * nT);
  w.child_ptr = take(sizeof(int32_t) * (S + 1));
  w.child_idx = take(sizeof(int32_t) * (S + 1));
  w.sub = take(sizeof(int64_t) * S);
  w.dfs_seg = take(sizeof(int32_t) * S);
  w.dfs_start = take(sizeof(int64_t) * S);
  w.ivcnt = take(sizeof(int32_t) * S);
  w.total = o;
  return w;
}

template <typename T>
static inline T* ws_at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }
template <typename T>
static inline const T* ws_at(const void* ws, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(ws) + off);
}

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace tt
