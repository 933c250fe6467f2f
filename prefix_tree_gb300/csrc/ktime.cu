// Launch timing: CUDA events around the launches of the attention and
// log-prob kernels, so that a caller can measure one kernel class's device
// time inside a larger sequence of calls (the path-at-a-time driver's chunk
// launches, the backward's launch) on the stream each kernel runs on. Off by
// default; while off a scope costs one relaxed load.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace tt {
namespace {

constexpr int kMaxRecords = 65536;

struct Record {
  int cls;
  cudaEvent_t ev0, ev1;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Record> g_pool;  // events are created once and reused
int g_used = 0;
int64_t g_dropped = 0;

}  // namespace

KtScope::KtScope(int cls, cudaStream_t st) : slot_(-1), st_(st) {
  if (!__atomic_load_n(&g_on, __ATOMIC_RELAXED)) return;
  // launches captured into a graph (tt_dta_plan_create) are not timed
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on) return;
  if (g_used >= kMaxRecords) {
    ++g_dropped;
    return;
  }
  if (g_used == (int)g_pool.size()) {
    Record r{cls, nullptr, nullptr};
    if (cudaEventCreate(&r.ev0) != cudaSuccess || cudaEventCreate(&r.ev1) != cudaSuccess) {
      ++g_dropped;
      return;
    }
    g_pool.push_back(r);
  }
  g_pool[g_used].cls = cls;
  if (cudaEventRecord(g_pool[g_used].ev0, st) != cudaSuccess) {
    ++g_dropped;
    return;
  }
  slot_ = g_used++;
}

KtScope::~KtScope() {
  if (slot_ < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(g_pool[slot_].ev1, st_);
}

}  // namespace tt

using namespace tt;

TT_API int tt_kernel_timing(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (on) {
    g_used = 0;
    g_dropped = 0;
  }
  __atomic_store_n(&g_on, on != 0, __ATOMIC_RELAXED);
  return TT_OK;
}

TT_API int tt_kernel_timing_read(double* ms_host, int64_t* launches_host, int n, int64_t* dropped_host) {
  if (!ms_host || !launches_host || n < 0) return TT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int c = 0; c < n; ++c) {
    ms_host[c] = 0.0;
    launches_host[c] = 0;
  }
  for (int i = 0; i < g_used; ++i) {
    const Record& r = g_pool[i];
    if (cudaEventSynchronize(r.ev1) != cudaSuccess) return TT_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.ev0, r.ev1) != cudaSuccess) return TT_ERR_CUDA;
    if (r.cls >= 0 && r.cls < n) {
      ms_host[r.cls] += ms;
      launches_host[r.cls] += 1;
    }
  }
  if (dropped_host) *dropped_host = g_dropped;
  return TT_OK;
}
