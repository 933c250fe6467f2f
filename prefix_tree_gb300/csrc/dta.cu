// Path-at-a-time tree attention (AReaL-DTA).
//
// "AREAL-DTA: Dynamic Tree Attention for Efficient Reinforcement Learning of
// Large Language Models", Key Contributions 1–2 and "Methodology in Plain
// English": walk the rollout tree depth-first keeping only the current
// root-to-node path (its tokens' K/V as a stack); forward each new segment
// against the cached path; once every descendant is done, backpropagate the
// segment (long segments in fixed-size query chunks, right to left) with the
// gradients of all descendant leaves already accumulated into the path, then
// pop it. Peak device memory is one path, not the tree.
//
// Host-side traversal (C++), device work on the caller's stream: D2D copies
// onto the path stack, chunk forward/backward kernels, fp32→bf16 conversion
// of completed key/value gradients. The visiting order ("Key Contributions" 2:
// visits reordered so that consecutive leaves share as much prefix as
// possible) is greedy: every DFS order gives consecutive leaves the same total
// shared prefix, so the greedy choice only settles ties, taken as longest root
// path first, then lowest segment index: at each segment the children are
// entered by decreasing depth (tokens) of their subtree's deepest leaf, ties
// by that leaf's index. Ascending segment index (the DFS layout's own order)
// is the alternative.
#include <algorithm>
#include <new>
#include <vector>

#include "common.cuh"

namespace tt {
namespace {

struct HostTree {
  int S = 0;
  int64_t N = 0, maxpath = 0;
  std::vector<int> parent, len, child_ptr, child_idx;
  std::vector<int64_t> start, pathlen;
  std::vector<int64_t> deep;   // tokens on the root path of the deepest leaf below each segment
  std::vector<int> deep_leaf;  // that leaf (lowest index among the deepest)
};

bool host_tree(const int32_t* parent, const int32_t* len, int32_t S, HostTree& t) {
  if (!parent || !len || S < 1 || parent[0] != -1) return false;
  t.S = S;
  t.parent.assign(parent, parent + S);
  t.len.assign(len, len + S);
  for (int s = 0; s < S; ++s) {
    if (len[s] < 1) return false;
    if (s > 0 && (parent[s] < 0 || parent[s] >= s)) return false;
    t.N += len[s];
  }
  t.child_ptr.assign(S + 1, 0);
  for (int s = 1; s < S; ++s) t.child_ptr[parent[s] + 1]++;
  for (int s = 0; s < S; ++s) t.child_ptr[s + 1] += t.child_ptr[s];
  t.child_idx.assign(S > 1 ? S - 1 : 1, 0);
  std::vector<int> fill(t.child_ptr.begin(), t.child_ptr.end() - 1);
  for (int s = 1; s < S; ++s) t.child_idx[fill[parent[s]]++] = s;
  std::vector<int64_t> sub(t.len.begin(), t.len.end());
  for (int s = S - 1; s > 0; --s) sub[parent[s]] += sub[s];
  t.start.assign(S, 0);
  t.pathlen.assign(S, 0);
  std::vector<int64_t> cur(S, 0);
  cur[0] = len[0];
  for (int s = 1; s < S; ++s) {
    const int p = parent[s];
    t.start[s] = cur[p];
    cur[p] += sub[s];
    cur[s] = t.start[s] + len[s];
    t.pathlen[s] = t.pathlen[p] + len[p];
  }
  for (int s = 0; s < S; ++s) t.maxpath = std::max<int64_t>(t.maxpath, t.pathlen[s] + len[s]);
  // deepest leaf of every subtree (children have larger indices than their parent)
  t.deep.assign(S, -1);
  t.deep_leaf.assign(S, S);
  for (int s = S - 1; s >= 0; --s) {
    if (t.child_ptr[s + 1] == t.child_ptr[s]) {
      t.deep[s] = t.pathlen[s] + len[s];
      t.deep_leaf[s] = s;
    }
    if (s > 0) {
      const int p = parent[s];
      if (t.deep[s] > t.deep[p] || (t.deep[s] == t.deep[p] && t.deep_leaf[s] < t.deep_leaf[p])) {
        t.deep[p] = t.deep[s];
        t.deep_leaf[p] = t.deep_leaf[s];
      }
    }
  }
  return true;
}

// Children of every segment in visiting order: ascending index (order 0) or
// greedy (order 1: deepest leaf first, ties by its index).
void order_children(HostTree& t, int order) {
  if (order != 1) return;
  for (int s = 0; s < t.S; ++s) {
    auto b = t.child_idx.begin() + t.child_ptr[s], e = t.child_idx.begin() + t.child_ptr[s + 1];
    std::stable_sort(b, e, [&](int x, int y) {
      return t.deep[x] != t.deep[y] ? t.deep[x] > t.deep[y] : t.deep_leaf[x] < t.deep_leaf[y];
    });
  }
}

struct DtaWs {
  size_t kst, vst, dka, dva, dsum, total;
};
DtaWs dta_layout(int64_t maxpath, int64_t chunk, int Hq, int Hkv, int d) {
  DtaWs w;
  const size_t rowk = (size_t)Hkv * d;
  size_t o = 0;
  auto take = [&](size_t b) { size_t r = o; o = align_up(o + b, 256); return r; };
  w.kst = take(maxpath * rowk * 2);
  w.vst = take(maxpath * rowk * 2);
  w.dka = take(maxpath * rowk * 4);
  w.dva = take(maxpath * rowk * 4);
  w.dsum = take(tt_tree_attn_chunk_bwd_workspace_bytes(chunk, Hq));
  w.total = o;
  return w;
}

__global__ void f32_to_bf16_kernel(const float* a, const float* b, __nv_bfloat16* x, __nv_bfloat16* y, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
  if (i >= n) return;
  const float2 u = *reinterpret_cast<const float2*>(a + i);
  const float2 v = *reinterpret_cast<const float2*>(b + i);
  *reinterpret_cast<__nv_bfloat162*>(x + i) = __floats2bfloat162_rn(u.x, u.y);
  *reinterpret_cast<__nv_bfloat162*>(y + i) = __floats2bfloat162_rn(v.x, v.y);
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API size_t tt_dta_workspace_bytes(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S,
                                     int64_t chunk, int Hq, int Hkv, int d) {
  HostTree t;
  if (chunk < 1 || Hq < 1 || Hkv < 1 || d < 1 || !host_tree(seg_parent_host, seg_len_host, S, t)) return 0;
  return dta_layout(t.maxpath, chunk, Hq, Hkv, d).total;
}

TT_API int tt_dta_leaf_order(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int order,
                             int32_t* leaves_host, int32_t capacity) {
  if (order != TT_DTA_ORDER_INDEX && order != TT_DTA_ORDER_GREEDY) return TT_ERR_INVALID_ARG;
  HostTree t;
  if (!host_tree(seg_parent_host, seg_len_host, S, t)) return TT_ERR_INVALID_TREE;
  order_children(t, order);
  std::vector<int> stack{0}, leaves;
  while (!stack.empty()) {
    const int s = stack.back();
    stack.pop_back();
    if (t.child_ptr[s + 1] == t.child_ptr[s]) leaves.push_back(s);
    for (int i = t.child_ptr[s + 1] - 1; i >= t.child_ptr[s]; --i) stack.push_back(t.child_idx[i]);
  }
  if (!leaves_host || capacity < (int64_t)leaves.size()) return TT_ERR_WORKSPACE;
  std::copy(leaves.begin(), leaves.end(), leaves_host);
  return (int)leaves.size();
}

TT_API int tt_dta_tree_attn(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                            int64_t chunk, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, const tt_bf16* dO,
                            tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int Hq, int Hkv, int d,
                            float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  return tt_dta_tree_attn_ordered(seg_parent_host, seg_len_host, S, N, chunk, TT_DTA_ORDER_GREEDY, Q, K, V, dO, O, LSE,
                                  dQ, dK, dV, Hq, Hkv, d, scale, ws, ws_bytes, err, stream);
}

// A plan: the traversal's device work for one tree, chunk size, order and
// set of buffers, captured once into a CUDA graph (copies, memsets and every
// chunk kernel as graph nodes); a launch replays it with one call, so the
// host walks the tree once and the GPU runs the ~3 launches per segment
// back to back.
struct tt_dta_plan_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

TT_API int tt_dta_plan_create(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                              int64_t chunk, int order, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                              const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int Hq,
                              int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                              tt_dta_plan* plan_out) {
  if (!plan_out) return TT_ERR_INVALID_ARG;
  *plan_out = nullptr;
  const int dev = current_device();
  if (dev < 0) return TT_ERR_CUDA;
  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return TT_ERR_CUDA;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return TT_ERR_CUDA;
  }
  const int rc = tt_dta_tree_attn_ordered(seg_parent_host, seg_len_host, S, N, chunk, order, Q, K, V, dO, O, LSE, dQ,
                                          dK, dV, Hq, Hkv, d, scale, ws, ws_bytes, err, reinterpret_cast<tt_stream_t>(cs));
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (rc != TT_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return rc != TT_OK ? rc : TT_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return TT_ERR_CUDA;
  }
  tt_dta_plan p = new (std::nothrow) tt_dta_plan_s;
  if (!p) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return TT_ERR_CUDA;
  }
  p->graph = g;
  p->exec = ex;
  p->device = dev;
  *plan_out = p;
  return TT_OK;
}

TT_API int tt_dta_plan_launch(tt_dta_plan plan, tt_stream_t stream) {
  if (!plan) return TT_ERR_INVALID_ARG;
  if (current_device() != plan->device) return TT_ERR_INVALID_ARG;
  return cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

TT_API int tt_dta_plan_destroy(tt_dta_plan plan) {
  if (!plan) return TT_OK;
  const bool ok = cudaGraphExecDestroy(plan->exec) == cudaSuccess && cudaGraphDestroy(plan->graph) == cudaSuccess;
  delete plan;
  return ok ? TT_OK : TT_ERR_CUDA;
}

TT_API int tt_dta_tree_attn_ordered(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                                    int64_t chunk, int order, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                                    const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV,
                                    int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                                    tt_stream_t stream) {
  if (!Q || !K || !V || !dO || !O || !LSE || !dQ || !dK || !dV || !ws || !err || chunk < 1) return TT_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1) return TT_ERR_INVALID_ARG;
  if (order != TT_DTA_ORDER_INDEX && order != TT_DTA_ORDER_GREEDY) return TT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (d != 64 && d != 128)) return TT_ERR_UNSUPPORTED;
  HostTree t;
  if (!host_tree(seg_parent_host, seg_len_host, S, t) || t.N != N) return TT_ERR_INVALID_TREE;
  order_children(t, order);
  const DtaWs L = dta_layout(t.maxpath, chunk, Hq, Hkv, d);
  if (ws_bytes < L.total) return TT_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  tt_bf16* kst = reinterpret_cast<tt_bf16*>(w + L.kst);
  tt_bf16* vst = reinterpret_cast<tt_bf16*>(w + L.vst);
  float* dka = reinterpret_cast<float*>(w + L.dka);
  float* dva = reinterpret_cast<float*>(w + L.dva);
  void* dsum = w + L.dsum;
  const size_t dsum_bytes = tt_tree_attn_chunk_bwd_workspace_bytes(chunk, Hq);
  const int64_t rowk = (int64_t)Hkv * d, rowq = (int64_t)Hq * d;

  auto chunks = [&](int s, std::vector<std::pair<int64_t, int64_t>>& out) {
    out.clear();
    for (int64_t c0 = 0; c0 < t.len[s]; c0 += chunk) out.emplace_back(c0, std::min<int64_t>(chunk, t.len[s] - c0));
  };
  auto enter = [&](int s) -> int {
    const int64_t base = t.pathlen[s], L0 = t.len[s], st0 = t.start[s];
    if (cudaMemcpyAsync(kst + base * rowk, K + st0 * rowk, L0 * rowk * 2, cudaMemcpyDeviceToDevice, st) ||
        cudaMemcpyAsync(vst + base * rowk, V + st0 * rowk, L0 * rowk * 2, cudaMemcpyDeviceToDevice, st) ||
        cudaMemsetAsync(dka + base * rowk, 0, L0 * rowk * 4, st) ||
        cudaMemsetAsync(dva + base * rowk, 0, L0 * rowk * 4, st))
      return TT_ERR_CUDA;
    std::vector<std::pair<int64_t, int64_t>> cs;
    chunks(s, cs);
    for (auto& c : cs) {
      const int64_t row = st0 + c.first;
      const int rc = tt_tree_attn_chunk_fwd(Q + row * rowq, c.second, base + c.first, kst, vst, O + row * rowq,
                                            LSE + row, N, Hq, Hkv, d, scale, err, stream);
      if (rc) return rc;
    }
    return TT_OK;
  };
  auto leave = [&](int s) -> int {
    const int64_t base = t.pathlen[s], L0 = t.len[s], st0 = t.start[s];
    std::vector<std::pair<int64_t, int64_t>> cs;
    chunks(s, cs);
    for (auto it = cs.rbegin(); it != cs.rend(); ++it) {
      const int64_t row = st0 + it->first;
      const int rc = tt_tree_attn_chunk_bwd(Q + row * rowq, it->second, base + it->first, kst, vst, O + row * rowq,
                                            LSE + row, N, dO + row * rowq, dQ + row * rowq, dka, dva, Hq, Hkv, d,
                                            scale, dsum, dsum_bytes, err, stream);
      if (rc) return rc;
    }
    const int64_t n = L0 * rowk;
    f32_to_bf16_kernel<<<(unsigned)((n / 2 + 255) / 256), 256, 0, st>>>(
        dka + base * rowk, dva + base * rowk, reinterpret_cast<__nv_bfloat16*>(dK + st0 * rowk),
        reinterpret_cast<__nv_bfloat16*>(dV + st0 * rowk), n);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  };
  // Iterative DFS: (segment, next child slot); enter on push, leave on pop.
  std::vector<std::pair<int, int>> stack;
  int rc = enter(0);
  if (rc) return rc;
  stack.emplace_back(0, t.child_ptr[0]);
  while (!stack.empty()) {
    auto& top = stack.back();
    const int s = top.first;
    if (top.second < t.child_ptr[s + 1]) {
      const int c = t.child_idx[top.second++];
      rc = enter(c);
      if (rc) return rc;
      stack.emplace_back(c, t.child_ptr[c]);
    } else {
      rc = leave(s);
      if (rc) return rc;
      stack.pop_back();
    }
  }
  return TT_OK;
}
