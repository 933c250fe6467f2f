// Tree build: DFS serialisation of a rollout prefix tree and the tile schedules
// of the attention kernels.
//
// "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix Reuse",
// Abstract: the tokens of a task form a prefix tree; DFS serialization visits
// every token exactly once; each token's loss weight is the fraction of
// branches through it. Children are visited in ascending segment index.
//
// Kernels:
//   seg_kernel   (1 CTA)   validation, child lists, subtree sizes, DFS offsets
//                          by per-parent cursors, depth/path length, leaf
//                          counts, interval counts, stats
//   iv_kernel    (grid)    per-segment merged ancestor intervals (walk up)
//   tok_kernel   (grid)    per-token seg / pos / send / leafcnt / weight
//   blk_kernel   (grid)    per-128-row block min/max of send, backward ranges
//   fwdcnt_kernel(grid)    key blocks per query tile, non-empty tile pairs
//   order_kernel (grid)    longest-first tile orders (stable rank)
#include "common.cuh"

namespace tt {
namespace {

struct BuildArgs {
  const int32_t* parent;
  const int32_t* len;
  int32_t S;
  int64_t N;
  tt_tree_out out;
  int64_t iv_cap;
  char* ws;
  TreeWs L;
  int32_t* err;
};

__device__ __forceinline__ int64_t* hdr_of(const BuildArgs& a) { return reinterpret_cast<int64_t*>(a.ws + a.L.hdr); }
template <typename T>
__device__ __forceinline__ T* at(const BuildArgs& a, size_t off) { return reinterpret_cast<T*>(a.ws + off); }

__global__ void seg_kernel(BuildArgs a) {
  __shared__ int bad;
  __shared__ unsigned long long tokens;
  const int S = a.S;
  if (threadIdx.x == 0) { bad = 0; tokens = 0; }
  __syncthreads();
  unsigned long long mine = 0;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int p = a.parent[s];
    const int l = a.len[s];
    if ((s == 0 && p != -1) || (s > 0 && (p < 0 || p >= s)) || l < 1) bad = 1;
    mine += (l > 0 ? (unsigned long long)l : 0ull);
  }
  atomicAdd(&tokens, mine);
  __syncthreads();
  int64_t* hdr = hdr_of(a);
  if (threadIdx.x != 0) return;
  hdr[0] = kTreeMagic;
  hdr[1] = a.N;
  hdr[2] = S;
  if (bad || (int64_t)tokens != a.N) {
    hdr[3] = 0;
    set_err(a.err, TT_ERR_INVALID_TREE);
    return;
  }
  // Sequential O(S) passes (segment counts are small; the work is negligible).
  int32_t* child_ptr = at<int32_t>(a, a.L.child_ptr);
  int32_t* child_idx = at<int32_t>(a, a.L.child_idx);
  int64_t* sub = at<int64_t>(a, a.L.sub);
  int32_t* ivcnt = at<int32_t>(a, a.L.ivcnt);
  int32_t* start = a.out.seg_start;
  int32_t* send = a.out.seg_subtree_end;
  int32_t* depth = a.out.seg_depth;
  int32_t* plen = a.out.seg_pathlen;
  int32_t* leaf = a.out.seg_leafcnt;

  for (int s = 0; s <= S; ++s) child_ptr[s] = 0;
  for (int s = 1; s < S; ++s) child_ptr[a.parent[s] + 1]++;
  for (int s = 0; s < S; ++s) child_ptr[s + 1] += child_ptr[s];
  for (int s = 0; s < S; ++s) ivcnt[s] = child_ptr[s];  // temporary fill cursor
  for (int s = 1; s < S; ++s) child_idx[ivcnt[a.parent[s]]++] = s;  // ascending per parent

  for (int s = 0; s < S; ++s) sub[s] = a.len[s];
  for (int s = S - 1; s > 0; --s) sub[a.parent[s]] += sub[s];
  // DFS offsets: a parent's children, taken in ascending index, are laid out
  // back to back right after the parent's own tokens.
  int64_t* cursor = at<int64_t>(a, a.L.dfs_start);  // reused as cursor scratch first
  start[0] = 0;
  cursor[0] = a.len[0];
  depth[0] = 0;
  plen[0] = 0;
  for (int s = 1; s < S; ++s) {
    const int p = a.parent[s];
    start[s] = (int32_t)cursor[p];
    cursor[p] += sub[s];
    cursor[s] = (int64_t)start[s] + a.len[s];
    depth[s] = depth[p] + 1;
    plen[s] = plen[p] + a.len[p];
  }
  for (int s = 0; s < S; ++s) send[s] = (int32_t)(start[s] + sub[s]);
  for (int s = S - 1; s >= 0; --s) {
    const int nch = child_ptr[s + 1] - child_ptr[s];
    if (nch == 0) leaf[s] = 1;
    else {
      int c = 0;
      for (int i = child_ptr[s]; i < child_ptr[s + 1]; ++i) c += leaf[child_idx[i]];
      leaf[s] = c;
    }
  }
  // Segments in DFS order (explicit stack in child_idx order).
  int32_t* dfs_seg = at<int32_t>(a, a.L.dfs_seg);
  {
    int32_t* stack = at<int32_t>(a, a.L.ivcnt);  // S entries suffice: each segment pushed once
    int top = 0, n = 0;
    stack[top++] = 0;
    while (top > 0) {
      const int s = stack[--top];
      dfs_seg[n++] = s;
      for (int i = child_ptr[s + 1] - 1; i >= child_ptr[s]; --i) stack[top++] = child_idx[i];
    }
  }
  int64_t* dfs_start = at<int64_t>(a, a.L.dfs_start);
  for (int i = 0; i < S; ++i) dfs_start[i] = start[dfs_seg[i]];
  // Interval counts: a segment extends its parent's list, merging when the
  // parent's range ends exactly where the segment starts.
  int64_t total = 0;
  for (int s = 0; s < S; ++s) {
    ivcnt[s] = s == 0 ? 1 : ivcnt[a.parent[s]] + ((start[a.parent[s]] + a.len[a.parent[s]] == start[s]) ? 0 : 1);
  }
  a.out.iv_ptr[0] = 0;
  for (int s = 0; s < S; ++s) {
    total += ivcnt[s];
    a.out.iv_ptr[s + 1] = (int32_t)total;
  }
  // Stats.
  int64_t B = leaf[0], branch_tokens = 0, pairs = 0, maxpath = 0;
  int maxdepth = 0;
  for (int s = 0; s < S; ++s) {
    const int64_t l = a.len[s], pl = plen[s];
    pairs += l * pl + l * (l + 1) / 2;
    if (child_ptr[s + 1] == child_ptr[s]) {
      branch_tokens += pl + l;
      if (pl + l > maxpath) maxpath = pl + l;
    }
    if (depth[s] > maxdepth) maxdepth = depth[s];
  }
  int64_t* st = a.out.stats;
  st[0] = B; st[1] = a.N; st[2] = branch_tokens; st[3] = pairs; st[4] = 0;
  st[5] = total; st[6] = maxdepth; st[7] = maxpath;
  hdr[4] = B;
  if (total > a.iv_cap) set_err(a.err, TT_ERR_WORKSPACE);
  hdr[3] = 1;
}

__global__ void iv_kernel(BuildArgs a) {
  const int64_t* hdr = hdr_of(a);
  if (hdr[3] == 0) return;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= a.S || a.out.stats[5] > a.iv_cap) return;
  const int32_t* start = a.out.seg_start;
  // Walk from s up to the root, emitting merged intervals from the back.
  int w = a.out.iv_ptr[s + 1] - 1;
  int32_t b = start[s], e = start[s] + a.len[s];
  int x = s;
  while (a.parent[x] >= 0) {
    const int p = a.parent[x];
    const int32_t pb = start[p], pe = start[p] + a.len[p];
    if (pe == b) b = pb;
    else {
      a.out.iv[2 * w] = b; a.out.iv[2 * w + 1] = e; --w;
      b = pb; e = pe;
    }
    x = p;
  }
  a.out.iv[2 * w] = b; a.out.iv[2 * w + 1] = e;
}

__global__ void tok_kernel(BuildArgs a) {
  const int64_t* hdr = hdr_of(a);
  if (hdr[3] == 0) return;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= a.N) return;
  const int64_t* dfs_start = at<int64_t>(a, a.L.dfs_start);
  const int32_t* dfs_seg = at<int32_t>(a, a.L.dfs_seg);
  int lo = 0, hi = a.S - 1;  // last i with dfs_start[i] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (dfs_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int s = dfs_seg[lo];
  const int32_t sd = a.out.seg_subtree_end[s];
  const int32_t n = a.out.seg_leafcnt[s];
  a.out.tok_seg[t] = s;
  a.out.tok_pos[t] = a.out.seg_pathlen[s] + (int32_t)(t - a.out.seg_start[s]);
  a.out.tok_send[t] = sd;
  a.out.tok_leafcnt[t] = n;
  a.out.tok_weight[t] = __fdiv_rn((float)n, (float)hdr[4]);
  at<int32_t>(a, a.L.send)[t] = sd;
}

__global__ void blk_kernel(BuildArgs a) {
  const int64_t* hdr = hdr_of(a);
  if (hdr[3] == 0) return;
  const int b = blockIdx.x;
  const int64_t t = (int64_t)b * kTile + threadIdx.x;
  int32_t* send = at<int32_t>(a, a.L.send);
  int mn = INT32_MAX, mx = 0;
  if (t < a.N) { mn = send[t]; mx = send[t]; }
  else send[t] = 0;  // padding keys are never visible
  for (int o = 16; o; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __shared__ int smn[kTile / 32], smx[kTile / 32];
  if ((threadIdx.x & 31) == 0) { smn[threadIdx.x >> 5] = mn; smx[threadIdx.x >> 5] = mx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    mn = smn[0]; mx = smx[0];
    for (int i = 1; i < kTile / 32; ++i) { mn = min(mn, smn[i]); mx = max(mx, smx[i]); }
    at<int32_t>(a, a.L.blk_min)[b] = mn;
    at<int32_t>(a, a.L.blk_max)[b] = mx;
    // queries of this key block: the contiguous range [b*128, mx)
    at<int32_t>(a, a.L.bwd_cnt)[b] = (mx + kTile - 1) / kTile - b;
  }
}

__global__ void fwdcnt_kernel(BuildArgs a, int nT) {
  const int64_t* hdr = hdr_of(a);
  if (hdr[3] == 0) return;
  const int T = blockIdx.x * blockDim.x + threadIdx.x;
  if (T >= nT) return;
  const int32_t* blk_max = at<int32_t>(a, a.L.blk_max);
  const int64_t q0 = (int64_t)T * kTile;
  int c = 0;
  for (int b = 0; b <= T; ++b) c += blk_max[b] > q0;
  at<int32_t>(a, a.L.fwd_cnt)[T] = c;
  atomicAdd(reinterpret_cast<unsigned long long*>(&a.out.stats[4]), (unsigned long long)c);
}

// Longest-first order: rank_i = #{j : cnt_j > cnt_i or (cnt_j == cnt_i and j < i)}.
__global__ void order_kernel(BuildArgs a, int nT) {
  const int64_t* hdr = hdr_of(a);
  if (hdr[3] == 0) return;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int which = blockIdx.y;
  const int32_t* cnt = at<int32_t>(a, which == 0 ? a.L.fwd_cnt : a.L.bwd_cnt);
  int32_t* order = at<int32_t>(a, which == 0 ? a.L.fwd_order : a.L.bwd_order);
  if (i >= nT) return;
  const int ci = cnt[i];
  int r = 0;
  for (int j = 0; j < nT; ++j) {
    const int cj = cnt[j];
    r += (cj > ci) || (cj == ci && j < i);
  }
  order[r] = i;
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API size_t tt_tree_workspace_bytes(int32_t S, int64_t N) {
  if (S < 1 || N < 1) return 0;
  return tree_ws_layout(S, N).total;
}

TT_API int tt_tree_build(const int32_t* seg_parent, const int32_t* seg_len, int32_t S, int64_t N,
                         const tt_tree_out* out, int64_t iv_capacity, void* ws, size_t ws_bytes, int32_t* err,
                         tt_stream_t stream) {
  if (!seg_parent || !seg_len || !out || !ws || !err || S < 1 || N < 1 || N > INT32_MAX - kTile || iv_capacity < 0)
    return TT_ERR_INVALID_ARG;
  const tt_tree_out& o = *out;
  if (!o.seg_start || !o.seg_subtree_end || !o.seg_depth || !o.seg_pathlen || !o.seg_leafcnt || !o.iv_ptr ||
      (!o.iv && iv_capacity > 0) || !o.tok_seg || !o.tok_pos || !o.tok_send || !o.tok_leafcnt || !o.tok_weight ||
      !o.stats)
    return TT_ERR_INVALID_ARG;
  BuildArgs a;
  a.parent = seg_parent; a.len = seg_len; a.S = S; a.N = N; a.out = o; a.iv_cap = iv_capacity;
  a.ws = static_cast<char*>(ws); a.L = tree_ws_layout(S, N); a.err = err;
  if (ws_bytes < a.L.total) return TT_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int nT = (int)((N + kTile - 1) / kTile);
  seg_kernel<<<1, 256, 0, st>>>(a);
  iv_kernel<<<(S + 127) / 128, 128, 0, st>>>(a);
  tok_kernel<<<(unsigned)((N + 255) / 256), 256, 0, st>>>(a);
  blk_kernel<<<nT, kTile, 0, st>>>(a);
  fwdcnt_kernel<<<(nT + 127) / 128, 128, 0, st>>>(a, nT);
  order_kernel<<<dim3((nT + 127) / 128, 2), 128, 0, st>>>(a, nT);
  TT_LAUNCH_CHECK();
  return TT_OK;
}

TT_API int tt_tree_schedules(const void* ws, int64_t N, int32_t* send, int32_t* blk_min, int32_t* blk_max,
                             int32_t* fwd_cnt, int32_t* fwd_order, int32_t* bwd_cnt, int32_t* bwd_order,
                             tt_stream_t stream) {
  if (!ws || N < 1 || N > INT32_MAX - kTile) return TT_ERR_INVALID_ARG;
  const TreeWs L = tree_ws_layout(0, N);
  const int64_t nT = (N + kTile - 1) / kTile;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(ws);
  struct Part {
    int32_t* dst;
    size_t off;
    int64_t n;
  } parts[] = {{send, L.send, nT * kTile}, {blk_min, L.blk_min, nT}, {blk_max, L.blk_max, nT},
               {fwd_cnt, L.fwd_cnt, nT},    {fwd_order, L.fwd_order, nT}, {bwd_cnt, L.bwd_cnt, nT},
               {bwd_order, L.bwd_order, nT}};
  for (const Part& p : parts) {
    if (!p.dst) continue;
    if (cudaMemcpyAsync(p.dst, w + p.off, (size_t)p.n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return TT_ERR_CUDA;
  }
  return TT_OK;
}
