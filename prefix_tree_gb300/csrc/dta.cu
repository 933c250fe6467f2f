// Path-at-a-time tree attention (AReaL-DTA).
//
// "AREAL-DTA: Dynamic Tree Attention for Efficient Reinforcement Learning of
// Large Language Models", Key Contributions 1–2 and "Methodology in Plain
// English": walk the rollout tree depth-first keeping only the current
// root-to-node path (its tokens' K/V as a stack); forward each new segment
// against the cached path; once every descendant is done, backpropagate the
// segment (long segments in fixed-size query chunks, right to left) with the
// gradients of all descendant leaves already accumulated into the path, then
// pop it. Peak device memory is one path per slot, not the tree: sibling
// leaves can run on up to `slots` path stacks at once (dta_run). Sibling
// leaves that lie next to each other in the DFS layout are also packed into
// one chunk of at most `chunk` rows behind their shared path (each leaf
// seeing the path and itself), so a stack holds at most its parent's path
// plus one chunk.
//
// Host-side traversal (C++), device work on the caller's stream: D2D copies
// onto the path stack, chunk forward/backward kernels, fp32→bf16 conversion
// of completed key/value gradients. The visiting order ("Key Contributions" 2:
// visits reordered so that each leaf and the next one have the longest
// possible common prefix) is greedy: every DFS order gives consecutive leaves the same total
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
  std::vector<int64_t> sub;    // rows of each segment's subtree (contiguous in the layout from start)
  std::vector<int> nseg;       // segments of each segment's subtree
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
  t.sub.assign(t.len.begin(), t.len.end());
  t.nseg.assign(S, 1);
  for (int s = S - 1; s > 0; --s) {
    t.sub[parent[s]] += t.sub[s];
    t.nseg[parent[s]] += t.nseg[s];
  }
  const std::vector<int64_t>& sub = t.sub;
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

constexpr int kMaxSlots = 8;
constexpr int kMaxPackSegs = 64;  // segments of one packed chunk

// Redundancy-free tree partitioning ("Tree Training", Abstract; the rule is
// this library's reading). A subtree is packable when it holds at most
// `budget` rows (the chunk size) and kMaxPackSegs segments. The traversal
// visits the segments that are not packable (their own rows in chunks of at
// most `budget` queries against their root path); the children of such a
// segment are taken in visiting order, and each run of consecutive packable
// children is cut into packs: whole sibling subtrees adjacent in the DFS
// layout (taken in layout order), at most `budget` rows and kMaxPackSegs
// segments per pack. A pack is processed as one chunk behind its parent's
// root path, every query seeing its ancestors only. If the whole tree is
// packable it is one pack with an empty path. Every row lies in exactly one
// chunk or pack, so no pair is computed twice, and a stack holds one root
// path plus at most `budget` rows.
bool packable(const HostTree& t, int c, int64_t budget) { return t.sub[c] <= budget && t.nseg[c] <= kMaxPackSegs; }
bool is_leaf(const HostTree& t, int s) { return t.child_ptr[s + 1] == t.child_ptr[s]; }

struct Pack {
  int64_t s0, st0, C;      // path rows; first layout row; rows
  int nseg;                // segments in its subtrees
  std::vector<int> roots;  // its sibling subtrees, in layout order
};
// A run of packable children of one segment -> packs, in layout order.
void pack_run(const HostTree& t, std::vector<int> run, int64_t budget, std::vector<Pack>& out) {
  out.clear();
  std::sort(run.begin(), run.end(), [&](int x, int y) { return t.start[x] < t.start[y]; });
  for (int c : run) {
    if (!out.empty()) {
      Pack& P = out.back();
      if (t.start[c] == P.st0 + P.C && P.C + t.sub[c] <= budget && P.nseg + t.nseg[c] <= kMaxPackSegs) {
        P.C += t.sub[c];
        P.nseg += t.nseg[c];
        P.roots.push_back(c);
        continue;
      }
    }
    out.push_back(Pack{t.pathlen[c], t.start[c], t.sub[c], t.nseg[c], {c}});
  }
}

// The partitions of the traversal, in layout order: packs (kind 0) and the
// chunks of the segments that are not packable (kind 1).
struct Part {
  int64_t first, rows, path;
  int kind;
};
void tree_partitions(const HostTree& t, int64_t budget, std::vector<Part>& out) {
  out.clear();
  if (packable(t, 0, budget)) {
    out.push_back(Part{0, t.N, 0, 0});
    return;
  }
  std::vector<int> stack{0}, run;
  std::vector<Pack> packs;
  auto close_run = [&]() {
    pack_run(t, run, budget, packs);
    run.clear();
    for (const Pack& P : packs) out.push_back(Part{P.st0, P.C, P.s0, 0});
  };
  while (!stack.empty()) {
    const int s = stack.back();
    stack.pop_back();
    for (int64_t c0 = 0; c0 < t.len[s]; c0 += budget)
      out.push_back(Part{t.start[s] + c0, std::min<int64_t>(budget, t.len[s] - c0), t.pathlen[s] + c0, 1});
    for (int i = t.child_ptr[s]; i < t.child_ptr[s + 1]; ++i) {
      const int c = t.child_idx[i];
      if (packable(t, c, budget)) {
        run.push_back(c);
        continue;
      }
      close_run();
      stack.push_back(c);
    }
    close_run();
  }
  std::sort(out.begin(), out.end(), [](const Part& x, const Part& y) { return x.first < y.first; });
}

// Rows of a path stack: the longest root-to-leaf path, a segment's path plus
// one budget of its packable children, or the whole tree when it is one pack.
int64_t stack_rows(const HostTree& t, int64_t budget) {
  if (packable(t, 0, budget)) return t.N;
  std::vector<int64_t> packsum(t.S, 0);
  for (int s = 1; s < t.S; ++s)
    if (packable(t, s, budget)) packsum[t.parent[s]] += t.sub[s];
  int64_t r = t.maxpath;
  for (int p = 0; p < t.S; ++p)
    if (packsum[p] > 0) r = std::max<int64_t>(r, t.pathlen[p] + t.len[p] + std::min<int64_t>(budget, packsum[p]));
  return r;
}

struct DtaWs {
  size_t kst, vst, dka, dva, snd, bmax, dsum, slot, total;  // offsets within a slot; bytes of a slot and of all slots
};
DtaWs dta_layout(int64_t rows, int64_t chunk, int Hq, int Hkv, int d, int slots) {
  DtaWs w;
  const size_t rowk = (size_t)Hkv * d;
  const size_t nblk = (size_t)(rows + 127) / 128;
  size_t o = 0;
  auto take = [&](size_t b) { size_t r = o; o = align_up(o + b, 256); return r; };
  w.kst = take(rows * rowk * 2);
  w.vst = take(rows * rowk * 2);
  w.dka = take(rows * rowk * 4);
  w.dva = take(rows * rowk * 4);
  w.snd = take(nblk * 128 * 4);  // send of a packed chunk, by stack row
  w.bmax = take(nblk * 4);       // its maximum per 128-row block
  w.dsum = take(tt_tree_attn_chunk_bwd_workspace_bytes(chunk, Hq));
  w.slot = o;
  w.total = o * (size_t)slots;
  return w;
}

// The send values and block maxima a packed chunk reads: one CTA of 128
// threads per 128-row block from floor(s0/128) to the block holding s0 + C − 1.
// send = INT32_MAX on the path, s0 + the local end of the subtree of a row's
// segment on the chunk, 0 past it.
struct PackSegs {
  int32_t n;
  int32_t start[kMaxPackSegs];  // local first row of each segment, increasing
  int32_t end[kMaxPackSegs];    // local end of its subtree
};
__global__ void pack_send_kernel(int32_t* snd, int32_t* bmax, int64_t s0, int64_t C, PackSegs ps) {
  __shared__ int32_t wmax[4];
  const int64_t b = s0 / 128 + blockIdx.x;
  const int64_t k = b * 128 + threadIdx.x;
  int32_t v = 0;
  if (k < s0) {
    v = INT32_MAX;
  } else if (k < s0 + C) {
    const int64_t i = k - s0;
    int j = 0;
    while (j + 1 < ps.n && ps.start[j + 1] <= i) ++j;
    v = (int32_t)(s0 + ps.end[j]);
  }
  snd[k] = v;
  const int32_t m = __reduce_max_sync(0xffffffffu, v);
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) bmax[b] = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
}

__global__ void f32_to_bf16_kernel(const float* a, const float* b, __nv_bfloat16* x, __nv_bfloat16* y, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;
  if (i >= n) return;
  const float2 u = *reinterpret_cast<const float2*>(a + i);
  const float2 v = *reinterpret_cast<const float2*>(b + i);
  *reinterpret_cast<__nv_bfloat162*>(x + i) = __floats2bfloat162_rn(u.x, u.y);
  *reinterpret_cast<__nv_bfloat162*>(y + i) = __floats2bfloat162_rn(v.x, v.y);
}

// a[i] += b[i], b[i] = 0 for the dK and dV accumulators (float4 units): a
// slot's sums over the shared prefix folded into slot 0.
__global__ void fold_kernel(float4* ak, float4* bk, float4* av, float4* bv, int64_t n4) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 x = ak[i], y = bk[i];
  ak[i] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
  bk[i] = z;
  x = av[i];
  y = bv[i];
  av[i] = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
  bv[i] = z;
}

struct DtaArgs {
  int64_t N, chunk;
  const tt_bf16 *Q, *K, *V, *dO;
  tt_bf16 *O, *dQ, *dK, *dV;
  float* LSE;
  int Hq, Hkv, d;
  float scale;
  int32_t* err;
};

// The traversal (the partitions of tree_partitions, in visiting order). A
// packable root is one pack. Otherwise segments that are not packable are
// entered and left on stream st with slot 0's stack; their K/V and zeroed
// accumulators are put into every slot, so that any slot holds the whole path
// above them. Each run of consecutive packable children (visiting order) is
// cut into packs (pack_run), each run as one packed chunk (a single leaf as a
// plain segment). When a segment's children are balanced (no unit — a child
// subtree that is not packable, or a pack — holds more than half of their
// attention work), all units are spread over the slots at once (longest first
// onto the least-loaded slot) and each slot runs its units whole, one after
// the other, on its own stream and stack. Otherwise the children are visited
// in order: those that are not packable recursively on st, and the packs of
// each run spread over the slots (pack i on slot i mod k). Either way,
// afterwards slots 1..k−1's sums over the shared path are added into slot 0's
// in slot order (then zeroed), so results do not depend on timing.
// `side` holds k streams (k > 1); events are appended to `events` for the
// caller to destroy (after a graph capture has ended).
int dta_run(const HostTree& t, const DtaArgs& A, char* ws, const DtaWs& L, int slots, cudaStream_t st,
            const std::vector<cudaStream_t>& side, std::vector<cudaEvent_t>& events) {
  struct Slot {
    tt_bf16 *kst, *vst;
    float *dka, *dva;
    int32_t *snd, *bmax;
    void* dsum;
  };
  std::vector<Slot> sl(slots);
  for (int j = 0; j < slots; ++j) {
    char* w = ws + (size_t)j * L.slot;
    sl[j] = {reinterpret_cast<tt_bf16*>(w + L.kst), reinterpret_cast<tt_bf16*>(w + L.vst),
             reinterpret_cast<float*>(w + L.dka), reinterpret_cast<float*>(w + L.dva),
             reinterpret_cast<int32_t*>(w + L.snd), reinterpret_cast<int32_t*>(w + L.bmax), w + L.dsum};
  }
  const size_t dsum_bytes = tt_tree_attn_chunk_bwd_workspace_bytes(A.chunk, A.Hq);
  const int64_t rowk = (int64_t)A.Hkv * A.d, rowq = (int64_t)A.Hq * A.d;
  auto chunks = [&](int s, std::vector<std::pair<int64_t, int64_t>>& out) {
    out.clear();
    for (int64_t c0 = 0; c0 < t.len[s]; c0 += A.chunk) out.emplace_back(c0, std::min<int64_t>(A.chunk, t.len[s] - c0));
  };
  // attention work (ancestor pairs) of each segment's subtree
  std::vector<double> work(t.S, 0.0);
  for (int s = t.S - 1; s >= 0; --s) {
    work[s] += (double)t.len[s] * ((double)t.pathlen[s] + 0.5 * (double)(t.len[s] + 1));
    if (s > 0) work[t.parent[s]] += work[s];
  }
  auto put = [&](int s, const Slot& x, cudaStream_t q) -> int {
    const int64_t base = t.pathlen[s], L0 = t.len[s], st0 = t.start[s];
    if (cudaMemcpyAsync(x.kst + base * rowk, A.K + st0 * rowk, L0 * rowk * 2, cudaMemcpyDeviceToDevice, q) ||
        cudaMemcpyAsync(x.vst + base * rowk, A.V + st0 * rowk, L0 * rowk * 2, cudaMemcpyDeviceToDevice, q) ||
        cudaMemsetAsync(x.dka + base * rowk, 0, L0 * rowk * 4, q) || cudaMemsetAsync(x.dva + base * rowk, 0, L0 * rowk * 4, q))
      return TT_ERR_CUDA;
    return TT_OK;
  };
  auto fwd_seg = [&](int s, const Slot& x, cudaStream_t q) -> int {
    const int64_t base = t.pathlen[s], st0 = t.start[s];
    std::vector<std::pair<int64_t, int64_t>> cs;
    chunks(s, cs);
    for (auto& c : cs) {
      const int64_t row = st0 + c.first;
      const int rc = tt_tree_attn_chunk_fwd(A.Q + row * rowq, c.second, base + c.first, x.kst, x.vst, A.O + row * rowq,
                                            A.LSE + row, A.N, A.Hq, A.Hkv, A.d, A.scale, A.err,
                                            reinterpret_cast<tt_stream_t>(q));
      if (rc) return rc;
    }
    return TT_OK;
  };
  auto bwd_seg = [&](int s, const Slot& x, cudaStream_t q) -> int {
    const int64_t base = t.pathlen[s], L0 = t.len[s], st0 = t.start[s];
    std::vector<std::pair<int64_t, int64_t>> cs;
    chunks(s, cs);
    for (auto it = cs.rbegin(); it != cs.rend(); ++it) {
      const int64_t row = st0 + it->first;
      const int rc = tt_tree_attn_chunk_bwd(A.Q + row * rowq, it->second, base + it->first, x.kst, x.vst,
                                            A.O + row * rowq, A.LSE + row, A.N, A.dO + row * rowq, A.dQ + row * rowq,
                                            x.dka, x.dva, A.Hq, A.Hkv, A.d, A.scale, x.dsum, dsum_bytes, A.err,
                                            reinterpret_cast<tt_stream_t>(q));
      if (rc) return rc;
    }
    const int64_t n = L0 * rowk;
    f32_to_bf16_kernel<<<(unsigned)((n / 2 + 255) / 256), 256, 0, q>>>(
        x.dka + base * rowk, x.dva + base * rowk, reinterpret_cast<__nv_bfloat16*>(A.dK + st0 * rowk),
        reinterpret_cast<__nv_bfloat16*>(A.dV + st0 * rowk), n);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  };
  // a leaf: enter and leave
  auto leaf_seg = [&](int c, const Slot& x, cudaStream_t q) -> int {
    int rc = put(c, x, q);
    if (!rc) rc = fwd_seg(c, x, q);
    if (!rc) rc = bwd_seg(c, x, q);
    return rc;
  };
  // a pack of subtrees: its rows onto the stack, its send values and block
  // maxima, one packed chunk forward and backward, its key/value gradients out
  auto run_packed = [&](const Pack& P, const Slot& x, cudaStream_t q) -> int {
    const int64_t s0 = P.s0, C = P.C, st0 = P.st0;
    if (cudaMemcpyAsync(x.kst + s0 * rowk, A.K + st0 * rowk, C * rowk * 2, cudaMemcpyDeviceToDevice, q) ||
        cudaMemcpyAsync(x.vst + s0 * rowk, A.V + st0 * rowk, C * rowk * 2, cudaMemcpyDeviceToDevice, q) ||
        cudaMemsetAsync(x.dka + s0 * rowk, 0, C * rowk * 4, q) || cudaMemsetAsync(x.dva + s0 * rowk, 0, C * rowk * 4, q))
      return TT_ERR_CUDA;
    // the pack's segments in layout order, with the local ends of their subtrees
    std::vector<int> segs, stk(P.roots.rbegin(), P.roots.rend());
    while (!stk.empty()) {
      const int u = stk.back();
      stk.pop_back();
      segs.push_back(u);
      for (int i = t.child_ptr[u + 1] - 1; i >= t.child_ptr[u]; --i) stk.push_back(t.child_idx[i]);
    }
    std::sort(segs.begin(), segs.end(), [&](int x1, int y1) { return t.start[x1] < t.start[y1]; });
    PackSegs ps{};
    ps.n = (int32_t)segs.size();
    for (size_t i = 0; i < segs.size(); ++i) {
      ps.start[i] = (int32_t)(t.start[segs[i]] - st0);
      ps.end[i] = (int32_t)(t.start[segs[i]] + t.sub[segs[i]] - st0);
    }
    const int64_t nblk = (s0 + C + 127) / 128 - s0 / 128;
    pack_send_kernel<<<(unsigned)nblk, 128, 0, q>>>(x.snd, x.bmax, s0, C, ps);
    if (cudaGetLastError() != cudaSuccess) return TT_ERR_CUDA;
    int rc = tt_tree_attn_chunk_fwd_packed(A.Q + st0 * rowq, C, s0, x.kst, x.vst, x.snd, x.bmax, A.O + st0 * rowq,
                                           A.LSE + st0, A.N, A.Hq, A.Hkv, A.d, A.scale, A.err,
                                           reinterpret_cast<tt_stream_t>(q));
    if (!rc)
      rc = tt_tree_attn_chunk_bwd_packed(A.Q + st0 * rowq, C, s0, x.kst, x.vst, x.snd, x.bmax, A.O + st0 * rowq,
                                         A.LSE + st0, A.N, A.dO + st0 * rowq, A.dQ + st0 * rowq, x.dka, x.dva, A.Hq,
                                         A.Hkv, A.d, A.scale, x.dsum, dsum_bytes, A.err,
                                         reinterpret_cast<tt_stream_t>(q));
    if (rc) return rc;
    const int64_t n = C * rowk;
    f32_to_bf16_kernel<<<(unsigned)((n / 2 + 255) / 256), 256, 0, q>>>(
        x.dka + s0 * rowk, x.dva + s0 * rowk, reinterpret_cast<__nv_bfloat16*>(A.dK + st0 * rowk),
        reinterpret_cast<__nv_bfloat16*>(A.dV + st0 * rowk), n);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  };
  // a single leaf runs as a segment (the plain chunk calls), anything else as a packed chunk
  auto run_pack = [&](const Pack& P, const Slot& x, cudaStream_t q) -> int {
    return P.roots.size() == 1 && is_leaf(t, P.roots[0]) ? leaf_seg(P.roots[0], x, q) : run_packed(P, x, q);
  };
  auto packable_c = [&](int c) { return packable(t, c, A.chunk); };
  auto enter_inner = [&](int s) -> int {
    for (int j = 0; j < slots; ++j) {
      const int rc = put(s, sl[j], st);
      if (rc) return rc;
    }
    return fwd_seg(s, sl[0], st);
  };
  auto event_on = [&](cudaStream_t q, cudaEvent_t* e) -> bool {
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
    events.push_back(*e);
    return cudaEventRecord(*e, q) == cudaSuccess;
  };
  // A whole subtree on one stack and stream, one segment after the other
  // (entered on push, left on pop).
  auto seq = [&](int c, const Slot& x, cudaStream_t q) -> int {
    std::vector<std::pair<int, int>> stk;
    int rc = put(c, x, q);
    if (!rc) rc = fwd_seg(c, x, q);
    if (rc) return rc;
    stk.emplace_back(c, t.child_ptr[c]);
    std::vector<int> run;
    std::vector<Pack> packs;
    while (!stk.empty()) {
      auto& top = stk.back();
      const int s = top.first;
      if (top.second < t.child_ptr[s + 1] && packable_c(t.child_idx[top.second])) {
        // the run of packable children from here (visiting order), as packs
        run.clear();
        while (top.second < t.child_ptr[s + 1] && packable_c(t.child_idx[top.second]))
          run.push_back(t.child_idx[top.second++]);
        pack_run(t, run, A.chunk, packs);
        for (const Pack& P : packs)
          if ((rc = run_pack(P, x, q))) return rc;
      } else if (top.second < t.child_ptr[s + 1]) {
        const int ch = t.child_idx[top.second++];
        rc = put(ch, x, q);
        if (!rc) rc = fwd_seg(ch, x, q);
        if (rc) return rc;
        stk.emplace_back(ch, t.child_ptr[ch]);
      } else {
        rc = bwd_seg(s, x, q);
        if (rc) return rc;
        stk.pop_back();
      }
    }
    return TT_OK;
  };
  // A unit of work under one parent: a child subtree (seg >= 0) or a pack.
  struct Unit {
    int seg;
    Pack pack;
  };
  auto run_unit = [&](const Unit& u, const Slot& x, cudaStream_t q) -> int {
    return u.seg >= 0 ? seq(u.seg, x, q) : run_pack(u.pack, x, q);
  };
  // `units` (children of `parent`, in visiting order) over the stacks: unit i
  // on stack slot_of[i], each stack's units in visiting order on its own
  // stream; then every stack is joined back into st and stacks 1.. have their
  // sums over parent's path added into stack 0 in stack order.
  auto fork_units = [&](const std::vector<Unit>& units, const std::vector<int>& slot_of, int used, int parent) -> int {
    int rc = TT_OK;
    if (used == 1) {
      for (const Unit& u : units)
        if (!rc) rc = run_unit(u, sl[0], st);
      return rc;
    }
    cudaEvent_t fork;
    if (!event_on(st, &fork)) rc = TT_ERR_CUDA;
    for (int j = 0; j < used && !rc; ++j)
      if (cudaStreamWaitEvent(side[j], fork, 0) != cudaSuccess) rc = TT_ERR_CUDA;
    for (size_t i = 0; i < units.size() && !rc; ++i) rc = run_unit(units[i], sl[slot_of[i]], side[slot_of[i]]);
    // join every stack's stream back into st, even after an error
    for (int j = 0; j < used; ++j) {
      cudaEvent_t e;
      if (!event_on(side[j], &e) || cudaStreamWaitEvent(st, e, 0) != cudaSuccess) rc = rc ? rc : TT_ERR_CUDA;
    }
    if (rc) return rc;
    const int64_t n4 = (t.pathlen[parent] + t.len[parent]) * rowk / 4;
    for (int j = 1; j < used; ++j)
      fold_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(
          reinterpret_cast<float4*>(sl[0].dka), reinterpret_cast<float4*>(sl[j].dka),
          reinterpret_cast<float4*>(sl[0].dva), reinterpret_cast<float4*>(sl[j].dva), n4);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  };
  // A run of packable children: its packs, pack i on stack i mod k.
  auto flush = [&](std::vector<int>& group, int parent) -> int {
    if (group.empty()) return TT_OK;
    std::vector<Pack> packs;
    pack_run(t, group, A.chunk, packs);
    group.clear();
    const int used = std::min<int>(slots, (int)packs.size());
    std::vector<Unit> units;
    std::vector<int> slot_of;
    for (size_t i = 0; i < packs.size(); ++i) {
      units.push_back(Unit{-1, packs[i]});
      slot_of.push_back((int)(i % used));
    }
    return fork_units(units, slot_of, used, parent);
  };
  // Balanced children: the children as units (inner children as subtrees,
  // each run of packable children as its packs, in visiting order); when no unit
  // holds more than half of their attention work (ancestor pairs), all units
  // are spread over the stacks at once, longest first onto the least-loaded
  // stack (ties: visiting order, lower stack), each stack running its units
  // in visiting order. Returns false (nothing enqueued) when s does not qualify.
  auto fork_children = [&](int s, int& rc) -> bool {
    if (slots < 2 || t.child_ptr[s + 1] - t.child_ptr[s] < 2) return false;
    std::vector<Unit> units;
    std::vector<double> uw;
    std::vector<int> run;
    std::vector<Pack> packs;
    auto close_run = [&]() {
      if (run.empty()) return;
      pack_run(t, run, A.chunk, packs);
      run.clear();
      for (const Pack& P : packs) {
        double w = 0.0;
        for (int c : P.roots) w += work[c];
        units.push_back(Unit{-1, P});
        uw.push_back(w);
      }
    };
    for (int i = t.child_ptr[s]; i < t.child_ptr[s + 1]; ++i) {
      const int c = t.child_idx[i];
      if (packable_c(c)) {
        run.push_back(c);
        continue;
      }
      close_run();
      units.push_back(Unit{c, Pack{}});
      uw.push_back(work[c]);
    }
    close_run();
    const int m = (int)units.size();
    if (m < 2) return false;
    double total = 0.0, mx = 0.0;
    for (double w : uw) {
      total += w;
      mx = std::max(mx, w);
    }
    if (mx > 0.5 * total) return false;
    const int used = std::min(slots, m);
    std::vector<int> by(m);
    for (int i = 0; i < m; ++i) by[i] = i;
    std::stable_sort(by.begin(), by.end(), [&](int x, int y) { return uw[x] > uw[y]; });
    std::vector<double> load(used, 0.0);
    std::vector<int> slot_of(m);
    for (int i : by) {
      int j = 0;
      for (int k = 1; k < used; ++k)
        if (load[k] < load[j]) j = k;
      slot_of[i] = j;
      load[j] += uw[i];
    }
    rc = fork_units(units, slot_of, used, s);
    return true;
  };
  // Iterative DFS: (segment, next child slot); segments with children are
  // entered on push and left on pop, packable children gathered into runs, or all
  // children forked at once when they are balanced.
  std::vector<std::pair<int, int>> stack;
  std::vector<int> group;
  if (packable_c(0)) return run_pack(Pack{0, 0, t.N, t.nseg[0], {0}}, sl[0], st);  // the whole tree is one pack
  int rc = enter_inner(0);
  if (rc) return rc;
  stack.emplace_back(0, t.child_ptr[0]);
  if (fork_children(0, rc)) {
    if (rc) return rc;
    stack.back().second = t.child_ptr[1];
  }
  while (!stack.empty()) {
    auto& top = stack.back();
    const int s = top.first;
    if (top.second < t.child_ptr[s + 1]) {
      const int c = t.child_idx[top.second++];
      if (packable_c(c)) {
        group.push_back(c);
        continue;
      }
      rc = flush(group, s);
      if (!rc) rc = enter_inner(c);
      if (rc) return rc;
      stack.emplace_back(c, t.child_ptr[c]);
      if (fork_children(c, rc)) {
        if (rc) return rc;
        stack.back().second = t.child_ptr[c + 1];
      }
    } else {
      rc = flush(group, s);
      if (!rc) rc = bwd_seg(s, sl[0], st);
      if (rc) return rc;
      stack.pop_back();
    }
  }
  return TT_OK;
}

// Validated arguments -> a ready traversal (host tree with its visiting order, layout).
int dta_prepare(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N, int64_t chunk,
                int order, int slots, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, const tt_bf16* dO,
                tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int Hq, int Hkv, int d, float scale,
                void* ws, size_t ws_bytes, int32_t* err, HostTree& t, DtaArgs& A, DtaWs& L) {
  if (!Q || !K || !V || !dO || !O || !LSE || !dQ || !dK || !dV || !ws || !err || chunk < 1) return TT_ERR_INVALID_ARG;
  if (slots < 1 || slots > kMaxSlots) return TT_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1) return TT_ERR_INVALID_ARG;
  if (order != TT_DTA_ORDER_INDEX && order != TT_DTA_ORDER_GREEDY) return TT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || (d != 64 && d != 128)) return TT_ERR_UNSUPPORTED;
  if (!host_tree(seg_parent_host, seg_len_host, S, t) || t.N != N) return TT_ERR_INVALID_TREE;
  order_children(t, order);
  L = dta_layout(stack_rows(t, chunk), chunk, Hq, Hkv, d, slots);
  if (ws_bytes < L.total) return TT_ERR_WORKSPACE;
  A = DtaArgs{N, chunk, Q, K, V, dO, O, dQ, dK, dV, LSE, Hq, Hkv, d, scale, err};
  return TT_OK;
}

// k non-blocking streams (none for k = 1); false if one cannot be created.
bool make_side_streams(int k, std::vector<cudaStream_t>& side) {
  side.clear();
  if (k < 2) return true;
  for (int j = 0; j < k; ++j) {
    cudaStream_t q;
    if (cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking) != cudaSuccess) return false;
    side.push_back(q);
  }
  return true;
}
void release(std::vector<cudaStream_t>& side, std::vector<cudaEvent_t>& events) {
  for (cudaEvent_t e : events) cudaEventDestroy(e);
  for (cudaStream_t q : side) cudaStreamDestroy(q);
  events.clear();
  side.clear();
}

}  // namespace
}  // namespace tt

using namespace tt;

TT_API size_t tt_dta_workspace_bytes_slots(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S,
                                           int64_t chunk, int Hq, int Hkv, int d, int slots) {
  HostTree t;
  if (chunk < 1 || Hq < 1 || Hkv < 1 || d < 1 || slots < 1 || slots > kMaxSlots ||
      !host_tree(seg_parent_host, seg_len_host, S, t))
    return 0;
  return dta_layout(stack_rows(t, chunk), chunk, Hq, Hkv, d, slots).total;
}

TT_API size_t tt_dta_workspace_bytes(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S,
                                     int64_t chunk, int Hq, int Hkv, int d) {
  return tt_dta_workspace_bytes_slots(seg_parent_host, seg_len_host, S, chunk, Hq, Hkv, d, TT_DTA_DEFAULT_SLOTS);
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

TT_API int tt_tree_partition(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t budget,
                             int order, int64_t* first_host, int64_t* rows_host, int64_t* path_host,
                             int32_t* kind_host, int32_t capacity) {
  if (budget < 1 || (order != TT_DTA_ORDER_INDEX && order != TT_DTA_ORDER_GREEDY) || capacity < 0)
    return TT_ERR_INVALID_ARG;
  HostTree t;
  if (!host_tree(seg_parent_host, seg_len_host, S, t)) return TT_ERR_INVALID_TREE;
  order_children(t, order);
  std::vector<Part> parts;
  tree_partitions(t, budget, parts);
  if (capacity == 0 && !first_host && !rows_host && !path_host && !kind_host) return (int)parts.size();
  if (!first_host || !rows_host || !path_host || !kind_host) return TT_ERR_INVALID_ARG;
  if (capacity < (int64_t)parts.size()) return TT_ERR_WORKSPACE;
  for (size_t i = 0; i < parts.size(); ++i) {
    first_host[i] = parts[i].first;
    rows_host[i] = parts[i].rows;
    path_host[i] = parts[i].path;
    kind_host[i] = parts[i].kind;
  }
  return (int)parts.size();
}

TT_API int tt_dta_tree_attn_slots(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                                  int64_t chunk, int order, int slots, const tt_bf16* Q, const tt_bf16* K,
                                  const tt_bf16* V, const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ,
                                  tt_bf16* dK, tt_bf16* dV, int Hq, int Hkv, int d, float scale, void* ws,
                                  size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  HostTree t;
  DtaArgs A;
  DtaWs L;
  int rc = dta_prepare(seg_parent_host, seg_len_host, S, N, chunk, order, slots, Q, K, V, dO, O, LSE, dQ, dK, dV, Hq,
                       Hkv, d, scale, ws, ws_bytes, err, t, A, L);
  if (rc) return rc;
  std::vector<cudaStream_t> side;
  std::vector<cudaEvent_t> events;
  if (!make_side_streams(slots, side)) {
    release(side, events);
    return TT_ERR_CUDA;
  }
  rc = dta_run(t, A, static_cast<char*>(ws), L, slots, reinterpret_cast<cudaStream_t>(stream), side, events);
  release(side, events);
  return rc;
}

TT_API int tt_dta_tree_attn_ordered(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                                    int64_t chunk, int order, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V,
                                    const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV,
                                    int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes, int32_t* err,
                                    tt_stream_t stream) {
  return tt_dta_tree_attn_slots(seg_parent_host, seg_len_host, S, N, chunk, order, TT_DTA_DEFAULT_SLOTS, Q, K, V, dO,
                                O, LSE, dQ, dK, dV, Hq, Hkv, d, scale, ws, ws_bytes, err, stream);
}

TT_API int tt_dta_tree_attn(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                            int64_t chunk, const tt_bf16* Q, const tt_bf16* K, const tt_bf16* V, const tt_bf16* dO,
                            tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK, tt_bf16* dV, int Hq, int Hkv, int d,
                            float scale, void* ws, size_t ws_bytes, int32_t* err, tt_stream_t stream) {
  return tt_dta_tree_attn_slots(seg_parent_host, seg_len_host, S, N, chunk, TT_DTA_ORDER_GREEDY, TT_DTA_DEFAULT_SLOTS,
                                Q, K, V, dO, O, LSE, dQ, dK, dV, Hq, Hkv, d, scale, ws, ws_bytes, err, stream);
}

// A plan: the traversal's device work for one tree, chunk size, order, slot
// count and set of buffers, captured once into a CUDA graph (copies, memsets,
// every chunk kernel, and the slots' streams as parallel branches); a launch
// replays it with one call, so the host walks the tree once.
struct tt_dta_plan_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

TT_API int tt_dta_plan_create(const int32_t* seg_parent_host, const int32_t* seg_len_host, int32_t S, int64_t N,
                              int64_t chunk, int order, int slots, const tt_bf16* Q, const tt_bf16* K,
                              const tt_bf16* V, const tt_bf16* dO, tt_bf16* O, float* LSE, tt_bf16* dQ, tt_bf16* dK,
                              tt_bf16* dV, int Hq, int Hkv, int d, float scale, void* ws, size_t ws_bytes,
                              int32_t* err, tt_dta_plan* plan_out) {
  if (!plan_out) return TT_ERR_INVALID_ARG;
  *plan_out = nullptr;
  HostTree t;
  DtaArgs A;
  DtaWs L;
  int rc = dta_prepare(seg_parent_host, seg_len_host, S, N, chunk, order, slots, Q, K, V, dO, O, LSE, dQ, dK, dV, Hq,
                       Hkv, d, scale, ws, ws_bytes, err, t, A, L);
  if (rc) return rc;
  const int dev = current_device();
  if (dev < 0) return TT_ERR_CUDA;
  std::vector<cudaStream_t> side;
  std::vector<cudaEvent_t> events;
  cudaStream_t cs;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return TT_ERR_CUDA;
  if (!make_side_streams(slots, side) || cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    release(side, events);
    cudaStreamDestroy(cs);
    (void)cudaGetLastError();
    return TT_ERR_CUDA;
  }
  rc = dta_run(t, A, static_cast<char*>(ws), L, slots, cs, side, events);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &g);
  release(side, events);
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
