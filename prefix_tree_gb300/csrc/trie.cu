// Prefix tree of a task's rollouts from their token sequences (host code):
// the step before tt_tree_build.
//
// "Tree Training", Abstract: the tokens of one task form a tree with shared
// prefixes, serialised in DFS order so every token is computed once.
// AReaL-DTA, Main Findings: rollouts that are prefixes of others are
// collapsed into the longer ones (fully-contained prefix sequences merged);
// compression = total sequence tokens / unique tree tokens, and the
// leaves-only rate counts only rollouts that are not prefixes of others.
//
// A node is a distinct prefix. Children are kept in order of first
// appearance (rollout order, then position); a segment is a maximal chain of
// nodes in which every node but the last has exactly one child; segments are
// numbered in DFS preorder, so tt_tree_build's ascending-index DFS reproduces
// the token order written here.
#include <algorithm>
#include <unordered_map>
#include <vector>

#include "common.cuh"

namespace tt {
namespace {

struct Node {
  int32_t tok;
  int32_t first_child = -1, last_child = -1, next_sibling = -1, nkids = 0;
};

}  // namespace
}  // namespace tt

using namespace tt;

TT_API int tt_trie_build(const int32_t* tokens_host, const int64_t* offsets_host, int32_t R, int64_t capacity,
                         int32_t* seg_parent_host, int32_t* seg_len_host, int32_t* tok_host, int64_t* rollout_end_host,
                         int64_t* counts_host) {
  if (!tokens_host || !offsets_host || !rollout_end_host || !counts_host || R < 1 || capacity < 0)
    return TT_ERR_INVALID_ARG;
  if (offsets_host[0] != 0) return TT_ERR_INVALID_ARG;
  for (int32_t r = 0; r < R; ++r)
    if (offsets_host[r + 1] <= offsets_host[r]) return TT_ERR_INVALID_TREE;  // empty rollout
  const int32_t first = tokens_host[0];
  for (int32_t r = 1; r < R; ++r)
    if (tokens_host[offsets_host[r]] != first) return TT_ERR_INVALID_TREE;  // several roots
  const int64_t total = offsets_host[R];

  // Trie: node 0 is the shared first token.
  std::vector<Node> nodes;
  nodes.reserve((size_t)std::min<int64_t>(total, (int64_t)1 << 20));
  nodes.push_back(Node{first});
  std::unordered_map<uint64_t, int32_t> child;
  child.reserve(1024);
  std::vector<int32_t> end_node(R);
  for (int32_t r = 0; r < R; ++r) {
    int32_t cur = 0;
    for (int64_t i = offsets_host[r] + 1; i < offsets_host[r + 1]; ++i) {
      // A node's first child is found through first_child, later children
      // (branch points) through the hash of (parent, token): shared
      // prefixes mostly follow first children, and a new node's chain of
      // new children needs no lookup at all.
      const int32_t tok = tokens_host[i];
      const int32_t fc = nodes[cur].first_child;
      if (fc >= 0 && nodes[fc].tok == tok) {
        cur = fc;
        continue;
      }
      const uint64_t key = ((uint64_t)(uint32_t)cur << 32) | (uint32_t)tok;
      if (nodes[cur].nkids >= 2) {
        auto it = child.find(key);
        if (it != child.end()) {
          cur = it->second;
          continue;
        }
      }
      if (nodes.size() >= (size_t)INT32_MAX) return TT_ERR_INVALID_ARG;
      const int32_t nn = (int32_t)nodes.size();
      nodes.push_back(Node{tok});
      Node& p = nodes[cur];
      if (p.last_child < 0) {
        p.first_child = nn;
      } else {
        nodes[p.last_child].next_sibling = nn;
        child.emplace(key, nn);
      }
      p.last_child = nn;
      ++p.nkids;
      cur = nn;
    }
    end_node[r] = cur;
  }
  const int64_t N = (int64_t)nodes.size();

  // Segments in DFS preorder with an explicit stack of (first node of a
  // segment, parent segment); children pushed in reverse so the first-seen
  // child is laid out first.
  std::vector<int64_t> dfs_index(nodes.size());
  std::vector<int32_t> par, len;
  std::vector<std::pair<int32_t, int32_t>> stack{{0, -1}};
  std::vector<int32_t> kids;
  int64_t pos = 0, leaf_tokens = 0;
  while (!stack.empty()) {
    const auto [start, parent_seg] = stack.back();
    stack.pop_back();
    const int32_t s = (int32_t)len.size();
    par.push_back(parent_seg);
    len.push_back(0);
    int32_t nd = start;
    for (;;) {
      dfs_index[nd] = pos;
      if (tok_host && pos < capacity) tok_host[pos] = nodes[nd].tok;
      ++pos;
      ++len[s];
      if (nodes[nd].nkids != 1) break;
      nd = nodes[nd].first_child;
    }
    if (nodes[nd].nkids == 0) {
      // depth of the leaf = tokens on its root path
      int64_t depth = 0;
      for (int32_t q = s; q >= 0; q = par[q]) depth += len[q];
      leaf_tokens += depth;
    }
    kids.clear();
    for (int32_t c = nodes[nd].first_child; c >= 0; c = nodes[c].next_sibling) kids.push_back(c);
    for (auto it = kids.rbegin(); it != kids.rend(); ++it) stack.emplace_back(*it, s);
  }
  const int64_t S = (int64_t)len.size();
  counts_host[0] = S;
  counts_host[1] = N;
  counts_host[2] = total;
  counts_host[3] = leaf_tokens;
  for (int32_t r = 0; r < R; ++r) rollout_end_host[r] = dfs_index[end_node[r]];
  if (S > capacity || N > capacity) return TT_ERR_WORKSPACE;
  if (!seg_parent_host || !seg_len_host || !tok_host) return TT_ERR_INVALID_ARG;
  for (int64_t s = 0; s < S; ++s) {
    seg_parent_host[s] = par[s];
    seg_len_host[s] = len[s];
  }
  return TT_OK;
}
