"""Tree tables of a rollout prefix tree laid out in DFS order (oracle, fp64/int).

Source: "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix
Reuse", Abstract — the tokens of one task form a tree with shared prefixes;
DFS serialization visits every token exactly once; each token's loss weight is
the fraction of branches passing through it. AReaL-DTA, "Main Findings" — the
compression rate is total sequence tokens over unique tree tokens.

Readings where the pages are silent (each listed in the design notes):
* a tree is given as segments: ``seg_parent[s]`` (−1 for the root, else an
  earlier segment) and ``seg_len[s] ≥ 1`` tokens;
* children are visited in ascending segment index;
* a branch is a root-to-leaf path of segments (leaf = segment without
  children); the position of a token is its 0-based depth along its path;
* an ancestor interval list is the sorted, maximal, half-open set of DFS
  token ranges covering a token's root-to-token path.

Everything is computed the plain way: recursive DFS, parent-pointer walks,
explicit sets. Test infrastructure only.
"""
from __future__ import annotations

import sys
from dataclasses import dataclass, field

import numpy as np


class TreeError(ValueError):
    """The segment arrays do not describe a valid topologically ordered tree."""


def validate(seg_parent, seg_len, N=None):
    par = [int(p) for p in seg_parent]
    ln = [int(x) for x in seg_len]
    if len(par) == 0 or len(par) != len(ln):
        raise TreeError("empty tree or length mismatch")
    if par[0] != -1:
        raise TreeError("segment 0 must be the root (parent −1)")
    for s in range(1, len(par)):
        if not (0 <= par[s] < s):
            raise TreeError(f"segment {s}: parent {par[s]} must lie in [0, {s})")
    if any(x < 1 for x in ln):
        raise TreeError("every segment needs at least one token")
    if N is not None and sum(ln) != N:
        raise TreeError("segment lengths do not sum to N")
    return par, ln


def children(seg_parent):
    par = [int(p) for p in seg_parent]
    ch = [[] for _ in par]
    for s in range(1, len(par)):
        ch[par[s]].append(s)
    for c in ch:
        c.sort()
    return ch


def dfs_preorder(seg_parent):
    """Segments in DFS preorder from the root, children in ascending index."""
    ch = children(seg_parent)
    order = []
    sys.setrecursionlimit(max(10000, 4 * len(ch) + 100))

    def visit(s):
        order.append(s)
        for c in ch[s]:
            visit(c)

    visit(0)
    return order


def segment_path(seg_parent, s):
    """Segments from the root down to s (inclusive), by walking parents."""
    path = []
    while s >= 0:
        path.append(int(s))
        s = int(seg_parent[s])
    return path[::-1]


@dataclass
class TreeTables:
    seg_parent: np.ndarray
    seg_len: np.ndarray
    order: list                 # segments in DFS preorder
    seg_start: np.ndarray       # DFS token offset of each segment
    seg_end: np.ndarray
    seg_subtree_end: np.ndarray  # end of the DFS span of the segment's subtree
    seg_depth: np.ndarray       # number of strict ancestor segments
    seg_pathlen: np.ndarray     # tokens on the path before the segment
    seg_leafcnt: np.ndarray     # leaves (childless segments) in the subtree
    iv_ptr: np.ndarray          # CSR offsets, [S+1]
    iv: np.ndarray              # [n_iv, 2] half-open (begin, end)
    tok_seg: np.ndarray
    tok_pos: np.ndarray
    tok_send: np.ndarray
    tok_leafcnt: np.ndarray
    tok_weight: np.ndarray      # float32(n)/float32(B)
    B: int
    N: int
    leaves: list
    stats: dict = field(default_factory=dict)

    @property
    def S(self):
        return len(self.seg_len)


def tables(seg_parent, seg_len, tile=128) -> TreeTables:
    par, ln = validate(seg_parent, seg_len)
    S, N = len(par), sum(ln)
    ch = children(par)
    order = dfs_preorder(par)

    # DFS layout: segments are laid out back to back in preorder.
    seg_start = np.zeros(S, np.int64)
    off = 0
    for s in order:
        seg_start[s] = off
        off += ln[s]
    seg_end = seg_start + np.asarray(ln, np.int64)

    # Subtree membership by parent walks (no reliance on the layout).
    in_subtree = [[] for _ in range(S)]
    for s in range(S):
        for a in segment_path(par, s):
            in_subtree[a].append(s)
    seg_subtree_end = np.array([max(seg_end[x] for x in in_subtree[s]) for s in range(S)], np.int64)
    leaves = [s for s in range(S) if not ch[s]]
    seg_leafcnt = np.array([sum(1 for x in in_subtree[s] if not ch[x]) for s in range(S)], np.int64)
    B = len(leaves)

    paths = [segment_path(par, s) for s in range(S)]
    seg_depth = np.array([len(p) - 1 for p in paths], np.int64)
    seg_pathlen = np.array([sum(ln[a] for a in p[:-1]) for p in paths], np.int64)

    # Canonical ancestor intervals of each segment (the segment's own range last).
    iv_ptr = [0]
    iv = []
    for s in range(S):
        ranges = sorted((int(seg_start[a]), int(seg_end[a])) for a in paths[s])
        merged = []
        for b, e in ranges:
            if merged and merged[-1][1] == b:
                merged[-1][1] = e
            else:
                merged.append([b, e])
        iv.extend(merged)
        iv_ptr.append(len(iv))

    tok_seg = np.zeros(N, np.int64)
    for s in range(S):
        tok_seg[seg_start[s]:seg_end[s]] = s
    t = np.arange(N)
    tok_pos = seg_pathlen[tok_seg] + (t - seg_start[tok_seg])
    tok_send = seg_subtree_end[tok_seg]
    tok_leafcnt = seg_leafcnt[tok_seg]
    tok_weight = (tok_leafcnt.astype(np.float32) / np.float32(B)).astype(np.float32)

    tt = TreeTables(
        seg_parent=np.asarray(par, np.int64), seg_len=np.asarray(ln, np.int64), order=order,
        seg_start=seg_start, seg_end=seg_end, seg_subtree_end=seg_subtree_end, seg_depth=seg_depth,
        seg_pathlen=seg_pathlen, seg_leafcnt=seg_leafcnt, iv_ptr=np.asarray(iv_ptr, np.int64),
        iv=np.asarray(iv, np.int64).reshape(-1, 2), tok_seg=tok_seg, tok_pos=tok_pos, tok_send=tok_send,
        tok_leafcnt=tok_leafcnt, tok_weight=tok_weight, B=B, N=N, leaves=leaves)
    br = branches(tt)
    tt.stats = dict(
        B=B, N=N,
        sum_branch_tokens=int(sum(len(b) for b in br)),
        useful_pairs=int(sum(len(token_ancestors(tt, x)) for x in range(N))) if N <= 4096
        else int(np.sum(tok_pos + 1)),
        tile_pairs=tile_pairs(tt, tile),
        iv_pairs=len(iv),
        max_depth=int(seg_depth.max()),
        max_path=int(max(len(b) for b in br)),
    )
    return tt


def token_ancestors(tt: TreeTables, t: int) -> np.ndarray:
    """Root-to-t path of token t (including t), as sorted DFS token indices, by walking parents."""
    s = int(tt.tok_seg[t])
    toks = []
    for a in segment_path(tt.seg_parent, s)[:-1]:
        toks.extend(range(int(tt.seg_start[a]), int(tt.seg_end[a])))
    toks.extend(range(int(tt.seg_start[s]), t + 1))
    return np.asarray(toks, np.int64)


def token_intervals(tt: TreeTables, t: int):
    """Interval list of token t: its segment's list with the last interval clipped at t+1."""
    s = int(tt.tok_seg[t])
    lst = [list(x) for x in tt.iv[tt.iv_ptr[s]:tt.iv_ptr[s + 1]]]
    lst[-1][1] = t + 1
    return lst


def branches(tt: TreeTables):
    """Token lists (DFS indices, root to leaf) of every root-to-leaf branch, leaves in DFS order."""
    out = []
    for leaf in sorted(tt.leaves, key=lambda s: tt.seg_start[s]):
        toks = []
        for a in segment_path(tt.seg_parent, leaf):
            toks.extend(range(int(tt.seg_start[a]), int(tt.seg_end[a])))
        out.append(np.asarray(toks, np.int64))
    return out


def compression(tt: TreeTables) -> float:
    """Total branch tokens over unique tree tokens (AReaL-DTA, "Main Findings")."""
    return sum(len(b) for b in branches(tt)) / tt.N


def tile_pairs(tt: TreeTables, tile=128) -> int:
    """Number of (query tile, key tile) pairs holding at least one ancestor pair."""
    nT = (tt.N + tile - 1) // tile
    hit = np.zeros((nT, nT), bool)
    for t in range(tt.N):
        for b, e in token_intervals(tt, t):
            hit[t // tile, b // tile:(e - 1) // tile + 1] = True
    return int(hit.sum())


def tile_schedules(tt: TreeTables, tile=128) -> dict:
    """Tile schedules of the attention kernels, from their plain definitions.

    With query tiles T and key blocks b of `tile` rows, a (T, b) pair is
    needed iff it holds at least one ancestor pair (k in b is an ancestor of
    q in T). Returns
    * send: tok_send zero-padded to whole blocks (a padding key is nobody's ancestor);
    * blk_min / blk_max: min / max of send over the real keys of each block;
    * fwd_cnt[T]: key blocks needed by query tile T; bwd_cnt[b]: query tiles
      needed by key block b (both from explicit interval lists);
    * fwd_order / bwd_order: tiles / blocks by decreasing count, ties by
      increasing index (longest first).
    """
    nT = (tt.N + tile - 1) // tile
    hit = np.zeros((nT, nT), bool)
    for t in range(tt.N):
        for b, e in token_intervals(tt, t):
            hit[t // tile, b // tile:(e - 1) // tile + 1] = True
    send = np.zeros(nT * tile, np.int64)
    send[:tt.N] = tt.tok_send
    blk_min = np.array([tt.tok_send[b * tile:min((b + 1) * tile, tt.N)].min() for b in range(nT)], np.int64)
    blk_max = np.array([tt.tok_send[b * tile:min((b + 1) * tile, tt.N)].max() for b in range(nT)], np.int64)
    fwd_cnt = hit.sum(axis=1).astype(np.int64)
    bwd_cnt = hit.sum(axis=0).astype(np.int64)
    longest_first = lambda cnt: np.array(sorted(range(nT), key=lambda i: (-int(cnt[i]), i)), np.int64)
    return dict(send=send, blk_min=blk_min, blk_max=blk_max, fwd_cnt=fwd_cnt, bwd_cnt=bwd_cnt,
                fwd_order=longest_first(fwd_cnt), bwd_order=longest_first(bwd_cnt))


def greedy_leaf_order(tt: TreeTables) -> list:
    """Order of visiting the leaves in which each next leaf has the longest possible common prefix with the one before
    (AReaL-DTA, "Key Contributions" 2 and "Methodology in Plain English": a greedy reordering of the DFS visits).

    A plain greedy walk over the leaves: start at the leaf with the longest root path (in tokens); from the
    current leaf, go to the unvisited leaf that shares the most prefix tokens with it; ties (the pages give no
    tie-break) go to the longer root path, then to the lower segment index. Every step compares explicit token
    paths. Returns the leaf segments in visiting order.
    """
    paths = {s: token_path(tt, s) for s in tt.leaves}

    def shared(a, b):
        pa, pb = paths[a], paths[b]
        n = min(len(pa), len(pb))
        k = 0
        while k < n and pa[k] == pb[k]:
            k += 1
        return k

    left = set(tt.leaves)
    cur = min(left, key=lambda s: (-len(paths[s]), s))
    order = [cur]
    left.remove(cur)
    while left:
        cur = min(left, key=lambda s: (-shared(order[-1], s), -len(paths[s]), s))
        order.append(cur)
        left.remove(cur)
    return order


def token_path(tt: TreeTables, s: int) -> list:
    """DFS token indices of the root-to-s path (all of segment s included), by walking parents."""
    toks = []
    for a in segment_path(tt.seg_parent, s):
        toks.extend(range(int(tt.seg_start[a]), int(tt.seg_end[a])))
    return toks
