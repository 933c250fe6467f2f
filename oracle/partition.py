"""Redundancy-free tree partitioning (oracle; test infrastructure only).

Source: "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix
Reuse", Abstract — a trajectory tree that does not fit on the GPU is split so
that no attention pair is computed twice and the device never holds more than
one root-to-leaf path at a time.
The pages give the two properties and no algorithm; the rule below is this
library's reading (it is the partition the path-at-a-time traversal runs):

* a subtree is *packable* when it holds at most ``budget`` tokens and at most
  ``max_segs`` segments;
* if the root's subtree is packable, the whole tree is one partition with an
  empty cached path;
* otherwise every segment that is not packable contributes its own tokens in
  chunks of at most ``budget`` (kind 1); chunk i attends to the segment's root
  path and the segment's earlier tokens;
* the children of such a segment, in visiting order, are taken in runs of
  consecutive packable children; each run is sorted by DFS position and cut
  greedily into packs of whole sibling subtrees that are adjacent in the DFS
  layout, at most ``budget`` tokens and ``max_segs`` segments each (kind 0);
  a pack attends to its parent's root path and to itself.

The visiting order is either ascending segment index or greedy: children in
the order in which the oracle's greedy leaf walk (tree.greedy_leaf_order)
first reaches a leaf of their subtree.

Partitions are returned as (first DFS token, tokens, cached path tokens,
kind), sorted by first token. Plain Python over the tree tables.
"""
from __future__ import annotations

from . import tree as _tree

MAX_SEGS = 64


def _visiting_children(tt, order):
    ch = _tree.children(tt.seg_parent)
    if order == "index":
        return ch
    if order != "greedy":
        raise ValueError(f"unknown order {order!r}")
    rank = {leaf: i for i, leaf in enumerate(_tree.greedy_leaf_order(tt))}
    first_leaf = {}
    for s in range(tt.S):
        first_leaf[s] = min(rank[x] for x in range(tt.S) if x in rank and
                            tt.seg_start[s] <= tt.seg_start[x] < tt.seg_subtree_end[s])
    return [sorted(c, key=lambda x: first_leaf[x]) for c in ch]


def subtree_tokens(tt, s):
    return int(tt.seg_subtree_end[s] - tt.seg_start[s])


def subtree_segments(tt, s):
    return sum(1 for x in range(tt.S) if tt.seg_start[s] <= tt.seg_start[x] < tt.seg_subtree_end[s])


def partitions(tt, budget, order="greedy", max_segs=MAX_SEGS):
    """The partitions of the tree for a token budget (see the module docstring)."""
    if budget < 1:
        raise ValueError("budget must be >= 1")
    kids = _visiting_children(tt, order)

    def packable(s):
        return subtree_tokens(tt, s) <= budget and subtree_segments(tt, s) <= max_segs

    if packable(0):
        return [(0, int(tt.N), 0, 0)]
    out = []

    def cut(run):
        packs = []  # [first, tokens, segments, path]
        for c in sorted(run, key=lambda x: tt.seg_start[x]):
            first, n, nseg = int(tt.seg_start[c]), subtree_tokens(tt, c), subtree_segments(tt, c)
            if packs and packs[-1][0] + packs[-1][1] == first and packs[-1][1] + n <= budget \
                    and packs[-1][2] + nseg <= max_segs:
                packs[-1][1] += n
                packs[-1][2] += nseg
            else:
                packs.append([first, n, nseg, int(tt.seg_pathlen[c])])
        for first, n, _, path in packs:
            out.append((first, n, path, 0))

    def visit(s):
        for c0 in range(0, int(tt.seg_len[s]), budget):
            out.append((int(tt.seg_start[s]) + c0, min(budget, int(tt.seg_len[s]) - c0), int(tt.seg_pathlen[s]) + c0, 1))
        run = []
        for c in kids[s]:
            if packable(c):
                run.append(c)
                continue
            cut(run)
            run = []
            visit(c)
        cut(run)

    visit(0)
    return sorted(out)


def partition_ancestor_check(tt, parts):
    """For every token t: the partition holding it, and whether every ancestor of t (its root-to-token path) lies in
    that partition's cached root path or in the partition itself at or before t. Returns (owner per token,
    violations). The cached path of a partition is the first `path` tokens of the root path of its first token."""
    owner = [-1] * int(tt.N)
    bad = []
    for i, (first, n, path, kind) in enumerate(parts):
        for t in range(first, first + n):
            if owner[t] != -1:
                bad.append(("twice", t))
            owner[t] = i
    for t in range(int(tt.N)):
        if owner[t] < 0:
            bad.append(("missing", t))
            continue
        first, n, path, kind = parts[owner[t]]
        root_path = _tree.token_path(tt, int(tt.tok_seg[t]))
        cached = set(root_path[:path]) if path else set()
        for a in _tree.token_ancestors(tt, t):
            a = int(a)
            if a not in cached and not (first <= a <= t):
                bad.append(("outside", t, a))
    return owner, bad
