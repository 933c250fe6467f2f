"""Prefix tree of a task's rollouts from their token sequences (oracle).

Sources: "Tree Training: Accelerating Agentic LLMs Training via Shared Prefix
Reuse", Abstract — the tokens of one task form a tree-structured trajectory
with shared prefixes, serialised in DFS order so every token is visited once.
"AREAL-DTA: Dynamic Tree Attention for Efficient Reinforcement Learning of
Large Language Models", Main Findings — rollouts that are prefixes of others
are collapsed into the longer ones (fully-contained prefix sequences are
merged); the compression rate is total sequence tokens over unique tree
tokens, and the leaves-only rate counts only rollouts that are not prefixes
of others.

Readings where the pages are silent (each listed in the design notes):
* every rollout is a non-empty token sequence, and all rollouts of a task
  share their first token (one root);
* a tree node is a distinct prefix; a segment is a maximal chain of nodes in
  which every node but the last has exactly one child, so a segment ends only
  at a leaf or at a branch point (a rollout ending inside a chain — a
  contained prefix, or a duplicate — does not split it);
* the children of a node are ordered by first appearance (rollout order, then
  position), and segments are numbered in DFS preorder, so parents precede
  children and tt_tree_build's ascending-index DFS gives the same layout.

Written the plain way: a dict-of-dicts trie and recursion. Test
infrastructure only.
"""
from __future__ import annotations

import sys
from dataclasses import dataclass


class TrieError(ValueError):
    """The rollouts do not form one prefix tree (empty rollout, several first tokens)."""


@dataclass
class Trie:
    seg_parent: list   # [S] parent segment, -1 for the root
    seg_len: list      # [S] tokens per segment
    tokens: list       # [N] token ids in DFS order
    rollout_end: list  # [R] DFS index of each rollout's last token
    total_tokens: int  # Σ rollout lengths
    leaf_tokens: int   # Σ lengths of the rollouts that are not prefixes of others (one per distinct leaf path)

    @property
    def S(self):
        return len(self.seg_len)

    @property
    def N(self):
        return len(self.tokens)


def build(rollouts) -> Trie:
    rollouts = [list(map(int, r)) for r in rollouts]
    if not rollouts or any(len(r) == 0 for r in rollouts):
        raise TrieError("every rollout needs at least one token")
    if len({r[0] for r in rollouts}) != 1:
        raise TrieError("rollouts do not share their first token")
    # node: {"tok": token, "kids": dict token -> node (insertion order = first appearance), "ends": [rollout ids]}
    root = {"tok": rollouts[0][0], "kids": {}, "ends": []}
    for r_id, r in enumerate(rollouts):
        node = root
        for tok in r[1:]:
            if tok not in node["kids"]:
                node["kids"][tok] = {"tok": tok, "kids": {}, "ends": []}
            node = node["kids"][tok]
        node["ends"].append(r_id)

    seg_parent, seg_len, tokens = [], [], []
    rollout_end = [None] * len(rollouts)
    sys.setrecursionlimit(max(10000, sys.getrecursionlimit()))

    def segment(first, parent_seg):
        """Lay out the segment starting at node `first`, then its child segments."""
        s = len(seg_len)
        seg_parent.append(parent_seg)
        seg_len.append(0)
        node = first
        while True:
            for r_id in node["ends"]:
                rollout_end[r_id] = len(tokens)
            tokens.append(node["tok"])
            seg_len[s] += 1
            if len(node["kids"]) != 1:
                break
            node = next(iter(node["kids"].values()))
        for child in node["kids"].values():
            segment(child, s)

    segment(root, -1)
    total = sum(len(r) for r in rollouts)
    # leaf paths: one per leaf node; its length is the node's depth + 1
    leaf_tokens = 0

    def leaves(node, depth):
        nonlocal leaf_tokens
        if not node["kids"]:
            leaf_tokens += depth + 1
        for c in node["kids"].values():
            leaves(c, depth + 1)

    leaves(root, 0)
    return Trie(seg_parent, seg_len, tokens, rollout_end, total, leaf_tokens)


def rollout_from_layout(trie: Trie, r_id: int) -> list:
    """The token sequence of rollout r_id read back from the layout: walk from its last token to the root."""
    start = []
    acc = 0
    for L in trie.seg_len:
        start.append(acc)
        acc += L
    idx = trie.rollout_end[r_id]
    seg = next(s for s in range(trie.S) if start[s] <= idx < start[s] + trie.seg_len[s])
    out = trie.tokens[start[seg]:idx + 1]
    seg = trie.seg_parent[seg]
    while seg >= 0:
        out = trie.tokens[start[seg]:start[seg] + trie.seg_len[seg]] + out
        seg = trie.seg_parent[seg]
    return out
