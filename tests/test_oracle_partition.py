"""Oracle pins for redundancy-free tree partitioning ("Tree Training", Abstract: no pair computed twice, at most one
root-to-leaf path held on the device; the rule is this library's reading, oracle/partition.py).

The hand-derived partitions of tests/golden/partition_small.json, and on random trees the properties the pages
state: every token is computed in exactly one partition, every ancestor of a token lies in its partition's cached
root path or in the partition at or before it (so the partition computes each ancestor pair once and needs nothing
else), a pack is whole sibling subtrees adjacent in the layout, and a partition needs at most the longest root path
plus the budget of tokens.
"""
import json
import os

import pytest

import synth
from oracle import partition as PT
from oracle import tree as T


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "partition_small.json")) as f:
        return json.load(f)["cases"]


def test_golden_partitions(golden_dir):
    for c in _golden(golden_dir):
        tab = T.tables(c["seg_parent"], c["seg_len"])
        for order in ("index", "greedy"):
            assert [list(p) for p in PT.partitions(tab, c["budget"], order)] == c["partitions"], c["why"]


def _trees():
    out = [synth.random_tree(700 + s, n_seg=3 + 4 * s, len_range=(1, 90), max_children=1 + s % 4) for s in range(10)]
    out.append(synth.random_tree(799, n_seg=120, len_range=(1, 5), max_children=6))  # many tiny segments
    out.append(synth.random_tree(798, n_seg=6, len_range=(40, 60), chain=True))
    return out


@pytest.mark.parametrize("shape", _trees(), ids=lambda s: f"S{s.S}N{s.N}")
@pytest.mark.parametrize("budget", [1, 7, 64, 200, 10 ** 6])
def test_partition_properties(shape, budget):
    tab = T.tables(shape.seg_parent, shape.seg_len)
    kids = T.children(shape.seg_parent)
    for order in ("index", "greedy"):
        parts = PT.partitions(tab, budget, order)
        owner, bad = PT.partition_ancestor_check(tab, parts)
        assert not bad, bad[:5]
        assert sum(p[1] for p in parts) == tab.N
        for first, n, path, kind in parts:
            assert 1 <= n <= max(budget, 1) or (kind == 0 and first == 0 and path == 0 and n == tab.N)
            assert path + n <= max(int(tab.seg_pathlen[s] + tab.seg_len[s]) for s in range(tab.S)) + budget
            segs = [s for s in range(tab.S) if first <= tab.seg_start[s] < first + n]
            if kind == 0:
                # whole subtrees of siblings: the pack's top segments share one parent, their subtrees tile it
                tops = [s for s in segs if s == 0 or not (first <= tab.seg_start[tab.seg_parent[s]] < first + n)]
                assert len({int(tab.seg_parent[s]) for s in tops}) == 1
                assert sum(PT.subtree_tokens(tab, s) for s in tops) == n
                assert len(segs) <= PT.MAX_SEGS
                p = int(tab.seg_parent[tops[0]])
                assert path == (0 if p < 0 else int(tab.seg_pathlen[p] + tab.seg_len[p]))
                assert all(s in kids[p] for s in tops) or p < 0
            else:
                # a chunk of one segment that is not packable
                assert len({int(tab.tok_seg[t]) for t in range(first, first + n)}) == 1
                s = int(tab.tok_seg[first])
                assert PT.subtree_tokens(tab, s) > budget or PT.subtree_segments(tab, s) > PT.MAX_SEGS
        # zero redundancy: each token's ancestor pairs are computed by its one partition
        assert sum(len(T.token_ancestors(tab, t)) for t in range(tab.N)) == tab.stats["useful_pairs"]


def test_whole_tree_fits_is_one_partition():
    sh = synth.random_tree(5, n_seg=10, len_range=(1, 20))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    assert PT.partitions(tab, tab.N) == [(0, tab.N, 0, 0)]
    # more segments than a pack may hold: not one partition any more
    many = synth.random_tree(6, n_seg=PT.MAX_SEGS + 1, len_range=(1, 2))
    tab2 = T.tables(many.seg_parent, many.seg_len)
    assert len(PT.partitions(tab2, tab2.N)) > 1


def test_ancestor_check_catches_planted_mistakes(golden_dir):
    """The property check is not vacuous: a cached path one token short, a pack that misses a token and a token
    counted twice are each reported."""
    c = _golden(golden_dir)[0]
    tab = T.tables(c["seg_parent"], c["seg_len"])
    good = [tuple(p) for p in c["partitions"]]
    assert not PT.partition_ancestor_check(tab, good)[1]
    short = [(f, n, p - 1 if k == 0 and p > 0 else p, k) for f, n, p, k in good]
    assert any(b[0] == "outside" for b in PT.partition_ancestor_check(tab, short)[1])
    missing = [good[0], (good[1][0], good[1][1] - 1, good[1][2], good[1][3])] + good[2:]
    assert any(b[0] == "missing" for b in PT.partition_ancestor_check(tab, missing)[1])
    twice = good + [good[-1]]
    assert any(b[0] == "twice" for b in PT.partition_ancestor_check(tab, twice)[1])
