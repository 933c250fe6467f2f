"""Pins of the trie oracle (rollout token sequences -> prefix tree in DFS layout)."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import tree as T
from oracle import trie as TR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "trie_small.json")


def random_rollouts(seed, n_roll=12, vocab=5, max_new=6):
    """Rollouts that share prefixes: each new one cuts an earlier one at a random point and continues with random
    tokens (a small vocabulary makes continuations collide), plus contained prefixes and duplicates."""
    rng = np.random.default_rng(seed)
    out = [[7] + list(rng.integers(0, vocab, rng.integers(0, max_new + 1)))]
    while len(out) < n_roll:
        base = out[rng.integers(0, len(out))]
        kind = rng.integers(0, 4)
        if kind == 0:
            out.append(base[:rng.integers(1, len(base) + 1)])          # contained prefix (or duplicate)
        else:
            cut = rng.integers(1, len(base) + 1)
            out.append(base[:cut] + list(rng.integers(0, vocab, rng.integers(1, max_new + 1))))
    return out


def test_golden():
    g = json.load(open(GOLDEN))
    t = TR.build(g["rollouts"])
    assert t.seg_parent == g["seg_parent"] and t.seg_len == g["seg_len"]
    assert t.tokens == g["tokens"] and t.rollout_end == g["rollout_end"]
    assert t.total_tokens == g["total_tokens"] and t.leaf_tokens == g["leaf_tokens"]


def check_invariants(t, rolls):
    # every rollout reads back from the layout
    for r_id, r in enumerate(rolls):
        assert TR.rollout_from_layout(t, r_id) == r
    # one node per distinct prefix
    prefixes = {tuple(r[:k]) for r in rolls for k in range(1, len(r) + 1)}
    assert t.N == len(prefixes)
    # segments end only at leaves or branch points
    kids = {s: 0 for s in range(t.S)}
    for s in range(1, t.S):
        assert 0 <= t.seg_parent[s] < s
        kids[t.seg_parent[s]] += 1
    assert all(k != 1 for k in kids.values()), "a segment with exactly one child"
    # leaves = the distinct rollouts that are not prefixes of another
    maximal = {tuple(r) for r in rolls if not any(len(o) > len(r) and o[:len(r)] == r for o in rolls)}
    assert sum(1 for k in kids.values() if k == 0) == len(maximal)
    assert t.leaf_tokens == sum(len(m) for m in maximal)
    assert t.total_tokens == sum(len(r) for r in rolls)
    # the layout is a valid tree for the tree tables, with one branch per maximal rollout
    tab = T.tables(np.array(t.seg_parent, np.int32), np.array(t.seg_len, np.int32))
    assert tab.B == len(maximal) and tab.N == t.N
    assert tab.stats["sum_branch_tokens"] == t.leaf_tokens


@pytest.mark.parametrize("seed", range(12))
def test_invariants_against_brute_force(seed):
    rolls = random_rollouts(seed)
    check_invariants(TR.build(rolls), rolls)


def test_order_of_rollouts_only_relabels():
    """Permuting rollouts changes child order (first appearance) but not the set of root-to-leaf sequences."""
    rolls = random_rollouts(3)
    a, b = TR.build(rolls), TR.build(list(reversed(rolls)))
    assert a.N == b.N and a.S == b.S and a.leaf_tokens == b.leaf_tokens
    seqs = lambda t, rs: sorted(tuple(TR.rollout_from_layout(t, i)) for i in range(len(rs)))
    assert seqs(a, rolls) == seqs(b, rolls)


def test_single_rollout_and_chain_of_prefixes():
    t = TR.build([[5, 6, 7]])
    assert (t.seg_parent, t.seg_len, t.tokens, t.rollout_end) == ([-1], [3], [5, 6, 7], [2])
    t = TR.build([[5], [5, 6], [5, 6, 7]])                  # every rollout a prefix of the last: one segment
    assert (t.seg_parent, t.seg_len, t.rollout_end, t.leaf_tokens) == ([-1], [3], [0, 1, 2], 3)


def test_errors():
    with pytest.raises(TR.TrieError):
        TR.build([[1, 2], [3]])                               # two first tokens: a forest
    with pytest.raises(TR.TrieError):
        TR.build([[1, 2], []])
    with pytest.raises(TR.TrieError):
        TR.build([])


def _split_segment(t, seg, at):
    """The layout with segment `seg` cut after `at` tokens into two chained segments (DFS numbering kept)."""
    par, ln = [], []
    for s in range(t.S):
        p = t.seg_parent[s]
        p = p + 1 if p > seg else (seg + 1 if p == seg else p)
        if s == seg:
            par += [p, seg]
            ln += [at, t.seg_len[s] - at]
        else:
            par.append(p)
            ln.append(t.seg_len[s])
    return TR.Trie(par, ln, t.tokens, t.rollout_end, t.total_tokens, t.leaf_tokens)


def test_planted_split_at_rollout_end_is_caught():
    """A builder that also split segments where a contained rollout ends (here r5's prefix r1 = [1,2,3,5,6]
    ends inside segment [5, 6, 8]) gives a layout the invariant checks reject."""
    g = json.load(open(GOLDEN))
    rolls = g["rollouts"]
    t = TR.build(rolls)
    check_invariants(t, rolls)
    bad = _split_segment(t, 3, 2)  # [5, 6] | [8]
    assert bad.seg_len == [2, 1, 1, 2, 1, 1] and bad.seg_parent == [-1, 0, 1, 1, 3, 0]
    with pytest.raises(AssertionError, match="exactly one child"):
        check_invariants(bad, rolls)
