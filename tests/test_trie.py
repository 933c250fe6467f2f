"""tt_trie_build (host code behind the C ABI) against the trie oracle, bit for bit."""
import numpy as np
import pytest

import synth
from oracle import tree as T
from oracle import trie as TR
from tests.test_oracle_trie import random_rollouts


@pytest.fixture(scope="module")
def tt():
    import prefix_tree_gb300 as tt
    return tt


def _same(lib_out, ref):
    assert lib_out["seg_parent"].tolist() == ref.seg_parent
    assert lib_out["seg_len"].tolist() == ref.seg_len
    assert lib_out["tokens"].tolist() == ref.tokens
    assert lib_out["rollout_end"].tolist() == ref.rollout_end
    assert lib_out["total_tokens"] == ref.total_tokens and lib_out["leaf_tokens"] == ref.leaf_tokens


@pytest.mark.parametrize("seed", range(20))
def test_matches_oracle(tt, seed):
    rolls = random_rollouts(seed, n_roll=5 + seed % 17, vocab=2 + seed % 6)
    _same(tt.trie_build(rolls), TR.build(rolls))


def test_golden_and_edge_cases(tt):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "trie_small.json")))
    _same(tt.trie_build(g["rollouts"]), TR.build(g["rollouts"]))
    for rolls in ([[5]], [[5, 6, 7]], [[5], [5], [5]], [[5], [5, 6], [5, 6, 7]], [[9, 1], [9, 2], [9, 3], [9, 1, 4]]):
        _same(tt.trie_build(rolls), TR.build(rolls))


def test_branches_of_the_benchmarked_tree_round_trip(tt):
    """The 1.7B-shaped tree's branches (token id = DFS position) give back its DFS layout exactly."""
    sh = synth.tree_shape(1)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    rolls = [list(b) for b in T.branches(tab)]           # DFS token indices along each root-to-leaf path
    out = tt.trie_build(rolls)
    assert out["tokens"].tolist() == list(range(tab.N))
    back = T.tables(out["seg_parent"], out["seg_len"])
    np.testing.assert_array_equal(back.tok_send, tab.tok_send)
    np.testing.assert_array_equal(back.tok_pos, tab.tok_pos)
    assert out["leaf_tokens"] == tab.stats["sum_branch_tokens"] and out["total_tokens"] == out["leaf_tokens"]


def test_errors(tt):
    with pytest.raises(tt.TTError):
        tt.trie_build([[1, 2], [3, 4]])                  # different first tokens
    with pytest.raises(tt.TTError):
        tt.trie_build([[1, 2], []])                      # empty rollout
    with pytest.raises(tt.TTError):
        tt.trie_build([])
    import ctypes
    L = tt.lib()
    toks = np.array([1, 2, 3, 1, 4], np.int32)
    offs = np.array([0, 3, 5], np.int64)
    ends = np.zeros(2, np.int64)
    counts = np.zeros(4, np.int64)
    small = np.zeros(2, np.int32)
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = L.tt_trie_build(vp(toks), vp(offs), 2, 2, vp(small), vp(small), vp(small), vp(ends), vp(counts))
    assert rc == -4 and counts.tolist() == [3, 4, 5, 5]  # capacity 2 < N: sizes still reported
