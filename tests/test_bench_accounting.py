"""The bench's FLOP accounting: its closed-form count of ancestor pairs (the useful-work unit of the attention
metric, 14·d·Hq·pairs per fwd+bwd) against the oracle's count from explicit ancestor sets."""
import numpy as np
import pytest

import bench
import synth
from oracle import tree as T


@pytest.mark.parametrize("seed,n_seg,lens", [(0, 1, (1, 1)), (1, 5, (1, 40)), (2, 12, (3, 200)), (3, 30, (1, 60)),
                                             (4, 9, (50, 400))])
def test_useful_pairs_matches_ancestor_sets(seed, n_seg, lens):
    sh = synth.random_tree(seed, n_seg=n_seg, len_range=lens, max_children=3)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    assert tab.N <= 4096  # the oracle counts explicit ancestor sets up to this size
    assert bench.useful_pairs(sh.seg_parent, sh.seg_len) == tab.stats["useful_pairs"]


@pytest.mark.parametrize("wid,pairs_m", [(1, 31.34), (3, 224.90), (4, 95.83)])
def test_useful_pairs_of_the_benchmarked_trees(wid, pairs_m):
    """The pair counts of the trees the bench times (the headline 8B-shaped tree and the side workloads) equal the
    oracle's Σ_t |anc(t)|, and its branch-token count the oracle's Σ_b |b|."""
    sh = synth.tree_shape(wid)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    p = bench.useful_pairs(sh.seg_parent, sh.seg_len)
    assert p == tab.stats["useful_pairs"] == int(np.sum(tab.tok_pos + 1))
    assert round(p / 1e6, 2) == pairs_m
    assert bench.branch_tokens(sh.seg_parent, sh.seg_len) == tab.stats["sum_branch_tokens"]


def test_oracle_sample_flops():
    """The CPU baseline's sample (one head, rows of the listed segments) is credited with exactly the ancestor
    pairs of those rows."""
    sh = synth.tree_shape(bench.HEADLINE)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    rows = np.concatenate([np.arange(tab.seg_start[s], tab.seg_end[s]) for s in bench.ORACLE_SEGMENTS])
    d = synth.HEADS[bench.HEADLINE][2]
    assert bench.oracle_flops() == 14.0 * d * int(np.sum(tab.tok_pos[rows] + 1))
    sh1 = synth.tree_shape(1)
    assert bench.oracle_flops(1, None) == 14.0 * 128 * bench.useful_pairs(sh1.seg_parent, sh1.seg_len)


def test_bench_trie_rollouts_rebuild_the_tree():
    """The bench's branch rollouts (from the segment arrays alone) rebuild the same DFS layout through the trie
    builder (checked with the oracle's tree tables)."""
    import prefix_tree_gb300 as tt
    sh = synth.tree_shape(1)
    out = tt.trie_build(bench.branch_rollouts(sh.seg_parent, sh.seg_len))
    a, b = T.tables(out["seg_parent"], out["seg_len"]), T.tables(sh.seg_parent, sh.seg_len)
    np.testing.assert_array_equal(a.tok_send, b.tok_send)
    assert out["total_tokens"] == b.stats["sum_branch_tokens"] and len(out["tokens"]) == b.N


@pytest.mark.parametrize("seed,chunk", [(5, 64), (6, 100), (7, 2048)])
def test_path_at_a_time_chunks_cover_each_pair_once(seed, chunk):
    """The traversal's chunk calls (segment s in chunks of `chunk` queries at path offset pathlen(s) + c0, each
    against its path prefix plus the causal part of the chunk) add up to the ancestor pairs: no redundant work."""
    sh = synth.random_tree(seed, n_seg=14, len_range=(1, 300), max_children=3)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    pairs = 0
    for s in range(tab.S):
        L, base = int(tab.seg_len[s]), int(tab.seg_pathlen[s])
        for c0 in range(0, L, chunk):
            C = min(chunk, L - c0)
            pairs += C * (base + c0) + C * (C + 1) // 2
    assert pairs == tab.stats["useful_pairs"] == bench.useful_pairs(sh.seg_parent, sh.seg_len)


def test_path_stack_folds_follow_the_fork_rule():
    """The bench's count of fold kernels: balanced children fork once at the top (8B-shaped tree: the root's 8
    equal subtrees over 2 stacks, one fold); a run of leaves is cut into packs first, and unbalanced units fall
    back to the runs' packs."""
    import bench
    import synth
    sh = synth.tree_shape(3)
    assert bench.dta_folds(sh.seg_parent, sh.seg_len) == 1
    assert bench.dta_folds(sh.seg_parent, sh.seg_len, slots=1) == 0
    # root with one big child (3 equal leaves below it) and one small leaf: unbalanced at the root
    par, ln = [-1, 0, 0, 1, 1, 1], [10, 500, 5, 50, 50, 50]
    assert bench.dta_folds(par, ln) == 0                # the whole tree (665 rows) is one pack
    assert bench.dta_folds(par, ln, chunk=100) == 1     # packs of 100 and 50 rows: unbalanced, the run forks
    assert bench.dta_folds(par, ln, chunk=50) == 1      # three one-leaf packs: balanced, all fork over 2 stacks
    assert bench.dta_folds(par, ln, chunk=50, slots=3) == 2
    # a chain: nothing forks
    assert bench.dta_folds([-1, 0, 1, 2], [5, 5, 5, 5]) == 0


def test_path_stack_launches_count_packs():
    """Kernel launches of the pass: a pack of subtrees is 5 launches (send fill, forward, pre-kernel, backward,
    conversion) where its segments alone would be 4 each."""
    import bench
    par, ln = [-1, 0, 0, 0], [300, 40, 40, 40]
    assert bench.dta_launches(par, ln, 2048) == 5  # the whole tree is one pack
    # 200-row chunks: the root in 2 chunks (7) + one pack of the three adjacent leaves (5)
    assert bench.dta_launches(par, ln, 200) == 7 + 5
    # an inner subtree that fits is packed whole: at 100-row chunks the root in 3 chunks (10) and one pack of
    # segment 1's subtree (70 rows) with the adjacent leaf 4 (10 rows); at 75 rows the root in 4 chunks (13), the
    # subtree pack (5) and leaf 4 alone as a segment (4), the two packs forked over 2 stacks (1 fold)
    assert bench.dta_launches([-1, 0, 1, 1, 0], [300, 30, 20, 20, 10], 100) == 10 + 5
    assert bench.dta_launches([-1, 0, 1, 1, 0], [300, 30, 20, 20, 10], 75) == 13 + 5 + 4 + 1
    # 80-row chunks: packs {1, 2} and {3} (5 + 4), the root in 4 chunks (13), then a fork of the two packs (1 fold)
    assert bench.dta_launches(par, ln, 80) == 13 + 5 + 4 + 1
