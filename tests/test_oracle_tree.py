"""Pins of oracle.tree against hand-derived fixtures, brute force and invariants.

Sources: "Tree Training" Abstract (DFS serialization; weight = fraction of
branches through a token); AReaL-DTA "Main Findings" (compression rate).
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import tree as T


@pytest.fixture(scope="module")
def golden(golden_dir):
    with open(os.path.join(golden_dir, "tree_small.json")) as f:
        return json.load(f)["trees"]


def test_golden_tables(golden):
    for g in golden:
        tt = T.tables(g["seg_parent"], g["seg_len"])
        assert tt.order == g["dfs_order"]
        for key in ("seg_start", "seg_subtree_end", "seg_depth", "seg_pathlen", "seg_leafcnt", "iv_ptr",
                    "tok_seg", "tok_pos", "tok_send", "tok_leafcnt"):
            np.testing.assert_array_equal(getattr(tt, key), g[key], err_msg=key)
        np.testing.assert_array_equal(tt.iv, np.asarray(g["iv"]))
        np.testing.assert_array_equal(tt.tok_weight, np.asarray(g["tok_weight"], np.float32))
        assert [b.tolist() for b in T.branches(tt)] == g["branches"]
        for k, v in g["stats"].items():
            assert tt.stats[k] == v, k
        assert T.compression(tt) == pytest.approx(g["compression"], abs=0)
        assert T.tile_pairs(tt, tile=4) == g["tile_pairs_tile4"]


def test_golden_tile_schedules(golden):
    """Tile schedules at tiles 2 and 4 against the hand-derived values (one of them with an empty tile pair)."""
    for g in golden:
        tt = T.tables(g["seg_parent"], g["seg_len"])
        for tile, want in g["schedules"].items():
            got = T.tile_schedules(tt, tile=int(tile))
            for k, v in want.items():
                np.testing.assert_array_equal(got[k], v, err_msg=f"{g['name']} tile {tile} {k}")


@pytest.mark.parametrize("seed,tile", [(3, 4), (5, 8), (8, 3), (11, 16)])
def test_tile_schedules_by_brute_force(seed, tile):
    """Counts from explicit ancestor sets (parent walks, not interval lists); both counts add up to the number of
    non-empty tile pairs; the orders are permutations sorted longest first."""
    shape = synth.random_tree(seed, n_seg=4 + 2 * seed, len_range=(1, 12), max_children=3)
    tt = T.tables(shape.seg_parent, shape.seg_len)
    sch = T.tile_schedules(tt, tile=tile)
    nT = (tt.N + tile - 1) // tile
    hit = np.zeros((nT, nT), bool)
    for t in range(tt.N):
        for k in T.token_ancestors(tt, t):
            hit[t // tile, k // tile] = True
    np.testing.assert_array_equal(sch["fwd_cnt"], hit.sum(axis=1))
    np.testing.assert_array_equal(sch["bwd_cnt"], hit.sum(axis=0))
    assert sch["fwd_cnt"].sum() == sch["bwd_cnt"].sum() == T.tile_pairs(tt, tile)
    for cnt, order in ((sch["fwd_cnt"], sch["fwd_order"]), (sch["bwd_cnt"], sch["bwd_order"])):
        assert sorted(order.tolist()) == list(range(nT))
        keys = [(-int(cnt[i]), int(i)) for i in order]
        assert keys == sorted(keys)
    assert (sch["send"][tt.N:] == 0).all() and len(sch["send"]) == nT * tile
    for b in range(nT):
        real = tt.tok_send[b * tile:(b + 1) * tile]
        assert sch["blk_min"][b] == min(real) and sch["blk_max"][b] == max(real)


def _random_trees():
    out = []
    for seed in range(12):
        out.append(synth.random_tree(seed, n_seg=1 + seed * 3, len_range=(1, 9), max_children=1 + seed % 4))
    out.append(synth.random_tree(99, n_seg=6, len_range=(1, 5), chain=True))
    return out


@pytest.mark.parametrize("shape", _random_trees(), ids=lambda s: f"S{s.S}N{s.N}")
def test_mask_identity_and_invariants(shape):
    """k ∈ anc(t) ⇔ k ≤ t < send[k], by brute-force parent walks; weight/leaf invariants."""
    tt = T.tables(shape.seg_parent, shape.seg_len)
    N = tt.N
    anc = np.zeros((N, N), bool)
    for t in range(N):
        anc[t, T.token_ancestors(tt, t)] = True
    k = np.arange(N)
    rule = (k[None, :] <= k[:, None]) & (k[:, None] < tt.tok_send[None, :])
    np.testing.assert_array_equal(anc, rule)
    # intervals cover exactly the ancestor set, sorted, maximal, half-open
    for t in range(N):
        ivs = T.token_intervals(tt, t)
        cover = np.zeros(N, bool)
        for i, (b, e) in enumerate(ivs):
            assert b < e
            if i:
                assert ivs[i - 1][1] < b, "adjacent intervals must be merged"
            cover[b:e] = True
        np.testing.assert_array_equal(cover, anc[t])
        assert len(ivs) <= tt.seg_depth[tt.tok_seg[t]] + 1
    # pos = |anc(t)| − 1
    np.testing.assert_array_equal(tt.tok_pos, anc.sum(1) - 1)
    # every token is visited exactly once by the layout
    assert sorted(np.concatenate([np.arange(tt.seg_start[s], tt.seg_end[s]) for s in range(tt.S)])) == list(range(N))
    # Σ_t n_t = Σ_b |b|; root weight 1; children leaf counts add up
    assert int(tt.tok_leafcnt.sum()) == tt.stats["sum_branch_tokens"]
    assert tt.tok_weight[0] == 1.0
    ch = T.children(tt.seg_parent)
    for s in range(tt.S):
        if ch[s]:
            assert sum(tt.seg_leafcnt[c] for c in ch[s]) == tt.seg_leafcnt[s]
        else:
            assert tt.seg_leafcnt[s] == 1
    # branch fraction: number of branches through t over B
    brs = T.branches(tt)
    through = np.zeros(N)
    for b in brs:
        through[b] += 1
    np.testing.assert_array_equal(tt.tok_weight, (through / len(brs)).astype(np.float32))
    assert tt.stats["useful_pairs"] == int(anc.sum())


def test_sibling_permutation_relabels_layout():
    """Renumbering siblings reorders the DFS layout but keeps the multiset of branch lengths."""
    a = T.tables([-1, 0, 0, 1, 2], [3, 2, 4, 1, 2])
    b = T.tables([-1, 0, 0, 2, 1], [3, 4, 2, 1, 2])
    assert sorted(len(x) for x in T.branches(a)) == sorted(len(x) for x in T.branches(b))
    assert a.stats["useful_pairs"] == b.stats["useful_pairs"]


def test_invalid_trees():
    with pytest.raises(T.TreeError):
        T.validate([0, 0], [1, 1])          # root must have parent −1
    with pytest.raises(T.TreeError):
        T.validate([-1, 1], [1, 1])         # parent must precede child (also rules out cycles)
    with pytest.raises(T.TreeError):
        T.validate([-1, 0], [1, 0])         # empty segment
    with pytest.raises(T.TreeError):
        T.validate([-1, 0], [1, 2], N=4)    # lengths must sum to N


@pytest.mark.parametrize("cfg,S,N,B,comp", [(0, 7, 196, 4, 2.31), (1, 21, 12669, 16, 3.94),
                                            (3, 73, 45379, 64, 7.95), (4, 59, 32136, 30, 3.45)])
def test_workload_shapes(cfg, S, N, B, comp):
    """Seed-0 workload trees: sizes, leaves and compression near the stated ≈4× / ≈8×."""
    sh = synth.tree_shape(cfg)
    assert (sh.S, sh.N) == (S, N)
    tt = T.tables(sh.seg_parent, sh.seg_len)
    assert tt.B == B
    assert T.compression(tt) == pytest.approx(comp, abs=0.005)
    # closed form for the two-level configs: Σ_b |b| = B·root + Σ_mid n_mid·len_mid + Σ_leaf len_leaf
    if cfg in (1, 3):
        fan = {1: 4, 3: 8}[cfg]
        ln = sh.seg_len
        closed = B * ln[0] + fan * ln[1:1 + fan].sum() + ln[1 + fan:].sum()
        assert tt.stats["sum_branch_tokens"] == closed


def test_golden_greedy_leaf_orders(golden_dir):
    with open(os.path.join(golden_dir, "tree_small.json")) as f:
        cases = json.load(f)["greedy_leaf_orders"]["cases"]
    for c in cases:
        tt = T.tables(c["seg_parent"], c["seg_len"])
        assert T.greedy_leaf_order(tt) == c["order"], c["why"]


@pytest.mark.parametrize("seed", range(10))
def test_greedy_leaf_order_properties(seed):
    """A permutation of the leaves that is a DFS order (every subtree's leaves consecutive), starting at a leaf with
    the longest root path; its consecutive shared-prefix total equals the closed form every DFS order attains:
    Σ over segments v of (children(v) − 1) · (tokens from the root through v)."""
    sh = synth.random_tree(200 + seed, n_seg=3 + 4 * seed, len_range=(1, 12), max_children=1 + seed % 4)
    tt = T.tables(sh.seg_parent, sh.seg_len)
    order = T.greedy_leaf_order(tt)
    assert sorted(order) == sorted(tt.leaves)
    pos = {s: i for i, s in enumerate(order)}
    for v in range(tt.S):
        sub = [x for x in tt.leaves if v in T.segment_path(tt.seg_parent, x)]
        idx = sorted(pos[x] for x in sub)
        assert idx == list(range(idx[0], idx[0] + len(idx))), f"leaves under segment {v} are not consecutive"
    depth = {x: int(tt.seg_pathlen[x] + tt.seg_len[x]) for x in tt.leaves}
    assert depth[order[0]] == max(depth.values())
    paths = {x: T.token_path(tt, x) for x in tt.leaves}
    total = 0
    for a, b in zip(order, order[1:]):
        total += len([1 for u, w in zip(paths[a], paths[b]) if u == w])
    ch = T.children(tt.seg_parent)
    closed = sum((len(ch[v]) - 1) * int(tt.seg_pathlen[v] + tt.seg_len[v]) for v in range(tt.S) if ch[v])
    assert total == closed
