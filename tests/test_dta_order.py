"""The path-at-a-time traversal's leaf order (tt_dta_leaf_order, host code behind the C ABI) against the oracle.

Greedy order: the oracle walks the leaves one by one (next = the unvisited leaf sharing the most prefix tokens with
the current one, ties to the longer root path, then the lower index); the library sorts each segment's children by
the depth of their deepest leaf. The two are independent computations of the same order. Index order: the leaves
in the DFS layout of tt_tree_build.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import tree as T


@pytest.fixture(scope="module")
def tt():
    import prefix_tree_gb300 as tt
    return tt


def _trees():
    out = [synth.random_tree(300 + s, n_seg=2 + 5 * s, len_range=(1, 30), max_children=1 + s % 5) for s in range(12)]
    out += [synth.tree_shape(w) for w in (0, 1, 3, 4)]
    return out


def test_golden_orders(tt, golden_dir):
    with open(os.path.join(golden_dir, "tree_small.json")) as f:
        cases = json.load(f)["greedy_leaf_orders"]["cases"]
    for c in cases:
        assert tt.dta_leaf_order(c["seg_parent"], c["seg_len"]).tolist() == c["order"], c["why"]


@pytest.mark.parametrize("shape", _trees(), ids=lambda s: f"S{s.S}N{s.N}")
def test_greedy_and_index_orders_match_oracle(tt, shape):
    tab = T.tables(shape.seg_parent, shape.seg_len)
    assert tt.dta_leaf_order(shape.seg_parent, shape.seg_len, tt.DTA_ORDER_GREEDY).tolist() == T.greedy_leaf_order(tab)
    dfs = sorted(tab.leaves, key=lambda s: tab.seg_start[s])
    assert tt.dta_leaf_order(shape.seg_parent, shape.seg_len, tt.DTA_ORDER_INDEX).tolist() == dfs


def test_errors(tt):
    with pytest.raises(tt.TTError):
        tt.dta_leaf_order([0, 0], [1, 1])          # no root
    with pytest.raises(tt.TTError):
        tt.dta_leaf_order([-1, 0], [1, 1], 7)      # unknown order
    par = np.array([-1, 0, 0], np.int32)
    ln = np.array([2, 2, 2], np.int32)
    out = np.zeros(1, np.int32)
    import ctypes
    rc = tt.lib().tt_dta_leaf_order(par.ctypes.data_as(ctypes.c_void_p), ln.ctypes.data_as(ctypes.c_void_p), 3, 1,
                                    out.ctypes.data_as(ctypes.c_void_p), 1)
    assert rc == -4  # two leaves, capacity one
