"""tt_tree_partition (host code behind the C ABI) against the oracle's partitioning rule (oracle/partition.py):
the same partitions, bit for bit, in both visiting orders and for several budgets."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import partition as PT
from oracle import tree as T


@pytest.fixture(scope="module")
def tt():
    import prefix_tree_gb300 as tt
    return tt


def _as_list(parts):
    first, rows, path, kind = parts
    return [[int(a), int(b), int(c), int(d)] for a, b, c, d in zip(first, rows, path, kind)]


def test_golden_partitions(tt, golden_dir):
    with open(os.path.join(golden_dir, "partition_small.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        for order in (tt.DTA_ORDER_INDEX, tt.DTA_ORDER_GREEDY):
            assert _as_list(tt.tree_partition(c["seg_parent"], c["seg_len"], c["budget"], order)) == c["partitions"]


def _trees():
    out = [synth.random_tree(900 + s, n_seg=3 + 5 * s, len_range=(1, 120), max_children=1 + s % 5) for s in range(10)]
    out.append(synth.random_tree(990, n_seg=150, len_range=(1, 6), max_children=7))
    out += [synth.tree_shape(w) for w in (0, 1, 4)]
    return out


@pytest.mark.parametrize("shape", _trees(), ids=lambda s: f"S{s.S}N{s.N}")
def test_matches_oracle(tt, shape):
    tab = T.tables(shape.seg_parent, shape.seg_len)
    for budget in (1, 37, 256, 2048, 10 ** 7):
        for order, name in ((tt.DTA_ORDER_INDEX, "index"), (tt.DTA_ORDER_GREEDY, "greedy")):
            got = _as_list(tt.tree_partition(shape.seg_parent, shape.seg_len, budget, order))
            assert got == [list(p) for p in PT.partitions(tab, budget, name)], (budget, name)


def test_arguments(tt):
    import ctypes
    L = tt.lib()
    par = np.array([-1, 0, 0], np.int32)
    ln = np.array([4, 2, 2], np.int32)
    vp = ctypes.c_void_p
    pp, lp = par.ctypes.data_as(vp), ln.ctypes.data_as(vp)
    assert L.tt_tree_partition(pp, lp, 3, 3, 1, None, None, None, None, 0) == 4   # count: root chunks 3+1, two packs
    assert L.tt_tree_partition(pp, lp, 3, 0, 1, None, None, None, None, 0) == -1  # budget < 1
    assert L.tt_tree_partition(pp, lp, 3, 3, 7, None, None, None, None, 0) == -1  # unknown order
    buf = np.zeros(4, np.int64)
    k = np.zeros(4, np.int32)
    bp, kp = buf.ctypes.data_as(vp), k.ctypes.data_as(vp)
    assert L.tt_tree_partition(pp, lp, 3, 3, 1, bp, bp, bp, kp, 1) == -4  # capacity too small
    bad = np.array([-1, 2, 0], np.int32)
    assert L.tt_tree_partition(bad.ctypes.data_as(vp), lp, 3, 3, 1, None, None, None, None, 0) == -2
