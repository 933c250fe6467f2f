"""tt_tree_build against the oracle: every table bit-exact (integers and fp32 weights), and the tile schedules
it writes for the attention kernels against the oracle's plain definition (tile 128)."""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import tree as T

pytestmark = pytest.mark.gpu


def _build(tt, par, ln, **kw):
    p = torch.tensor(np.asarray(par, np.int32), device="cuda")
    l = torch.tensor(np.asarray(ln, np.int32), device="cuda")
    return tt.tree_build(p, l, **kw)


def _compare_schedules(tt, dev, ref):
    got = {k: v.cpu().numpy() for k, v in tt.tree_schedules(dev).items()}
    want = T.tile_schedules(ref, tile=128)
    for k, v in want.items():
        np.testing.assert_array_equal(got[k], v, err_msg=f"schedule {k}")


def _compare(dev, ref, tt=None):
    for key in ("seg_start", "seg_subtree_end", "seg_depth", "seg_pathlen", "seg_leafcnt", "iv_ptr", "tok_seg",
                "tok_pos", "tok_send", "tok_leafcnt"):
        np.testing.assert_array_equal(getattr(dev, key).cpu().numpy(), getattr(ref, key), err_msg=key)
    n_iv = int(ref.iv_ptr[-1])
    np.testing.assert_array_equal(dev.iv[:n_iv].cpu().numpy(), ref.iv)
    w = dev.tok_weight.cpu().numpy()
    assert w.dtype == np.float32
    np.testing.assert_array_equal(w.view(np.uint32), ref.tok_weight.view(np.uint32))
    st = dev.stats.cpu().numpy()
    s = ref.stats
    assert list(st) == [s["B"], s["N"], s["sum_branch_tokens"], s["useful_pairs"], s["tile_pairs"], s["iv_pairs"],
                        s["max_depth"], s["max_path"]]
    if tt is not None:
        _compare_schedules(tt, dev, ref)


def test_golden(tt, golden_dir):
    for g in json.load(open(os.path.join(golden_dir, "tree_small.json")))["trees"]:
        dev = _build(tt, g["seg_parent"], g["seg_len"]).check()
        _compare(dev, T.tables(g["seg_parent"], g["seg_len"]), tt)


@pytest.mark.parametrize("seed", range(8))
def test_random_trees(tt, seed):
    sh = synth.random_tree(seed, n_seg=1 + 9 * seed, len_range=(1, 300), max_children=1 + seed % 5)
    dev = _build(tt, sh.seg_parent, sh.seg_len).check()
    _compare(dev, T.tables(sh.seg_parent, sh.seg_len), tt)


@pytest.mark.parametrize("cfg", [0, 1, 3, 4])
def test_workload_trees(tt, cfg):
    sh = synth.tree_shape(cfg)
    dev = _build(tt, sh.seg_parent, sh.seg_len).check()
    _compare(dev, T.tables(sh.seg_parent, sh.seg_len), tt)


def test_wide_deep_tree(tt):
    # 600 segments, chain + fan-out mix, several hundred 128-token tiles
    sh = synth.random_tree(123, n_seg=600, len_range=(1, 100), max_children=2)
    dev = _build(tt, sh.seg_parent, sh.seg_len).check()
    _compare(dev, T.tables(sh.seg_parent, sh.seg_len), tt)


@pytest.mark.parametrize("par,ln", [([0, 0], [1, 1]), ([-1, 1], [2, 2]), ([-1, 0], [3, 0]), ([-1, 5, 0], [1, 1, 1])])
def test_invalid_tree_sets_error(tt, par, ln):
    dev = _build(tt, par, ln, N=max(1, sum(x for x in ln if x > 0)))
    assert int(dev.err.item()) == -2
    # attention given that workspace refuses to run and reports the same error
    N = dev.N
    Q = torch.zeros(N, 1, 64, dtype=torch.bfloat16, device="cuda")
    err = tt.new_err("cuda")
    tt.tree_attn_fwd(dev, Q, Q, Q, err=err)
    assert int(err.item()) == -2


def test_interval_capacity_too_small(tt):
    sh = synth.tree_shape(3)
    ref = T.tables(sh.seg_parent, sh.seg_len)
    dev = _build(tt, sh.seg_parent, sh.seg_len, iv_capacity=5)
    assert int(dev.err.item()) == -4
    assert int(dev.stats[5].item()) == ref.stats["iv_pairs"]


def test_single_token(tt):
    dev = _build(tt, [-1], [1]).check()
    assert dev.tok_weight.item() == 1.0 and dev.stats.cpu().tolist()[:4] == [1, 1, 1, 1]
