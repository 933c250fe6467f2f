"""Tree attention fwd/bwd (tt_tree_attn_fwd / tt_tree_attn_bwd) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import tree as T
from tests._util import GRAD_RL2, LSE_RTOL, O_ATOL, dev_to_f64, f64, rel_l2, to_dev_bf16, workload_oracle

pytestmark = pytest.mark.gpu


def run_gpu(tt, sh, inp, tiles=None):
    par = torch.tensor(sh.seg_parent, device="cuda")
    ln = torch.tensor(sh.seg_len, device="cuda")
    tree = tt.tree_build(par, ln).check()
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    O, LSE = tt.tree_attn_fwd(tree, Q, K, V, tiles=tiles)
    dQ, dK, dV = tt.tree_attn_bwd(tree, Q, K, V, O, LSE, dO)
    torch.cuda.synchronize()
    tree.check()
    return dict(O=dev_to_f64(O), LSE=LSE.cpu().numpy().astype(np.float64), dQ=dev_to_f64(dQ), dK=dev_to_f64(dK),
                dV=dev_to_f64(dV))


def check_full(got, ref, heads=None, kv_heads=None):
    O, LSE, dQ, dK, dV = ref
    hs = slice(None) if heads is None else heads
    gs = slice(None) if kv_heads is None else kv_heads
    assert np.abs(got["O"][:, hs] - O[:, hs]).max() <= O_ATOL
    assert np.abs(got["LSE"][hs] - LSE[hs]).max() / np.abs(LSE[hs]).max() <= LSE_RTOL
    assert (np.abs(got["LSE"][hs] - LSE[hs]) <= LSE_RTOL * np.abs(LSE[hs]) + 1e-5).all()
    assert rel_l2(got["dQ"][:, hs], dQ[:, hs]) <= GRAD_RL2
    assert rel_l2(got["dK"][:, gs], dK[:, gs]) <= GRAD_RL2
    assert rel_l2(got["dV"][:, gs], dV[:, gs]) <= GRAD_RL2


def oracle_inputs(inp):
    return [f64(inp[k]) for k in ("Q", "K", "V", "dO")]


@pytest.mark.parametrize("seed,n_seg,lens,heads", [
    (0, 6, (50, 300), (2, 1, 64)),
    (1, 9, (1, 200), (4, 2, 128)),
    (2, 14, (20, 140), (3, 3, 64)),
    (3, 5, (100, 400), (6, 2, 128)),
    (4, 25, (1, 60), (5, 1, 128)),
    (5, 3, (129, 257), (2, 2, 64)),
])
def test_random_trees(tt, seed, n_seg, lens, heads):
    sh = synth.random_tree(seed, n_seg=n_seg, len_range=lens, max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=heads)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.tree_attention_segments(tab, *oracle_inputs(inp))
    check_full(run_gpu(tt, sh, inp), ref)


def test_tiny_workload_vs_branches(tt):
    inp = synth.attention_inputs(0)
    sh = inp["tree"]
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.tree_attention_branches(tab, *oracle_inputs(inp))
    check_full(run_gpu(tt, sh, inp), ref)


@pytest.mark.parametrize("kind", ["single", "chain", "star", "one_token_segments"])
def test_special_trees(tt, kind):
    if kind == "single":
        sh = synth.TreeShape(np.array([-1], np.int32), np.array([333], np.int32), np.random.default_rng(0))
    elif kind == "chain":
        sh = synth.random_tree(7, n_seg=7, len_range=(10, 100), chain=True)
    elif kind == "star":
        par = np.array([-1] + [0] * 40, np.int32)
        sh = synth.TreeShape(par, np.array([200] + [7 + 3 * i for i in range(40)], np.int32),
                             np.random.default_rng(1))
    else:
        sh = synth.random_tree(8, n_seg=150, len_range=(1, 1), max_children=4)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.tree_attention_segments(tab, *oracle_inputs(inp))
    got = run_gpu(tt, sh, inp)
    check_full(got, ref)
    if kind in ("single", "chain"):   # reduces to plain causal attention over the sequence
        o, lse = A.causal_attention_forward(*oracle_inputs(inp)[:3], scale=1 / np.sqrt(128))
        assert np.abs(got["O"] - o).max() <= O_ATOL


def _sample_rows(tab, n, seed=0):
    rng = np.random.default_rng(seed)
    firsts = tab.seg_start[:min(tab.S, 40)]
    lasts = tab.seg_end[:min(tab.S, 40)] - 1
    return np.unique(np.r_[firsts, lasts, rng.integers(0, tab.N, n)])


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_workload_full_size(tt, cfg):
    """Full-size workloads: O/LSE on sampled rows of every head; gradients (and O/LSE) in full for every KV group
    of the Qwen3-1.7B-shaped tree, for the last KV group of the larger trees."""
    groups = tuple(range(8)) if cfg == 1 else (7,)
    inp, tab, ref = workload_oracle(cfg, groups)
    sh = inp["tree"]
    got = run_gpu(tt, sh, inp)
    Qf, Kf, Vf, dOf = oracle_inputs(inp)
    rows = _sample_rows(tab, 96)
    o, lse = A.ancestor_rows_forward(tab, Qf, Kf, Vf, rows)
    assert np.abs(got["O"][rows] - o).max() <= O_ATOL
    assert (np.abs(got["LSE"][:, rows] - lse) <= LSE_RTOL * np.abs(lse) + 1e-5).all()
    G = inp["hq"] // inp["hkv"]
    for g in groups:
        check_full(got, ref, heads=slice(g * G, (g + 1) * G), kv_heads=[g])


@pytest.mark.parametrize("tiles", [1, 2])
@pytest.mark.parametrize("seed,n_seg,lens,heads", [
    (40, 9, (30, 400), (4, 2, 128)),   # head pairs (even group size)
    (41, 12, (1, 300), (5, 1, 128)),   # tile pairs, odd number of query tiles possible
    (42, 6, (100, 500), (3, 3, 64)),   # tile pairs, one head per group
    (43, 20, (1, 90), (8, 2, 64)),     # head pairs, many short segments
    (44, 10, (20, 300), (6, 2, 128)),  # odd group size over two groups: one head pair + the last head's tile pairs
    (45, 7, (50, 400), (14, 2, 64)),   # group size 7: three head pairs per group + tile pairs
])
def test_forward_schedules(tt, tiles, seed, n_seg, lens, heads):
    """One query tile per CTA and two per CTA (head or tile pairs) both match the oracle."""
    sh = synth.random_tree(seed, n_seg=n_seg, len_range=lens, max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=heads)
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.tree_attention_segments(tab, *oracle_inputs(inp))
    check_full(run_gpu(tt, sh, inp, tiles=tiles), ref)


def test_kernel_timing_counts_launches(tt):
    """Launch timing sees one forward and one backward launch per whole-tree fwd+bwd."""
    sh = synth.random_tree(44, n_seg=6, len_range=(50, 300), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tt.kernel_timing(True)
    run_gpu(tt, sh, inp)
    tt.kernel_timing(False)
    times, dropped = tt.kernel_timing_read()
    assert dropped == 0
    assert [times[c][1] for c in ("fwd", "bwd", "logprob")] == [1, 1, 0]
    assert all(times[c][0] > 0 for c in ("fwd", "bwd"))
    tt.kernel_timing(True)  # clears
    assert tt.kernel_timing_read()[0]["fwd"] == (0.0, 0)
    tt.kernel_timing(False)
