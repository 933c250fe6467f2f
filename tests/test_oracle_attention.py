"""Pins of oracle.attention: library routines, finite differences, brute force, reductions.

Sources: "Tree Training" Abstract (tree-exact attention matching independent
branches); AReaL-DTA Key Contributions 1–2 (gradients of all descendant leaves
accumulate into the shared prefix; right-to-left query chunks).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import tree as T


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _sdpa(q, k, v, scale, C_off=None):
    """PyTorch fp64 scaled_dot_product_attention with a bottom-right causal mask (GQA expanded)."""
    C, hq, d = q.shape
    P, hkv, _ = k.shape
    G = hq // hkv
    qt = torch.tensor(q).permute(1, 0, 2)
    kt = torch.tensor(k).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.tensor(v).permute(1, 0, 2).repeat_interleave(G, 0)
    mask = torch.arange(P)[None, :] <= (P - C + torch.arange(C))[:, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)


@pytest.mark.parametrize("C,P,hq,hkv,d", [(7, 7, 1, 1, 8), (5, 12, 4, 2, 16), (12, 12, 6, 3, 4), (1, 9, 2, 1, 8)])
def test_causal_forward_vs_torch_sdpa(C, P, hq, hkv, d):
    rng = np.random.default_rng(C * 100 + P)
    q, k, v = _rand(rng, C, hq, d), _rand(rng, P, hkv, d), _rand(rng, P, hkv, d)
    scale = 1 / np.sqrt(d)
    o, lse = A.causal_attention_forward(q, k, v, scale)
    ref = _sdpa(q, k, v, scale).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)
    # LSE: logsumexp of the visible scaled scores, via torch.logsumexp
    G = hq // hkv
    for h in range(hq):
        s = torch.tensor(scale * q[:, h] @ k[:, h // G].T)
        s[torch.arange(P)[None, :] > (P - C + torch.arange(C))[:, None]] = -float("inf")
        np.testing.assert_allclose(lse[h], torch.logsumexp(s, 1).numpy(), rtol=1e-13)


@pytest.mark.parametrize("C,P,hq,hkv,d", [(6, 6, 2, 1, 8), (4, 11, 4, 2, 8)])
def test_causal_backward_vs_torch_autograd(C, P, hq, hkv, d):
    rng = np.random.default_rng(7 + C)
    q, k, v, do = _rand(rng, C, hq, d), _rand(rng, P, hkv, d), _rand(rng, P, hkv, d), _rand(rng, C, hq, d)
    scale = 0.3
    dq, dk, dv = A.causal_attention_backward(q, k, v, do, scale)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = hq // hkv
    mask = torch.arange(P)[None, :] <= (P - C + torch.arange(C))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2), kt.permute(1, 0, 2).repeat_interleave(G, 0),
        vt.permute(1, 0, 2).repeat_interleave(G, 0), attn_mask=mask, scale=scale)
    (out * torch.tensor(do).permute(1, 0, 2)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_tree_backward_finite_differences():
    """Central differences of Σ_t ⟨dO_t, O_t⟩ pin the tree gradient itself."""
    sh = synth.random_tree(3, n_seg=4, len_range=(1, 3))
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(1)
    N, hq, hkv, d = tt.N, 2, 1, 3
    Q, K, V, dO = _rand(rng, N, hq, d), _rand(rng, N, hkv, d), _rand(rng, N, hkv, d), _rand(rng, N, hq, d)
    _, _, dQ, dK, dV = A.tree_attention_branches(tt, Q, K, V, dO, scale=0.7)

    def f(Q_, K_, V_):
        O, _ = A.tree_attention_branches(tt, Q_, K_, V_, scale=0.7)
        return float((O * dO).sum())

    eps = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args = [Q, K, V]
            i = [id(Q), id(K), id(V)].index(id(X))
            args[i] = Xp
            fp = f(*args)
            args[i] = Xm
            num[idx] = (fp - f(*args)) / (2 * eps)
        np.testing.assert_allclose(G, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("seed,n_seg,hq,hkv", [(0, 5, 2, 1), (1, 7, 3, 3), (2, 4, 4, 2)])
def test_branch_segment_bruteforce_agree(seed, n_seg, hq, hkv):
    sh = synth.random_tree(seed, n_seg=n_seg, len_range=(1, 5))
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(seed + 10)
    d = 4
    Q, K, V, dO = _rand(rng, tt.N, hq, d), _rand(rng, tt.N, hkv, d), _rand(rng, tt.N, hkv, d), _rand(rng, tt.N, hq, d)
    ref = A.tree_attention_bruteforce(tt, Q, K, V, dO)
    for got in (A.tree_attention_branches(tt, Q, K, V, dO), A.tree_attention_segments(tt, Q, K, V, dO),
                A.dta_chunked(tt, Q, K, V, dO, chunk=2)):
        for x, y in zip(got, ref):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)
    o, lse = A.ancestor_rows_forward(tt, Q, K, V, [0, tt.N - 1])
    np.testing.assert_allclose(o, ref[0][[0, tt.N - 1]], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref[1][:, [0, tt.N - 1]], rtol=1e-12)


def test_single_segment_is_causal_attention():
    rng = np.random.default_rng(5)
    N, hq, hkv, d = 17, 2, 1, 8
    tt = T.tables([-1], [N])
    Q, K, V = _rand(rng, N, hq, d), _rand(rng, N, hkv, d), _rand(rng, N, hkv, d)
    O, LSE = A.tree_attention_branches(tt, Q, K, V)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, 1 / np.sqrt(d)).permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_chain_tree_is_one_causal_sequence():
    sh = synth.random_tree(4, n_seg=5, len_range=(1, 6), chain=True)
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(6)
    hq, hkv, d = 2, 2, 4
    Q, K, V = _rand(rng, tt.N, hq, d), _rand(rng, tt.N, hkv, d), _rand(rng, tt.N, hkv, d)
    O, _ = A.tree_attention_segments(tt, Q, K, V)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, 1 / np.sqrt(d)).permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_sibling_permutation_invariance():
    """Swapping two siblings' indices permutes the layout; per-token results follow the tokens."""
    par_a, len_a = [-1, 0, 0, 1, 2], [3, 2, 4, 1, 2]
    par_b, len_b = [-1, 0, 0, 2, 1], [3, 4, 2, 1, 2]   # segments 1<->2 swapped (children follow)
    ta, tb = T.tables(par_a, len_a), T.tables(par_b, len_b)
    swap = {0: 0, 1: 2, 2: 1, 3: 3, 4: 4}
    perm = np.zeros(ta.N, np.int64)          # token of a -> token of b
    for s in range(ta.S):
        perm[ta.seg_start[s]:ta.seg_end[s]] = np.arange(tb.seg_start[swap[s]], tb.seg_end[swap[s]])
    rng = np.random.default_rng(8)
    Q, K, V, dO = _rand(rng, ta.N, 2, 4), _rand(rng, ta.N, 1, 4), _rand(rng, ta.N, 1, 4), _rand(rng, ta.N, 2, 4)
    Qb, Kb, Vb, dOb = (np.empty_like(x) for x in (Q, K, V, dO))
    for x, xb in ((Q, Qb), (K, Kb), (V, Vb), (dO, dOb)):
        xb[perm] = x
    ra = A.tree_attention_branches(ta, Q, K, V, dO)
    rb = A.tree_attention_branches(tb, Qb, Kb, Vb, dOb)
    np.testing.assert_allclose(ra[0], rb[0][perm], rtol=1e-12)
    np.testing.assert_allclose(ra[1], rb[1][:, perm], rtol=1e-12)
    for i in (2, 3, 4):
        np.testing.assert_allclose(ra[i], rb[i][perm], rtol=1e-11, atol=1e-13)


def test_shared_prefix_gradient_sums_descendants():
    """dK/dV of a prefix token = Σ over branches of that branch's own causal-attention gradient."""
    sh = synth.random_tree(11, n_seg=6, len_range=(2, 4))
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(2)
    Q, K, V, dO = _rand(rng, tt.N, 1, 4), _rand(rng, tt.N, 1, 4), _rand(rng, tt.N, 1, 4), _rand(rng, tt.N, 1, 4)
    _, _, _, dK, dV = A.tree_attention_segments(tt, Q, K, V, dO)
    # root token 0 is seen by every token: its dV is Σ_t P_t0 dO_t over all t
    O, LSE = A.tree_attention_segments(tt, Q, K, V)
    p0 = np.exp(0.5 * (Q[:, 0] @ K[0, 0]) - LSE[0])
    np.testing.assert_allclose(dV[0, 0], p0 @ dO[:, 0], rtol=1e-12)


def test_planted_mistake_is_caught():
    """A wrong mask (strictly-below-diagonal) in a copy of the forward fails the SDPA pin."""
    rng = np.random.default_rng(0)
    q, k, v = _rand(rng, 5, 1, 4), _rand(rng, 5, 1, 4), _rand(rng, 5, 1, 4)
    bad = np.zeros_like(q)
    for i in range(5):
        s = 0.5 * (k[:i + 1, 0] @ q[i, 0])
        s[-1] = -np.inf if i else s[-1]          # drops the diagonal key
        p = np.exp(s - s.max())
        bad[i, 0] = p @ v[:i + 1, 0] / p.sum()
    ref = _sdpa(q, k, v, 0.5).permute(1, 0, 2).numpy()
    assert not np.allclose(bad, ref, rtol=1e-6)
    good, _ = A.causal_attention_forward(q, k, v, 0.5)
    np.testing.assert_allclose(good, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("seed,chunk", [(7, 16), (8, 5)])
def test_dta_greedy_order_equals_segments(seed, chunk):
    """The path-at-a-time traversal in the greedy leaf order gives the same forward and gradients as the
    per-segment definition (the visiting order changes only the order of the accumulations)."""
    sh = synth.random_tree(seed, n_seg=9, len_range=(3, 20), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(2, 1, 64))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    args = [synth.bf16_bits_to_f32(inp[k]).astype(np.float64) for k in ("Q", "K", "V", "dO")]
    ref = A.tree_attention_segments(tab, *args)
    got = A.dta_chunked(tab, *args, chunk=chunk, leaf_order=T.greedy_leaf_order(tab))
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-12)
