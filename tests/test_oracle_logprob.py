"""Pins of oracle.logprob: the branch-average identity, closed forms and library routines.

Source: "Tree Training" Abstract — the mean of the branch losses is one sum over
tokens, each scaled by the share of branches that contain it.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import logprob as L
from oracle import tree as T


@pytest.mark.parametrize("seed,n_seg", [(0, 1), (1, 4), (2, 9), (3, 15)])
def test_branch_average_equals_weighted_token_loss(seed, n_seg):
    sh = synth.random_tree(seed, n_seg=n_seg, len_range=(1, 7))
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(seed)
    V = 11
    z = rng.standard_normal((tt.N, V)) * 2
    y = rng.integers(0, V, tt.N)
    lp_b, loss_b, dl_b = L.branch_average_loss(tt, z, y, g=1.7)
    w = tt.tok_leafcnt / tt.B          # exact fp64 branch fraction
    lp_w, loss_w, dl_w = L.weighted_token_loss(z, y, w, g=1.7)
    assert abs(loss_b - loss_w) <= 1e-12 * abs(loss_w)
    np.testing.assert_allclose(lp_b, lp_w, rtol=1e-14)
    np.testing.assert_allclose(dl_b, dl_w, rtol=1e-12, atol=1e-15)


def test_identity_on_tiny_workload():
    inp = synth.logprob_inputs(0)
    tt = T.tables(inp["tree"].seg_parent, inp["tree"].seg_len)
    z = synth.bf16_bits_to_f32(inp["logits"]).astype(np.float64)
    _, loss_b, _ = L.branch_average_loss(tt, z, inp["targets"])
    _, loss_w, _ = L.weighted_token_loss(z, inp["targets"], tt.tok_leafcnt / tt.B)
    assert abs(loss_b - loss_w) <= 1e-9 * abs(loss_w)


def test_vs_torch_log_softmax_and_autograd():
    rng = np.random.default_rng(3)
    z = rng.standard_normal((9, 37)) * 3
    y = rng.integers(0, 37, 9)
    w = rng.random(9)
    lp, loss, dl = L.weighted_token_loss(z, y, w, g=0.5)
    zt = torch.tensor(z, requires_grad=True)
    lpt = torch.log_softmax(zt, 1)[torch.arange(9), torch.tensor(y)]
    lt = -(torch.tensor(w) * lpt).sum()
    (0.5 * lt).backward()
    np.testing.assert_allclose(lp, lpt.detach().numpy(), rtol=1e-14)
    assert loss == pytest.approx(lt.item(), rel=1e-14)
    np.testing.assert_allclose(dl, zt.grad.numpy(), rtol=1e-12, atol=1e-16)


def test_closed_forms():
    # uniform logits: log p = −ln V exactly, softmax = 1/V
    V = 1000
    lp, loss, dl = L.weighted_token_loss(np.full((3, V), 0.75), [0, 5, 999], [1.0, 0.5, 0.25])
    np.testing.assert_allclose(lp, -np.log(V), rtol=1e-15)
    assert loss == pytest.approx(1.75 * np.log(V), rel=1e-15)
    assert dl[0, 0] == pytest.approx(1 / V - 1) and dl[1, 0] == pytest.approx(0.5 / V)
    # V = 1: log p = 0, dlogits = 0
    lp, loss, dl = L.weighted_token_loss(np.array([[3.0], [-2.0]]), [0, 0], [1.0, 1.0])
    assert np.all(lp == 0) and loss == 0 and np.all(dl == 0)
    # two classes, logits (0, ln 3): softmax (1/4, 3/4)
    lp, loss, dl = L.weighted_token_loss(np.array([[0.0, np.log(3.0)]]), [0], [2.0])
    assert lp[0] == pytest.approx(np.log(0.25), rel=1e-15)
    np.testing.assert_allclose(dl[0], [2 * (0.25 - 1), 2 * 0.75], rtol=1e-14)


def test_sampled_loss_matches_full():
    rng = np.random.default_rng(4)
    z = rng.standard_normal((700, 50))
    y = rng.integers(0, 50, 700)
    w = rng.random(700)
    lp_full, loss_full, _ = L.weighted_token_loss(z, y, w, want_dlogits=False)
    lp, loss = L.weighted_loss_sampled(lambda lo, hi: z[lo:hi], 700, y, w, chunk=128)
    np.testing.assert_allclose(lp, lp_full, rtol=1e-15)
    assert loss == pytest.approx(loss_full, rel=1e-14)


def test_planted_mean_loss_breaks_identity():
    """Per-branch MEAN loss (the other reading) does not equal the leaf-fraction weighting."""
    sh = synth.random_tree(5, n_seg=5, len_range=(2, 9))
    tt = T.tables(sh.seg_parent, sh.seg_len)
    rng = np.random.default_rng(0)
    z = rng.standard_normal((tt.N, 6))
    y = rng.integers(0, 6, tt.N)
    brs = T.branches(tt)
    lse, _ = L.log_softmax_rows(z)
    lp = z[np.arange(tt.N), y] - lse
    mean_loss = np.mean([-lp[b].mean() for b in brs])
    _, loss_w, _ = L.weighted_token_loss(z, y, tt.tok_leafcnt / tt.B)
    assert abs(mean_loss - loss_w) > 1e-3 * abs(loss_w)
