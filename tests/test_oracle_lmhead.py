"""Pins of oracle.lmhead: the LM head's loss and gradients against cases fixed by the mathematics.

Source: "Tree Training", Abstract (weighted per-token loss == branch-average
loss); the LM head is the product z = H·Wᵀ in front of it.
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import lmhead as LH
from oracle import logprob as L


def _case(seed, N=7, V=13, Hd=5):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, Hd))
    W = rng.standard_normal((V, Hd))
    y = rng.integers(0, V, N)
    w = rng.random(N)
    return H, W, y, w


def test_identity_head_reduces_to_the_log_prob_loss():
    """W = I (V = Hd): z = H exactly, so every output is the (pinned) weighted log-prob of H."""
    H, _, y, w = _case(0, N=9, V=6, Hd=6)
    out = LH.lmhead_weighted_loss(H, np.eye(6), y, w, g=1.3)
    lp, loss, dz = L.weighted_token_loss(H, y, w, g=1.3)
    np.testing.assert_array_equal(out["logp"], lp)
    assert out["loss"] == loss
    np.testing.assert_array_equal(out["dH"], dz)  # dz·I
    np.testing.assert_array_equal(out["dW"], dz.T @ H)


def test_equal_rows_give_uniform_log_probs():
    """All vocabulary rows equal: every logit of a row is the same, so logp = −log V and lse = z + log V."""
    rng = np.random.default_rng(1)
    N, V, Hd = 6, 37, 8
    H = rng.standard_normal((N, Hd))
    W = np.tile(rng.standard_normal(Hd), (V, 1))
    y = rng.integers(0, V, N)
    out = LH.lmhead_weighted_loss(H, W, y, np.ones(N))
    np.testing.assert_allclose(out["logp"], -math.log(V), rtol=1e-14)
    np.testing.assert_allclose(out["lse"], H @ W[0] + math.log(V), rtol=1e-13, atol=1e-13)
    assert abs(out["loss"] - N * math.log(V)) <= 1e-12 * N * math.log(V)


def test_brute_force_loops():
    """Scalar loops: dot products, log-sum-exp with math.fsum, the weighted sum."""
    H, W, y, w = _case(2)
    out = LH.lmhead_weighted_loss(H, W, y, w, want_grads=False)
    total = []
    for t in range(H.shape[0]):
        z = [math.fsum(H[t, k] * W[v, k] for k in range(H.shape[1])) for v in range(W.shape[0])]
        m = max(z)
        lse = m + math.log(math.fsum(math.exp(x - m) for x in z))
        assert abs(out["logp"][t] - (z[y[t]] - lse)) <= 1e-12
        total.append(-w[t] * (z[y[t]] - lse))
    assert abs(out["loss"] - math.fsum(total)) <= 1e-12


@pytest.mark.parametrize("which", ["H", "W"])
def test_gradients_by_central_differences(which):
    """dH and dW are the gradients of g·loss: checked entry by entry against (f(x+ε) − f(x−ε)) / 2ε."""
    H, W, y, w = _case(3, N=4, V=6, Hd=3)
    g = 0.7
    out = LH.lmhead_weighted_loss(H, W, y, w, g=g)
    X = H if which == "H" else W
    eps = 1e-6
    for idx in np.ndindex(X.shape):
        Xp, Xm = X.copy(), X.copy()
        Xp[idx] += eps
        Xm[idx] -= eps
        args_p = (Xp, W) if which == "H" else (H, Xp)
        args_m = (Xm, W) if which == "H" else (H, Xm)
        fp = LH.lmhead_weighted_loss(*args_p, y, w, want_grads=False)["loss"]
        fm = LH.lmhead_weighted_loss(*args_m, y, w, want_grads=False)["loss"]
        assert abs(g * (fp - fm) / (2 * eps) - out["d" + which][idx]) <= 1e-6


def test_gradients_vs_autograd():
    H, W, y, w = _case(4, N=11, V=17, Hd=6)
    out = LH.lmhead_weighted_loss(H, W, y, w, g=2.0)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    lp = torch.log_softmax(Ht @ Wt.T, 1)[torch.arange(11), torch.tensor(y)]
    (2.0 * -(torch.tensor(w) * lp).sum()).backward()
    np.testing.assert_allclose(out["dH"], Ht.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out["dW"], Wt.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_sampled_rows_match_the_full_computation():
    d = synth.lmhead_inputs(0, n_rows=40, vocab=3001, hidden=64)
    H = synth.bf16_bits_to_f32(d["H"]).astype(np.float64)
    W = synth.bf16_bits_to_f32(d["W"]).astype(np.float64)
    out = LH.lmhead_weighted_loss(H, W, d["targets"], np.ones(40), want_grads=False)
    rows = np.array([0, 7, 39])
    lse, logp = LH.lmhead_rows(H, W, d["targets"], rows, vchunk=700)
    np.testing.assert_allclose(lse, out["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(logp, out["logp"][rows], rtol=1e-12, atol=1e-13)


def test_generator_scale():
    """W's scale 2/√Hd gives logits with about the log-prob workload's N(0, 2²) spread."""
    d = synth.lmhead_inputs(0, n_rows=64, vocab=4096, hidden=256)
    z = LH.logits(synth.bf16_bits_to_f32(d["H"]), synth.bf16_bits_to_f32(d["W"]))
    assert 1.8 < z.std() < 2.2
