"""LM head fused with the weighted log-prob loss (oracle).

Source: "Tree Training", Abstract: averaging the per-branch losses equals one
pass over the tree's tokens with each token's term scaled by the share of
branches through it, so every token's log-probability is computed once. The
LM head in front of that loss is the plain product of the final hidden
states with the vocabulary matrix: the logit of vocabulary entry v at row t
is <H_t, W_v>. The pages give no detail of this step; readings:
* H is [N, Hd] (one row per tree token, the caller aligns row t with the
  prediction of token t as for the log-prob loss), W is [V, Hd] (the layout
  of a linear layer's weight), z = H·Wᵀ;
* the loss on z is exactly the weighted log-prob of oracle.logprob
  (branch loss = sum of its tokens' negative log-probabilities);
* the gradients are those of g·loss: dz = g·w_t·(softmax_t − onehot(y_t)),
  dH = dz·W, dW = dzᵀ·H.

Test infrastructure only: used by the tests, the smoke check and the CPU
baseline leg of the benchmark, never by the library. fp64 throughout on the
bf16 values the GPU receives, widened exactly.
"""
from __future__ import annotations

import numpy as np

from .logprob import log_softmax_rows, weighted_token_loss


def logits(H, W):
    """z = H·Wᵀ in fp64 (library matrix product)."""
    return np.asarray(H, np.float64) @ np.asarray(W, np.float64).T


def lmhead_weighted_loss(H, W, targets, weights, g=1.0, want_grads=True):
    """logp [N], lse [N], loss, and (if want_grads) dH [N, Hd], dW [V, Hd] of g·loss."""
    z = logits(H, W)
    lse, _ = log_softmax_rows(z)
    logp, loss, dz = weighted_token_loss(z, targets, weights, g=g, want_dlogits=want_grads)
    out = {"logp": logp, "lse": lse, "loss": loss}
    if want_grads:
        out["dH"] = dz @ np.asarray(W, np.float64)
        out["dW"] = dz.T @ np.asarray(H, np.float64)
    return out


def lmhead_rows(H, W, targets, rows, vchunk=16384, widen=None):
    """lse and logp of the selected rows only, W taken in vocabulary chunks.

    For matrices too large to hold z (or W) in fp64: row t's logits are formed
    chunk by chunk and folded into a running maximum and rescaled sum.
    `widen` maps a slice of W to fp64 (default: a plain conversion; pass the
    bf16-bits widening for raw bf16 storage).
    """
    widen = (lambda x: np.asarray(x, np.float64)) if widen is None else widen
    h = np.asarray(H, np.float64)[np.asarray(rows)]
    V = W.shape[0]
    m = np.full(len(rows), -np.inf)
    s = np.zeros(len(rows))
    zt = np.empty(len(rows))
    y = np.asarray(targets)[np.asarray(rows)]
    for lo in range(0, V, vchunk):
        hi = min(V, lo + vchunk)
        z = h @ widen(W[lo:hi]).T
        cm = z.max(axis=1)
        nm = np.maximum(m, cm)
        s = s * np.exp(m - nm) + np.exp(z - nm[:, None]).sum(axis=1)
        m = nm
        inside = (y >= lo) & (y < hi)
        zt[inside] = z[inside, y[inside] - lo]
    lse = m + np.log(s)
    return lse, zt - lse
