"""Per-token log-probabilities, the branch-average loss and its weighted-token form (oracle).

Source: "Tree Training", Abstract. The mean of the per-branch losses, each
branch taken on its own, is the same number as one sum over the tree's tokens
in which a token's term is scaled by the share of branches that contain it;
so each token's log-probability needs to be computed only once.

Readings where the pages are silent:
* a branch's loss is the SUM of its tokens' negative log-probabilities (only
  then is the weight exactly the branch fraction n_t / B);
* row t of the logits predicts token t's target (the caller aligns rows);
* dlogits is the gradient of g·loss.

Test infrastructure only. fp64 throughout; inputs are the bf16 values the GPU
receives, widened exactly.
"""
from __future__ import annotations

import numpy as np

from . import tree as _tree


def log_softmax_rows(z):
    """logsumexp per row and log p = z − lse, computed stably in fp64."""
    z = np.asarray(z, np.float64)
    m = z.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(z - m).sum(axis=1))
    return lse, z - lse[:, None]


def weighted_token_loss(logits, targets, weights, g=1.0, want_dlogits=True):
    """logp_t = z_{t,y_t} − lse_t;  loss = −Σ_t w_t logp_t;  dlogits = g w_t (softmax_t − onehot(y_t))."""
    z = np.asarray(logits, np.float64)
    y = np.asarray(targets, np.int64)
    w = np.asarray(weights, np.float64)
    lse, _ = log_softmax_rows(z)
    rows = np.arange(z.shape[0])
    logp = z[rows, y] - lse
    loss = float(-(w * logp).sum())
    if not want_dlogits:
        return logp, loss, None
    p = np.exp(z - lse[:, None])
    p[rows, y] -= 1.0
    return logp, loss, g * w[:, None] * p


def branch_average_loss(tt, logits, targets, g=1.0):
    """Loss averaged over independently linearised branches (the definition).

    Each branch b is an ordinary sequence; its loss is L_b = −Σ_{t∈b} log p_t.
    The tree loss is (1/B)·Σ_b L_b. dlogits: each branch copy of row t
    contributes (1/B)(softmax_t − onehot(y_t)), scatter-added onto tree rows,
    times g. Returns (per-token logp, loss, dlogits).
    """
    z = np.asarray(logits, np.float64)
    y = np.asarray(targets, np.int64)
    brs = _tree.branches(tt)
    B = len(brs)
    logp_tree = np.full(z.shape[0], np.nan)
    total = 0.0
    dlogits = np.zeros_like(z)
    for br in brs:
        lse, _ = log_softmax_rows(z[br])
        lp = z[br, y[br]] - lse
        total += -lp.sum()
        logp_tree[br] = lp
        p = np.exp(z[br] - lse[:, None])
        p[np.arange(len(br)), y[br]] -= 1.0
        np.add.at(dlogits, br, p / B)
    return logp_tree, total / B, g * dlogits


def weighted_loss_sampled(logits_rows_fn, n_rows, targets, weights, chunk=256):
    """Loss −Σ w_t logp_t over a logits matrix too large for fp64 in memory.

    `logits_rows_fn(lo, hi)` returns the rows [lo, hi) widened to fp64; rows
    are processed in fixed blocks. Returns (logp [n_rows], loss).
    """
    logp = np.empty(n_rows)
    for lo in range(0, n_rows, chunk):
        hi = min(n_rows, lo + chunk)
        lp, _, _ = weighted_token_loss(logits_rows_fn(lo, hi), targets[lo:hi], weights[lo:hi],
                                       want_dlogits=False)
        logp[lo:hi] = lp
    return logp, float(-(np.asarray(weights, np.float64) * logp).sum())
