"""Tree attention, forward and backward, in fp64 (oracle).

Source: "Tree Training", Abstract — full attention adapted to the DFS layout
so that every token's result matches the independent per-branch computation
exactly; AReaL-DTA, Key Contributions 1 and "Methodology in Plain English" —
the tree walked path by path from the root, shared prefix segments backpropagated once
with the gradients of all descendant leaves accumulated; Key Contributions 2 —
long suffixes split into fixed-length query chunks processed right to left.

Definitions used (readings where the pages are silent):
* token t attends to anc(t), its root-to-t path including t;
* scores are scale·q·k with scale = 1/√d; LSE is the natural-log
  log-sum-exp of the scaled scores;
* grouped-query attention: query head h uses key/value head h // (Hq/Hkv);
* the backward pass is the vector-Jacobian product of Σ_t ⟨dO_t, O_t⟩.

Inputs are the bf16 values the GPU receives, widened exactly to fp64.
Test infrastructure only.
"""
from __future__ import annotations

import numpy as np

from . import tree as _tree


def _group(hq, hkv):
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return hq // hkv


def causal_attention_forward(q, k, v, scale, heads=None):
    """Ordinary causal softmax attention of C query rows at the end of a P-row path.

    q: [C, Hq, d]; k, v: [P, Hkv, d]. Query row i sits at path position
    P − C + i and attends to keys 0 … P − C + i. Returns O [C, Hq, d] and
    LSE [Hq, C]; heads outside `heads` are left as NaN.
    """
    C, hq, d = q.shape
    P, hkv, _ = k.shape
    G = _group(hq, hkv)
    qpos = P - C + np.arange(C)
    visible = np.arange(P)[None, :] <= qpos[:, None]
    O = np.full((C, hq, d), np.nan)
    LSE = np.full((hq, C), np.nan)
    for h in (range(hq) if heads is None else heads):
        s = scale * (q[:, h, :] @ k[:, h // G, :].T)
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        O[:, h, :] = (p @ v[:, h // G, :]) / l
        LSE[h] = (m + np.log(l))[:, 0]
    return O, LSE


def causal_attention_backward(q, k, v, dO, scale, heads=None):
    """Vector-Jacobian product of causal_attention_forward for upstream dO.

    Textbook softmax-attention backward, recomputing P:
    dV = Pᵀ dO;  dP = dO Vᵀ;  dS = P ⊙ (dP − rowsum(dO ⊙ O));
    dQ = scale·dS K;  dK = scale·dSᵀ Q. Key/value gradients of a group sum over
    its query heads. Returns dq [C,Hq,d], dk, dv [P,Hkv,d] (zero for heads
    outside `heads`).
    """
    C, hq, d = q.shape
    P, hkv, _ = k.shape
    G = _group(hq, hkv)
    qpos = P - C + np.arange(C)
    visible = np.arange(P)[None, :] <= qpos[:, None]
    dq = np.zeros((C, hq, d))
    dk = np.zeros((P, hkv, d))
    dv = np.zeros((P, hkv, d))
    for h in (range(hq) if heads is None else heads):
        g = h // G
        s = np.where(visible, scale * (q[:, h, :] @ k[:, g, :].T), -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        o = p @ v[:, g, :]
        do = dO[:, h, :]
        dv[:, g, :] += p.T @ do
        dp = do @ v[:, g, :].T
        ds = p * (dp - np.sum(do * o, axis=1, keepdims=True))
        dq[:, h, :] = scale * (ds @ k[:, g, :])
        dk[:, g, :] += scale * (ds.T @ q[:, h, :])
    return dq, dk, dv


def _heads_of(kv_heads, hq, hkv):
    if kv_heads is None:
        return None
    G = _group(hq, hkv)
    return [h for g in kv_heads for h in range(g * G, (g + 1) * G)]


def tree_attention_branches(tt, Q, K, V, dO=None, scale=None, kv_heads=None, rtol=1e-10):
    """Tree attention by linearising every root-to-leaf branch (the definition).

    Each branch runs ordinary causal attention on its own token sequence. A
    tree token appears in n_t branches; all copies of O_t / LSE_t must agree
    (asserted, "Tree Training" Abstract). For the backward, each copy receives
    dO_t / n_t, so the summed branch gradients are the VJP of Σ_t ⟨dO_t, O_t⟩;
    branch-copy gradients are scatter-added back onto tree tokens.
    `kv_heads` restricts the work to the query heads of those KV groups.
    """
    N, hq, d = Q.shape
    hkv = K.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    heads = _heads_of(kv_heads, hq, hkv)
    hs = list(range(hq)) if heads is None else heads
    O = np.full((N, hq, d), np.nan)
    LSE = np.full((hq, N), np.nan)
    seen = np.zeros(N, bool)
    ncopies = np.zeros(N, np.int64)
    brs = _tree.branches(tt)
    for br in brs:
        o, lse = causal_attention_forward(Q[br], K[br], V[br], scale, heads=hs)
        fresh = ~seen[br]
        old = br[~fresh]
        if old.size:
            np.testing.assert_allclose(o[~fresh][:, hs], O[old][:, hs], rtol=rtol, atol=1e-12)
            np.testing.assert_allclose(lse[hs][:, ~fresh], LSE[hs][:, old], rtol=rtol, atol=1e-12)
        O[br[fresh]] = o[fresh]
        LSE[:, br[fresh]] = lse[:, fresh]
        seen[br] = True
        ncopies[br] += 1
    assert seen.all(), "every token lies on some branch"
    if dO is None:
        return O, LSE
    dQ = np.zeros((N, hq, d))
    dK = np.zeros((N, hkv, d))
    dV = np.zeros((N, hkv, d))
    for br in brs:
        share = dO[br] / ncopies[br][:, None, None]
        dq, dk, dv = causal_attention_backward(Q[br], K[br], V[br], share, scale, heads=hs)
        np.add.at(dQ, br, dq)
        np.add.at(dK, br, dk)
        np.add.at(dV, br, dv)
    return O, LSE, dQ, dK, dV


def tree_attention_segments(tt, Q, K, V, dO=None, scale=None, kv_heads=None):
    """Tree attention one segment at a time (each token computed once).

    The rows of segment s are the last len(s) rows of ordinary causal
    attention over the root-to-s token path, so they are computed by
    causal_attention_forward on that path; their VJP contributions to the
    path's keys and values are scatter-added onto the tree tokens. This is
    the branch definition with each token kept in one copy, i.e. the
    path-at-a-time traversal of AReaL-DTA ("Methodology in Plain English").
    """
    N, hq, d = Q.shape
    hkv = K.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    heads = _heads_of(kv_heads, hq, hkv)
    O = np.full((N, hq, d), np.nan)
    LSE = np.full((hq, N), np.nan)
    if dO is not None:
        dQ = np.zeros((N, hq, d))
        dK = np.zeros((N, hkv, d))
        dV = np.zeros((N, hkv, d))
    for s in range(tt.S):
        path = np.concatenate([np.arange(tt.seg_start[a], tt.seg_end[a])
                               for a in _tree.segment_path(tt.seg_parent, s)])
        rows = np.arange(tt.seg_start[s], tt.seg_end[s])
        o, lse = causal_attention_forward(Q[rows], K[path], V[path], scale, heads=heads)
        O[rows] = o
        LSE[:, rows] = lse
        if dO is not None:
            dq, dk, dv = causal_attention_backward(Q[rows], K[path], V[path], dO[rows], scale, heads=heads)
            dQ[rows] = dq
            dK[path] += dk   # path indices are distinct: an ordinary scatter-add
            dV[path] += dv
    if dO is None:
        return O, LSE
    return O, LSE, dQ, dK, dV


def tree_attention_bruteforce(tt, Q, K, V, dO, scale=None):
    """Scalar-loop tree attention on explicit ancestor sets (tiny trees only).

    For every token t and head h: anc(t) from a parent walk, scores
    s_k = scale·q_t·k_k, P = softmax over anc(t), O_t = Σ P_k v_k. The
    gradient of Σ_t ⟨dO_t, O_t⟩ is accumulated term by term:
    dv_k += P_k dO_t; dS_k = P_k (dO_t·v_k − dO_t·O_t);
    dq_t += scale dS_k k_k; dk_k += scale dS_k q_t.
    """
    N, hq, d = Q.shape
    hkv = K.shape[1]
    G = _group(hq, hkv)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    O = np.zeros((N, hq, d))
    LSE = np.zeros((hq, N))
    dQ = np.zeros((N, hq, d))
    dK = np.zeros((N, hkv, d))
    dV = np.zeros((N, hkv, d))
    for t in range(N):
        anc = [int(x) for x in _tree.token_ancestors(tt, t)]
        for h in range(hq):
            g = h // G
            s = [scale * sum(Q[t, h, i] * K[k, g, i] for i in range(d)) for k in anc]
            m = max(s)
            e = [np.exp(x - m) for x in s]
            z = sum(e)
            p = [x / z for x in e]
            o = [sum(p[j] * V[anc[j], g, i] for j in range(len(anc))) for i in range(d)]
            O[t, h] = o
            LSE[h, t] = m + np.log(z)
            dot_do_o = sum(dO[t, h, i] * o[i] for i in range(d))
            for j, k in enumerate(anc):
                dp = sum(dO[t, h, i] * V[k, g, i] for i in range(d))
                ds = p[j] * (dp - dot_do_o)
                for i in range(d):
                    dV[k, g, i] += p[j] * dO[t, h, i]
                    dQ[t, h, i] += scale * ds * K[k, g, i]
                    dK[k, g, i] += scale * ds * Q[t, h, i]
    return O, LSE, dQ, dK, dV


def ancestor_rows_forward(tt, Q, K, V, tokens, scale=None, heads=None):
    """O and LSE of selected tokens only, from each token's explicit ancestor set.

    Used to check full-size runs on sampled rows. Returns O [len, Hq, d] and
    LSE [Hq, len].
    """
    N, hq, d = Q.shape
    hkv = K.shape[1]
    G = _group(hq, hkv)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    hs = list(range(hq)) if heads is None else list(heads)
    O = np.full((len(tokens), hq, d), np.nan)
    LSE = np.full((hq, len(tokens)), np.nan)
    for i, t in enumerate(tokens):
        anc = _tree.token_ancestors(tt, int(t))
        for h in hs:
            s = scale * (K[anc, h // G, :] @ Q[t, h, :])
            m = s.max()
            p = np.exp(s - m)
            O[i, h] = (p @ V[anc, h // G, :]) / p.sum()
            LSE[h, i] = m + np.log(p.sum())
    return O, LSE


def dta_chunked(tt, Q, K, V, dO, chunk, scale=None, kv_heads=None, leaf_order=None):
    """Path-at-a-time traversal with fixed-size query chunks (AReaL-DTA).

    Walks segments in DFS order keeping the current root-to-segment path.
    Entering a segment forwards its tokens in chunks of at most `chunk`
    queries (each chunk is causal attention against the path prefix that
    ends at the chunk). Leaving a segment — after all its descendants —
    backpropagates its chunks right to left, accumulating key/value gradients
    into the path; the segment's own key/value gradients are then complete
    (AReaL-DTA, Key Contributions 1–2, "Methodology in Plain English").
    Children are entered in ascending segment index, or, with `leaf_order`
    (a visiting order of the leaves, e.g. tree.greedy_leaf_order), so that
    the leaves are reached in that order (it must be a DFS order: the leaves
    of every subtree consecutive).
    """
    N, hq, d = Q.shape
    hkv = K.shape[1]
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    heads = _heads_of(kv_heads, hq, hkv)
    ch = _tree.children(tt.seg_parent)
    if leaf_order is not None:
        # a child's rank: the position of the first of its subtree's leaves in leaf_order
        pos = {int(x): i for i, x in enumerate(leaf_order)}
        first = {}
        for s in range(tt.S):
            for a in _tree.segment_path(tt.seg_parent, s):
                if s in pos:
                    first[a] = min(first.get(a, len(pos)), pos[s])
        ch = [sorted(c, key=lambda x: first[x]) for c in ch]
    O = np.full((N, hq, d), np.nan)
    LSE = np.full((hq, N), np.nan)
    dQ = np.zeros((N, hq, d))
    dK = np.zeros((N, hkv, d))
    dV = np.zeros((N, hkv, d))
    dk_acc = {}
    dv_acc = {}

    def visit(s, path):
        path = np.concatenate([path, np.arange(tt.seg_start[s], tt.seg_end[s])])
        base = len(path) - tt.seg_len[s]
        for t in path[base:]:
            dk_acc[int(t)] = np.zeros((hkv, d))
            dv_acc[int(t)] = np.zeros((hkv, d))
        pieces = [(c0, min(c0 + chunk, int(tt.seg_len[s]))) for c0 in range(0, int(tt.seg_len[s]), chunk)]
        for c0, c1 in pieces:
            rows = path[base + c0: base + c1]
            kp = path[:base + c1]
            o, lse = causal_attention_forward(Q[rows], K[kp], V[kp], scale, heads=heads)
            O[rows] = o
            LSE[:, rows] = lse
        for c in ch[s]:
            visit(c, path)
        for c0, c1 in reversed(pieces):
            rows = path[base + c0: base + c1]
            kp = path[:base + c1]
            dq, dk, dv = causal_attention_backward(Q[rows], K[kp], V[kp], dO[rows], scale, heads=heads)
            dQ[rows] = dq
            for j, t in enumerate(kp):
                dk_acc[int(t)] += dk[j]
                dv_acc[int(t)] += dv[j]
        for t in path[base:]:
            dK[t] = dk_acc.pop(int(t))
            dV[t] = dv_acc.pop(int(t))

    visit(0, np.zeros(0, np.int64))
    return O, LSE, dQ, dK, dV
