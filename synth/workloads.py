"""Seeded synthetic workloads for the prefix-tree attention / weighted-log-prob path.

This module generates inputs only: tree shapes (segment parent / length
arrays), bf16 tensors, targets. It holds none of the method's arithmetic (no
DFS layout, no weights, no attention, no softmax), so both the CPU oracle and
the CUDA-path tests and bench can draw their inputs from it without sharing
any computation.

Tree shapes follow the five workloads of the tree-training pages (rollout
trees with shared prefixes, "Tree Training" abstract; τ²-bench-like
compression ≈ 4× and ≈ 8×, AReaL-DTA "Main Findings"), with Qwen3 head shapes.

Random values: every tensor is drawn as bf16 directly, by inverse-CDF lookup.
One 16-bit uniform draw u selects the bf16-rounded normal quantile
Φ⁻¹((u + 0.5) / 65536)·σ. This is a normal distribution discretised at
2⁻¹⁶ in probability (tails clipped at ≈4.3σ), exact at bf16 resolution, and
~50× faster than drawing fp32 normals and rounding them. The draws come from
``numpy.random.default_rng(seed)`` in a fixed order:
tree structure (breadth-first creation order), then Q, K, V, dO, then logits,
then targets.
"""
from __future__ import annotations

import functools
from dataclasses import dataclass

import numpy as np
import torch
from scipy.special import ndtri

__all__ = [
    "CONFIG_NAMES", "TreeShape", "tree_shape", "random_tree",
    "bf16_bits_to_f32", "f32_to_bf16_bits", "normal_bf16",
    "attention_inputs", "logprob_inputs", "lmhead_inputs", "HEADS",
]

CONFIG_NAMES = {
    0: "tiny tree, 1 head, d=64, V=1000",
    1: "Qwen3-1.7B-shaped tree attention (16/8 heads, d=128), 16 leaves",
    2: "weighted log-prob over config-1 tree, V=151936",
    3: "Qwen3-8B-shaped GRPO tree (32/8 heads, d=128), 64 leaves",
    4: "deep agentic tree, Qwen3-14B-shaped (40/8 heads, d=128)",
}

# (Hq, Hkv, d) per attention workload
HEADS = {0: (1, 1, 64), 1: (16, 8, 128), 3: (32, 8, 128), 4: (40, 8, 128)}


@dataclass
class TreeShape:
    seg_parent: np.ndarray  # int32 [S]; -1 for the root, parent < child otherwise
    seg_len: np.ndarray     # int32 [S]; >= 1
    rng: np.random.Generator  # positioned after the structure draws

    @property
    def S(self) -> int:
        return int(self.seg_parent.shape[0])

    @property
    def N(self) -> int:
        return int(self.seg_len.sum())


def _u(rng, lo, hi):
    """One uniform integer in [lo, hi] (inclusive)."""
    return int(rng.integers(lo, hi + 1))


def _two_level(rng, root_len, n1, len1, n2, len2):
    par, ln = [-1], [root_len]
    for _ in range(n1):
        par.append(0)
        ln.append(len1 if isinstance(len1, int) else _u(rng, *len1))
    for c in range(1, n1 + 1):
        for _ in range(n2):
            par.append(c)
            ln.append(len2 if isinstance(len2, int) else _u(rng, *len2))
    return par, ln


def _deep_agentic(rng, levels=6, cap_tokens=65536, cap_leaves=128, lens=(32, 1024), kids=(1, 3)):
    """Breadth-first random tree: root plus `levels` levels of children.

    Each node draws its child count, then each child's length. Creation stops
    once the unique-token total reaches `cap_tokens` (the last segment is
    truncated) and no new branch is opened once `cap_leaves` leaves exist.
    """
    par, ln, depth = [-1], [_u(rng, *lens)], [0]
    total, leaves = ln[0], 1
    queue, stop = [0], False
    while queue and not stop:
        s = queue.pop(0)
        if depth[s] >= levels:
            continue
        for i in range(_u(rng, *kids)):
            if i > 0 and leaves >= cap_leaves:
                break
            length = _u(rng, *lens)
            if total + length >= cap_tokens:
                length, stop = cap_tokens - total, True
            par.append(s)
            ln.append(length)
            depth.append(depth[s] + 1)
            total += length
            if i > 0:
                leaves += 1
            queue.append(len(par) - 1)
            if stop:
                break
    return par, ln


def tree_shape(cfg: int, seed: int = 0) -> TreeShape:
    """Segment tree of workload `cfg` (0..4); config 2 reuses config 1's tree."""
    rng = np.random.default_rng(seed)
    if cfg == 0:
        par, ln = _two_level(rng, 64, 2, 32, 2, (8, 24))
    elif cfg in (1, 2):
        par, ln = _two_level(rng, 2048, 4, (256, 768), 4, (256, 768))
    elif cfg == 3:
        par, ln = _two_level(rng, 4096, 8, 1024, 8, (256, 768))
    elif cfg == 4:
        par, ln = _deep_agentic(rng)
    else:
        raise ValueError(f"unknown workload {cfg}")
    return TreeShape(np.asarray(par, np.int32), np.asarray(ln, np.int32), rng)


def random_tree(seed: int, n_seg: int, len_range=(1, 40), max_children=3, chain=False) -> TreeShape:
    """Small random topological tree for tests: segment s>0 picks a parent < s.

    chain=True gives a single path (every segment has one child).
    """
    rng = np.random.default_rng(seed)
    par = [-1]
    nchild = [0]
    for s in range(1, n_seg):
        if chain:
            p = s - 1
        else:
            cand = [p for p in range(s) if nchild[p] < max_children]
            p = int(cand[int(rng.integers(0, len(cand)))])
        par.append(p)
        nchild[p] += 1
        nchild.append(0)
    ln = [int(rng.integers(len_range[0], len_range[1] + 1)) for _ in range(n_seg)]
    return TreeShape(np.asarray(par, np.int32), np.asarray(ln, np.int32), rng)


# ----------------------------------------------------------------------------- bf16 helpers
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even), returned as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits (uint16) to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@functools.lru_cache(maxsize=8)
def _quantile_table(sigma: float) -> torch.Tensor:
    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    q = (ndtri(p) * sigma).astype(np.float32)
    return torch.from_numpy(f32_to_bf16_bits(q).view(np.int16))


def normal_bf16(rng: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    """bf16 bits (uint16) of N(0, sigma²) samples, by 16-bit quantile lookup."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.int16)
    tab = _quantile_table(float(sigma))
    step = 1 << 26
    for lo in range(0, n, step):
        m = min(step, n - lo)
        u = rng.integers(0, 2**32, size=(m + 1) // 2, dtype=np.uint32).view(np.int16)[:m]
        idx = torch.from_numpy(u).to(torch.int32) & 0xFFFF
        torch.index_select(tab, 0, idx, out=out[lo:lo + m])
    return out.numpy().view(np.uint16).reshape(shape)


# ----------------------------------------------------------------------------- workloads
def attention_inputs(cfg: int, seed: int = 0, tree: TreeShape | None = None, heads=None):
    """Tree + bf16 Q, K, V, dO (uint16 bits) of attention workload `cfg`.

    Q/dO are [N, Hq, d], K/V are [N, Hkv, d], token-major. `tree`/`heads`
    override the shape (random test trees); the draws then continue on the
    tree's own generator.
    """
    if tree is None:
        tree = tree_shape(cfg, seed)
    hq, hkv, d = heads if heads is not None else HEADS[cfg]
    sig = 1.0 / np.sqrt(8.0) if cfg == 0 else 1.0
    rng, N = tree.rng, tree.N
    Q = normal_bf16(rng, (N, hq, d), sig)
    K = normal_bf16(rng, (N, hkv, d), sig)
    V = normal_bf16(rng, (N, hkv, d), sig)
    dO = normal_bf16(rng, (N, hq, d), 1.0)
    return dict(tree=tree, Q=Q, K=K, V=V, dO=dO, hq=hq, hkv=hkv, d=d)


def logprob_inputs(cfg: int, seed: int = 0, tree: TreeShape | None = None, vocab=None):
    """Tree + bf16 logits [N, V] ~ N(0, 2²) and int32 targets uniform in [0, V).

    Config 0 draws its logits after its attention tensors (same generator);
    config 2 regenerates config 1's tree and draws logits right after it.
    """
    if tree is None:
        if cfg == 0:
            tree = attention_inputs(0, seed)["tree"]
        elif cfg == 2:
            tree = tree_shape(2, seed)
        else:
            raise ValueError("log-prob workloads are configs 0 and 2")
    V = vocab if vocab is not None else (1000 if cfg == 0 else 151936)
    rng, N = tree.rng, tree.N
    logits = normal_bf16(rng, (N, V), 2.0)
    targets = rng.integers(0, V, size=N).astype(np.int32)
    return dict(tree=tree, logits=logits, targets=targets, V=V)


def lmhead_inputs(seed: int = 0, tree: TreeShape | None = None, vocab: int = 151936, hidden: int = 2048,
                  n_rows: int | None = None):
    """Hidden states H [N, Hd] ~ N(0, 1) and vocabulary matrix W [V, Hd] ~ N(0, (2/√Hd)²), both bf16, and int32
    targets uniform in [0, V): the LM head in front of the log-prob workload (Qwen3-1.7B hidden size 2048,
    Qwen3 vocabulary). W's scale gives logits z = H·Wᵀ with about the N(0, 2²) spread of the log-prob
    workload's logits. Default tree: config 2's (= config 1's) tree; `n_rows` overrides N (no tree then).
    Draw order: tree, H, W, targets.
    """
    if n_rows is None:
        tree = tree_shape(2, seed) if tree is None else tree
        rng, N = tree.rng, tree.N
    else:
        rng, N = np.random.default_rng(seed), int(n_rows)
    H = normal_bf16(rng, (N, hidden), 1.0)
    W = normal_bf16(rng, (vocab, hidden), 2.0 / np.sqrt(hidden))
    targets = rng.integers(0, vocab, size=N).astype(np.int32)
    return dict(tree=tree, H=H, W=W, targets=targets, V=vocab, Hd=hidden)
