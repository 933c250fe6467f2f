"""The attention kernels are deterministic: repeated calls give identical bits.

Every kernel of the path accumulates in a fixed order (no atomics), so any
difference between two calls on the same inputs exposes a race between the
roles of a kernel (for example a tensor-memory buffer reused before its
readers are done). Oracle parity on sampled rows can miss such a race; a
bitwise comparison over many calls of the full workload does not.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu


def _setup(tt, cfg):
    inp = synth.attention_inputs(cfg)
    sh = inp["tree"]
    tree = tt.tree_build(torch.tensor(sh.seg_parent, device="cuda"), torch.tensor(sh.seg_len, device="cuda")).check()
    return tree, [to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO")]


def _bits(x):
    return x.view(torch.int16).clone() if x.dtype == torch.bfloat16 else x.clone()


@pytest.mark.parametrize("cfg,reps", [(1, 24), (4, 8)])
def test_tree_fwd_bwd_bitwise_repeatable(tt, cfg, reps):
    tree, (Q, K, V, dO) = _setup(tt, cfg)
    ref = None
    for _ in range(reps):
        O, LSE = tt.tree_attn_fwd(tree, Q, K, V)
        dQ, dK, dV = tt.tree_attn_bwd(tree, Q, K, V, O, LSE, dO)
        torch.cuda.synchronize()
        cur = [_bits(x) for x in (O, LSE, dQ, dK, dV)]
        if ref is None:
            ref = cur
            continue
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), ref, cur):
            assert torch.equal(a, b), f"{name}: {int((a != b).sum())} elements differ between calls"


@pytest.mark.parametrize("tiles", [1, 2])  # one or two query tiles per forward CTA
def test_chunk_fwd_bwd_bitwise_repeatable(tt, tiles):
    rng = np.random.default_rng(7)
    C, s0, hq, hkv, d = 2048, 3000, 16, 8, 128
    P = s0 + C
    q, k, v, do = (to_dev_bf16(synth.normal_bf16(rng, s)) for s in ((C, hq, d), (P, hkv, d), (P, hkv, d), (C, hq, d)))
    ref = None
    for _ in range(8):
        o, lse = tt.tree_attn_chunk_fwd(q, s0, k, v, tiles=tiles)
        dk = torch.zeros(P, hkv, d, device="cuda")
        dv = torch.zeros(P, hkv, d, device="cuda")
        dq = tt.tree_attn_chunk_bwd(q, s0, k, v, o, lse, do, dk, dv)
        torch.cuda.synchronize()
        cur = [_bits(x) for x in (o, lse, dq, dk, dv)]
        if ref is None:
            ref = cur
            continue
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), ref, cur):
            assert torch.equal(a, b), f"chunk {name}: {int((a != b).sum())} elements differ between calls"


def test_path_at_a_time_bitwise_repeatable(tt):
    """The path-at-a-time driver (a chunk forward and backward per path segment) repeats bit for bit."""
    inp = synth.attention_inputs(1)
    sh = inp["tree"]
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    ref = None
    for _ in range(4):
        outs = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=2048)
        torch.cuda.synchronize()
        cur = [_bits(x) for x in outs]
        if ref is None:
            ref = cur
            continue
        for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), ref, cur):
            assert torch.equal(a, b), f"path-at-a-time {name}: {int((a != b).sum())} elements differ between calls"
