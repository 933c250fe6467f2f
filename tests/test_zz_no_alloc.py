"""The no-allocation chunk backward agrees with the regular chunk backward.

tt_tree_attn_chunk_bwd_noalloc is for callers that cannot allocate device
memory at call time (a runtime that owns all device memory through its own
pool, or a latency path that cannot afford cudaMalloc's implicit
synchronisation). It keeps its scratch in a static device array instead of
a caller workspace. This test calls it twice in a row through the C ABI,
with different chunk shapes so that stale scratch from the first call would
show, and compares each result with tt_tree_attn_chunk_bwd bit for bit: both
run the same deterministic kernels on the same inputs, only the scratch
differs. A third call fills the static array exactly (Hq·roundup(C, 128) at
its limit). The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(tt, seed, C, s0, hq, hkv, d):
    lib = tt.lib()
    rng = np.random.default_rng(seed)
    P = s0 + C
    q, k, v, do = (to_dev_bf16(synth.normal_bf16(rng, s)) for s in ((C, hq, d), (P, hkv, d), (P, hkv, d), (C, hq, d)))
    scale = 1.0 / np.sqrt(d)
    err = tt.new_err("cuda")
    o, lse = tt.tree_attn_chunk_fwd(q, s0, k, v, err=err)
    # regular entry point (caller workspace)
    dk_ref = torch.zeros(P, hkv, d, device="cuda")
    dv_ref = torch.zeros(P, hkv, d, device="cuda")
    dq_ref = tt.tree_attn_chunk_bwd(q, s0, k, v, o, lse, do, dk_ref, dv_ref, err=err)
    # no-allocation entry point, straight through the C ABI
    dq = torch.empty_like(q)
    dk = torch.zeros(P, hkv, d, device="cuda")
    dv = torch.zeros(P, hkv, d, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.tt_tree_attn_chunk_bwd_noalloc(_vp(q), C, s0, _vp(k), _vp(v), _vp(o), _vp(lse), C, _vp(do), _vp(dq),
                                            _vp(dk), _vp(dv), hq, hkv, d, ctypes.c_float(scale), _vp(err), stream)
    assert rc == 0, lib.tt_status_string(rc)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for name, got, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        assert torch.equal(got, ref), f"{name}: {int((got != ref).sum())} elements differ from the regular call"


def test_no_alloc_chunk_bwd_matches_regular(tt):
    # two calls in a row on the shared scratch, different shapes
    _case(tt, 1, C=700, s0=300, hq=8, hkv=2, d=128)
    _case(tt, 2, C=129, s0=2048, hq=4, hkv=4, d=64)


def test_no_alloc_at_the_limit(tt):
    # Hq · roundup(C, 128) = 64 · 4096 = 262144: the whole static array
    _case(tt, 3, C=4096, s0=0, hq=64, hkv=8, d=128)


def test_no_alloc_rejects_oversized_chunk(tt):
    lib = tt.lib()
    fake = ctypes.c_void_p(4096)  # rejected before any pointer is used
    rc = lib.tt_tree_attn_chunk_bwd_noalloc(fake, 4097, 0, fake, fake, fake, fake, 4097, fake, fake, fake, fake, 64, 8,
                                            128, ctypes.c_float(0.1), fake, None)
    assert rc == -4
