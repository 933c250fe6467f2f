"""The bounded-wait timeout path of the tensor-memory forward, forced on purpose.

tt_tree_attn_fwd_stall_test makes the MMA-issuing thread of each CTA wait, in
the middle of its pipeline (before its second key block), on a barrier that
nothing arrives at, with a 10 ms limit. The wait expires; the kernel must then
stop its other roles, wait for every TMA copy and tensor-core operation it
already issued, free tensor memory and report TT_ERR_TIMEOUT in the error word,
leaving the context usable: the next normal calls on the same stream must
match the oracle. No wait here is unbounded and nothing faults on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import tree as T
from tests._util import GRAD_RL2, LSE_RTOL, O_ATOL, dev_to_f64, f64, rel_l2, to_dev_bf16

pytestmark = pytest.mark.gpu

TT_ERR_TIMEOUT = -6


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("tiles", [1, 2])
def test_forward_wait_expires_then_calls_recover(tt, tiles):
    sh = synth.random_tree(61, n_seg=9, len_range=(80, 300), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    tree = tt.tree_build(torch.tensor(sh.seg_parent, device="cuda"), torch.tensor(sh.seg_len, device="cuda")).check()
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    N, hq, d = Q.shape
    hkv = K.shape[1]
    O = torch.empty_like(Q)
    LSE = torch.empty(hq, N, dtype=torch.float32, device="cuda")
    err = tt.new_err("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = tt.lib().tt_tree_attn_fwd_stall_test(_vp(tree.ws), _vp(Q), _vp(K), _vp(V), _vp(O), _vp(LSE), N, hq, hkv, d,
                                               ctypes.c_float(1.0 / np.sqrt(d)), tiles, 10_000_000, _vp(err), stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == TT_ERR_TIMEOUT
    # the same stream, the same buffers: normal forward and backward match the oracle
    err2 = tt.new_err("cuda")
    O2, LSE2 = tt.tree_attn_fwd(tree, Q, K, V, out=(O, LSE), err=err2, tiles=tiles)
    dQ, dK, dV = tt.tree_attn_bwd(tree, Q, K, V, O2, LSE2, dO, err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    ref = A.tree_attention_segments(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")))
    assert np.abs(dev_to_f64(O2) - ref[0]).max() <= O_ATOL
    lse = LSE2.cpu().numpy().astype(np.float64)
    assert (np.abs(lse - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for got, r in ((dQ, ref[2]), (dK, ref[3]), (dV, ref[4])):
        assert rel_l2(dev_to_f64(got), r) <= GRAD_RL2


def test_stall_test_rejects_bad_limits(tt):
    fake = ctypes.c_void_p(4096)  # rejected before any pointer is used
    for ns in (0, -1, 10_000_000_001):
        rc = tt.lib().tt_tree_attn_fwd_stall_test(fake, fake, fake, fake, fake, fake, 128, 1, 1, 64,
                                                   ctypes.c_float(0.125), 1, ns, fake, None)
        assert rc == -1
