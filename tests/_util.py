"""Shared helpers of the test-suite: input conversion, comparison metrics, cached oracle results."""
import functools

import numpy as np
import torch

import synth


def to_dev_bf16(bits, device="cuda"):
    """uint16 bf16 bits (numpy) -> CUDA bf16 tensor (bit-exact)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def f64(bits):
    """uint16 bf16 bits -> exact fp64 values for the oracle."""
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def dev_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))


# Tolerances of the path (stated by the workload definition): attention O max
# abs 2e-2, LSE max rel 1e-3, dQ/dK/dV relative L2 1e-2, logp / loss 1e-4 abs.
O_ATOL = 2e-2
LSE_RTOL = 1e-3
GRAD_RL2 = 1e-2
LOGP_ATOL = 1e-4
# dlogits are bf16 (no stated tolerance; derived from the arithmetic): bf16
# output rounding has unit roundoff 2^-8 (3.9e-3 relative at worst), the
# per-element exponentials are kept as f16 (2^-11), fp32 ops add ~2^-20:
# 2^-8 + 2^-11 + 2^-20 < 5e-3 relative, plus an absolute floor for values
# that are below the f16 normal range of the stored exponentials.
DLOGIT_RTOL = 5e-3
DLOGIT_ATOL = 1e-7


@functools.lru_cache(maxsize=2)
def workload_oracle(wid, kv_groups):
    """Seeded inputs of attention workload `wid` and the fp64 oracle's whole-tree O, LSE, dQ, dK, dV for the
    query heads of `kv_groups` (a tuple), one segment at a time (cached: several tests compare against it)."""
    from oracle import attention as A
    from oracle import tree as T
    inp = synth.attention_inputs(wid)
    sh = inp["tree"]
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.tree_attention_segments(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), kv_heads=list(kv_groups))
    return inp, tab, ref
