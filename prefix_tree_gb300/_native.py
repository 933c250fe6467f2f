"""ctypes binding of libtt (include/tt.h): argument marshalling only.

Every computation runs in the CUDA library; this module allocates outputs and
workspaces with PyTorch on the tensors' device, passes raw pointers and the
current CUDA stream, and raises on a non-zero status. There is no fallback: a
missing libtt.so raises immediately.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtt.so")

TT_OK = 0
_STATUS = {0: "TT_OK", -1: "TT_ERR_INVALID_ARG", -2: "TT_ERR_INVALID_TREE", -3: "TT_ERR_UNSUPPORTED",
           -4: "TT_ERR_WORKSPACE", -5: "TT_ERR_CUDA", -6: "TT_ERR_TIMEOUT"}

_vp, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_int = ctypes.c_int


class TTError(RuntimeError):
    def __init__(self, code, what=""):
        self.code = int(code)
        super().__init__(f"{what}: {_STATUS.get(self.code, self.code)} ({lib().tt_status_string(self.code).decode()})")


class _TreeOut(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("seg_start", "seg_subtree_end", "seg_depth", "seg_pathlen", "seg_leafcnt", "iv_ptr",
                                   "iv", "tok_seg", "tok_pos", "tok_send", "tok_leafcnt", "tok_weight", "stats")]


_SIGS = {
    "tt_tree_workspace_bytes": (_sz, [_i32, _i64]),
    "tt_tree_build": (_int, [_vp, _vp, _i32, _i64, ctypes.POINTER(_TreeOut), _i64, _vp, _sz, _vp, _vp]),
    "tt_tree_schedules": (_int, [_vp, _i64] + [_vp] * 7 + [_vp]),
    "tt_tree_attn_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _vp, _vp]),
    "tt_tree_attn_fwd_tiles": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _int, _vp, _vp]),
    "tt_tree_attn_fwd_stall_test": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _int, _i64, _vp,
                                           _vp]),
    "tt_tree_attn_bwd_workspace_bytes": (_sz, [_i64, _int]),
    "tt_tree_attn_bwd": (_int, [_vp] * 10 + [_i64, _int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_tree_attn_chunk_fwd": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _vp, _vp]),
    "tt_tree_attn_chunk_fwd_tiles": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _int,
                                            _vp, _vp]),
    "tt_tree_attn_chunk_fwd_split": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _f32, _int,
                                            _vp, _vp]),
    "tt_tree_attn_chunk_bwd_workspace_bytes": (_sz, [_i64, _int]),
    "tt_tree_attn_chunk_bwd": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _int, _int, _int,
                                      _f32, _vp, _sz, _vp, _vp]),
    "tt_tree_attn_chunk_fwd_packed": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int,
                                             _f32, _vp, _vp]),
    "tt_tree_attn_chunk_bwd_packed": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp,
                                             _vp, _int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_tree_attn_chunk_bwd_noalloc": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _int,
                                              _int, _int, _f32, _vp, _vp]),
    "tt_dta_workspace_bytes": (_sz, [_vp, _vp, _i32, _i64, _int, _int, _int]),
    "tt_dta_tree_attn": (_int, [_vp, _vp, _i32, _i64, _i64] + [_vp] * 9 + [_int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_dta_tree_attn_ordered": (_int, [_vp, _vp, _i32, _i64, _i64, _int] + [_vp] * 9
                                 + [_int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_tree_partition": (_int, [_vp, _vp, _i32, _i64, _int, _vp, _vp, _vp, _vp, _i32]),
    "tt_dta_leaf_order": (_int, [_vp, _vp, _i32, _int, _vp, _i32]),
    "tt_dta_plan_create": (_int, [_vp, _vp, _i32, _i64, _i64, _int, _int] + [_vp] * 9
                           + [_int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_dta_workspace_bytes_slots": (_sz, [_vp, _vp, _i32, _i64, _int, _int, _int, _int]),
    "tt_dta_tree_attn_slots": (_int, [_vp, _vp, _i32, _i64, _i64, _int, _int] + [_vp] * 9
                               + [_int, _int, _int, _f32, _vp, _sz, _vp, _vp]),
    "tt_dta_plan_launch": (_int, [_vp, _vp]),
    "tt_dta_plan_destroy": (_int, [_vp]),
    "tt_weighted_logprob": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _vp]),
    "tt_lmhead_logprob_workspace_bytes": (_sz, [_i64, _i64]),
    "tt_lmhead_logprob": (_int, [_vp, _vp, _i64, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "tt_lmhead_logprob_bwd_workspace_bytes": (_sz, [_i64, _i64]),
    "tt_lmhead_logprob_bwd": (_int, [_vp, _vp, _i64, _i64, _int, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _sz, _vp, _vp]),
    "tt_status_string": (ctypes.c_char_p, [_int]),
    "tt_version": (_int, []),
    "tt_trie_build": (_int, [_vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp, _vp]),
    "tt_kernel_timing": (_int, [_int]),
    "tt_kernel_timing_read": (_int, [_vp, _vp, _int, _vp]),
}

_LIB = None


def lib():
    """The loaded libtt (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtt.so is not built ({LIB_PATH}); run prefix_tree_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def exported_symbols():
    return list(_SIGS)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev=None):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(rc, what):
    if rc != TT_OK:
        raise TTError(rc, what)


def _need(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims")


def new_err(device):
    """A zeroed device error word (see tt.h)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_err(err, what="device"):
    """Synchronise on the error word and raise if a kernel recorded an error."""
    code = int(err.item())
    if code != 0:
        raise TTError(code, what)


# --------------------------------------------------------------------------- tree build
@dataclass
class Tree:
    """Device tables of a DFS-serialised tree plus the attention workspace."""
    S: int
    N: int
    seg_start: torch.Tensor
    seg_subtree_end: torch.Tensor
    seg_depth: torch.Tensor
    seg_pathlen: torch.Tensor
    seg_leafcnt: torch.Tensor
    iv_ptr: torch.Tensor
    iv: torch.Tensor
    tok_seg: torch.Tensor
    tok_pos: torch.Tensor
    tok_send: torch.Tensor
    tok_leafcnt: torch.Tensor
    tok_weight: torch.Tensor
    stats: torch.Tensor
    ws: torch.Tensor
    err: torch.Tensor

    def check(self):
        check_err(self.err, "tt_tree_build")
        return self


def tree_build(seg_parent: torch.Tensor, seg_len: torch.Tensor, N: int | None = None, iv_capacity: int | None = None,
               err: torch.Tensor | None = None) -> Tree:
    _need(seg_parent, torch.int32, "seg_parent", 1)
    _need(seg_len, torch.int32, "seg_len", 1)
    S = seg_parent.numel()
    dev = seg_parent.device
    if N is None:
        N = int(seg_len.sum().item())
    if iv_capacity is None:
        iv_capacity = S * (S + 1) // 2
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(seg_start=torch.empty(S, **i32), seg_subtree_end=torch.empty(S, **i32),
               seg_depth=torch.empty(S, **i32), seg_pathlen=torch.empty(S, **i32),
               seg_leafcnt=torch.empty(S, **i32), iv_ptr=torch.empty(S + 1, **i32),
               iv=torch.empty(max(1, iv_capacity), 2, **i32), tok_seg=torch.empty(N, **i32),
               tok_pos=torch.empty(N, **i32), tok_send=torch.empty(N, **i32), tok_leafcnt=torch.empty(N, **i32),
               tok_weight=torch.empty(N, dtype=torch.float32, device=dev),
               stats=torch.zeros(8, dtype=torch.int64, device=dev))
    nbytes = lib().tt_tree_workspace_bytes(S, N)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    err = new_err(dev) if err is None else err
    s = _TreeOut(**{k: _p(v).value for k, v in out.items()})
    rc = lib().tt_tree_build(_p(seg_parent), _p(seg_len), S, N, ctypes.byref(s), iv_capacity, _p(ws), nbytes,
                             _p(err), _stream(dev))
    _check(rc, "tt_tree_build")
    return Tree(S=S, N=N, ws=ws, err=err, **out)


def tree_schedules(tree: Tree) -> dict:
    """The tile schedules the tree build wrote (tt_tree_schedules), as int32 device tensors."""
    nT = (tree.N + 127) // 128
    dev = tree.ws.device
    names = ("send", "blk_min", "blk_max", "fwd_cnt", "fwd_order", "bwd_cnt", "bwd_order")
    out = {n: torch.empty(nT * 128 if n == "send" else nT, dtype=torch.int32, device=dev) for n in names}
    _check(lib().tt_tree_schedules(_p(tree.ws), tree.N, *(_p(out[n]) for n in names), _stream(dev)),
           "tt_tree_schedules")
    return out


# --------------------------------------------------------------------------- attention
def _heads(Q, K):
    N, hq, d = Q.shape
    return N, hq, K.shape[1], d


def tree_attn_fwd(tree: Tree, Q, K, V, scale=None, out=None, err=None, tiles=None):
    """O [N,Hq,d] bf16, LSE [Hq,N] fp32 of tree attention (tt_tree_attn_fwd; with `tiles` = 1 or 2 the
    forward schedule is fixed through tt_tree_attn_fwd_tiles)."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _need(t, torch.bfloat16, n, 3)
    N, hq, hkv, d = _heads(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    O = torch.empty_like(Q) if out is None else out[0]
    LSE = torch.empty(hq, N, dtype=torch.float32, device=Q.device) if out is None else out[1]
    err = tree.err if err is None else err
    if tiles is None:
        rc = lib().tt_tree_attn_fwd(_p(tree.ws), _p(Q), _p(K), _p(V), _p(O), _p(LSE), N, hq, hkv, d, scale, _p(err),
                                    _stream(Q.device))
    else:
        rc = lib().tt_tree_attn_fwd_tiles(_p(tree.ws), _p(Q), _p(K), _p(V), _p(O), _p(LSE), N, hq, hkv, d, scale,
                                          int(tiles), _p(err), _stream(Q.device))
    _check(rc, "tt_tree_attn_fwd")
    return O, LSE


def tree_attn_bwd(tree: Tree, Q, K, V, O, LSE, dO, scale=None, out=None, ws=None, err=None):
    """dQ, dK, dV (bf16) of tree attention (tt_tree_attn_bwd)."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V"), (O, "O"), (dO, "dO")):
        _need(t, torch.bfloat16, n, 3)
    _need(LSE, torch.float32, "LSE", 2)
    N, hq, hkv, d = _heads(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dQ, dK, dV = (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)) if out is None else out
    nbytes = lib().tt_tree_attn_bwd_workspace_bytes(N, hq)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    err = tree.err if err is None else err
    rc = lib().tt_tree_attn_bwd(_p(tree.ws), _p(Q), _p(K), _p(V), _p(O), _p(LSE), _p(dO), _p(dQ), _p(dK), _p(dV), N,
                                hq, hkv, d, scale, _p(ws), ws.numel(), _p(err), _stream(Q.device))
    _check(rc, "tt_tree_attn_bwd")
    return dQ, dK, dV


def tree_attn_chunk_fwd(q, s0, k_path, v_path, o=None, lse=None, lse_ld=None, scale=None, err=None, tiles=None,
                        splits=None, send=None, blk_max=None):
    """Chunk-vs-path forward: q [C,Hq,d] at path offset s0 against k/v_path [s0+C,Hkv,d] (`tiles` as in
    tree_attn_fwd; `splits` = key-range splits per tile on the one-tile schedule, 0 = chosen, 1..4 fixed).
    `send` and `blk_max` (int32 device tensors, tt_tree_attn_chunk_fwd_packed) make it a packed chunk of sibling
    subtrees."""
    C, hq, d = q.shape
    hkv = k_path.shape[1]
    if k_path.shape[0] < s0 + C:
        raise ValueError("k_path must hold s0 + C rows")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q) if o is None else o
    lse_ld = C if lse_ld is None else lse_ld
    lse = torch.empty(hq, lse_ld, dtype=torch.float32, device=q.device) if lse is None else lse
    err = new_err(q.device) if err is None else err
    if send is not None:
        if tiles is not None or splits is not None:
            raise ValueError("a packed chunk takes no tiles or splits")
        rc = lib().tt_tree_attn_chunk_fwd_packed(_p(q), C, s0, _p(k_path), _p(v_path), _p(send), _p(blk_max), _p(o),
                                                 _p(lse), lse_ld, hq, hkv, d, scale, _p(err), _stream(q.device))
    elif splits is not None:
        if tiles is not None:
            raise ValueError("give tiles or splits, not both")
        rc = lib().tt_tree_attn_chunk_fwd_split(_p(q), C, s0, _p(k_path), _p(v_path), _p(o), _p(lse), lse_ld, hq, hkv,
                                                d, scale, int(splits), _p(err), _stream(q.device))
    elif tiles is None:
        rc = lib().tt_tree_attn_chunk_fwd(_p(q), C, s0, _p(k_path), _p(v_path), _p(o), _p(lse), lse_ld, hq, hkv, d,
                                          scale, _p(err), _stream(q.device))
    else:
        rc = lib().tt_tree_attn_chunk_fwd_tiles(_p(q), C, s0, _p(k_path), _p(v_path), _p(o), _p(lse), lse_ld, hq, hkv,
                                                d, scale, int(tiles), _p(err), _stream(q.device))
    _check(rc, "tt_tree_attn_chunk_fwd")
    return o, lse


def tree_attn_chunk_bwd(q, s0, k_path, v_path, o, lse, dO, dk_acc, dv_acc, lse_ld=None, dq=None, scale=None,
                        err=None, ws=None, send=None, blk_max=None):
    """Chunk-vs-path backward: returns dq; accumulates fp32 dk_acc / dv_acc in place (`send`, `blk_max`: a packed
    chunk, tt_tree_attn_chunk_bwd_packed)."""
    C, hq, d = q.shape
    hkv = k_path.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    lse_ld = C if lse_ld is None else lse_ld
    nbytes = lib().tt_tree_attn_chunk_bwd_workspace_bytes(C, hq)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device) if ws is None else ws
    err = new_err(q.device) if err is None else err
    if send is not None:
        rc = lib().tt_tree_attn_chunk_bwd_packed(_p(q), C, s0, _p(k_path), _p(v_path), _p(send), _p(blk_max), _p(o),
                                                 _p(lse), lse_ld, _p(dO), _p(dq), _p(dk_acc), _p(dv_acc), hq, hkv, d,
                                                 scale, _p(ws), ws.numel(), _p(err), _stream(q.device))
    else:
        rc = lib().tt_tree_attn_chunk_bwd(_p(q), C, s0, _p(k_path), _p(v_path), _p(o), _p(lse), lse_ld, _p(dO),
                                          _p(dq), _p(dk_acc), _p(dv_acc), hq, hkv, d, scale, _p(ws), ws.numel(),
                                          _p(err), _stream(q.device))
    _check(rc, "tt_tree_attn_chunk_bwd")
    return dq


DTA_ORDER_INDEX, DTA_ORDER_GREEDY = 0, 1
DTA_DEFAULT_SLOTS = 2  # TT_DTA_DEFAULT_SLOTS


def dta_workspace_bytes(seg_parent_host, seg_len_host, chunk, hq, hkv, d, slots=DTA_DEFAULT_SLOTS):
    """Device scratch bytes of the path-at-a-time pass for this tree, chunk size and slot count
    (tt_dta_workspace_bytes_slots)."""
    import numpy as np
    par = np.ascontiguousarray(seg_parent_host, dtype=np.int32)
    ln = np.ascontiguousarray(seg_len_host, dtype=np.int32)
    n = lib().tt_dta_workspace_bytes_slots(par.ctypes.data_as(_vp), ln.ctypes.data_as(_vp), len(par), chunk, hq, hkv,
                                           d, slots)
    if n == 0:
        raise TTError(-2, "tt_dta_workspace_bytes")
    return n


def tree_partition(seg_parent_host, seg_len_host, budget, order=DTA_ORDER_GREEDY):
    """The partitions of the path-at-a-time traversal for a token budget (tt_tree_partition), in DFS layout order:
    numpy arrays (first row, rows, cached path rows, kind: 0 pack of sibling subtrees, 1 chunk of one segment)."""
    import numpy as np
    par = np.ascontiguousarray(seg_parent_host, dtype=np.int32)
    ln = np.ascontiguousarray(seg_len_host, dtype=np.int32)
    pp, lp = par.ctypes.data_as(_vp), ln.ctypes.data_as(_vp)
    n = lib().tt_tree_partition(pp, lp, len(par), int(budget), order, None, None, None, None, 0)
    _check(n if n < 0 else 0, "tt_tree_partition")
    first, rows, path = (np.zeros(n, np.int64) for _ in range(3))
    kind = np.zeros(n, np.int32)
    rc = lib().tt_tree_partition(pp, lp, len(par), int(budget), order, first.ctypes.data_as(_vp),
                                 rows.ctypes.data_as(_vp), path.ctypes.data_as(_vp), kind.ctypes.data_as(_vp), n)
    _check(rc if rc < 0 else 0, "tt_tree_partition")
    return first, rows, path, kind


def dta_leaf_order(seg_parent_host, seg_len_host, order=DTA_ORDER_GREEDY):
    """Leaves (segment ids) in the order the path-at-a-time traversal reaches them (tt_dta_leaf_order)."""
    import numpy as np
    par = np.ascontiguousarray(seg_parent_host, dtype=np.int32)
    ln = np.ascontiguousarray(seg_len_host, dtype=np.int32)
    out = np.empty(max(len(par), 1), np.int32)
    n = lib().tt_dta_leaf_order(par.ctypes.data_as(_vp), ln.ctypes.data_as(_vp), len(par), order,
                                out.ctypes.data_as(_vp), len(out))
    if n < 0:
        raise TTError(n, "tt_dta_leaf_order")
    return out[:n].copy()


def dta_tree_attn(seg_parent_host, seg_len_host, Q, K, V, dO, chunk=2048, scale=None, err=None, ws=None, out=None,
                  order=DTA_ORDER_GREEDY, slots=DTA_DEFAULT_SLOTS):
    """Whole-tree fwd+bwd by path-at-a-time traversal (tt_dta_tree_attn_slots): O, LSE, dQ, dK, dV
    (written into `out` = (O, LSE, dQ, dK, dV) when given); `order` = DTA_ORDER_GREEDY or DTA_ORDER_INDEX;
    `slots` = sibling leaves processed at once (1 = the one-path traversal)."""
    import numpy as np
    par = np.ascontiguousarray(seg_parent_host, dtype=np.int32)
    ln = np.ascontiguousarray(seg_len_host, dtype=np.int32)
    N, hq, hkv, d = _heads(Q, K)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    pp, lp = par.ctypes.data_as(_vp), ln.ctypes.data_as(_vp)
    if ws is None:
        nbytes = lib().tt_dta_workspace_bytes_slots(pp, lp, len(par), chunk, hq, hkv, d, slots)
        if nbytes == 0:
            raise TTError(-2, "tt_dta_workspace_bytes")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    if out is None:
        O, dQ = torch.empty_like(Q), torch.empty_like(Q)
        dK, dV = torch.empty_like(K), torch.empty_like(V)
        LSE = torch.empty(hq, N, dtype=torch.float32, device=Q.device)
    else:
        O, LSE, dQ, dK, dV = out
    err = new_err(Q.device) if err is None else err
    rc = lib().tt_dta_tree_attn_slots(pp, lp, len(par), N, chunk, order, slots, _p(Q), _p(K), _p(V), _p(dO), _p(O),
                                      _p(LSE), _p(dQ), _p(dK), _p(dV), hq, hkv, d, scale, _p(ws), ws.numel(), _p(err),
                                      _stream(Q.device))
    _check(rc, "tt_dta_tree_attn")
    return O, LSE, dQ, dK, dV


class DtaPlan:
    """The path-at-a-time pass of one tree captured once into a CUDA graph (tt_dta_plan_create); launch() enqueues
    the whole pass with one call. The input and output tensors are bound at creation: write new inputs into them
    and keep them alive while the plan exists. `outputs` = (O, LSE, dQ, dK, dV)."""

    def __init__(self, seg_parent_host, seg_len_host, Q, K, V, dO, chunk=2048, scale=None, err=None, ws=None,
                 out=None, order=DTA_ORDER_GREEDY, slots=DTA_DEFAULT_SLOTS):
        import numpy as np
        self._plan = None
        par = np.ascontiguousarray(seg_parent_host, dtype=np.int32)
        ln = np.ascontiguousarray(seg_len_host, dtype=np.int32)
        N, hq, hkv, d = _heads(Q, K)
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        pp, lp = par.ctypes.data_as(_vp), ln.ctypes.data_as(_vp)
        nbytes = lib().tt_dta_workspace_bytes_slots(pp, lp, len(par), chunk, hq, hkv, d, slots)
        if nbytes == 0:
            raise TTError(-2, "tt_dta_workspace_bytes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=Q.device) if ws is None else ws
        if out is None:
            out = (torch.empty_like(Q), torch.empty(hq, N, dtype=torch.float32, device=Q.device), torch.empty_like(Q),
                   torch.empty_like(K), torch.empty_like(V))
        self.outputs = tuple(out)
        self.err = new_err(Q.device) if err is None else err
        self.device = Q.device
        self._keep = (Q, K, V, dO)
        O, LSE, dQ, dK, dV = self.outputs
        plan = ctypes.c_void_p(0)
        rc = lib().tt_dta_plan_create(pp, lp, len(par), N, chunk, order, slots, _p(Q), _p(K), _p(V), _p(dO), _p(O),
                                      _p(LSE),
                                      _p(dQ), _p(dK), _p(dV), hq, hkv, d, scale, _p(self.ws), self.ws.numel(),
                                      _p(self.err), ctypes.byref(plan))
        _check(rc, "tt_dta_plan_create")
        self._plan = plan

    def launch(self):
        """Enqueue the pass on the current stream; returns the output tensors."""
        _check(lib().tt_dta_plan_launch(self._plan, _stream(self.device)), "tt_dta_plan_launch")
        return self.outputs

    def close(self):
        if self._plan is not None and self._plan.value:
            _check(lib().tt_dta_plan_destroy(self._plan), "tt_dta_plan_destroy")
        self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------------------- log-prob
def weighted_logprob(logits, targets, weights=None, g=1.0, want_dlogits=True, out=None, err=None):
    """logp fp32 [N], loss fp64 (device scalar), dlogits bf16 [N,V] or None (tt_weighted_logprob). `logits` may be a
    row-padded view (rows ld >= V elements apart, elements contiguous); dlogits then has the same row stride."""
    if not isinstance(logits, torch.Tensor) or not logits.is_cuda or logits.dtype != torch.bfloat16 or logits.dim() != 2:
        raise TypeError("logits must be a 2-D bf16 CUDA tensor")
    N, V = logits.shape
    ld = logits.stride(0) if N > 1 else V
    if logits.stride(1) != 1 or ld < V:
        raise ValueError("logits rows must be contiguous (stride(1) == 1, stride(0) >= V)")
    _need(targets, torch.int32, "targets", 1)
    if weights is not None:
        _need(weights, torch.float32, "weights", 1)
    dev = logits.device
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        loss = torch.empty(1, dtype=torch.float64, device=dev)
        dl = torch.empty(N, ld, dtype=torch.bfloat16, device=dev)[:, :V] if want_dlogits else None
    else:
        logp, loss, dl = out
    if dl is not None and (dl.shape != logits.shape or dl.stride() != logits.stride()):
        raise ValueError("dlogits must have the shape and strides of logits")
    err = new_err(dev) if err is None else err
    rc = lib().tt_weighted_logprob(_p(logits), N, V, ld, _p(targets), _p(weights), g, _p(logp), _p(loss), _p(dl),
                                   _p(err), _stream(dev))
    _check(rc, "tt_weighted_logprob")
    return logp, loss, dl


def lmhead_logprob(hidden, w_vocab, targets, weights=None, out=None, ws=None, err=None):
    """LM head fused with the weighted log-prob (tt_lmhead_logprob): logits z = hidden·w_vocabᵀ are never stored.
    hidden [N,Hd] bf16, w_vocab [V,Hd] bf16 -> (logp fp32 [N], lse fp32 [N], loss fp64 device scalar)."""
    _need(hidden, torch.bfloat16, "hidden", 2)
    _need(w_vocab, torch.bfloat16, "w_vocab", 2)
    _need(targets, torch.int32, "targets", 1)
    if weights is not None:
        _need(weights, torch.float32, "weights", 1)
    N, Hd = hidden.shape
    V = w_vocab.shape[0]
    if w_vocab.shape[1] != Hd:
        raise ValueError("hidden and w_vocab must share Hd")
    dev = hidden.device
    if out is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        loss = torch.empty(1, dtype=torch.float64, device=dev)
    else:
        logp, lse, loss = out
    nbytes = lib().tt_lmhead_logprob_workspace_bytes(N, V)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if ws is None else ws
    err = new_err(dev) if err is None else err
    rc = lib().tt_lmhead_logprob(_p(hidden), _p(w_vocab), N, V, Hd, _p(targets), _p(weights), _p(logp), _p(lse),
                                 _p(loss), _p(ws), ws.numel(), _p(err), _stream(dev))
    _check(rc, "tt_lmhead_logprob")
    return logp, lse, loss


def lmhead_logprob_bwd(hidden, w_vocab, targets, lse, weights=None, g=1.0, out=None, ws=None, err=None):
    """Gradients of g·loss of lmhead_logprob (tt_lmhead_logprob_bwd): d_hidden bf16 [N,Hd], d_w_vocab fp32 [V,Hd]."""
    _need(hidden, torch.bfloat16, "hidden", 2)
    _need(w_vocab, torch.bfloat16, "w_vocab", 2)
    _need(targets, torch.int32, "targets", 1)
    _need(lse, torch.float32, "lse", 1)
    if weights is not None:
        _need(weights, torch.float32, "weights", 1)
    N, Hd = hidden.shape
    V = w_vocab.shape[0]
    dev = hidden.device
    if out is None:
        dh = torch.empty_like(hidden)
        dw = torch.empty(V, Hd, dtype=torch.float32, device=dev)
    else:
        dh, dw = out
    if ws is None:
        ws = torch.empty(lib().tt_lmhead_logprob_bwd_workspace_bytes(N, V), dtype=torch.uint8, device=dev)
    err = new_err(dev) if err is None else err
    rc = lib().tt_lmhead_logprob_bwd(_p(hidden), _p(w_vocab), N, V, Hd, _p(targets), _p(weights), g, _p(lse), _p(dh),
                                     _p(dw), _p(ws), ws.numel(), _p(err), _stream(dev))
    _check(rc, "tt_lmhead_logprob_bwd")
    return dh, dw


KERNEL_CLASSES = ("fwd", "bwd", "logprob", "lmhead")  # TT_KT_* order


def kernel_timing(on: bool):
    """Turn launch timing on (clearing earlier records) or off (tt_kernel_timing)."""
    _check(lib().tt_kernel_timing(1 if on else 0), "kernel_timing")


def kernel_timing_read():
    """{class: (milliseconds, launches)} of the launches timed since kernel_timing(True), and the
    number of launches that were not timed (tt_kernel_timing_read; waits for the recorded events)."""
    n = len(KERNEL_CLASSES)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    dropped = ctypes.c_int64(0)
    _check(lib().tt_kernel_timing_read(ctypes.cast(ms, _vp), ctypes.cast(cnt, _vp), n, ctypes.byref(dropped)),
           "kernel_timing_read")
    return {c: (ms[i], cnt[i]) for i, c in enumerate(KERNEL_CLASSES)}, dropped.value


def trie_build(rollouts):
    """Prefix tree of rollouts given as sequences of token ids (tt_trie_build, host only).

    Returns a dict of numpy arrays: seg_parent [S], seg_len [S] (int32; valid tree_build inputs), tokens [N]
    (token ids in DFS order), rollout_end [R] (DFS index of each rollout's last token), and the counts
    total_tokens and leaf_tokens (compression = total_tokens / N; leaves-only = leaf_tokens / N)."""
    import numpy as np
    seqs = [np.asarray(r, dtype=np.int32).ravel() for r in rollouts]
    R = len(seqs)
    offsets = np.zeros(R + 1, np.int64)
    if R:
        offsets[1:] = np.cumsum([len(x) for x in seqs])
    toks = np.concatenate(seqs) if R else np.zeros(0, np.int32)
    cap = max(int(offsets[-1]), 1)
    par, ln, tok = (np.empty(cap, np.int32) for _ in range(3))
    ends = np.empty(max(R, 1), np.int64)
    counts = np.zeros(4, np.int64)
    vp = lambda a: a.ctypes.data_as(_vp)
    _check(lib().tt_trie_build(vp(toks), vp(offsets), R, cap, vp(par), vp(ln), vp(tok), vp(ends), vp(counts)),
           "trie_build")
    S, N = int(counts[0]), int(counts[1])
    return {"seg_parent": par[:S].copy(), "seg_len": ln[:S].copy(), "tokens": tok[:N].copy(),
            "rollout_end": ends[:R].copy(), "total_tokens": int(counts[2]), "leaf_tokens": int(counts[3])}
