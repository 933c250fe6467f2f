"""libtt loads, exports every symbol include/tt.h declares, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from prefix_tree_gb300 import build, lib
    build.build()
    return lib()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "tt.h")).read()
    return sorted(set(re.findall(r"TT_API\s+[\w\s\*]+?\b(tt_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    from prefix_tree_gb300 import exported_symbols
    syms = header_symbols()
    assert len(syms) >= 12
    for s in syms:
        assert hasattr(L, s), s
    assert sorted(exported_symbols()) == syms


def test_host_only_entry_points(L):
    assert L.tt_version() == 203  # 2.03: packed chunks (sibling subtrees, block maxima) and tree partitioning
    assert L.tt_status_string(0) == b"TT_OK"
    assert b"INVALID_TREE" in L.tt_status_string(-2)
    assert L.tt_tree_workspace_bytes(7, 196) > 196 * 4
    assert L.tt_tree_workspace_bytes(0, 196) == 0
    assert L.tt_tree_attn_bwd_workspace_bytes(196, 4) >= 196 * 4 * 4
    par = np.array([-1, 0, 0, 1], np.int32)
    ln = np.array([5, 3, 2, 4], np.int32)
    vp = ctypes.c_void_p
    n = L.tt_dta_workspace_bytes(par.ctypes.data_as(vp), ln.ctypes.data_as(vp), 4, 2048, 2, 1, 64)
    assert n >= 12 * 64 * 2 * 2          # path stack of the longest path (12 tokens)
    bad = np.array([-1, 2, 0, 1], np.int32)  # parent must precede child
    assert L.tt_dta_workspace_bytes(bad.ctypes.data_as(vp), ln.ctypes.data_as(vp), 4, 2048, 2, 1, 64) == 0
    # one path stack per slot: the default is two, slots outside 1..8 are rejected
    ws1 = L.tt_dta_workspace_bytes_slots(par.ctypes.data_as(vp), ln.ctypes.data_as(vp), 4, 2048, 2, 1, 64, 1)
    ws2 = L.tt_dta_workspace_bytes_slots(par.ctypes.data_as(vp), ln.ctypes.data_as(vp), 4, 2048, 2, 1, 64, 2)
    assert ws2 == 2 * ws1 == n
    for bad_slots in (0, 9):
        assert L.tt_dta_workspace_bytes_slots(par.ctypes.data_as(vp), ln.ctypes.data_as(vp), 4, 2048, 2, 1, 64,
                                              bad_slots) == 0
    # many short leaves: a stack also holds the parent's path plus one chunk of its leaves packed behind it
    par2 = np.array([-1, 0, 0, 0, 0], np.int32)
    ln2 = np.array([10, 3, 3, 3, 3], np.int32)
    rowk = 1 * 64
    for chunk, rows in ((2048, 22), (5, 15)):  # 10 + min(chunk, 12) rows against a longest path of 13
        m = L.tt_dta_workspace_bytes_slots(par2.ctypes.data_as(vp), ln2.ctypes.data_as(vp), 5, chunk, 2, 1, 64, 1)
        assert m >= rows * rowk * (2 + 2 + 4 + 4) + rows * 4


def test_kernel_timing_host_side(L):
    """Launch timing: on/off and reading with no launches recorded need no GPU."""
    import prefix_tree_gb300 as tt
    tt.kernel_timing(True)
    times, dropped = tt.kernel_timing_read()
    assert times == {c: (0.0, 0) for c in tt.KERNEL_CLASSES} and dropped == 0
    tt.kernel_timing(False)
    assert L.tt_kernel_timing_read(None, None, 4, None) == -1  # TT_ERR_INVALID_ARG


def test_host_side_argument_errors(L):
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    # unsupported head_dim / head grouping
    assert L.tt_tree_attn_fwd(fake, fake, fake, fake, fake, fake, 100, 4, 2, 96, 0.1, fake, None) == -3
    assert L.tt_tree_attn_fwd(fake, fake, fake, fake, fake, fake, 100, 3, 2, 64, 0.1, fake, None) == -3
    # null pointer / empty
    assert L.tt_tree_attn_fwd(None, fake, fake, fake, fake, fake, 100, 4, 2, 64, 0.1, fake, None) == -1
    assert L.tt_tree_build(fake, fake, 0, 10, None, 0, fake, 0, fake, None) == -1
    assert L.tt_weighted_logprob(fake, 10, 5, 4, fake, None, 1.0, fake, fake, None, fake, None) == -1  # ld < V
    # invalid host tree for the path-at-a-time driver
    par = np.array([0, 0], np.int32)
    ln = np.array([1, 1], np.int32)
    vp = ctypes.c_void_p
    args = [par.ctypes.data_as(vp), ln.ctypes.data_as(vp), 2, 2, 2048] + [fake] * 9 + [1, 1, 64, 0.125, fake, 1 << 20,
                                                                                    fake, None]
    assert L.tt_dta_tree_attn(*args) == -2
    # packed chunks: send (16-byte aligned) and the per-block maxima are required
    cargs = [fake, 64, 100, fake, fake]
    tail = [fake, fake, 64, 2, 1, 64, 0.125, fake, None]
    assert L.tt_tree_attn_chunk_fwd_packed(*cargs, None, fake, *tail) == -1
    assert L.tt_tree_attn_chunk_fwd_packed(*cargs, fake, None, *tail) == -1
    assert L.tt_tree_attn_chunk_fwd_packed(*cargs, ctypes.c_void_p(4100), fake, *tail) == -1
    btail = [fake, fake, 64, fake, fake, fake, fake, 2, 1, 64, 0.125, fake, 1 << 20, fake, None]
    assert L.tt_tree_attn_chunk_bwd_packed(*cargs, None, fake, *btail) == -1
    assert L.tt_tree_attn_chunk_bwd_packed(*cargs, fake, None, *btail) == -1
    assert L.tt_tree_attn_chunk_bwd_packed(*cargs, ctypes.c_void_p(4100), fake, *btail) == -1
