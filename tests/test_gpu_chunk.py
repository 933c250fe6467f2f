"""Chunk-vs-path attention (tt_tree_attn_chunk_fwd/bwd) and the path-at-a-time
driver (tt_dta_tree_attn) against the oracle and against whole-tree mode."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as A
from oracle import tree as T
from tests._util import GRAD_RL2, LSE_RTOL, O_ATOL, dev_to_f64, f64, rel_l2, to_dev_bf16, workload_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("C,s0,hq,hkv,d", [(1, 0, 1, 1, 64), (77, 0, 2, 1, 64), (200, 333, 4, 2, 128),
                                           (2048, 1000, 8, 2, 128), (129, 4096, 2, 2, 64), (513, 31, 6, 3, 128)])
def test_chunk_vs_oracle(tt, C, s0, hq, hkv, d):
    rng = np.random.default_rng(C + s0)
    P = s0 + C
    q, k, v, do = (synth.normal_bf16(rng, s) for s in ((C, hq, d), (P, hkv, d), (P, hkv, d), (C, hq, d)))
    scale = 1 / np.sqrt(d)
    o_ref, lse_ref = A.causal_attention_forward(f64(q), f64(k), f64(v), scale)
    dq_ref, dk_ref, dv_ref = A.causal_attention_backward(f64(q), f64(k), f64(v), f64(do), scale)
    qd, kd, vd, dod = (to_dev_bf16(x) for x in (q, k, v, do))
    err = tt.new_err("cuda")
    o, lse = tt.tree_attn_chunk_fwd(qd, s0, kd, vd, err=err)
    # accumulation: start from a non-zero buffer and check += semantics
    base_k = torch.randn(P, hkv, d, device="cuda")
    base_v = torch.randn(P, hkv, d, device="cuda")
    dka, dva = base_k.clone(), base_v.clone()
    dq = tt.tree_attn_chunk_bwd(qd, s0, kd, vd, o, lse, dod, dka, dva, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(dev_to_f64(o) - o_ref).max() <= O_ATOL
    assert (np.abs(lse.cpu().numpy() - lse_ref) <= LSE_RTOL * np.abs(lse_ref) + 1e-5).all()
    assert rel_l2(dev_to_f64(dq), dq_ref) <= GRAD_RL2
    assert rel_l2((dka - base_k).cpu().numpy(), dk_ref) <= GRAD_RL2
    assert rel_l2((dva - base_v).cpu().numpy(), dv_ref) <= GRAD_RL2


def _pack_send(tab, s0):
    """send and blk_max of a packed chunk (tt_tree_attn_chunk_fwd_packed) for the local tree `tab` whose root segment
    is the path (s0 tokens) and whose other segments are the chunk: the tree-mode send (end of the subtree of each
    token's segment; the path's tokens get the tree's end, s0 + C, the least allowed), 0 past the chunk. The entries
    the call must never read (send below 128·floor(s0/128), blk_max below floor(s0/128)) hold -7."""
    C = int(tab.N) - s0
    n = (s0 + C + 127) // 128 * 128
    send = np.zeros(n, np.int64)
    send[:s0 + C] = tab.tok_send
    bmax = send.reshape(-1, 128).max(1)
    send[:s0 // 128 * 128] = -7
    bmax[:s0 // 128] = -7
    return torch.tensor(send.astype(np.int32), device="cuda"), torch.tensor(bmax.astype(np.int32), device="cuda")


# (path tokens, the chunk's segments as (parent among them or -1 for the path, tokens), heads): unaligned path,
# aligned segments, one-token segments, few CTAs over a long path (key-range splits), enough CTAs for the paired
# two-tile schedule, a single segment (the causal chunk), and subtrees with inner segments (send not monotone)
@pytest.mark.parametrize("s0,segs,heads", [
    (333, [(-1, 100), (-1, 50), (-1, 200)], (4, 2, 128)),
    (128, [(-1, 128)] * 4, (2, 1, 64)),
    (1000, [(-1, 1)] * 7 + [(-1, 60), (-1, 3)], (2, 2, 64)),
    (4096, [(-1, 100), (-1, 50)], (2, 1, 64)),
    (200, [(-1, 600), (-1, 600), (-1, 500)], (32, 8, 128)),
    (77, [(-1, 300)], (4, 2, 128)),
    (333, [(-1, 100), (0, 50), (0, 60), (-1, 200), (3, 10), (4, 1)], (4, 2, 128)),
    (130, [(-1, 300), (0, 140), (1, 100), (0, 7), (-1, 90)], (2, 1, 64)),
    (257, [(-1, 200), (0, 300), (0, 300), (1, 400), (-1, 500)], (32, 8, 128)),
    (257, [(-1, 900), (0, 300), (-1, 700)], (24, 8, 64)),   # odd group size: paired schedule on adjacent tiles
    (1000, [(-1, 700), (-1, 650), (0, 300)], (32, 8, 64)),  # d = 64 on the paired schedule
])
def test_packed_chunk_vs_oracle(tt, s0, segs, heads):
    """A packed chunk (sibling subtrees behind their shared path) against the oracle on the tree "path as the root,
    the subtrees as its children": O, LSE, dQ of the chunk rows, and the dK/dV it accumulates on every path and
    chunk row (the oracle's dO is zero on the path rows, so only the chunk's queries contribute)."""
    hq, hkv, d = heads
    par = np.array([-1] + [0 if p < 0 else p + 1 for p, _ in segs], np.int32)
    ln = np.array([s0] + [n for _, n in segs], np.int32)
    C = int(ln[1:].sum())
    sh = synth.TreeShape(par, ln, np.random.default_rng(s0 + C))
    tab = T.tables(par, ln)
    inp = synth.attention_inputs(None, tree=sh, heads=heads)
    inp["dO"][:s0] = 0
    ref = A.tree_attention_segments(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")))
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    send, bmax = _pack_send(tab, s0)
    err = tt.new_err("cuda")
    q, do = Q[s0:].contiguous(), dO[s0:].contiguous()
    o, lse = tt.tree_attn_chunk_fwd(q, s0, K, V, err=err, send=send, blk_max=bmax)
    base_k = torch.randn(s0 + C, hkv, d, device="cuda")
    base_v = torch.randn(s0 + C, hkv, d, device="cuda")
    dka, dva = base_k.clone(), base_v.clone()
    dq = tt.tree_attn_chunk_bwd(q, s0, K, V, o, lse, do, dka, dva, err=err, send=send, blk_max=bmax)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(dev_to_f64(o) - ref[0][s0:]).max() <= O_ATOL
    lr = ref[1][:, s0:]
    assert (np.abs(lse.cpu().numpy() - lr) <= LSE_RTOL * np.abs(lr) + 1e-5).all()
    assert rel_l2(dev_to_f64(dq), ref[2][s0:]) <= GRAD_RL2
    assert rel_l2((dka - base_k).cpu().numpy(), ref[3]) <= GRAD_RL2
    assert rel_l2((dva - base_v).cpu().numpy(), ref[4]) <= GRAD_RL2
    # one segment: the same as the unpacked chunk up to fp32 rounding
    if len(segs) == 1:
        o2, lse2 = tt.tree_attn_chunk_fwd(q, s0, K, V, err=err)
        torch.cuda.synchronize()
        assert (o2.float() - o.float()).abs().max().item() <= 2 ** -7
        assert (lse2 - lse).abs().max().item() <= 1e-5


def test_packed_chunk_arguments(tt):
    q = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(128, 1, 64, dtype=torch.bfloat16, device="cuda")
    send = torch.zeros(129, dtype=torch.int32, device="cuda")
    bmax = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(tt.TTError) as e:
        tt.tree_attn_chunk_fwd(q, 64, kv, kv, send=send[1:], blk_max=bmax)  # not 16-byte aligned
    assert e.value.code == -1
    with pytest.raises(tt.TTError) as e:
        tt.tree_attn_chunk_fwd(q, 64, kv, kv, send=send)  # no block maxima
    assert e.value.code == -1
    with pytest.raises(ValueError):
        tt.tree_attn_chunk_fwd(q, 64, kv, kv, send=send, blk_max=bmax, tiles=2)


def _dta(tt, sh, inp, chunk):
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    err = tt.new_err("cuda")
    out = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=chunk, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


@pytest.mark.parametrize("seed,chunk", [(0, 64), (1, 100), (2, 2048)])
def test_dta_small_trees(tt, seed, chunk):
    sh = synth.random_tree(seed, n_seg=8, len_range=(30, 260), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk)
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in _dta(tt, sh, inp, chunk)]
    assert np.abs(got[0] - ref[0]).max() <= O_ATOL
    assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for i in (2, 3, 4):
        assert rel_l2(got[i], ref[i]) <= GRAD_RL2


def _leafy_tree(seed):
    """Root, 40 one-token leaves, an inner child with 6 leaves of 20..140 tokens, 9 leaves of 1..90 tokens."""
    rng = np.random.default_rng(seed)
    par = [-1] + [0] * 40 + [0] + [41] * 6 + [0] * 9
    ln = [300] + [1] * 40 + [50] + list(rng.integers(20, 141, 6)) + list(rng.integers(1, 91, 9))
    return synth.TreeShape(np.array(par, np.int32), np.array(ln, np.int32), rng)


@pytest.mark.parametrize("seed,chunk", [(0, 2048), (1, 100), (2, 17)])
def test_dta_packed_leaves(tt, seed, chunk):
    """Runs of sibling leaves packed into chunks (cut by the chunk size, by the 32-segment limit of a pack and by
    the inner child between runs) against the oracle's path-at-a-time traversal."""
    sh = _leafy_tree(seed)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 64))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk)
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in _dta(tt, sh, inp, chunk)]
    assert np.abs(got[0] - ref[0]).max() <= O_ATOL
    assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for i in (2, 3, 4):
        assert rel_l2(got[i], ref[i]) <= GRAD_RL2


@pytest.mark.parametrize("seed,chunk", [(10, 128), (11, 512), (12, 100000)])
def test_dta_packed_subtrees(tt, seed, chunk):
    """Trees whose inner subtrees fit a chunk (packed whole, send not monotone over the pack), and with a large
    chunk the whole tree as one pack with an empty path, against the oracle's path-at-a-time traversal; the
    traversal's partitions are those of tt_tree_partition (pinned against the oracle's rule on the CPU)."""
    sh = synth.random_tree(seed, n_seg=40, len_range=(1, 70), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 64))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    first, rows, path, kind = tt.tree_partition(sh.seg_parent, sh.seg_len, chunk)
    assert int(rows.sum()) == tab.N and (kind == 0).any()
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk)
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in _dta(tt, sh, inp, chunk)]
    assert np.abs(got[0] - ref[0]).max() <= O_ATOL
    assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for i in (2, 3, 4):
        assert rel_l2(got[i], ref[i]) <= GRAD_RL2


@pytest.mark.parametrize("wid,groups", [(3, (7,)), (1, (0, 7)), (4, (7,))])  # the 8B-shaped result is still cached
def test_dta_full_size_vs_oracle(tt, wid, groups):
    """The path-at-a-time pass the bench times (2048-query chunks) on the Qwen3-1.7B-, 8B- and deep agentic
    14B-shaped trees (the last with 5 query heads per KV head: the paired forward on adjacent tiles): O, LSE, dQ, dK,
    dV of whole KV groups against the fp64 oracle (per-branch exactness: "Tree Training", Abstract)."""
    inp, tab, ref = workload_oracle(wid, groups)
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy().astype(np.float64)
           for x in _dta(tt, inp["tree"], inp, 2048)]
    O, LSE, dQ, dK, dV = got
    G = inp["hq"] // inp["hkv"]
    for g in groups:
        hs = slice(g * G, (g + 1) * G)
        assert np.abs(O[:, hs] - ref[0][:, hs]).max() <= O_ATOL
        assert (np.abs(LSE[hs] - ref[1][hs]) <= LSE_RTOL * np.abs(ref[1][hs]) + 1e-5).all()
        assert rel_l2(dQ[:, hs], ref[2][:, hs]) <= GRAD_RL2
        assert rel_l2(dK[:, g], ref[3][:, g]) <= GRAD_RL2
        assert rel_l2(dV[:, g], ref[4][:, g]) <= GRAD_RL2


@pytest.mark.parametrize("chunk", [2048, 4096])
def test_dta_equals_whole_tree_on_grpo_workload(tt, chunk):
    """Config 3 (root 4096 = two 2048-query chunks, or one with the 4096 variant of AReaL-DTA "Main Findings"):
    chunk mode == whole-tree mode."""
    inp = synth.attention_inputs(3)
    sh = inp["tree"]
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    tree = tt.tree_build(torch.tensor(sh.seg_parent, device="cuda"), torch.tensor(sh.seg_len, device="cuda"))
    O, LSE = tt.tree_attn_fwd(tree, Q, K, V)
    dQ, dK, dV = tt.tree_attn_bwd(tree, Q, K, V, O, LSE, dO)
    O2, LSE2, dQ2, dK2, dV2 = _dta(tt, sh, inp, chunk)
    tree.check()
    # both are bf16 results of the same sums in different tile orders
    assert (O.float() - O2.float()).abs().max().item() <= O_ATOL
    assert ((LSE - LSE2).abs() <= LSE_RTOL * LSE.abs() + 1e-5).all()
    for a, b in ((dQ, dQ2), (dK, dK2), (dV, dV2)):
        assert rel_l2(b.float().cpu().numpy(), a.float().cpu().numpy()) <= GRAD_RL2
    # and against the oracle on sampled rows
    tab = T.tables(sh.seg_parent, sh.seg_len)
    rows = np.r_[0, 2047, 2048, 4095, 4096, tab.N - 1]
    o, lse = A.ancestor_rows_forward(tab, f64(inp["Q"]), f64(inp["K"]), f64(inp["V"]), rows)
    assert np.abs(dev_to_f64(O2)[rows] - o).max() <= O_ATOL


@pytest.mark.parametrize("tiles", [1, 2])
@pytest.mark.parametrize("C,s0,hq,hkv,d", [(300, 129, 4, 2, 128), (385, 0, 3, 1, 64), (1000, 2500, 2, 2, 128),
                                           (640, 77, 3, 3, 128)])  # last: tile pairs, odd tile count (5)
def test_chunk_forward_schedules(tt, tiles, C, s0, hq, hkv, d):
    """The chunk forward matches causal attention with one or two query tiles per CTA."""
    rng = np.random.default_rng(7 * C + s0)
    P = s0 + C
    q, k, v = (synth.normal_bf16(rng, s) for s in ((C, hq, d), (P, hkv, d), (P, hkv, d)))
    o_ref, lse_ref = A.causal_attention_forward(f64(q), f64(k), f64(v), 1 / np.sqrt(d))
    err = tt.new_err("cuda")
    o, lse = tt.tree_attn_chunk_fwd(to_dev_bf16(q), s0, to_dev_bf16(k), to_dev_bf16(v), err=err, tiles=tiles)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(dev_to_f64(o) - o_ref).max() <= O_ATOL
    assert (np.abs(lse.cpu().numpy() - lse_ref) <= LSE_RTOL * np.abs(lse_ref) + 1e-5).all()


@pytest.mark.parametrize("splits", [1, 2, 3, 4])
@pytest.mark.parametrize("C,s0,hq,hkv,d", [(77, 0, 2, 1, 64),       # one key block: the other splits see none
                                           (128, 100, 2, 2, 128),   # row 0 sees no key of the second split
                                           (300, 129, 4, 2, 128), (640, 5120, 4, 1, 128), (385, 1000, 3, 3, 64)])
def test_chunk_forward_key_splits(tt, splits, C, s0, hq, hkv, d):
    """Key-range splits merged in distributed shared memory match causal attention (online-softmax merge of
    disjoint key sets), including splits with no key block and rows with no visible key in a split."""
    rng = np.random.default_rng(11 * C + s0 + splits)
    P = s0 + C
    q, k, v = (synth.normal_bf16(rng, s) for s in ((C, hq, d), (P, hkv, d), (P, hkv, d)))
    o_ref, lse_ref = A.causal_attention_forward(f64(q), f64(k), f64(v), 1 / np.sqrt(d))
    err = tt.new_err("cuda")
    lse_ld = C + 5
    o, lse = tt.tree_attn_chunk_fwd(to_dev_bf16(q), s0, to_dev_bf16(k), to_dev_bf16(v), err=err, lse_ld=lse_ld,
                                    splits=splits)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.abs(dev_to_f64(o) - o_ref).max() <= O_ATOL
    lse = lse.cpu().numpy()[:, :C]
    assert (np.abs(lse - lse_ref) <= LSE_RTOL * np.abs(lse_ref) + 1e-5).all()


def test_chunk_forward_split_arguments(tt):
    x = torch.zeros(128, 1, 64, dtype=torch.bfloat16, device="cuda")
    for bad in (-1, 5):
        with pytest.raises(RuntimeError):
            tt.tree_attn_chunk_fwd(x, 0, x, x, splits=bad)


@pytest.mark.parametrize("seed,chunk", [(10, 96), (11, 300)])
def test_dta_orders_vs_oracle(tt, seed, chunk):
    """Greedy and index visiting orders both match the oracle's traversal in the greedy order (a tree with ties
    between subtrees of equal depth, chunks smaller than segments)."""
    sh = synth.random_tree(seed, n_seg=12, len_range=(40, 400), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk,
                        leaf_order=T.greedy_leaf_order(tab))
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    for order in (tt.DTA_ORDER_GREEDY, tt.DTA_ORDER_INDEX):
        err = tt.new_err("cuda")
        out = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=chunk, err=err, order=order)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in out]
        assert np.abs(got[0] - ref[0]).max() <= O_ATOL
        assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
        for i in (2, 3, 4):
            assert rel_l2(got[i], ref[i]) <= GRAD_RL2


def test_dta_plan_matches_the_direct_call_bitwise(tt):
    """A captured plan replays exactly the direct call's work: bitwise-equal outputs, twice, and new inputs written
    into the bound tensors are picked up."""
    sh = synth.random_tree(21, n_seg=10, len_range=(40, 500), max_children=3)
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    plan = tt.DtaPlan(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=256)
    for _ in range(2):
        got = plan.launch()
        direct = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=256)
        torch.cuda.synchronize()
        assert int(plan.err.item()) == 0
        for a, b in zip(direct, got):
            assert torch.equal(a, b)
    Q.mul_(0.5)
    got = plan.launch()
    direct = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=256)
    torch.cuda.synchronize()
    for a, b in zip(direct, got):
        assert torch.equal(a, b)
    plan.close()


def test_dta_plan_rejects_an_invalid_tree(tt):
    Q = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tt.TTError) as e:
        tt.DtaPlan(np.array([-1, 2, 0], np.int32), np.array([4, 3, 3], np.int32), Q, Q, Q, Q, chunk=64)
    assert e.value.code == -2


def _grpo_like(seed, n_mid=3, n_leaf=5):
    """Root, n_mid children, n_leaf leaves under each (runs of sibling leaves), short random lengths."""
    rng = np.random.default_rng(seed)
    par, ln = [-1], [int(rng.integers(200, 400))]
    for m in range(n_mid):
        par.append(0)
        ln.append(int(rng.integers(100, 300)))
        mid = len(par) - 1
        for _ in range(n_leaf):
            par.append(mid)
            ln.append(int(rng.integers(30, 260)))
    return synth.TreeShape(np.array(par, np.int32), np.array(ln, np.int32), rng)


@pytest.mark.parametrize("slots", [1, 2, 3])
@pytest.mark.parametrize("maker,chunk", [(lambda: _grpo_like(40), 128), (lambda: _grpo_like(41, 2, 7), 2048),
                                         (lambda: synth.random_tree(42, n_seg=14, len_range=(30, 300),
                                                                    max_children=4), 100)])
def test_dta_slots_vs_oracle(tt, slots, maker, chunk):
    """Sibling leaves spread over 1, 2 or 3 path stacks (own streams, prefix sums folded in slot order) match the
    oracle's traversal; the results do not depend on timing (two runs bitwise equal)."""
    sh = maker()
    inp = synth.attention_inputs(None, tree=sh, heads=(4, 2, 128))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk,
                        leaf_order=T.greedy_leaf_order(tab))
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    runs = []
    for _ in range(2):
        err = tt.new_err("cuda")
        runs.append(tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=chunk, err=err, slots=slots))
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in runs[0]]
    assert np.abs(got[0] - ref[0]).max() <= O_ATOL
    assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for i in (2, 3, 4):
        assert rel_l2(got[i], ref[i]) <= GRAD_RL2


def test_dta_slot_count_checked(tt):
    sh = _grpo_like(43, 1, 2)
    Q = torch.zeros(sh.N, 2, 64, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for bad in (0, 9):
        with pytest.raises(tt.TTError) as e:
            tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, Q, Q, Q, chunk=64, ws=ws, slots=bad)
        assert e.value.code == -1


@pytest.mark.parametrize("seed", range(24))
def test_dta_random_partitions(tt, seed):
    """Random trees (chains, bushes, many one-token segments) under random chunk sizes and 1–3 path stacks: every
    output against the oracle's path-at-a-time traversal, so that every kind of partition (chunks of large segments,
    packs of leaves, packs of inner subtrees, the whole tree as one pack) and every fork rule meets it."""
    rng = np.random.default_rng(1000 + seed)
    n_seg = int(rng.integers(2, 40))
    lo = int(rng.choice([1, 1, 5, 20]))
    sh = synth.random_tree(2000 + seed, n_seg=n_seg, len_range=(lo, lo + int(rng.integers(1, 150))),
                           max_children=int(rng.integers(1, 6)), chain=bool(seed % 11 == 0))
    chunk = int(rng.choice([16, 37, 64, 128, 300, 1000, 100000]))
    slots = int(rng.integers(1, 4))
    inp = synth.attention_inputs(None, tree=sh, heads=(2, 1, 64))
    tab = T.tables(sh.seg_parent, sh.seg_len)
    first, rows, path, kind = tt.tree_partition(sh.seg_parent, sh.seg_len, chunk)
    assert int(rows.sum()) == tab.N
    ref = A.dta_chunked(tab, *(f64(inp[k]) for k in ("Q", "K", "V", "dO")), chunk=chunk)
    Q, K, V, dO = (to_dev_bf16(inp[k]) for k in ("Q", "K", "V", "dO"))
    err = tt.new_err("cuda")
    out = tt.dta_tree_attn(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=chunk, err=err, slots=slots)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = [dev_to_f64(x) if x.dtype == torch.bfloat16 else x.cpu().numpy() for x in out]
    assert np.abs(got[0] - ref[0]).max() <= O_ATOL, (n_seg, chunk, slots)
    assert (np.abs(got[1] - ref[1]) <= LSE_RTOL * np.abs(ref[1]) + 1e-5).all()
    for i in (2, 3, 4):
        assert rel_l2(got[i], ref[i]) <= GRAD_RL2, (i, n_seg, chunk, slots)
