"""Benchmark of the prefix-tree training hot path on one GB300 (or N replicas).

Headline workload: the Qwen3-8B-shaped GRPO rollout tree (4096-token root, 8
children of 1024 tokens, 8 leaves of U[256,768] tokens under each: 64
leaves, 45,379 unique tokens, 7.95x compression; 32 query / 8 key-value
heads, d = 128). One step = one pass of every hot-path stage:
  tree build -> whole-tree attention forward -> backward ->
  path-at-a-time (2048-query chunks, right to left) forward+backward of the
  same tree (a plan: the traversal captured once into a CUDA graph, one
  launch per step) -> weighted log-prob + loss + dlogits over the 12,669 tokens of
  the Qwen3-1.7B-shaped tree at V = 151,936 (logits [12669, 151936] bf16).
Inputs are synthetic, seeded and resident in HBM before timing.

value = useful tree-attention TFLOP/s of the whole-tree forward+backward of
the headline tree (only ancestor pairs count: 14·d·Hq·pairs). The other
attention workloads (tiny tree, Qwen3-1.7B-shaped tree, deep agentic
14B-shaped tree) and the 4096-query path-at-a-time variant are timed after
the steps, each on its own with L2 flushed before every iteration, and
reported under `workloads`. `roofline` is for the kernel class with the most
device time per step, timed by CUDA events the library records around each
of its launches on the launch's own stream (tt_kernel_timing) over a second
run of the same steps; its algorithmic work is the step's useful work of
that class: forward 4, backward kernel 10 (S, dP, dV, dK, dQ; the S and dP
its dQ CTAs form again are not credited) flops per ancestor pair per d·Hq,
for the whole-tree call and the path-at-a-time chunks; log-prob 4·N·V + 12·N
bytes. Fractions are of the measured burst bf16 peak (the steps run well
under a second) and of the measured HBM copy bandwidth. Timing: CUDA events
on the launching stream, W warm-up steps, K timed steps bracketed by
barrier + synchronize. L2: the log-prob stage streams 7.7 GB (>> 129 MB L2)
between consecutive attention passes, and its own inputs exceed L2.

--impl reference times the CPU oracle (the reference arm of this build) on a
bounded sample of the headline workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-attn fwd+bwd useful TFLOPS (% bf16 peak); weighted-logprob HBM GB/s"
HEADLINE = 3  # synthetic workload id of the Qwen3-8B-shaped GRPO tree
WORKLOAD = ("Qwen3-8B-shaped GRPO tree attention (Hq=32, Hkv=8, d=128; 4096-token root, 8x1024, 64 leaves "
            "U[256,768], N=45379, 7.95x compression), fwd+bwd whole-tree and path-at-a-time (2048-query chunks) "
            "+ weighted log-prob over the Qwen3-1.7B-shaped tree's 12669 tokens at V=151936 (seed 0)")
# The other attention workloads, reported after the steps (id: description).
SIDE_WORKLOADS = {
    0: "tiny tree (root 64, 2x32, 4 leaves U[8,24]; N=196), 1 head, d=64",
    1: "Qwen3-1.7B-shaped tree (2048-token root, 4x4 branches U[256,768]; N=12669), Hq=16, Hkv=8, d=128",
    4: "deep agentic Qwen3-14B-shaped tree (7 segment levels, U[1,3] children, U[32,1024] lengths; N=32136), "
       "Hq=40, Hkv=8, d=128",
}
CHUNK = 2048
CHUNK_VARIANT = 4096
CPU_ORACLE_THREADS = os.cpu_count() or 1
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
# DRAM bytes (read + write) of one log-prob row at V = 151936 measured by ncu
# (a 2048-row launch: 623.3 MB read + 562.2 MB written).
LP_TRAFFIC_VOCAB = 151936
LP_TRAFFIC_PER_ROW = (623346176 + 562226176) / 2048
# ncu DRAM bytes (read + write) of the whole-tree forward and backward launches
# per attention workload (the backward's small pre-kernel not included);
# workloads without a capture report null.
ATTN_TRAFFIC = {
    1: {"fwd": 110959360 + 22983936, "bwd": 403075328 + 80562944},
    3: {"fwd": 1193966848 + 340193024, "bwd": 9384893952 + 529950976},
    4: {"fwd": 1037719808 + 296361728, "bwd": 8349900288 + 430888704},
}
# The LM head fused with the log-prob loss: config 2's tree (N = 12669) through
# a Qwen3-1.7B-shaped head (hidden 2048) at the Qwen3 vocabulary.
LMHEAD = dict(vocab=151936, hidden=2048)
LMHEAD_WORKLOAD = ("LM head fused with the weighted log-prob: H [12669, 2048] x W [151936, 2048] bf16 "
                   "(Qwen3-1.7B hidden size and vocabulary over the Qwen3-1.7B-shaped tree), logits never stored")
LMHEAD_ORACLE_ROWS = 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tt", choices=["tt", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-side", action="store_true", help="skip the other workloads after the steps")
    ap.add_argument("--stage", default="all", choices=["all", "attn", "logprob", "lmhead"],
                    help="profiling aid: run only the attention stages, only the log-prob stage, or only the fused "
                         "LM-head call (--steps iterations after --warmup, one JSON line)")
    ap.add_argument("--workload", type=int, default=HEADLINE, choices=[0, 1, 3, 4],
                    help="profiling aid: attention workload of the steps (default: the headline tree)")
    ap.add_argument("--lp-rows", type=int, default=0,
                    help="profiling aid: log-prob over only the first R rows (0 = all)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing
def dist_setup(n):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cpu"):
    """Maximum of a float over all ranks (identity at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- peaks, clocks
def peaks():
    """(HBM GB/s, burst bf16 TFLOP/s, sustained bf16 TFLOP/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs") or p.get("hbm_GBs")
        bf = p.get("bf16_tflops")
        if hbm and bf:
            return float(hbm), float(bf), float(p.get("bf16_tflops_sustained") or bf), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []
        self.window = (0.0, float("inf"))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a moment to start: wait (at most 3 s) for its first sample
            t_end = time.perf_counter() + 3.0
            while not self.lines and time.perf_counter() < t_end:
                time.sleep(0.01)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def timed(self, t0, t1):
        """Keep only the samples that arrived while the timed steps ran (plus one interval)."""
        self.window = (t0, t1 + 0.06)

    def summary(self):
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if not (self.window[0] <= ts <= self.window[1]):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        if power:
            out["power_w_max"] = max(power)
        return out


# ----------------------------------------------------------------------------- workloads
def useful_pairs(seg_parent, seg_len):
    """Σ_t |anc(t)| = Σ_s len·pathlen + len(len+1)/2 (host arithmetic on the segment arrays)."""
    pl = [0] * len(seg_len)
    tot = 0
    for s in range(len(seg_len)):
        if s:
            pl[s] = pl[seg_parent[s]] + int(seg_len[seg_parent[s]])
        L = int(seg_len[s])
        tot += L * pl[s] + L * (L + 1) // 2
    return tot


def branch_tokens(seg_parent, seg_len):
    """Σ over root-to-leaf branches of their lengths (the tokens a per-branch computation would process)."""
    S = len(seg_len)
    has_child = [False] * S
    for c in range(1, S):
        has_child[seg_parent[c]] = True
    pl = [0] * S
    tot = 0
    for s in range(S):
        if s:
            pl[s] = pl[seg_parent[s]] + int(seg_len[seg_parent[s]])
        if not has_child[s]:
            tot += pl[s] + int(seg_len[s])
    return tot


def _bf16(bits, device=None, pin=False):
    import numpy as np
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if pin:
        return t.pin_memory()
    return t.to(device)


def attention_case(wid, device, pin=False):
    """Seeded inputs of one attention workload on `device` (and pinned host copies if `pin`)."""
    import torch

    import synth
    att = synth.attention_inputs(wid)
    sh = att["tree"]
    c = dict(wid=wid, sh=sh, N=sh.N, hq=att["hq"], hkv=att["hkv"], d=att["d"],
             P=useful_pairs(sh.seg_parent, sh.seg_len), branch_tokens=branch_tokens(sh.seg_parent, sh.seg_len))
    host = {k: _bf16(att[k], pin=True) for k in ("Q", "K", "V", "dO")} if pin else None
    c["host"] = None
    if pin:
        host["par"] = torch.tensor(sh.seg_parent).pin_memory()
        host["len"] = torch.tensor(sh.seg_len).pin_memory()
        c["host"] = host
        c["dev"] = {k: v.to(device, non_blocking=True) for k, v in host.items()}
    else:
        c["dev"] = {k: _bf16(att[k], device) for k in ("Q", "K", "V", "dO")}
        c["dev"]["par"] = torch.tensor(sh.seg_parent, device=device)
        c["dev"]["len"] = torch.tensor(sh.seg_len, device=device)
    torch.cuda.synchronize(device)
    return c


def logprob_case(device, lp_rows=0):
    import torch

    import synth
    lp = synth.logprob_inputs(2)
    if lp_rows:
        lp = dict(lp, logits=lp["logits"][:lp_rows], targets=lp["targets"][:lp_rows])
    sh = lp["tree"]
    c = dict(V=lp["V"], n=lp["logits"].shape[0], logits=_bf16(lp["logits"], device),
             targets=torch.tensor(lp["targets"], device=device),
             par=torch.tensor(sh.seg_parent, device=device), len=torch.tensor(sh.seg_len, device=device))
    torch.cuda.synchronize(device)
    return c


def branch_rollouts(seg_parent, seg_len):
    """The tree's root-to-leaf token sequences (one rollout per leaf), with a distinct token id per tree node,
    from the segment arrays alone (host arithmetic)."""
    import numpy as np
    S = len(seg_len)
    first = np.concatenate([[0], np.cumsum(np.asarray(seg_len, np.int64))[:-1]])
    has_child = np.zeros(S, bool)
    for c in range(1, S):
        has_child[seg_parent[c]] = True
    out = []
    for leaf in range(S):
        if has_child[leaf]:
            continue
        path, s = [], leaf
        while s >= 0:
            path.append(np.arange(first[s], first[s] + seg_len[s], dtype=np.int32))
            s = seg_parent[s] if s else -1
        out.append(np.concatenate(path[::-1]))
    return out


def time_trie_build(tt, seg_parent, seg_len, reps=10):
    """Host time of tt_trie_build (the step before the tree build) on the tree's branch rollouts."""
    rolls = branch_rollouts(seg_parent, seg_len)
    out = tt.trie_build(rolls)
    t0 = time.perf_counter()
    for _ in range(reps):
        out = tt.trie_build(rolls)
    ms = (time.perf_counter() - t0) / reps * 1e3
    tot = out["total_tokens"]
    return {"ms": round(ms, 3), "rollouts": len(rolls), "rollout_tokens": tot, "unique_tokens": len(out["tokens"]),
            "segments": len(out["seg_len"]), "compression": round(tot / len(out["tokens"]), 3),
            "mtokens_per_s": round(tot / ms / 1e3, 2), "where": "host (C++), the step before the tree build"}


def _dta_walk(seg_parent, seg_len, chunk, slots=2):
    """(kernel launches, fold kernels) of one path-at-a-time pass: the driver's rules restated on the host.

    Layout: DFS preorder, children by index. Visiting order: greedy (children by decreasing depth of their deepest
    leaf, ties by that leaf's index). A subtree is packable when it holds <= `chunk` rows and <= 64 segments; a
    packable root makes the whole tree one pack. Otherwise a run of consecutive packable children (visiting order)
    is cut into packs: whole subtrees adjacent in the layout (taken in layout order), <= `chunk` rows and <= 64
    segments each; a pack holding one leaf is a plain segment. A segment's children as units (children that are not
    packable as subtrees, runs as their packs): with slots > 1, >= 2 children, >= 2 units and none holding more than
    half of their ancestor pairs, all units fork over min(slots, units) stacks and nothing below them forks;
    otherwise the children that are not packable are visited the same way and each run's packs fork over
    min(slots, packs) stacks. A fork over u stacks ends with u - 1 folds. Launches: a segment = its forward chunks
    + (pre-kernel + backward) per chunk + one gradient conversion; any other pack = send fill, forward, pre-kernel,
    backward, conversion."""
    S = len(seg_len)
    ln = [int(x) for x in seg_len]
    par = [int(x) for x in seg_parent]
    kids = [[] for _ in range(S)]
    for c in range(1, S):
        kids[par[c]].append(c)
    sub, nseg = ln[:], [1] * S
    for c in range(S - 1, 0, -1):
        sub[par[c]] += sub[c]
        nseg[par[c]] += nseg[c]
    start, pathlen, cur = [0] * S, [0] * S, [0] * S
    cur[0] = ln[0]
    for c in range(1, S):
        p = par[c]
        start[c], cur[p] = cur[p], cur[p] + sub[c]
        cur[c] = start[c] + ln[c]
        pathlen[c] = pathlen[p] + ln[p]
    deep, deep_leaf = [-1] * S, [S] * S
    for s in range(S - 1, -1, -1):
        if not kids[s]:
            deep[s], deep_leaf[s] = pathlen[s] + ln[s], s
        if s > 0:
            p = par[s]
            if deep[s] > deep[p] or (deep[s] == deep[p] and deep_leaf[s] < deep_leaf[p]):
                deep[p], deep_leaf[p] = deep[s], deep_leaf[s]
    for s in range(S):
        kids[s].sort(key=lambda c: (-deep[c], deep_leaf[c]))
    work = [ln[s] * (pathlen[s] + 0.5 * (ln[s] + 1)) for s in range(S)]
    for c in range(S - 1, 0, -1):
        work[par[c]] += work[c]

    def packable(c):
        return sub[c] <= chunk and nseg[c] <= 64

    def packs_of(run):
        out = []  # [roots, rows, segments]
        for c in sorted(run, key=lambda x: start[x]):
            if out:
                P = out[-1]
                if start[c] == start[P[0][0]] + P[1] and P[1] + sub[c] <= chunk and P[2] + nseg[c] <= 64:
                    P[0].append(c)
                    P[1] += sub[c]
                    P[2] += nseg[c]
                    continue
            out.append([[c], sub[c], nseg[c]])
        return [P[0] for P in out]

    def seg_launches(s):
        return math.ceil(ln[s] / chunk) * 3 + 1

    def pack_launches(P):
        return seg_launches(P[0]) if len(P) == 1 and not kids[P[0]] else 5

    def units_of(s):  # [(kind, item, work)] in visiting order
        units, run = [], []
        for c in kids[s] + [None]:
            if c is not None and packable(c):
                run.append(c)
                continue
            for P in packs_of(run):
                units.append(("pack", P, sum(work[x] for x in P)))
            run = []
            if c is not None:
                units.append(("seg", c, work[c]))
        return units

    def seq_launches(c):  # a subtree that is not packable, on one stack
        n = seg_launches(c)
        for kind, item, _ in units_of(c):
            n += pack_launches(item) if kind == "pack" else seq_launches(item)
        return n

    if packable(0):
        return pack_launches([0]), 0
    launches, folds = seg_launches(0), 0
    stack = [0]
    while stack:
        s = stack.pop()
        units = units_of(s)
        ws = [w for _, _, w in units]
        if slots > 1 and len(kids[s]) >= 2 and len(units) >= 2 and max(ws) <= 0.5 * sum(ws):
            launches += sum(pack_launches(i) if k == "pack" else seq_launches(i) for k, i, _ in units)
            folds += min(slots, len(units)) - 1
            continue
        run = []
        for c in kids[s] + [None]:
            if c is not None and packable(c):
                run.append(c)
                continue
            if run:
                P = packs_of(run)
                launches += sum(pack_launches(x) for x in P)
                if slots > 1 and len(P) >= 2:
                    folds += min(slots, len(P)) - 1
            run = []
            if c is not None:
                launches += seg_launches(c)
                stack.append(c)
    return launches, folds


def dta_folds(seg_parent, seg_len, slots=2, chunk=2048):
    """Fold kernels of one path-at-a-time pass (_dta_walk)."""
    return _dta_walk(seg_parent, seg_len, chunk, slots)[1]


def dta_launches(seg_parent, seg_len, chunk, slots=2):
    """Kernel launches of one path-at-a-time pass, folds included (_dta_walk)."""
    n, f = _dta_walk(seg_parent, seg_len, chunk, slots)
    return n + f


def time_lmhead(tt, device, flush, bf16_peak, iters=10, warmup=3):
    """tt_lmhead_logprob on the LM-head workload: median CUDA-event time of the call (L2 flushed before every
    iteration; W alone is 622 MB) and the fused kernel's own launch time (tt_kernel_timing)."""
    import numpy as np
    import torch

    import synth
    d = synth.lmhead_inputs(0, **LMHEAD)
    H, W = _bf16(d["H"], device), _bf16(d["W"], device)
    N, Hd = H.shape
    V = W.shape[0]
    y = torch.tensor(d["targets"], device=device)
    wts = torch.tensor(np.random.default_rng(1).random(N).astype(np.float32), device=device)
    out = (torch.empty(N, dtype=torch.float32, device=device), torch.empty(N, dtype=torch.float32, device=device),
           torch.empty(1, dtype=torch.float64, device=device))
    ws = torch.empty(tt.lib().tt_lmhead_logprob_workspace_bytes(N, V), dtype=torch.uint8, device=device)
    err = tt.new_err(device)
    stream = torch.cuda.current_stream(device)
    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def one(ev):
        flush.add_(1)
        ev[0].record(stream)
        tt.lmhead_logprob(H, W, y, wts, out=out, ws=ws, err=err)
        ev[1].record(stream)

    for _ in range(warmup):
        one(mk())
    evs = [mk() for _ in range(iters)]
    for ev in evs:
        one(ev)
    torch.cuda.synchronize(device)
    tt.kernel_timing(True)
    for _ in range(iters):
        one(mk())
    torch.cuda.synchronize(device)
    tt.kernel_timing(False)
    kt, _ = tt.kernel_timing_read()
    tt.check_err(err, "LM head")
    ms = statistics.median(ev[0].elapsed_time(ev[1]) for ev in evs)
    k_ms = kt["lmhead"][0] / max(kt["lmhead"][1], 1)
    # backward (tt_lmhead_logprob_bwd: dz, dH = dz·W, dW = dzᵀ·H), after the forward's lse
    lse = out[1]
    grads = (torch.empty_like(H), torch.empty(V, Hd, dtype=torch.float32, device=device))
    wsb = torch.empty(tt.lib().tt_lmhead_logprob_bwd_workspace_bytes(N, V), dtype=torch.uint8, device=device)

    def one_bwd(ev):
        flush.add_(1)
        ev[0].record(stream)
        tt.lmhead_logprob_bwd(H, W, y, lse, wts, out=grads, ws=wsb, err=err)
        ev[1].record(stream)

    for _ in range(warmup):
        one_bwd(mk())
    evs_b = [mk() for _ in range(iters)]
    for ev in evs_b:
        one_bwd(ev)
    torch.cuda.synchronize(device)
    tt.check_err(err, "LM head backward")
    ms_b = statistics.median(ev[0].elapsed_time(ev[1]) for ev in evs_b)
    del wsb, grads
    flops = 2.0 * N * V * Hd
    tf, ktf = flops / (ms * 1e-3) / 1e12, flops / (k_ms * 1e-3) / 1e12
    tfb = 3 * flops / (ms_b * 1e-3) / 1e12
    return {"workload": LMHEAD_WORKLOAD, "rows": N, "vocab": V, "hidden": Hd, "useful_gflop": round(flops / 1e9, 1),
            "iters": iters, "l2": "flushed before every iteration", "ms": round(ms, 4), "tflops": round(tf, 2),
            "frac": round(tf / bf16_peak, 4), "tokens_per_s": round(N / (ms * 1e-3)),
            "roofline": {"bound": "tensor", "kernel": "lmhead_gemm_kernel (forward: log-sum-exp epilogue)",
                         "achieved": round(ktf, 2), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(ktf / bf16_peak, 4), "ms_per_launch": round(k_ms, 4), "traffic": None,
                         "algorithmic_flops": flops, "peak_source": "measured burst"},
            "backward": {"ms": round(ms_b, 4), "useful_gflop": round(3 * flops / 1e9, 1), "tflops": round(tfb, 2),
                         "frac": round(tfb / bf16_peak, 4),
                         "work": "dz = g·w·(softmax − onehot) from recomputed logits, dH = dz·W, dW = dzᵀ·H"},
            "fwd_bwd_ms": round(ms + ms_b, 4),
            "fwd_bwd_tflops": round(4 * flops / ((ms + ms_b) * 1e-3) / 1e12, 2),
            "fwd_bwd_frac": round(4 * flops / ((ms + ms_b) * 1e-3) / 1e12 / bf16_peak, 4),
            "logits_bytes_not_stored": 2 * N * V}


def attn_flops(c):
    return 4.0 * c["d"] * c["hq"] * c["P"], 10.0 * c["d"] * c["hq"] * c["P"]


# ----------------------------------------------------------------------------- GPU arm
def time_side_workload(tt, c, device, flush, bf16_peak, iters=10, warmup=3, dta_chunk=None):
    """Whole-tree fwd and bwd (or the path-at-a-time pass with `dta_chunk`) of one workload, L2 flushed before
    every timed iteration; median CUDA-event times."""
    import torch
    dv = c["dev"]
    stream = torch.cuda.current_stream(device)
    tree = tt.tree_build(dv["par"], dv["len"]).check()
    Q, K, V, dO = dv["Q"], dv["K"], dv["V"], dv["dO"]
    err = tt.new_err(device)
    O = torch.empty_like(Q)
    LSE = torch.empty(c["hq"], c["N"], dtype=torch.float32, device=device)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    bws = torch.empty(tt.lib().tt_tree_attn_bwd_workspace_bytes(c["N"], c["hq"]), dtype=torch.uint8, device=device)
    sh = c["sh"]
    if dta_chunk:
        dws = torch.empty(tt.dta_workspace_bytes(sh.seg_parent, sh.seg_len, dta_chunk, c["hq"], c["hkv"], c["d"]),
                          dtype=torch.uint8, device=device)
        plan = tt.DtaPlan(sh.seg_parent, sh.seg_len, Q, K, V, dO, chunk=dta_chunk, err=err, ws=dws,
                          out=(O, LSE, dQ, dK, dV))

    def one(ev):
        flush.add_(1)
        ev[0].record(stream)
        if dta_chunk:
            plan.launch()
            ev[1].record(stream)
        else:
            tt.tree_attn_fwd(tree, Q, K, V, out=(O, LSE), err=err)
            ev[1].record(stream)
            tt.tree_attn_bwd(tree, Q, K, V, O, LSE, dO, out=(dQ, dK, dV), ws=bws, err=err)
        ev[2].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(warmup):
        one(mk())
    evs = [mk() for _ in range(iters)]
    for ev in evs:
        one(ev)
    torch.cuda.synchronize(device)
    tt.check_err(err, f"workload {c['wid']}")
    t_a = statistics.median(ev[0].elapsed_time(ev[1]) for ev in evs)
    t_b = statistics.median(ev[1].elapsed_time(ev[2]) for ev in evs)
    ff, fb = attn_flops(c)
    tot = t_a + t_b
    out = {"tokens": c["N"], "pairs": c["P"], "heads": [c["hq"], c["hkv"], c["d"]],
           "useful_gflop": round((ff + fb) / 1e9, 3), "iters": iters, "l2": "flushed before every iteration"}
    if dta_chunk:
        out.update({"chunk": dta_chunk, "ms": round(tot, 4)})
    else:
        out.update({"fwd_ms": round(t_a, 4), "bwd_ms": round(t_b, 4), "ms": round(tot, 4),
                    "fwd_tflops": round(ff / (t_a * 1e-3) / 1e12, 2), "bwd_tflops": round(fb / (t_b * 1e-3) / 1e12, 2)})
        if c["wid"] in ATTN_TRAFFIC:
            # ncu DRAM bytes of one whole-tree launch of each kernel on this tree
            out["traffic"] = dict(ATTN_TRAFFIC[c["wid"]])
    tfl = (ff + fb) / (tot * 1e-3) / 1e12
    out.update({"tflops": round(tfl, 2), "frac": round(tfl / bf16_peak, 4),
                "tokens_per_s": round(c["N"] / (tot * 1e-3)),
                "branch_tokens_per_s": round(c["branch_tokens"] / (tot * 1e-3))})
    return out


def run_tt(args, rank, world, local):
    import torch

    import prefix_tree_gb300 as tt
    from prefix_tree_gb300 import build as _b
    _b.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    do_attn, do_lp = args.stage in ("all", "attn"), args.stage in ("all", "logprob")
    c = attention_case(args.workload, device, pin=not args.no_e2e and args.stage == "all")
    lpc = logprob_case(device, args.lp_rows) if do_lp else None
    sh, N, hq, hkv, d, P = c["sh"], c["N"], c["hq"], c["hkv"], c["d"], c["P"]
    dv = c["dev"]
    flops_fwd, flops_bwd = attn_flops(c)
    stream = torch.cuda.current_stream(device)

    # persistent buffers (allocation outside the timed region)
    tree = tt.tree_build(dv["par"], dv["len"])
    O = torch.empty_like(dv["Q"])
    LSE = torch.empty(hq, N, dtype=torch.float32, device=device)
    dQ, dK, dV = torch.empty_like(dv["Q"]), torch.empty_like(dv["K"]), torch.empty_like(dv["V"])
    bws = torch.empty(tt.lib().tt_tree_attn_bwd_workspace_bytes(N, hq), dtype=torch.uint8, device=device)
    dws = torch.empty(tt.dta_workspace_bytes(sh.seg_parent, sh.seg_len, CHUNK, hq, hkv, d), dtype=torch.uint8,
                      device=device)
    dta_out = (torch.empty_like(O), torch.empty_like(LSE), torch.empty_like(dQ), torch.empty_like(dK),
               torch.empty_like(dV))
    # the path-at-a-time pass as a captured plan (host traversal once, one graph launch per step)
    dta_plan = tt.DtaPlan(sh.seg_parent, sh.seg_len, dv["Q"], dv["K"], dv["V"], dv["dO"], chunk=CHUNK, ws=dws,
                          out=dta_out, err=None) if do_attn else None
    err = tt.new_err(device)
    if do_lp:
        lp_tree = tt.tree_build(lpc["par"], lpc["len"]).check()
        w = lp_tree.tok_weight[:lpc["n"]].contiguous()
        logp = torch.empty(lpc["n"], dtype=torch.float32, device=device)
        loss = torch.empty(1, dtype=torch.float64, device=device)
        dl = torch.empty_like(lpc["logits"])
        lp_bytes = 4.0 * lpc["n"] * lpc["V"] + 12.0 * lpc["n"]
    torch.cuda.synchronize(device)
    tree.check()

    names = ["tree_build", "attn_fwd", "attn_bwd", "dta_chunk", "logprob"]

    def step(ev, plan=True):
        ev[0].record(stream)
        t = tt.tree_build(dv["par"], dv["len"], N=N, err=err)
        ev[1].record(stream)
        if do_attn:
            tt.tree_attn_fwd(t, dv["Q"], dv["K"], dv["V"], out=(O, LSE), err=err)
        ev[2].record(stream)
        if do_attn:
            tt.tree_attn_bwd(t, dv["Q"], dv["K"], dv["V"], O, LSE, dv["dO"], out=(dQ, dK, dV), ws=bws, err=err)
        ev[3].record(stream)
        if do_attn and plan:
            dta_plan.launch()
        elif do_attn:
            tt.dta_tree_attn(sh.seg_parent, sh.seg_len, dv["Q"], dv["K"], dv["V"], dv["dO"], chunk=CHUNK, err=err,
                             ws=dws, out=dta_out)
        ev[4].record(stream)
        if do_lp:
            tt.weighted_logprob(lpc["logits"], lpc["targets"], w, out=(logp, loss, dl), err=err)
        ev[5].record(stream)
        return t

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    evs = [mk() for _ in range(args.steps)]
    # the clock sampler starts with the warm-up, so that its first samples
    # (nvidia-smi takes a while to start) fall inside the timed steps
    with ClockSampler(local) as clocks:
        for _ in range(args.warmup):
            step(mk())
        torch.cuda.synchronize(device)
        tt.check_err(err, "warm-up")
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(evs[i])
        torch.cuda.synchronize(device)
        t1 = time.perf_counter()
        wall = t1 - t0
        clocks.timed(t0, t1)
    barrier(world)
    tt.check_err(err, "timed steps")
    per = {n: [] for n in names}
    for ev in evs:
        for j, n in enumerate(names):
            per[n].append(ev[j].elapsed_time(ev[j + 1]))
    mean = {n: sum(v) / len(v) for n, v in per.items()}
    step_ms = sum(mean.values())
    attn_ms = mean["attn_fwd"] + mean["attn_bwd"]
    # whole-job numbers: max time over ranks, work of all ranks
    attn_ms_max = max_over_ranks(attn_ms, world, device)
    step_ms_max = max_over_ranks(step_ms, world, device)
    tflops = world * (flops_fwd + flops_bwd) / max(attn_ms_max * 1e-3, 1e-12) / 1e12
    fwd_tflops = flops_fwd / max(mean["attn_fwd"] * 1e-3, 1e-12) / 1e12
    bwd_tflops = flops_bwd / max(mean["attn_bwd"] * 1e-3, 1e-12) / 1e12
    dta_tflops = (flops_fwd + flops_bwd) / max(mean["dta_chunk"] * 1e-3, 1e-12) / 1e12

    # Device time per kernel class, from CUDA events the library records on
    # each launch's own stream (tt_kernel_timing), over a second run of the
    # same steps; the dominant class is the one with the most time per step.
    # (the path-at-a-time pass by the direct call here: the launches of a
    # captured plan carry no per-launch events)
    tt.kernel_timing(True)
    for _ in range(args.steps):
        step(mk(), plan=False)
    torch.cuda.synchronize(device)
    tt.kernel_timing(False)
    kt, kt_dropped = tt.kernel_timing_read()
    tt.check_err(err, "kernel timing steps")
    if do_attn:
        tt.check_err(dta_plan.err, "path-at-a-time plan")
    kt_ms = {k: kt[k][0] / args.steps for k in tt.KERNEL_CLASSES}
    kt_launches = {k: kt[k][1] / args.steps for k in tt.KERNEL_CLASSES}
    # Algorithmic work per step of each class: the whole-tree call and the
    # path-at-a-time chunks each cover the P ancestor pairs once. Forward:
    # S and P·V (4·d·Hq per pair); backward kernel (dK/dV and dQ CTAs in one
    # launch): S, dP, dV, dK, dQ (10: the S and dP its dQ CTAs form again are
    # counted once); log-prob 4·N·V + 12·N bytes. Masked and skipped work is
    # not credited.
    n_calls = 2 if do_attn else 0
    kt_work = {"fwd": n_calls * 4.0 * d * hq * P, "bwd": n_calls * 10.0 * d * hq * P,
               "logprob": lp_bytes if do_lp else 0.0, "lmhead": 0.0}
    dom = max(tt.KERNEL_CLASSES, key=lambda k: kt_ms[k])
    dom_names = {"fwd": "fwd_tc_kernel", "bwd": "bwd_tc_kernel (dK/dV and dQ CTAs)", "logprob": "wlp_cluster_kernel",
                 "lmhead": "lmhead_fwd_kernel"}
    lp_traffic = (round(LP_TRAFFIC_PER_ROW * lpc["n"]) if do_lp and lpc["V"] == LP_TRAFFIC_VOCAB else None)
    per_launch_ms = kt_ms[dom] / max(kt_launches[dom], 1e-12)
    per_launch_work = kt_work[dom] / max(kt_launches[dom], 1e-12)
    if dom == "logprob":
        achieved = per_launch_work / max(per_launch_ms * 1e-3, 1e-12) / 1e9
        roofline = {"bound": "hbm", "kernel": dom_names[dom], "achieved": round(achieved, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": lp_traffic,
                    "algorithmic_bytes": round(per_launch_work)}
    else:
        achieved = per_launch_work / max(per_launch_ms * 1e-3, 1e-12) / 1e12
        # The class mixes the whole-tree launch with the path-at-a-time chunk
        # launches; ncu bytes exist for the whole-tree launch only (see
        # attention_roofline), so the class's per-launch traffic is not given.
        roofline = {"bound": "tensor", "kernel": dom_names[dom], "achieved": round(achieved, 2), "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": round(achieved / bf16_peak, 4), "traffic": None,
                    "traffic_note": "ncu DRAM bytes are for the whole-tree launch only: attention_roofline",
                    "algorithmic_flops": round(per_launch_work)}
    roofline.update({"launches_per_step": kt_launches[dom], "ms_per_launch": round(per_launch_ms, 4),
                     "peak_source": peak_src + (" burst" if dom != "logprob" else ""),
                     "timing": "CUDA events around each launch on its stream"})
    kernel_times = {}
    for k in tt.KERNEL_CLASSES:
        e = {"ms_per_step": round(kt_ms[k], 4), "launches_per_step": kt_launches[k]}
        if kt_ms[k] > 0 and kt_work[k] > 0:
            if k == "logprob":
                e["gbs"] = round(kt_work[k] / (kt_ms[k] * 1e-3) / 1e9, 1)
                e["frac"] = round(e["gbs"] / hbm_peak, 4)
            else:
                e["tflops"] = round(kt_work[k] / (kt_ms[k] * 1e-3) / 1e12, 2)
                e["frac"] = round(e["tflops"] / bf16_peak, 4)
        kernel_times[k] = e
    res = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD if args.workload == HEADLINE else SIDE_WORKLOADS[args.workload],
                   "tokens": N, "pairs": P, "heads": [hq, hkv, d], "chunk": CHUNK,
                   "vocab": lpc["V"] if do_lp else None, "logprob_rows": lpc["n"] if do_lp else None,
                   "parallelism": f"replicas{world}",
                   "l2": "inputs > L2: the 7.7 GB log-prob stage streams between attention passes"},
        "value_fraction_of_peak": round(tflops / world / bf16_peak, 4),
        "peaks": {"bf16_burst_tflops": bf16_peak, "bf16_sustained_tflops": bf16_sus, "hbm_gbs": hbm_peak,
                  "source": peak_src, "fractions_use": "burst bf16 (steps run well under a second)"},
        "parts_ms": {n: round(mean[n], 4) for n in names},
        "attn_tflops": {"fwd": round(fwd_tflops, 2), "bwd": round(bwd_tflops, 2),
                        "fwd_frac": round(fwd_tflops / bf16_peak, 4), "bwd_frac": round(bwd_tflops / bf16_peak, 4),
                        "dta_chunk_fwd_bwd": round(dta_tflops, 2), "dta_chunk_frac": round(dta_tflops / bf16_peak, 4)},
        "tokens_per_s": round(N / (attn_ms * 1e-3)),
        "branch_tokens_per_s": round(c["branch_tokens"] / (attn_ms * 1e-3)),
        "roofline": roofline,
        "kernel_ms_per_step": kernel_times,
        "kernel_timing_dropped": kt_dropped,
        "attention_roofline": {
            "fwd_tc_kernel (whole-tree launch)": {"bound": "tensor", "achieved": round(fwd_tflops, 2), "unit": "TFLOP/s",
                              "peak": bf16_peak, "frac": round(fwd_tflops / bf16_peak, 4),
                              "traffic": ATTN_TRAFFIC.get(args.workload, {}).get("fwd")},
            "tt_tree_attn_bwd (prep_kernel + bwd_tc_kernel)": {
                "bound": "tensor", "achieved": round(bwd_tflops, 2), "unit": "TFLOP/s", "peak": bf16_peak,
                "frac": round(bwd_tflops / bf16_peak, 4), "traffic": ATTN_TRAFFIC.get(args.workload, {}).get("bwd")}},
        "gpu_launches": args.steps * ((6 + 1 + 2 + dta_launches(sh.seg_parent, sh.seg_len, CHUNK)) if do_attn else 6)
        # the log-prob call: its cluster kernel (and the row kernel on the SMs the clusters leave idle, counted by
        # the launch-timing pass) and the loss kernel
        + args.steps * ((round(kt_launches["logprob"]) + 1) if do_lp else 0),
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if do_lp:
        lp_gbs = world * lp_bytes / max(max_over_ranks(mean["logprob"], world, device) * 1e-3, 1e-12) / 1e9
        res["logprob"] = {"value": round(lp_gbs, 1), "unit": "GB/s", "ms": round(mean["logprob"], 4),
                          "frac": round(lp_gbs / world / hbm_peak, 4), "peak": hbm_peak, "peak_source": peak_src,
                          "workload": "weighted log-prob, logits [12669, 151936] bf16 (Qwen3-1.7B-shaped tree)"}
        res["logprob_roofline"] = {"bound": "hbm", "kernel": "wlp_cluster_kernel (tt_weighted_logprob call)",
                                   "achieved": round(lp_gbs / world, 1), "peak": hbm_peak, "unit": "GB/s",
                                   "frac": round(lp_gbs / world / hbm_peak, 4), "traffic": lp_traffic,
                                   "algorithmic_bytes": round(lp_bytes)}
    res["trie_build"] = time_trie_build(tt, sh.seg_parent, sh.seg_len)
    if args.stage != "all":
        res["config"]["stage"] = args.stage
    if not args.no_e2e and args.stage == "all":
        res["e2e"] = e2e_tt(args, tt, c, device, flops_fwd + flops_bwd, world)
    if not args.no_side and args.stage == "all" and args.workload == HEADLINE:
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        side = {}
        for wid, desc in SIDE_WORKLOADS.items():
            sc = attention_case(wid, device)
            side[str(wid)] = dict(workload=desc, **time_side_workload(tt, sc, device, flush, bf16_peak))
            del sc
        side["3_path_at_a_time_4096"] = dict(
            workload="headline tree, path-at-a-time pass with 4096-query chunks",
            **time_side_workload(tt, c, device, flush, bf16_peak, dta_chunk=CHUNK_VARIANT))
        side["3_path_at_a_time_2048"] = dict(
            workload="headline tree, path-at-a-time pass with 2048-query chunks (as in the steps)",
            **time_side_workload(tt, c, device, flush, bf16_peak, dta_chunk=CHUNK))
        side["3_whole_tree"] = dict(workload="headline tree, whole-tree fwd+bwd timed alone",
                                    **time_side_workload(tt, c, device, flush, bf16_peak))
        side["2_lmhead"] = time_lmhead(tt, device, flush, bf16_peak)
        res["workloads"] = side
    return res


def e2e_tt(args, tt, c, device, flops, world):
    """Same metric through the public API with host (pinned) inputs and outputs; copies are timed.

    The timed loop runs the way a training loop feeds a GPU: each step uploads its own inputs (tree arrays, Q, K, V,
    dO) from pinned host memory and downloads its own gradients (dQ, dK, dV), on two copy streams, so that step i+1's
    upload and step i-1's download overlap step i's compute. Inputs are double-buffered: an upload starts only after
    the compute two steps back is done, so at most two steps' inputs are resident. `serial` is the same steps with
    no overlap across steps (a step's copies start after the previous step's work)."""
    import torch
    host = c["host"]
    N = c["N"]
    outs = [torch.empty(host[k].shape, dtype=torch.bfloat16).pin_memory() for k in ("Q", "K", "V")]
    keys = ("par", "len", "Q", "K", "V", "dO")
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = sum(o.numel() * o.element_size() for o in outs)
    cur = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def upload(after):
        # one step's inputs on the upload stream, once `after` (the compute that last used the other buffer) is done
        if after is not None:
            up.wait_event(after)
        with torch.cuda.stream(up):
            dv = {k: host[k].to(device, non_blocking=True) for k in keys}
            ready = torch.cuda.Event()
            ready.record(up)
        return dv, ready

    def compute(dv, ready):
        # tree build, forward, backward on the compute stream; the gradients go home on the download stream
        cur.wait_event(ready)
        for x in dv.values():
            x.record_stream(cur)
        t = tt.tree_build(dv["par"], dv["len"], N=N)
        O, LSE = tt.tree_attn_fwd(t, dv["Q"], dv["K"], dv["V"])
        g = tt.tree_attn_bwd(t, dv["Q"], dv["K"], dv["V"], O, LSE, dv["dO"])
        done = torch.cuda.Event()
        done.record(cur)
        down.wait_event(done)
        with torch.cuda.stream(down):
            for o, x in zip(outs, g):
                x.record_stream(down)
                o.copy_(x, non_blocking=True)
        return done

    def pipelined(steps):
        up.wait_stream(cur)
        done = [None, None]
        nxt = upload(None)
        for i in range(steps):
            if done[i % 2] is not None:
                done[i % 2].synchronize()  # the host stays two steps ahead, so the allocator's pool stays warm
            this = nxt
            if i + 1 < steps:
                nxt = upload(done[(i + 1) % 2])
            done[i % 2] = compute(*this)
        cur.wait_stream(down)

    def serial(steps):
        for _ in range(steps):
            up.wait_stream(cur)
            compute(*upload(None))
            cur.wait_stream(down)

    def timed(run):
        run(max(3, args.warmup))
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(cur)
        run(args.steps)
        e1.record(cur)
        torch.cuda.synchronize(device)
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)

    ms = timed(pipelined)
    ms_serial = timed(serial)
    rate = lambda t: round(world * flops / (t * 1e-3) / 1e12, 3)
    return {"value": rate(ms), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "serial": {"value": rate(ms_serial), "ms_per_step": round(ms_serial, 4),
                       "scope": "the same steps with no overlap across steps"},
            "scope": "headline tree: every step uploads its tree arrays, Q, K, V and dO from pinned host memory, runs "
                     "tree build -> attention fwd -> bwd, and downloads dQ, dK, dV; uploads and downloads run on two "
                     "copy streams beside the compute (step i+1's upload and step i-1's download during step i, inputs "
                     "double-buffered); the first upload and the last download are inside the timed region (the "
                     "attention metric only; the log-prob stage is not in this number)"}


# ----------------------------------------------------------------------------- CPU oracle
# Bounded sample of the headline tree for the CPU oracle: one query head (its
# KV head 0), forward + backward of the rows of 10 segments (the root, its
# first child and that child's 8 leaves), each against its root path, by the
# fp64 oracle's causal attention; plus the fp64 weighted log-prob of 32 rows.
ORACLE_SEGMENTS = [0, 1] + list(range(9, 17))
ORACLE_SAMPLE = ("one query head of the Qwen3-8B-shaped tree: fp64 forward+backward of the rows of segments "
                 "0, 1, 9..16 (root, first child, its 8 leaves) against their root paths, plus the fp64 weighted "
                 "log-prob of 32 rows at V=151936")


def oracle_sample_code(steps, warmup, wid, segments):
    return f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import synth
from oracle import attention as A, logprob as L, tree as T
att = synth.attention_inputs({wid})
lp = synth.logprob_inputs(2)
sh = att["tree"]
f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
Q, K, V, dO = (f(att[k][:, :1]) for k in ("Q", "K", "V", "dO"))
z = f(lp["logits"][:32])
segs = {segments!r}
times = []
for i in range({warmup} + {steps}):
    t0 = time.perf_counter()
    tab = T.tables(sh.seg_parent, sh.seg_len)
    if segs is None:
        A.tree_attention_segments(tab, Q, K, V, dO)
    else:
        sc = 1.0 / np.sqrt(Q.shape[2])
        for s in segs:
            path = np.concatenate([np.arange(tab.seg_start[a], tab.seg_end[a])
                                   for a in T.segment_path(tab.seg_parent, s)])
            rows = np.arange(tab.seg_start[s], tab.seg_end[s])
            A.causal_attention_forward(Q[rows], K[path], V[path], sc)
            A.causal_attention_backward(Q[rows], K[path], V[path], dO[rows], sc)
    L.weighted_token_loss(z, lp["targets"][:32], tab.tok_weight[:32])
    if i >= {warmup}:
        times.append(time.perf_counter() - t0)
print(json.dumps({{"times": times}}))
"""


def run_oracle(steps, warmup, wid=HEADLINE, segments=ORACLE_SEGMENTS):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(CPU_ORACLE_THREADS)
    r = subprocess.run([sys.executable, "-c", oracle_sample_code(steps, warmup, wid, segments)], env=env,
                       capture_output=True, text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["times"]


def oracle_flops(wid=HEADLINE, segments=ORACLE_SEGMENTS):
    """Useful fwd+bwd flops of one head over the sampled segments' rows (all rows if segments is None)."""
    import synth
    sh = synth.tree_shape(wid)
    d = synth.HEADS[wid][2]
    if segments is None:
        return 14.0 * d * useful_pairs(sh.seg_parent, sh.seg_len)
    pl = [0] * sh.S
    for s in range(1, sh.S):
        pl[s] = pl[sh.seg_parent[s]] + int(sh.seg_len[sh.seg_parent[s]])
    pairs = sum(int(sh.seg_len[s]) * pl[s] + int(sh.seg_len[s]) * (int(sh.seg_len[s]) + 1) // 2 for s in segments)
    return 14.0 * d * pairs


LMHEAD_ORACLE_CODE = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import synth
from oracle import lmhead as LH
d = synth.lmhead_inputs(0, vocab={LMHEAD['vocab']}, hidden={LMHEAD['hidden']})
f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
rows = np.arange({LMHEAD_ORACLE_ROWS})
t0 = time.perf_counter()
LH.lmhead_rows(f(d["H"][rows]), d["W"], d["targets"][rows], rows, widen=f)
print(json.dumps({{"seconds": time.perf_counter() - t0}}))
"""


def lmhead_cpu_baseline():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(CPU_ORACLE_THREADS)
    r = subprocess.run([sys.executable, "-c", LMHEAD_ORACLE_CODE], env=env, capture_output=True, text=True,
                       timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("LM-head oracle sample failed:\n" + r.stderr[-2000:])
    t = json.loads(r.stdout.strip().splitlines()[-1])["seconds"]
    flops = 2.0 * LMHEAD_ORACLE_ROWS * LMHEAD["vocab"] * LMHEAD["hidden"]
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "seconds": round(t, 3),
            "sample": f"fp64 LM head + log-sum-exp of {LMHEAD_ORACLE_ROWS} rows over the whole vocabulary "
                      "(W widened chunk by chunk)"}


def cpu_baseline():
    t = run_oracle(1, 0)[0]
    out = {"value": round(oracle_flops() / t / 1e12, 6), "unit": "TFLOP/s", "cores": CPU_ORACLE_THREADS,
           "kind": "oracle", "sample": ORACLE_SAMPLE, "seconds": round(t, 3), "workloads": {}}
    for wid in (0, 1, 4):
        tw = run_oracle(1, 0, wid, None)[0]
        out["workloads"][str(wid)] = {"value": round(oracle_flops(wid, None) / tw / 1e12, 6), "unit": "TFLOP/s",
                                      "seconds": round(tw, 3), "sample": "one query head, every row of the tree, "
                                      "fp64 forward+backward (+ 32 log-prob rows)"}
    out["workloads"]["2_lmhead"] = lmhead_cpu_baseline()
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    times = run_oracle(args.steps, args.warmup)
    t = sum(times) / len(times)
    v = oracle_flops() / t / 1e12
    return {"metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "parallelism": "cpu-oracle"},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": CPU_ORACLE_THREADS, "kind": "oracle",
                             "sample": ORACLE_SAMPLE},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_lmhead_stage(args, local):
    """Profiling aid: only the fused LM-head call, --warmup + --steps iterations."""
    import torch

    import prefix_tree_gb300 as tt
    from prefix_tree_gb300 import build as _b
    _b.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    _, bf16_peak, _, _ = peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    r = time_lmhead(tt, device, flush, bf16_peak, iters=args.steps, warmup=args.warmup)
    return dict(r, stage="lmhead")


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.stage == "lmhead":
        if rank == 0:
            print(json.dumps(run_lmhead_stage(args, local)), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    # CPU baseline first, in a fresh subprocess (no fork after CUDA initialisation)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()
    res = run_tt(args, rank, world, local)
    if rank == 0:
        if cpu is not None:
            res["cpu_baseline"] = cpu
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
