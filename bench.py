"""Benchmark of the prefix-tree training hot path on one GB300 (or N replicas).

One step = one pass of every hot-path stage over the Qwen3-1.7B-shaped rollout
tree (2048-token prompt, 4 x 4 branches, 12,669 unique tokens, 16/8 heads,
d=128):
  tree build -> tree attention forward -> tree attention backward ->
  path-at-a-time (2048-query chunk) forward+backward of the same tree ->
  weighted log-prob + loss + dlogits over logits [12669, 151936] bf16.
Inputs are synthetic, seeded and resident in HBM before timing.

value = useful tree-attention TFLOP/s of the whole-tree forward+backward
(only ancestor pairs count: 14·d·Hq·pairs per step); the log-prob stage is
reported as HBM GB/s (4·N·V + 12·N algorithmic bytes). `roofline` is for the
kernel class with the most device time per step, timed by CUDA events the
library records around each of its launches on the launch's own stream
(tt_kernel_timing) over a second run of the same steps; its algorithmic work
per launch is the step's work of that class (forward 4, dQ 6, dK/dV 8 flops
per ancestor pair per d·Hq, for the whole-tree call and the path-at-a-time
chunks; log-prob bytes as above) over the class's launches. Timing: CUDA events on
the launching stream, W warm-up steps, K timed steps bracketed by barrier +
synchronize. L2: the log-prob stage streams 7.7 GB (>> 129 MB L2) between
consecutive attention passes, and its own inputs exceed L2.

--impl reference times the CPU oracle (the reference arm of this build) on a
bounded sample of the same workload, on the host cores.
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
WORKLOAD = ("Qwen3-1.7B-shaped tree attention (Hq=16, Hkv=8, d=128; 2048-token root, 4x4 branches U[256,768], "
            "N=12669, 16 leaves, 3.94x compression) + weighted log-prob over its tokens at V=151936 (seed 0)")
CPU_ORACLE_THREADS = os.cpu_count() or 1
# DRAM bytes (read + write) per launch measured by ncu on this build's kernels:
# log-prob at V = 151936 per row (2048-row launch: 623.3 MB read + 562.2 MB
# written), tree-attention forward and backward (dq + dkdv) on the workload.
LP_TRAFFIC_VOCAB = 151936
LP_TRAFFIC_PER_ROW = (623346176 + 562226176) / 2048
ATTN_FWD_TRAFFIC = 109455616 + 23435264
ATTN_BWD_TRAFFIC = 168829696 + 31970816 + 260049408 + 29090816
# DRAM bytes (read + written) per step of each attention kernel class over
# all of its launches in a step (whole-tree call and path-at-a-time chunks),
# from an ncu capture of one step; None where not captured for these kernels.
KT_TRAFFIC_PER_STEP = {"fwd": 441414400, "dq": 559690496, "dkdv": 1157959424}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tt", choices=["tt", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stage", default="all", choices=["all", "attn", "logprob"],
                    help="profiling aid: run only the attention stages or only the log-prob stage")
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
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs") or p.get("hbm_GBs")
        bf = p.get("bf16_tflops_sustained") or p.get("bf16_tflops")
        if hbm and bf:
            return float(hbm), float(bf), "measured"
    return 6800.0, 1900.0, "fallback"


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
        sm, mx, reasons = [], [], set()
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
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload
def make_workload(device, stage="all", lp_rows=0):
    import numpy as np
    import torch

    import synth
    att = synth.attention_inputs(1)
    if stage == "attn":
        lp = dict(logits=np.zeros((1, 8), np.uint16), targets=np.zeros(1, np.int32), V=8)
    else:
        lp = synth.logprob_inputs(2)
        if lp_rows:
            lp = dict(lp, logits=lp["logits"][:lp_rows], targets=lp["targets"][:lp_rows])
    sh = att["tree"]

    def bf(bits, pin=False):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory() if pin else t.to(device)

    host = dict(Q=bf(att["Q"], True), K=bf(att["K"], True), V=bf(att["V"], True), dO=bf(att["dO"], True),
                logits=bf(lp["logits"], True), par=torch.tensor(sh.seg_parent).pin_memory(),
                len=torch.tensor(sh.seg_len).pin_memory(), targets=torch.tensor(lp["targets"]).pin_memory())
    dev = {k: v.to(device, non_blocking=True) for k, v in host.items()}
    torch.cuda.synchronize(device)
    return att, lp, sh, host, dev


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


def dta_launches(seg_len, chunk):
    # per segment: forward chunks (1 kernel each), backward chunks (3 each), one gradient conversion
    return sum(math.ceil(int(L) / chunk) * 4 + 1 for L in seg_len)


# ----------------------------------------------------------------------------- GPU arm
def run_tt(args, rank, world, local):
    import torch

    import prefix_tree_gb300 as tt
    from prefix_tree_gb300 import build as _b
    _b.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    att, lp, sh, host, dev = make_workload(device, args.stage, args.lp_rows)
    N, hq, hkv, d = att["tree"].N, att["hq"], att["hkv"], att["d"]
    V = lp["V"]
    n_lp = dev["logits"].shape[0]
    w_lp = None
    P = useful_pairs(sh.seg_parent, sh.seg_len)
    flops_fwd, flops_bwd = 4.0 * d * hq * P, 10.0 * d * hq * P
    lp_bytes = 4.0 * n_lp * V + 12.0 * n_lp
    chunk = 2048
    stream = torch.cuda.current_stream(device)

    # persistent buffers (allocation outside the timed region)
    tree = tt.tree_build(dev["par"], dev["len"])
    torch.cuda.synchronize(device)
    w = tree.tok_weight[:n_lp].contiguous() if args.stage != "attn" else None
    O = torch.empty_like(dev["Q"])
    LSE = torch.empty(hq, N, dtype=torch.float32, device=device)
    dQ, dK, dV = torch.empty_like(dev["Q"]), torch.empty_like(dev["K"]), torch.empty_like(dev["V"])
    bws = torch.empty(tt.lib().tt_tree_attn_bwd_workspace_bytes(N, hq), dtype=torch.uint8, device=device)
    logp = torch.empty(n_lp, dtype=torch.float32, device=device)
    loss = torch.empty(1, dtype=torch.float64, device=device)
    dl = torch.empty_like(dev["logits"])
    err = tt.new_err(device)

    names = ["tree_build", "attn_fwd", "attn_bwd", "dta_chunk", "logprob"]

    do_attn, do_lp = args.stage in ("all", "attn"), args.stage in ("all", "logprob")

    def step(ev):
        ev[0].record(stream)
        t = tt.tree_build(dev["par"], dev["len"], N=N, err=err)
        ev[1].record(stream)
        if do_attn:
            tt.tree_attn_fwd(t, dev["Q"], dev["K"], dev["V"], out=(O, LSE), err=err)
        ev[2].record(stream)
        if do_attn:
            tt.tree_attn_bwd(t, dev["Q"], dev["K"], dev["V"], O, LSE, dev["dO"], out=(dQ, dK, dV), ws=bws, err=err)
        ev[3].record(stream)
        if do_attn:
            tt.dta_tree_attn(sh.seg_parent, sh.seg_len, dev["Q"], dev["K"], dev["V"], dev["dO"], chunk=chunk,
                             err=err)
        ev[4].record(stream)
        if do_lp:
            tt.weighted_logprob(dev["logits"], dev["targets"], w, out=(logp, loss, dl), err=err)
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
    lp_ms_max = max_over_ranks(mean["logprob"], world, device)
    tflops = world * (flops_fwd + flops_bwd) / max(attn_ms_max * 1e-3, 1e-12) / 1e12
    lp_gbs = world * lp_bytes / max(lp_ms_max * 1e-3, 1e-12) / 1e9
    hbm_peak, bf16_peak, peak_src = peaks()

    bwd_tflops = flops_bwd / max(mean["attn_bwd"] * 1e-3, 1e-12) / 1e12
    fwd_tflops = flops_fwd / max(mean["attn_fwd"] * 1e-3, 1e-12) / 1e12
    lp_traffic = round(LP_TRAFFIC_PER_ROW * n_lp) if do_lp and V == LP_TRAFFIC_VOCAB and LP_TRAFFIC_PER_ROW else None

    # Device time per kernel class, from CUDA events the library records on
    # each launch's own stream (tt_kernel_timing), over a second run of the
    # same steps; the dominant class is the one with the most time per step.
    tt.kernel_timing(True)
    for _ in range(args.steps):
        step(mk())
    torch.cuda.synchronize(device)
    tt.kernel_timing(False)
    kt, kt_dropped = tt.kernel_timing_read()
    tt.check_err(err, "kernel timing steps")
    kt_ms = {c: kt[c][0] / args.steps for c in tt.KERNEL_CLASSES}
    kt_launches = {c: kt[c][1] / args.steps for c in tt.KERNEL_CLASSES}
    # Algorithmic work per step of each class: the whole-tree call and the
    # path-at-a-time chunks each cover the P ancestor pairs once; forward
    # S and P·V (4·d·Hq per pair), dQ kernel S, dP, dQ (6), dK/dV kernel
    # Sᵀ, dPᵀ, dV, dK (8: S and dP are formed again, as the forward keeps no
    # P); log-prob 4·N·V + 12·N bytes. Masked and skipped work is not credited.
    n_attn_calls = 2 if do_attn else 0
    kt_work = {"fwd": n_attn_calls * 4.0 * d * hq * P, "dq": n_attn_calls * 6.0 * d * hq * P,
               "dkdv": n_attn_calls * 8.0 * d * hq * P, "logprob": lp_bytes if do_lp else 0.0}
    dom = max(tt.KERNEL_CLASSES, key=lambda c: kt_ms[c])
    dom_names = {"fwd": "fwd_tc_kernel", "dq": "dq_tc_kernel", "dkdv": "dkdv_tc_kernel",
                 "logprob": "wlp_cluster_kernel"}
    per_launch_ms = kt_ms[dom] / max(kt_launches[dom], 1e-12)
    per_launch_work = kt_work[dom] / max(kt_launches[dom], 1e-12)
    if dom == "logprob":
        achieved = per_launch_work / max(per_launch_ms * 1e-3, 1e-12) / 1e9
        roofline = {"bound": "hbm", "kernel": dom_names[dom], "achieved": round(achieved, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": lp_traffic,
                    "algorithmic_bytes": round(per_launch_work)}
    else:
        achieved = per_launch_work / max(per_launch_ms * 1e-3, 1e-12) / 1e12
        tr = KT_TRAFFIC_PER_STEP.get(dom) if do_attn and args.stage == "all" else None
        roofline = {"bound": "tensor", "kernel": dom_names[dom], "achieved": round(achieved, 2), "peak": bf16_peak,
                    "unit": "TFLOP/s", "frac": round(achieved / bf16_peak, 4),
                    "traffic": None if tr is None else round(tr / max(kt_launches[dom], 1e-12)),
                    "algorithmic_flops": round(per_launch_work)}
    roofline.update({"launches_per_step": kt_launches[dom], "ms_per_launch": round(per_launch_ms, 4),
                     "peak_source": peak_src, "timing": "CUDA events around each launch on its stream"})
    kernel_times = {c: {"ms_per_step": round(kt_ms[c], 4), "launches_per_step": kt_launches[c]}
                    for c in tt.KERNEL_CLASSES}
    attn_roofline = {
        "fwd_tc_kernel": {"bound": "tensor", "achieved": round(fwd_tflops, 2), "unit": "TFLOP/s",
                          "peak": bf16_peak, "frac": round(fwd_tflops / bf16_peak, 4),
                          "traffic": ATTN_FWD_TRAFFIC},
        "tt_tree_attn_bwd (prep + dq_tc_kernel + dkdv_tc_kernel)": {
            "bound": "tensor", "achieved": round(bwd_tflops, 2), "unit": "TFLOP/s", "peak": bf16_peak,
            "frac": round(bwd_tflops / bf16_peak, 4), "traffic": ATTN_BWD_TRAFFIC},
    }
    parts = {n: round(mean[n], 4) for n in names}
    res = {
        "metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": N, "pairs": P, "heads": [hq, hkv, d], "vocab": V,
                   "chunk": chunk, "parallelism": f"replicas{world}",
                   "l2": "inputs > L2: the 7.7 GB log-prob stage streams between attention passes"},
        "value_fraction_of_peak": round(tflops / world / bf16_peak, 4),
        "logprob": {"value": round(lp_gbs, 1), "unit": "GB/s", "ms": round(mean["logprob"], 4),
                    "frac": round(lp_gbs / world / hbm_peak, 4), "peak": hbm_peak, "peak_source": peak_src},
        "parts_ms": parts,
        "attn_tflops": {"fwd": round(flops_fwd / max(mean["attn_fwd"] * 1e-3, 1e-12) / 1e12, 2),
                        "bwd": round(bwd_tflops, 2),
                        "dta_chunk_fwd_bwd": round((flops_fwd + flops_bwd) / max(mean["dta_chunk"] * 1e-3, 1e-12)
                                                   / 1e12, 2)},
        "roofline": roofline,
        "kernel_ms_per_step": kernel_times,
        "kernel_timing_dropped": kt_dropped,
        "logprob_roofline": {"bound": "hbm", "kernel": "wlp_cluster_kernel (tt_weighted_logprob call)",
                             "achieved": round(lp_gbs / world, 1), "peak": hbm_peak, "unit": "GB/s",
                             "frac": round(lp_gbs / world / hbm_peak, 4), "traffic": lp_traffic,
                             "algorithmic_bytes": round(lp_bytes)},
        "attention_roofline": attn_roofline,
        "gpu_launches": args.steps * (6 + 1 + 3 + dta_launches(sh.seg_len, chunk) + 2),
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
    }
    res["trie_build"] = time_trie_build(tt, sh.seg_parent, sh.seg_len)
    if args.stage != "all":
        res["config"]["stage"] = args.stage
        res["config"]["lp_rows"] = n_lp
    if not args.no_e2e and args.stage == "all":
        res["e2e"] = e2e_tt(args, tt, host, device, hq, flops_fwd + flops_bwd, world)
    return res


def e2e_tt(args, tt, host, device, hq, flops, world):
    """Same metric through the public API with host (pinned) inputs and outputs; copies are timed."""
    import torch
    N = host["Q"].shape[0]
    outs = [torch.empty(host[k].shape, dtype=torch.bfloat16).pin_memory() for k in ("Q", "K", "V")]
    keys = ("par", "len", "Q", "K", "V", "dO")
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = sum(o.numel() * o.element_size() for o in outs)

    def one():
        dv = {k: host[k].to(device, non_blocking=True) for k in keys}
        t = tt.tree_build(dv["par"], dv["len"], N=N)
        O, LSE = tt.tree_attn_fwd(t, dv["Q"], dv["K"], dv["V"])
        g = tt.tree_attn_bwd(t, dv["Q"], dv["K"], dv["V"], O, LSE, dv["dO"])
        for o, x in zip(outs, g):
            o.copy_(x, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record()
    for _ in range(args.steps):
        one()
    e1.record()
    torch.cuda.synchronize(device)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ----------------------------------------------------------------------------- CPU oracle
ORACLE_SAMPLE = ("one query head (h=0, its KV head 0) of the whole-tree attention forward+backward over all 12669 "
                 "tokens by the per-segment fp64 oracle, plus the fp64 weighted log-prob of 32 rows")


def oracle_sample_code(steps, warmup):
    return f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
import synth
from oracle import attention as A, logprob as L, tree as T
att = synth.attention_inputs(1)
lp = synth.logprob_inputs(2)
sh = att["tree"]
f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
Q, K, V, dO = (f(att[k][:, :1]) for k in ("Q", "K", "V", "dO"))
z = f(lp["logits"][:32])
times = []
for i in range({warmup} + {steps}):
    t0 = time.perf_counter()
    tab = T.tables(sh.seg_parent, sh.seg_len)
    A.tree_attention_segments(tab, Q, K, V, dO)
    L.weighted_token_loss(z, lp["targets"][:32], tab.tok_weight[:32])
    if i >= {warmup}:
        times.append(time.perf_counter() - t0)
print(json.dumps({{"times": times}}))
"""


def run_oracle(steps, warmup):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(CPU_ORACLE_THREADS)
    r = subprocess.run([sys.executable, "-c", oracle_sample_code(steps, warmup)], env=env, capture_output=True,
                       text=True, timeout=3600)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["times"]


def oracle_flops():
    import synth
    sh = synth.tree_shape(1)
    return 14.0 * 128 * 1 * useful_pairs(sh.seg_parent, sh.seg_len)


def cpu_baseline():
    times = run_oracle(1, 0)
    t = times[0]
    return {"value": round(oracle_flops() / t / 1e12, 6), "unit": "TFLOP/s", "cores": CPU_ORACLE_THREADS,
            "kind": "oracle", "sample": ORACLE_SAMPLE, "seconds": round(t, 3)}


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


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
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
