#!/usr/bin/env python
"""Benchmark: prefix-tree attention forward + backward on GB300.

One step = one pass of the whole hot path over one synthetic tree: the forward
kernel, then the backward's three stages.  The default workload is the largest
one, the long shared context (a 32,768-token prefix with 64 branches of 1-3
segments of log-uniform length in [1024, 8192]; 64 query heads, 8 kv heads,
head_dim 128, bf16; about 480k compact tokens).  The metric is useful TFLOP/s,
counting only attended (ancestor) pairs: 4*d per pair and q-head forward, 10*d
backward.  The same line also carries the smaller workloads (tiny binary tree,
GRPO star, segment tree, agentic tree), each timed the same way.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload.

    python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import math
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-attn fwd+bwd useful TFLOP/s (ancestor pairs) and % of bf16 TC peak, 1 GB300"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 512 << 20          # larger than the 129 MB L2
FALLBACK_BF16_TFLOPS = 1900.0

DESCRIPTIONS = {
    "grpo_star": "GRPO-style star tree: 1024-token prompt + 16 responses U[256,1024]; 32q/8kv heads, d=128",
    "segment_tree": "segment tree: 512-token prompt, 256-token segments, binary x4, early stop + fallback "
                    "to 16 leaves; 32q/8kv heads, d=128",
    "agentic_tree": "irregular agentic tree ~64k compact tokens, 4-6x expansion; 32q/8kv heads, d=128",
    "tiny_binary": "tiny binary tree 64 + 2x32 + 4x32 tokens; 2 heads, d=64",
    "long_context": "long shared context: 32768-token prefix + 64 chains of 1-3 log-U[1k,8k] segments; "
                    "64q/8kv heads, d=128",
    "long_context_4b": "long shared context, first 4 of its 64 branches (58,232 tokens); 48q/6kv heads, d=128 "
                       "(6 GB: the case profiler captures run on; the backward takes the long context's "
                       "chunk and CTA order)",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_context")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-expanded", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="time the named workload only")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU sample")
    ap.add_argument("--extras", action="store_true",
                    help="instead of the step, time the calls around it (tree batching, loss boundary, "
                         "subtree advantages, tree linear attention); one JSON line each")
    ap.add_argument("--extras-small", action="store_true",
                    help="with --extras: GRPO star only and a 32,768-token vocabulary (a few GB on the device, "
                         "for profiler captures)")
    return ap.parse_args()


def useful_flops(pairs: int, hq: int, d: int):
    return 4.0 * d * pairs * hq, 10.0 * d * pairs * hq


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "prefix_tree_attention_attn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (same hash); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[2] == src_hash:
            return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples go to BENCH_OUT_DIR (default: a temporary directory)
        out = os.environ.get("BENCH_OUT_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out, f"clocks_bench_{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the oracle on a bounded sample (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

# Workloads where one kv-group of the full expansion is too large for the host
# (the long shared context: about 1e14 fp64 FLOP per kv-group) take the
# row / key sample; the others take whole kv-groups.
ROW_KEY_SAMPLE = {"long_context", "long_context_4b"}


def oracle_group_step(tree, x, heads, scale, groups):
    """fp64 oracle forward + backward on kv-groups ``groups`` (their q-heads
    and kv-head) of the workload; returns the useful FLOPs it covers."""
    from oracle import attention as OA
    G = heads.group
    pairs = None
    flops = 0.0
    for g in groups:
        qs = slice(g * G, (g + 1) * G)
        q, k, v, do = x["q"][:, qs], x["k"][:, g:g + 1], x["v"][:, g:g + 1], x["do"][:, qs]
        OA.forward(tree.parent, tree.seg_len, q, k, v, scale, check_copies=False)
        OA.backward(tree.parent, tree.seg_len, q, k, v, do, scale)
        if pairs is None:
            from oracle import plan as OP
            pairs = OP.pair_count(tree.parent, tree.seg_len)
        flops += 14.0 * heads.d * pairs * G
    return flops


class RowKeySample:
    """Rows and keys of one tree that the fp64 oracle evaluates one by one, on
    kv-group 0 (q-heads 0..G-1, kv-head 0): O, LSE and dQ of a row over its own
    root-to-node path, and dK, dV of a key near the end of a leaf segment over
    its descendant queries.  Each is credited with its share of a full step's
    useful FLOPs: 10*d per (row, key on its path) pair and q-head (forward 4*d;
    S, dP and dQ of the backward 6*d) and 4*d per (key, descendant query) pair
    and q-head (dV and dK).  Summed over every row and key of the tree these
    shares give the step's 14*d*pairs*hq."""

    ROWS_PER_STEP, KEYS_PER_STEP = 4, 1

    def __init__(self, tree, d, G, seed=0):
        import numpy as np
        from oracle import layout as OL
        self.tree, self.d, self.G = tree, d, G
        order, off, N = OL.packed_layout(tree.parent, tree.seg_len)
        self.N = N
        self.tn = OL.token_nodes(tree.parent, tree.seg_len)
        self.off = off
        ch = OL.children(tree.parent)
        self.above, self.sub_end = {}, {}
        for u in order:
            p = tree.parent[u]
            self.above[u] = 0 if p < 0 else self.above[p] + tree.seg_len[p]
        for u in reversed(order):
            self.sub_end[u] = self.sub_end[ch[u][-1]] if ch[u] else int(off[u]) + tree.seg_len[u]
        self.rng = np.random.default_rng(seed)
        self.leaves = OL.leaves(tree.parent)

    def path_len(self, i):
        u = int(self.tn[i])
        return self.above[u] + (i - int(self.off[u])) + 1

    def descendants(self, j):
        return self.sub_end[int(self.tn[j])] - j

    def draw(self):
        rows = sorted(int(r) for r in self.rng.choice(self.N, size=self.ROWS_PER_STEP, replace=False))
        keys = []
        for l in self.rng.choice(self.leaves, size=self.KEYS_PER_STEP, replace=False):
            end = int(self.off[l]) + self.tree.seg_len[l]
            keys.append(end - 1 - int(self.rng.integers(0, min(8, self.tree.seg_len[l]))))
        return rows, sorted(keys)

    def step(self, xg, scale):
        """One bounded sample: returns the useful FLOPs credited to it."""
        from oracle import attention as OA
        t = self.tree
        rows, keys = self.draw()
        OA.forward_rows(t.parent, t.seg_len, xg["q"], xg["k"], xg["v"], scale, rows)
        OA.backward_rows_dq(t.parent, t.seg_len, xg["q"], xg["k"], xg["v"], xg["do"], scale, rows)
        OA.backward_keys_dkdv(t.parent, t.seg_len, xg["q"], xg["k"], xg["v"], xg["do"], scale, keys)
        return self.d * self.G * (10.0 * sum(self.path_len(i) for i in rows)
                                  + 4.0 * sum(self.descendants(j) for j in keys))

    def describe(self):
        return (f"fp64 oracle on kv-group 0 ({self.G} q-heads, 1 kv-head): per step O, LSE and dQ of "
                f"{self.ROWS_PER_STEP} random rows over their root-to-node paths and dK, dV of "
                f"{self.KEYS_PER_STEP} key(s) near a leaf end, credited 10*d per (row, path key) pair and 4*d per "
                f"(key, descendant) pair per q-head")


def group_slice(x, G):
    """kv-group 0 of a tensor set, on the host (q-heads 0..G-1, kv-head 0)."""
    return {"q": x["q"][:, :G].contiguous().cpu(), "k": x["k"][:, :1].contiguous().cpu(),
            "v": x["v"][:, :1].contiguous().cpu(), "do": x["do"][:, :G].contiguous().cpu()}


def cpu_baseline(name, tree, x, heads, scale, target_s):
    """Time the oracle as it stands until about ``target_s`` seconds have been
    spent: whole kv-groups one at a time, or row / key samples (ROW_KEY_SAMPLE)."""
    t0 = time.perf_counter()
    flops = 0.0
    if name in ROW_KEY_SAMPLE:
        xg = group_slice(x, heads.group)
        smp = RowKeySample(tree, heads.d, heads.group)
        t0 = time.perf_counter()
        n = 0
        while True:
            flops += smp.step(xg, scale)
            n += 1
            if time.perf_counter() - t0 >= target_s:
                break
        dt = time.perf_counter() - t0
        sample = f"{n} steps of: {smp.describe()}; {dt:.1f} s"
    else:
        groups = 0
        while groups < heads.hkv:
            flops += oracle_group_step(tree, x, heads, scale, [groups])
            groups += 1
            if time.perf_counter() - t0 >= target_s:
                break
        dt = time.perf_counter() - t0
        sample = (f"fp64 numpy oracle, fwd+bwd of {groups} of {heads.hkv} kv-head groups "
                  f"({groups * heads.group} q-heads) of the full tree, {dt:.1f} s")
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": sample + "; numpy BLAS default threads", "cpu_model": cpu_model(),
            "blas_threads": blas_threads()}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def blas_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from workloads import tensors as WX
    from workloads import trees as WT
    tree = WT.load_tree(args.workload)
    heads, rec = WX.HEADS[base_name(args.workload)], WX.VALUE_RECIPES[args.workload]
    if args.workload in ROW_KEY_SAMPLE:
        # kv-group 0 drawn on the host with the workload's recipe and seed (the GPU
        # arm draws this workload on the device)
        xg = WX.draw_inputs(tree.n_tokens, WX.HeadConfig(heads.group, 1, heads.d), rec,
                            1000 + WX.SEEDS[args.workload])
        smp = RowKeySample(tree, heads.d, heads.group)
        one = lambda: smp.step(xg, rec.scale)
        sample = "per step: " + smp.describe()
    else:
        _, _, x = WX.workload_inputs(args.workload, tree.n_tokens)
        one = lambda: oracle_group_step(tree, x, heads, rec.scale, [0])
        sample = (f"fp64 numpy oracle fwd+bwd on kv-head group 0 ({heads.group} q-heads, 1 kv-head) of "
                  f"the full tree per step")
    for _ in range(args.warmup):
        one()
    times, flops = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops += one()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = flops / total / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": DESCRIPTIONS.get(args.workload, args.workload),
                                        "name": args.workload, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }))


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

DEFAULT_WORKLOAD = "long_context"
# timed too, each in its own region, and reported inside the same line
OTHER_WORKLOADS = ("tiny_binary", "grpo_star", "segment_tree", "agentic_tree")
# drawn on the device (a CUDA generator with the workload's seed): the host
# would take minutes for ~9e9 normal samples
DEVICE_DRAWN = {"long_context", "long_context_4b"}
# steps at least this long keep the tensor core busy for seconds: their
# roofline takes the sustained bf16 peak, shorter ones the burst peak
LONG_STEP_MS = 100.0


def base_name(name: str) -> str:
    return "tiny_binary" if name.startswith("tiny_binary") else name


def max_over_ranks(local_ms: float, world: int, device=None) -> float:
    """The slowest rank's timed-region length (every rank runs its own tree;
    the job is done when the last one is)."""
    if world <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job useful TFLOP/s: the units all ranks processed over the
    slowest rank's time (weak scaling: each rank holds one tree)."""
    return flops_per_step * steps * world / (max_ms / 1e3) / 1e12


def chain_batches(TA, lens, hq, hkv, d, budget_bytes):
    """Split chains (token counts `lens`, in order) into equal contiguous
    batches, doubling the batch count until one batch's device bytes (Q, K, V,
    dO, O, dQ, dK, dV in bf16, LSE, backward workspace) fit in budget_bytes,
    or every batch holds one chain."""
    def batch_bytes(ls):
        pb = TA.TreePlan([-1] * len(ls), ls)
        nt = pb.n_tokens
        ws = pb.workspace_size(hq, hkv, d)[1]
        pb.close()
        return nt * (4 * hq + 4 * hkv) * d * 2 + 4 * hq * nt + ws

    n_batches = 1
    while True:
        per = -(-len(lens) // n_batches)
        groups = [lens[i:i + per] for i in range(0, len(lens), per)]
        if max(batch_bytes(gl) for gl in groups) <= budget_bytes or per == 1:
            return groups
        n_batches *= 2


def workload_tree(WT, name):
    if name == "long_context_4b":     # the long-context recipe's first 4 branches
        return WT.long_context_tree(seed=5, branches=4)
    return WT.load_tree(name)


def device_inputs(WX, name, n_tokens, dev):
    """Seeded bf16 Q, K, V, dO of a workload on the device."""
    if name == "long_context_4b":
        heads, rec = WX.HeadConfig(48, 6, 128), WX.VALUE_RECIPES["long_context"]
        return heads, rec, WX.draw_inputs(n_tokens, heads, rec, 1005, device=str(dev), chunk_rows=65536)
    heads, rec = WX.HEADS[base_name(name)], WX.VALUE_RECIPES[name]
    if name in DEVICE_DRAWN:
        return heads, rec, WX.draw_inputs(n_tokens, heads, rec, 1000 + WX.SEEDS[name], device=str(dev),
                                          chunk_rows=65536)
    _, _, x = WX.workload_inputs(name, n_tokens)
    return heads, rec, {n: t.to(dev) for n, t in x.items()}


def timed_hot_path(torch, TA, plan, x, heads, scale, steps, warmup, flush, around=None, graph_out=None):
    """Warm up, then time ``steps`` steps (forward, backward pre / main / post)
    with CUDA events on the launching stream, L2 flushed (untimed) before
    each.  ``around`` = (enter, leave) callables wrapped round the timed
    region.  Returns per-step [fwd, pre, main, post] milliseconds.  With
    ``graph_out`` (a dict), the same step is also captured once in a CUDA graph
    (the launch-bound small trees: five launches per step become one) and its
    replays timed the same way; the per-step milliseconds land in
    graph_out["ms"]."""
    hq, hkv, d = heads.hq, heads.hkv, heads.d
    N = plan.n_tokens
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o = torch.empty_like(q)
    lse = torch.empty((hq, N), dtype=torch.float32, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(plan.workspace_size(hq, hkv, d)[1], 1), dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        if evs:
            evs[0].record(stream)
        TA.tree_attn_fwd(plan, q, k, v, scale, o=o, lse=lse)
        for si, stage in enumerate((TA.BWD_PRE, TA.BWD_MAIN, TA.BWD_POST)):
            if evs:
                evs[1 + si].record(stream)
            TA.tree_attn_bwd(plan, q, k, v, o, lse, do, scale, dq=dq, dk=dk, dv=dv, workspace=ws, stages=stage)
        if evs:
            evs[4].record(stream)

    for _ in range(max(warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    if TA.device_status() != 0:
        raise RuntimeError("device status non-zero after warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    if around:
        around[0]()
    torch.cuda.synchronize()
    for kk in range(steps):
        flush.fill_(kk & 0xff)             # evict L2 between timed steps (not timed)
        step(evs[kk])
    torch.cuda.synchronize()
    if around:
        around[1]()
    status = TA.device_status()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    per = [[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in evs]
    if graph_out is not None:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
        ge = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for kk in range(steps):
            flush.fill_(kk & 0xff)
            ge[kk][0].record()
            g.replay()
            ge[kk][1].record()
        torch.cuda.synchronize()
        if TA.device_status() != 0:
            raise RuntimeError("device status non-zero after graph replays")
        graph_out["ms"] = [a.elapsed_time(b) for a, b in ge]
        del g
    del o, lse, dq, dk, dv, ws
    return per


def stage_summary(per, f_fwd, f_bwd):
    fwd_ms = statistics.mean(p[0] for p in per)
    pre_ms = statistics.mean(p[1] for p in per)
    main_ms = statistics.mean(p[2] for p in per)
    post_ms = statistics.mean(p[3] for p in per)
    step_ms = [sum(p) for p in per]
    return {"ms_per_step": statistics.mean(step_ms), "ms_per_step_median": statistics.median(step_ms),
            "fwd_ms": fwd_ms, "bwd_pre_ms": pre_ms, "bwd_main_ms": main_ms, "bwd_post_ms": post_ms,
            "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12, "bwd_main_tflops": f_bwd / (main_ms / 1e3) / 1e12,
            "tflops": (f_fwd + f_bwd) / (statistics.mean(step_ms) / 1e3) / 1e12}


def launches_per_step(plan):
    # forward, backward pre, backward main, dQ conversion, split dK/dV sum
    return 4 + (1 if plan.info["n_split_kv_tiles"] > 0 else 0)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import prefix_tree_attention_attn_gb300 as TA
    from workloads import tensors as WX
    from workloads import trees as WT

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    name = args.workload
    tree = workload_tree(WT, name)
    heads, rec, x = device_inputs(WX, name, tree.n_tokens, dev)
    hq, hkv, d, scale = heads.hq, heads.hkv, heads.d, rec.scale
    t_plan = time.perf_counter()
    for _ in range(5):
        TA.TreePlan(tree.parent, tree.seg_len).close()
    plan_ms = (time.perf_counter() - t_plan) * 1e3 / 5   # host planner, reported on its own
    plan = TA.TreePlan(tree.parent, tree.seg_len)
    N = plan.n_tokens
    f_fwd, f_bwd = useful_flops(plan.n_pairs, hq, d)
    flops_step = f_fwd + f_bwd
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    clocks = ClockSampler(local)
    wall = {}

    def enter():
        clocks.start()
        time.sleep(0.3)                    # let the sampler start
        barrier()
        torch.cuda.synchronize()
        wall["t0"] = time.perf_counter()

    def leave():
        barrier()
        wall["s"] = time.perf_counter() - wall["t0"]

    per = timed_hot_path(torch, TA, plan, x, heads, scale, args.steps, args.warmup, flush, (enter, leave))
    clk = clocks.stop()
    summ = stage_summary(per, f_fwd, f_bwd)
    total_ms = sum(sum(p) for p in per)
    total_max_ms = max_over_ranks(total_ms, world, dev)
    value = job_throughput(flops_step, args.steps, world, total_max_ms)

    peak_burst, peak_sus, peak_src = measured_peaks()
    long_step = summ["ms_per_step"] >= LONG_STEP_MS
    peak = peak_sus if long_step else peak_burst
    peak_name = f"{peak_src} bf16 {'sustained' if long_step else 'burst'}"
    # the backward's tensor-core kernel is bwd_fs_kernel (bwd_fs.cu) for d = 128, bwd_kernel (bwd.cu) else
    bwd_name, bwd_src = ("bwd_fs_kernel", "bwd_fs.cu") if d == 128 else ("bwd_kernel", "bwd.cu")
    main_ms, fwd_ms = summ["bwd_main_ms"], summ["fwd_ms"]
    dominant = (bwd_name, main_ms, f_bwd, bwd_src) if main_ms >= fwd_ms else ("fwd_kernel", fwd_ms, f_fwd, "fwd.cu")
    achieved = dominant[2] / (dominant[1] / 1e3) / 1e12
    src_hash = kernel_source_hash([dominant[3], "ptx.cuh"])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(dominant[0], name, src_hash),
                "kernel": dominant[0], "peak_source": peak_name, "kernel_src_hash": src_hash,
                "algorithmic": f"{'10' if dominant[0] != 'fwd_kernel' else '4'}*d*pairs*hq = {dominant[2]:.4g} FLOP "
                               f"per launch / mean CUDA-event launch time {dominant[1]:.4g} ms"}

    # ---- end to end through the public API, host buffers ------------------
    e2e = None
    if not args.no_e2e and (rank == 0 or world > 1):
        pin = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in ("q", "k", "v", "do")}
        for n in pin:
            pin[n].copy_(x[n])
        outs = {"o": torch.empty((N, hq, d), dtype=torch.bfloat16, pin_memory=True),
                "lse": torch.empty((hq, N), dtype=torch.float32, pin_memory=True),
                "dq": torch.empty((N, hq, d), dtype=torch.bfloat16, pin_memory=True),
                "dk": torch.empty((N, hkv, d), dtype=torch.bfloat16, pin_memory=True),
                "dv": torch.empty((N, hkv, d), dtype=torch.bfloat16, pin_memory=True)}
        h2d = sum(t_.numel() * t_.element_size() for t_ in pin.values())
        d2h = sum(t_.numel() * t_.element_size() for t_ in outs.values())
        # a bounded number of end-to-end steps: about 20 s at most
        e2e_steps = max(3, min(args.steps, 20, int(20e3 / (1.5 * summ["ms_per_step"] + 1.0))))
        e2e_warm = 2 if long_step else max(3, args.warmup)
        side = torch.cuda.Stream(device=dev)        # the dO upload overlaps the forward

        copy_ev = []    # per step: events around the q/k/v upload and the output download

        def e2e_step():
            main = torch.cuda.current_stream(dev)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            copy_ev.append(ev)
            # inputs the forward needs first; the plan is built on the host meanwhile
            ev[0].record(main)
            qd, kd, vd = (pin[n].to(dev, non_blocking=True) for n in ("q", "k", "v"))
            ev[1].record(main)
            side.wait_stream(main)
            with torch.cuda.stream(side):
                dod = pin["do"].to(dev, non_blocking=True)   # arrives during the forward
            p2 = TA.TreePlan(tree.parent, tree.seg_len)      # a new tree each step: plan on the host
            oo, ll = TA.tree_attn_fwd(p2, qd, kd, vd, scale)
            main.wait_stream(side)
            a, b, c = TA.tree_attn_bwd(p2, qd, kd, vd, oo, ll, dod, scale)
            # The outputs leave after the backward.  Measured on one box, long shared
            # context: 1.90-1.96 s per step this way; 1.93-1.98 s with O and LSE
            # leaving during the backward (the copy slows it); 2.09-2.17 s with
            # device buffers made once and reused.
            ev[2].record(main)
            for nm, src in (("o", oo), ("lse", ll), ("dq", a), ("dk", b), ("dv", c)):
                outs[nm].copy_(src, non_blocking=True)
            ev[3].record(main)
            torch.cuda.synchronize(dev)      # the step's results are on the host
            p2.close()

        for _ in range(e2e_warm):   # first-touch costs: allocator pools, plan upload
            e2e_step()
        barrier()
        t0 = time.perf_counter()
        e2e_each = []
        for _ in range(e2e_steps):
            t1 = time.perf_counter()
            e2e_step()
            e2e_each.append(time.perf_counter() - t1)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        timed_ev = copy_ev[-e2e_steps:]
        qkv_bytes = sum(pin[n].numel() * pin[n].element_size() for n in ("q", "k", "v"))
        h2d_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in timed_ev)
        d2h_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in timed_ev)
        e2e = {"value": flops_step * world / e2e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": e2e_steps,
               "ms_each": [round(t_ * 1e3, 2) for t_ in e2e_each],
               "qkv_upload_ms": h2d_ms, "qkv_upload_gbs": qkv_bytes / h2d_ms / 1e6,
               "download_ms": d2h_ms, "download_gbs": d2h / d2h_ms / 1e6,
               "includes": "host plan build + device upload, H2D of q/k/v/dO from pinned memory, fwd+bwd, "
                           "D2H of o/lse/dq/dk/dv after the backward; dO arrives during the forward (side "
                           "stream)"}
        del pin, outs
        torch.cuda.empty_cache()

    # ---- same kernels on the expanded trajectories ---------------------------
    # Every root-to-leaf trajectory as its own chain.  When the whole expanded
    # forest does not fit in half of the free device memory (the long shared
    # context: ~2.5 M tokens), the chains run in equal batches one after another
    # inside each timed step, and the step time is the sum.
    expanded = None
    if not args.no_expanded and rank == 0:
        ft = WT.expanded_forest(tree)
        groups = chain_batches(TA, list(ft.seg_len), hq, hkv, d, 0.5 * torch.cuda.mem_get_info(dev)[0])
        eplans = [TA.TreePlan([-1] * len(gl), gl) for gl in groups]
        Ne = sum(pb.n_tokens for pb in eplans)
        Nmax = max(pb.n_tokens for pb in eplans)
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        xe = {n: (torch.randn((Nmax, h, d), generator=g, device=dev, dtype=torch.float32)).to(torch.bfloat16)
              for n, h in (("q", hq), ("k", hkv), ("v", hkv), ("do", hq))}
        wse = torch.empty(max(max(pb.workspace_size(hq, hkv, d)[1] for pb in eplans), 1), dtype=torch.uint8,
                          device=dev)

        def estep():
            for pb in eplans:
                nb = pb.n_tokens
                qb, kb, vb, dob = (xe[n][:nb] for n in ("q", "k", "v", "do"))
                oo, ll = TA.tree_attn_fwd(pb, qb, kb, vb, scale)
                TA.tree_attn_bwd(pb, qb, kb, vb, oo, ll, dob, scale, workspace=wse)

        for _ in range(1 if long_step else 3):
            estep()
        torch.cuda.synchronize()
        ee = []
        for _ in range(2 if long_step else min(args.steps, 20)):
            flush.fill_(3)
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record()
            estep()
            b_.record()
            ee.append((a_, b_))
        torch.cuda.synchronize()
        ems = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ee)
        expanded = {"ms_per_step": ems, "speedup": ems / summ["ms_per_step"], "n_tokens": Ne,
                    "pairs": sum(pb.n_pairs for pb in eplans), "chain_batches": len(eplans), "steps": len(ee)}
        for pb in eplans:
            pb.close()
        del xe, wse
        torch.cuda.empty_cache()

    # ---- the smaller workloads, each timed the same way ----------------------
    others = []
    if rank == 0 and world == 1 and name == DEFAULT_WORKLOAD and not args.no_others:
        for wn in OTHER_WORKLOADS:
            tw = WT.load_tree(wn)
            hw, rw, xw = device_inputs(WX, wn, tw.n_tokens, dev)
            pw = TA.TreePlan(tw.parent, tw.seg_len)
            ff, fb = useful_flops(pw.n_pairs, hw.hq, hw.d)
            gr = {}
            pr = timed_hot_path(torch, TA, pw, xw, hw, rw.scale, min(args.steps, 20), 3, flush, graph_out=gr)
            sw = stage_summary(pr, ff, fb)
            gms = statistics.mean(gr["ms"])
            sw["graph"] = {"ms_per_step": gms, "tflops": (ff + fb) / (gms / 1e3) / 1e12,
                           "what": "the same five launches captured once in a CUDA graph and replayed"}
            sw.update({"name": wn, "workload": DESCRIPTIONS[wn], "n_tokens": pw.n_tokens, "pairs": pw.n_pairs,
                       "hq": hw.hq, "hkv": hw.hkv, "d": hw.d, "steps": len(pr),
                       "pct_peak": 100.0 * sw["tflops"] / peak_burst, "peak": f"{peak_src} bf16 burst"})
            others.append(sw)
            pw.close()
            del xw

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(name, tree, x, heads, scale, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": total_max_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": DESCRIPTIONS.get(name, name), "name": name,
                       "n_tokens": N, "pairs": plan.n_pairs, "hq": hq, "hkv": hkv, "d": d,
                       "softmax_scale": scale, "l2": "flushed between timed steps (512 MB write, untimed)",
                       "inputs": "drawn on the device" if name in DEVICE_DRAWN else "drawn on the host, copied",
                       "parallelism": f"replicas x{world} (independent trees per GPU)"},
            "pct_peak": 100.0 * value / world / peak, "peak_source": peak_name,
            "ms_per_step_median": summ["ms_per_step_median"],
            "plan_ms_host": plan_ms,
            "fwd_ms": summ["fwd_ms"], "bwd_pre_ms": summ["bwd_pre_ms"], "bwd_main_ms": summ["bwd_main_ms"],
            "bwd_post_ms": summ["bwd_post_ms"], "fwd_tflops": summ["fwd_tflops"],
            "bwd_main_tflops": summ["bwd_main_tflops"],
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step(plan) * args.steps,
            "clocks": clk,
            "speedup_vs_expanded": expanded["speedup"] if expanded else None,
            "expanded": expanded,
            "other_workloads": others,
            "wall_s_timed_region": wall.get("s"),
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_extras(args):
    """The calls around the attention, each timed on its own: host batching of
    many trees, weights folded into dO, per-trajectory log-probs from compact
    logits (vocabulary 152,064, the Qwen2.5 LM-head width), subtree advantages."""
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from prefix_tree_attention_attn_gb300 import TreePlan
    from prefix_tree_attention_attn_gb300 import batch as TB
    from prefix_tree_attention_attn_gb300 import loss as TL
    from workloads import tensors as WX
    from workloads import trees as WT

    hbm = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            hbm = float(json.load(f)["hbm_gbs"])
    except Exception:
        hbm = 6800.0

    # -- batching: 2048 trees (segment trees and GRPO stars of varied seeds), 8 replicas
    trees = []
    for sd in range(1024):
        a, b = WT.segment_tree(seed=100 + sd), WT.grpo_star_tree(seed=5000 + sd)
        trees += [(a.parent, a.seg_len), (b.parent, b.seg_len)]
    batch = TB.TreeBatch(trees)
    t0 = time.perf_counter()
    reps = 5
    for _ in range(reps):
        pairs, toks = batch.work()
        rep, load = TB.batch_assign(pairs, 8)
        n_forests = 0
        for r in range(8):
            mb, n_mb = TB.batch_microbatches(pairs, toks, rep, r, 65536)
            for m in range(n_mb):
                batch.forest(mb == m)
                n_forests += 1
    host_ms = (time.perf_counter() - t0) * 1e3 / reps
    print(json.dumps({"metric": "tree batching (work, LPT over 8 replicas, 64k-token microbatches, forests)",
                      "value": len(trees) / (host_ms / 1e3), "unit": "trees/s", "ms_per_batch": host_ms,
                      "config": {"trees": len(trees), "replicas": 8, "microbatches": n_forests,
                                 "max_replica_pairs_over_mean": float(load.max() / load.mean())},
                      "dtype": "int64", "cores": 1}))

    dev = torch.device("cuda:0")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed_steps(fn, iters, warm):
        for _ in range(warm):
            fn()
        ms = []
        for _ in range(iters):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    # the tiny binary tree is latency-bound alone (one launch for 3.9e7 FLOP); 4,096 copies
    # packed as one forest by the batching calls run in one fwd + bwd call
    tiny = WT.load_tree("tiny_binary")
    copies = 4096
    fpar, fseg, _ = TB.TreeBatch([(tiny.parent, tiny.seg_len)] * copies).forest([True] * copies)
    fplan = TreePlan(fpar, fseg)
    th, trc = WX.HEADS["tiny_binary"], WX.VALUE_RECIPES["tiny_binary"]
    tx = WX.draw_inputs(fplan.n_tokens, th, trc, 1000 + WX.SEEDS["tiny_binary"], device="cuda")
    from prefix_tree_attention_attn_gb300 import tree_attn_bwd, tree_attn_fwd

    def tiny_step():
        o_, l_ = tree_attn_fwd(fplan, tx["q"], tx["k"], tx["v"], trc.scale)
        tree_attn_bwd(fplan, tx["q"], tx["k"], tx["v"], o_, l_, tx["do"], trc.scale)

    ms = timed_steps(tiny_step, 10, 3)
    ff, fb = useful_flops(fplan.n_pairs, th.hq, th.d)
    print(json.dumps({"metric": METRIC + " (variant: tiny binary tree x 4096 as one forest)",
                      "value": (ff + fb) / (ms / 1e3) / 1e12, "unit": UNIT, "ms": ms,
                      "pct_peak": 100 * (ff + fb) / (ms / 1e3) / 1e12 / measured_peaks()[0],
                      "config": {"workload": "tiny_binary x 4096 forest", "n_tokens": fplan.n_tokens,
                                 "pairs": fplan.n_pairs, "hq": th.hq, "hkv": th.hkv, "d": th.d}, "dtype": "bf16"}))
    del tx

    def timed(fn, iters=20, warm=3):
        return timed_steps(fn, iters, warm)

    t = WT.load_tree("grpo_star")
    heads, rec = WX.HEADS["grpo_star"], WX.VALUE_RECIPES["grpo_star"]
    plan = TreePlan(t.parent, t.seg_len)
    x = WX.draw_inputs(t.n_tokens, heads, rec, 1000 + WX.SEEDS["grpo_star"], device="cuda")
    mult, _ = TL.token_info(plan)
    w = torch.as_tensor(mult, dtype=torch.float32, device=dev)
    do = x["do"]
    out = torch.empty_like(do)
    ms = timed(lambda: TL.scale_rows(do, w, out=out))
    nbytes = 2 * do.numel() * 2 + w.numel() * 4
    print(json.dumps({"metric": "multiplicity weights folded into dO (scale_rows)", "value": nbytes / ms / 1e6,
                      "unit": "GB/s", "ms": ms, "roofline": {"bound": "hbm", "peak": hbm, "frac": nbytes / ms / 1e6 / hbm},
                      "config": {"workload": "grpo_star dO [11167, 32, 128] bf16"}, "dtype": "bf16"}))

    V = 32768 if args.extras_small else 152064
    g = torch.Generator(device="cuda").manual_seed(9)
    logits = (torch.randn(t.n_tokens, V, generator=g, device=dev) * 2.0).to(torch.bfloat16)
    tokens = torch.randint(0, V, (t.n_tokens,), generator=g, device=dev, dtype=torch.int32)
    lse, lp = TL.traj_logprobs(plan, logits, tokens)
    ms = timed(lambda: TL.traj_logprobs(plan, logits, tokens, row_lse=lse, out=lp), iters=10)
    nbytes = logits.numel() * 2 + lp.numel() * (4 + 8 + 4 + 2) + t.n_tokens * 4
    print(json.dumps({"metric": "per-trajectory next-token log-probs from compact logits", "value": nbytes / ms / 1e6,
                      "unit": "GB/s", "ms": ms, "roofline": {"bound": "hbm", "peak": hbm, "frac": nbytes / ms / 1e6 / hbm},
                      "config": {"workload": f"grpo_star logits [11167, {V}] bf16", "predictions": lp.numel(),
                                 "expanded_rows_avoided": int(t.n_expanded - t.n_tokens)}, "dtype": "bf16"}))
    del logits

    # linear attention over the tree (chunks of <= 128 tokens, state handed to children)
    from prefix_tree_attention_attn_gb300.linear import linear_workspace, tree_linear_bwd, tree_linear_fwd
    for wname in ("grpo_star",) if args.extras_small else ("grpo_star", "long_context"):
        tl = WT.load_tree(wname)
        hl, rl = WX.HEADS[wname], WX.VALUE_RECIPES[wname]
        xl = WX.draw_inputs(tl.n_tokens, hl, rl, 1000 + WX.SEEDS[wname], device="cuda", chunk_rows=65536)
        pl = TreePlan(tl.parent, tl.seg_len)
        nc, wsb = linear_workspace(pl, hl.hkv, hl.d)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        dec = torch.full((hl.hkv,), 0.999, dtype=torch.float32, device=dev)
        ol = torch.empty_like(xl["q"])
        run = lambda: tree_linear_fwd(pl, xl["q"], xl["k"], xl["v"], dec, 1 / math.sqrt(hl.d), o=ol, workspace=ws)
        ms = timed(run, iters=10 if wname == "grpo_star" else 3, warm=2)
        # tensor work issued: per chunk and kv-head K^T V (2 d^2 128), per chunk and
        # q-head Q K^T, Q S_in and P V (3 x 2 x 128 x 128 x d)
        flops = nc * (hl.hkv * 2 * hl.d * hl.d * 128 + hl.hq * 3 * 2 * 128 * 128 * hl.d)
        print(json.dumps({"metric": "tree linear attention forward (chunked, state handoff at branch points)",
                          "value": tl.n_tokens / (ms / 1e3), "unit": "compact tokens/s", "ms": ms,
                          "roofline": {"bound": "tensor", "achieved": flops / ms / 1e9, "unit": "TFLOP/s",
                                       "peak": measured_peaks()[0],
                                       "frac": flops / ms / 1e9 / measured_peaks()[0]},
                          "config": {"workload": wname, "chunks": nc, "hq": hl.hq, "hkv": hl.hkv, "d": hl.d,
                                     "decay": 0.999, "workspace_bytes": wsb}, "dtype": "bf16"}))
        dql, dkl, dvl = torch.empty_like(xl["q"]), torch.empty_like(xl["k"]), torch.empty_like(xl["v"])
        runb = lambda: tree_linear_bwd(pl, xl["q"], xl["k"], xl["v"], xl["do"], dec, 1 / math.sqrt(hl.d), dq=dql,
                                       dk=dkl, dv=dvl, workspace=ws)
        msb = timed(runb, iters=10 if wname == "grpo_star" else 3, warm=2)
        # tensor work issued: dQ is the forward's; F per chunk and q-head Q^T dO (2 d^2 128);
        # per chunk and kv-head V Rsum^T and K Rsum (2 x 2 x 128 d^2); per chunk and
        # q-head K Q^T, V dO^T, P^T dO and dA^T Q (4 x 2 x 128 x 128 x d)
        flops_b = flops + nc * (hl.hq * 2 * hl.d * hl.d * 128 + hl.hkv * 4 * 128 * hl.d * hl.d
                                + hl.hq * 4 * 2 * 128 * 128 * hl.d)
        print(json.dumps({"metric": "tree linear attention backward (dQ, dK, dV; adjoint state summed over children)",
                          "value": tl.n_tokens / (msb / 1e3), "unit": "compact tokens/s", "ms": msb,
                          "roofline": {"bound": "tensor", "achieved": flops_b / msb / 1e9, "unit": "TFLOP/s",
                                       "peak": measured_peaks()[0],
                                       "frac": flops_b / msb / 1e9 / measured_peaks()[0]},
                          "config": {"workload": wname, "chunks": nc, "hq": hl.hq, "hkv": hl.hkv, "d": hl.d,
                                     "decay": 0.999}, "dtype": "bf16"}))
        del xl, ws, ol, dql, dkl, dvl

    ta = WT.load_tree("agentic_tree")
    pa = TreePlan(ta.parent, ta.seg_len)
    L, _ = TL.trajectory_info(pa)
    r = torch.randn(L, device=dev)
    TL.subtree_advantage(pa, r, flags=TL.NORM_STD)
    ms = timed(lambda: TL.subtree_advantage(pa, r, flags=TL.NORM_STD), iters=20)
    print(json.dumps({"metric": "subtree advantages (per trajectory, node and compact token)", "value": ms * 1e3,
                      "unit": "us", "higher_is_better": False,
                      "config": {"workload": "agentic_tree", "nodes": ta.n_nodes, "leaves": L,
                                 "tokens": ta.n_tokens}, "dtype": "f32"}))


def main():
    args = parse_args()
    if args.extras:
        run_extras(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
