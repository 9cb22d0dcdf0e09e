"""Benchmark of one EAGLE-2 draft-tree verification step on GB300.

A step is the whole hot path over one batch of synthetic inputs that are
already resident in HBM: D x et_tree_expand, et_tree_rerank,
et_tree_mask_posids, et_tree_attention, et_verify_accept.  Steps are replayed
from CUDA graphs over R rotating input sets whose combined footprint is
larger than L2, so every step reads its logits and KV from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead (the only other implementation of this path), on a bounded sample.

Multi-GPU: each rank is an independent replica on its own GPU with its own
sequences (the step has no exchange), so scaling is weak and there is no
collective in the data path; a barrier and a max-over-ranks of the timed
region are the only communication.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
DEFAULT_WORKLOAD = "llama2-7b"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def attention_bytes(wl, prefix_lens):
    """Bytes one et_tree_attention launch must move: KV prefix + tree K/V + Q + O."""
    el = 2 if wl.dtype == "bf16" else 4
    kv = sum(2 * wl.Hkv * int(L) * wl.d * el for L in prefix_lens)
    B = len(prefix_lens)
    tree = 2 * B * wl.N * wl.Hkv * wl.d * el
    qo = 2 * B * wl.N * wl.Hq * wl.d * el
    return kv + tree + qo


def step_bytes(wl, cfg, prefix_lens, expanded_rows):
    """Bytes a step reads from its inputs: expanded draft rows, the N target rows and the attention bytes."""
    B = len(prefix_lens)
    return B * (expanded_rows + wl.N) * wl.V * 4 + attention_bytes(wl, prefix_lens)


# ---------------------------------------------------------------------------
# clocks sampling (nvidia-smi during the timed region)
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, csv_path=""):
        self.proc = None
        self.gpu = gpu_index
        self.csv_path = csv_path  # where to keep the raw samples ("" = nowhere)
        self.out = None

    def __enter__(self):
        if self.csv_path:
            try:
                self.out = open(self.csv_path, "w")
            except OSError:
                self.out = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
            if self.out:
                self.out.write("\n".join(self.lines) + "\n")
        if self.out:
            self.out.close()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------
ORACLE_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle as O
from speculative_decoding_eagle_gb300 import workloads as W
wl = W.WORKLOADS[{name!r}].with_(B=1)
cfg = O.TreeCfg(B=1, V=wl.V, depth=wl.depth, topk=wl.topk, m=wl.m, n=wl.n, temperature=wl.temperature)
C = O.num_candidates(cfg)
budget = {budget}
done, spent, parts = 0, 0.0, {{}}
b = 0
while spent < budget and done < {max_steps}:
    target, draft, rmap = W.logit_tables(wl, C, batch=range(b, b + 1))
    L = int(W.prefix_lengths(wl, b + 1)[b])
    x = W.qkv(wl, b, L)
    u = W.uniforms(wl, b)[None]
    root = W.root_tokens(wl, b + 1)[b:b + 1]
    t0 = time.perf_counter()
    tree = O.build_tree(cfg, draft, rmap, root)
    t1 = time.perf_counter()
    mask, pos = O.mask_posids(tree.flat_parent, tree.flat_depth, np.array([L]))
    q = W.as_float(wl, x["q"])[None].astype(np.float64)
    kp = [W.as_float(wl, x["k_prefix"]).astype(np.float64)]
    vp = [W.as_float(wl, x["v_prefix"]).astype(np.float64)]
    kt = W.as_float(wl, x["k_tree"])[None].astype(np.float64)
    vt = W.as_float(wl, x["v_tree"])[None].astype(np.float64)
    t2 = time.perf_counter()
    O.tree_attention(q, kp, vp, kt, vt, mask, wl.d ** -0.5)
    t3 = time.perf_counter()
    mode = O.GREEDY if "greedy" in wl.accept else O.STOCH_POINT
    O.verify_accept(cfg, mode, tree.flat_tok, tree.flat_parent, tree.flat_node, target, rmap, uniforms=u)
    t4 = time.perf_counter()
    spent += (t1 - t0) + (t3 - t2) + (t4 - t3) + (t2 - t1)
    for k, v in (("tree", t1 - t0), ("mask_conv", t2 - t1), ("attention", t3 - t2), ("accept", t4 - t3)):
        parts[k] = parts.get(k, 0.0) + v
    done += 1
    b += 1
print(json.dumps({{"steps": done, "seconds": spent, "parts": parts}}))
"""


ORACLE_WORKER = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle as O
from speculative_decoding_eagle_gb300 import workloads as W
wl = W.WORKLOADS[{name!r}].with_(B=1)
cfg = O.TreeCfg(B=1, V=wl.V, depth=wl.depth, topk=wl.topk, m=wl.m, n=wl.n, temperature=wl.temperature)
C = O.num_candidates(cfg)
b = {worker}
target, draft, rmap = W.logit_tables(wl, C, batch=range(b, b + 1))
L = int(W.prefix_lengths(wl, b + 1)[b])
x = W.qkv(wl, b, L)
u = W.uniforms(wl, b)[None]
root = W.root_tokens(wl, b + 1)[b:b + 1]
q = W.as_float(wl, x["q"])[None].astype(np.float64)
kp = [W.as_float(wl, x["k_prefix"]).astype(np.float64)]
vp = [W.as_float(wl, x["v_prefix"]).astype(np.float64)]
kt = W.as_float(wl, x["k_tree"])[None].astype(np.float64)
vt = W.as_float(wl, x["v_tree"])[None].astype(np.float64)
mode = O.GREEDY if "greedy" in wl.accept else O.STOCH_POINT
start = {start_at}
while time.time() < start:
    time.sleep(0.005)
t0 = time.time()
done = 0
while time.time() - t0 < {budget}:
    tree = O.build_tree(cfg, draft, rmap, root)
    mask, pos = O.mask_posids(tree.flat_parent, tree.flat_depth, np.array([L]))
    O.tree_attention(q, kp, vp, kt, vt, mask, wl.d ** -0.5)
    O.verify_accept(cfg, mode, tree.flat_tok, tree.flat_parent, tree.flat_node, target, rmap, uniforms=u)
    done += 1
print(json.dumps({{"steps": done, "t0": t0, "t1": time.time(), "late": t0 - start}}))
"""


def host_cores() -> int:
    """Cores this process may run on (the box's count is read, not assumed)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_baseline_all_cores(name, budget_s=10.0, lead_s=None):
    """The oracle on every host core at once: one process per core, one BLAS
    thread each, each timing full steps of its own sequence from a common
    wall-clock start; throughput = all completed steps / (last end - start)."""
    P = host_cores()
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    lead = lead_s if lead_s is not None else 20.0 + 0.5 * P  # input generation before the common start
    start_at = time.time() + lead
    procs = [subprocess.Popen([sys.executable, "-c", ORACLE_WORKER.format(root=ROOT, name=name, worker=w,
                                                                           start_at=start_at, budget=budget_s)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
             for w in range(P)]
    res = []
    for pr in procs:
        out, err = pr.communicate(timeout=900)
        if pr.returncode != 0:
            raise RuntimeError("oracle worker failed:\n" + err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    steps = sum(r["steps"] for r in res)
    span = max(r["t1"] for r in res) - start_at
    late = max(r["late"] for r in res)
    return {"value": steps / span, "unit": "steps/s", "cores": P, "kind": "oracle",
            "sample": f"{steps} full steps of the {name} workload (batch 1) on {P} processes, one per core, "
                      f"one BLAS thread each, {budget_s:.0f} s from a common start; input generation untimed",
            "seconds": round(span, 3), "late_start_s": round(late, 3)}


def oracle_baseline(name, budget_s=15.0, max_steps=80):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    code = ORACLE_SNIPPET.format(root=ROOT, name=name, budget=budget_s, max_steps=max_steps)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle baseline failed:\n" + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["steps"] / d["seconds"], "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{d['steps']} full steps of the {name} workload (batch 1, fresh seeded inputs each), "
                      f"fp64 numpy, 1 BLAS thread; input generation untimed",
            "seconds": round(d["seconds"], 3), "parts_s": {k: round(v, 3) for k, v in d["parts"].items()}}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
# DRAM traffic of the attention kernel, from the committed ncu summary of the
# same build: the summary records a hash of the kernel's sources, and the
# figure is reported only while the sources still hash the same
# ---------------------------------------------------------------------------
ATTN_SOURCES = ("et_attention_tc.cu", "et_attn_internal.h", "et_common.cuh", "et_tc.cuh", "et_attention.cu")


def attention_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(ROOT, "speculative_decoding_eagle_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_attention_traffic(workload: str, batch: int, prefix: int):
    """Bytes per launch (DRAM read + write) that ncu measured for this
    workload on this exact kernel source, or None."""
    import glob
    import re
    want = attention_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "attn_*.md"))):
        txt = open(path).read()
        m = re.search(r"^traffic: workload=(\S+) batch=(\d+) prefix=(\d+) bytes_per_launch=(\d+) "
                      r"sources_sha256=([0-9a-f]{64})$", txt, flags=re.M)
        if m and m.group(1) == workload and int(m.group(2)) == batch and int(m.group(3)) == prefix \
                and m.group(5) == want:
            return int(m.group(4))
    return None


# ---------------------------------------------------------------------------
# replicas: each rank runs whole steps on its own sequences (no data-path
# collective); only the timing is reduced, as the maximum over ranks
# ---------------------------------------------------------------------------
def step_spread(step_ms):
    """Median, 10th and 90th percentiles (linear interpolation) of per-step times in ms."""
    xs = sorted(float(x) for x in step_ms)
    if not xs:
        return {"median_ms": None, "p10_ms": None, "p90_ms": None}

    def pct(p):
        k = (len(xs) - 1) * p / 100.0
        lo = int(k)
        hi = min(lo + 1, len(xs) - 1)
        return xs[lo] + (xs[hi] - xs[lo]) * (k - lo)
    return {"median_ms": round(pct(50), 5), "p10_ms": round(pct(10), 5), "p90_ms": round(pct(90), 5)}


def shard_offsets(rank: int, n_sets: int, batch: int):
    """First sequence index of each of rank `rank`'s input sets: ranks and
    sets cover disjoint, consecutive blocks of `batch` sequences."""
    return [(rank * n_sets + r) * batch for r in range(n_sets)]


def reduce_step_ms(step_ms: float, world: int, device=None) -> float:
    """The slowest rank's time per step (all ranks wait for it)."""
    if world <= 1:
        return step_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([step_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(step_ms: float, world: int) -> float:
    """Steps per second of all ranks together (weak scaling: one step per rank)."""
    return world * 1000.0 / step_ms


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    from speculative_decoding_eagle_gb300 import step as S
    from speculative_decoding_eagle_gb300 import workloads as W

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if rank == 0 or world == 1:
        build_lib.build()
    if world > 1:
        dist.barrier()
    E.load()
    wl = W.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.with_(B=args.batch)
    if args.prefix:
        wl = wl.with_(prefix=args.prefix, ragged=False)
    mode = None if args.mode == "auto" else {"greedy": E.ET_ACCEPT_GREEDY, "stoch": E.ET_ACCEPT_STOCH_POINT,
                                              "draftq": E.ET_ACCEPT_STOCH_DRAFTQ}[args.mode]
    st = S.VerifyStep(wl, mode=mode, num_splits=args.splits,
                      attn_impl={"auto": E.ATTN_AUTO, "mma": E.ATTN_MMA_SYNC, "tcgen05": E.ATTN_TCGEN05}[args.attn])
    cfg = st.cfg
    prefix = W.prefix_lengths(wl, cfg.B)
    expanded = sum(E.et_layer_expanded(cfg, l) for l in range(cfg.depth))
    per_step = step_bytes(wl, cfg, prefix, expanded)
    R = args.sets or max(2, int(np.ceil(2 * L2_BYTES / per_step)) + 1)
    # rank r's sequences are disjoint from every other rank's (weak scaling)
    sets = []
    for b0 in shard_offsets(rank, R, cfg.B):
        sets.append(S.to_device(wl, S.host_inputs(wl, st.C, cfg.B, b0=b0)))
    st.prepare(sets[0])
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    # eager warm-up on a side stream, then one graph per input set
    with torch.cuda.stream(stream):
        for r in range(R):
            st.run(sets[r], stream=stream)
    stream.synchronize()
    graphs = []
    if not args.eager:
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                st.run(sets[r], stream=stream)
            graphs.append(g)
    torch.cuda.synchronize()

    def one_step(i):
        if graphs:
            graphs[i % R].replay()
        else:
            with torch.cuda.stream(stream):
                st.run(sets[i % R], stream=stream)

    for i in range(args.warmup):
        one_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # graphs replay on the current stream; eager steps run on the side stream
    cur = torch.cuda.current_stream() if graphs else stream
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]  # the end of each step
    with Clocks(local, args.clocks_csv) as clk:
        t_wall = time.perf_counter()
        ev0.record(cur)
        for i in range(args.steps):
            one_step(i)
            marks[i].record(cur)
        ev1.record(cur)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    step_ms = reduce_step_ms(ev0.elapsed_time(ev1) / args.steps, world, device="cuda")
    steps_per_s = whole_job_rate(step_ms, world)
    spread = step_spread([(ev0 if i == 0 else marks[i - 1]).elapsed_time(marks[i]) for i in range(args.steps)])

    # ---- the same step without graphs (every launch from the host) ----
    eager_ms = None
    if graphs:
        ke = max(3, min(50, args.steps))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(ke):
                st.run(sets[i % R], stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        eager_ms = round(e0.elapsed_time(e1) / ke, 5)

    # ---- attention alone (the standalone split plan): a graph of K launches over the rotating sets ----
    K = max(8, min(200, args.steps))
    sa = S.VerifyStep(wl, mode=mode, num_splits=args.splits, overlap=False,
                      attn_impl={"auto": E.ATTN_AUTO, "mma": E.ATTN_MMA_SYNC, "tcgen05": E.ATTN_TCGEN05}[args.attn])
    sa.prepare(sets[0])
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for r in range(R):
            sa.run(sets[r], stream=stream)  # its own trees and masks
    stream.synchronize()
    with torch.cuda.graph(ga, stream=stream):
        for i in range(K):
            sa.attention(sets[i % R], stream=stream)
    ga.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    ga.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    attn_us = e0.elapsed_time(e1) * 1000.0 / K
    attn_b = attention_bytes(wl, prefix)
    hbm_peak, bf16_peak, peak_src = _peaks()
    achieved = attn_b / (attn_us * 1e-6) / 1e9

    # ---- each call of the step alone, graph-timed the same way: which kernel dominates ----
    def graph_us(call):
        with torch.cuda.stream(stream):
            for r in range(R):
                call(sets[r])
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                call(sets[i % R])
        g.replay()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(cur)
        g.replay()
        a1.record(cur)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) * 1000.0 / K

    tree_us = graph_us(lambda inp: st.build_tree(inp, stream=stream))
    accept_us = graph_us(lambda inp: st.accept(inp, stream=stream))
    # the step's own attention (its split count chosen to stream beside the tree build): what it adds to the tree
    tree_attn_us = graph_us(lambda inp: (st.build_tree(inp, stream=stream), st.attention(inp, stream=stream)))
    tree_b = 4 * wl.V * expanded * cfg.B          # one fp32 logits row per expanded node
    accept_b = 4 * wl.V * cfg.N * cfg.B           # every flat row's target logits (what the kernel reads)
    # the acceptance's algorithmic minimum: the rows on the accepted paths and each stop row
    path_rows = []
    for r in range(R):
        st.accept(sets[r], stream=stream)
        stream.synchronize()
        path_rows.append(int((st.accept_len.cpu() + 1).clamp(max=wl.depth + 1).sum()))
    accept_path_b = int(round(4 * wl.V * sum(path_rows) / len(path_rows)))
    parts = [("et_tree_build", tree_us, tree_b, "latency: D dependent layers, each a DRAM round trip, "
                                                 "two cluster barriers and a cross-cluster handshake"),
             ("et_tree_attention", attn_us, attn_b, "hbm"),
             ("et_verify_accept", accept_us, accept_b, "latency: one row per cluster, then the walk")]
    total_us = sum(p_[1] for p_ in parts)
    step_kernels = {"calls": [{"call": n_, "us_alone": round(u_, 3), "share_of_sum": round(u_ / total_us, 3),
                               "bytes": b_, "GBps": round(b_ / (u_ * 1e-6) / 1e9, 1),
                               "frac_hbm": round(b_ / (u_ * 1e-6) / 1e9 / hbm_peak, 4), "bound": bd_}
                              for n_, u_, b_, bd_ in parts],
                    # bytes the acceptance moves (every flat row) and its algorithmic minimum (the path rows)
                    "accept_moved_bytes": accept_b, "accept_algorithmic_bytes": accept_path_b,
                    "attention_alone_splits": E.et_tree_attention_splits(sa.shape),
                    "attention_in_step_splits": E.et_tree_attention_splits(st.shape),
                    "tree_then_attention_us": round(tree_attn_us, 3),
                    "attention_adds_to_tree_us": round(tree_attn_us - tree_us, 3)}

    # ---- attention alone at the other target shapes, at the batched sweep's shape, and the
    # batched sweep's whole step: in a child process, so that a failure there cannot end this one ----
    shapes, batched, sweep = [], [], []
    if not args.no_attn_shapes and local == 0:  # the child runs on device 0: the first rank's GPU
        ex = run_extras_child(args)
        shapes, batched, sweep = ex["tree_attention_shapes"], ex["tree_attention_batched"], ex["sweep_step"]

    # ---- KV commit of the accepted paths (the step after acceptance), timed alone ----
    commit = time_kv_commit(st, sets[0], wl, cfg, prefix, stream, K)

    # ---- a static draft tree of the same size, flattened from the same draft table ----
    static = time_static_tree(wl, cfg, sets[0], stream, K)

    # ---- the draft LM head that produces one layer's logits (tcgen05) ----
    lm_head = time_lm_head(wl, cfg, stream, K, hbm_peak)

    # ---- end to end through the public API with host buffers ----
    e2e = run_e2e(args, st, sets, wl, stream, host_tables=True)
    e2e["whole_copy"] = run_e2e(args, st, sets, wl, stream, host_tables=False)

    launches = st.launches() * args.steps
    out = {
        "metric": "tree-verify steps/s (1 GB300, batch 1) with tree-attention HBM GB/s",
        "value": round(steps_per_s, 2), "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "step_spread": spread,
        "eager_ms_per_step": eager_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 attention (fp32 accumulate), fp32 logits" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded Zipf target logits, noisy draft logits, N(0,1) Q/K/V)",
        "config": {"workload": wl.name, "batch": cfg.B, "V": wl.V, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "prefix": int(prefix.max()), "depth": wl.depth, "topk": wl.topk, "m": wl.m, "n": wl.n,
                   "accept": {0: "greedy", 1: "stoch_point", 2: "stoch_draftq"}[st.mode],
                   "attention_splits": E.et_tree_attention_splits(st.shape),
                   "attention_kernel": {0: "auto", 1: "mma.sync", 2: "tcgen05"}[st.attn_impl] if st.attn_impl else
                   ("fp32 cores" if wl.dtype != "bf16" else ("tcgen05" if wl.d == 128 else "mma.sync")),
                   "l2": f"inputs larger than L2: {R} rotating input sets, {per_step / 1e6:.1f} MB read per step",
                   "cuda_graphs": bool(graphs), "parallelism": f"replicas x{world}"},
        "tree_attention": {"us_per_launch": round(attn_us, 3), "splits": E.et_tree_attention_splits(sa.shape),
                           "GBps": round(achieved, 1),
                           "pct_of_8TBps": round(100 * achieved / 8000.0, 2), "bytes": attn_b},
        "tree_attention_shapes": shapes,
        "tree_attention_batched": batched,
        "sweep_step": sweep,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": args.traffic if args.traffic is not None else
                     recorded_attention_traffic(wl.name, cfg.B, int(prefix.max())),
                     "peak_source": peak_src, "kernel": "et_tree_attention"},
        "step_kernels": step_kernels,
        "e2e": e2e,
        "kv_commit": commit,
        "static_tree": static,
        "lm_head": lm_head,
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        try:
            one = oracle_baseline(wl.name)
            try:
                allc = oracle_baseline_all_cores(wl.name)
                out["cpu_baseline"] = dict(allc, one_core=one)
            except Exception as ex:  # keep the one-core figure
                out["cpu_baseline"] = dict(one, all_cores_error=str(ex)[:300])
        except Exception as ex:  # report, never hide
            out["cpu_baseline"] = {"error": str(ex)[:300]}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def attention_flops(wl, prefix_lens):
    """FLOPs one et_tree_attention launch performs as the kernel tiles it: Q K^T
    and P V of every row over its prefix and the N tree rows (2 x 2 x d each)."""
    return sum(4 * wl.N * wl.Hq * wl.d * (int(L) + wl.N) for L in prefix_lens)


# further attention shapes timed in the same run (batch 1): the two HBM-bound
# shapes at prefix 4096 and the tensor-core-bound GQA shape
ATTN_SHAPES = (("llama2-7b", 4096), ("llama2-13b", 4096), ("llama2-70b", 8192))


def time_attention_shape(name, prefix, stream, K, hbm_peak, bf16_peak):
    """et_tree_attention alone at one more shape, batch 1: one tree (from the
    shape's own seeded draft logits) gives the mask; Q/K/V rotate over sets
    whose combined size exceeds L2; CUDA events around a graph of K launches."""
    import dataclasses
    import numpy as np
    import torch
    from speculative_decoding_eagle_gb300 import step as S
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS[name].with_(B=1, prefix=prefix, ragged=False)
    st = S.VerifyStep(wl, overlap=False)  # the standalone split plan
    base = S.to_device(wl, S.host_inputs(wl, st.C))
    st.run(base, stream=stream)  # the mask of a real tree
    stream.synchronize()
    nb = attention_bytes(wl, [prefix])
    R = max(2, int(np.ceil(2 * L2_BYTES / nb)) + 1)
    sets = [base]
    kind = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    for r in range(1, R):
        x = W.qkv(wl, r, prefix)

        def up(a):
            a = np.ascontiguousarray(a)
            if wl.dtype == "bf16":
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
            return torch.from_numpy(a).cuda()
        sets.append(dataclasses.replace(base, q=up(x["q"])[None], k_prefix=up(x["k_prefix"].reshape(-1, wl.d)),
                                        v_prefix=up(x["v_prefix"].reshape(-1, wl.d)), k_tree=up(x["k_tree"])[None],
                                        v_tree=up(x["v_tree"])[None]))
    with torch.cuda.stream(stream):
        for r in range(R):
            st.attention(sets[r], stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(K):
            st.attention(sets[i % R], stream=stream)
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    gbs = nb / (us * 1e-6) / 1e9
    fl = attention_flops(wl, [prefix])
    tfs = fl / (us * 1e-6) / 1e12
    out = {"workload": name, "batch": 1, "prefix": prefix, "Hq": wl.Hq, "Hkv": wl.Hkv, "N": wl.N,
           "splits": E_splits(st), "us_per_launch": round(us, 3), "bytes": nb, "GBps": round(gbs, 1),
           "pct_of_8TBps": round(100.0 * gbs / 8000.0, 2), "frac_hbm": round(gbs / hbm_peak, 4),
           "flops": fl, "TFLOPs": round(tfs, 1), "frac_bf16": round(tfs / bf16_peak, 4),
           "bound": "tensor" if fl / nb > 300 else "hbm", "status": int(st.dev_status.item())}
    del sets, base, g
    torch.cuda.empty_cache()
    return out


def time_attention_batch(B, stream, K, hbm_peak, seed=11, splits=0):
    """et_tree_attention alone at the batched sweep's shape: B sequences of
    7B heads (32 x 128, bf16) with ragged prefixes ~ U{512 .. 16384} (the
    workload's own seeded lengths) and an EAGLE-2-sized tree of n = 60 each.
    Q/K/V are N(0,1) drawn on the device (the timing needs no oracle); the
    mask comes from et_tree_mask_posids on a seeded random tree (parent of
    row i drawn from rows < i).  The standalone split plan; a graph of K
    launches over inputs far larger than L2."""
    import numpy as np
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS["sweep-7b"].with_(B=B)
    cfg = E.TreeCfg(B=B, V=wl.V, depth=wl.depth, topk=wl.topk, m=wl.m, n=wl.n, temperature=1.0)
    N = cfg.N
    prefix = W.prefix_lengths(wl, B)
    kv_row0 = np.concatenate([[0], np.cumsum(wl.Hkv * prefix.astype(np.int64))[:-1]]).astype(np.int64)
    rows = int(wl.Hkv * prefix.astype(np.int64).sum())
    gen = torch.Generator(device="cuda").manual_seed(seed)
    bf = dict(dtype=torch.bfloat16, device="cuda", generator=gen)
    q = torch.randn((B, N, wl.Hq, wl.d), **bf)
    kp = torch.randn((rows, wl.d), **bf)
    vp = torch.randn((rows, wl.d), **bf)
    kt = torch.randn((B, N, wl.Hkv, wl.d), **bf)
    vt = torch.randn((B, N, wl.Hkv, wl.d), **bf)
    rng = np.random.default_rng(seed)
    par = np.full((B, N), -1, np.int32)
    dep = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            par[b, i] = rng.integers(0, i)
            dep[b, i] = dep[b, par[b, i]] + 1
    tree = E.TreeBuffers.allocate(cfg)
    tree.flat_parent.copy_(torch.from_numpy(par))
    tree.flat_depth.copy_(torch.from_numpy(dep))
    plen = torch.from_numpy(prefix).cuda()
    row0 = torch.from_numpy(kv_row0).cuda()
    mask = torch.zeros((B, N, (N + 63) // 64), dtype=torch.int64, device="cuda")
    posids = torch.zeros((B, N), dtype=torch.int32, device="cuda")
    E.et_tree_mask_posids(cfg, tree, plen, mask, posids)
    shape = E.AttnShape(B=B, N=N, Hq=wl.Hq, Hkv=wl.Hkv, d=wl.d, dtype=E.ET_BF16, scale=wl.d ** -0.5,
                        max_prefix=int(prefix.max()), kv_rows=rows, num_splits=splits)
    ws = E.new_workspace(E.et_tree_attention_workspace_size(shape))
    out = torch.zeros((B, N, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, wl.Hq, N), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    call = lambda: E.et_tree_attention(shape, q, kp, vp, row0, plen, kt, vt, mask, out, lse=lse, ws=ws,
                                       dev_status=status, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            call()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    nbytes = attention_bytes(wl, prefix)
    gbps = nbytes / (us * 1e-6) / 1e9
    res = {"workload": "sweep-7b", "batch": B, "prefix_mean": round(float(prefix.mean()), 1),
           "prefix_min": int(prefix.min()), "prefix_max": int(prefix.max()),
           "splits": E.et_tree_attention_splits(shape), "us_per_launch": round(us, 3), "bytes": nbytes,
           "GBps": round(gbps, 1), "pct_of_8TBps": round(100 * gbps / 8000.0, 2),
           "frac_hbm": round(gbps / hbm_peak, 4), "bound": "hbm", "status": int(status.item())}
    del q, kp, vp, kt, vt, ws, out
    torch.cuda.empty_cache()
    return res


def sweep_logit_tables(wl, rows, gen, with_target=True):
    """Target and draft logit tables of `rows` nodes drawn on the device with
    the workload's recipe: target -slope * ln(rank) + N(0, 1) over a random
    permutation of the vocabulary per node, draft = target + N(0, sigma^2)."""
    import torch
    dev = dict(device="cuda", generator=gen)
    target = torch.empty((rows, wl.V), dtype=torch.float32, device="cuda")
    draft = torch.empty_like(target)
    by_rank = -wl.slope * torch.log(torch.arange(1, wl.V + 1, device="cuda", dtype=torch.float32))
    for r0 in range(0, rows, 256):
        r1 = min(rows, r0 + 256)
        perm = torch.argsort(torch.rand((r1 - r0, wl.V), **dev), dim=1)  # the token at each rank
        z = by_rank.expand(r1 - r0, -1) + torch.randn((r1 - r0, wl.V), **dev)
        target[r0:r1].scatter_(1, perm, z)
        draft[r0:r1] = target[r0:r1] + wl.sigma * torch.randn((r1 - r0, wl.V), **dev)
        del perm, z
    if not with_target:
        del target
        return None, draft
    return target, draft


def time_tree_batch(B, stream, K, hbm_peak, seed=23, per_layer=False):
    """et_tree_build alone at the batched sweep's shape (B sequences, V =
    32000, depth 6, top-k 10, m 10, n 60; draft logits drawn on the device
    as in the sweep step, about 2 GB at B = 32): a graph of one build
    replayed K times (per_layer: D et_tree_expand launches and
    et_tree_rerank_mask instead).  The algorithmic bytes are the expanded
    rows' logits (B * sum of m_l rows of V fp32) -- the rerank reads a few
    KB."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import step as S
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS["sweep-7b"].with_(B=B)
    st = S.VerifyStep(wl, per_layer=per_layer)
    cfg, R = st.cfg, st.C + 1
    gen = torch.Generator(device="cuda").manual_seed(seed)
    _, draft = sweep_logit_tables(wl, B * R, gen, with_target=False)
    row_of_node = (torch.arange(B, dtype=torch.int32, device="cuda")[:, None] * R
                   + torch.arange(R, dtype=torch.int32, device="cuda")[None, :]).contiguous()
    prefix = torch.from_numpy(W.prefix_lengths(wl, B)).cuda()
    st.tree.root_tok = torch.from_numpy(W.root_tokens(wl, B)).cuda()
    inp = S.StepInputs(draft=draft, target=None, row_of_node=row_of_node, root_tok=st.tree.root_tok,
                       prefix_len=prefix, kv_row0=None, q=None, k_prefix=None, v_prefix=None, k_tree=None,
                       v_tree=None, uniforms=None, host={})
    call = lambda: st.build_tree(inp, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(K):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    rows = B * sum(E.et_layer_expanded(cfg, l) for l in range(cfg.depth))
    tb = rows * wl.V * 4
    res = {"workload": "sweep-7b", "batch": B, "us_per_tree": round(us, 2), "launches": st.launches() - 2,
           "rows_expanded": rows, "logit_bytes": tb, "GBps": round(tb / (us * 1e-6) / 1e9, 1),
           "frac_of_measured_hbm": round(tb / (us * 1e-6) / 1e9 / hbm_peak, 4), "replays": K,
           "status": int(st.dev_status.item())}
    del draft, st
    torch.cuda.empty_cache()
    return res


def time_accept_batch(B, stream, K, hbm_peak, seed=23):
    """et_verify_accept alone (point-mass) at the batched sweep's shape: the
    tree is built once from the sweep's device-drawn draft logits, then a
    graph of one acceptance call is replayed K times over the target table.
    The algorithmic bytes are the logit rows on the accepted paths plus the
    stop rows (at most D + 1 rows of V fp32 per sequence)."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import step as S
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS["sweep-7b"].with_(B=B)
    st = S.VerifyStep(wl)
    cfg, R, N = st.cfg, st.C + 1, st.cfg.N
    gen = torch.Generator(device="cuda").manual_seed(seed)
    target, draft = sweep_logit_tables(wl, B * R, gen)
    row_of_node = (torch.arange(B, dtype=torch.int32, device="cuda")[:, None] * R
                   + torch.arange(R, dtype=torch.int32, device="cuda")[None, :]).contiguous()
    prefix = torch.from_numpy(W.prefix_lengths(wl, B)).cuda()
    inp = S.StepInputs(draft=draft, target=target, row_of_node=row_of_node,
                       root_tok=torch.from_numpy(W.root_tokens(wl, B)).cuda(), prefix_len=prefix, kv_row0=None,
                       q=None, k_prefix=None, v_prefix=None, k_tree=None, v_tree=None,
                       uniforms=torch.rand((B, N), device="cuda", generator=gen), host={})
    st.build_tree(inp, stream=stream)
    call = lambda: st.accept(inp, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(K):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    acc = st.accept_len.cpu()
    rows = int((acc + 1).clamp(max=wl.depth + 1).sum())  # the path rows and each stop row
    pb = rows * wl.V * 4
    res = {"workload": "sweep-7b", "batch": B, "accept": "stoch_point", "us_per_call": round(us, 2),
           "mean_accept_len": round(float(acc.float().mean()), 3), "rows_on_paths": rows, "path_bytes": pb,
           "GBps": round(pb / (us * 1e-6) / 1e9, 1), "replays": K, "status": int(st.dev_status.item())}
    del inp, target, draft, st
    torch.cuda.empty_cache()
    return res


def time_sweep_step(B, stream, K, hbm_peak, seed=23, n=None):
    """The whole verification step at the batched sweep's shape: B sequences
    of 7B heads with ragged prefixes ~ U{512 .. 16384} (the workload's seeded
    lengths), EAGLE-2 trees of depth 6, top-k 10, m 10, n 60, point-mass
    stochastic acceptance.  The inputs follow the same recipe as the seeded
    host generators but are drawn on the device (about 9 GB at B = 32, which
    the host would take minutes to write): target logits -slope * ln(rank) +
    N(0, 1) over a random permutation of the vocabulary per node, draft =
    target + N(0, sigma^2), Q/K/V ~ N(0, 1) in bf16.  One CUDA graph per
    step, replayed K times over inputs far larger than L2; each call also
    timed alone."""
    import numpy as np
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import step as S
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS["sweep-7b"].with_(B=B)
    if n is not None:
        wl = wl.with_(n=n)
    st = S.VerifyStep(wl)
    cfg, C = st.cfg, st.C
    R, N = C + 1, cfg.N
    gen = torch.Generator(device="cuda").manual_seed(seed)
    target, draft = sweep_logit_tables(wl, B * R, gen)
    prefix = W.prefix_lengths(wl, B)
    kv_row0 = np.concatenate([[0], np.cumsum(wl.Hkv * prefix.astype(np.int64))[:-1]]).astype(np.int64)
    kv_rows = int(wl.Hkv * prefix.astype(np.int64).sum())
    bf = dict(dtype=torch.bfloat16, device="cuda", generator=gen)
    inp = S.StepInputs(
        draft=draft, target=target,
        row_of_node=(torch.arange(B, dtype=torch.int32, device="cuda")[:, None] * R
                     + torch.arange(R, dtype=torch.int32, device="cuda")[None, :]).contiguous(),
        root_tok=torch.from_numpy(W.root_tokens(wl, B)).cuda(),
        prefix_len=torch.from_numpy(prefix).cuda(), kv_row0=torch.from_numpy(kv_row0).cuda(),
        q=torch.randn((B, N, wl.Hq, wl.d), **bf), k_prefix=torch.randn((kv_rows, wl.d), **bf),
        v_prefix=torch.randn((kv_rows, wl.d), **bf), k_tree=torch.randn((B, N, wl.Hkv, wl.d), **bf),
        v_tree=torch.randn((B, N, wl.Hkv, wl.d), **bf),
        uniforms=torch.rand((B, N), device="cuda", generator=gen), host={"prefix_len": prefix})
    st.prepare(inp)
    cur = torch.cuda.current_stream()

    def graph_us(call):
        with torch.cuda.stream(stream):
            for _ in range(2):
                call()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            call()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(K):
            g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / K

    step_us = graph_us(lambda: st.run(inp, stream=stream))
    tree_us = graph_us(lambda: st.build_tree(inp, stream=stream))
    attn_us = graph_us(lambda: st.attention(inp, stream=stream))
    accept_us = graph_us(lambda: st.accept(inp, stream=stream))
    attn_b = attention_bytes(wl, prefix)
    res = {"workload": "sweep-7b", "batch": B, "n": cfg.n, "prefix_mean": round(float(prefix.mean()), 1),
           "accept": "stoch_point", "ms_per_step": round(step_us / 1000.0, 4),
           "steps_per_s": round(1e6 / step_us, 1), "sequences_per_s": round(B * 1e6 / step_us, 1),
           "tree_launches": st.launches() - 2, "attention_splits": E.et_tree_attention_splits(st.shape),
           "calls_alone_us": {"tree": round(tree_us, 2), "attention": round(attn_us, 2),
                              "accept": round(accept_us, 2)},
           "attention_GBps": round(attn_b / (attn_us * 1e-6) / 1e9, 1),
           "attention_pct_of_8TBps": round(100 * attn_b / (attn_us * 1e-6) / 8e12, 2),
           "inputs": "drawn on the device with the workload's recipe", "status": int(st.dev_status.item())}
    del inp, target, draft, st
    torch.cuda.empty_cache()
    return res


def E_splits(st):
    from speculative_decoding_eagle_gb300 import binding as E
    return E.et_tree_attention_splits(st.shape)


def time_kv_commit(st, inp, wl, cfg, prefix, stream, K):
    """et_kv_commit of the accepted paths of one step into caches with room
    for them; algorithmic bytes = read + write of the committed K/V rows."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    B, Hkv, d = cfg.B, wl.Hkv, wl.d
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    cap = int(prefix.max()) + wl.depth + 1
    kc = torch.zeros((B * Hkv * cap, d), dtype=dt, device="cuda")
    vc = torch.zeros_like(kc)
    kv_row0 = torch.arange(B, dtype=torch.int64, device="cuda") * Hkv * cap
    new_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    shape = E.CommitShape(B=B, N=cfg.N, Hkv=Hkv, d=d, path_len=wl.depth + 1,
                          dtype=E.ET_BF16 if wl.dtype == "bf16" else E.ET_F32, kv_head_stride=cap,
                          kv_rows=B * Hkv * cap)
    with torch.cuda.stream(stream):
        st.run(inp, stream=stream)
    stream.synchronize()

    def one():
        E.et_kv_commit(shape, inp.k_tree, inp.v_tree, st.accept_len, st.path, kc, vc, kv_row0, inp.prefix_len,
                       new_len, dev_status=st.dev_status, stream=stream)
    with torch.cuda.stream(stream):
        one()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            one()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    rows = int(st.accept_len.sum().item()) + B
    nbytes = rows * Hkv * d * kc.element_size() * 2 * 2
    return {"us_per_launch": round(us, 3), "rows_committed": rows, "bytes": nbytes,
            "GBps": round(nbytes / (us * 1e-6) / 1e9, 2), "bound": "latency (a few KB per sequence)"}


LM_HIDDEN = {"llama2-7b": 4096, "llama2-13b": 5120, "llama2-70b": 8192, "sweep-7b": 4096}


def time_lm_head(wl, cfg, stream, K, hbm_peak):
    """et_lm_head for one expansion layer (B x m feature rows) against a
    synthetic bf16 LM head [V, H]; two weight copies alternate so that every
    launch streams its weight from HBM (each is larger than L2)."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    H = LM_HIDDEN.get(wl.name)
    M = cfg.B * wl.m
    if H is None or M > 64:
        return None
    g = torch.Generator(device="cuda").manual_seed(0xEA61)
    ws = [(0.02 * torch.randn((wl.V, H), device="cuda", generator=g)).to(torch.bfloat16) for _ in range(2)]
    x = torch.randn((M, H), device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty((M, wl.V), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for w in ws:
            E.et_lm_head(x, w, out, dev_status=status, stream=stream)
    stream.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(K):
            E.et_lm_head(x, ws[i % 2], out, dev_status=status, stream=stream)
    gr.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    gr.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    nbytes = wl.V * H * 2 + M * H * 2 + M * wl.V * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    del ws
    return {"M": M, "H": H, "V": wl.V, "us_per_launch": round(us, 3), "bytes": nbytes, "GBps": round(gbs, 1),
            "frac": round(gbs / hbm_peak, 4), "bound": "hbm (weight streamed once)",
            "status": int(status.item())}


STATIC_WIDTHS = (4, 2, 2, 1, 1)  # 61 flat rows, the size of the 7B dynamic tree


def time_static_tree(wl, cfg, inp, stream, K):
    """et_static_tree over the step's draft table (one launch per step)."""
    import numpy as np
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import workloads as W
    if wl.V > 32768:
        return None
    parent, rank = W.static_shape(STATIC_WIDTHS)
    B, N = cfg.B, parent.size
    per_seq = inp.draft.shape[0] // B
    if per_seq < N:
        return None
    rmap = torch.from_numpy((np.arange(B)[:, None] * per_seq + np.arange(N)[None, :]).astype(np.int32)).cuda()
    tb = E.TreeBuffers.allocate_flat(B, N, root_tok=inp.root_tok)
    par_d, rank_d = torch.from_numpy(parent).cuda(), torch.from_numpy(rank).cuda()
    k = max(STATIC_WIDTHS)

    def one():
        E.et_static_tree(B, wl.V, k, par_d, rank_d, inp.draft, rmap, tb, stream=stream)
    with torch.cuda.stream(stream):
        one()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(K):
            one()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / K
    internal = int(np.unique(parent[1:]).size)
    nbytes = B * internal * wl.V * 4
    # children drawn from q = softmax(draft / T) instead of ranked (two launches)
    u = torch.rand((B, N), device="cuda", generator=torch.Generator(device="cuda").manual_seed(7))
    ws = E.new_workspace(E.load().et_static_tree_workspace_size(E.ctypes.byref(E.StaticCfgC(B, wl.V, N, 1, 1.0))))

    def drawn():
        E.et_static_tree_sampled(B, wl.V, 1.0, par_d, inp.draft, rmap, u, tb, ws=ws, stream=stream)
    with torch.cuda.stream(stream):
        drawn()
    stream.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        for _ in range(K):
            drawn()
    g2.replay()
    torch.cuda.synchronize()
    e0.record(cur)
    g2.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    us_s = e0.elapsed_time(e1) * 1000.0 / K
    return {"widths": list(STATIC_WIDTHS), "rows": N, "us_per_launch": round(us, 3), "bytes": nbytes,
            "GBps": round(nbytes / (us * 1e-6) / 1e9, 1), "sampled_us": round(us_s, 3), "bound": "latency at batch 1"}


def run_e2e(args, st, sets, wl, stream, host_tables=True):
    """Steps through the public API with the inputs in pinned host memory,
    each step reading its result (accept_len, path, tokens) device -> host.
    Double-buffered like a serving loop: step i+1's copies run on a copy
    stream while step i computes, and the host waits for step i-2 (whose
    buffers it reuses) before issuing step i.

    host_tables: the draft and target logit tables (one row per candidate
    node, 131 MB at the 7B shape) stay in pinned host memory and the tree
    build and the acceptance read only the rows they use over the host link
    (NVLink-C2C on Grace-Blackwell); everything else is copied each step.
    Otherwise every input is copied whole."""
    import dataclasses
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    names = ("draft", "target", "row_of_node", "root_tok", "prefix_len", "kv_row0", "q", "k_prefix", "v_prefix",
             "k_tree", "v_tree", "uniforms")
    tables = ("draft", "target") if host_tables else ()
    copied_names = tuple(n for n in names if n not in tables)
    nbuf = 2
    R = min(len(sets), 2)
    host = [{n: getattr(sets[r], n).cpu().pin_memory() for n in names} for r in range(R)]
    dev = [sets[0], sets[1] if len(sets) > 1 else sets[0]]
    if dev[1] is dev[0]:
        nbuf = 1
    # the inputs a step is given: device buffers, with the tables left in host memory
    step_in = [[dataclasses.replace(dev[k], **{n: host[r][n] for n in tables}) for r in range(R)]
               for k in range(2)]
    outs = [st.accept_len, st.path, st.tokens]
    host_out = [[t.cpu().pin_memory() for t in outs] for _ in range(2)]
    h2d = sum(host[0][n].numel() * host[0][n].element_size() for n in copied_names)
    cfg = st.cfg
    expanded_rows = cfg.B * sum(E.et_layer_expanded(cfg, l) for l in range(cfg.depth))
    path_rows = [0]  # target rows the acceptance walks read, summed over the consumed steps
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    K = max(3, min(20, args.steps))
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    issued = [False, False]

    def one(i):
        k = i % nbuf
        if issued[k]:
            done[k].synchronize()  # step i-2 finished: its device inputs and host result buffer are free
            path_rows[0] += int(host_out[k][0].sum()) + cfg.B  # the host consumes that step's result
        with torch.cuda.stream(copy_stream):
            for n in copied_names:
                getattr(dev[k], n).copy_(host[i % R][n], non_blocking=True)
            copied[k].record(copy_stream)
        with torch.cuda.stream(stream):
            stream.wait_event(copied[k])
            st.run(step_in[k][i % R], stream=stream)
            for d, hh in zip(outs, host_out[k]):
                hh.copy_(d, non_blocking=True)
            done[k].record(stream)
        issued[k] = True

    # warm-up: with the tables in host memory, one untimed pass of K steps (the GPU's first reads of
    # freshly pinned pages run about twice as slow until their translations are cached)
    for i in range(K if host_tables else 2):
        one(i)
    torch.cuda.synchronize()
    issued[:] = [False, False]
    path_rows[0] = 0
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(copy_stream)
    for i in range(K):
        one(i)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(e0.elapsed_time(e1), wall * 1000.0) / K
    consumed = K - min(K, nbuf)  # steps whose result the loop read back before the last ones
    table_bytes = 0
    if host_tables and consumed > 0:
        # every expanded draft row; the target rows on the walked paths (8 or more sequences) or every flat row
        target_rows = path_rows[0] / consumed if cfg.B >= 8 else cfg.B * cfg.N
        table_bytes = int((expanded_rows + target_rows) * wl.V * 4)
    out = {"value": round(1000.0 / ms, 2), "unit": "steps/s", "h2d_bytes_per_step": int(h2d + table_bytes),
           "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4), "steps": K,
           "h2d_GBps": round((h2d + table_bytes) / (ms * 1e-3) / 1e9, 1)}
    if host_tables:
        out["copied_bytes_per_step"] = int(h2d)
        out["table_rows_read_bytes_per_step"] = int(table_bytes)
        out["pipeline"] = ("logit tables stay in pinned host memory, the kernels read the rows they use over the "
                           "host link; the other inputs of step i+1 copy while step i computes (two device sets)")
    else:
        out["pipeline"] = "every input of step i+1 copies while step i computes (two device input sets)"
    return out


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    from speculative_decoding_eagle_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    times = []
    base = None
    for i in range(args.warmup + args.steps):
        r = oracle_baseline(wl.name, budget_s=max(1.0, 20.0 / max(1, args.steps + args.warmup)), max_steps=2)
        if i >= args.warmup:
            times.append(1.0 / r["value"])
            base = r
    v = len(times) / sum(times)
    out = {"impl": "reference", "metric": "tree-verify steps/s (1 GB300, batch 1) with tree-attention HBM GB/s",
           "value": round(v, 4), "unit": "steps/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1000.0 / v, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": wl.name, "batch": 1, "V": wl.V, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                      "prefix": int(wl.prefix), "depth": wl.depth, "topk": wl.topk, "m": wl.m, "n": wl.n,
                      "accept": "greedy" if "greedy" in wl.accept else "stoch_point",
                      "parallelism": f"replicas x{world}"},
           "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": base["sample"] if base else "",
                            "value": round(v, 4)},
           "e2e": {"value": round(v, 4), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_split_sweep(args):
    """Attention alone at each KV split count: one JSON line per count (a
    tuning aid; the step's own plan picks the count by default).  Timing as in
    the step bench: CUDA events around a graph of K launches over input sets
    that together exceed L2."""
    import numpy as np
    import torch
    from speculative_decoding_eagle_gb300 import binding as E, build_lib, step as S
    from speculative_decoding_eagle_gb300 import workloads as W
    build_lib.build()
    E.load()
    wl = W.WORKLOADS[args.workload]
    if args.batch:
        wl = wl.with_(B=args.batch)
    if args.prefix:
        wl = wl.with_(prefix=args.prefix, ragged=False)
    st0 = S.VerifyStep(wl)
    cfg = st0.cfg
    prefix = W.prefix_lengths(wl, cfg.B)
    abytes = attention_bytes(wl, prefix)
    R = args.sets or max(2, int(np.ceil(2 * L2_BYTES / abytes)) + 1)
    sets = [S.to_device(wl, S.host_inputs(wl, st0.C, cfg.B, b0=r * cfg.B)) for r in range(R)]
    K = max(8, min(200, args.steps))
    stream = torch.cuda.Stream()
    for splits in [int(x) for x in args.splits_sweep.split(",")]:
        st = S.VerifyStep(wl, num_splits=splits, attn_impl=E.ATTN_TCGEN05, overlap=False)
        st.prepare(sets[0])
        with torch.cuda.stream(stream):
            for r in range(R):
                st.run(sets[r], stream=stream)  # trees and masks of every set
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(K):
                st.attention(sets[i % R], stream=stream)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()  # a graph replays on the current stream
        e0.record(cur)
        g.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000.0 / K
        print(json.dumps({"workload": wl.name, "batch": cfg.B, "prefix": int(max(prefix)), "splits": splits,
                          "splits_used": E.et_tree_attention_splits(st.shape), "us_per_launch": round(us, 2),
                          "GBps": round(abytes / us / 1e3, 1), "launches": K, "input_sets": R}), flush=True)


def extras_sections(args, K, hbm_peak, bf16_peak):
    """The bench line's secondary measurements (each guarded: an error is
    reported in its entry): attention alone at the other target shapes, at
    the batched sweep's shape, and the batched sweep's whole step."""
    import torch
    stream = torch.cuda.Stream()
    shapes, batched, sweep = [], [], []
    for name, L in ATTN_SHAPES:
        try:
            shapes.append(time_attention_shape(name, L, stream, K, hbm_peak, bf16_peak))
        except Exception as ex:  # report, keep the rest
            print(f"attention at {name}, prefix {L}: {ex!r}", file=sys.stderr, flush=True)
            shapes.append({"workload": name, "prefix": L, "error": str(ex)[:300]})
    for Bs in (16, 32):
        try:
            batched.append(time_attention_batch(Bs, stream, max(4, min(20, K)), hbm_peak))
        except Exception as ex:  # report, keep the rest
            print(f"batched attention, batch {Bs}: {ex!r}", file=sys.stderr, flush=True)
            batched.append({"workload": "sweep-7b", "batch": Bs, "error": str(ex)[:300]})
    # the sweep's grid: batches at the kept-tree size n = 60 and other sizes at batch 16; batch 32 last
    for Bs, n in ((1, 60), (4, 60), (16, 60), (16, 16), (16, 32), (16, 100), (32, 60)):
        try:
            sweep.append(time_sweep_step(Bs, stream, max(3, min(10, K)), hbm_peak, n=n))
        except Exception as ex:  # report, keep the rest
            print(f"sweep step, batch {Bs}, n {n}: {ex!r}", file=sys.stderr, flush=True)
            sweep.append({"workload": "sweep-7b", "batch": Bs, "n": n, "error": str(ex)[:300]})
    return {"tree_attention_shapes": shapes, "tree_attention_batched": batched, "sweep_step": sweep}


def run_extras(args):
    """--extras: the secondary sections alone, one JSON line (the child process of the main bench)."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    torch.cuda.set_device(0)
    hbm_peak, bf16_peak, _ = _peaks()
    print(json.dumps(extras_sections(args, max(8, min(200, args.steps)), hbm_peak, bf16_peak)), flush=True)


def run_extras_child(args):
    """Runs --extras in a child process on the same GPU and returns its sections; a child that fails
    leaves an error entry in each section instead of ending the bench."""
    cmd = [sys.executable, os.path.abspath(__file__), "--extras", "--steps", str(args.steps)]
    env = dict(os.environ)
    try:
        p = subprocess.run(cmd, capture_output=True, text=True, timeout=1200, env=env)
        lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
        if p.returncode == 0 and lines:
            sys.stderr.write(p.stderr[-2000:])
            return json.loads(lines[-1])
        err = f"child exited {p.returncode}: {p.stderr.strip()[-300:]}"
    except Exception as ex:
        err = f"child failed: {ex!r}"[:300]
    print(err, file=sys.stderr, flush=True)
    return {"tree_attention_shapes": [{"error": err}], "tree_attention_batched": [{"error": err}],
            "sweep_step": [{"error": err}]}


def run_attn_batch(args):
    """Attention alone at the batched sweep's shape (one JSON line); the
    command the batched attention's ncu summary is captured from."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    torch.cuda.set_device(0)
    hbm_peak, _, _ = _peaks()
    res = time_attention_batch(args.attn_batch, torch.cuda.Stream(), max(4, min(20, args.steps)), hbm_peak,
                               splits=args.splits)
    print(json.dumps(res))


def run_tree_batch(args):
    """The tree build alone at the batched sweep's shape (one JSON line); the
    command the batched expansion's ncu summary is captured from."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    torch.cuda.set_device(0)
    hbm_peak, _, _ = _peaks()
    E.et_set_expand_kernel({"auto": E.ET_EXPAND_AUTO, "cluster": E.ET_EXPAND_CLUSTER,
                            "block": E.ET_EXPAND_BLOCK}[args.expand_kernel])
    res = time_tree_batch(args.tree_batch, torch.cuda.Stream(), max(4, min(50, args.steps)), hbm_peak,
                          per_layer=args.per_layer)
    res["expand_kernel"] = args.expand_kernel
    res["per_layer"] = bool(args.per_layer)
    print(json.dumps(res))


def run_sweep_batch(args):
    """The batched sweep's whole step at one batch (and --sweep-n kept-tree size), one JSON line; the
    command the sweep step's launch list is captured from."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    torch.cuda.set_device(0)
    hbm_peak, _, _ = _peaks()
    print(json.dumps(time_sweep_step(args.sweep_batch, torch.cuda.Stream(), max(3, min(10, args.steps)), hbm_peak,
                                     n=args.sweep_n or None)))


def run_accept_batch(args):
    """Acceptance alone at the batched sweep's shape (one JSON line); the
    command the batched acceptance's ncu summary is captured from."""
    import torch
    from speculative_decoding_eagle_gb300 import binding as E
    from speculative_decoding_eagle_gb300 import build_lib
    build_lib.build()
    E.load()
    torch.cuda.set_device(0)
    hbm_peak, _, _ = _peaks()
    print(json.dumps(time_accept_batch(args.accept_batch, torch.cuda.Stream(), max(4, min(50, args.steps)), hbm_peak)))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--mode", default="auto", choices=["auto", "greedy", "stoch", "draftq"])
    ap.add_argument("--prefix", type=int, default=0, help="override the workload's KV-prefix length")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--attn", default="auto", choices=["auto", "mma", "tcgen05"], help="attention kernel")
    ap.add_argument("--sets", type=int, default=0)
    ap.add_argument("--eager", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-attn-shapes", action="store_true", help="skip timing attention at the other target shapes")
    ap.add_argument("--clocks-csv", default="", help="also write the raw nvidia-smi samples of the timed region here")
    ap.add_argument("--splits-sweep", default="", help="comma-separated KV split counts: time attention alone at each")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per attention launch from an ncu capture of the same kernel")
    ap.add_argument("--attn-batch", type=int, default=0,
                    help="only time attention alone at the batched sweep's shape with this batch (one JSON line)")
    ap.add_argument("--tree-batch", type=int, default=0,
                    help="only time the tree build alone at the batched sweep's shape with this batch (one JSON line)")
    ap.add_argument("--expand-kernel", default="auto", choices=["auto", "cluster", "block"],
                    help="expansion row code (et_set_expand_kernel)")
    ap.add_argument("--extras", action="store_true",
                    help="only the secondary sections (other attention shapes, batched attention, sweep steps)")
    ap.add_argument("--sweep-batch", type=int, default=0,
                    help="only the batched sweep's whole step at this batch (one JSON line)")
    ap.add_argument("--sweep-n", type=int, default=0, help="with --sweep-batch: the kept-tree size n")
    ap.add_argument("--accept-batch", type=int, default=0,
                    help="only time the acceptance alone at the batched sweep's shape with this batch (one JSON line)")
    ap.add_argument("--per-layer", action="store_true",
                    help="with --tree-batch: the tree as D et_tree_expand launches and the rerank")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.splits_sweep:
        run_split_sweep(args)
    elif args.attn_batch:
        run_attn_batch(args)
    elif args.tree_batch:
        run_tree_batch(args)
    elif args.accept_batch:
        run_accept_batch(args)
    elif args.sweep_batch:
        run_sweep_batch(args)
    elif args.extras:
        run_extras(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
