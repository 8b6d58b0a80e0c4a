#!/usr/bin/env python
"""Benchmark: prefix-tree attention forward + backward, useful TFLOP/s.

A step is one pass of the whole path over one batch of synthetic input:
block map from the tree (labels + tile classes + lists), forward (O, LSE) and
backward (Delta preprocess, dK/dV, dQ).  Useful work per step is
4*D*Hq*pairs (forward) + 10*D*Hq*pairs (backward), where pairs is the number
of kept (q, kv) token pairs per head; masked pairs inside partial tiles are
not counted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C] [--impl ours|reference]

One JSON line is printed by rank 0.  Multi-GPU runs (torchrun, one process
per GPU) run one replica of the workload per GPU: the groups of the path are
independent, so nothing is exchanged on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefix-tree attn fwd+bwd useful TFLOP/s (unmasked pairs), % of bf16 peak"
L2_FLUSH_BYTES = 256 << 20


def draft_pairs(st) -> int:
    """Kept (q, kv) pairs per head of a draft-block layout: per kept block and
    token k, the context of the anchor's document before the anchor (within
    the window of real position anchor + k, if any), plus the block itself
    (k + 1 tokens when causal, all of it otherwise)."""
    import numpy as np

    total = 0
    S, bs = int(st.ctx_len), int(st.block_size)
    for b, a in enumerate(int(x) for x in st.anchors):
        if st.block_keep is not None and not st.block_keep[b]:
            continue
        lo, hi = 0, a
        if st.ctx_doc is not None:
            idx = np.nonzero(np.asarray(st.ctx_doc) == st.anchor_doc[b])[0]
            lo, hi = (int(idx[0]), min(int(idx[-1]) + 1, a)) if idx.size else (0, 0)
            if lo >= hi:
                lo = hi = 0
        for k in range(bs):
            c0 = max(lo, a + k - st.window + 1) if st.window > 0 else lo
            total += max(hi - c0, 0) + (k + 1 if st.causal else bs)
    return total


def useful_pairs(st) -> int:
    """Kept (q, kv) pairs per head, from the tree: each node's own causal
    triangle plus its tokens times all ancestor tokens (draft-block layouts:
    draft_pairs)."""
    if hasattr(st, "anchors"):
        return draft_pairs(st)
    parent = {}
    for p in st.paths():
        for a, b in zip(p[:-1], p[1:]):
            parent[b] = a
    total = 0
    for n, ln in enumerate(int(x) for x in st.node_lengths):
        anc = 0
        a = parent.get(n)
        while a is not None:
            anc += int(st.node_lengths[a])
            a = parent.get(a)
        total += ln * (ln + 1) // 2 + ln * anc
    return total


# DRAM bytes (read + write) per launch of the tensor-core kernels, from one
# `ncu --set full` capture of the current kernels on each workload (the
# per-kernel counter summaries under profiles/).  A kernel changed since its
# capture must be removed from this table (its traffic is then reported null).
MEASURED_TRAFFIC = {
    (2, "fwd_tc"): 35.06e6, (2, "bwd_fused"): 253.6e6,
    (3, "fwd_tc"): 927.5e6, (3, "bwd_dkdv"): 3435e6, (3, "bwd_dq"): 1186e6,
    (7, "fwd_tc"): 351.3e6,
}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank runs the same per-GPU workload (replicas,
    weak scaling), so the job processes world x the units of one rank in the
    slowest rank's time."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM (4 sub-partitions x 32)
SM_MAX_GHZ = 2.07  # maximum SM clock of the GB300


def num_sms() -> int:
    import torch

    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def euler_intervals(st):
    """Pre-order index (tin) and end of subtree (tout) of every node, children in id order."""
    import numpy as np

    n = int(st.node_lengths.size)
    parent = [-1] * n
    for p in st.paths():
        for a, b in zip(p[:-1], p[1:]):
            parent[b] = a
    children = [[] for _ in range(n)]
    for i in range(n):
        if parent[i] >= 0:
            children[parent[i]].append(i)
    tin = np.zeros(n, np.int64)
    tout = np.zeros(n, np.int64)
    counter = 0
    stack = [(r, False) for r in reversed([i for i in range(n) if parent[i] < 0])]
    while stack:
        u, done = stack.pop()
        if done:
            tout[u] = counter
            continue
        tin[u] = counter
        counter += 1
        stack.append((u, True))
        stack.extend((c, False) for c in reversed(children[u]))
    return tin, tout


def dense_keep_mask(st, device):
    """[T, T] bool: row q keeps column k when k's node is q's node or an ancestor of it (k's pre-order
    interval holds q's) and k <= q in the flat order."""
    import numpy as np
    import torch

    tin, tout = euler_intervals(st)
    node_of = np.repeat(np.arange(st.node_lengths.size), st.node_lengths)
    ti = torch.as_tensor(tin[node_of], device=device)
    to = torch.as_tensor(tout[node_of], device=device)
    idx = torch.arange(int(node_of.size), device=device)
    return (ti[None, :] <= ti[:, None]) & (ti[:, None] < to[None, :]) & (idx[None, :] <= idx[:, None])


def sdpa_dense_mask(st, Q, K, V, dO, steps):
    """torch scaled_dot_product_attention forward + backward with the dense [T, T] keep mask."""
    import torch
    import torch.nn.functional as F

    mask = dense_keep_mask(st, Q.device)
    T = Q.shape[0]
    q4, k4, v4, g4 = (x.transpose(0, 1).unsqueeze(0).contiguous() for x in (Q, K, V, dO))
    q4.requires_grad_()
    k4.requires_grad_()
    v4.requires_grad_()

    def one():
        q4.grad = k4.grad = v4.grad = None
        o = F.scaled_dot_product_attention(q4, k4, v4, attn_mask=mask, enable_gqa=True)
        o.backward(g4)

    one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    return {"ms_per_step": a.elapsed_time(b) / steps, "what": "torch SDPA forward + backward, dense bool mask, "
            f"GQA, same inputs (torch {torch.__version__})", "mask_mb": T * T / 1e6}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"pt_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names[1:], parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def cpu_oracle_run(st, cfg, seed, max_units=None):
    """Run the fp64 oracle forward + backward on a prefix of the workload's
    independent units (whole groups / documents) and return (useful flops, seconds,
    threads, description)."""
    from oracle import oracle as orc
    from prefix_tree_block_gb300 import workloads as W

    Hq, Hkv, D = cfg["Hq"], cfg["Hkv"], cfg["D"]
    if hasattr(st, "anchors"):  # draft blocks: the dense fp64 oracle on the first blocks
        from oracle import draft as odr

        nb = 64 if max_units is None else 16
        sub = W.DraftStructure(ctx_len=int(st.anchors[nb - 1]), anchors=st.anchors[:nb], block_size=st.block_size,
                               block_keep=None if st.block_keep is None else st.block_keep[:nb],
                               causal=st.causal, window=st.window,
                               ctx_doc=None if st.ctx_doc is None else st.ctx_doc[:int(st.anchors[nb - 1])],
                               anchor_doc=None if st.anchor_doc is None else st.anchor_doc[:nb])
        q, k, v, do = W.make_tensors(sub.T, Hq, Hkv, D, cfg["dtype"], seed)
        mask = odr.draft_mask(**sub.kwargs())
        t0 = time.perf_counter()
        odr.masked_attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), mask)
        odr.masked_attn_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), do.double().numpy(), mask)
        dt = time.perf_counter() - t0
        flops = 14.0 * D * Hq * useful_pairs(sub)
        what = (f"fp64 dense-mask oracle forward+backward (numpy, BLAS on all cores) over the first {nb} of "
                f"{st.anchors.size} blocks (T={sub.T}), all {Hq} heads")
        return flops, dt, os.cpu_count() or 1, what
    if "group_specs" in st.meta:
        specs = st.meta["group_specs"][: max_units or len(st.meta["group_specs"])]
        sub = W.grpo_structure(specs)
        what = f"{len(specs)} of {len(st.meta['group_specs'])} groups"
    elif "doc_lengths" in st.meta:
        docs = st.meta["doc_lengths"][: max_units or len(st.meta["doc_lengths"])]
        sub = W.docs_structure(docs)
        what = f"{len(docs)} of {len(st.meta['doc_lengths'])} documents"
    else:
        sub = st
        what = "the whole tree"
    q, k, v, do = W.make_tensors(sub.T, Hq, Hkv, D, cfg["dtype"], seed)
    lab = orc.structure_labels(sub)
    nth = orc.default_threads()
    t0 = time.perf_counter()
    orc.attn_fwd(q, k, v, lab, n_threads=nth)
    orc.attn_bwd(q, k, v, do, lab, n_threads=nth)
    dt = time.perf_counter() - t0
    flops = 14.0 * D * Hq * useful_pairs(sub)
    return flops, dt, nth, f"fp64 oracle forward+backward over {what} (T={sub.T}) of the workload, all {Hq} heads"


def run_reference(args, cfg, st):
    """The reference arm: the fp64 CPU oracle, timed on this host's cores, on
    a bounded sample (one group) per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_oracle_run(st, cfg, args.workload, max_units=1)
    flops = secs = 0.0
    desc, nth = "", 1
    for _ in range(args.steps):
        f, s, nth, desc = cpu_oracle_run(st, cfg, args.workload, max_units=1)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg["name"], "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_device(workload, steps, warmup, with_dense, flush, dist, local, world):
    """Device-resident measurement of one workload: the step (map build from
    the host layout, forward, backward) timed over `steps` steps with the L2
    flushed before each, the per-kernel durations from a second timed pass,
    forward and backward fractions of the bf16 peak, the roofline of the
    dominant kernel and the dense-masked comparison."""
    import torch

    import prefix_tree_block_gb300 as pt
    from prefix_tree_block_gb300 import workloads as W

    cfg = dict(W.CONFIGS[workload])
    st = W.config_structure(workload)
    Hq, Hkv, D, dtype = cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["dtype"]
    T = st.T
    pairs = useful_pairs(st)
    flops_fwd = 4.0 * D * Hq * pairs
    flops_step = flops_fwd * 3.5
    q, k, v, do = W.make_tensors(T, Hq, Hkv, D, dtype, workload)
    dev = torch.device("cuda", local)
    Q, K, V, dO = (x.to(dev) for x in (q, k, v, do))
    O = torch.empty_like(Q)
    LSE = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    ws = torch.empty(pt.bwd_workspace_bytes(T, Hq, D), dtype=torch.uint8, device=dev)
    draft = hasattr(st, "anchors")
    if draft:
        host_layout = [a for a in (st.anchors, st.block_keep, st.ctx_doc, st.anchor_doc) if a is not None]
        make_map = lambda: pt.build_blockmap_draft(**st.kwargs())
    else:
        nl, pp, pn = st.node_lengths, st.path_ptr, st.path_nodes
        host_layout = [nl, pp, pn]
        make_map = lambda: pt.build_blockmap_tree(nl, pp, pn, 128, 128)
    stream = torch.cuda.current_stream()

    def step(dense=False):
        bm = make_map()
        if dense:
            d = bm.dense()
            bm.free()
            bm = d
        pt.attn_fwd(Q, K, V, bm, O=O, LSE=LSE)
        pt.attn_bwd(dO, Q, K, V, O, LSE, bm, dQ=dQ, dK=dK, dV=dV, workspace=ws)
        bm.free()

    for _ in range(warmup):
        step()
    pt.sync_status()

    def timed(n, fn):
        evs = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = pt.launch_count()
    pt.profile_reset()
    # the step time: no events inside the step (an event between two kernels
    # costs the launch overlap, about 3 us per boundary)
    times = timed(steps, step)
    launches = pt.launch_count() - launches0
    torch.cuda.synchronize()
    # per-kernel durations: the same K steps again, each kernel bracketed by
    # CUDA events on its stream
    pt.profile_enable(True)
    timed(steps, step)
    pt.profile_enable(False)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    pt.sync_status()
    total_ms = max_over_ranks(sum(times), dist, dev)
    ms_step = total_ms / steps
    value = whole_job_tflops(world, flops_step, steps, total_ms)

    kernels = {}
    for name in ("blockmap_classify", "blockmap_lists", "fwd_tc", "fwd_simt", "bwd_prep", "bwd_dkdv",
                 "bwd_dkdv_finalize", "bwd_fused", "bwd_fused_finalize", "bwd_dv", "bwd_dk", "bwd_dq", "bwd_simt"):
        n, ms = pt.profile_read(name)
        if n:  # (the per-kernel pass runs the same `steps` steps; some kernels launch several times a step)
            kernels[name] = {"launches": n, "ms_per_launch": ms / n, "ms_per_step": ms / steps}
    pt.profile_reset()

    # ---- forward and backward fractions, roofline of the dominant kernel ----
    peak_tf, peak_gbs, peak_src = peaks()
    fwd_ms = sum(kernels[k]["ms_per_step"] for k in ("fwd_tc", "fwd_simt") if k in kernels)
    bwd_ms = sum(kernels[k]["ms_per_step"] for k in kernels if k.startswith("bwd_"))
    fwd_tf = flops_fwd / (fwd_ms * 1e-3) / 1e12 if fwd_ms else None
    bwd_tf = 2.5 * flops_fwd / (bwd_ms * 1e-3) / 1e12 if bwd_ms else None
    # head_dim 512: each backward launch builds one 256-column half of its output and recomputes S
    # (and dP): S^T + half of dV = 3D, S^T + dP^T + half of dK (or S + dP + half of dQ) = 5D
    wide2 = D == 512
    per_launch_flops = {  # useful-pair flops of each kernel: 2D per pair and head for each of its products
        "fwd_tc": 4.0 * D * Hq * pairs,
        "bwd_dkdv": 8.0 * D * Hq * pairs,
        "bwd_fused": 10.0 * D * Hq * pairs,  # head_dim 64 one pass: S^T, dP^T, dV, dK, dQ
        "bwd_dv": (3.0 if wide2 else 4.0) * D * Hq * pairs,  # head_dim 256: S^T and dV
        "bwd_dk": (5.0 if wide2 else 6.0) * D * Hq * pairs,  # head_dim 256: S^T, dP^T and dK
        "bwd_dq": (5.0 if wide2 else 6.0) * D * Hq * pairs,
        # CUDA-core kernels (fp32 inputs, head dims without a tensor-core path): useful flops
        "fwd_simt": 4.0 * D * Hq * pairs,
        "bwd_simt": 10.0 * D * Hq * pairs,
    }
    tc = {k: v for k, v in kernels.items() if k in per_launch_flops}
    roofline = None
    if tc:
        dom = max(tc, key=lambda k: tc[k]["ms_per_step"])  # the most time per step
        ach = per_launch_flops[dom] / (tc[dom]["ms_per_launch"] * 1e-3) / 1e12
        if dom.endswith("_simt"):  # fp32 FMA pipes: SMs x 128 lanes x 2 flop x max SM clock
            fp32_peak = FP32_LANES_PER_SM * num_sms() * 2 * SM_MAX_GHZ / 1e3
            roofline = {"kernel": dom, "bound": "alu", "achieved": ach, "peak": fp32_peak, "unit": "TFLOP/s",
                        "frac": ach / fp32_peak, "traffic": None,
                        "peak_source": f"derived: {num_sms()} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2 flop x "
                                       f"{SM_MAX_GHZ} GHz"}
        else:
            roofline = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak_tf, "unit": "TFLOP/s",
                        "frac": ach / peak_tf, "traffic": MEASURED_TRAFFIC.get((workload, dom)),
                        "peak_source": f"{peak_src} bf16 burst"}

    # ---- HBM-bound kernels: algorithmic bytes per step against the measured copy peak ----
    mp = make_map()
    nnz, n_part = mp.nnz, mp.nnz - mp.n_full
    mp.free()
    tpad = -(-T // 128) * 128
    elt = 2 if dtype == "bf16" else 4
    fused = "bwd_fused" in kernels
    algo = {
        # dO and O read, LSE read, Delta and LSE*log2(e) written; with the one-pass
        # backward also its fp32 dQ accumulator zeroed
        "bwd_prep": 2 * T * Hq * D * elt + 4 * T * Hq + 8 * tpad * Hq + (4 * tpad * Hq * D if fused else 0),
        # the map: per listed tile its q-major and kv-major entries (18 B), 2 x 2 KB of
        # keep bits per partial tile; tree maps also the token table (8 B) and each
        # token's node (4 B)
        "blockmap": 18 * nnz + 4096 * n_part + (0 if draft else 12 * tpad),
    }
    if fused:  # the fp32 accumulator read, dQ written
        algo["bwd_fused_finalize"] = 4 * tpad * Hq * D + elt * T * Hq * D
    hbm = {"peak_gbs": peak_gbs}
    for name, nbytes in algo.items():
        if name == "blockmap":
            ms = sum(kernels[k]["ms_per_step"] for k in ("blockmap_classify", "blockmap_lists") if k in kernels)
        else:
            ms = kernels[name]["ms_per_step"] if name in kernels else 0.0
        if ms > 0:
            gbs = nbytes / (ms * 1e-3) / 1e9
            hbm[name] = {"algorithmic_bytes": int(nbytes), "ms": ms, "achieved_gbs": gbs, "frac_of_hbm": gbs / peak_gbs}

    # ---- dense-masked comparison (same kernels, every tile partial) ---------
    dense = None
    if with_dense:
        step(dense=True)
        dt = timed(max(2, min(5, steps)), lambda: step(dense=True))
        dense = {"ms_per_step": sum(dt) / len(dt), "speedup": (sum(dt) / len(dt)) / ms_step}
    pt.sync_status()
    out = {
        "workload": cfg["name"], "T": T, "useful_pairs_per_head": pairs, "useful_tflop_per_step": flops_step / 1e12,
        "steps": steps, "ms_per_step": ms_step, "value": value, "unit": "TFLOP/s",
        "frac_of_peak": value / world / peak_tf,
        "fwd": {"ms": fwd_ms, "tflops": fwd_tf, "frac_of_peak": fwd_tf / peak_tf if fwd_tf else None},
        "bwd": {"ms": bwd_ms, "tflops": bwd_tf, "frac_of_peak": bwd_tf / peak_tf if bwd_tf else None},
        "kernels": kernels, "roofline": roofline, "hbm": hbm, "dense_masked": dense, "gpu_launches": int(launches),
        "_ctx": {"tensors": (Q, K, V, dO, q, k, v, do), "grads": (dQ, dK, dV), "make_map": make_map,
                 "host_layout": host_layout, "stream": stream, "timed": timed},
    }
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2, help="workload 1..7 (default 2: GRPO batch)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true")
    ap.add_argument("--no-fold", action="store_true")
    ap.add_argument("--no-other-workloads", dest="all_workloads", action="store_false",
                    help="with the default workload 2, skip the workloads 3..7 section")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from prefix_tree_block_gb300 import workloads as W

    cfg = dict(W.CONFIGS[args.workload])
    st = W.config_structure(args.workload)
    if args.impl == "reference":
        run_reference(args, cfg, st)
        return

    import torch

    import prefix_tree_block_gb300 as pt
    from prefix_tree_block_gb300 import build as ptbuild

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        ptbuild.build()
    if dist is not None:
        dist.barrier()
    pt.load_library()

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=torch.device("cuda", local))
    sampler = ClockSampler(local)
    sampler.start()
    res = measure_device(args.workload, args.steps, args.warmup, not args.no_dense, flush, dist, local, world)
    ctx = res.pop("_ctx")
    # the other workloads of the set, in the same run: the same measurement
    # (fewer steps), each with its own inputs and map
    others = {}
    if args.all_workloads and args.workload == 2:
        for c in (3, 4, 5, 6, 7):
            n = max(3, min(args.steps, 20)) if c != 7 else 3
            r = measure_device(c, n, 3, c != 7 and not args.no_dense, flush, dist, local, world)
            r.pop("_ctx")
            others[str(c)] = r
            torch.cuda.empty_cache()
    clocks = sampler.stop()
    Q, K, V, dO, q, k, v, do = ctx["tensors"]
    dQ, dK, dV = ctx["grads"]
    make_map, host_layout, stream, timed = ctx["make_map"], ctx["host_layout"], ctx["stream"], ctx["timed"]
    Hq, Hkv, D, dtype = cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["dtype"]
    T = st.T
    draft = hasattr(st, "anchors")
    flops_step = res["useful_tflop_per_step"] * 1e12
    ms_step = res["ms_per_step"]
    value = res["value"]
    peak_tf, peak_gbs, peak_src = peaks()
    dev = torch.device("cuda", local)
    if not draft:
        nl, pp, pn = st.node_lengths, st.path_ptr, st.path_nodes

    # ---- secondary context: torch SDPA over a dense [T, T] boolean mask ------
    # (the pre-block-sparse path the drafter PR replaced).  The mask is
    # keep(q, kv) = node(kv) is an ancestor-or-self of node(q) and kv <= q,
    # from the tree's Euler intervals; forward and backward with GQA.
    sdpa = None
    if not args.no_dense and not draft and T <= 32768:
        try:
            sdpa = sdpa_dense_mask(st, Q, K, V, dO, max(2, min(3, args.steps)))
            sdpa["speedup"] = sdpa["ms_per_step"] / ms_step
        except Exception as e:  # noqa: BLE001 - context only: report why it could not run
            sdpa = {"unavailable": f"{type(e).__name__}: {str(e)[:160]}"}
        torch.cuda.empty_cache()

    # ---- end to end through the C ABI with host buffers ---------------------
    # Every step builds its map from the host tree arrays, uploads Q, K, V, dO
    # from pinned host memory and downloads dQ, dK, dV (pt_hoststep: two
    # device buffer sets, copies on their own streams, overlapped with the
    # kernels of the neighbouring steps).  One timed region over all steps,
    # ended after the last download; no L2 flush (the inputs arrive by copy).
    hq, hk, hv, hdo = (x.pin_memory() for x in (q, k, v, do))
    hdq, hdk, hdv = (torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (Q, K, V))
    hs = pt.HostStep(Q.dtype, T, Hq, Hkv, D)

    def e2e_step():
        bm = make_map()
        hs.run(hq, hk, hv, hdo, bm, hdq, hdk, hdv)
        bm.free()

    for _ in range(2):
        e2e_step()
    hs.sync()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(args.steps):
        e2e_step()
    hs.sync()
    eb.record(stream)
    torch.cuda.synchronize()
    pt.sync_status()
    hs.free()
    e2e_ms = max_over_ranks(ea.elapsed_time(eb), dist, dev)
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v, do)) + sum(int(a.nbytes) for a in host_layout)
    d2h = sum(x.numel() * x.element_size() for x in (dQ, dK, dV))
    e2e = {"value": whole_job_tflops(world, flops_step, args.steps, e2e_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms / args.steps,
           "path": "map built from host arrays + pt_hoststep_run from pinned host buffers, copies overlapped"}

    # ---- shared-prefix fold of the rollouts (HBM-bound data movement) -------
    # The workload's samples as rollout rows of hidden states (Hq*D per token,
    # the attention's input width): fold (rollouts -> flat), unfold (flat ->
    # rollouts, padding zeroed) and the adjoint of unfold (summed gradient).
    # Algorithmic bytes: fold 2*T*W; unfold T*W + S*L*W; unfold_grad
    # copies*W + T*W (copies = the rollout entries that hold a token).
    fold = None
    if not args.no_fold and not draft:
        L = int(max(sum(int(st.node_lengths[n]) for n in p) for p in st.paths()))
        plan = pt.fold_plan(nl, pp, pn, L)
        width = Hq * D
        hflat = torch.randn(T, width, device=dev).to(Q.dtype)
        roll = plan.unfold(hflat)
        flat_out = torch.empty_like(hflat)
        droll = torch.randn(roll.shape, device=dev).to(Q.dtype)
        S = plan.n_samples
        es = hflat.element_size()
        copies = int(sum(sum(int(st.node_lengths[n]) for n in p) for p in st.paths()))
        algo = {"fold": 2 * T * width * es, "unfold": (T + S * L) * width * es,
                "unfold_grad": (copies + T) * width * es}
        calls = {"fold": lambda: plan.fold(roll, out=flat_out), "unfold": lambda: plan.unfold(hflat, out=roll),
                 "unfold_grad": lambda: plan.unfold_grad(droll, out=flat_out)}
        fold = {"workload": f"{S} rollout rows of {L} tokens x {width} {dtype} (T={T} flat tokens)"}
        for name, fn in calls.items():
            for _ in range(3):
                fn()
            pt.profile_reset()
            pt.profile_enable(True)
            timed(args.steps, fn)
            pt.profile_enable(False)
            n, ms = pt.profile_read(name)
            ach = algo[name] / (ms / n * 1e-3) / 1e9
            fold[name] = {"ms_per_launch": ms / n, "algorithmic_bytes": algo[name], "achieved_gbs": ach,
                          "frac_of_hbm": ach / peak_gbs}
        fold["hbm_peak_gbs"] = peak_gbs
        fold["l2"] = "flushed before every launch (256 MB write, untimed)"
        pt.profile_reset()
        plan.free()
        pt.sync_status()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, s, nth, desc = cpu_oracle_run(st, cfg, args.workload)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": nth, "kind": "oracle", "sample": desc,
               "seconds": s}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "frac_of_peak": res["frac_of_peak"], "fwd": res["fwd"], "bwd": res["bwd"],
            "config": {"workload": cfg["name"], "T": T, "Hq": Hq, "Hkv": Hkv, "head_dim": D,
                       "useful_pairs_per_head": res["useful_pairs_per_head"],
                       "useful_tflop_per_step": flops_step / 1e12,
                       "tiles": "128x128", "l2": "flushed before every step (256 MB write, untimed)",
                       "parallelism": f"replicas x{world}"},
            "kernels": res["kernels"], "kernel_timing": "second pass of the same steps with an event pair per kernel",
            "roofline": res["roofline"], "hbm": res["hbm"], "dense_masked": res["dense_masked"], "sdpa_dense_mask": sdpa,
            "e2e": e2e,
            "gpu_launches": res["gpu_launches"], "clocks": clocks, "cpu_baseline": cpu, "fold": fold,
        }
        if others:
            line["workloads"] = others
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
