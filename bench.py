#!/usr/bin/env python
"""Benchmark of the tree-packed training hot path on GB300.

One step = one pass over one packed tree of the attention path: depth RoPE on Q
and K, tree attention forward (tile metadata + kernel), tree attention backward
(metadata, Delta, dQ/dK/dV) and the inverse RoPE on dQ and dK. The metric is
tree-attention forward+backward TFLOP/s counted on allowed (query, key) pairs
only (4*d per pair and query head forward, 10*d backward), with packed tokens/s
beside it. The shared-logit log-prob forward and backward run on their own
workload in the same process and are reported under "lm_head".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank packs its own tree (seed = rank): weak scaling, no
collective on the data path; only a barrier and a max over ranks of the timed
region. L2 is flushed (256 MiB write) before every timed step. ``--impl
reference`` times the float64 CPU oracle on the host cores instead (rank 0
only), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import resource
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "tree-attn fwd+bwd TFLOP/s on allowed pairs (% BF16 peak); packed tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


# ----------------------------------------------------------------------------- helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="agentic_long",
                    choices=["agentic_short", "agentic_long", "galton_watson", "tiny_fp32"])
    ap.add_argument("--secondary-steps", type=int, default=20,
                    help="timed steps of each tree that is not the headline workload")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--attn-heads", default="",
                    help="HQ,HKV: the attention trees with fewer heads (a smaller case for ncu captures; "
                         "not a bench configuration)")
    ap.add_argument("--lm-steps", type=int, default=3)
    ap.add_argument("--lm-rows", type=int, default=8192,
                    help="packed rows of the LM-head tree (mean path count 2.2); smaller for profiling")
    ap.add_argument("--no-lm", action="store_true")
    ap.add_argument("--conv-steps", type=int, default=10)
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--gateway-steps", type=int, default=5)
    ap.add_argument("--no-gateway", action="store_true")
    ap.add_argument("--gdn-steps", type=int, default=5)
    ap.add_argument("--no-gdn", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--leg-rest-s", type=float, default=2.0,
                    help="idle seconds before each leg after the headline, so that one leg's power "
                         "state (the LM GEMMs run at the power cap) does not carry into the next")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of graph replays")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="reference arm: target wall time of the whole run")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int) -> int:
    """Each rank packs its own tree: the workload seed is the rank."""
    return rank


def reduce_max(x: float, world: int) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from before the warm-up
    until after the timed region; each line is stamped with the host time it arrived, so
    the samples inside the timed window can be picked out (the nearest ones when the
    window is shorter than the sampling period)."""
    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.perf_counter(), line.strip().split(", ")))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(0.3)
        return self

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        good = [(t, r) for t, r in self.rows if len(r) >= len(self.FIELDS)]
        inside = [x for x in good if t0 <= x[0] <= t1 + 0.02]
        chosen = inside
        if not chosen and good:
            chosen = sorted(good, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))[:2]
        sm, mx, reasons = [], [], set()
        for _, r in chosen:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "samples_in_window": len(inside), "reasons": sorted(reasons)}


def source_sha(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "tree_masked_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str, sources) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, only while the kernel's
    sources are unchanged since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not d or d.get("source_sha") != source_sha(*sources):
        return None
    return float(d["bytes_per_launch"])


# ----------------------------------------------------------------------------- workload
def attention_workload(name: str, seed: int):
    tree = synth.CONFIGS[name]["tree"](seed=seed)
    c = synth.CONFIGS[name]
    return tree, c


def describe(name, T, P, n_seqs, n_tokens, c):
    return {
        "workload": name,
        "tree": {"agentic_short": "shared 256-token prompt, 4 trajectories x 4 steps x 128-token branches",
                 "agentic_long": "shared 1024-token prompt, 8 trajectories x 8 steps x 256-token branches, "
                                 "sibling sharing p=0.3",
                 "galton_watson": "Galton-Watson tree, depth <= 8 levels, fanout U{1,2,3}, segments "
                                  "U[64,512], 16384 packed tokens",
                 "tiny_fp32": "24-token prefix, children of 20 and 8 tokens, the 8 splitting into 12+12"}[name],
        "T_packed": int(T), "allowed_pairs": int(P), "input_sequences": int(n_seqs),
        "unpacked_tokens": int(n_tokens), "por": round(1.0 - T / n_tokens, 4),
        "Hq": c["Hq"], "Hkv": c["Hkv"], "d": c["d"],
        "l2": "flushed before every timed step (256 MiB write)",
        "step": "tree_rope(q, k) -> tree_attn_fwd -> tree_attn_bwd_rope (backward, and the inverse "
                "rotation of dq, dk fused into the kernel that writes them)",
    }


def attn_flops(P, Hq, d):
    return 4.0 * d * P * Hq, 10.0 * d * P * Hq


# ----------------------------------------------------------------------------- our arm
class AttnStep:
    """One packed tree's attention step on the device: RoPE, forward, backward with the
    inverse rotation fused. Holds the tree, its host (pinned) and device tensors."""

    def __init__(self, tma, name: str, seed: int, dev, heads=None):
        import torch
        self.tma, self.name, self.dev = tma, name, dev
        self.tree, c = attention_workload(name, seed)
        if heads is not None:  # fewer heads of the same tree: a smaller case for profiling
            c = dict(c, Hq=heads[0], Hkv=heads[1])
        self.c = c
        pk = tma.tree_pack(self.tree.seqs)
        self.T, self.Hq, self.Hkv, self.d = pk["T"], c["Hq"], c["Hkv"], c["d"]
        self.P = int((pk["position_ids"].astype(np.int64) + 1).sum())
        self.n_tokens = sum(len(s) for s in self.tree.seqs)
        self.f_fwd, self.f_bwd = attn_flops(self.P, self.Hq, self.d)
        self.td = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
        self.host = synth.attention_config(name, self.T, seed=seed)
        if heads is not None:
            q_, k_, v_, do_ = self.host
            self.host = tuple(np.ascontiguousarray(x) for x in
                              (q_[:, :self.Hq], k_[:, :self.Hkv], v_[:, :self.Hkv], do_[:, :self.Hq]))
        pin = lambda a: torch.from_numpy(a).to(self.td).pin_memory()
        self.hq, self.hk, self.hv, self.hdo = (pin(a) for a in self.host)
        self.q, self.k, self.v, self.do = (x.to(dev) for x in (self.hq, self.hk, self.hv, self.hdo))
        self.pos = torch.from_numpy(pk["position_ids"]).to(dev)
        self.end = torch.from_numpy(pk["subtree_end"]).to(dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((self.Hq, self.T), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = (torch.empty_like(x) for x in (self.q, self.k, self.v))
        self.dcode = 1 if self.td == torch.bfloat16 else 0
        self.ws = torch.empty(tma.tree_attn_workspace_size(self.T, self.Hq, self.Hkv, self.d, self.dcode),
                              dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def step(self, ev=None, b=None):
        """One step on the leg's device tensors, or on those of buffer set `b`."""
        tma, s = self.tma, self.stream
        b = self if b is None else b
        if ev: ev[0].record(s)
        tma.tree_rope(b.q, b.k, b.pos)
        if ev: ev[1].record(s)
        tma.tree_attn_fwd(b.q, b.k, b.v, b.end, workspace=b.ws, out=b.o, lse=b.lse)
        if ev: ev[2].record(s)
        # backward with the inverse rotation of dq, dk fused into the kernel that writes them
        tma.tree_attn_bwd_rope(b.q, b.k, b.v, b.o, b.do, b.lse, b.end, b.pos,
                               workspace=b.ws, grads=(b.dq, b.dk, b.dv))
        if ev: ev[3].record(s)

    def describe(self):
        return describe(self.name, self.T, self.P, len(self.tree.seqs), self.n_tokens, self.c)

    def measure(self, K: int, warmup: int, flush, use_graph: bool, world: int = 1, clocks=None):
        """Warm-up, K eager steps with per-call events (the per-kernel split), then K timed
        steps (CUDA-graph replays unless use_graph is false), L2 flushed before each."""
        import torch
        tma, stream = self.tma, self.stream
        for _ in range(max(warmup, 0)):
            flush.zero_()
            self.step()
        torch.cuda.synchronize()
        tma.tree_check_device_status()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        barrier(world)
        torch.cuda.synchronize()
        n0 = tma.tree_launch_count()
        # the library brackets each call's main kernel with events (read after each step)
        tma.tree_kernel_timing(True)
        main_ms = []
        for s in range(K):
            flush.zero_()
            self.step(evs[s])
            main_ms.append((tma.tree_kernel_last_ms(0), tma.tree_kernel_last_ms(1)))
        tma.tree_kernel_timing(False)
        torch.cuda.synchronize()
        launches_per_step = (tma.tree_launch_count() - n0) / K
        op_ms = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs])  # [K, 3]
        graph = None
        if use_graph:
            # the step's launches captured once into a CUDA graph (static shapes and
            # buffers), then replayed: the timed steps are K replays
            side = torch.cuda.Stream(self.dev)
            side.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                self.step()
            stream.wait_stream(side)
            for _ in range(2):
                flush.zero_()
                graph.replay()
            torch.cuda.synchronize()
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        barrier(world)
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for s in range(K):
            flush.zero_()
            gev[s][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                self.step()
            gev[s][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        w1 = time.perf_counter()
        clk = clocks.stop(w0, w1) if clocks is not None else None
        tma.tree_check_device_status()
        step_ms = np.array([e[0].elapsed_time(e[1]) for e in gev])
        total_s = reduce_max(float(step_ms.sum()) / 1e3, world)
        return {"total_s": total_s, "wall_s": w1 - w0, "op_ms": op_ms, "main_ms": np.array(main_ms),
                "launches_per_step": launches_per_step, "graph": graph is not None, "clocks": clk}

    def roofline(self, m, peak, peak_src):
        """Roofline of the dominant kernel call (the backward on every bf16 tree), with the
        main kernel's own duration from the library's event brackets."""
        names = ["tree_rope", "tree_attn_fwd", "tree_attn_bwd_rope"]
        avg = m["op_ms"].mean(axis=0)
        main = m["main_ms"].mean(axis=0)  # [fwd, bwd] main-kernel ms (-1: not bracketed)
        dom = int(np.argmax(avg))
        if dom == 0:  # RoPE cannot dominate a bf16 tree; kept for completeness
            dom = 2
        fl = self.f_fwd if dom == 1 else self.f_bwd
        kms = float(main[dom - 1])
        timed_kernel = kms > 0
        dur = kms if timed_kernel else float(avg[dom])
        achieved = fl / (dur / 1e3) / 1e12
        kname = {1: "attn_fwd_tc_kernel", 2: "attn_bwd_tc_kernel"}[dom] if timed_kernel else names[dom]
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "of": peak_src, "kernel": kname,
                "kernel_ms": round(dur, 4), "kernel_flops": fl, "call": names[dom],
                "call_achieved": round(fl / (avg[dom] / 1e3) / 1e12, 2)}
        key = {1: "attn_fwd", 2: "attn_bwd"}[dom]
        roof["traffic"] = profiled_traffic(f"{key}:{self.name}", kernel_sources(self.tma, key))
        roof["per_call_ms"] = {n: round(float(x), 4) for n, x in zip(names, avg)}
        roof["main_kernel_ms"] = {"attn_fwd_tc_kernel": round(float(main[0]), 4),
                                  "attn_bwd_tc_kernel": round(float(main[1]), 4)}
        if main[0] > 0:
            fa = self.f_fwd / (main[0] / 1e3) / 1e12
            roof["attn_fwd_tc_kernel"] = {"achieved": round(fa, 2), "frac": round(fa / peak, 4)}
        if main[1] > 0:
            ba = self.f_bwd / (main[1] / 1e3) / 1e12
            roof["attn_bwd_tc_kernel"] = {"achieved": round(ba, 2), "frac": round(ba / peak, 4)}
        roof["kernel_family"] = {"attn_fwd": self.tma.tree_kernel_path(0, self.dcode, self.d),
                                 "attn_bwd": self.tma.tree_kernel_path(1, self.dcode, self.d)}
        return roof

    def e2e(self, K: int, flush, world: int = 1):
        """The same step through the public API with host buffers, as a training loop runs
        it: every step packs its tree on the host (tree_pack, position_ids and subtree_end
        only), copies Q, K, V, dO, positions and subtree_end from pinned memory to the
        device, runs the step and copies dQ, dK, dV back into pinned memory. Two device
        buffer sets and three streams let step s + 1's inputs travel while step s computes
        and step s - 1's gradients come back; the host packs step s + 1's tree meanwhile."""
        import types
        import torch
        tma, dev, comp = self.tma, self.dev, self.stream
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        sets = [self]
        extra = types.SimpleNamespace()
        extra.q, extra.k, extra.v, extra.do = (torch.empty_like(x) for x in (self.q, self.k, self.v, self.do))
        extra.pos, extra.end = torch.empty_like(self.pos), torch.empty_like(self.end)
        extra.o, extra.lse = torch.empty_like(self.o), torch.empty_like(self.lse)
        extra.dq, extra.dk, extra.dv = (torch.empty_like(x) for x in (self.dq, self.dk, self.dv))
        extra.ws = torch.empty_like(self.ws)
        sets.append(extra)
        hgrad = [tuple(torch.empty(x.shape, dtype=self.td).pin_memory() for x in (self.dq, self.dk, self.dv))
                 for _ in range(2)]
        hpos = [torch.empty(self.T, dtype=torch.int32).pin_memory() for _ in range(2)]
        hend = [torch.empty(self.T, dtype=torch.int32).pin_memory() for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in (self.hq, self.hk, self.hv, self.hdo, hpos[0], hend[0]))
        d2h = sum(x.numel() * x.element_size() for x in hgrad[0])
        ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("h2d", "comp", "d2h")}

        def pack_into(b):
            p2 = tma.tree_pack(self.tree.seqs, fields=("position_ids", "subtree_end"))
            hpos[b].numpy()[:] = p2["position_ids"]
            hend[b].numpy()[:] = p2["subtree_end"]

        def run(n):
            torch.cuda.synchronize()
            used = [False, False]
            pack_into(0)
            for s_ in range(n):
                b, S = s_ & 1, sets[s_ & 1]
                if used[b]:
                    h2d_s.wait_event(ev["comp"][b])  # step s - 2 is done with this set's inputs
                with torch.cuda.stream(h2d_s):
                    for dst, src in ((S.pos, hpos[b]), (S.end, hend[b]), (S.q, self.hq), (S.k, self.hk),
                                     (S.v, self.hv), (S.do, self.hdo)):
                        dst.copy_(src, non_blocking=True)
                    ev["h2d"][b].record(h2d_s)
                comp.wait_event(ev["h2d"][b])
                if used[b]:
                    comp.wait_event(ev["d2h"][b])  # step s - 2's gradients have left this set
                flush.zero_()
                self.step(b=S)
                ev["comp"][b].record(comp)
                d2h_s.wait_event(ev["comp"][b])
                with torch.cuda.stream(d2h_s):
                    for dst, src in zip(hgrad[b], (S.dq, S.dk, S.dv)):
                        dst.copy_(src, non_blocking=True)
                    ev["d2h"][b].record(d2h_s)
                used[b] = True
                if s_ + 1 < n:
                    if s_ >= 1:
                        ev["h2d"][b ^ 1].synchronize()  # step s - 1's index copies have left hpos/hend
                    pack_into(b ^ 1)
            torch.cuda.synchronize()

        run(3)
        barrier(world)
        w0 = time.perf_counter()
        run(K)
        e_s = reduce_max(time.perf_counter() - w0, world)
        return {"value": round((self.f_fwd + self.f_bwd) * K * world / e_s / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e_s * 1e3 / K, 4),
                "includes": "per step: tree_pack on the host, pinned H2D of Q,K,V,dO,positions,subtree_end, "
                            "the step, D2H of dQ,dK,dV into pinned buffers, L2 flush write; two device buffer "
                            "sets and separate copy streams overlap step s+1's H2D and step s-1's D2H with "
                            "step s, and the host packs the next tree meanwhile; wall clock around all K steps"}


def secondary_entry(leg: AttnStep, m, peak, peak_src):
    """A smaller summary line for the trees that are not the headline workload."""
    flops = leg.f_fwd + leg.f_bwd
    K = len(m["op_ms"])
    value = flops * K / m["total_s"] / 1e12
    return {"config": leg.describe(), "value": round(value, 3), "unit": "TFLOP/s",
            "ms_per_step": round(m["total_s"] * 1e3 / K, 4), "steps": K,
            "pct_bf16_peak": round(100.0 * value / peak, 2),
            "packed_tokens_per_s": round(leg.T * K / m["total_s"], 1),
            "step_mode": "CUDA-graph replay of the device step" if m["graph"] else "eager launches",
            "roofline": leg.roofline(m, peak, peak_src)}


def run_ours(args):
    import torch
    import tree_masked_attention_gb300 as tma
    from tree_masked_attention_gb300 import build as _b
    _b.build()

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    heads = tuple(int(x) for x in args.attn_heads.split(",")) if args.attn_heads else None
    leg = AttnStep(tma, args.workload, rank_seed(rank), dev, heads)
    K = args.steps
    clocks = ClockSampler(local).start()
    m = leg.measure(K, args.warmup, flush, use_graph=not args.no_graph, world=world, clocks=clocks)
    total_s = m["total_s"]
    flops_step = leg.f_fwd + leg.f_bwd
    value = flops_step * K * world / total_s / 1e12
    launches = int(round(m["launches_per_step"] * K))
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_s * 1e3 / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": leg.c["dtype"], "data": "synthetic",
        "config": leg.describe(),
        "pct_bf16_peak": round(100.0 * value / (peak * world), 2),
        "packed_tokens_per_s": round(leg.T * K * world / total_s, 1),
        "wall_s_timed_region": round(m["wall_s"], 4),
        "step_mode": "CUDA-graph replay of the device step" if m["graph"] else "eager launches",
        "gpu_launches": int(launches),
        "gpu_launches_note": f"{m['launches_per_step']:g} library kernels per step (counted on eager steps) x {K} steps",
        "eager_ms_per_step": round(float(m["op_ms"].sum(axis=1).mean()), 4),
        "clocks": m["clocks"],
        "roofline": leg.roofline(m, peak, peak_src),
    }
    if not args.no_e2e:
        out["e2e"] = leg.e2e(K, flush, world)

    def rest():
        torch.cuda.synchronize()
        time.sleep(max(args.leg_rest_s, 0.0))

    # the other bf16 trees, each with its own roofline (rank 0, one GPU's worth of work)
    if rank == 0 and not args.no_secondary:
        sec = {}
        for name in ("galton_watson", "agentic_long", "agentic_short"):
            if name == args.workload:
                continue
            rest()
            other = AttnStep(tma, name, 0, dev, heads)
            m2 = other.measure(max(args.secondary_steps, 1), 3, flush, use_graph=not args.no_graph)
            sec[name] = secondary_entry(other, m2, peak, peak_src)
            del other
        out["secondary"] = sec

    if not args.no_lm and rank == 0:
        rest()
        out["lm_head"] = run_lm_head(args, dev, peaks, peak_src)
    if not args.no_conv and rank == 0:
        rest()
        out["conv1d"] = run_conv1d(args, dev, peaks, peak_src, flush)
    if not args.no_gateway and rank == 0:
        rest()
        out["gateway"] = run_gateway(args, dev, peaks, peak_src, flush)
    if not args.no_gdn and rank == 0:
        rest()
        out["gdn"] = run_gdn(args, dev, flush)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, leg.tree, leg.host, leg.P, budget_s=25.0)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def kernel_sources(tma, key):
    """Source files of the kernel that a roofline entry describes."""
    if key == "attn_fwd":
        return ["attn_tc.cu"] if tma.tree_kernel_path(0, 1, 128) == 1 else ["attn_simt.cu"]
    return ["attn_bwd_tc.cu"] if tma.tree_kernel_path(1, 1, 128) == 1 else ["attn_simt.cu"]


def run_lm_head(args, dev, peaks, peak_src):
    """Shared-logit log-prob forward + backward on the 8192 x 4096 x 128256 workload."""
    import torch
    import tree_masked_attention_gb300 as tma
    rows = rows_arg = args.lm_rows
    tree = synth.lm_head_tree(rows=rows, occ_range=(round(rows * 17500 / 8192), round(rows * 18500 / 8192)))
    pk = tma.tree_pack(tree.seqs)
    T, K, V = pk["T"], 4096, 128256
    n_occ = pk["n_occ"]
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    h = torch.randn((T, K), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((K, V), generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(7)
    tg = torch.from_numpy(rng.integers(0, V, size=n_occ).astype(np.int32)).to(dev)
    gl = torch.from_numpy(-(1.0 - rng.random(n_occ)).astype(np.float32)).to(dev)
    rp = torch.from_numpy(pk["occ_row_ptr"]).to(dev)
    pm = torch.from_numpy(pk["occ_perm"]).to(dev)
    ws = torch.empty(tma.tree_logprob_workspace_size(T, K, V, n_occ, 1), dtype=torch.uint8, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    logp = torch.empty(n_occ, dtype=torch.float32, device=dev)
    dh, dw = torch.empty_like(h), torch.empty_like(w)
    rows = int((np.diff(pk["occ_row_ptr"]) > 0).sum())
    f_gemm = 2.0 * rows * K * V
    stream = torch.cuda.current_stream(dev)

    # a policy-gradient step: per-occurrence advantages and old log-probs (the current
    # ones perturbed), the clipped objective's gradient feeds the backward
    tma.tree_logprob_fwd(h, w, rp, pm, tg, workspace=ws, lse=lse, logp=logp)
    adv = torch.randn(n_occ, generator=g, device=dev, dtype=torch.float32)
    old_lp = logp + 0.3 * torch.randn(n_occ, generator=g, device=dev, dtype=torch.float32)

    def step(ev=None):
        if ev: ev[0].record(stream)
        tma.tree_logprob_fwd(h, w, rp, pm, tg, workspace=ws, lse=lse, logp=logp)
        if ev: ev[1].record(stream)
        tma.tree_policy_loss(logp, old_lp, adv, eps_low=0.2, grad=gl)
        if ev: ev[2].record(stream)
        tma.tree_logprob_bwd(h, w, lse, rp, pm, tg, gl, workspace=ws, grads=(dh, dw))
        if ev: ev[3].record(stream)

    step()
    torch.cuda.synchronize()
    n = max(args.lm_steps, 1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for s in range(n):
        step(evs[s])
    torch.cuda.synchronize()
    tma.tree_check_device_status()
    ms3 = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs]).mean(axis=0)
    ms = np.array([ms3[0], ms3[2]])  # the two GEMM phases; the objective is reported apart
    peak = float(peaks["bf16_tflops"])
    fwd_t = f_gemm / (ms[0] / 1e3) / 1e12
    bwd_t = 3 * f_gemm / (ms[1] / 1e3) / 1e12
    tot = 4 * f_gemm / (float(ms3.sum()) / 1e3) / 1e12  # whole step, objective included
    dom = 1 if ms[1] >= ms[0] else 0
    ach = bwd_t if dom else fwd_t
    return {
        "workload": f"lm_head: hidden {T}x{K} bf16, W_LM {K}x{V} bf16, {n_occ} occurrences over {rows} rows "
                    "(source rows from a Galton-Watson tree of 8192 tokens), targets U[0,V), weights U(0,1]",
        "value": round(tot, 3), "unit": "TFLOP/s", "steps": n,
        "ms_fwd": round(float(ms[0]), 3), "ms_bwd": round(float(ms[1]), 3),
        "ms_policy_loss": round(float(ms3[1]), 4),
        "step": "tree_logprob_fwd -> tree_policy_loss (clipped objective, eps 0.2) -> tree_logprob_bwd",
        "flops_per_step": 4 * f_gemm, "pct_bf16_peak": round(100 * tot / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(ach / peak, 4), "of": peak_src,
                     "kernel": "tree_logprob_bwd" if dom else "tree_logprob_fwd",
                     "traffic": (profiled_traffic(("lm_bwd" if dom else "lm_fwd") + ":lm_head", ["lm_tc.cu"])
                                 if rows_arg == 8192 else None),
                     "traffic_unit": "DRAM bytes per call (all of the call's launches)"},
        "kernel_family": {"fwd": tma.tree_kernel_path(2, 1, 128), "bwd": tma.tree_kernel_path(3, 1, 128)},
        "data": "synthetic (seeded torch generator on device)",
    }


def run_conv1d(args, dev, peaks, peak_src, flush):
    """Tree-correct causal depthwise conv1d (kernel size 4) forward and backward on the
    16384-row Galton-Watson tree at 8192 channels (bf16): the short convolution of an
    SSM layer. HBM-bound; L2 flushed before every call, CUDA events on the stream."""
    import torch
    import tree_masked_attention_gb300 as tma
    tree = synth.galton_watson()
    pk = tma.tree_pack(tree.seqs)
    T, C, K = pk["T"], 8192, 4
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    x = torch.randn((T, C), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    dy = torch.randn((T, C), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    w = (0.5 * torch.randn((C, K), generator=g, device=dev, dtype=torch.float32)).to(torch.bfloat16)
    b = (0.1 * torch.randn(C, generator=g, device=dev, dtype=torch.float32)).to(torch.bfloat16)
    par = torch.from_numpy(pk["parent_row"]).to(dev)
    end = torch.from_numpy(pk["subtree_end"]).to(dev)
    pos = torch.from_numpy(pk["position_ids"]).to(dev)
    y, dx = torch.empty_like(x), torch.empty_like(x)
    dw = torch.empty((C, K), dtype=torch.float32, device=dev)
    db = torch.empty(C, dtype=torch.float32, device=dev)
    ws = torch.empty(tma.tree_conv1d_workspace_size(T, C, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = max(args.conv_steps, 1)
    for _ in range(3):
        tma.tree_conv1d_fwd(x, w, par, bias=b, out=y)
        tma.tree_conv1d_bwd(x, w, dy, end, pos, workspace=ws, grads=(dx, dw, db))
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    kern = []
    # the library brackets each call's kernels with events right at the launches, so the
    # kernel times carry none of the host's call overhead; the call times (events recorded
    # from Python around each call) are reported beside them
    tma.tree_kernel_timing(True)
    for s in range(n):
        flush.zero_()
        evs[s][0].record(stream)
        tma.tree_conv1d_fwd(x, w, par, bias=b, out=y)
        evs[s][1].record(stream)
        flush.zero_()
        evs[s][2].record(stream)
        tma.tree_conv1d_bwd(x, w, dy, end, pos, workspace=ws, grads=(dx, dw, db))
        evs[s][3].record(stream)
        kern.append((tma.tree_kernel_last_ms(2), tma.tree_kernel_last_ms(3)))
    tma.tree_kernel_timing(False)
    torch.cuda.synchronize()
    tma.tree_check_device_status()
    call_f = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    call_b = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    kern = np.array(kern)
    f_ms = float(kern[:, 0].mean()) if (kern[:, 0] > 0).all() else call_f
    b_ms = float(kern[:, 1].mean()) if (kern[:, 1] > 0).all() else call_b
    el = 2
    # algorithmic bytes: forward reads x and writes y once, reads parent_row and the taps;
    # backward reads x and dy and writes dx once, reads subtree_end, positions and the
    # taps, writes dw and dbias (the per-tile partial sums are not counted)
    f_bytes = 2.0 * T * C * el + 4.0 * T + C * (K + 1) * el
    b_bytes = 3.0 * T * C * el + 8.0 * T + C * K * el + 4.0 * C * (K + 1)
    hbm = float(peaks["hbm_gbs"])
    fg, bg = f_bytes / (f_ms / 1e3) / 1e9, b_bytes / (b_ms / 1e3) / 1e9
    dom_b = b_ms >= f_ms
    return {
        "workload": f"conv1d: Galton-Watson tree of {T} rows, {C} channels, kernel size {K}, bf16, with bias",
        "value": round((f_bytes + b_bytes) / ((f_ms + b_ms) / 1e3) / 1e9, 1), "unit": "GB/s",
        "ms_fwd": round(f_ms, 4), "ms_bwd": round(b_ms, 4), "steps": n,
        "call_ms": {"fwd": round(call_f, 4), "bwd": round(call_b, 4)},
        "gbs_fwd": round(fg, 1), "gbs_bwd": round(bg, 1),
        "step": "tree_conv1d_fwd -> tree_conv1d_bwd (dx, dw, dbias), L2 flushed before each call",
        "roofline": {"bound": "hbm", "achieved": round(bg if dom_b else fg, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round((bg if dom_b else fg) / hbm, 4), "of": peak_src,
                     "kernel": "tree_conv1d_bwd" if dom_b else "tree_conv1d_fwd",
                     "bytes_per_launch": b_bytes if dom_b else f_bytes,
                     "traffic": profiled_traffic(("conv1d_bwd" if dom_b else "conv1d_fwd") + ":galton_watson_c8192_k4",
                                                 ["conv1d.cu"])},
        "data": "synthetic (seeded torch generator on device)",
    }


def run_gateway(args, dev, peaks, peak_src, flush):
    """Partition-gateway attention: the long-prompt agentic tree cut below its shared
    1024-token prompt. The prompt is the parent partition; every trajectory subtree is a
    child partition whose gateway past is the prompt (all ancestors, bias 0). Each step
    runs every child's tree_attn_fwd_gateway and tree_attn_bwd_gateway (the prompt rows'
    dK / dV summed over the children in fp32). TFLOP/s on allowed pairs of the children."""
    import torch
    import tree_masked_attention_gb300 as tma
    tree = synth.agentic_long()
    pk = tma.tree_pack(tree.seqs)
    c = synth.CONFIGS["agentic_long"]
    Hq, Hkv, d = c["Hq"], c["Hkv"], c["d"]
    end, par, pos = pk["subtree_end"], pk["parent_row"], pk["position_ids"]
    prompt_end = int(pk["node_end"][0])          # the shared prompt: the root node
    P = prompt_end + 1
    kids = [int(r) for r in range(P, pk["T"]) if par[r] == prompt_end]
    T = pk["T"]
    q_all, k_all, v_all, do_all = synth.attention_config("agentic_long", T, seed=0)
    bf = torch.bfloat16
    past_k = torch.from_numpy(k_all[:P]).to(bf)
    past_v = torch.from_numpy(v_all[:P]).to(bf)
    bias = torch.zeros(P, dtype=torch.float32, device=dev)
    parts, pairs = [], 0
    for r in kids:
        rows = slice(r, int(end[r]) + 1)
        n = int(end[r]) + 1 - r
        ce = (end[rows] - r).astype(np.int32)
        parts.append(dict(
            q=torch.from_numpy(q_all[rows]).to(bf).to(dev), do=torch.from_numpy(do_all[rows]).to(bf).to(dev),
            k=torch.cat([past_k, torch.from_numpy(k_all[rows]).to(bf)]).to(dev),
            v=torch.cat([past_v, torch.from_numpy(v_all[rows]).to(bf)]).to(dev),
            end=torch.from_numpy(ce).to(dev), n=n))
        pairs += int((pos[rows].astype(np.int64) + 1).sum())   # every past row is an ancestor
    ws = torch.empty(max(tma.tree_attn_gateway_workspace_size(P, p["n"], Hq, Hkv, d, 1) for p in parts),
                     dtype=torch.uint8, device=dev)
    dkp = torch.zeros((P, Hkv, d), dtype=torch.float32, device=dev)
    dvp = torch.zeros_like(dkp)
    for p in parts:
        p["o"] = torch.empty_like(p["q"])
        p["lse"] = torch.empty((Hq, p["n"]), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dkp.zero_()
        dvp.zero_()
        for p in parts:
            tma.tree_attn_fwd_gateway(p["q"], p["k"], p["v"], bias, p["end"], workspace=ws, out=p["o"], lse=p["lse"])
        for p in parts:
            tma.tree_attn_bwd_gateway(p["q"], p["k"], p["v"], p["o"], p["do"], p["lse"], bias, p["end"],
                                      dk_past=dkp, dv_past=dvp, workspace=ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(args.gateway_steps, 1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for s in range(n):
        flush.zero_()
        evs[s][0].record(stream)
        step()
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    tma.tree_check_device_status()
    ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    fl = 14.0 * d * pairs * Hq
    tf = fl / (ms / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    return {
        "workload": f"gateway: long-prompt agentic tree ({T} rows) cut below its {P}-token prompt; "
                    f"{len(parts)} child partitions of {min(p['n'] for p in parts)}-{max(p['n'] for p in parts)} rows, "
                    f"each with the prompt as gateway past; bf16, {Hq}/{Hkv} heads, d = {d}",
        "value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4), "steps": n,
        "allowed_pairs": pairs, "flops_per_step": fl, "pct_bf16_peak": round(100 * tf / peak, 2),
        "step": "tree_attn_fwd_gateway for every child, then tree_attn_bwd_gateway for every child "
                "(prompt dK / dV summed in fp32); L2 flushed before each step",
        "data": "synthetic (the long-prompt agentic configuration's seeded Q, K, V, dO)",
    }


def run_gdn(args, dev, flush):
    """Gated DeltaNet with tree state routing on the 16384-row Galton-Watson tree: 16
    heads, Dk = Dv = 128, bf16 q / k / v / dO, fp32 gates. Forward and backward, each
    timed with CUDA events after an L2 flush; packed tokens/s of the forward+backward
    step, and the recurrence's own arithmetic (3 products of the [Dv, Dk] state per
    token and head forward: S k, the rank-1 update, S q)."""
    import torch
    import tree_masked_attention_gb300 as tma
    tree = synth.galton_watson()
    pk = tma.tree_pack(tree.seqs)
    T, H, D = pk["T"], 16, 128
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    q = (torch.randn((T, H, D), generator=g, device=dev) / D ** 0.5).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((T, H, D), generator=g, device=dev), dim=-1).to(torch.bfloat16)
    v = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    do = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    gate = -0.2 * torch.rand((T, H), generator=g, device=dev)
    beta = torch.rand((T, H), generator=g, device=dev)
    ns, ne, npar = (torch.from_numpy(pk[n]).to(dev) for n in ("node_start", "node_end", "node_parent"))
    ws = torch.empty(tma.tree_gdn_bwd_workspace_size(T, len(pk["node_start"]), H, D, D), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(v)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(gate),
             torch.empty_like(beta))
    stream = torch.cuda.current_stream(dev)
    # the step: the forward on the backward-sized workspace, then the backward that takes
    # the forward's states from it (tree_gdn_bwd_saved); the backward that recomputes them
    # from the inputs alone (tree_gdn_bwd) is timed beside it
    for _ in range(2):
        tma.tree_gdn_fwd(q, k, v, gate, beta, ns, ne, npar, workspace=ws, out=o)
        tma.tree_gdn_bwd(q, k, v, gate, beta, do, ns, ne, npar, workspace=ws, grads=grads, saved=True)
        tma.tree_gdn_bwd(q, k, v, gate, beta, do, ns, ne, npar, workspace=ws, grads=grads)
    torch.cuda.synchronize()
    n = max(args.gdn_steps, 1)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
    for s in range(n):
        flush.zero_()
        evs[s][0].record(stream)
        tma.tree_gdn_fwd(q, k, v, gate, beta, ns, ne, npar, workspace=ws, out=o)
        evs[s][1].record(stream)
        flush.zero_()
        evs[s][2].record(stream)
        tma.tree_gdn_bwd(q, k, v, gate, beta, do, ns, ne, npar, workspace=ws, grads=grads, saved=True)
        evs[s][3].record(stream)
        flush.zero_()
        evs[s][4].record(stream)
        tma.tree_gdn_bwd(q, k, v, gate, beta, do, ns, ne, npar, workspace=ws, grads=grads)
        evs[s][5].record(stream)
    torch.cuda.synchronize()
    tma.tree_check_device_status()
    f_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    b_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in evs]))
    r_ms = float(np.mean([e[4].elapsed_time(e[5]) for e in evs]))
    fl = 6.0 * D * D * H * T
    return {
        "workload": f"gdn: Galton-Watson tree of {T} rows ({len(pk['node_start'])} nodes), {H} heads, Dk = Dv = {D}, "
                    "bf16 q/k/v/dO, fp32 gates",
        "value": round(T / ((f_ms + b_ms) / 1e3), 1), "unit": "packed tokens/s (forward + backward)",
        "ms_fwd": round(f_ms, 4), "ms_bwd": round(b_ms, 4), "ms_bwd_recompute": round(r_ms, 4), "steps": n,
        "fwd_tokens_per_s": round(T / (f_ms / 1e3), 1),
        "fwd_recurrence_tflops": round(fl / (f_ms / 1e3) / 1e12, 3),
        # fp32 on the CUDA cores: the ALU roofline is 152 SMs x 128 fp32 lanes x 2 FLOP per FMA
        # at the 2070 MHz maximum SM clock = 80.5 TFLOP/s; the algorithmic work counted is the
        # recurrence's, 6 Dk Dv per row and head forward and twice that backward (the chunked
        # form's extra products -- the triangular factors -- are not counted)
        "roofline": {"bound": "alu", "achieved": round(2 * fl / (b_ms / 1e3) / 1e12, 3), "peak": 80.5,
                     "unit": "TFLOP/s", "frac": round(2 * fl / (b_ms / 1e3) / 1e12 / 80.5, 4),
                     "of": "152 SMs x 128 fp32 FMA lanes x 2 x 2.07 GHz", "kernel": "tree_gdn_bwd_saved",
                     "traffic": None},
        "kernels": "fwd: gdn_setup, gdn_prep (chunk-parallel factors), gdn_chain (state chain over 32-column "
                   "slices), gdn_out; bwd (saved): setup, gdn_bprep (chain-independent products), gdn_bchain "
                   "(state-gradient chain), gdn_grads; bwd (recompute): setup, prep, chain, bprep, bchain, "
                   "grads (fp32 CUDA cores)",
        "data": "synthetic (seeded torch generator on device)",
    }


# ----------------------------------------------------------------------------- oracle timing
def _oracle_sample(ref, qkvdo, n_heads, n_paths, Hq, Hkv):
    """The oracle's forward and backward over the first n_paths input sequences (their
    union is a sub-tree: every prefix of a path is on it) for n_heads query heads. Returns
    wall seconds, CPU seconds and the allowed pairs of that sub-tree."""
    import oracle
    q, k, v, do = qkvdo
    G = Hq // Hkv
    n_kv = max(1, n_heads // G) if n_heads >= G else 1
    n_heads = n_kv * G if n_heads >= G else n_heads
    hs, ks = slice(0, n_heads), slice(0, n_kv)
    paths = ref["paths"][:n_paths]
    rows = np.unique(np.concatenate([np.asarray(p, dtype=np.int64) for p in paths]))
    pairs = int((ref["position_ids"][rows].astype(np.int64) + 1).sum())
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    oracle.attn_ref_fwd(q[:, hs], k[:, ks], v[:, ks], paths)
    oracle.attn_ref_bwd(q[:, hs], k[:, ks], v[:, ks], do[:, hs], paths)
    wall = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    return wall, cpu, pairs, n_heads


def _oracle_plan(ref, qkvdo, Hq, Hkv, budget_s):
    """Sample size (query heads, leading input sequences) whose oracle pass takes about
    budget_s: the oracle's cost grows with n_heads * sum of squared path lengths, so one
    calibration pass over the first sixteenth of the paths on one head sets the scale."""
    lens = np.array([len(p) for p in ref["paths"]], dtype=np.float64)
    cost = np.cumsum(lens ** 2)
    n_cal = max(1, len(lens) // 16)
    wall, _, _, _ = _oracle_sample(ref, qkvdo, 1, n_cal, Hq, Hkv)
    per_unit = max(wall, 1e-4) / cost[n_cal - 1]
    if per_unit * cost[-1] <= budget_s:  # the whole tree fits: add heads
        return int(max(1, min(Hq, budget_s // (per_unit * cost[-1])))), len(lens)
    n_paths = int(np.searchsorted(cost, budget_s / per_unit, side="right"))
    return 1, max(1, n_paths)


def _sample_text(n_heads, n_paths, ref, Hq):
    return (f"oracle fwd+bwd (float64 NumPy, per-path unpacked causal attention) over the sub-tree of the "
            f"first {n_paths} of {len(ref['paths'])} input sequences, {n_heads} of {Hq} query heads; "
            f"FLOPs counted on that sub-tree's allowed pairs")


def cpu_baseline(name, tree, qkvdo, P, budget_s=25.0):
    """The oracle (float64 NumPy, per-path unpacked attention) on the host cores, on a
    bounded sample of the same workload (a leading sub-tree, some query heads)."""
    import oracle
    c = synth.CONFIGS[name]
    Hq, Hkv, d = c["Hq"], c["Hkv"], c["d"]
    ref = oracle.pack_ref(tree.seqs)
    n_heads, n_paths = _oracle_plan(ref, qkvdo, Hq, Hkv, budget_s)
    wall, cpu, pairs, n_heads = _oracle_sample(ref, qkvdo, n_heads, n_paths, Hq, Hkv)
    f = sum(attn_flops(pairs, n_heads, d))
    return {"value": round(f / wall / 1e12, 6), "unit": "TFLOP/s", "cores": max(1, round(cpu / wall)),
            "kind": "oracle", "sample": _sample_text(n_heads, n_paths, ref, Hq) + f"; {wall:.2f} s wall, {cpu:.1f} s CPU"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle  # the reference arm: the oracle is the reference
    tree, c = attention_workload(args.workload, 0)
    ref = oracle.pack_ref(tree.seqs)
    T = ref["T"]
    P = int((ref["position_ids"].astype(np.int64) + 1).sum())
    qkvdo = synth.attention_config(args.workload, T, seed=0)
    Hq, Hkv, d = c["Hq"], c["Hkv"], c["d"]
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    n_heads, n_paths = _oracle_plan(ref, qkvdo, Hq, Hkv, per_step)
    for _ in range(max(args.warmup - 1, 0)):
        _oracle_sample(ref, qkvdo, n_heads, n_paths, Hq, Hkv)
    walls, cpus = [], []
    for _ in range(args.steps):
        w, cp, pairs, nh = _oracle_sample(ref, qkvdo, n_heads, n_paths, Hq, Hkv)
        walls.append(w)
        cpus.append(cp)
    f = sum(attn_flops(pairs, nh, d))
    tot = sum(walls)
    value = f * args.steps / tot / 1e12
    cores = max(1, round(sum(cpus) / tot))
    out = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot * 1e3 / args.steps, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": describe(args.workload, T, P, len(tree.seqs), sum(len(s) for s in tree.seqs), c),
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                            "sample": _sample_text(nh, n_paths, ref, Hq) + " per step"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
