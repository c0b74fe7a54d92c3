"""Throughput of the MoE greedy-verify step on synthetic inputs.

Workload (the full verify step): the 12-layer stack (hidden 1280, 64 routed
SwiGLU experts of 896 with top-6 routing plus 2 shared experts, vocabulary
129,280), B=32 sequences in flight (concurrency 32) with K=3 drafts each.
A draft equals the target's greedy token with probability 0.75, else it is a
uniform random id (about 2.73 tokens committed per step); a sequence stops
at 1,085 committed tokens and a new one with a fresh start id takes its slot.

One bench step = one verify step (all layers, lm_head, argmax) plus the
acceptance kernel for the 32 sequences.  `value` is committed tokens per
second with every step's inputs already in HBM; `e2e` is the same metric
through moe_verify_decode_host with host buffers (copies in the timed
region).  The weights (5.8 GB touched per step) are larger than L2, so no
flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank drives its own GPU with its own 32 sequences
(replicas: nothing is exchanged on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_speculative_decoding_router_gb300 import synth as S  # noqa: E402

METRIC = "committed tokens/s, MoE verify step (B=32, K=3)"
UNIT = "tokens/s"
B_SEQ, K_DRAFT, P_MATCH, PAGE_TOKENS = 32, 3, 0.75, 1085
WORKLOAD = "moe_verify_full_b32_k3_p0.75"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------- trajectory

class Trajectory:
    """Host simulation of the decode loop with a known greedy table g.

    Sequence slot b holds one page at a time: last committed id, tokens
    committed so far, and a step counter for the draft coins.  Finished pages
    (1,085 tokens) are replaced by a new start id.  Targets are g of each
    verify token, so the outcome of every step is known in advance."""

    def __init__(self, g: np.ndarray, rank: int, B=B_SEQ, K=K_DRAFT, p=P_MATCH,
                 page_tokens=PAGE_TOKENS):
        self.g, self.B, self.K, self.page = g, B, K, page_tokens
        self.V = len(g)
        self.src = S.DraftSource(p, self.V, K)
        self.rank = rank
        self.page_id = np.arange(B, dtype=np.int64) + rank * 1_000_000
        self.next_page = B
        self.last = S.start_ids(B, self.V, first=rank * 1_000_000).astype(np.int64)
        self.done = np.zeros(B, dtype=np.int64)
        self.steps = np.zeros(B, dtype=np.int64)
        self._rows = np.arange(B)

    def drafts(self):
        truth = np.empty((self.B, self.K), dtype=np.int64)
        x = self.last
        for i in range(self.K):
            x = self.g[x]
            truth[:, i] = x
        d = self.src.drafts_batch(self.page_id, self.steps, truth)
        return self.last.astype(np.int32), d

    def advance(self, committed: np.ndarray, alen: np.ndarray) -> int:
        """Apply one step's outcome; returns the committed tokens it counts."""
        n = np.asarray(alen, dtype=np.int64)
        take = np.minimum(n + 1, self.page - self.done)
        self.done += take
        self.steps += 1
        self.last = np.asarray(committed, dtype=np.int64)[self._rows, n]
        for b in np.flatnonzero(self.done >= self.page):
            self.page_id[b] = self.rank * 1_000_000 + self.next_page
            self.next_page += 1
            self.last[b] = int(S.start_ids(1, self.V, first=int(self.page_id[b]))[0])
            self.done[b] = 0
            self.steps[b] = 0
        return int(take.sum())

    def expected(self, ctx_ids: np.ndarray, drafts: np.ndarray):
        toks = np.concatenate([ctx_ids.reshape(-1, 1), drafts], axis=1).astype(np.int64)
        y = self.g[toks].astype(np.int32)
        match = drafts == y[:, :-1]
        n = np.where(match.all(axis=1), self.K, np.argmin(match, axis=1))
        keep = np.arange(self.K + 1)[None, :] <= n[:, None]
        committed = np.where(keep, y, -1).astype(np.int32)
        return committed, n.astype(np.int32)


# ------------------------------------------------------------ clocks sampling

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [l for _, l in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- our arm

def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def expert_weight_bytes(topk_idx_layer: np.ndarray, cfg) -> float:
    """Algorithmic bytes of one expert-FFN launch (one layer): the gate, up and
    down weights of every touched expert (routed + shared), once.
    Intermediate activations are not counted.  topk_idx_layer: [T, k]."""
    touched = len(np.unique(topk_idx_layer)) + cfg.n_shared
    return float(touched * 3 * cfg.expert_inter * cfg.hidden * 2)


def step_bytes(topk_idx: np.ndarray, cfg, T: int) -> float:
    """Algorithmic bytes of one verify step: the touched experts' weights of
    every layer, the routers, the norms' gains, the whole lm_head, the
    embedding rows of the verify tokens, ids in and out.  topk_idx: [L, T, k]."""
    L, d, E, V = cfg.n_layers, cfg.hidden, cfg.n_experts, cfg.vocab
    b = sum(expert_weight_bytes(topk_idx[l], cfg) for l in range(L))
    return b + L * E * d * 2 + (L + 1) * d * 2 + V * d * 2 + T * d * 2 + T * 4 * 3


def step_flops(cfg, T: int) -> float:
    """Flops of one verify step, selected-expert work only: routed and shared
    expert rows (gate, up, down), the routers, the lm_head."""
    L, d, E, k, S, I, V = (cfg.n_layers, cfg.hidden, cfg.n_experts, cfg.top_k, cfg.n_shared,
                           cfg.expert_inter, cfg.vocab)
    return float(L * (T * (k + S) * 6 * d * I + 2 * T * d * E) + 2 * T * d * V)


def kernel_digest() -> str:
    """Digest of the CUDA sources of the kernels, to tell whether a stored ncu
    figure was taken on the kernels that run now."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_speculative_decoding_router_gb300", "csrc")
    for name in ("gemm.cu", "route.cu", "ptx.cuh", "internal.h"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def greedy_table(ctx, V: int, K: int, dev, max_batch: int):
    """The library's own greedy target of every id, max_batch * (K+1) ids per call."""
    import torch
    g = np.empty(V, dtype=np.int32)
    chunk = max_batch * (K + 1)
    all_ids = torch.arange(V, dtype=torch.int32, device=dev)
    for s0 in range(0, V, chunk):
        n = min(chunk, V - s0)
        Bn = (n + K) // (K + 1)
        ids = torch.zeros(Bn * (K + 1), dtype=torch.int32, device=dev)
        ids[:n] = all_ids[s0:s0 + n]
        ids = ids.view(Bn, K + 1)
        tg = ctx.step(ids[:, 0].contiguous(), ids[:, 1:].contiguous() if K else None)
        g[s0:s0 + n] = tg.view(-1)[:n].cpu().numpy()
    return g


class Plan:
    """A decode trajectory planned on the host from a greedy table: every
    step's inputs, its expected commits and the tokens it counts."""

    def __init__(self, g, rank, B, K, p, total):
        traj = Trajectory(g, rank, B=B, K=K, p=p)
        self.ctx = np.empty((total, B), np.int32)
        self.dr = np.empty((total, B, K), np.int32)
        self.com = np.empty((total, B, K + 1), np.int32)
        self.alen = np.empty((total, B), np.int32)
        self.counted = np.zeros(total, np.int64)
        for i in range(total):
            c, d = traj.drafts()
            com, n = traj.expected(c, d)
            self.ctx[i], self.dr[i], self.com[i], self.alen[i] = c, d, com, n
            self.counted[i] = traj.advance(com, n)


class StepGraph:
    """step + accept on fixed buffers, captured as one CUDA graph; each replay
    copies the step's inputs in from HBM and its outputs out."""

    def __init__(self, ctx, B, K, dev, stamps=None):
        import torch
        self.B, self.K = B, K
        self.in_ctx = torch.zeros((B,), dtype=torch.int32, device=dev)
        self.in_dr = torch.zeros((B, K), dtype=torch.int32, device=dev)
        self.tg = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        self.com = torch.empty_like(self.tg)
        self.alen = torch.empty((B,), dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.stream.wait_stream(torch.cuda.current_stream())
        dr = self.in_dr if K else None

        def body():
            ctx.step(self.in_ctx, dr, target_ids=self.tg, stream=self.stream)
            ctx.accept(dr, self.tg, committed=self.com, accept_len=self.alen, stream=self.stream)

        with torch.cuda.stream(self.stream):
            body()
        self.stream.synchronize()
        if stamps is not None:
            ctx.set_stamps(stamps)
        try:
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                body()
        finally:
            if stamps is not None:
                ctx.set_stamps(None)
        torch.cuda.current_stream().wait_stream(self.stream)

    def run(self, d_ctx, d_dr, i, d_com=None, d_alen=None):
        self.in_ctx.copy_(d_ctx[i], non_blocking=True)
        if self.K:
            self.in_dr.copy_(d_dr[i], non_blocking=True)
        self.graph.replay()
        if d_com is not None:
            d_com[i].copy_(self.com, non_blocking=True)
            d_alen[i].copy_(self.alen, non_blocking=True)


def timed_plan(ctx, plan, B, K, warmup, steps, dev, dist=None, clocks=None):
    """Replays the plan's steps through one step graph; returns (ms for the
    timed steps, commits [steps, B, K+1], accept lengths [steps, B], clocks)."""
    import torch
    d_ctx = torch.from_numpy(plan.ctx).to(dev)
    d_dr = torch.from_numpy(plan.dr).to(dev)
    total = warmup + steps
    d_com = torch.empty((total, B, K + 1), dtype=torch.int32, device=dev)
    d_alen = torch.empty((total, B), dtype=torch.int32, device=dev)
    sg = StepGraph(ctx, B, K, dev)
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        sg.run(d_ctx, d_dr, i, d_com, d_alen)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    ev0.record(stream)
    for i in range(warmup, total):
        sg.run(d_ctx, d_dr, i, d_com, d_alen)
    ev1.record(stream)
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    if dist:
        dist.barrier()
    clk = None
    if clocks:
        time.sleep(0.2)
        clocks.stop()
        clk = clocks.summary(w0, w1)
    ms = ev0.elapsed_time(ev1)
    return ms, d_com[warmup:].cpu().numpy(), d_alen[warmup:].cpu().numpy(), clk


def probe_pass(ctx, cfg, plan, B, K, first, n, dev):
    """Routing of steps first .. first+n-1 of a plan (eager, with the probe):
    returns a list of topk_idx [L, T, k] arrays."""
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND
    T = B * (K + 1)
    probe, pt = BND.make_probe(cfg.n_layers, T, cfg, topk=True, hidden=False, device=dev)
    out = []
    for i in range(first, first + n):
        ctx.step(torch.from_numpy(plan.ctx[i]).to(dev),
                 torch.from_numpy(plan.dr[i]).to(dev) if K else None, probe=probe)
        out.append(pt["topk_idx"].cpu().numpy())
    return out


def fractions(bytes_per_step, flops_per_step, ms_per_step, peaks):
    hbm, _, tf_sus, _ = peaks
    gbs = bytes_per_step / (ms_per_step * 1e-3) / 1e9
    tfs = flops_per_step / (ms_per_step * 1e-3) / 1e12
    return {"hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "tensor_tflops": round(tfs, 1), "tensor_frac": round(tfs / tf_sus, 4)}


def in_graph_stamps(ctx, cfg, plan, B, K, first, n, dev):
    """Per-launch device times of the step's kernels inside a graph-replayed
    step (launch timestamps): returns arrays [n, 2L+1, 3] of (start, ready,
    end) in ns relative to each step's first start."""
    import torch
    L = cfg.n_layers
    stamps = torch.zeros((2 * L + 1, 4), dtype=torch.int64, device=dev)
    init = torch.zeros_like(stamps)
    init[:, 0] = -1
    sg = StepGraph(ctx, B, K, dev, stamps=stamps)
    d_ctx = torch.from_numpy(plan.ctx).to(dev)
    d_dr = torch.from_numpy(plan.dr).to(dev)
    out = []
    for i in range(first, first + n):
        stamps.copy_(init)
        sg.run(d_ctx, d_dr, i)
        torch.cuda.synchronize()
        st = stamps.cpu().numpy().view(np.uint64)[:, :3].astype(np.float64)
        out.append(st - st[0, 0])
    return np.stack(out)


def run_ours(args, rank, world, local):
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    base = S.FULL_ZIPF if args.zipf else S.FULL
    cfg = base if not args.layers else __import__("dataclasses").replace(base, n_layers=args.layers)
    # the workload's batch shape; profiling runs may time another one
    Bq = args.batch if (args.profile and args.batch) else B_SEQ
    Kq = args.drafts if (args.profile and args.drafts is not None) else K_DRAFT
    t_setup = time.perf_counter()
    w_host = S.make_weights(cfg)
    w_dev = BND.weights_to_device(w_host, device=dev)
    ctx = BND.MoeVerify(cfg, w_dev, max_batch=Bq if args.profile else 1024,
                        max_k=Kq if args.profile else K_DRAFT)
    ctx.set_layer_kernel(args.layer_kernel)
    del w_dev
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()

    # the library's greedy table over the whole vocabulary (profiling runs use
    # a random table instead: same kernels, same shapes)
    V = cfg.vocab
    if args.profile:
        g = S.uniform_ids(V, 99, 0, V).astype(np.int32)
    else:
        g = greedy_table(ctx, V, Kq, dev, 1024)
    assert ctx.sync_status() == BND.OK

    total = args.warmup + args.steps
    plan = Plan(g, rank, Bq, Kq, P_MATCH, total)
    setup_s = time.perf_counter() - t_setup

    clocks = ClockSampler(local)
    ms, got_com, got_alen, clk = timed_plan(ctx, plan, Bq, Kq, args.warmup, args.steps, dev,
                                            dist, clocks)

    if args.profile and args.attn:
        line = run_attn(w_host, args, dev, peaks, B=Bq, K=Kq, layers=args.layers)
        line["clocks"] = clk
        if rank == 0:
            print(json.dumps(line), flush=True)
        ctx.close()
        return

    if args.profile and args.draft_head:
        line = run_decode_iteration(args, ctx, cfg, w_host, dev, Bq, Kq, stream)
        line["clocks"] = clk
        if rank == 0:
            print(json.dumps(line), flush=True)
        ctx.close()
        return

    if args.profile:
        # per-launch windows inside the graph-replayed step (launch timestamps)
        st = in_graph_stamps(ctx, cfg, plan, Bq, Kq, args.warmup, args.steps, dev)
        L = cfg.n_layers
        win = (st[:, :, 2] - st[:, :, 1]) * 1e-3  # us
        if rank == 0:
            print(json.dumps({"profile": True, "layers": cfg.n_layers, "batch": Bq, "drafts": Kq,
                              "zipf": bool(args.zipf), "steps": args.steps,
                              "ms_per_step": round(ms / args.steps, 4),
                              "in_graph_us": {
                                  "ffn_per_layer": [round(x, 2) for x in win[:, 1:2 * L:2].mean(0)],
                                  "routing_per_layer": [round(x, 2)
                                                        for x in win[:, 0:2 * L:2].mean(0)],
                                  # from the previous launch's end to the routing's end
                                  # (all of the routing's blocks, every wave)
                                  "routing_span_per_layer": [
                                      round(x, 2) for x in
                                      ((st[:, 2:2 * L:2, 2] - st[:, 1:2 * L - 1:2, 2]) * 1e-3)
                                      .mean(0)],
                                  "layer_period": round(float(np.mean(np.diff(
                                      st[:, 1:2 * L:2, 2], axis=1))) * 1e-3, 2),
                                  "lm_head": round(float(win[:, 2 * L].mean()), 2),
                                  "step_span": round(float(st[:, 2 * L, 2].mean()) * 1e-3, 2)},
                              "clocks": clk}), flush=True)
        ctx.close()
        return

    # every timed step committed exactly what the planned trajectory says
    mism = int(np.sum(np.any(got_com != plan.com[args.warmup:], axis=2)) +
               np.sum(got_alen != plan.alen[args.warmup:]))
    status = ctx.sync_status()
    tokens = float(plan.counted[args.warmup:].sum())

    # end to end: the same steps through the host-buffer entry point
    e_tokens, e_s = run_e2e(ctx, g, rank, Bq, Kq, args, dist)

    # roofline of the dominant kernel (the expert FFN), weights-only bytes:
    # in-graph launch times from the launch timestamps, and the
    # event-bracketed (serialised) launch times beside them
    T = Bq * (Kq + 1)
    routing = probe_pass(ctx, cfg, plan, Bq, Kq, args.warmup, args.steps, dev)
    ffn_bytes = [expert_weight_bytes(idx[l], cfg) for idx in routing for l in range(cfg.n_layers)]
    st = in_graph_stamps(ctx, cfg, plan, Bq, Kq, args.warmup, args.steps, dev)
    L = cfg.n_layers
    ffn_win = (st[:, 1:2 * L:2, 2] - st[:, 1:2 * L:2, 1]) * 1e-6      # ms, [steps, L]
    ffn_start = (st[:, 1:2 * L:2, 2] - st[:, 1:2 * L:2, 0]) * 1e-6
    layer_period = np.diff(np.concatenate([np.zeros((st.shape[0], 1)), st[:, 1:2 * L:2, 2]],
                                          axis=1), axis=1) * 1e-6
    lm_win = (st[:, 2 * L, 2] - st[:, 2 * L, 1]) * 1e-6
    route_win = (st[:, 0:2 * L:2, 2] - st[:, 0:2 * L:2, 1]) * 1e-6
    ffn_ms_graph = float(np.mean(ffn_win))
    ctx.set_timing(True)
    ctx.get_timing(reset=True)
    d_ctx = torch.from_numpy(plan.ctx).to(dev)
    d_dr = torch.from_numpy(plan.dr).to(dev)
    for i in range(args.warmup, total):
        tg = ctx.step(d_ctx[i], d_dr[i])
        ctx.accept(d_dr[i], tg)
    fam_ms, fam_n = ctx.get_timing(reset=True)
    ctx.set_timing(False)
    ffn_ms_events = fam_ms[0] / max(1, fam_n[0])
    mean_ffn_bytes = float(np.mean(ffn_bytes))
    achieved = mean_ffn_bytes / (ffn_ms_graph * 1e-3) / 1e9
    traffic, traffic_note = stored_traffic()
    flops = step_flops(cfg, T)
    sbytes = float(np.mean([step_bytes(idx, cfg, T) for idx in routing]))

    # the other workloads, measured in the same run
    configs = {
        "single_layer_t4": run_single_layer(ctx, cfg, dev, peaks),
        "zipf_b256_k3_p0.576": run_zipf(w_host, rank, args, dev, peaks),
        "sweep": run_sweep(ctx, cfg, g, rank, dev, peaks),
        f"attn_b32_k3_pos{ATTN_LO}_{ATTN_HI}": run_attn(w_host, args, dev, peaks,
                                                         steps=min(args.steps, 20)),
    }

    if dist:
        ms, e_s, tokens, e_tokens = whole_job(ms, e_s, tokens, e_tokens, dev)
    value = tokens / (ms / 1e3)
    ms_step = ms / args.steps
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights, uniform start ids, drafts right w.p. 0.75)",
        "config": {"workload": WORKLOAD, "layers": cfg.n_layers, "hidden": cfg.hidden,
                   "experts": f"{cfg.n_experts}x{cfg.expert_inter} top-{cfg.top_k} + "
                              f"{cfg.n_shared} shared", "vocab": cfg.vocab, "batch": Bq,
                   "drafts": Kq, "p_match": P_MATCH, "page_tokens": PAGE_TOKENS,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (5.8 GB of weights per step)",
                   "cuda_graph": True},
        "e2e": {"value": round(e_tokens / e_s, 1), "unit": UNIT,
                "h2d_bytes_per_step": Bq * 4 + Bq * Kq * 4,
                "d2h_bytes_per_step": Bq * (Kq + 1) * 4 + Bq * 4},
        "gpu_launches": int(args.steps * (2 * cfg.n_layers + 3)),
        "roofline": {"kernel": "expert FFN (gate/up + SwiGLU + down + combine)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peaks[0], "unit": "GB/s",
                     "frac": round(achieved / peaks[0], 4), "peak_source": peaks[3],
                     "traffic": traffic, "traffic_note": traffic_note,
                     "alg_bytes_per_launch": round(mean_ffn_bytes),
                     "alg_bytes": "touched experts' gate, up and down weights, once",
                     "launch_ms": round(ffn_ms_graph, 5),
                     "launch_ms_source": "in-graph launch timestamps: last CTA end minus the "
                                         "return of the wait for the routing kernel",
                     "launch_ms_from_cta_start": round(float(np.mean(ffn_start)), 5),
                     "launch_ms_events": round(ffn_ms_events, 5),
                     "tensor": dict(scope="whole step, selected-expert flops",
                                    flops_per_step=round(flops),
                                    **{k: v for k, v in fractions(sbytes, flops, ms_step,
                                                                  peaks).items()
                                       if k.startswith("tensor")},
                                    peak_tflops=peaks[2], peak_kind="bf16 sustained")},
        "step": dict(alg_bytes_per_step=round(sbytes), **fractions(sbytes, flops, ms_step, peaks)),
        "in_graph_ms": {"ffn_per_layer": round(ffn_ms_graph, 5),
                        "layer_period": round(float(np.mean(layer_period[:, 1:])), 5),
                        "routing_per_layer": round(float(np.mean(route_win)), 5),
                        "lm_head": round(float(np.mean(lm_win)), 5)},
        "configs": configs,
        "clocks": clk,
        "committed_per_step": round(tokens / args.steps / world, 3),
        "check": {"mismatched_rows": mism, "status": status},
        "setup_s": round(setup_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = cpu_baseline(cfg, w_host, plan, g,
                                                            args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if dist:
        dist.destroy_process_group()


def stored_traffic():
    """ncu's DRAM bytes per expert-FFN launch, if they were taken on the
    kernels that run now (else None, with the reason)."""
    prof = os.path.join(ROOT, "profiles", "ffn_traffic.json")
    if not os.path.exists(prof):
        return None, "no ncu capture stored"
    with open(prof) as f:
        d = json.load(f)
    if d.get("kernel_digest") != kernel_digest():
        return None, "kernel sources changed since the ncu capture"
    return d.get("bytes_per_launch"), d.get("note", "")


def run_e2e(ctx, g, rank, Bq, Kq, args, dist):
    """The timed steps through moe_verify_decode_host on pinned host buffers,
    with the host building each next step's drafts."""
    import torch
    h_ctx = torch.empty((Bq,), dtype=torch.int32, pin_memory=True).numpy()
    h_dr = torch.empty((Bq, Kq), dtype=torch.int32, pin_memory=True).numpy()
    h_com = torch.empty((Bq, Kq + 1), dtype=torch.int32, pin_memory=True).numpy()
    h_alen = torch.empty((Bq,), dtype=torch.int32, pin_memory=True).numpy()
    etraj = Trajectory(g, rank, B=Bq, K=Kq)
    cur = torch.cuda.current_stream()
    c, d = etraj.drafts()
    for i in range(args.warmup):
        h_ctx[:], h_dr[:] = c, d
        ctx.decode_host(h_ctx, h_dr, h_com, h_alen, stream=cur)
        etraj.advance(h_com, h_alen)
        c, d = etraj.drafts()
    e_tokens = 0
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = time.perf_counter()
    for i in range(args.steps):
        h_ctx[:], h_dr[:] = c, d
        ctx.decode_host(h_ctx, h_dr, h_com, h_alen, stream=cur)
        e_tokens += etraj.advance(h_com, h_alen)
        c, d = etraj.drafts()
    e1 = time.perf_counter()
    return e_tokens, e1 - e0


def run_single_layer(ctx, cfg, dev, peaks, reps=20):
    """One decoder block on T = 4 bf16 hidden rows through moe_verify_layer,
    cycling over the 12 distinct layers of the stack (12 x ~160 MB, far more
    than L2, so no repeat is served from L2): device time per call and the
    touched weights' bytes per second."""
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND
    T, L = 4, cfg.n_layers
    hin = S.hidden_input(T, cfg.hidden, seed=S.SEED_HIDDEN)
    h_in = torch.from_numpy(hin.view(np.int16)).to(dev).view(torch.bfloat16)
    h_out = torch.empty_like(h_in)
    probe, pt = BND.make_probe(1, T, cfg, topk=True, hidden=False, device=dev)
    nbytes = []
    for l in range(L):
        ctx.layer(l, h_in, h_out=h_out, probe=probe)
        idx = pt["topk_idx"].cpu().numpy()[0]
        nbytes.append(expert_weight_bytes(idx, cfg) + cfg.n_experts * cfg.hidden * 2 +
                      cfg.hidden * 2 + 2 * T * cfg.hidden * 2)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l in range(L):
            ctx.layer(l, h_in, h_out=h_out, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for l in range(L):
            ctx.layer(l, h_in, h_out=h_out, stream=s)
    with torch.cuda.stream(s):
        for _ in range(3):
            graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            graph.replay()
        e1.record(s)
    torch.cuda.synchronize()
    ms_call = e0.elapsed_time(e1) / (reps * L)
    b = float(np.mean(nbytes))
    gbs = b / (ms_call * 1e-3) / 1e9
    return {"tokens": T, "layers_cycled": L, "calls": reps * L, "ms_per_call": round(ms_call, 5),
            "alg_bytes_per_call": round(b), "hbm_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks[0], 4),
            "entry_point": "moe_verify_layer (routing + expert FFN + bf16 output), graph-replayed"}


def run_zipf(w_host, rank, args, dev, peaks):
    """Batch 256 x (1 + 3 drafts) on the stack with the Zipf(s=1.2) router
    bias, drafts right with probability 0.576: committed tokens/s, time per
    step and both roofline fractions (touched experts' bytes; selected-expert
    flops against the sustained bf16 peak)."""
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND
    cfg = S.FULL_ZIPF
    B, K, p = 256, 3, 0.576
    w = dict(w_host)
    w["router_bias"] = S.router_bias(cfg)
    ctx = BND.MoeVerify(cfg, BND.weights_to_device(w, device=dev), max_batch=B, max_k=K)
    torch.cuda.empty_cache()
    try:
        g = greedy_table(ctx, cfg.vocab, K, dev, B)
        total = args.warmup + args.steps
        plan = Plan(g, rank, B, K, p, total)
        ms, com, alen, _ = timed_plan(ctx, plan, B, K, args.warmup, args.steps, dev)
        mism = int(np.sum(np.any(com != plan.com[args.warmup:], axis=2)) +
                   np.sum(alen != plan.alen[args.warmup:]))
        routing = probe_pass(ctx, cfg, plan, B, K, args.warmup, min(args.steps, 5), dev)
        T = B * (K + 1)
        sbytes = float(np.mean([step_bytes(idx, cfg, T) for idx in routing]))
        touched = float(np.mean([[len(np.unique(idx[l])) for l in range(cfg.n_layers)]
                                 for idx in routing]))
        top_share = float(np.mean([np.bincount(idx[l].reshape(-1), minlength=cfg.n_experts).max()
                                   / T for idx in routing for l in range(cfg.n_layers)]))
        ms_step = ms / args.steps
        fr = fractions(sbytes, step_flops(cfg, T), ms_step, peaks)
        status = ctx.sync_status()
    finally:
        ctx.close()
    tokens = float(plan.counted[args.warmup:].sum())
    out = {"batch": B, "drafts": K, "p_match": p, "steps": args.steps,
           "value": round(tokens / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms_step, 4),
           "committed_per_step": round(tokens / args.steps, 2),
           "alg_bytes_per_step": round(sbytes), "flops_per_step": round(step_flops(cfg, T)),
           "touched_routed_experts_per_layer": round(touched, 1),
           "busiest_expert_token_share": round(top_share, 3)}
    out.update(fr)
    out["binding"] = "tensor" if fr["tensor_frac"] > fr["hbm_frac"] else "hbm"
    out["check"] = {"mismatched_rows": mism, "status": status}
    return out


def run_sweep(ctx, cfg, g, rank, dev, peaks, warmup=3, steps=10):
    """B in {1, 8, 32, 128} x K in {1, 2, 3} x p in {0.576, 0.75}: committed
    tokens/s, time per step and roofline fractions per point.  Each entry is
    [B, K, p, ms_per_step, tokens_per_s, hbm_frac, tensor_frac]."""
    out, mism = [], 0
    for B in (1, 8, 32, 128):
        for K in (1, 2, 3):
            for p in (0.576, 0.75):
                plan = Plan(g, rank, B, K, p, warmup + steps)
                ms, com, alen, _ = timed_plan(ctx, plan, B, K, warmup, steps, dev)
                mism += int(np.sum(np.any(com != plan.com[warmup:], axis=2)) +
                            np.sum(alen != plan.alen[warmup:]))
                T = B * (K + 1)
                routing = probe_pass(ctx, cfg, plan, B, K, warmup, 2, dev)
                sbytes = float(np.mean([step_bytes(idx, cfg, T) for idx in routing]))
                fr = fractions(sbytes, step_flops(cfg, T), ms / steps, peaks)
                tok = float(plan.counted[warmup:].sum())
                out.append([B, K, p, round(ms / steps, 4), round(tok / (ms / 1e3), 1),
                            fr["hbm_frac"], fr["tensor_frac"]])
    return {"columns": ["batch", "drafts", "p_match", "ms_per_step", "tokens_per_s", "hbm_frac",
                        "tensor_frac"], "steps_per_point": steps, "points": out,
            "check": {"mismatched_rows": mism}}


ATTN_LO, ATTN_HI = 512, 4096


def run_attn(w_host, args, dev, peaks, B=32, K=3, lo=ATTN_LO, hi=ATTN_HI, steps=None, layers=0):
    """The stack with attention (the library's reading of the decoder's
    unspecified attention: 10 heads of 128, rotary positions, a bf16 key/value
    cache), B=32 sequences at positions drawn uniformly from [512, 4096), K=3
    drafts.  Each sequence's cache holds the keys and values of a synthetic
    prompt, fed through the verify call beforehand (calls of 16 tokens); the
    timed step re-verifies the prompt's tokens at each sequence's position
    (the same cache rows are rewritten).  Returns verify tokens/s, the time per
    step, each kernel's in-graph time per launch, and the attention kernel's
    roofline: its bytes are every cached key and value of the sequences'
    positions once, plus q read and the output written."""
    import dataclasses
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND
    cfg = S.FULL_ATTN if not layers else dataclasses.replace(S.FULL_ATTN, n_layers=layers)
    L, d = cfg.n_layers, cfg.hidden
    steps = steps or args.steps
    w = dict(w_host)
    w.update(S.make_attn_weights(cfg))
    pos = (lo + S.uniform_ids(B, 8, 0, hi - lo - K)).astype(np.int64)
    n = int(-(-(int(pos.max()) + K + 1) // 16) * 16)
    ctx = BND.MoeVerify(cfg, BND.weights_to_device(w, device=dev), max_batch=B, max_k=15,
                        max_pos=n)
    del w
    torch.cuda.empty_cache()
    try:
        prompts = S.uniform_ids(B * n, 7, 0, cfg.vocab, 123456789).astype(np.int64).reshape(B, n)
        d_prompts = torch.from_numpy(prompts.astype(np.int32)).to(dev)
        for p0 in range(0, n, 16):
            ctx.step_attn(d_prompts[:, p0].contiguous(), d_prompts[:, p0 + 1:p0 + 16].contiguous(),
                          torch.full((B,), p0, dtype=torch.int32, device=dev))
        torch.cuda.synchronize()
        rows = np.arange(B)
        in_ctx = torch.from_numpy(prompts[rows, pos].astype(np.int32)).to(dev)
        in_dr = torch.from_numpy(np.stack([prompts[b, pos[b] + 1: pos[b] + 1 + K]
                                           for b in range(B)]).astype(np.int32)).to(dev)
        in_pos = torch.from_numpy(pos.astype(np.int32)).to(dev)
        tg = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
        com = torch.empty_like(tg)
        alen = torch.empty((B,), dtype=torch.int32, device=dev)
        stamps = torch.zeros((6 * L + 1, 4), dtype=torch.int64, device=dev)
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())

        def body():
            ctx.step_attn(in_ctx, in_dr, in_pos, target_ids=tg, stream=s)
            ctx.accept(in_dr, tg, committed=com, accept_len=alen, stream=s)

        graphs = []
        for with_stamps in (False, True):
            with torch.cuda.stream(s):
                body()
            s.synchronize()
            if with_stamps:
                ctx.set_stamps(stamps)
            try:
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=s):
                    body()
            finally:
                ctx.set_stamps(None)
            graphs.append(gr)
        with torch.cuda.stream(s):
            for _ in range(args.warmup):
                graphs[0].replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(steps):
                graphs[0].replay()
            e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        # per-launch windows (last CTA end minus the latest return of the wait
        # for the preceding launch), averaged over replays
        init = torch.zeros_like(stamps)
        init[:, 0] = -1
        wins = []
        for _ in range(min(steps, 10)):
            stamps.copy_(init)
            with torch.cuda.stream(s):
                graphs[1].replay()
            s.synchronize()
            st = stamps.cpu().numpy().view(np.uint64)[:, :3].astype(np.float64)
            wins.append((st[:, 2] - st[:, 1]) * 1e-6)
        win = np.mean(np.stack(wins), axis=0)  # ms per launch slot
        status = ctx.sync_status()
    finally:
        ctx.close()
    T = B * (K + 1)
    keys = float(np.sum(pos + K + 1))
    attn_bytes = keys * d * 2 * 2 + T * d * 4 + T * d * 2
    attn_ms = float(np.mean(win[2:6 * L:6]))
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    rows_qkv = -(-3 * d // 128) * 128
    qkv_bytes = rows_qkv * d * 2 + T * d * 2 + T * d * 4 + 2 * T * d * 2
    o_bytes = d * d * 2 + T * d * 2 + 2 * T * d * 4
    qkv_ms, o_ms = float(np.mean(win[1:6 * L:6])), float(np.mean(win[3:6 * L:6]))
    kib = {"attn_rmsnorm": win[0:6 * L:6], "qkv_projection": win[1:6 * L:6],
           "attention": win[2:6 * L:6], "o_projection": win[3:6 * L:6],
           "routing": win[4:6 * L:6], "expert_ffn": win[5:6 * L:6]}
    return {"batch": B, "drafts": K, "positions": f"uniform in [{lo}, {hi})",
            "mean_position": round(float(pos.mean()), 1), "steps": steps,
            "value": round(T / (ms * 1e-3), 1), "unit": "verify tokens/s",
            "ms_per_step": round(ms, 4),
            "in_graph_ms_per_launch": {k: round(float(np.mean(v)), 5) for k, v in kib.items()},
            "in_graph_ms_lm_head": round(float(win[6 * L]), 5),
            "roofline": {"kernel": "attention over the key/value cache", "bound": "hbm",
                         "achieved": round(achieved, 1), "peak": peaks[0], "unit": "GB/s",
                         "frac": round(achieved / peaks[0], 4), "peak_source": peaks[3],
                         "alg_bytes_per_launch": round(attn_bytes),
                         "alg_bytes": "each sequence's cached keys and values of positions "
                                      "0 .. pos + K once, q read, output written",
                         "launch_ms": round(attn_ms, 5),
                         "launch_ms_source": "in-graph launch timestamps"},
            "projections": {"qkv_gbs": round(qkv_bytes / (qkv_ms * 1e-3) / 1e9, 1),
                            "o_gbs": round(o_bytes / (o_ms * 1e-3) / 1e9, 1),
                            "alg_bytes": "weights once, activations in and out"},
            "cache_fill": f"{n} prompt tokens per sequence through the verify call (16 per call)",
            "check": {"status": status}}


def whole_job(ms, e_s, tokens, e_tokens, device):
    """Whole-job figures over the ranks of the default process group: the
    slowest rank's device and end-to-end times, every rank's committed tokens."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, e_s, tokens, e_tokens], dtype=torch.float64, device=device)
    mx, sm = t.clone(), t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(mx[1]), float(sm[2]), float(sm[3])


def run_decode_iteration(args, ctx, cfg, w_host, dev, Bq, Kq, stream):
    """Timing of one whole decode iteration on the device (profiling only):
    verify step + accept + draft inputs + the FastMTP draft head (K steps),
    captured as one CUDA graph whose outputs feed its inputs, so replays run
    the decode loop autonomously.  The draft head has random weights, so its
    drafts are rarely accepted; the line reports time, not speed-up."""
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND
    dw = S.make_draft_weights(S.DRAFT, w_host)
    dctx = BND.MoeVerify(S.DRAFT, BND.weights_to_device(dw, device=dev), max_batch=Bq, max_k=0)
    start = torch.from_numpy(S.start_ids(Bq, cfg.vocab).astype(np.int32)).to(dev)
    in_c = start.clone()
    in_d = torch.zeros((Bq, Kq), dtype=torch.int32, device=dev)
    tg = torch.empty((Bq, Kq + 1), dtype=torch.int32, device=dev)
    com, alen = torch.empty_like(tg), torch.empty((Bq,), dtype=torch.int32, device=dev)
    h = torch.empty((Bq, cfg.hidden), dtype=torch.float32, device=dev)
    t = torch.empty((Bq,), dtype=torch.int32, device=dev)
    out_d = torch.empty((Bq, Kq), dtype=torch.int32, device=dev)
    committed = torch.zeros((), dtype=torch.int64, device=dev)
    cs = torch.cuda.Stream(device=dev)
    cs.wait_stream(stream)

    def iteration(draft=True):
        ctx.step(in_c, in_d, target_ids=tg, stream=cs)
        ctx.accept(in_d, tg, committed=com, accept_len=alen, stream=cs)
        ctx.draft_inputs(com, alen, h_out=h, t_out=t, stream=cs)
        if draft:
            dctx.draft(h, t, Kq, drafts=out_d, stream=cs)
        committed.add_((alen + 1).sum())
        in_c.copy_(t)
        in_d.copy_(out_d)

    graphs = {}
    for key in (True, False):
        with torch.cuda.stream(cs):
            iteration(key)
        cs.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            iteration(key)
        graphs[key] = g
    times = {}
    for key in (True, False):
        # replays and events on the same stream (a replay runs on the
        # current stream)
        with torch.cuda.stream(cs):
            in_c.copy_(start)
            in_d.zero_()
            for _ in range(args.warmup):
                graphs[key].replay()
            cs.synchronize()
            committed.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cs)
            for _ in range(args.steps):
                graphs[key].replay()
            e1.record(cs)
        torch.cuda.synchronize()
        times[key] = (e0.elapsed_time(e1) / args.steps, float(committed.item()) / args.steps)
    status = (ctx.sync_status(), dctx.sync_status())
    dctx.close()
    ms_it, com_it = times[True]
    ms_verify = times[False][0]
    return {"profile": True, "decode_iteration": True, "batch": Bq, "drafts": Kq,
            "steps": args.steps, "ms_per_iteration": round(ms_it, 4),
            "ms_verify_accept": round(ms_verify, 4), "ms_draft_head": round(ms_it - ms_verify, 4),
            "committed_per_iteration": round(com_it, 2),
            "note": "random draft weights: drafts are rarely accepted", "status": list(status)}


# ------------------------------------------------------------ CPU baseline

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_baseline(cfg, w_host, plan, g, budget_s=20.0):
    """The oracle, as it stands, on a bounded sample of the workload's verify
    tokens (one token per thread at a time), scaled to committed tokens/s.
    Its targets are also compared with the library's greedy table, which the
    timed steps' commits were checked against: returns (baseline, parity)."""
    import oracle as O
    orc = O.Oracle(cfg, w_host)
    toks = np.concatenate([plan.ctx[..., None], plan.dr], axis=2).reshape(-1)
    cores = _cores()
    import concurrent.futures as fut
    done = 0
    res = []
    t0 = time.perf_counter()
    with fut.ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < budget_s and done < len(toks):
            batch = toks[done:done + cores]
            res += list(ex.map(orc.forward_token, batch))
            done += len(batch)
    dt = time.perf_counter() - t0
    per_verify_token = float(plan.counted.sum()) / (len(plan.counted) * B_SEQ * (K_DRAFT + 1))
    value = done / dt * per_verify_token
    base = {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} verify tokens of the workload's first steps in {dt:.1f} s "
                      f"(fp64, one token per thread), scaled by {per_verify_token:.3f} committed "
                      f"tokens per verify token"}
    diffs = [(int(x), r["logit_gap"]) for x, r in zip(toks[:done], res)
             if r["target"] != int(g[int(x)])]
    parity = {"verify_tokens": done, "target_diffs": len(diffs),
              "diff_logit_gaps": [round(gap, 5) for _, gap in diffs],
              "what": "free-running fp64 oracle targets vs the library's targets for the same "
                      "tokens of the timed trajectory (a difference needs a small oracle gap)"}
    return base, parity


# -------------------------------------------------------- reference arm

def run_reference(args, rank, world, local):
    """The oracle timed as the reference arm: each step evaluates one verify
    token per host core (a bounded sample of one verify step)."""
    if rank != 0:
        return
    import oracle as O
    cfg = S.FULL
    w_host = S.make_weights(cfg)
    orc = O.Oracle(cfg, w_host)
    cores = _cores()
    V = cfg.vocab
    toks = S.uniform_ids((args.warmup + args.steps) * cores, S.SEED_START_IDS, 11, V)
    import concurrent.futures as fut
    per_verify_token = expected_commit_ratio()
    with fut.ThreadPoolExecutor(max_workers=cores) as ex:
        for i in range(args.warmup):
            list(ex.map(orc.target, toks[i * cores:(i + 1) * cores]))
        t0 = time.perf_counter()
        for i in range(args.warmup, args.warmup + args.steps):
            list(ex.map(orc.target, toks[i * cores:(i + 1) * cores]))
        dt = time.perf_counter() - t0
    value = args.steps * cores / dt * per_verify_token
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": f"{cores} verify tokens per step"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{cores} verify tokens per step (one per thread), scaled by "
                                   f"{per_verify_token:.4f} committed tokens per verify token"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def expected_commit_ratio():
    """Committed tokens per verify token when each draft matches w.p. p:
    (1 + p + ... + p^K) / (K + 1)."""
    return sum(P_MATCH ** i for i in range(K_DRAFT + 1)) / (K_DRAFT + 1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--profile", action="store_true",
                    help="timing loop only (random greedy table; no e2e, roofline or CPU legs)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: a shorter stack (same per-layer shapes)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling only: sequences per step (default 32)")
    ap.add_argument("--drafts", type=int, default=None,
                    help="profiling only: drafts per sequence, 0..15 (default 3)")
    ap.add_argument("--zipf", action="store_true",
                    help="profiling only: the stack with the Zipf(s=1.2) router bias")
    ap.add_argument("--draft-head", action="store_true",
                    help="profiling only: time whole decode iterations with the FastMTP draft head")
    ap.add_argument("--attn", action="store_true",
                    help="profiling only: the stack with attention at positions in [512, 4096)")
    ap.add_argument("--layer-kernel", type=int, default=0,
                    help="profiling only: steps of at most this many verify tokens route inside "
                         "the expert-FFN kernel (0..8; 0, the default: a routing launch per layer)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if (args.layers or args.batch or args.drafts is not None or args.draft_head
            or args.zipf or args.attn) and not args.profile:
        ap.error("--layers, --batch, --drafts, --zipf, --draft-head and --attn are for "
                 "profiling runs only (--profile)")
    if args.layer_kernel and not args.profile:
        ap.error("--layer-kernel is for profiling runs only (--profile)")
    if not 0 <= args.layer_kernel <= 8:
        ap.error("--layer-kernel must be in 0..8")
    if args.attn and (args.zipf or args.draft_head):
        ap.error("--attn runs the stack without the Zipf bias or the draft head")
    if args.draft_head and (args.layers or (args.drafts is not None and args.drafts < 1)):
        ap.error("--draft-head needs the full stack and at least one draft")
    if args.drafts is not None and not 0 <= args.drafts <= 15:
        ap.error("--drafts must be in 0..15")
    if (args.batch or B_SEQ) * ((K_DRAFT if args.drafts is None else args.drafts) + 1) > 4096:
        ap.error("--batch x (--drafts + 1) must be at most 4096 verify tokens")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
