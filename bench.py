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
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def algorithmic_ffn_bytes(topk_idx: np.ndarray, cfg) -> float:
    """Bytes one expert-FFN launch (one layer) must move at least: the gate,
    up and down weights of every touched expert (routed + shared) once, the
    expert-major normalised inputs read once, the SwiGLU rows written and read
    once (bf16), and the weighted fp32 outputs written once.  topk_idx: [T, k]."""
    T = topk_idx.shape[0]
    touched = len(np.unique(topk_idx)) + cfg.n_shared
    rows = T * (cfg.top_k + cfg.n_shared)
    d, I = cfg.hidden, cfg.expert_inter
    return touched * 3 * I * d * 2 + rows * d * 2 + 2 * rows * I * 2 + rows * d * 4


def run_ours(args, rank, world, local):
    import torch
    from moe_speculative_decoding_router_gb300 import binding as BND

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    cfg = S.FULL if not args.layers else __import__("dataclasses").replace(S.FULL, n_layers=args.layers)
    # the workload's batch shape; profiling runs may time another one
    Bq = args.batch if (args.profile and args.batch) else B_SEQ
    Kq = args.drafts if (args.profile and args.drafts is not None) else K_DRAFT
    t_setup = time.perf_counter()
    w_host = S.make_weights(cfg)
    w_dev = BND.weights_to_device(w_host, device=dev)
    ctx = BND.MoeVerify(cfg, w_dev, max_batch=Bq if args.profile else 1024,
                        max_k=Kq if args.profile else K_DRAFT)
    del w_dev
    torch.cuda.empty_cache()
    stream = torch.cuda.current_stream()

    # greedy table g over the whole vocabulary, 4,096 verify tokens per call
    # (profiling runs use a random table instead: same kernels, same shapes)
    V = cfg.vocab
    g = np.empty(V, dtype=np.int32)
    if args.profile:
        g[:] = S.uniform_ids(V, 99, 0, V)
    chunk = 1024 * (Kq + 1)
    all_ids = torch.arange(V, dtype=torch.int32, device=dev)
    for s0 in (range(0, V, chunk) if not args.profile else ()):
        n = min(chunk, V - s0)
        Bn = (n + Kq) // (Kq + 1)
        ids = torch.zeros(Bn * (Kq + 1), dtype=torch.int32, device=dev)
        ids[:n] = all_ids[s0:s0 + n]
        ids = ids.view(Bn, Kq + 1)
        tg = ctx.step(ids[:, 0].contiguous(), ids[:, 1:].contiguous())
        g[s0:s0 + n] = tg.view(-1)[:n].cpu().numpy()
    assert ctx.sync_status() == BND.OK

    # the decode trajectory, planned on the host
    total = args.warmup + args.steps
    traj = Trajectory(g, rank, B=Bq, K=Kq)
    plan_ctx = np.empty((total, Bq), np.int32)
    plan_dr = np.empty((total, Bq, Kq), np.int32)
    plan_com = np.empty((total, Bq, Kq + 1), np.int32)
    plan_alen = np.empty((total, Bq), np.int32)
    counted = np.zeros(total, np.int64)
    for i in range(total):
        c, d = traj.drafts()
        com, n = traj.expected(c, d)
        plan_ctx[i], plan_dr[i], plan_com[i], plan_alen[i] = c, d, com, n
        counted[i] = traj.advance(com, n)
    setup_s = time.perf_counter() - t_setup

    d_ctx = torch.from_numpy(plan_ctx).to(dev)
    d_dr = torch.from_numpy(plan_dr).to(dev)
    d_tg = torch.empty((total, Bq, Kq + 1), dtype=torch.int32, device=dev)
    d_com = torch.empty_like(d_tg)
    d_alen = torch.empty((total, Bq), dtype=torch.int32, device=dev)

    # one CUDA graph per step: step + accept on fixed buffers, inputs copied in
    in_ctx = torch.empty((Bq,), dtype=torch.int32, device=dev)
    in_dr = torch.empty((Bq, Kq), dtype=torch.int32, device=dev)
    out_tg = torch.empty((Bq, Kq + 1), dtype=torch.int32, device=dev)
    out_com = torch.empty_like(out_tg)
    out_alen = torch.empty((Bq,), dtype=torch.int32, device=dev)
    in_ctx.copy_(d_ctx[0])
    in_dr.copy_(d_dr[0])
    cs = torch.cuda.Stream(device=dev)
    cs.wait_stream(stream)
    graph = None
    if not args.no_graph:
        with torch.cuda.stream(cs):
            ctx.step(in_ctx, in_dr, target_ids=out_tg, stream=cs)
            ctx.accept(in_dr, out_tg, committed=out_com, accept_len=out_alen, stream=cs)
        cs.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            ctx.step(in_ctx, in_dr, target_ids=out_tg, stream=cs)
            ctx.accept(in_dr, out_tg, committed=out_com, accept_len=out_alen, stream=cs)
    stream.wait_stream(cs)

    def run_step(i):
        if graph is not None:
            in_ctx.copy_(d_ctx[i], non_blocking=True)
            in_dr.copy_(d_dr[i], non_blocking=True)
            graph.replay()
            d_com[i].copy_(out_com, non_blocking=True)
            d_alen[i].copy_(out_alen, non_blocking=True)
        else:
            ctx.step(d_ctx[i], d_dr[i], target_ids=d_tg[i])
            ctx.accept(d_dr[i], d_tg[i], committed=d_com[i], accept_len=d_alen[i])

    for i in range(args.warmup):
        run_step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    ev0.record(stream)
    for i in range(args.warmup, total):
        run_step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    if dist:
        dist.barrier()
    time.sleep(0.2)
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.summary(w0, w1)

    if args.profile and args.draft_head:
        line = run_decode_iteration(args, ctx, cfg, w_host, dev, Bq, Kq, stream)
        line["clocks"] = clk
        if rank == 0:
            print(json.dumps(line), flush=True)
        ctx.close()
        return

    if args.profile:
        if rank == 0:
            print(json.dumps({"profile": True, "layers": cfg.n_layers, "batch": Bq, "drafts": Kq,
                              "steps": args.steps, "ms_per_step": round(ms / args.steps, 4),
                              "clocks": clk}), flush=True)
        ctx.close()
        return

    # every timed step committed exactly what the planned trajectory says
    got_com = d_com[args.warmup:].cpu().numpy()
    got_alen = d_alen[args.warmup:].cpu().numpy()
    mism = int(np.sum(np.any(got_com != plan_com[args.warmup:], axis=2)) +
               np.sum(got_alen != plan_alen[args.warmup:]))
    status = ctx.sync_status()
    tokens = float(counted[args.warmup:].sum())

    # end to end: the same steps through the host-buffer entry point
    h_ctx = torch.empty((Bq,), dtype=torch.int32, pin_memory=True).numpy()
    h_dr = torch.empty((Bq, Kq), dtype=torch.int32, pin_memory=True).numpy()
    h_com = torch.empty((Bq, Kq + 1), dtype=torch.int32, pin_memory=True).numpy()
    h_alen = torch.empty((Bq,), dtype=torch.int32, pin_memory=True).numpy()
    etraj = Trajectory(g, rank, B=Bq, K=Kq)
    cur = torch.cuda.current_stream()
    pre = [etraj.drafts()]
    for i in range(args.warmup):
        c, d = pre[-1]
        h_ctx[:], h_dr[:] = c, d
        ctx.decode_host(h_ctx, h_dr, h_com, h_alen, stream=cur)
        etraj.advance(h_com, h_alen)
        pre.append(etraj.drafts())
    e_tokens = 0
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0 = time.perf_counter()
    c, d = pre[-1]
    for i in range(args.steps):
        h_ctx[:], h_dr[:] = c, d
        ctx.decode_host(h_ctx, h_dr, h_com, h_alen, stream=cur)
        e_tokens += etraj.advance(h_com, h_alen)
        c, d = etraj.drafts()
    e1 = time.perf_counter()
    e_s = e1 - e0

    # roofline of the dominant kernel (the expert FFN): CUDA events around
    # each of its launches over the same steps, probes give the touched experts
    peak_gbs, peak_tf, peak_kind = measured_peaks()
    ctx.set_timing(True)
    ctx.get_timing(reset=True)
    alg_bytes = 0.0
    probe, pt = BND.make_probe(cfg.n_layers, Bq * (Kq + 1), cfg, topk=True, hidden=False,
                               device=dev)
    for i in range(args.warmup, total):
        ctx.step(d_ctx[i], d_dr[i], target_ids=d_tg[i], probe=probe)
        ctx.accept(d_dr[i], d_tg[i], committed=d_com[i], accept_len=d_alen[i])
        idx = pt["topk_idx"].cpu().numpy()
        for l in range(cfg.n_layers):
            alg_bytes += algorithmic_ffn_bytes(idx[l], cfg)
    fam_ms, fam_n = ctx.get_timing(reset=True)
    ctx.set_timing(False)
    ffn_launch_ms = fam_ms[0] / max(1, fam_n[0])
    ffn_bytes = alg_bytes / max(1, fam_n[0])
    achieved = ffn_bytes / (ffn_launch_ms * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "ffn_traffic.json")
    if os.path.exists(prof):
        with open(prof) as f:
            traffic = json.load(f).get("bytes_per_launch")

    if dist:
        ms, e_s, tokens, e_tokens = whole_job(ms, e_s, tokens, e_tokens, dev)
    value = tokens / (ms / 1e3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) bf16 weights, uniform start ids, drafts right w.p. 0.75)",
        "config": {"workload": WORKLOAD, "layers": cfg.n_layers, "hidden": cfg.hidden,
                   "experts": f"{cfg.n_experts}x{cfg.expert_inter} top-{cfg.top_k} + "
                              f"{cfg.n_shared} shared", "vocab": cfg.vocab, "batch": Bq,
                   "drafts": Kq, "p_match": P_MATCH, "page_tokens": PAGE_TOKENS,
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (5.8 GB of weights per step)",
                   "cuda_graph": graph is not None},
        "e2e": {"value": round(e_tokens / e_s, 1), "unit": UNIT,
                "h2d_bytes_per_step": Bq * 4 + Bq * Kq * 4,
                "d2h_bytes_per_step": Bq * (Kq + 1) * 4 + Bq * 4},
        "gpu_launches": int(args.steps * (2 * cfg.n_layers + 3)),
        "roofline": {"kernel": "expert FFN (gate/up + SwiGLU + down + combine)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak_gbs, "unit": "GB/s",
                     "frac": round(achieved / peak_gbs, 4), "peak_source": peak_kind,
                     "traffic": traffic, "launch_ms": round(ffn_launch_ms, 5),
                     "alg_bytes_per_launch": round(ffn_bytes)},
        "clocks": clk,
        "committed_per_step": round(tokens / args.steps / world, 3),
        "check": {"mismatched_rows": mism, "status": status},
        "kernel_ms_per_step": {"expert_ffn": round(fam_ms[0] / args.steps, 4),
                               "lm_head": round(fam_ms[2] / args.steps, 4),
                               "routing_and_norm": round(fam_ms[3] / args.steps, 4),
                               "note": "serialised by the per-launch events"},
        "setup_s": round(setup_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, w_host, plan_ctx, plan_dr, counted, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if dist:
        dist.destroy_process_group()


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


def cpu_baseline(cfg, w_host, plan_ctx, plan_dr, counted, budget_s=20.0):
    """The oracle, as it stands, on a bounded sample of the workload's verify
    tokens (one token per thread at a time), scaled to committed tokens/s."""
    import oracle as O
    orc = O.Oracle(cfg, w_host)
    toks = np.concatenate([plan_ctx[..., None], plan_dr], axis=2).reshape(-1)
    cores = _cores()
    import concurrent.futures as fut
    done = 0
    t0 = time.perf_counter()
    with fut.ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < budget_s and done < len(toks):
            batch = toks[done:done + cores]
            list(ex.map(orc.target, batch))
            done += len(batch)
    dt = time.perf_counter() - t0
    per_verify_token = float(counted.sum()) / (len(counted) * B_SEQ * (K_DRAFT + 1))
    value = done / dt * per_verify_token
    return {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done} verify tokens of the workload's first steps in {dt:.1f} s "
                      f"(fp64, one token per thread), scaled by {per_verify_token:.3f} committed "
                      f"tokens per verify token"}


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
    ap.add_argument("--draft-head", action="store_true",
                    help="profiling only: time whole decode iterations with the FastMTP draft head")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if (args.layers or args.batch or args.drafts is not None or args.draft_head) and not args.profile:
        ap.error("--layers, --batch, --drafts and --draft-head are for profiling runs only (--profile)")
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
