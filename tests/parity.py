"""Comparison of the CUDA path with the oracle, shared by the GPU tests.

Exact quantities (routing sets, argmax ids, accept lengths, committed
tokens) are compared exactly, except where the oracle's own top-k selection
gap (logit units) or top-2 logit gap is below 1e-3; those near ties are
counted and reported.

Each decoder block and the final argmax are checked teacher-forced: the
oracle evaluates block l on the GPU's own residual stream entering block l
(read from the hidden-state probe, fp32 values taken exactly in fp64).  The
whole trajectory is held to the hidden-state tolerance: max relative error
2e-2 per token and block, taken as max|gpu - ref| / max|ref| against the
oracle run along the GPU's routing.

Every checked token is also run through the oracle free-running (its own
routing from the token id on).  Over 12 blocks the fp32 path drifts from
fp64: the bf16 rounding of the normalised input and of the SwiGLU product
turns last-bit differences into whole-ulp steps that compound, so free-running
routing and targets can differ from the GPU's where the oracle's own gap is
small.  Such differences are bounded, not just counted:
  - the first block where the free-running routing set differs from the GPU's
    must have an oracle selection gap below FREE_ROUTE_BAND (logit units);
  - a target that differs while every block's routing agrees must have an
    oracle top-2 logit gap below FREE_LOGIT_BAND.
A difference at a larger gap fails.  The bands come from the drift measured
on the GPU at full size: along the same routing the lm_head logits of the GPU
and of the oracle differ by at most 0.033 (max relative error 1.1e-2; the
full-size logits test re-measures it on every run and checks it against the
band), and a flip needs an oracle top-2 gap below the sum of the two
candidates' errors, so at most 0.067; the band is that, rounded up.  Router
logits have the same scale (a bf16-normalised row times N(0, 0.02) weights
over d = 1280, standard deviation ~0.72) and drift alike, so the routing band
is the same.

Every call's counts are kept in RECORD; the conftest prints them at the end
of the run (and writes them as JSON where PARITY_RECORD names a file).
"""
import concurrent.futures as fut
import os

import numpy as np

TIE = 1e-3
REL = 2e-2
# one block, teacher-forced: only last-bit differences of the inputs' bf16
# rounding separate the two sides
BLOCK_REL = 2e-3
# free-running differences must sit below these gaps (logit units)
FREE_ROUTE_BAND = 8e-2
FREE_LOGIT_BAND = 8e-2

RECORD = []


def threads():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref), axis=-1)
    return np.max(np.abs(got - ref), axis=-1) / np.maximum(den, 1e-30)


def _same_sets(a, b):
    return set(np.asarray(a).tolist()) == set(np.asarray(b).tolist())


def check_tokens(orc, ids, gpu_targets, probe_idx=None, probe_w=None, probe_hidden=None,
                 sample=None, nthreads=None, label=None):
    """Check verify tokens ids[t] with GPU targets gpu_targets[t].

    With probes (topk_idx [L,T,k], topk_w [L,T,k], hidden [L+1,T,d]) every
    block and the final argmax are checked teacher-forced, the whole
    trajectory against the oracle run along the GPU's routing, and the
    free-running oracle's routing and target against the GPU's within the
    bands.  Without probes the targets are compared with the free-running
    oracle (exact outside the tie band).  Returns the counts, which are also
    appended to RECORD under `label`."""
    T = len(ids)
    sample = list(range(T) if sample is None else sample)
    nthreads = nthreads or threads()

    def one(t):
        out = {"route_ties": 0, "logit_tie": 0, "free_diff": 0, "free_gap": None,
               "free_route_layers": 0, "free_route_gap": None, "free_diff_route_agrees": None,
               "max_rel": 0.0, "max_block_rel": 0.0, "max_free_rel": 0.0, "fail": None}
        x = int(ids[t])
        if probe_hidden is None:
            r = orc.forward_token(x)
            if int(gpu_targets[t]) != r["target"]:
                if r["logit_gap"] < TIE:
                    out["logit_tie"] = 1
                else:
                    out["fail"] = (f"token {t} (id {x}): gpu target {int(gpu_targets[t])} "
                                   f"oracle {r['target']} logit gap {r['logit_gap']:.3g}")
            return out
        H = np.asarray(probe_hidden[:, t, :], dtype=np.float64)
        L = H.shape[0] - 1
        emb = orc.w["embed"][x] if orc.w.get("embed") is not None else None
        if emb is not None:
            e0 = (emb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            if not np.array_equal(H[0], e0):
                out["fail"] = f"token {t}: residual stream entering block 0 is not E[{x}]"
                return out
        for l in range(L):
            gsel = np.ascontiguousarray(probe_idx[l, t, :])
            h_new, sel, wts, gap, _ = orc.layer(l, H[l], force_sel=gsel)
            if not _same_sets(gsel, sel):
                if gap < TIE:
                    out["route_ties"] += 1
                else:
                    out["fail"] = (f"token {t} (id {x}) block {l}: gpu experts "
                                   f"{sorted(gsel.tolist())} oracle {sorted(sel.tolist())} "
                                   f"gap {gap:.3g}")
                    return out
            if probe_w is not None:
                err = np.max(np.abs(probe_w[l, t, :] - wts) / np.maximum(np.abs(wts), 1e-12))
                if err > BLOCK_REL:
                    out["fail"] = f"token {t} block {l}: routing weights rel err {err:.3g}"
                    return out
            e = float(rel_err(H[l + 1], h_new))
            out["max_block_rel"] = max(out["max_block_rel"], e)
            if e > BLOCK_REL:
                out["fail"] = f"token {t} block {l}: teacher-forced block output rel err {e:.3g}"
                return out
        tgt, lgap, _ = orc.head(H[L])
        if int(gpu_targets[t]) != tgt:
            if lgap < TIE:
                out["logit_tie"] = 1
            else:
                out["fail"] = (f"token {t} (id {x}): gpu target {int(gpu_targets[t])} oracle on "
                               f"the gpu's final residual {tgt}, logit gap {lgap:.3g}")
                return out
        # free-running: the oracle's own routing from the token id on
        free = orc.forward_token(x)
        gsel_all = np.ascontiguousarray(probe_idx[:, t, :])
        differ = [l for l in range(L) if not _same_sets(gsel_all[l], free["sel"][l])]
        out["free_route_layers"] = len(differ)
        if differ:
            l0 = differ[0]
            out["free_route_gap"] = float(free["route_gap"][l0])
            if out["free_route_gap"] >= FREE_ROUTE_BAND:
                out["fail"] = (f"token {t} (id {x}): free-running routing first differs at block "
                               f"{l0} with oracle selection gap {out['free_route_gap']:.3g} "
                               f">= {FREE_ROUTE_BAND}")
                return out
            # the whole trajectory along the GPU's routing
            forced = orc.forward_token(x, force_sel=gsel_all)
        else:
            forced = free
            out["max_free_rel"] = float(np.max(rel_err(H, free["hidden"])))
        e = rel_err(H, forced["hidden"])
        out["max_rel"] = float(np.max(e))
        if out["max_rel"] > REL:
            out["fail"] = f"token {t}: hidden rel err per block {np.round(e, 5).tolist()}"
            return out
        if free["target"] != int(gpu_targets[t]):
            out["free_diff"] = 1
            out["free_gap"] = free["logit_gap"]
            out["free_diff_route_agrees"] = not differ
            if not differ and free["logit_gap"] >= FREE_LOGIT_BAND:
                out["fail"] = (f"token {t} (id {x}): free-running target {free['target']} vs gpu "
                               f"{int(gpu_targets[t])} with identical routing, oracle logit gap "
                               f"{free['logit_gap']:.3g} >= {FREE_LOGIT_BAND}")
                return out
        return out

    with fut.ThreadPoolExecutor(max_workers=nthreads) as ex:
        res = list(ex.map(one, sample))
    fails = [r["fail"] for r in res if r["fail"]]
    assert not fails, "\n".join(fails[:10])
    stats = {"label": label, "tokens": len(res),
             "route_ties": sum(r["route_ties"] for r in res),
             "logit_ties": sum(r["logit_tie"] for r in res)}
    if probe_hidden is not None:
        stats.update({
            "free_running_target_diffs": sum(r["free_diff"] for r in res),
            "free_running_diff_logit_gaps": [round(r["free_gap"], 5) for r in res
                                             if r["free_diff"]],
            "free_running_diffs_with_same_routing": sum(1 for r in res if r["free_diff"]
                                                        and r["free_diff_route_agrees"]),
            "free_running_route_diff_tokens": sum(1 for r in res if r["free_route_layers"]),
            "free_running_first_route_gaps": [round(r["free_route_gap"], 5) for r in res
                                              if r["free_route_gap"] is not None],
            "max_hidden_rel": max([r["max_rel"] for r in res] + [0.0]),
            "max_free_hidden_rel": max([r["max_free_rel"] for r in res] + [0.0]),
            "max_block_rel": max([r["max_block_rel"] for r in res] + [0.0])})
    RECORD.append(stats)
    return stats


def record(label, **counts):
    """Adds counts of a test that does not go through check_tokens."""
    RECORD.append(dict(label=label, **counts))


# The stack with attention, one block teacher-forced: the attention sub-block
# adds bf16 roundings of its own (k, v and the attention output), each a
# last-bit difference at most between the two sides, so a block keeps the
# tolerance of BLOCK_REL.  A cached key or value is the bf16 rounding of a sum
# whose inputs (the bf16-normalised row) may already differ by a last bit
# between the sides, which moves the sum by up to a small fraction of the
# row's scale (not of the element's: an element near zero has a large
# relative error); the rounding then adds at most one bf16 step of the
# element (2^-7 of its magnitude).  So |gpu - oracle| <= KV_STEP |oracle| +
# rel * max|oracle row|, rel = BLOCK_REL teacher-forced.
KV_STEP = 2.0 ** -7
# The attention sub-block alone, teacher-forced, on the same grounds as a MoE
# block: its sides differ by last-bit flips of bf16 roundings (the normalised
# row, k, v, the attention output), so it keeps BLOCK_REL.  (Measured at full
# size: max 2.2e-4, median 7e-7; the MoE part on the GPU's post-attention
# residual: max 9.3e-4.)
ATTN_REL = BLOCK_REL


def kv_within(g, o, rel):
    """Cached key/value rows g (GPU) and o (oracle), [..., n] float64: the
    elements outside the bound above (an empty array when all are inside)."""
    scale = np.max(np.abs(o), axis=-1, keepdims=True)
    return np.nonzero(np.abs(g - o) > KV_STEP * np.abs(o) + rel * scale)


def _bf16_to_f64(a):
    a = np.asarray(a)
    if a.dtype == np.uint16 or a.dtype == np.int16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def check_attn_tokens(orc, ids, seq, pos, gpu_targets, probe_idx, probe_w, probe_hidden, kcache,
                      vcache, sample=None, nthreads=None, label=None):
    """Teacher-forced check of the stack with attention.

    ids[t], seq[t], pos[t]: token t's id, sequence slot and position;
    probe_* as for check_tokens, the hidden states [2L + 1, T, d] (entering
    each block's attention and its MoE part, and after the last block);
    kcache / vcache: the GPU's caches after the step as bf16 bit patterns [L,
    slots, heads, max_pos, hd].  For each block the oracle's attention
    sub-block runs on the GPU's residual and the GPU's cached keys and values
    of positions < pos (its own key and value of pos are compared with the
    GPU's) and its output is compared with the GPU's residual entering the MoE
    part, which the oracle's MoE block then runs on along the GPU's routing;
    the final argmax is checked on the GPU's final residual.  Returns the
    counts (also appended to RECORD)."""
    T = len(ids)
    sample = list(range(T) if sample is None else sample)
    nthreads = nthreads or threads()
    c = orc.cfg
    L, d = c.n_layers, c.hidden

    def cache_rows(arr, l, b, n):
        # [heads, n, hd] -> [n, d]
        x = _bf16_to_f64(arr[l, b, :, :n, :])
        return np.ascontiguousarray(x.transpose(1, 0, 2).reshape(n, d))

    def one(t):
        out = {"route_ties": 0, "logit_tie": 0, "kv_steps": 0, "kv_vals": 0,
               "max_block_rel": 0.0, "max_attn_rel": 0.0, "fail": None}
        x, b, p = int(ids[t]), int(seq[t]), int(pos[t])
        H = np.asarray(probe_hidden[:, t, :], dtype=np.float64)
        e0 = _bf16_to_f64(orc.w["embed"][x])
        if not np.array_equal(H[0], e0):
            out["fail"] = f"token {t}: residual stream entering block 0 is not E[{x}]"
            return out
        for l in range(L):
            kc = cache_rows(kcache, l, b, p + 1)
            vc = cache_rows(vcache, l, b, p + 1)
            gk, gv = kc[p].copy(), vc[p].copy()
            h_att, _ = orc.attn_block(l, H[2 * l], p, kc, vc)
            e = float(rel_err(H[2 * l + 1], h_att))
            out["max_attn_rel"] = max(out["max_attn_rel"], e)
            if e > ATTN_REL:
                out["fail"] = f"token {t} block {l}: teacher-forced attention output rel err {e:.3g}"
                return out
            for g, o in ((gk, kc[p]), (gv, vc[p])):
                out["kv_vals"] += d
                out["kv_steps"] += int(np.count_nonzero(g != o))
                bad = kv_within(g, o, BLOCK_REL)[0]
                if bad.size:
                    i = int(bad[0])
                    out["fail"] = (f"token {t} block {l}: cached key/value at position {p} dim {i}"
                                   f" gpu {g[i]:.6g} oracle {o[i]:.6g} (row scale "
                                   f"{np.max(np.abs(o)):.3g})")
                    return out
            gsel = np.ascontiguousarray(probe_idx[l, t, :])
            h_new, sel, wts, gap, _ = orc.layer(l, H[2 * l + 1], force_sel=gsel)
            if not _same_sets(gsel, sel):
                if gap < TIE:
                    out["route_ties"] += 1
                else:
                    out["fail"] = (f"token {t} (id {x}) block {l}: gpu experts "
                                   f"{sorted(gsel.tolist())} oracle {sorted(sel.tolist())} "
                                   f"gap {gap:.3g}")
                    return out
            err = np.max(np.abs(probe_w[l, t, :] - wts) / np.maximum(np.abs(wts), 1e-12))
            if err > BLOCK_REL:
                out["fail"] = f"token {t} block {l}: routing weights rel err {err:.3g}"
                return out
            e = float(rel_err(H[2 * l + 2], h_new))
            out["max_block_rel"] = max(out["max_block_rel"], e)
            if e > BLOCK_REL:
                out["fail"] = f"token {t} block {l}: teacher-forced block output rel err {e:.3g}"
                return out
        tgt, lgap, _ = orc.head(H[2 * L])
        if int(gpu_targets[t]) != tgt:
            if lgap < TIE:
                out["logit_tie"] = 1
            else:
                out["fail"] = (f"token {t} (id {x}): gpu target {int(gpu_targets[t])} oracle on "
                               f"the gpu's final residual {tgt}, logit gap {lgap:.3g}")
        return out

    with fut.ThreadPoolExecutor(max_workers=nthreads) as ex:
        res = list(ex.map(one, sample))
    fails = [r["fail"] for r in res if r["fail"]]
    assert not fails, "\n".join(fails[:10])
    stats = {"label": label, "tokens": len(res),
             "route_ties": sum(r["route_ties"] for r in res),
             "logit_ties": sum(r["logit_tie"] for r in res),
             "kv_values": sum(r["kv_vals"] for r in res),
             "kv_values_differing": sum(r["kv_steps"] for r in res),
             "max_block_rel": max([r["max_block_rel"] for r in res] + [0.0]),
             "max_attn_rel": max([r["max_attn_rel"] for r in res] + [0.0])}
    RECORD.append(stats)
    return stats
