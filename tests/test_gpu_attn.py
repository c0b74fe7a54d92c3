"""GPU parity of the stack with attention against the fp64 oracle.

The pages name the decoder but not its attention; the library reads it as
pre-norm multi-head attention with rotary positions and a bf16 key/value cache
before each MoE block (the oracle's attention sub-block states the reading).
The verify step then depends on each sequence's prefix: these tests feed
prompts through the verify call (drafts = the prompt's next tokens), decode
with speculation, and check every target against the oracle, teacher-forced
on the GPU's own residual stream and cache, and free-running over whole
sequences.
"""
import concurrent.futures as fut

import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S
import parity
from parity import FREE_LOGIT_BAND, FREE_ROUTE_BAND, REL, TIE, check_attn_tokens, threads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SEED_PROMPTS = 7


def _B():
    from moe_speculative_decoding_router_gb300 import binding
    return binding


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _prompts(n_seq, n, V, first=0):
    ids = S.uniform_ids(n_seq * n, SEED_PROMPTS, 0, V, first)
    return np.asarray(ids, dtype=np.int64).reshape(n_seq, n)


def _feed(ctx, seqs, K, start=0, probe_last=False):
    """Feeds seqs [B, n] (n - start a multiple of K + 1) through verify calls
    of K + 1 tokens per sequence at positions start, start + K + 1, ...;
    returns the targets [B, n - start] (target j: the greedy next id after
    the sequence's tokens 0 .. start + j) and, with probe_last, the last
    call's (ids, positions, targets, probe tensors)."""
    B_ = _B()
    Bn, n = seqs.shape
    K1 = K + 1
    assert (n - start) % K1 == 0
    out = []
    last = None
    for p0 in range(start, n, K1):
        ctxids = _i32(seqs[:, p0])
        drafts = _i32(seqs[:, p0 + 1: p0 + K1]) if K > 0 else None
        pos = _i32(np.full(Bn, p0))
        probe = pt = None
        if probe_last and p0 + K1 == n:
            probe, pt = B_.make_probe(ctx.cfg.n_layers, Bn * K1, ctx.cfg)
        out.append(ctx.step_attn(ctxids, drafts, pos, probe=probe))
        if probe is not None:
            last = (seqs[:, p0: p0 + K1].reshape(-1), np.repeat(np.full(Bn, p0), K1) +
                    np.tile(np.arange(K1), Bn), out[-1], pt)
    tg = torch.cat(out, dim=1).cpu().numpy()
    assert ctx.sync_status() == 0
    return tg, last


def _cache_np(ctx):
    k, v = ctx.kv_cache()
    torch.cuda.synchronize()
    return (k.view(torch.int16).cpu().numpy().view(np.uint16),
            v.view(torch.int16).cpu().numpy().view(np.uint16))


def _oracle_seqs(orc, seqs, caches=False):
    with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
        return list(ex.map(lambda s: orc.forward_seq(s, caches=caches), list(seqs)))


def _compare_free(gpu_targets, refs, first, label):
    """GPU targets [B, n - first] against the oracle's free-running targets of
    positions first .. n-1.  A difference must sit where the oracle's top-2
    logit gap is below FREE_LOGIT_BAND, or where one of the sequence's block
    selections up to that position has a gap below FREE_ROUTE_BAND (a routing
    decision that the fp32 and fp64 paths may take apart, and which then
    reaches every later position through the cache)."""
    diffs, ties, routed = 0, 0, 0
    for b, r in enumerate(refs):
        ref = r["targets"][first:]
        got = gpu_targets[b]
        route_min = np.minimum.accumulate(np.min(r["route_gaps"], axis=1))[first:]
        for j in np.nonzero(got != ref)[0]:
            diffs += 1
            lg = r["logit_gaps"][first + j]
            if lg < TIE:
                ties += 1
            elif route_min[j] < FREE_ROUTE_BAND:
                routed += 1
            else:
                assert lg < FREE_LOGIT_BAND, (
                    f"{label}: sequence {b} position {first + j}: gpu {got[j]} oracle {ref[j]}, "
                    f"logit gap {lg:.3g}, smallest selection gap so far {route_min[j]:.3g}")
    parity.record(label, tokens=int(gpu_targets.size), free_running_diffs=diffs,
                  near_ties=ties, after_close_routing=routed)
    return diffs


# ------------------------------------------------------------------ fixtures

@pytest.fixture(scope="module")
def tiny_attn():
    B = _B()
    cfg = S.TINY_ATTN
    w = S.make_weights(cfg)
    ctx = B.MoeVerify(cfg, B.weights_to_device(w), max_batch=8, max_k=15, max_pos=20480)
    yield ctx, O.Oracle(cfg, w)
    ctx.close()


@pytest.fixture(scope="module")
def full_attn():
    B = _B()
    cfg = S.FULL_ATTN
    w = S.make_weights(cfg)
    ctx = B.MoeVerify(cfg, B.weights_to_device(w), max_batch=8, max_k=3, max_pos=256)
    torch.cuda.empty_cache()
    yield ctx, O.Oracle(cfg, w)
    ctx.close()


# ----------------------------------------------------------------- tiny stack

@pytest.mark.parametrize("Bn,K", [(1, 0), (5, 3), (3, 15), (8, 1)])
def test_tiny_attn_prompts_match_oracle(tiny_attn, Bn, K):
    """Prompts of 48 tokens through verify calls of K + 1 tokens: every
    target equals the oracle's greedy next id after the prefix (outside the
    bands), and the cached keys and values are the oracle's free-running ones
    within the trajectory tolerance (parity.kv_within with REL)."""
    ctx, orc = tiny_attn
    n = 48
    seqs = _prompts(Bn, n, orc.cfg.vocab, first=100 * K)
    tg, _ = _feed(ctx, seqs, K)
    refs = _oracle_seqs(orc, seqs, caches=True)
    _compare_free(tg, refs, 0, f"attn tiny prompts B={Bn} K={K}")
    kc, vc = _cache_np(ctx)
    L, d = orc.cfg.n_layers, orc.cfg.hidden
    differing, worst = 0, 0.0
    for b, r in enumerate(refs):
        for name, gpu, ref in (("key", kc, r["kcache"]), ("value", vc, r["vcache"])):
            g = parity._bf16_to_f64(gpu[:, b, :, :n, :]).transpose(0, 2, 1, 3).reshape(L, n, d)
            bad = parity.kv_within(g, ref, REL)
            assert bad[0].size == 0, (f"{name} cache, sequence {b}, layer {bad[0][0]} position "
                                      f"{bad[1][0]}")
            differing += int(np.count_nonzero(g != ref))
            worst = max(worst, float(np.max(parity.rel_err(g, ref))))
    parity.record(f"attn tiny cache B={Bn} K={K}", values=int(2 * Bn * L * n * d),
                  differing=differing, max_row_rel=round(worst, 6))


def test_tiny_attn_teacher_forced(tiny_attn):
    """After 32-token prompts, one verify call at a different position per
    sequence (earlier positions overwritten by new tokens): every token
    checked teacher-forced on the GPU's residual stream and cache."""
    ctx, orc = tiny_attn
    Bn, K = 6, 3
    seqs = _prompts(Bn, 32, orc.cfg.vocab, first=5000)
    _feed(ctx, seqs, K)
    pos0 = np.array([31, 20, 0, 7, 28, 13])
    new = _prompts(Bn, K + 1, orc.cfg.vocab, first=7000)
    B_ = _B()
    probe, pt = B_.make_probe(orc.cfg.n_layers, Bn * (K + 1), orc.cfg)
    tg = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(pos0), probe=probe)
    assert ctx.sync_status() == 0
    kc, vc = _cache_np(ctx)
    ids = new.reshape(-1)
    seq = np.repeat(np.arange(Bn), K + 1)
    pos = np.repeat(pos0, K + 1) + np.tile(np.arange(K + 1), Bn)
    check_attn_tokens(orc, ids, seq, pos, tg.cpu().numpy().reshape(-1),
                      pt["topk_idx"].cpu().numpy(), pt["topk_w"].cpu().numpy(),
                      pt["hidden"].cpu().numpy(), kc, vc, label="attn tiny teacher-forced")


def test_tiny_attn_long_context(tiny_attn):
    """Eight sequences of ~20,000 positions: the split width reaches its
    1,024-key limit and each sequence's keys span ~20 splits merged by the
    last to finish.  The first 3,008 positions of sequence 0 are checked
    free-running against the oracle, and a final call at a different
    position per sequence is checked teacher-forced on every token."""
    ctx, orc = tiny_attn
    Bn, K, n = 8, 15, 20464
    seqs = _prompts(Bn, n, orc.cfg.vocab, first=10 ** 6)
    tg, _ = _feed(ctx, seqs, K)
    m = 3008
    ref = orc.forward_seq(seqs[0, :m])
    _compare_free(tg[:1, :m], [ref], 0, "attn tiny long context, sequence 0 free-running")
    pos0 = n - np.array([0, 5, 17, 300, 1000, 2003, 64, 1]) - (K + 1)
    new = _prompts(Bn, K + 1, orc.cfg.vocab, first=9 * 10 ** 6)
    B_ = _B()
    probe, pt = B_.make_probe(orc.cfg.n_layers, Bn * (K + 1), orc.cfg)
    tgl = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(pos0), probe=probe)
    assert ctx.sync_status() == 0
    kc, vc = _cache_np(ctx)
    ids = new.reshape(-1)
    seq = np.repeat(np.arange(Bn), K + 1)
    pos = np.repeat(pos0, K + 1) + np.tile(np.arange(K + 1), Bn)
    check_attn_tokens(orc, ids, seq, pos, tgl.cpu().numpy().reshape(-1),
                      pt["topk_idx"].cpu().numpy(), pt["topk_w"].cpu().numpy(),
                      pt["hidden"].cpu().numpy(), kc, vc,
                      label="attn tiny long context teacher-forced")


def test_tiny_attn_speculative_decoding_is_lossless(tiny_attn):
    """Prompts, then ten verify + accept iterations with drafts from the
    oracle's greedy continuation, each replaced by a random id with
    probability 1 - p: the committed tokens are the oracle's greedy
    continuation (outside near ties), whatever the drafts."""
    ctx, orc = tiny_attn
    Bn, K, n0, iters, p = 6, 3, 8, 10, 0.6
    V = orc.cfg.vocab
    prompts = _prompts(Bn, n0, V, first=3 * 10 ** 6)
    tg, _ = _feed(ctx, prompts, K)
    # the oracle's greedy continuation, long enough for every commit
    horizon = n0 + 1 + iters * (K + 1) + K
    greedy = []
    for b in range(Bn):
        s = list(prompts[b])
        while len(s) < horizon:
            s.append(int(orc.forward_seq(s)["targets"][-1]))
        greedy.append(s)
    toks = [list(prompts[b]) + [int(tg[b, -1])] for b in range(Bn)]
    rng = np.random.default_rng(11)
    accepted = 0
    for it in range(iters):
        pos = np.array([len(t) - 1 for t in toks])
        ctxids = np.array([t[-1] for t in toks])
        drafts = np.zeros((Bn, K), dtype=np.int64)
        for b in range(Bn):
            for i in range(K):
                g = greedy[b][len(toks[b]) + i]
                drafts[b, i] = g if rng.random() < p else int(rng.integers(0, V))
        tgt = ctx.step_attn(_i32(ctxids), _i32(drafts), _i32(pos))
        com, alen = ctx.accept(_i32(drafts), tgt)
        com, alen = com.cpu().numpy(), alen.cpu().numpy()
        for b in range(Bn):
            nacc = int(alen[b])
            accepted += nacc
            toks[b].extend(int(x) for x in com[b, : nacc + 1])
    assert ctx.sync_status() == 0
    # every committed token is the oracle's greedy next id after the
    # committed prefix before it (a near tie may go either way)
    ties = 0
    for b in range(Bn):
        got = toks[b]
        ref = orc.forward_seq(got)
        for i in range(n0 - 1, len(got) - 1):
            if got[i + 1] != ref["targets"][i]:
                assert ref["logit_gaps"][i] < TIE, f"sequence {b} position {i + 1}"
                ties += 1
    parity.record("attn tiny speculative decoding", iterations=iters, accepted=accepted,
                  near_ties=ties)


def test_tiny_attn_out_of_range_positions(tiny_attn):
    """A sequence whose positions leave [0, max_pos) gets targets -1, writes
    nothing to the cache and raises the id-range status; the others are as
    in a call without it."""
    ctx, orc = tiny_attn
    K = 3
    seqs = _prompts(4, 8, orc.cfg.vocab, first=4 * 10 ** 6)
    _feed(ctx, seqs, K)
    new = _prompts(4, K + 1, orc.cfg.vocab, first=5 * 10 ** 6)
    good = np.array([4, 4, 4, 4])
    ref = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(good)).cpu().numpy()
    assert ctx.sync_status() == 0
    kc0, vc0 = _cache_np(ctx)
    bad = np.array([4, -1, 4, ctx.max_pos - K])
    got = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(bad)).cpu().numpy()
    assert ctx.sync_status() == _B().ERR_ID_RANGE
    assert np.all(got[1] == -1) and np.all(got[3] == -1)
    assert np.array_equal(got[[0, 2]], ref[[0, 2]])
    kc1, vc1 = _cache_np(ctx)
    assert np.array_equal(kc0, kc1) and np.array_equal(vc0, vc1)


def test_attn_host_argument_errors(tiny_attn):
    """The calls of the attention-free stack refuse a context with attention,
    and the attention call checks its arguments on the host."""
    ctx, orc = tiny_attn
    B_ = _B()
    ids = _i32(np.zeros(2))
    dr = _i32(np.zeros((2, 3)))
    with pytest.raises(B_.MoeVerifyError) as e:
        ctx.step(ids, dr)
    assert e.value.code == B_.ERR_ARG
    lib = B_.load()
    tg = _i32(np.zeros((2, 4)))
    s = torch.cuda.current_stream().cuda_stream
    assert lib.moe_verify_step_attn(ctx.handle, ids.data_ptr(), dr.data_ptr(), None, 2, 3,
                                    tg.data_ptr(), None, s) == B_.ERR_ARG
    assert lib.moe_verify_step_attn(ctx.handle, ids.data_ptr(), dr.data_ptr(), ids.data_ptr(), 9,
                                    3, tg.data_ptr(), None, s) == B_.ERR_ARG
    assert lib.moe_verify_step_attn(ctx.handle, ids.data_ptr(), dr.data_ptr(), ids.data_ptr(), 2,
                                    16, tg.data_ptr(), None, s) == B_.ERR_ARG


# ----------------------------------------------------------------- full size

def test_full_attn_prompts_teacher_forced_and_free_running(full_attn):
    """Full size (12 layers, hidden 1280, 10 heads of 128, vocabulary
    129,280): 8 prompts of 32 tokens in verify calls of 4; the last call is
    checked teacher-forced on every token, and every target of every call
    against the oracle's free-running sequence within the bands."""
    ctx, orc = full_attn
    Bn, K, n = 8, 3, 32
    seqs = _prompts(Bn, n, orc.cfg.vocab, first=6 * 10 ** 6)
    tg, last = _feed(ctx, seqs, K, probe_last=True)
    ids, pos, tgl, pt = last
    kc, vc = _cache_np(ctx)
    check_attn_tokens(orc, ids, np.repeat(np.arange(Bn), K + 1), pos, tgl.cpu().numpy().reshape(-1),
                      pt["topk_idx"].cpu().numpy(), pt["topk_w"].cpu().numpy(),
                      pt["hidden"].cpu().numpy(), kc, vc, label="attn full teacher-forced")
    refs = _oracle_seqs(orc, seqs)
    _compare_free(tg, refs, 0, "attn full prompts B=8 K=3 n=32 free-running")


def test_full_attn_decode_loop(full_attn):
    """Full size: prompts of 16, then four verify + accept iterations with
    drafts from the GPU's own previous targets (right where the chain holds)
    mixed with random ids; every call's tokens teacher-forced (sampled), the
    commits exactly the acceptance rule on the targets."""
    ctx, orc = full_attn
    B_ = _B()
    Bn, K, n0 = 8, 3, 16
    V = orc.cfg.vocab
    prompts = _prompts(Bn, n0, V, first=7 * 10 ** 6)
    tg, _ = _feed(ctx, prompts, K)
    toks = [list(prompts[b]) + [int(tg[b, -1])] for b in range(Bn)]
    rng = np.random.default_rng(12)
    prev = None
    for it in range(4):
        pos = np.array([len(t) - 1 for t in toks])
        ctxids = np.array([t[-1] for t in toks])
        drafts = rng.integers(0, V, size=(Bn, K))
        if prev is not None:
            keep = rng.random((Bn, K)) < 0.5
            drafts = np.where(keep, prev, drafts)
        probe, pt = B_.make_probe(orc.cfg.n_layers, Bn * (K + 1), orc.cfg)
        tgt = ctx.step_attn(_i32(ctxids), _i32(drafts), _i32(pos), probe=probe)
        com, alen = ctx.accept(_i32(drafts), tgt)
        tgn, com, alen = tgt.cpu().numpy(), com.cpu().numpy(), alen.cpu().numpy()
        wc, wl, _ = O.accept(drafts, tgn, V)
        assert np.array_equal(com, wc) and np.array_equal(alen, wl)
        kc, vc = _cache_np(ctx)
        ids = np.concatenate([ctxids.reshape(-1, 1), drafts], axis=1).reshape(-1)
        allpos = np.repeat(pos, K + 1) + np.tile(np.arange(K + 1), Bn)
        sample = list(range(0, Bn * (K + 1), 3))
        check_attn_tokens(orc, ids, np.repeat(np.arange(Bn), K + 1), allpos, tgn.reshape(-1),
                          pt["topk_idx"].cpu().numpy(), pt["topk_w"].cpu().numpy(),
                          pt["hidden"].cpu().numpy(), kc, vc, sample=sample,
                          label=f"attn full decode step {it}")
        for b in range(Bn):
            nacc = int(alen[b])
            toks[b].extend(int(x) for x in com[b, : nacc + 1])
        prev = tgn[:, 1:]
    assert ctx.sync_status() == 0


def test_full_attn_same_bits_on_any_grid(full_attn):
    """The step with attention gives the same bits with one CTA, with more
    CTAs than fit on the GPU at once, and with the default grid."""
    ctx, orc = full_attn
    B_ = _B()
    Bn, K = 8, 3
    seqs = _prompts(Bn, 20, orc.cfg.vocab, first=8 * 10 ** 6)
    _feed(ctx, seqs[:, :16], K)
    new = seqs[:, 16:20]
    pos = np.full(Bn, 16)
    outs = []
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for g in (0, 1, 2 * sms + 3):
        ctx.set_grid(g)
        probe, pt = B_.make_probe(orc.cfg.n_layers, Bn * (K + 1), orc.cfg)
        tg = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(pos), probe=probe)
        torch.cuda.synchronize()
        outs.append((tg.cpu().numpy(), pt["hidden"].cpu().numpy()))
    ctx.set_grid(0)
    assert ctx.sync_status() == 0
    for tg, hid in outs[1:]:
        assert np.array_equal(tg, outs[0][0])
        assert np.array_equal(hid, outs[0][1])


def test_full_attn_graph_capture(full_attn):
    """The step with attention captured in a CUDA graph and replayed gives
    the targets of the direct call."""
    ctx, orc = full_attn
    Bn, K = 8, 3
    seqs = _prompts(Bn, 24, orc.cfg.vocab, first=9 * 10 ** 6)
    _feed(ctx, seqs[:, :20], K)
    c = _i32(seqs[:, 20])
    dr = _i32(seqs[:, 21:24])
    pos = _i32(np.full(Bn, 20))
    direct = ctx.step_attn(c, dr, pos).clone()
    out = torch.empty_like(direct)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ctx.step_attn(c, dr, pos, target_ids=out, stream=s)
    for _ in range(2):
        out.fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, direct)
    assert ctx.sync_status() == 0


# ------------------------------------------------------------- other shapes

@pytest.mark.parametrize("n_heads", [1, 2])
def test_tiny_attn_other_head_widths(n_heads):
    """Head widths 64 (one 128-byte swizzled box per key row) and 32 (the
    64-byte swizzle): prompts of 48 in calls of 4, every target and the cache
    against the oracle."""
    import dataclasses
    B_ = _B()
    cfg = dataclasses.replace(S.TINY_ATTN, n_heads=n_heads, name=f"tiny_attn_h{n_heads}")
    w = S.make_weights(cfg)
    ctx = B_.MoeVerify(cfg, B_.weights_to_device(w), max_batch=3, max_k=3, max_pos=64)
    try:
        orc = O.Oracle(cfg, w)
        n = 48
        seqs = _prompts(3, n, cfg.vocab, first=11000 + n_heads)
        tg, _ = _feed(ctx, seqs, 3)
        refs = _oracle_seqs(orc, seqs, caches=True)
        _compare_free(tg, refs, 0, f"attn tiny hd={cfg.hidden // n_heads} prompts")
        kc, vc = _cache_np(ctx)
        L, d = cfg.n_layers, cfg.hidden
        for b, r in enumerate(refs):
            for name, gpu, ref in (("key", kc, r["kcache"]), ("value", vc, r["vcache"])):
                g = parity._bf16_to_f64(gpu[:, b, :, :n, :]).transpose(0, 2, 1, 3).reshape(L, n, d)
                bad = parity.kv_within(g, ref, REL)
                assert bad[0].size == 0, f"{name} cache, sequence {b}"
    finally:
        ctx.close()


@pytest.fixture(scope="module")
def full_attn_long():
    B_ = _B()
    cfg = S.FULL_ATTN
    w = S.make_weights(cfg)
    ctx = B_.MoeVerify(cfg, B_.weights_to_device(w), max_batch=4, max_k=15, max_pos=2304)
    torch.cuda.empty_cache()
    yield ctx, O.Oracle(cfg, w)
    ctx.close()


def test_full_attn_long_context_teacher_forced(full_attn_long):
    """Full size at ~2,000 positions: four prompts of 2,048 tokens fed in calls
    of 16, then one call per sequence at a different position; with 4
    sequences the split width is 256 keys, so each sequence's keys span ~8
    splits merged by the last to finish.  Every token of the last call is
    checked teacher-forced (attention part, MoE part, routing, target) on the
    GPU's residual stream and cache."""
    ctx, orc = full_attn_long
    B_ = _B()
    Bn, K, n = 4, 15, 2048
    seqs = _prompts(Bn, n, orc.cfg.vocab, first=12 * 10 ** 6)
    _feed(ctx, seqs, K)
    pos0 = np.array([n - 16, n - 16 - 333, n - 16 - 1000, 700])
    new = _prompts(Bn, K + 1, orc.cfg.vocab, first=13 * 10 ** 6)
    probe, pt = B_.make_probe(orc.cfg.n_layers, Bn * (K + 1), orc.cfg)
    tg = ctx.step_attn(_i32(new[:, 0]), _i32(new[:, 1:]), _i32(pos0), probe=probe)
    assert ctx.sync_status() == 0
    kc, vc = _cache_np(ctx)
    ids = new.reshape(-1)
    seq = np.repeat(np.arange(Bn), K + 1)
    pos = np.repeat(pos0, K + 1) + np.tile(np.arange(K + 1), Bn)
    sample = sorted(set(range(0, Bn * (K + 1), 5)) | {K, 2 * K + 1, Bn * (K + 1) - 1})
    check_attn_tokens(orc, ids, seq, pos, tg.cpu().numpy().reshape(-1),
                      pt["topk_idx"].cpu().numpy(), pt["topk_w"].cpu().numpy(),
                      pt["hidden"].cpu().numpy(), kc, vc, sample=sample,
                      label="attn full long context (~2,000 positions) teacher-forced")
