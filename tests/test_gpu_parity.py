"""GPU parity: the CUDA path through the C ABI against the fp64 oracle."""
import os

import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S
import parity
from parity import REL, TIE, check_tokens, rel_err, threads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _B():
    from moe_speculative_decoding_router_gb300 import binding
    return binding


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


# ------------------------------------------------------------------ fixtures

@pytest.fixture(scope="module")
def tiny():
    B = _B()
    w = S.make_weights(S.TINY)
    ctx = B.MoeVerify(S.TINY, B.weights_to_device(w), max_batch=128, max_k=3)
    yield ctx, O.Oracle(S.TINY, w)
    ctx.close()


@pytest.fixture(scope="module")
def layer():
    B = _B()
    w = S.make_weights(S.LAYER)
    ctx = B.MoeVerify(S.LAYER, B.weights_to_device(w), max_batch=4096, max_k=0)
    yield ctx, O.Oracle(S.LAYER, w)
    ctx.close()


@pytest.fixture(scope="module")
def full():
    B = _B()
    w = S.make_weights(S.FULL)
    ctx = B.MoeVerify(S.FULL, B.weights_to_device(w), max_batch=32, max_k=3)
    torch.cuda.empty_cache()
    yield ctx, O.Oracle(S.FULL, w)
    ctx.close()


# ----------------------------------------------------------------- tiny stack

def test_tiny_every_id_matches_oracle(tiny):
    """All 512 ids as 128 sequences x (1 + 3 drafts): routing per layer,
    residual stream, targets."""
    ctx, orc = tiny
    B = _B()
    ids = np.arange(512, dtype=np.int32).reshape(128, 4)
    probe, pt = B.make_probe(S.TINY.n_layers, 512, S.TINY)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    got = tg.cpu().numpy().reshape(-1)
    stats = check_tokens(orc, ids.reshape(-1), got, pt["topk_idx"].cpu().numpy(),
                         pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(),
                         label="tiny, all 512 ids")
    g = np.loadtxt(os.path.join(GOLDEN, "tiny_g_table.txt"), dtype=np.int64)
    mism = np.nonzero(got != g[ids.reshape(-1)])[0]
    assert len(mism) <= stats["logit_ties"] + stats["route_ties"], mism
    print("tiny:", stats)


# T = 68 and 96 reach the tokens-on-M lm_head with ragged chunks (65..128 tokens)
# T = 260, 300, 400, 512: lm_head on CTA pairs (260 and 300: the last 256-token
# chunk holds 4 and 44 tokens, so the odd CTA of its pairs holds none)
@pytest.mark.parametrize("Bn,K", [(1, 0), (1, 3), (3, 1), (4, 3), (17, 3), (24, 3), (128, 0),
                                  (77, 2), (65, 3), (75, 3), (100, 3), (128, 3)])
def test_tiny_batch_shapes(tiny, Bn, K):
    ctx, orc = tiny
    ids = S.uniform_ids(Bn * (K + 1), 41 + Bn, K, 512).reshape(Bn, K + 1)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]) if K else None)
    got = tg.cpu().numpy().reshape(-1)
    check_tokens(orc, ids.reshape(-1), got, label=f"tiny B={Bn} K={K}")


# T = 4: vocabulary rows on M; T = 80: tokens on M; T = 280, 512: CTA pairs
@pytest.mark.parametrize("Bn", [1, 20, 70, 128])
def test_tiny_logits_probe(tiny, Bn):
    ctx, orc = tiny
    B = _B()
    if Bn == 1:
        ids = np.array([[5, 9, 300, 511]], dtype=np.int32)
    else:
        ids = S.uniform_ids(Bn * 4, 61, 3, 512).reshape(Bn, 4)
    T = ids.size
    probe, pt = B.make_probe(S.TINY.n_layers, T, S.TINY, logits=True)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    lg = pt["logits"].cpu().numpy()
    # the argmax is the probe's own logits' argmax (ties to the lowest id)
    assert np.array_equal(tg.cpu().numpy().reshape(-1), np.argmax(lg, axis=1))
    for t in range(T):
        r = orc.forward_token(int(ids.reshape(-1)[t]),
                              force_sel=pt["topk_idx"].cpu().numpy()[:, t, :], logits=True)
        assert rel_err(lg[t], r["logits"]) <= REL


@pytest.fixture(scope="module")
def tiny3():
    """The tiny stack with an odd layer count (expert counters alternate
    between two buffers by layer parity)."""
    import dataclasses
    B = _B()
    cfg = dataclasses.replace(S.TINY, n_layers=3)
    w = S.make_weights(cfg)
    ctx = B.MoeVerify(cfg, B.weights_to_device(w), max_batch=64, max_k=3)
    yield ctx, O.Oracle(cfg, w), cfg
    ctx.close()


def test_tiny_odd_layers_steps_and_layer_calls_interleaved(tiny3):
    """Steps and single-block calls in any order leave every counter clean:
    each call matches the oracle on its own."""
    ctx, orc, cfg = tiny3
    B = _B()
    for rnd in range(3):
        for Bn, K in [(32, 3), (5, 1), (64, 3)]:
            ids = S.uniform_ids(Bn * (K + 1), 900 + 7 * rnd + Bn, K, cfg.vocab).reshape(Bn, K + 1)
            tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]))
            check_tokens(orc, ids.reshape(-1), tg.cpu().numpy().reshape(-1),
                         label=f"tiny 3 layers B={Bn} K={K} round {rnd}")
        T = 9 + rnd
        hin = S.hidden_input(T, cfg.hidden, seed=S.SEED_HIDDEN + 50 + rnd)
        hin_t = torch.from_numpy(hin.view(np.int16)).cuda().view(torch.bfloat16)
        probe, pt = B.make_probe(1, T, cfg)
        hout = ctx.layer(rnd % cfg.n_layers, hin_t, probe=probe)
        got = hout.view(torch.int16).cpu().numpy().view(np.uint16)
        gsel = pt["topk_idx"].cpu().numpy()[0]
        for t in range(T):
            _, _, sel, _, gap = orc.layer_bf16(rnd % cfg.n_layers, hin[t])
            if set(sel.tolist()) != set(gsel[t].tolist()):
                assert gap < TIE, (rnd, t, gap)
            _, f64, _, _, _ = orc.layer_bf16(rnd % cfg.n_layers, hin[t], force_sel=gsel[t])
            assert rel_err(S.bf16_bits_to_f32(got[t]), f64) <= REL, (rnd, t)
    assert ctx.sync_status() == B.OK


# ---------------------------------------------------------- single MoE block

@pytest.mark.parametrize("T", [4, 1, 37, 128, 300, 1024, 4096])
def test_layer_matches_oracle(layer, T):
    """One block at hidden 1280, 64 experts of 896, top-6, 2 shared: routing
    sets, weights and the bf16 output."""
    ctx, orc = layer
    B = _B()
    hin = S.hidden_input(T, 1280, seed=S.SEED_HIDDEN + T)
    hin_t = torch.from_numpy(hin.view(np.int16)).cuda().view(torch.bfloat16)
    probe, pt = B.make_probe(1, T, S.LAYER)
    hout = ctx.layer(0, hin_t, probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    got = hout.view(torch.int16).cpu().numpy().view(np.uint16)
    gsel = pt["topk_idx"].cpu().numpy()[0]
    gw = pt["topk_w"].cpu().numpy()[0]
    sample = range(T) if T <= 128 else sorted(set(np.linspace(0, T - 1, 96).astype(int).tolist()))
    ties = 0

    def one(t):
        _, _, sel, _, gap = orc.layer_bf16(0, hin[t])
        tie = 0
        if set(sel.tolist()) != set(gsel[t].tolist()):
            assert gap < TIE, (t, sorted(sel.tolist()), sorted(gsel[t].tolist()), gap)
            tie = 1
        out, f64, _, wts, _ = orc.layer_bf16(0, hin[t], force_sel=gsel[t])
        assert np.max(np.abs(gw[t] - wts) / np.abs(wts)) <= REL
        e = rel_err(S.bf16_bits_to_f32(got[t]), f64)
        assert e <= REL, (t, e)
        return tie

    import concurrent.futures as fut
    with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
        ties = sum(ex.map(one, sample))
    print(f"layer T={T}: {len(sample)} tokens checked, {ties} routing near ties")


# ------------------------------------------------------------ the full stack

def test_full_step_batch32_k3_every_token(full):
    """The 12-layer stack, B=32 sequences x (1 + 3 drafts): all 128 verify
    tokens against the oracle, every block teacher-forced and free-running."""
    ctx, orc = full
    B = _B()
    ids = S.uniform_ids(32 * 4, S.SEED_START_IDS, 7, S.FULL.vocab).reshape(32, 4)
    probe, pt = B.make_probe(S.FULL.n_layers, 128, S.FULL)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    got = tg.cpu().numpy().reshape(-1)
    stats = check_tokens(orc, ids.reshape(-1), got, pt["topk_idx"].cpu().numpy(),
                         pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(),
                         label="full B=32 K=3, all 128 tokens")
    print("full:", stats)


def test_full_logits_probe_sampled(full):
    """lm_head logits at full size (hidden 1280, vocabulary 129,280), T = 128
    (the tokens-on-M form): on sampled tokens, within max relative error 2e-2
    of the oracle's logits along the GPU's routing, and their argmax is the
    GPU's target.  Records the largest absolute logit difference, which the
    free-running logit band is set from."""
    ctx, orc = full
    B = _B()
    ids = S.uniform_ids(32 * 4, S.SEED_START_IDS, 9, S.FULL.vocab).reshape(32, 4)
    probe, pt = B.make_probe(S.FULL.n_layers, 128, S.FULL, logits=True)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    got = tg.cpu().numpy().reshape(-1)
    idx = pt["topk_idx"].cpu().numpy()
    sample = list(range(0, 128, 8))
    lg = pt["logits"].cpu().numpy()[sample]
    assert np.array_equal(np.argmax(lg, axis=1), got[sample])

    def one(j):
        t = sample[j]
        r = orc.forward_token(int(ids.reshape(-1)[t]), force_sel=idx[:, t, :], logits=True)
        return float(rel_err(lg[j], r["logits"])), float(np.max(np.abs(lg[j] - r["logits"])))

    import concurrent.futures as fut
    with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
        res = list(ex.map(one, range(len(sample))))
    worst_rel = max(r[0] for r in res)
    worst_abs = max(r[1] for r in res)
    parity.record("full B=32 K=3 logits, 16 tokens", tokens=len(sample),
                  max_logit_rel=round(worst_rel, 6), max_logit_abs_diff=round(worst_abs, 6))
    assert worst_rel <= REL, res
    # a free-running target flip with identical routing needs a top-2 gap
    # below the two logits' errors: the band must cover that
    assert 2 * worst_abs < parity.FREE_LOGIT_BAND, worst_abs


def test_full_batch_invariance(full):
    """A token's target and residual stream do not depend on the rest of the
    batch (same bits alone and inside a batch of 32)."""
    ctx, _ = full
    B = _B()
    ids = S.uniform_ids(32 * 4, 77, 1, S.FULL.vocab).reshape(32, 4)
    pa, ta = B.make_probe(S.FULL.n_layers, 128, S.FULL, topk=False)
    big = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pa).cpu().numpy()
    ha = ta["hidden"].cpu().numpy()
    for b in (0, 13, 31):
        pb, tb = B.make_probe(S.FULL.n_layers, 4, S.FULL, topk=False)
        one = ctx.step(_i32(ids[b:b + 1, 0]), _i32(ids[b:b + 1, 1:]), probe=pb).cpu().numpy()
        assert np.array_equal(one[0], big[b])
        assert np.array_equal(tb["hidden"].cpu().numpy(), ha[:, 4 * b:4 * b + 4, :])


def test_full_step_same_bits_on_any_grid(full):
    """The persistent kernels on fewer CTAs than SMs (a context that holds
    part of the GPU) and on twice as many as fit at once (CTAs that start
    only after others have finished): targets and every block's residual
    stream are the same bits as on one CTA per SM, with no wait running out."""
    ctx, _ = full
    B = _B()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ids = S.uniform_ids(32 * 4, 88, 1, S.FULL.vocab).reshape(32, 4)
    pa, ta = B.make_probe(S.FULL.n_layers, 128, S.FULL, topk=False)
    want = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pa).cpu().numpy()
    hw = ta["hidden"].cpu().numpy()
    assert ctx.sync_status() == B.OK
    try:
        for ctas in (19, 2 * sms, 1):
            ctx.set_grid(ctas)
            pb, tb = B.make_probe(S.FULL.n_layers, 128, S.FULL, topk=False)
            got = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pb).cpu().numpy()
            assert ctx.sync_status() == B.OK, ctas
            assert np.array_equal(got, want), ctas
            assert np.array_equal(tb["hidden"].cpu().numpy(), hw), ctas
    finally:
        ctx.set_grid(0)
    with pytest.raises(B.MoeVerifyError):
        ctx.set_grid(-1)
    with pytest.raises(B.MoeVerifyError):
        ctx.set_grid(8 * sms + 1)


# B = 1 with the layer kernel: routing and expert items in one launch per layer
@pytest.mark.parametrize("Bn,fused", [(32, False), (1, False), (1, True)])
def test_full_step_launch_stamps(full, Bn, fused):
    """Launch timestamps of a graph-replayed step: each launch starts before
    it ends, and its wait for the preceding launch returns only after that
    launch's last CTA has ended (the dependency the launch chain relies on;
    in the single-kernel layer, the expert items start only after the layer's
    routing tasks have ended).  Targets are unchanged by the stamps."""
    ctx, _ = full
    L = S.FULL.n_layers
    ids = S.uniform_ids(Bn * 4, 89, 1, S.FULL.vocab).reshape(Bn, 4)
    ctxi, dr = _i32(ids[:, 0]), _i32(ids[:, 1:])
    want = ctx.step(ctxi, dr).clone()
    stamps = torch.zeros((2 * L + 1, 4), dtype=torch.int64, device="cuda")
    init = torch.zeros_like(stamps)
    init[:, 0] = -1  # all bits set: UINT64_MAX as the library reads it
    tg = torch.empty((Bn, 4), dtype=torch.int32, device="cuda")
    ctx.set_stamps(stamps)
    ctx.set_layer_kernel(8 if fused else 0)
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ctx.step(ctxi, dr, target_ids=tg, stream=s)
    finally:
        ctx.set_stamps(None)
        ctx.set_layer_kernel(0)
    for _ in range(2):
        stamps.copy_(init)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(tg, want)
        st = stamps.cpu().numpy().view(np.uint64)
        assert np.all(st[:, 0] < st[:, 2]), st
        assert np.all(st[:, 1] <= st[:, 2]) and np.all(st[:, 1] > 0), st
        for j in range(1, 2 * L + 1):
            assert st[j, 1] >= st[j - 1, 2], (j, st[j - 1], st[j])
        ffn_us = (st[1:2 * L:2, 2] - st[1:2 * L:2, 1]) / 1e3
        assert np.all(ffn_us > 5) and np.all(ffn_us < 2000), ffn_us


def test_full_decode_host_matches_device(full):
    """The host-buffer entry point (a graph per (B, K) after its first call)
    returns what step + accept return, over repeated and alternating shapes."""
    ctx, _ = full
    for rep in range(3):
        for Bn, K in [(32, 3), (5, 1), (32, 3), (1, 0), (17, 2)]:
            ids = S.uniform_ids(Bn * (K + 1), 91 + rep, 1 + Bn + K, S.FULL.vocab).reshape(Bn, K + 1)
            ctxi = _i32(ids[:, 0])
            dr = _i32(ids[:, 1:]) if K else None
            tg = ctx.step(ctxi, dr)
            com, alen = ctx.accept(dr, tg)
            hc = np.zeros((Bn, K + 1), np.int32)
            ha = np.zeros(Bn, np.int32)
            ctx.decode_host(np.ascontiguousarray(ids[:, 0]),
                            np.ascontiguousarray(ids[:, 1:]) if K else None, hc, ha)
            assert np.array_equal(hc, com.cpu().numpy()), (rep, Bn, K)
            assert np.array_equal(ha, alen.cpu().numpy()), (rep, Bn, K)


def test_full_graph_capture(full):
    ctx, _ = full
    ids = S.uniform_ids(32 * 4, 93, 1, S.FULL.vocab).reshape(32, 4)
    ctxi, dr = _i32(ids[:, 0]), _i32(ids[:, 1:])
    tg = torch.empty((32, 4), dtype=torch.int32, device="cuda")
    com = torch.empty((32, 4), dtype=torch.int32, device="cuda")
    alen = torch.empty((32,), dtype=torch.int32, device="cuda")
    want = ctx.step(ctxi, dr).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ctx.step(ctxi, dr, target_ids=tg, stream=s)
        ctx.accept(dr, tg, committed=com, accept_len=alen, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(tg, want)
    wc, wl, _ = O.accept(ids[:, 1:], want.cpu().numpy(), S.FULL.vocab)
    assert np.array_equal(com.cpu().numpy(), wc) and np.array_equal(alen.cpu().numpy(), wl)


# --------------------------------------------------------------- acceptance

@pytest.mark.parametrize("Bn,K", [(1, 0), (1, 1), (7, 3), (1000, 3), (33, 15), (64, 2)])
def test_accept_matches_oracle(tiny, Bn, K):
    ctx, _ = tiny
    rng = np.random.default_rng(Bn * 31 + K)
    y = rng.integers(0, 4, size=(Bn, K + 1)).astype(np.int32)
    d = rng.integers(0, 4, size=(Bn, K)).astype(np.int32)
    if Bn > 2:  # a few invalid rows: id -1 and id == V
        if K:
            d.reshape(-1)[rng.integers(0, d.size, 2)] = -1
        y[rng.integers(0, Bn), rng.integers(0, K + 1)] = 512
    com, alen = ctx.accept(_i32(d) if K else None, _i32(y))
    wc, wl, wbad = O.accept(d, y, 512)
    assert np.array_equal(com.cpu().numpy(), wc)
    assert np.array_equal(alen.cpu().numpy(), wl)
    rc = ctx.sync_status()
    B = _B()
    assert rc == (B.ERR_ID_RANGE if wbad else B.OK)


def test_step_flags_out_of_range_ids(tiny):
    ctx, _ = tiny
    B = _B()
    assert ctx.sync_status() == B.OK
    ids = np.array([[1, 2, 3, 4], [512, 5, 6, 7], [8, -3, 9, 10]], dtype=np.int32)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:])).cpu().numpy()
    assert tg[1, 0] == -1 and tg[2, 1] == -1
    assert np.all(tg[0] >= 0) and tg[1, 1] >= 0
    assert ctx.sync_status() == B.ERR_ID_RANGE
    assert ctx.sync_status() == B.OK
    com, alen = ctx.accept(_i32(ids[:, 1:]), _i32(tg))
    assert alen.cpu().numpy()[1] == -1 and alen.cpu().numpy()[2] == -1


def test_bounded_waits_give_up_and_report(tiny):
    """A wait on an mbarrier phase nothing completes and a spin on a flag
    nothing sets both give up after their limit and raise the timeout bit;
    the context keeps working afterwards."""
    ctx, orc = tiny
    B = _B()
    ctx.sync_status()  # clear what earlier tests on this context left
    limit = 2_000_000  # 2 ms each
    rc, elapsed = B.check_bounded_wait(limit)
    assert rc == B.OK, B.strerror(rc)
    assert 2 * limit <= elapsed < 2 * limit + 50_000_000, elapsed
    ids = S.uniform_ids(8, 77, 3, 512).reshape(2, 4)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]))
    check_tokens(orc, ids.reshape(-1), tg.cpu().numpy().reshape(-1),
                 label="tiny after the bounded-wait check")
    assert ctx.sync_status() == B.OK


def test_host_argument_errors(tiny):
    ctx, _ = tiny
    B = _B()
    with pytest.raises(B.MoeVerifyError) as e:
        ctx.step(_i32(np.zeros(129)), _i32(np.zeros((129, 3))))
    assert e.value.code == B.ERR_ARG
    with pytest.raises(B.MoeVerifyError) as e:
        ctx.step(_i32(np.zeros(4)), _i32(np.zeros((4, 4))))
    assert e.value.code == B.ERR_ARG
    with pytest.raises(B.MoeVerifyError) as e:
        ctx.layer(5, torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == B.ERR_ARG


# ------------------------------------------------ skewed routing and the sweep

@pytest.fixture(scope="module")
def full_zipf(full):
    """The full stack with the Zipf(s=1.2) router bias, room for 256 x 4 tokens."""
    B = _B()
    w = dict(full[1].w)
    w["router_bias"] = S.router_bias(S.FULL_ZIPF)
    ctx = B.MoeVerify(S.FULL_ZIPF, B.weights_to_device(w), max_batch=256, max_k=3)
    torch.cuda.empty_cache()
    yield ctx, O.Oracle(S.FULL_ZIPF, w)
    ctx.close()


def test_full_zipf_batch256_k3_sampled(full_zipf):
    """Skewed routing, 1,024 verify tokens: one expert takes almost every
    token (its rows are cut into several items).  Routing and residual stream
    of every token come from the probes; 128 sampled tokens against the oracle."""
    ctx, orc = full_zipf
    B = _B()
    ids = S.uniform_ids(256 * 4, S.SEED_START_IDS, 13, S.FULL.vocab).reshape(256, 4)
    probe, pt = B.make_probe(S.FULL.n_layers, 1024, S.FULL)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    idx = pt["topk_idx"].cpu().numpy()
    counts = np.bincount(idx[0].reshape(-1), minlength=64)
    assert counts[0] > 512, counts[:8]           # the skew is there
    sample = list(range(3, 1024, 8))
    stats = check_tokens(orc, ids.reshape(-1), tg.cpu().numpy().reshape(-1), idx,
                         pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(), sample=sample,
                         label="zipf B=256 K=3, 128 of 1024 tokens")
    print("zipf:", stats, "layer-0 expert counts (top 4):", sorted(counts)[-4:])


@pytest.mark.parametrize("Bn", [1, 8, 32, 128])
@pytest.mark.parametrize("K", [1, 2, 3])
def test_sweep_shapes_sampled(full, Bn, K):
    """The sweep's shapes (B in {1, 8, 32, 128} x K in {1, 2, 3}): every
    block and the target of sampled tokens, teacher-forced."""
    ctx, orc = full
    B = _B()
    if Bn > 32:
        pytest.skip("covered by the 256-sequence context below")
    T = Bn * (K + 1)
    ids = S.uniform_ids(T, 61 + Bn, K, S.FULL.vocab).reshape(Bn, K + 1)
    probe, pt = B.make_probe(S.FULL.n_layers, T, S.FULL)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    sample = sorted(set(np.linspace(0, T - 1, min(T, 4)).astype(int).tolist()))
    check_tokens(orc, ids.reshape(-1), tg.cpu().numpy().reshape(-1), pt["topk_idx"].cpu().numpy(),
                 pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(), sample=sample,
                 label=f"sweep B={Bn} K={K}")


@pytest.mark.parametrize("K", [1, 2, 3])
def test_sweep_batch128_sampled(full_zipf_free, K):
    ctx, orc = full_zipf_free
    B = _B()
    T = 128 * (K + 1)
    ids = S.uniform_ids(T, 67, K, S.FULL.vocab).reshape(128, K + 1)
    probe, pt = B.make_probe(S.FULL.n_layers, T, S.FULL)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    sample = sorted(set(np.linspace(0, T - 1, 4).astype(int).tolist()))
    check_tokens(orc, ids.reshape(-1), tg.cpu().numpy().reshape(-1), pt["topk_idx"].cpu().numpy(),
                 pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(), sample=sample,
                 label=f"sweep B=128 K={K}")


def test_full_batch_invariance_across_ffn_forms(full_zipf_free):
    """Inside a batch of 512 verify tokens the expert FFN runs token-major
    (rows on the MMA's M side); alone, a sequence's 4 tokens run weight-major.
    Targets and every block's residual stream are the same bits either way."""
    ctx, _ = full_zipf_free
    B = _B()
    ids = S.uniform_ids(128 * 4, 78, 1, S.FULL.vocab).reshape(128, 4)
    pa, ta = B.make_probe(S.FULL.n_layers, 512, S.FULL, topk=False)
    big = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pa).cpu().numpy()
    ha = ta["hidden"].cpu().numpy()
    for b in (0, 77, 127):
        pb, tb = B.make_probe(S.FULL.n_layers, 4, S.FULL, topk=False)
        one = ctx.step(_i32(ids[b:b + 1, 0]), _i32(ids[b:b + 1, 1:]), probe=pb).cpu().numpy()
        assert np.array_equal(tb["hidden"].cpu().numpy(), ha[:, 4 * b:4 * b + 4, :]), b
        assert np.array_equal(one[0], big[b]), b


@pytest.fixture(scope="module")
def full_zipf_free(full):
    """The full stack without bias, room for 128 x 4 tokens."""
    B = _B()
    ctx = B.MoeVerify(S.FULL, B.weights_to_device(full[1].w), max_batch=128, max_k=3)
    torch.cuda.empty_cache()
    yield ctx, full[1]
    ctx.close()


@pytest.mark.parametrize("Bn,K,p", [(8, 2, 0.576), (32, 3, 0.75), (1, 1, 0.576)])
def test_decode_loop(full, Bn, K, p):
    """A few decode iterations through step + accept on the GPU, drafts taken
    from the oracle's greedy chain with probability p.  Each step's targets are
    checked teacher-forced against the oracle (every block and the final
    argmax, exact outside near ties); the commits are exactly the acceptance
    rule applied to those targets.  Commits that differ from the oracle's own
    free-running chain are counted; every verify token whose GPU target
    differs from the oracle's free-running target is among the checked
    tokens, so each such difference lies inside the free-running bands."""
    ctx, orc = full
    B = _B()
    V = S.FULL.vocab
    src = S.DraftSource(p, V, K, seed=5)
    last = S.start_ids(Bn, V, first=900).astype(np.int64)
    memo = {}

    def g(x):
        if x not in memo:
            memo[x] = orc.target(int(x))
        return memo[x]

    import concurrent.futures as fut
    drift = 0
    committed_total = 0
    for step in range(3):
        with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
            list(ex.map(g, sorted(set(last.tolist()))))
        chains = np.zeros((Bn, K + 1), dtype=np.int64)
        for b in range(Bn):
            x = int(last[b])
            for i in range(K + 1):
                if i > 0 and x not in memo:
                    memo[x] = orc.target(x)
                x = g(x)
                chains[b, i] = x
        drafts = np.stack([src.drafts(b, step, chains[b, :K]) for b in range(Bn)])
        T = Bn * (K + 1)
        probe, pt = B.make_probe(S.FULL.n_layers, T, S.FULL)
        tg = ctx.step(_i32(last), _i32(drafts), probe=probe)
        com, alen = ctx.accept(_i32(drafts), tg)
        tg, com, alen = tg.cpu().numpy(), com.cpu().numpy(), alen.cpu().numpy()
        ids = np.concatenate([last.reshape(-1, 1), drafts], axis=1).reshape(-1)
        with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
            list(ex.map(g, sorted(set(ids.tolist()) - set(memo))))
        free_diff = [t for t in range(T) if int(tg.reshape(-1)[t]) != memo[int(ids[t])]]
        sample = sorted(set(np.linspace(0, T - 1, min(T, 8)).astype(int).tolist()) |
                        set(free_diff))
        check_tokens(orc, ids, tg.reshape(-1), pt["topk_idx"].cpu().numpy(),
                     pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(), sample=sample,
                     label=f"decode B={Bn} K={K} p={p} step {step}")
        wc, wl, _ = O.accept(drafts, tg, V)
        assert np.array_equal(com, wc) and np.array_equal(alen, wl)
        for b in range(Bn):
            n = int(alen[b])
            committed_total += n + 1
            drift += int(np.sum(com[b, : n + 1] != chains[b, : n + 1]))
            last[b] = int(com[b, n])
    parity.record(f"decode loop B={Bn} K={K} p={p}, 3 steps", committed=committed_total,
                  differ_from_oracle_chain=drift)
    print(f"decode B={Bn} K={K} p={p}: {committed_total} committed, "
          f"{drift} differ from the oracle's free-running chain")


# ------------------------------------------------------------- draft head

@pytest.fixture(scope="module")
def tiny_draft():
    B = _B()
    tw = S.make_weights(S.TINY)
    dw = S.make_draft_weights(S.DRAFT_TINY, tw)
    dctx = B.MoeVerify(S.DRAFT_TINY, B.weights_to_device(dw), max_batch=128, max_k=0)
    yield dctx, O.Oracle(S.DRAFT_TINY, dw)
    dctx.close()


def _check_drafts(dorc, h, t, drafts, hidden, K):
    """Each sequence's draft chain against the oracle's from the same inputs:
    equal until a step whose top-2 logit gap is below the tie band (then the
    rest of that chain is not compared); states within REL before it."""
    ties = 0
    for b in range(h.shape[0]):
        od, oh, og = dorc.draft(h[b].astype(np.float64), int(t[b]), K)
        for i in range(K):
            if drafts[b, i] != od[i]:
                assert og[i] < TIE, (b, i, int(drafts[b, i]), int(od[i]), og[i])
                ties += 1
                break
            assert rel_err(hidden[i, b], oh[i]) <= REL, (b, i)
    return ties


def test_draft_head_tiny_matches_oracle(tiny, tiny_draft):
    ctx, _ = tiny
    dctx, dorc = tiny_draft
    B = _B()
    L = S.TINY.n_layers
    ids = S.uniform_ids(128 * 4, 301, 3, 512).reshape(128, 4)
    probe, pt = B.make_probe(L, 512, S.TINY)
    dr = _i32(ids[:, 1:])
    tg = ctx.step(_i32(ids[:, 0]), dr, probe=probe)
    com, alen = ctx.accept(dr, tg)
    h, t = ctx.draft_inputs(com, alen)
    # the inputs: final residual and committed token of each accepted position
    n = np.maximum(alen.cpu().numpy(), 0)
    rows = np.arange(128) * 4 + n
    hfin = pt["hidden"].cpu().numpy()[L]
    assert np.array_equal(h.cpu().numpy(), hfin[rows])
    assert np.array_equal(t.cpu().numpy(), com.cpu().numpy()[np.arange(128), n])
    drafts, hidden = dctx.draft(h, t, 3, hidden=True)
    torch.cuda.synchronize()
    assert dctx.sync_status() == B.OK
    ties = _check_drafts(dorc, h.cpu().numpy(), t.cpu().numpy(), drafts.cpu().numpy(),
                         hidden.cpu().numpy(), 3)
    print(f"draft tiny: 128 chains x 3 steps, {ties} logit near ties")


def test_decode_loop_with_draft_head_is_lossless(tiny, tiny_draft):
    """Verify, accept and draft on the device, drafts fed back: whatever the
    draft head proposes, the committed stream is plain greedy decoding."""
    ctx, _ = tiny
    dctx, _ = tiny_draft
    g = np.loadtxt(os.path.join(GOLDEN, "tiny_g_table.txt"), dtype=np.int64)
    Bn, K = 16, 3
    start = S.uniform_ids(Bn, 402, 0, 512).astype(np.int64)
    streams = [[] for _ in range(Bn)]
    # a first verify step without drafts, then K drafts per step
    tg = ctx.step(_i32(start), None)
    com, alen = ctx.accept(None, tg)
    accepted = 0
    for it in range(12):
        comh, nh = com.cpu().numpy(), alen.cpu().numpy()
        for b in range(Bn):
            streams[b] += [int(x) for x in comh[b, : nh[b] + 1]]
        accepted += int(nh.sum()) if it else 0
        h, t = ctx.draft_inputs(com, alen)
        dr = dctx.draft(h, t, K)
        tg = ctx.step(t, dr)
        com, alen = ctx.accept(dr, tg)
    assert ctx.sync_status() == _B().OK and dctx.sync_status() == _B().OK
    for b in range(Bn):
        x, want = int(start[b]), []
        for _ in range(len(streams[b])):
            x = int(g[x])
            want.append(x)
        assert streams[b] == want, b
    print(f"decode loop: {sum(map(len, streams))} tokens committed, {accepted} drafts accepted")


@pytest.fixture(scope="module")
def full_draft():
    B = _B()
    tw = S.make_weights(S.FULL)
    dw = S.make_draft_weights(S.DRAFT, tw)
    dctx = B.MoeVerify(S.DRAFT, B.weights_to_device(dw), max_batch=32, max_k=0)
    torch.cuda.empty_cache()
    yield dctx, O.Oracle(S.DRAFT, dw)
    dctx.close()


def test_draft_head_full_sampled(full, full_draft):
    """The 1280-wide draft block (one 5120-wide SwiGLU) with the 129,280-token
    head, B = 32 after a K = 3 verify step: 8 sampled chains vs the oracle."""
    ctx, _ = full
    dctx, dorc = full_draft
    ids = S.uniform_ids(32 * 4, 511, 3, S.FULL.vocab).reshape(32, 4)
    dr = _i32(ids[:, 1:])
    tg = ctx.step(_i32(ids[:, 0]), dr)
    com, alen = ctx.accept(dr, tg)
    h, t = ctx.draft_inputs(com, alen)
    drafts, hidden = dctx.draft(h, t, 3, hidden=True)
    torch.cuda.synchronize()
    assert dctx.sync_status() == _B().OK
    pick = np.linspace(0, 31, 8).astype(int)
    hh, tt = h.cpu().numpy()[pick], t.cpu().numpy()[pick]
    dd, hd = drafts.cpu().numpy()[pick], hidden.cpu().numpy()[:, pick]
    import concurrent.futures as fut

    def one(j):
        return _check_drafts(dorc, hh[j:j + 1], tt[j:j + 1], dd[j:j + 1], hd[:, j:j + 1], 3)

    with fut.ThreadPoolExecutor(max_workers=threads()) as ex:
        ties = sum(ex.map(one, range(len(pick))))
    print(f"draft full: 8 chains x 3 steps, {ties} logit near ties")


def test_decode_iteration_in_one_graph(full, full_draft):
    """Verify step, accept, draft inputs and the K-step draft captured as one
    CUDA graph: replays match the same calls made eagerly."""
    ctx, _ = full
    dctx, _ = full_draft
    Bn, K = 32, 3
    ids = S.uniform_ids(Bn * 4, 612, 3, S.FULL.vocab).reshape(Bn, 4)
    c0, d0 = _i32(ids[:, 0]), _i32(ids[:, 1:])
    # eager reference for three iterations
    ref = []
    c, d = c0.clone(), d0.clone()
    for _ in range(3):
        tg = ctx.step(c, d)
        com, alen = ctx.accept(d, tg)
        h, t = ctx.draft_inputs(com, alen)
        d = dctx.draft(h, t, K)
        c = t
        ref.append((com.clone(), d.clone()))
    # the same iteration as one graph on fixed buffers
    in_c, in_d = c0.clone(), d0.clone()
    tg = torch.empty((Bn, K + 1), dtype=torch.int32, device="cuda")
    com = torch.empty_like(tg)
    alen = torch.empty((Bn,), dtype=torch.int32, device="cuda")
    h = torch.empty((Bn, S.FULL.hidden), dtype=torch.float32, device="cuda")
    t = torch.empty((Bn,), dtype=torch.int32, device="cuda")
    out_d = torch.empty((Bn, K), dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())

    def iteration():
        ctx.step(in_c, in_d, target_ids=tg, stream=st)
        ctx.accept(in_d, tg, committed=com, accept_len=alen, stream=st)
        ctx.draft_inputs(com, alen, h_out=h, t_out=t, stream=st)
        dctx.draft(h, t, K, drafts=out_d, stream=st)

    with torch.cuda.stream(st):
        iteration()
    st.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        iteration()
    in_c.copy_(c0)
    in_d.copy_(d0)
    for r in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(com, ref[r][0]), r
        assert torch.equal(out_d, ref[r][1]), r
        in_c.copy_(t)
        in_d.copy_(out_d)


@pytest.fixture(scope="module")
def full_two_layers():
    """Two blocks of the full-width stack, room for 128 x 4 tokens."""
    import dataclasses
    B = _B()
    cfg = dataclasses.replace(S.FULL, n_layers=2, name="full_two_layers")
    ctx = B.MoeVerify(cfg, B.weights_to_device(S.make_weights(cfg)), max_batch=128, max_k=3)
    torch.cuda.empty_cache()
    yield ctx, cfg
    ctx.close()


def test_large_batch_same_bits_on_any_grid(full_two_layers):
    """512 tokens (token-major expert FFN, lm_head on CTA pairs) on 1 CTA
    (the lm_head falls back to single CTAs: no pair fits), 3 CTAs (one pair)
    and twice as many as fit at once: targets and every block's residual
    stream are the same bits as on one CTA per SM."""
    ctx, cfg = full_two_layers
    B = _B()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ids = S.uniform_ids(128 * 4, 91, 1, cfg.vocab).reshape(128, 4)
    pa, ta = B.make_probe(cfg.n_layers, 512, cfg, topk=False)
    want = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pa).cpu().numpy()
    hw = ta["hidden"].cpu().numpy()
    assert ctx.sync_status() == B.OK
    try:
        for ctas in (3, 2 * sms, 1):
            ctx.set_grid(ctas)
            pb, tb = B.make_probe(cfg.n_layers, 512, cfg, topk=False)
            got = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=pb).cpu().numpy()
            assert ctx.sync_status() == B.OK, ctas
            assert np.array_equal(got, want), ctas
            assert np.array_equal(tb["hidden"].cpu().numpy(), hw), ctas
    finally:
        ctx.set_grid(0)
