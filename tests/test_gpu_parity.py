"""GPU parity: the CUDA path through the C ABI against the fp64 oracle."""
import os

import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S
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
                         pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy())
    g = np.loadtxt(os.path.join(GOLDEN, "tiny_g_table.txt"), dtype=np.int64)
    mism = np.nonzero(got != g[ids.reshape(-1)])[0]
    assert len(mism) <= stats["logit_ties"] + stats["route_ties"], mism
    print("tiny:", stats)


@pytest.mark.parametrize("Bn,K", [(1, 0), (1, 3), (3, 1), (4, 3), (128, 0), (77, 2)])
def test_tiny_batch_shapes(tiny, Bn, K):
    ctx, orc = tiny
    ids = S.uniform_ids(Bn * (K + 1), 41 + Bn, K, 512).reshape(Bn, K + 1)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]) if K else None)
    got = tg.cpu().numpy().reshape(-1)
    check_tokens(orc, ids.reshape(-1), got)


def test_tiny_logits_probe(tiny):
    ctx, orc = tiny
    B = _B()
    ids = np.array([[5, 9, 300, 511]], dtype=np.int32)
    probe, pt = B.make_probe(S.TINY.n_layers, 4, S.TINY, logits=True)
    ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    lg = pt["logits"].cpu().numpy()
    for t in range(4):
        r = orc.forward_token(int(ids[0, t]), force_sel=pt["topk_idx"].cpu().numpy()[:, t, :],
                              logits=True)
        assert rel_err(lg[t], r["logits"]) <= REL


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

def test_full_step_batch32_k3_sampled(full):
    """The 12-layer stack, B=32 sequences x (1 + 3 drafts): every token's
    routing and residual stream from the probes, 32 tokens against the oracle."""
    ctx, orc = full
    B = _B()
    ids = S.uniform_ids(32 * 4, S.SEED_START_IDS, 7, S.FULL.vocab).reshape(32, 4)
    probe, pt = B.make_probe(S.FULL.n_layers, 128, S.FULL)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe)
    torch.cuda.synchronize()
    assert ctx.sync_status() == B.OK
    got = tg.cpu().numpy().reshape(-1)
    sample = list(range(0, 128, 4))
    stats = check_tokens(orc, ids.reshape(-1), got, pt["topk_idx"].cpu().numpy(),
                         pt["topk_w"].cpu().numpy(), pt["hidden"].cpu().numpy(), sample=sample)
    print("full:", stats)


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


def test_full_decode_host_matches_device(full):
    ctx, _ = full
    ids = S.uniform_ids(32 * 4, 91, 1, S.FULL.vocab).reshape(32, 4)
    ctxi, dr = _i32(ids[:, 0]), _i32(ids[:, 1:])
    tg = ctx.step(ctxi, dr)
    com, alen = ctx.accept(dr, tg)
    hc = np.zeros((32, 4), np.int32)
    ha = np.zeros(32, np.int32)
    ctx.decode_host(np.ascontiguousarray(ids[:, 0]), np.ascontiguousarray(ids[:, 1:]), hc, ha)
    assert np.array_equal(hc, com.cpu().numpy())
    assert np.array_equal(ha, alen.cpu().numpy())


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
