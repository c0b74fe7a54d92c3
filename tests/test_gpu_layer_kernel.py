"""The single-kernel layer (each layer's routing inside the expert-FFN
kernel) for steps of at most 8 verify tokens: the same bits as the two-launch
layer (routing kernel, then expert FFN), on any grid and across calls that
switch between the two, and the oracle's targets, checked per block."""
import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S
from parity import check_tokens

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _B():
    from moe_speculative_decoding_router_gb300 import binding
    return binding


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.fixture(scope="module")
def full():
    B = _B()
    w = S.make_weights(S.FULL)
    ctx = B.MoeVerify(S.FULL, B.weights_to_device(w), max_batch=32, max_k=7)
    torch.cuda.empty_cache()
    yield ctx, O.Oracle(S.FULL, w)
    ctx.close()


@pytest.fixture(scope="module")
def tiny():
    B = _B()
    w = S.make_weights(S.TINY)
    ctx = B.MoeVerify(S.TINY, B.weights_to_device(w), max_batch=8, max_k=7)
    yield ctx, O.Oracle(S.TINY, w)
    ctx.close()


def _run(ctx, cfg, ids, fused, topk=True):
    """One step on ids [B, K+1] with the layer kernel on (8) or off (0):
    targets and the probes as numpy arrays."""
    B = _B()
    Bn, K1 = ids.shape
    ctx.set_layer_kernel(8 if fused else 0)
    pr, t = B.make_probe(cfg.n_layers, Bn * K1, cfg, topk=topk)
    tg = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]) if K1 > 1 else None, probe=pr)
    out = {"targets": tg.cpu().numpy()}
    out.update({k: v.cpu().numpy() for k, v in t.items()})
    assert ctx.sync_status() == B.OK
    return out


@pytest.mark.parametrize("Bn,K", [(1, 0), (1, 1), (1, 3), (2, 3), (1, 7), (4, 1), (3, 1)])
def test_full_layer_kernel_same_bits_as_two_launches(full, Bn, K):
    ctx, _ = full
    ids = S.uniform_ids(Bn * (K + 1), 300 + 10 * Bn + K, 1, S.FULL.vocab).reshape(Bn, K + 1)
    try:
        a = _run(ctx, S.FULL, ids, True)
        b = _run(ctx, S.FULL, ids, False)
    finally:
        ctx.set_layer_kernel(0)
    for key in ("targets", "topk_idx", "topk_w", "hidden"):
        assert np.array_equal(a[key], b[key]), key


def test_full_layer_kernel_any_grid(full):
    """One CTA (it routes all 8 tokens, then runs every expert item), a few,
    and twice as many as fit at once: the same bits as one CTA per SM."""
    ctx, _ = full
    B = _B()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ids = S.uniform_ids(8, 321, 1, S.FULL.vocab).reshape(2, 4)
    want = _run(ctx, S.FULL, ids, True, topk=False)
    try:
        for ctas in (1, 3, 7, 2 * sms):
            ctx.set_grid(ctas)
            got = _run(ctx, S.FULL, ids, True, topk=False)
            assert np.array_equal(got["targets"], want["targets"]), ctas
            assert np.array_equal(got["hidden"], want["hidden"]), ctas
    finally:
        ctx.set_grid(0)
        ctx.set_layer_kernel(0)
    assert ctx.sync_status() == B.OK


def test_full_layer_kernel_interleaved_with_two_launch_steps(full):
    """Calls that alternate between the single-kernel layer (T <= 8) and the
    two launches (larger T, or the layer kernel off) leave the counters each
    form expects: every call gives what it gives alone."""
    ctx, _ = full
    shapes = [(1, 3), (32, 3), (2, 3), (1, 0), (16, 1), (1, 7), (8, 0), (1, 3)]
    calls = [S.uniform_ids(b * (k + 1), 400 + i, 1, S.FULL.vocab).reshape(b, k + 1)
             for i, (b, k) in enumerate(shapes)]
    try:
        want = [_run(ctx, S.FULL, ids, False, topk=False)["targets"] for ids in calls]
        for rep in range(2):
            for i, ids in enumerate(calls):
                got = _run(ctx, S.FULL, ids, (i + rep) % 3 != 2, topk=False)["targets"]
                assert np.array_equal(got, want[i]), (rep, i, shapes[i])
    finally:
        ctx.set_layer_kernel(0)


def test_full_layer_kernel_matches_oracle(full):
    """The single-kernel layer at B = 2, K = 3 (8 tokens): every block and the
    final argmax teacher-forced against the oracle, the trajectory within the
    hidden-state tolerance."""
    ctx, orc = full
    ids = S.uniform_ids(8, 333, 1, S.FULL.vocab).reshape(2, 4)
    r = _run(ctx, S.FULL, ids, True)
    ctx.set_layer_kernel(0)
    check_tokens(orc, ids.reshape(-1), r["targets"].reshape(-1), probe_idx=r["topk_idx"],
                 probe_w=r["topk_w"], probe_hidden=r["hidden"], label="full layer kernel B=2 K=3")


@pytest.mark.parametrize("Bn,K", [(1, 0), (1, 3), (2, 3), (1, 7)])
def test_tiny_layer_kernel_matches_oracle(tiny, Bn, K):
    ctx, orc = tiny
    ids = S.uniform_ids(Bn * (K + 1), 500 + 10 * Bn + K, K, S.TINY.vocab).reshape(Bn, K + 1)
    r = _run(ctx, S.TINY, ids, True)
    check_tokens(orc, ids.reshape(-1), r["targets"].reshape(-1), probe_idx=r["topk_idx"],
                 probe_w=r["topk_w"], probe_hidden=r["hidden"],
                 label=f"tiny layer kernel B={Bn} K={K}")
    b = _run(ctx, S.TINY, ids, False)
    for key in ("targets", "topk_idx", "topk_w", "hidden"):
        assert np.array_equal(r[key], b[key]), key
    ctx.set_layer_kernel(0)


def test_full_layer_kernel_decode_host(full):
    """The host-buffer entry point (one captured graph per shape) with the
    single-kernel layer: the same commits as with the two launches."""
    ctx, _ = full
    B = _B()
    out = {}
    try:
        for fused in (True, False):
            ctx.set_layer_kernel(8 if fused else 0)
            res = []
            for i, (Bn, K) in enumerate([(1, 3), (1, 1), (2, 3), (1, 3)]):
                ids = S.uniform_ids(Bn * (K + 1), 600 + i, 1, S.FULL.vocab).reshape(Bn, K + 1)
                com = np.zeros((Bn, K + 1), dtype=np.int32)
                alen = np.zeros(Bn, dtype=np.int32)
                ctx.decode_host(np.ascontiguousarray(ids[:, 0]),
                                np.ascontiguousarray(ids[:, 1:]) if K else None, com, alen)
                res.append((com.copy(), alen.copy()))
            out[fused] = res
            assert ctx.sync_status() == B.OK
    finally:
        ctx.set_layer_kernel(0)
    for (c1, a1), (c0, a0) in zip(out[True], out[False]):
        assert np.array_equal(c1, c0) and np.array_equal(a1, a0)


def test_layer_kernel_argument_range(full):
    ctx, _ = full
    B = _B()
    for bad in (-1, 9):
        with pytest.raises(B.MoeVerifyError):
            ctx.set_layer_kernel(bad)
    ctx.set_layer_kernel(0)
