"""The allocation-free greedy head (moe_verify_greedy_head_noalloc).

Callers that cannot allocate device memory (their memory belongs to another
allocator with a fixed budget, they must not stall other streams, or they run
where CUDA allocation calls are not allowed) use this entry point: its
scratch is a fixed array inside the library.  Here it must give the same
targets as the regular verify step on the step's own final residual stream,
and the oracle's greedy head on those rows (outside the 1e-3 logit band), on
consecutive calls, including a call with fewer rows and a narrower hidden size
after a larger one (the shared scratch then still holds the earlier call's
rows), and it must not change the device's free memory once its first call on
the device has looked up the array's address.

This file sorts last so that a run which stops at the first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TIE = 1e-3


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _step_final_residual(B, ctx, cfg, Bn, K, seed):
    """A verify step; returns (its targets [T], its final residual rows [T, d])."""
    ids = S.uniform_ids(Bn * (K + 1), seed, 3, cfg.vocab).reshape(Bn, K + 1)
    T = Bn * (K + 1)
    probe, pt = B.make_probe(cfg.n_layers, T, cfg, topk=False)
    want = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]) if K else None, probe=probe).reshape(-1)
    return want, pt["hidden"][cfg.n_layers].contiguous()


def _check_against_oracle(orc, h_final, got):
    """Each row's target equals the oracle's greedy head on the same residual
    row, unless the oracle's own top-2 logit gap is below the tie band."""
    H = h_final.cpu().numpy().astype(np.float64)
    g = got.cpu().numpy()
    ties = 0
    for t in range(H.shape[0]):
        tgt, gap, _ = orc.head(H[t])
        if int(g[t]) != tgt:
            assert gap < TIE, (t, int(g[t]), tgt, gap)
            ties += 1
    return ties


def _noalloc(B, h_final, wd, cfg, check_free_memory):
    got = torch.full((h_final.shape[0],), -5, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    B.greedy_head_noalloc(h_final, wd["final_norm"], wd["lm_head"], cfg.rms_eps, target_ids=got)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    if check_free_memory:
        assert free1 == free0, "the call changed the device's free memory"
    return got


@pytest.mark.parametrize("cfg", [S.TINY, S.LAYER], ids=["tiny_d64", "layer_d1280"])
def test_noalloc_head_matches_step_on_two_calls(cfg):
    from moe_speculative_decoding_router_gb300 import binding as B
    w = S.make_weights(cfg)
    wd = B.weights_to_device(w)
    orc = O.Oracle(cfg, w)
    ctx = B.MoeVerify(cfg, wd, max_batch=64, max_k=3)
    try:
        # T = 128 (tokens on the MMA's M side), then T = 150 (vocabulary on M)
        for call, (Bn, K) in enumerate(((32, 3), (50, 2))):
            want, h_final = _step_final_residual(B, ctx, cfg, Bn, K, 500 + call)
            # the first call on the device may load the module
            got = _noalloc(B, h_final, wd, cfg, check_free_memory=call == 1)
            assert torch.equal(got, want), (got.cpu().numpy(), want.cpu().numpy())
            _check_against_oracle(orc, h_final, got)
        assert ctx.sync_status() == B.OK
    finally:
        ctx.close()


def test_noalloc_head_small_narrow_call_after_large_wide_one():
    """T = 150 rows of hidden 1280, then T = 4 rows of hidden 64: the second
    call's tiles cover scratch rows that still hold the first call's values;
    only its own rows may count."""
    from moe_speculative_decoding_router_gb300 import binding as B
    results = []
    for cfg, (Bn, K), seed in ((S.LAYER, (50, 2), 700), (S.TINY, (1, 3), 701),
                               (S.TINY, (3, 0), 702)):
        w = S.make_weights(cfg)
        wd = B.weights_to_device(w)
        ctx = B.MoeVerify(cfg, wd, max_batch=64, max_k=3)
        try:
            want, h_final = _step_final_residual(B, ctx, cfg, Bn, K, seed)
            got = _noalloc(B, h_final, wd, cfg, check_free_memory=True)
            assert torch.equal(got, want), (cfg.hidden, got.cpu().numpy(), want.cpu().numpy())
            _check_against_oracle(O.Oracle(cfg, w), h_final, got)
            assert ctx.sync_status() == B.OK
            results.append(got.cpu().numpy())
        finally:
            ctx.close()
    assert [len(r) for r in results] == [150, 4, 3]


def test_noalloc_head_rejects_sizes_beyond_its_scratch():
    from moe_speculative_decoding_router_gb300 import binding as B
    lib = B.load()
    h = torch.zeros((257, 64), dtype=torch.float32, device="cuda")
    g = torch.ones((4096,), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((512, 4096), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((257,), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.moe_verify_greedy_head_noalloc(h.data_ptr(), g.data_ptr(), W.data_ptr(), 257, 64,
                                              512, 1e-6, out.data_ptr(), s) == B.ERR_UNSUPPORTED
    assert lib.moe_verify_greedy_head_noalloc(h.data_ptr(), g.data_ptr(), W.data_ptr(), 4, 4096,
                                              512, 1e-6, out.data_ptr(), s) == B.ERR_UNSUPPORTED
    assert lib.moe_verify_greedy_head_noalloc(None, g.data_ptr(), W.data_ptr(), 4, 64, 512, 1e-6,
                                              out.data_ptr(), s) == B.ERR_ARG
