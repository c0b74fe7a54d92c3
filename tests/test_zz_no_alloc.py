"""The allocation-free greedy head (moe_verify_greedy_head_noalloc).

Callers that cannot allocate device memory (their memory belongs to another
allocator with a fixed budget, they must not stall other streams, or they run
where CUDA allocation calls are not allowed) use this entry point: its
scratch is a fixed array inside the library.  Here it must give the same
targets as the regular verify step on the step's own final residual stream,
on two calls in a row, and it must not change the device's free memory once
its first call on the device has looked up the array's address.

This file sorts last so that a run which stops at the first failure has run
every other test before it; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from moe_speculative_decoding_router_gb300 import synth as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("cfg", [S.TINY, S.LAYER], ids=["tiny_d64", "layer_d1280"])
def test_noalloc_head_matches_step_on_two_calls(cfg):
    from moe_speculative_decoding_router_gb300 import binding as B
    w = S.make_weights(cfg)
    wd = B.weights_to_device(w)
    ctx = B.MoeVerify(cfg, wd, max_batch=64, max_k=3)
    try:
        outs = []
        for call, (Bn, K) in enumerate(((32, 3), (50, 2))):
            ids = S.uniform_ids(Bn * (K + 1), 500 + call, 3, cfg.vocab).reshape(Bn, K + 1)
            T = Bn * (K + 1)
            probe, pt = B.make_probe(cfg.n_layers, T, cfg, topk=False)
            want = ctx.step(_i32(ids[:, 0]), _i32(ids[:, 1:]), probe=probe).reshape(-1)
            h_final = pt["hidden"][cfg.n_layers].contiguous()
            got = torch.full((T,), -5, dtype=torch.int32, device="cuda")
            torch.cuda.synchronize()
            free0 = torch.cuda.mem_get_info()[0]
            B.greedy_head_noalloc(h_final, wd["final_norm"], wd["lm_head"], cfg.rms_eps,
                                  target_ids=got)
            torch.cuda.synchronize()
            free1 = torch.cuda.mem_get_info()[0]
            if call == 1:  # the first call on the device may load the module
                assert free1 == free0, "the call changed the device's free memory"
            assert torch.equal(got, want), (got.cpu().numpy(), want.cpu().numpy())
            outs.append(got.cpu().numpy())
        assert ctx.sync_status() == B.OK
    finally:
        ctx.close()


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
