"""The Python binding's argument marshalling, without a GPU: arrays of the
wrong type, layout or shape are refused with ValueError before the library is
called (the library reads every buffer as a dense array from its pointer)."""
import numpy as np
import pytest
import torch

from moe_speculative_decoding_router_gb300 import binding as B
from moe_speculative_decoding_router_gb300 import synth as S


def _detached_context():
    """A MoeVerify object with no library context behind it: any call that got
    past the argument checks would fail on the missing library."""
    m = B.MoeVerify.__new__(B.MoeVerify)
    m.cfg, m.lib, m.handle = S.TINY, None, None
    return m


def test_host_int32_arrays():
    ok = np.zeros((4, 3), np.int32)
    assert B._host_i32(ok, "a", (4, 3)) is ok
    with pytest.raises(ValueError):
        B._host_i32(np.zeros((4, 3), np.int64), "a", (4, 3))           # dtype
    with pytest.raises(ValueError):
        B._host_i32(np.zeros((3, 4), np.int32).T, "a", (4, 3))         # not C-contiguous
    with pytest.raises(ValueError):
        B._host_i32(np.zeros((4, 2), np.int32), "a", (4, 3))           # shape
    with pytest.raises(ValueError):
        B._host_i32([[0, 0, 0]] * 4, "a", (4, 3))                       # not an array
    ro = np.zeros((4, 3), np.int32)
    ro.flags.writeable = False
    assert B._host_i32(ro, "a", (4, 3)) is ro
    with pytest.raises(ValueError):
        B._host_i32(ro, "a", (4, 3), writable=True)


def test_device_tensors_must_be_on_the_gpu():
    for t in (torch.zeros(4, dtype=torch.int32), np.zeros(4, np.int32), None):
        with pytest.raises(ValueError):
            B._dev_i32(t, "ids")
        with pytest.raises(ValueError):
            B._check_dev(t, torch.float32, "h")


def test_decode_host_refuses_bad_host_buffers_before_the_call():
    m = _detached_context()
    Bn, K = 4, 3
    ctx_ids = np.zeros(Bn, np.int32)
    drafts = np.zeros((Bn, K), np.int32)
    com = np.zeros((Bn, K + 1), np.int32)
    alen = np.zeros(Bn, np.int32)
    bad = [
        (ctx_ids.astype(np.int64), drafts, com, alen),          # 64-bit ids
        (ctx_ids, drafts.astype(np.int64), com, alen),
        (ctx_ids, np.zeros((K, Bn), np.int32).T, com, alen),    # strided drafts
        (ctx_ids, drafts, np.zeros((Bn, K), np.int32), alen),   # committed too small
        (ctx_ids, drafts, com, np.zeros(Bn + 1, np.int32)),
        (ctx_ids.reshape(Bn, 1), drafts, com, alen),            # 2-D context ids
    ]
    for args in bad:
        with pytest.raises(ValueError):
            m.decode_host(*args)


def test_device_calls_refuse_host_tensors_before_the_call():
    m = _detached_context()
    c = torch.zeros(4, dtype=torch.int32)
    d = torch.zeros((4, 3), dtype=torch.int32)
    tg = torch.zeros((4, 4), dtype=torch.int32)
    with pytest.raises(ValueError):
        m.step(c, d)
    with pytest.raises(ValueError):
        m.step(torch.zeros((4, 1), dtype=torch.int32), d)       # 2-D context ids
    with pytest.raises(ValueError):
        m.accept(d, tg)
    with pytest.raises(ValueError):
        m.layer(0, torch.zeros((4, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        m.layer(0, torch.zeros(64, dtype=torch.bfloat16))        # 1-D hidden state
    with pytest.raises(ValueError):
        m.draft_inputs(tg, c)
    with pytest.raises(ValueError):
        m.draft(torch.zeros((4, 64)), c, 3)
    with pytest.raises(ValueError):
        B.greedy_head_noalloc(torch.zeros((4, 64)), torch.zeros(64, dtype=torch.bfloat16),
                              torch.zeros((512, 64), dtype=torch.bfloat16), 1e-6)
