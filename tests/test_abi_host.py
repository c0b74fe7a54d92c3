"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and its host-only checks behave."""
import ctypes
import os
import re
import subprocess

import pytest

from moe_speculative_decoding_router_gb300 import binding as B
from moe_speculative_decoding_router_gb300 import build as build_mod
from moe_speculative_decoding_router_gb300 import synth as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_entry_points():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            names |= set(re.findall(r"^MOE_VERIFY_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M))
    return names


def test_library_builds_and_exports_every_declared_symbol():
    path = build_mod.build()
    names = declared_entry_points()
    assert {"moe_verify_init", "moe_verify_step", "moe_verify_accept"} <= names
    lib = ctypes.CDLL(path)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert names == exported, (names ^ exported)
    assert set(B.EXPORTED) == names


def test_library_links_no_torch_and_no_oracle():
    out = subprocess.run(["ldd", build_mod.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "oracle" not in out and "synth" not in out


def test_strerror_covers_every_status():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert B.strerror(code) and B.strerror(code) != "unknown status"
    assert B.strerror(-99) == "unknown status"


def test_check_config():
    assert B.check_config(S.FULL, 32, 3) == B.OK
    assert B.check_config(S.TINY, 4, 3) == B.OK
    assert B.check_config(S.FULL, 0, 3) == B.ERR_ARG
    assert B.check_config(S.FULL, 32, 16) == B.ERR_ARG
    assert B.check_config(S.FULL, 4096, 3) == B.ERR_UNSUPPORTED     # T = 16384 tokens
    import dataclasses
    assert B.check_config(dataclasses.replace(S.FULL, hidden=1000), 32, 3) == B.ERR_UNSUPPORTED
    assert B.check_config(dataclasses.replace(S.FULL, top_k=65), 32, 3) == B.ERR_ARG
    assert B.check_config(dataclasses.replace(S.FULL, rms_eps=0.0), 32, 3) == B.ERR_ARG
    assert B.device_bytes(S.FULL, 0, 3) == 0


_ARG, _UNS = "arg", "unsupported"


@pytest.mark.parametrize("field,value,want", [
    ("n_layers", 0, _ARG), ("n_layers", 257, _ARG), ("n_layers", 256, None),
    ("hidden", 63, _ARG), ("hidden", 8256, _ARG), ("hidden", 1000, _UNS), ("hidden", 64, None),
    ("n_experts", 0, _ARG), ("n_experts", 257, _ARG),
    ("top_k", 0, _ARG), ("top_k", 17, _ARG), ("top_k", 64, _ARG),   # more than n_experts = 8
    ("top_k", 8, None),                                               # every expert selected
    ("n_shared", -1, _ARG), ("n_shared", 9, _ARG), ("n_shared", 0, None),
    ("expert_inter", 0, _ARG), ("expert_inter", 8193, _ARG),
    ("shared_inter", 0, _ARG), ("shared_inter", 8193, _ARG),
    ("vocab", 1, _ARG), ("vocab", (1 << 30) + 1, _ARG), ("vocab", 2, None),
    ("rms_eps", 0.0, _ARG), ("rms_eps", float("nan"), _ARG), ("rms_eps", 1.0, _ARG),
    ("rms_eps", -1e-6, _ARG),
])
def test_check_config_refusals(field, value, want):
    """Each refusal rule of moe_verify_check_config at its boundary, on the
    tiny shape (8 experts, top-2, one shared expert, d = 64)."""
    import dataclasses
    cfg = dataclasses.replace(S.TINY, **{field: value})
    code = {None: B.OK, _ARG: B.ERR_ARG, _UNS: B.ERR_UNSUPPORTED}[want]
    assert B.check_config(cfg, 4, 3) == code


@pytest.mark.parametrize("max_batch,max_k,want", [
    (0, 3, B.ERR_ARG), (4, -1, B.ERR_ARG), (4, 16, B.ERR_ARG),
    (256, 15, B.OK),                   # 4096 verify tokens: the largest workspace
    (257, 15, B.ERR_UNSUPPORTED), (4097, 0, B.ERR_UNSUPPORTED), (4096, 0, B.OK),
])
def test_check_config_workspace_limits(max_batch, max_k, want):
    assert B.check_config(S.TINY, max_batch, max_k) == want


def test_device_bytes_is_weights_plus_workspace():
    n = B.device_bytes(S.FULL, 32, 3)
    per_expert = 3 * 896 * 1280 * 2
    weights = 12 * 66 * per_expert + 2 * 129280 * 1280 * 2
    assert weights < n < weights * 1.05


def test_null_arguments_fail_on_the_host():
    lib = B.load()
    assert lib.moe_verify_step(None, None, None, 1, 0, None, None, None) == B.ERR_ARG
    assert lib.moe_verify_accept(None, None, None, 1, 0, None, None, None) == B.ERR_ARG
    assert lib.moe_verify_layer(None, 0, None, 1, None, None, None) == B.ERR_ARG
    assert lib.moe_verify_sync_status(None) == B.ERR_ARG
    assert lib.moe_verify_check_config(None) == B.ERR_ARG
    h = ctypes.c_void_p()
    assert lib.moe_verify_init(None, None, None, ctypes.byref(h)) == B.ERR_ARG
    assert h.value is None
    lib.moe_verify_destroy(None)


def test_bounded_wait_check_rejects_limits_on_the_host():
    """Out-of-range limits are refused before any device work."""
    assert B.check_bounded_wait(10)[0] == B.ERR_ARG
    assert B.check_bounded_wait(2_000_000_000)[0] == B.ERR_ARG


def test_entry_points_refuse_null_and_out_of_range_arguments_on_the_host():
    """Argument errors come back as MOE_VERIFY_ERR_ARG before any device work
    (so they need no GPU): null contexts and pointers, sizes out of range."""
    L = B.load()
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails its checks first
    assert L.moe_verify_step(None, p, p, 1, 0, p, None, None) == B.ERR_ARG
    assert L.moe_verify_accept(None, p, p, 1, 0, p, p, None) == B.ERR_ARG
    assert L.moe_verify_layer(None, 0, p, 1, p, None, None) == B.ERR_ARG
    assert L.moe_verify_decode_host(None, p, p, 1, 0, p, p, None) == B.ERR_ARG
    assert L.moe_verify_draft(None, p, p, 1, 1, p, None, None) == B.ERR_ARG
    assert L.moe_verify_draft_inputs(None, p, p, 1, 0, p, p, None) == B.ERR_ARG
    assert L.moe_verify_greedy_head_noalloc(None, p, p, 1, 64, 512, 1e-6, p, None) == B.ERR_ARG
    assert L.moe_verify_check_bounded_wait(999, None, None) == B.ERR_ARG
    assert L.moe_verify_check_bounded_wait(1_000_000_001, None, None) == B.ERR_ARG
    assert L.moe_verify_sync_status(None) == B.ERR_ARG
