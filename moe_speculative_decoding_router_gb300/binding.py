"""Python binding of the C ABI in include/moe_verify.h.

Argument marshalling only: every step of the verify path runs in the CUDA
library.  Tensors are PyTorch CUDA tensors (device memory and streams are the
only things PyTorch provides here).  If the library cannot be loaded the
calls raise; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

from . import build as _build

_P = ctypes.c_void_p
_i32 = ctypes.c_int32

OK = 0
ERR_ARG = -1
ERR_CUDA = -2
ERR_OOM = -3
ERR_ID_RANGE = -4
ERR_TIMEOUT = -5
ERR_UNSUPPORTED = -6

EXPORTED = ("moe_verify_init", "moe_verify_step", "moe_verify_accept", "moe_verify_layer",
            "moe_verify_decode_host", "moe_verify_sync_status", "moe_verify_destroy",
            "moe_verify_strerror", "moe_verify_check_config", "moe_verify_device_bytes",
            "moe_verify_set_timing", "moe_verify_get_timing", "moe_verify_greedy_head_noalloc",
            "moe_verify_check_bounded_wait", "moe_verify_draft", "moe_verify_draft_inputs",
            "moe_verify_set_grid", "moe_verify_set_layer_kernel", "moe_verify_set_stamps",
            "moe_verify_init_attn", "moe_verify_step_attn", "moe_verify_kv_cache")


class Config(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("hidden", _i32), ("n_experts", _i32), ("top_k", _i32),
                ("n_shared", _i32), ("expert_inter", _i32), ("shared_inter", _i32),
                ("vocab", _i32), ("rms_eps", ctypes.c_float), ("max_batch", _i32),
                ("max_k", _i32)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("final_norm", _P), ("lm_head", _P), ("norm", _P),
                ("router", _P), ("router_bias", _P), ("w_gate", _P), ("w_up", _P),
                ("w_down", _P), ("s_gate", _P), ("s_up", _P), ("s_down", _P)]


class AttnConfig(ctypes.Structure):
    _fields_ = [("n_heads", _i32), ("max_pos", _i32), ("rope_theta", ctypes.c_float)]


class AttnWeights(ctypes.Structure):
    _fields_ = [("attn_norm", _P), ("w_q", _P), ("w_k", _P), ("w_v", _P), ("w_o", _P)]


class Probe(ctypes.Structure):
    _fields_ = [("topk_idx", _P), ("topk_w", _P), ("hidden", _P), ("logits", _P)]


class MoeVerifyError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


_lib = None


def load(build_if_missing: bool = True):
    """Load libmoe_verify.so (building it first if needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing; run the build first")
    L = ctypes.CDLL(path)
    L.moe_verify_init.restype = _i32
    L.moe_verify_init.argtypes = [_P, _P, _P, ctypes.POINTER(_P)]
    L.moe_verify_step.restype = _i32
    L.moe_verify_step.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_accept.restype = _i32
    L.moe_verify_accept.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_layer.restype = _i32
    L.moe_verify_layer.argtypes = [_P, _i32, _P, _i32, _P, _P, _P]
    L.moe_verify_decode_host.restype = _i32
    L.moe_verify_decode_host.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_sync_status.restype = _i32
    L.moe_verify_sync_status.argtypes = [_P]
    L.moe_verify_destroy.restype = None
    L.moe_verify_destroy.argtypes = [_P]
    L.moe_verify_strerror.restype = ctypes.c_char_p
    L.moe_verify_strerror.argtypes = [_i32]
    L.moe_verify_check_config.restype = _i32
    L.moe_verify_check_config.argtypes = [_P]
    L.moe_verify_device_bytes.restype = ctypes.c_uint64
    L.moe_verify_device_bytes.argtypes = [_P]
    L.moe_verify_set_timing.restype = _i32
    L.moe_verify_set_timing.argtypes = [_P, _i32]
    L.moe_verify_get_timing.restype = _i32
    L.moe_verify_get_timing.argtypes = [_P, _P, _P, _i32]
    L.moe_verify_draft.restype = _i32
    L.moe_verify_draft.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_draft_inputs.restype = _i32
    L.moe_verify_draft_inputs.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_check_bounded_wait.restype = _i32
    L.moe_verify_check_bounded_wait.argtypes = [ctypes.c_int64, _P, _P]
    L.moe_verify_set_grid.restype = _i32
    L.moe_verify_set_grid.argtypes = [_P, _i32]
    L.moe_verify_set_layer_kernel.restype = _i32
    L.moe_verify_set_layer_kernel.argtypes = [_P, _i32]
    L.moe_verify_set_stamps.restype = _i32
    L.moe_verify_set_stamps.argtypes = [_P, _P]
    L.moe_verify_init_attn.restype = _i32
    L.moe_verify_init_attn.argtypes = [_P, _P, _P, _P, _P, ctypes.POINTER(_P)]
    L.moe_verify_step_attn.restype = _i32
    L.moe_verify_step_attn.argtypes = [_P, _P, _P, _P, _i32, _i32, _P, _P, _P]
    L.moe_verify_kv_cache.restype = _i32
    L.moe_verify_kv_cache.argtypes = [_P, ctypes.POINTER(_P), ctypes.POINTER(_P)]
    L.moe_verify_greedy_head_noalloc.restype = _i32
    L.moe_verify_greedy_head_noalloc.argtypes = [_P, _P, _P, _i32, _i32, _i32, ctypes.c_float, _P,
                                                 _P]
    _lib = L
    return L


def strerror(code: int) -> str:
    return load().moe_verify_strerror(int(code)).decode()


def make_config(cfg, max_batch: int, max_k: int) -> Config:
    """Config struct from a shape record with the synthetic module's field names."""
    return Config(cfg.n_layers, cfg.hidden, cfg.n_experts, cfg.top_k, cfg.n_shared,
                  cfg.expert_inter, cfg.shared_inter, cfg.vocab, float(cfg.rms_eps),
                  int(max_batch), int(max_k))


def check_config(cfg, max_batch: int, max_k: int) -> int:
    c = make_config(cfg, max_batch, max_k)
    return int(load().moe_verify_check_config(ctypes.byref(c)))


def device_bytes(cfg, max_batch: int, max_k: int) -> int:
    c = make_config(cfg, max_batch, max_k)
    return int(load().moe_verify_device_bytes(ctypes.byref(c)))


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check_dev(t, dtype, name: str, shape=None):
    """t must be a contiguous CUDA tensor of `dtype` (and `shape`, where given):
    the library reads and writes it as a dense array from its data pointer."""
    import torch
    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype
            or not t.is_contiguous()):
        raise ValueError(f"{name}: a contiguous CUDA tensor of {dtype} is expected")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(shape)} expected, got {tuple(t.shape)}")
    return t


def _dev_i32(t, name: str = "ids", shape=None):
    import torch
    return _check_dev(t, torch.int32, name, shape)


def _host_i32(a, name: str, shape, writable: bool = False):
    """a must be a C-contiguous int32 numpy array of `shape`."""
    if (not isinstance(a, np.ndarray) or a.dtype != np.int32 or not a.flags["C_CONTIGUOUS"]
            or a.shape != tuple(shape)):
        raise ValueError(f"{name}: a C-contiguous int32 array of shape {tuple(shape)} is expected")
    if writable and not a.flags["WRITEABLE"]:
        raise ValueError(f"{name}: a writable array is expected")
    return a


def weights_to_device(w: Dict[str, np.ndarray], device="cuda") -> Dict[str, object]:
    """Upload the synthetic module's weight dict (bf16 bit patterns) to the GPU."""
    import torch
    out = {}
    for k, v in w.items():
        if v is None:
            continue
        if v.dtype == np.uint16:
            out[k] = torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).to(device).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(device)
    return out


class _DeviceArray:
    """A raw device allocation seen through the CUDA array interface (int16
    elements), for a tensor view that does not own the memory."""

    def __init__(self, ptr: int, shape):
        self.__cuda_array_interface__ = {"shape": tuple(int(x) for x in shape), "typestr": "<i2",
                                         "data": (int(ptr), False), "version": 3, "strides": None}


class MoeVerify:
    """One library context: weights and workspace on the current CUDA device.
    A shape record with n_heads > 0 makes a context of the stack with
    attention (moe_verify_init_attn), whose key/value cache holds max_pos
    positions per sequence slot."""

    def __init__(self, cfg, weights: Dict[str, object], max_batch: int, max_k: int, stream=None,
                 max_pos: int = 0):
        import torch
        self.lib = load()
        self.cfg = cfg
        self.max_batch, self.max_k = int(max_batch), int(max_k)
        self.attn = getattr(cfg, "n_heads", 0) > 0
        self.max_pos = int(max_pos)
        if self.attn and self.max_pos < 1:
            raise ValueError("max_pos: the positions held per sequence are needed with attention")
        self._c = make_config(cfg, max_batch, max_k)
        dw = {k: (v if isinstance(v, torch.Tensor) else None) for k, v in weights.items()}
        if any(v is None for v in dw.values()):
            dw = weights_to_device(weights)
        L = cfg.n_layers
        keep = []

        def per_layer(name):
            t = dw.get(name)
            if t is None:
                return None
            arr = (_P * L)(*[t[l].data_ptr() for l in range(L)])
            keep.append(arr)
            return ctypes.cast(arr, _P)

        W = Weights(_ptr(dw["embed"]), _ptr(dw["final_norm"]), _ptr(dw["lm_head"]),
                    per_layer("norm"), per_layer("router"), per_layer("router_bias"),
                    per_layer("w_gate"), per_layer("w_up"), per_layer("w_down"),
                    per_layer("s_gate"), per_layer("s_up"), per_layer("s_down"))
        h = _P()
        if self.attn:
            A = AttnConfig(int(cfg.n_heads), self.max_pos, float(cfg.rope_theta))
            AW = AttnWeights(per_layer("attn_norm"), per_layer("w_q"), per_layer("w_k"),
                             per_layer("w_v"), per_layer("w_o"))
            rc = self.lib.moe_verify_init_attn(ctypes.byref(self._c), ctypes.byref(W),
                                               ctypes.byref(A), ctypes.byref(AW),
                                               _stream_handle(stream), ctypes.byref(h))
            if rc != OK:
                raise MoeVerifyError(rc, "moe_verify_init_attn")
        else:
            rc = self.lib.moe_verify_init(ctypes.byref(self._c), ctypes.byref(W),
                                          _stream_handle(stream), ctypes.byref(h))
            if rc != OK:
                raise MoeVerifyError(rc, "moe_verify_init")
        self.handle = h
        del keep, dw

    # -- the calls -----------------------------------------------------------
    def step(self, context_ids, draft_ids, target_ids=None, probe: Optional[Probe] = None,
             stream=None):
        import torch
        if getattr(context_ids, "ndim", 0) != 1:
            raise ValueError("context_ids: a 1-D tensor [B] is expected")
        context_ids = _dev_i32(context_ids, "context_ids")
        B = context_ids.shape[0]
        K = 0 if draft_ids is None else draft_ids.shape[1]
        if K > 0:
            _dev_i32(draft_ids, "draft_ids", (B, K))
        if target_ids is None:
            target_ids = torch.empty((B, K + 1), dtype=torch.int32, device=context_ids.device)
        _dev_i32(target_ids, "target_ids", (B, K + 1))
        rc = self.lib.moe_verify_step(self.handle, _ptr(context_ids),
                                      _ptr(draft_ids) if K > 0 else None, B, K, _ptr(target_ids),
                                      ctypes.byref(probe) if probe is not None else None,
                                      _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_step")
        return target_ids

    def step_attn(self, context_ids, draft_ids, positions, target_ids=None,
                  probe: Optional[Probe] = None, stream=None):
        """moe_verify_step_attn: positions [B] int32 (device) is each
        sequence's position of its context token."""
        import torch
        if getattr(context_ids, "ndim", 0) != 1:
            raise ValueError("context_ids: a 1-D tensor [B] is expected")
        context_ids = _dev_i32(context_ids, "context_ids")
        B = context_ids.shape[0]
        K = 0 if draft_ids is None else draft_ids.shape[1]
        if K > 0:
            _dev_i32(draft_ids, "draft_ids", (B, K))
        _dev_i32(positions, "positions", (B,))
        if target_ids is None:
            target_ids = torch.empty((B, K + 1), dtype=torch.int32, device=context_ids.device)
        _dev_i32(target_ids, "target_ids", (B, K + 1))
        rc = self.lib.moe_verify_step_attn(self.handle, _ptr(context_ids),
                                           _ptr(draft_ids) if K > 0 else None, _ptr(positions), B,
                                           K, _ptr(target_ids),
                                           ctypes.byref(probe) if probe is not None else None,
                                           _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_step_attn")
        return target_ids

    def kv_cache(self):
        """moe_verify_kv_cache: (keys, values) as bf16 tensor views [L,
        max_batch, n_heads, max_pos, head width] of the context's cache (valid
        while the context lives)."""
        import torch
        kp, vp = _P(), _P()
        rc = self.lib.moe_verify_kv_cache(self.handle, ctypes.byref(kp), ctypes.byref(vp))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_kv_cache")
        c = self.cfg
        shape = (c.n_layers, self.max_batch, c.n_heads, self.max_pos, c.hidden // c.n_heads)
        k = torch.as_tensor(_DeviceArray(kp.value, shape), device="cuda").view(torch.bfloat16)
        v = torch.as_tensor(_DeviceArray(vp.value, shape), device="cuda").view(torch.bfloat16)
        return k, v

    def accept(self, draft_ids, target_ids, committed=None, accept_len=None, stream=None):
        import torch
        if getattr(target_ids, "ndim", 0) != 2:
            raise ValueError("target_ids: a 2-D tensor [B, K + 1] is expected")
        B, K1 = target_ids.shape
        K = K1 - 1
        _dev_i32(target_ids, "target_ids")
        if K > 0 and draft_ids is not None:
            _dev_i32(draft_ids, "draft_ids", (B, K))
        if committed is None:
            committed = torch.empty((B, K1), dtype=torch.int32, device=target_ids.device)
        if accept_len is None:
            accept_len = torch.empty((B,), dtype=torch.int32, device=target_ids.device)
        _dev_i32(committed, "committed", (B, K1))
        _dev_i32(accept_len, "accept_len", (B,))
        rc = self.lib.moe_verify_accept(self.handle, _ptr(draft_ids) if K > 0 else None,
                                        _ptr(target_ids), B, K, _ptr(committed), _ptr(accept_len),
                                        _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_accept")
        return committed, accept_len

    def layer(self, layer: int, h_in, h_out=None, probe: Optional[Probe] = None, stream=None):
        import torch
        if getattr(h_in, "ndim", 0) != 2:
            raise ValueError("h_in: a 2-D tensor [T, hidden] is expected")
        T = h_in.shape[0]
        _check_dev(h_in, torch.bfloat16, "h_in", (T, self.cfg.hidden))
        if h_out is None:
            h_out = torch.empty_like(h_in)
        _check_dev(h_out, torch.bfloat16, "h_out", (T, self.cfg.hidden))
        rc = self.lib.moe_verify_layer(self.handle, int(layer), _ptr(h_in), T, _ptr(h_out),
                                       ctypes.byref(probe) if probe is not None else None,
                                       _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_layer")
        return h_out

    def draft_inputs(self, committed, accept_len, h_out=None, t_out=None, stream=None):
        """moe_verify_draft_inputs: (h [B, d] fp32, t [B] int32) of each
        sequence's last accepted position after step + accept."""
        import torch
        if getattr(committed, "ndim", 0) != 2:
            raise ValueError("committed: a 2-D tensor [B, K + 1] is expected")
        B, K1 = committed.shape
        _dev_i32(committed, "committed")
        _dev_i32(accept_len, "accept_len", (B,))
        if h_out is None:
            h_out = torch.empty((B, self.cfg.hidden), dtype=torch.float32, device=committed.device)
        if t_out is None:
            t_out = torch.empty((B,), dtype=torch.int32, device=committed.device)
        _check_dev(h_out, torch.float32, "h_out", (B, self.cfg.hidden))
        _dev_i32(t_out, "t_out", (B,))
        rc = self.lib.moe_verify_draft_inputs(self.handle, _ptr(committed), _ptr(accept_len), B,
                                              K1 - 1, _ptr(h_out), _ptr(t_out),
                                              _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_draft_inputs")
        return h_out, t_out

    def draft(self, h_prev, t_prev, K: int, drafts=None, hidden: bool = False, stream=None):
        """moe_verify_draft on this (one-layer draft-block) context: drafts
        [B, K] int32, and the state after each step [K, B, d] when hidden."""
        import torch
        if getattr(t_prev, "ndim", 0) != 1:
            raise ValueError("t_prev: a 1-D tensor [B] is expected")
        B = t_prev.shape[0]
        _dev_i32(t_prev, "t_prev")
        _check_dev(h_prev, torch.float32, "h_prev", (B, self.cfg.hidden))
        if drafts is None:
            drafts = torch.empty((B, K), dtype=torch.int32, device=t_prev.device)
        _dev_i32(drafts, "drafts", (B, K))
        hid = (torch.empty((K, B, self.cfg.hidden), dtype=torch.float32, device=t_prev.device)
               if hidden else None)
        rc = self.lib.moe_verify_draft(self.handle, _ptr(h_prev), _ptr(t_prev), B, int(K),
                                       _ptr(drafts), _ptr(hid), _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_draft")
        return (drafts, hid) if hidden else drafts

    def decode_host(self, context_ids: np.ndarray, draft_ids: Optional[np.ndarray],
                    committed: np.ndarray, accept_len: np.ndarray, stream=None):
        """Host buffers in and out (any C-contiguous int32 arrays: the library
        stages them through its own pinned buffer)."""
        if getattr(context_ids, "ndim", 0) != 1:
            raise ValueError("context_ids: a 1-D array [B] is expected")
        B = context_ids.shape[0]
        K = 0 if draft_ids is None else draft_ids.shape[1]
        _host_i32(context_ids, "context_ids", (B,))
        if K > 0:
            _host_i32(draft_ids, "draft_ids", (B, K))
        _host_i32(committed, "committed", (B, K + 1), writable=True)
        _host_i32(accept_len, "accept_len", (B,), writable=True)
        rc = self.lib.moe_verify_decode_host(
            self.handle, context_ids.ctypes.data,
            draft_ids.ctypes.data if K > 0 else None, B, K, committed.ctypes.data,
            accept_len.ctypes.data, _stream_handle(stream))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_decode_host")
        return committed, accept_len

    def sync_status(self) -> int:
        return int(self.lib.moe_verify_sync_status(self.handle))

    def set_timing(self, enable: bool):
        rc = self.lib.moe_verify_set_timing(self.handle, 1 if enable else 0)
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_set_timing")

    def set_grid(self, ctas: int):
        """moe_verify_set_grid: CTAs of the persistent kernels (0: one per SM)."""
        rc = self.lib.moe_verify_set_grid(self.handle, int(ctas))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_set_grid")

    def set_layer_kernel(self, max_tokens: int):
        """moe_verify_set_layer_kernel: steps of at most max_tokens verify
        tokens run one launch per layer (0: off)."""
        rc = self.lib.moe_verify_set_layer_kernel(self.handle, int(max_tokens))
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_set_layer_kernel")

    def set_stamps(self, stamps):
        """moe_verify_set_stamps: a device int64 tensor [2L + 1, 4] ([6L + 1, 4]
        with attention; viewed as uint64 by the library), or None to stop."""
        import torch
        if stamps is not None:
            per = 6 if self.attn else 2
            _check_dev(stamps, torch.int64, "stamps", (per * self.cfg.n_layers + 1, 4))
        rc = self.lib.moe_verify_set_stamps(self.handle, _ptr(stamps) if stamps is not None else None)
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_set_stamps")

    def get_timing(self, reset: bool = True):
        ms = (ctypes.c_double * 4)()
        n = (ctypes.c_int64 * 4)()
        rc = self.lib.moe_verify_get_timing(self.handle, ms, n, 1 if reset else 0)
        if rc != OK:
            raise MoeVerifyError(rc, "moe_verify_get_timing")
        return list(ms), list(n)

    def close(self):
        if getattr(self, "handle", None):
            self.lib.moe_verify_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass


def greedy_head_noalloc(h, final_norm, lm_head, rms_eps: float, target_ids=None, stream=None):
    """moe_verify_greedy_head_noalloc: argmax of lm_head . bf16(RMSNorm(h) * g)
    for each row of h [T, d] (fp32 CUDA tensor), with no device allocation
    inside the call (target_ids may be passed preallocated)."""
    import torch
    if getattr(h, "ndim", 0) != 2 or getattr(lm_head, "ndim", 0) != 2:
        raise ValueError("h [T, d] and lm_head [V, d] are expected")
    T, d = h.shape
    V = lm_head.shape[0]
    _check_dev(h, torch.float32, "h")
    _check_dev(final_norm, torch.bfloat16, "final_norm", (d,))
    _check_dev(lm_head, torch.bfloat16, "lm_head", (V, d))
    if target_ids is None:
        target_ids = torch.empty((T,), dtype=torch.int32, device=h.device)
    _dev_i32(target_ids, "target_ids", (T,))
    rc = load().moe_verify_greedy_head_noalloc(_ptr(h), _ptr(final_norm), _ptr(lm_head), T, d, V,
                                                float(rms_eps), _ptr(target_ids),
                                                _stream_handle(stream))
    if rc != OK:
        raise MoeVerifyError(rc, "moe_verify_greedy_head_noalloc")
    return target_ids


def check_bounded_wait(limit_ns: int, stream=None):
    """moe_verify_check_bounded_wait: returns (status, elapsed ns of the two
    waits that nothing completes)."""
    el = ctypes.c_int64(0)
    # an out-of-range limit is refused on the host, before any stream is needed
    ok_limit = 1000 <= int(limit_ns) <= 1_000_000_000
    rc = load().moe_verify_check_bounded_wait(int(limit_ns), ctypes.byref(el),
                                              _stream_handle(stream) if ok_limit else None)
    return int(rc), int(el.value)


def make_probe(L: int, T: int, cfg, topk: bool = True, hidden: bool = True, logits: bool = False,
               device="cuda"):
    """Allocate probe buffers; returns (Probe struct, dict of tensors).  For
    a shape record with attention the hidden states are [2L + 1, T, d]
    (entering each block's attention and its MoE part, and after the last)."""
    import torch
    t = {}
    rows = 2 * L + 1 if getattr(cfg, "n_heads", 0) > 0 else L + 1
    if topk:
        t["topk_idx"] = torch.full((L, T, cfg.top_k), -7, dtype=torch.int32, device=device)
        t["topk_w"] = torch.zeros((L, T, cfg.top_k), dtype=torch.float32, device=device)
    if hidden:
        t["hidden"] = torch.zeros((rows, T, cfg.hidden), dtype=torch.float32, device=device)
    if logits:
        t["logits"] = torch.zeros((T, cfg.vocab), dtype=torch.float32, device=device)
    p = Probe(_ptr(t.get("topk_idx")), _ptr(t.get("topk_w")), _ptr(t.get("hidden")),
              _ptr(t.get("logits")))
    return p, t


__all__ = ["load", "MoeVerify", "MoeVerifyError", "Probe", "AttnConfig", "AttnWeights",
           "make_probe", "check_config",
           "device_bytes", "strerror", "weights_to_device", "check_bounded_wait", "EXPORTED"]
