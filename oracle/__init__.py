"""Python binding of the fp64 oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it.  The product library never imports it.

The binding only marshals arguments; every step of the arithmetic runs in the
C file, single-threaded per call.  ``Oracle.targets`` may run several calls at
once on separate threads (ctypes releases the GIL), one token per call, which
changes no arithmetic.
"""
from __future__ import annotations

import concurrent.futures as _fut
import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_i32 = ctypes.c_int32


class OracleConfig(ctypes.Structure):
    _fields_ = [("n_layers", _i32), ("hidden", _i32), ("n_experts", _i32), ("top_k", _i32),
                ("n_shared", _i32), ("expert_inter", _i32), ("shared_inter", _i32),
                ("vocab", _i32), ("rms_eps", ctypes.c_double)]


class OracleAttnWeights(ctypes.Structure):
    _fields_ = [("n_heads", _i32), ("rope_theta", ctypes.c_double), ("attn_norm", _P), ("w_q", _P),
                ("w_k", _P), ("w_v", _P), ("w_o", _P)]


class OracleWeights(ctypes.Structure):
    _fields_ = [("embed", _P), ("final_norm", _P), ("lm_head", _P), ("norm", _P), ("router", _P),
                ("router_bias", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P),
                ("s_gate", _P), ("s_up", _P), ("s_down", _P)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc: -O2, no fast-math, no FMA contraction."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                                   "-shared", "-fvisibility=hidden", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        # A test that plants a mistake in a copy of the C source points
        # MOE_ORACLE_LIB at the compiled copy.
        path = os.environ.get("MOE_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        L.oracle_bf16_value.restype = ctypes.c_double
        L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_rmsnorm_bf16.restype = None
        L.oracle_rmsnorm_bf16.argtypes = [_P, _P, _i32, ctypes.c_double, _P]
        L.oracle_router.restype = None
        L.oracle_router.argtypes = [_P, _P, _P, _i32, _i32, _i32, _P, _P, _P, _P, _P]
        L.oracle_swiglu_expert.restype = None
        L.oracle_swiglu_expert.argtypes = [_P, _P, _P, _P, _i32, _i32, _P]
        L.oracle_layer.restype = None
        L.oracle_layer.argtypes = [_P, _P, _i32, _P, _P, _P, _P, _P, _P]
        L.oracle_forward_token.restype = _i32
        L.oracle_forward_token.argtypes = [_P, _P, _i32] + [_P] * 8
        L.oracle_verify_step.restype = _i32
        L.oracle_verify_step.argtypes = [_P, _P, _P, _P, _i32, _i32, _P]
        L.oracle_accept.restype = _i32
        L.oracle_accept.argtypes = [_P, _P, _i32, _i32, _i32, _P, _P]
        L.oracle_head.restype = _i32
        L.oracle_head.argtypes = [_P, _P, _P, _P, _P]
        L.oracle_layer_bf16.restype = None
        L.oracle_layer_bf16.argtypes = [_P, _P, _i32, _P, _P, _P, _P, _P, _P, _P]
        L.oracle_draft.restype = _i32
        L.oracle_draft.argtypes = [_P, _P, _P, _i32, _i32, _P, _P, _P]
        L.oracle_rope.restype = None
        L.oracle_rope.argtypes = [_P, _i32, _i32, ctypes.c_double]
        L.oracle_attn_block.restype = None
        L.oracle_attn_block.argtypes = [_P, _P, _i32, _P, _i32, _P, _P, _P]
        L.oracle_forward_seq.restype = _i32
        L.oracle_forward_seq.argtypes = [_P, _P, _P, _P, _i32, _P, _P, _P, _P, _P, _P]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def round_bf16(x: float) -> int:
    return int(lib().oracle_round_bf16(float(x)))


def bf16_value(b: int) -> float:
    return float(lib().oracle_bf16_value(int(b) & 0xFFFF))


def rmsnorm_bf16(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.uint16)
    out = np.empty(h.shape[-1], dtype=np.uint16)
    lib().oracle_rmsnorm_bf16(_ptr(h), _ptr(g), h.shape[-1], float(eps), _ptr(out))
    return out


def router(xhat: np.ndarray, W: np.ndarray, k: int, bias: Optional[np.ndarray] = None):
    """Returns (z, p, sel, p_sel, gap) for one token."""
    xhat = np.ascontiguousarray(xhat, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    E, d = W.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    z, p = np.empty(E), np.empty(E)
    sel, psel, gap = np.empty(k, np.int32), np.empty(k), np.empty(1)
    lib().oracle_router(_ptr(xhat), _ptr(W), _ptr(b), E, d, k, _ptr(z), _ptr(p), _ptr(sel),
                        _ptr(psel), _ptr(gap))
    return z, p, sel, psel, float(gap[0])


def swiglu_expert(xhat, Wg, Wu, Wd) -> np.ndarray:
    xhat = np.ascontiguousarray(xhat, dtype=np.uint16)
    Wg, Wu, Wd = (np.ascontiguousarray(a, dtype=np.uint16) for a in (Wg, Wu, Wd))
    I, d = Wg.shape
    y = np.empty(d)
    lib().oracle_swiglu_expert(_ptr(xhat), _ptr(Wg), _ptr(Wu), _ptr(Wd), d, I, _ptr(y))
    return y


def rope(x: np.ndarray, pos: int, theta: float = 10000.0) -> np.ndarray:
    """The rotary embedding of one head vector (a rotated copy)."""
    y = np.array(x, dtype=np.float64, copy=True)
    lib().oracle_rope(_ptr(y), y.shape[0], int(pos), float(theta))
    return y


def accept(drafts: np.ndarray, targets: np.ndarray, V: int):
    """Returns (committed [B,K+1], accept_len [B], bad_rows)."""
    drafts = np.ascontiguousarray(drafts, dtype=np.int32)
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    B, K1 = targets.shape
    K = K1 - 1
    if drafts.size == 0:
        drafts = np.zeros((B, max(K, 0)), dtype=np.int32)
    committed = np.empty((B, K1), dtype=np.int32)
    alen = np.empty(B, dtype=np.int32)
    bad = lib().oracle_accept(_ptr(drafts), _ptr(targets), B, K, V, _ptr(committed), _ptr(alen))
    return committed, alen, int(bad)


class Oracle:
    """The fp64 target stack over a set of bf16 weights (numpy uint16 arrays,
    the dict layout of the synthetic-input module)."""

    def __init__(self, cfg, weights: Dict[str, np.ndarray]):
        self.cfg = cfg
        self.w = {k: (np.ascontiguousarray(v) if v is not None else None) for k, v in weights.items()}
        L = cfg.n_layers
        self._c = OracleConfig(cfg.n_layers, cfg.hidden, cfg.n_experts, cfg.top_k, cfg.n_shared,
                               cfg.expert_inter, cfg.shared_inter, cfg.vocab, float(cfg.rms_eps))
        self._keep = []

        def per_layer(name):
            a = self.w.get(name)
            if a is None:
                return None
            arr = (ctypes.c_void_p * L)(*[a[l].ctypes.data for l in range(L)])
            self._keep.append(arr)
            return ctypes.cast(arr, ctypes.c_void_p)

        self._w = OracleWeights(
            _ptr(self.w.get("embed")), _ptr(self.w["final_norm"]), _ptr(self.w.get("lm_head")),
            per_layer("norm"), per_layer("router"), per_layer("router_bias"), per_layer("w_gate"),
            per_layer("w_up"), per_layer("w_down"), per_layer("s_gate"), per_layer("s_up"),
            per_layer("s_down"))
        self._cp = ctypes.byref(self._c)
        self._wp = ctypes.byref(self._w)
        self._ap = None
        if getattr(cfg, "n_heads", 0) > 0:
            self._a = OracleAttnWeights(cfg.n_heads, float(cfg.rope_theta), per_layer("attn_norm"),
                                        per_layer("w_q"), per_layer("w_k"), per_layer("w_v"),
                                        per_layer("w_o"))
            self._ap = ctypes.byref(self._a)

    # -- one token through the whole stack --------------------------------
    def forward_token(self, x: int, force_sel: Optional[np.ndarray] = None, logits: bool = False):
        c = self.cfg
        L, k, d = c.n_layers, c.top_k, c.hidden
        sel = np.empty((L, k), np.int32)
        wts = np.empty((L, k))
        gaps = np.empty(L)
        hid = np.empty((L + 1, d))
        xf = np.empty(d, np.uint16)
        lg = np.empty(c.vocab) if logits else None
        lgap = np.empty(1)
        fs = None if force_sel is None else np.ascontiguousarray(force_sel, dtype=np.int32)
        y = lib().oracle_forward_token(self._cp, self._wp, int(x), _ptr(fs), _ptr(sel), _ptr(wts),
                                       _ptr(gaps), _ptr(hid), _ptr(xf), _ptr(lg), _ptr(lgap))
        return dict(target=int(y), sel=sel, w=wts, route_gap=gaps, hidden=hid, xhat_f=xf,
                    logits=lg, logit_gap=float(lgap[0]))

    def target(self, x: int) -> int:
        return int(lib().oracle_forward_token(self._cp, self._wp, int(x), *([None] * 8)))

    def targets(self, ids: Sequence[int], nthreads: int = 1, **kw):
        """forward_token over many ids; nthreads > 1 runs one call per thread."""
        ids = [int(i) for i in ids]
        if nthreads <= 1 or len(ids) <= 1:
            return [self.forward_token(i, **kw) for i in ids]
        with _fut.ThreadPoolExecutor(max_workers=nthreads) as ex:
            return list(ex.map(lambda i: self.forward_token(i, **kw), ids))

    def g_table(self, ids: Sequence[int], nthreads: int = 1) -> np.ndarray:
        ids = [int(i) for i in ids]
        if nthreads <= 1:
            return np.array([self.target(i) for i in ids], dtype=np.int32)
        with _fut.ThreadPoolExecutor(max_workers=nthreads) as ex:
            return np.array(list(ex.map(self.target, ids)), dtype=np.int32)

    # -- the verify step and the layer entry point -------------------------
    def verify_step(self, context_ids: np.ndarray, drafts: np.ndarray) -> np.ndarray:
        context_ids = np.ascontiguousarray(context_ids, dtype=np.int32)
        B = context_ids.shape[0]
        drafts = np.ascontiguousarray(drafts, dtype=np.int32).reshape(B, -1)
        K = drafts.shape[1]
        out = np.empty((B, K + 1), dtype=np.int32)
        rc = lib().oracle_verify_step(self._cp, self._wp, _ptr(context_ids), _ptr(drafts), B, K,
                                      _ptr(out))
        if rc != 0:
            raise ValueError("verify token id outside [0, V)")
        return out

    def layer(self, l: int, h: np.ndarray, force_sel: Optional[np.ndarray] = None):
        """One block on fp64 hidden h [d] (a copy is updated).  Returns
        (h_new, sel, w, gap, xhat)."""
        c = self.cfg
        hh = np.array(h, dtype=np.float64, copy=True)
        sel = np.empty(c.top_k, np.int32)
        wts = np.empty(c.top_k)
        gap = np.empty(1)
        xh = np.empty(c.hidden, np.uint16)
        fs = None if force_sel is None else np.ascontiguousarray(force_sel, dtype=np.int32)
        lib().oracle_layer(self._cp, self._wp, int(l), _ptr(hh), _ptr(fs), _ptr(sel), _ptr(wts),
                           _ptr(gap), _ptr(xh))
        return hh, sel, wts, float(gap[0]), xh

    def head(self, h: np.ndarray, logits: bool = False):
        """Final RMSNorm + lm_head argmax on residual h [d].  Returns
        (target, top-2 logit gap, logits or None)."""
        hh = np.ascontiguousarray(h, dtype=np.float64)
        lg = np.empty(self.cfg.vocab) if logits else None
        gap = np.empty(1)
        y = lib().oracle_head(self._cp, self._wp, _ptr(hh), _ptr(lg), _ptr(gap))
        return int(y), float(gap[0]), lg

    def draft(self, h_prev: np.ndarray, t_prev: int, K: int):
        """The FastMTP draft head with this instance as the draft block (one
        layer, one expert): K recursive steps from residual h_prev [d] and
        token t_prev.  Returns (drafts [K], hidden after each step [K, d],
        top-2 logit gaps [K])."""
        d = self.cfg.hidden
        hp = np.ascontiguousarray(h_prev, dtype=np.float64)
        drafts = np.empty(K, np.int32)
        hid = np.empty((K, d))
        gaps = np.empty(K)
        rc = lib().oracle_draft(self._cp, self._wp, _ptr(hp), int(t_prev), int(K), _ptr(drafts),
                                _ptr(hid), _ptr(gaps))
        if rc != 0:
            raise ValueError("draft token id outside [0, V)")
        return drafts, hid, gaps

    # -- the stack with attention (configs with n_heads > 0) ---------------
    def attn_block(self, l: int, h: np.ndarray, pos: int, kc: np.ndarray, vc: np.ndarray):
        """Attention sub-block of layer l on one token at position pos:
        returns (h after it, o before W_o).  kc, vc: [pos + 1, d] float64
        caches of this layer (rows < pos read, row pos written in place)."""
        hh = np.array(h, dtype=np.float64, copy=True)
        assert kc.dtype == np.float64 and kc.flags["C_CONTIGUOUS"] and kc.shape[0] >= pos + 1
        assert vc.dtype == np.float64 and vc.flags["C_CONTIGUOUS"] and vc.shape[0] >= pos + 1
        o = np.empty(self.cfg.hidden)
        lib().oracle_attn_block(self._cp, self._ap, int(l), _ptr(hh), int(pos), _ptr(kc), _ptr(vc),
                                _ptr(o))
        return hh, o

    def forward_seq(self, ids: Sequence[int], caches: bool = False, hidden: bool = False):
        """A whole sequence with attention: greedy target after every prefix,
        top-2 logit gaps, selection gaps [n, L]; with caches=True the key and
        value caches [L, n, d], with hidden=True the residual stream entering
        each block and after the last, [n, L+1, d]."""
        c = self.cfg
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        n, L, d = ids.shape[0], c.n_layers, c.hidden
        tg = np.empty(n, np.int32)
        lg = np.empty(n)
        rg = np.empty((n, L))
        kc = np.empty((L, n, d)) if caches else None
        vc = np.empty((L, n, d)) if caches else None
        hid = np.empty((n, L + 1, d)) if hidden else None
        rc = lib().oracle_forward_seq(self._cp, self._wp, self._ap, _ptr(ids), n, _ptr(tg), _ptr(lg),
                                      _ptr(rg), _ptr(kc), _ptr(vc), _ptr(hid))
        if rc != 0:
            raise ValueError("token id outside [0, V)")
        return dict(targets=tg, logit_gaps=lg, route_gaps=rg, kcache=kc, vcache=vc, hidden=hid)

    def layer_bf16(self, l: int, h_in: np.ndarray, force_sel: Optional[np.ndarray] = None):
        """The bf16-in/bf16-out block on one token.  Returns
        (h_out_bf16, h_out_f64, sel, w, gap)."""
        c = self.cfg
        h_in = np.ascontiguousarray(h_in, dtype=np.uint16)
        out = np.empty(c.hidden, np.uint16)
        f64 = np.empty(c.hidden)
        sel = np.empty(c.top_k, np.int32)
        wts = np.empty(c.top_k)
        gap = np.empty(1)
        fs = None if force_sel is None else np.ascontiguousarray(force_sel, dtype=np.int32)
        lib().oracle_layer_bf16(self._cp, self._wp, int(l), _ptr(h_in), _ptr(fs), _ptr(out),
                                _ptr(f64), _ptr(sel), _ptr(wts), _ptr(gap))
        return out, f64, sel, wts, float(gap[0])
