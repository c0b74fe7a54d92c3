"""Seeded synthetic inputs for the MoE greedy-verify step.

This module builds the workload's inputs and nothing else: weights, start ids,
draft coins and draft ids.  It contains none of the verify step's arithmetic.
The CUDA library and the fp64 oracle both take its arrays as plain inputs.

The element generator is host C (``synth.c``): a counter-based splitmix64
stream per (seed, tensor id) with Box-Muller normals, rounded once to bf16.

Model shapes follow the DeepSeek-3B-MoE decoder that "Jina AI Releases
jina-ocr-v1, a 3.4B MoE Document Parser With Built-In Speculative Decoding"
describes in its architecture paragraph (12 layers, 64 routed experts, two
shared experts, top-6 routing).  Hidden 1280, expert intermediate 896 and
vocabulary 129,280 are the workload's stated sizes.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Seeds of the workload's streams.
SEED_WEIGHTS = 0
SEED_START_IDS = 1
SEED_DRAFTS = 2
SEED_HIDDEN = 3
SEED_DRAFT_HEAD = 4

# Stream ids inside a seed.  Weights: embed, then per layer eight tensors,
# then the final norm and the lm_head.
TID_EMBED = 0
_LAYER_TENSORS = ("norm", "router", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down")
TID_DRAFT_COIN = 1
TID_DRAFT_ID = 2


def tid_layer(layer: int, name: str) -> int:
    return 1 + 8 * layer + _LAYER_TENSORS.index(name)


def tid_final_norm(n_layers: int) -> int:
    return 1 + 8 * n_layers


def tid_lm_head(n_layers: int) -> int:
    return 2 + 8 * n_layers


_ATTN_TENSORS = ("w_q", "w_k", "w_v", "w_o")


def tid_attn(n_layers: int, layer: int, name: str) -> int:
    """Attention projections come after every tensor of the attention-free
    stack, so adding attention changes none of those streams."""
    return 3 + 8 * n_layers + 4 * layer + _ATTN_TENSORS.index(name)


def build(force: bool = False) -> str:
    """Compile the generator with gcc (in-tree, host only)."""
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-fvisibility=hidden",
                                   "-o", tmp, _SRC, "-lm", "-lpthread"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
        L.synth_draw.restype = u64
        L.synth_draw.argtypes = [u64, u64, u64]
        L.synth_normal.restype = ctypes.c_double
        L.synth_normal.argtypes = [u64, u64, u64]
        L.synth_bf16_of.restype = ctypes.c_uint16
        L.synth_bf16_of.argtypes = [ctypes.c_double]
        L.synth_normal_bf16.restype = None
        L.synth_normal_bf16.argtypes = [ctypes.c_void_p, i64, u64, u64, u64, ctypes.c_double, i32]
        L.synth_ids.restype = None
        L.synth_ids.argtypes = [ctypes.c_void_p, i64, u64, u64, u64, i64, i32]
        L.synth_uniform.restype = None
        L.synth_uniform.argtypes = [ctypes.c_void_p, i64, u64, u64, u64, i32]
        L.synth_uniform_at.restype = None
        L.synth_uniform_at.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, u64, u64]
        L.synth_ids_at.restype = None
        L.synth_ids_at.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64, u64, u64, i64]
        _lib = L
    return _lib


def _threads(n: Optional[int]) -> int:
    if n:
        return n
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def normal_bf16(shape, seed: int, tid: int, sigma: float, first: int = 0,
                nthreads: Optional[int] = None) -> np.ndarray:
    """bf16 bit patterns (uint16) of sigma * N(0,1), element i drawn at first+i."""
    out = np.empty(shape, dtype=np.uint16)
    lib().synth_normal_bf16(out.ctypes.data, out.size, seed, tid, first, float(sigma), _threads(nthreads))
    return out


def uniform_ids(n: int, seed: int, tid: int, modulus: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().synth_ids(out.ctypes.data, n, seed, tid, first, modulus, 1)
    return out


def uniform01(n: int, seed: int, tid: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_uniform(out.ctypes.data, n, seed, tid, first, 1)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Shape of the MoE decoder stack on the verify path."""
    n_layers: int
    hidden: int
    n_experts: int
    top_k: int
    n_shared: int
    expert_inter: int
    shared_inter: int
    vocab: int
    rms_eps: float = 1e-6
    sigma: float = 0.02          # std of every weight tensor
    zipf_s: float = 0.0          # >0: per-expert router bias -s*ln(e+1)
    name: str = ""
    n_heads: int = 0             # >0: attention before each MoE block (head width hidden/n_heads)
    rope_theta: float = 10000.0


# Tiny correctness instance: 2 layers, d=64, 8 experts of 32, top-2, one
# shared expert, vocab 512, weights N(0, 0.05).
TINY = ModelConfig(2, 64, 8, 2, 1, 32, 32, 512, sigma=0.05, name="tiny")
# One layer at the decoder's expert layout (hidden 1280, 64 x 896, top-6, 2
# shared).  The single-block entry point never touches the vocabulary, so a
# small one keeps the embedding and lm_head cheap.
LAYER = ModelConfig(1, 1280, 64, 6, 2, 896, 896, 512, name="layer")
# The full 12-layer stack with the 129,280-token vocabulary.
FULL = ModelConfig(12, 1280, 64, 6, 2, 896, 896, 129280, name="full")
# The full stack with Zipf(s=1.2)-skewed routing.
FULL_ZIPF = dataclasses.replace(FULL, zipf_s=1.2, name="full_zipf")
# The stacks with attention before each MoE block (the pages give no shape:
# heads of width 128 at hidden 1280, 16 at hidden 64).
TINY_ATTN = dataclasses.replace(TINY, n_heads=4, name="tiny_attn")
FULL_ATTN = dataclasses.replace(FULL, n_heads=10, name="full_attn")


# FastMTP draft heads: one dense block applied recursively, sharing the
# verifier's embedding, final norm and lm_head.  The pages give no width:
# 4 x hidden.  A SwiGLU FFN is a sum over its intermediate units, so the dense
# block of width 4d is held as 8 always-on (shared, weight 1) experts of width
# d/2 -- its units in 8 groups -- which gives the GPU eight times as many
# down-projection items; the stack's one routed expert has zero weights.
DRAFT_TINY = ModelConfig(1, 64, 1, 1, 8, 32, 32, 512, sigma=0.05, name="draft_tiny")
DRAFT = ModelConfig(1, 1280, 1, 1, 8, 64, 640, 129280, name="draft")


def make_draft_weights(cfg: ModelConfig, target: Dict[str, np.ndarray],
                       seed: int = SEED_DRAFT_HEAD,
                       nthreads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """The draft block's own weights (seeded stream SEED_DRAFT_HEAD; the
    routed expert zeroed, so the block is the dense FFN of the shared
    experts) plus the verifier's embedding, final norm and lm_head (the same
    arrays)."""
    w = make_weights(cfg, seed=seed, with_embed=False, with_lm_head=False, nthreads=nthreads)
    for k in ("w_gate", "w_up", "w_down"):
        w[k] = np.zeros_like(w[k])
    for k in ("embed", "final_norm", "lm_head"):
        w[k] = target[k]
    return w


def router_bias(cfg: ModelConfig) -> Optional[np.ndarray]:
    """Zipf routing skew: b_e = -s * ln(e + 1), the same in every layer, fp32."""
    if cfg.zipf_s <= 0:
        return None
    e = np.arange(cfg.n_experts, dtype=np.float64)
    b = (-cfg.zipf_s * np.log(e + 1.0)).astype(np.float32)
    return np.ascontiguousarray(np.broadcast_to(b, (cfg.n_layers, cfg.n_experts)))


def make_weights(cfg: ModelConfig, seed: int = SEED_WEIGHTS, with_embed: bool = True,
                 with_lm_head: bool = True, nthreads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All weights of the stack as bf16 bit patterns (uint16), PyTorch Linear layout [out, in].

    RMSNorm gains are unit (the workload fixes them at 1).
    """
    L, d, E, I, S, Is, V = (cfg.n_layers, cfg.hidden, cfg.n_experts, cfg.expert_inter,
                            cfg.n_shared, cfg.shared_inter, cfg.vocab)
    sg = cfg.sigma
    one = np.uint16(0x3F80)
    w: Dict[str, np.ndarray] = {}
    w["norm"] = np.full((L, d), one, dtype=np.uint16)
    w["final_norm"] = np.full((d,), one, dtype=np.uint16)
    for name, shape in (("router", (E, d)), ("w_gate", (E, I, d)), ("w_up", (E, I, d)),
                        ("w_down", (E, d, I)), ("s_gate", (S, Is, d)), ("s_up", (S, Is, d)),
                        ("s_down", (S, d, Is))):
        arr = np.empty((L,) + shape, dtype=np.uint16)
        for l in range(L):
            lib().synth_normal_bf16(arr[l].ctypes.data, arr[l].size, seed, tid_layer(l, name), 0,
                                    float(sg), _threads(nthreads))
        w[name] = arr
    if with_embed:
        w["embed"] = normal_bf16((V, d), seed, TID_EMBED, sg, nthreads=nthreads)
    if with_lm_head:
        w["lm_head"] = normal_bf16((V, d), seed, tid_lm_head(L), sg, nthreads=nthreads)
    rb = router_bias(cfg)
    if rb is not None:
        w["router_bias"] = rb
    if cfg.n_heads > 0:
        w.update(make_attn_weights(cfg, seed, nthreads))
    return w


def make_attn_weights(cfg: ModelConfig, seed: int = SEED_WEIGHTS,
                      nthreads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """The attention tensors alone (the entries that make_weights adds for a
    shape record with n_heads > 0): unit attn_norm gains and W_q, W_k, W_v,
    W_o [L, d, d]."""
    L, d = cfg.n_layers, cfg.hidden
    w: Dict[str, np.ndarray] = {"attn_norm": np.full((L, d), np.uint16(0x3F80), dtype=np.uint16)}
    for name in _ATTN_TENSORS:
        arr = np.empty((L, d, d), dtype=np.uint16)
        for l in range(L):
            lib().synth_normal_bf16(arr[l].ctypes.data, arr[l].size, seed, tid_attn(L, l, name),
                                    0, float(cfg.sigma), _threads(nthreads))
        w[name] = arr
    return w


def hidden_input(T: int, d: int, seed: int = SEED_HIDDEN) -> np.ndarray:
    """Input hidden states for the single-layer case: N(0,1) rounded to bf16, [T, d]."""
    return normal_bf16((T, d), seed, 0, 1.0)


def start_ids(B: int, V: int, seed: int = SEED_START_IDS, first: int = 0) -> np.ndarray:
    """Uniform start ids in [0, V)."""
    return uniform_ids(B, seed, 0, V, first)


class DraftSource:
    """Synthetic stand-in for the draft head.

    Draft i of a sequence whose greedy continuation is G[c+1], G[c+2], ... is
    G[c+1+i] with probability p, else a uniform id in [0, V).  The coin and the
    replacement id are counter-indexed by (sequence, step, i), so both are
    reproducible and independent per position.
    """

    def __init__(self, p: float, V: int, K: int, seed: int = SEED_DRAFTS):
        self.p, self.V, self.K, self.seed = float(p), int(V), int(K), seed
        self._lanes = np.arange(self.K, dtype=np.uint64).reshape(1, -1)

    def _index(self, seq: int, step: int, i: int) -> int:
        return ((seq * 1_000_003 + step) * 16 + i)

    def drafts_batch(self, seqs, steps, truth) -> np.ndarray:
        """drafts() for many sequences at once: seqs [B], steps [B],
        truth [B, K] -> [B, K] int32 (the same draws, counter-indexed)."""
        seqs = np.asarray(seqs, dtype=np.uint64)
        steps = np.asarray(steps, dtype=np.uint64)
        truth = np.asarray(truth).reshape(len(seqs), self.K)
        # counter index of (sequence, step, i), as in _index
        j = ((seqs * np.uint64(1_000_003) + steps) * np.uint64(16))[:, None] + self._lanes
        u = np.empty(j.shape, dtype=np.float64)
        ids = np.empty(j.shape, dtype=np.int32)
        L = lib()
        L.synth_uniform_at(u.ctypes.data, j.ctypes.data, j.size, self.seed, TID_DRAFT_COIN)
        L.synth_ids_at(ids.ctypes.data, j.ctypes.data, j.size, self.seed, TID_DRAFT_ID, self.V)
        hit = u < self.p
        ids[hit] = truth[hit]
        return ids

    def drafts(self, seq: int, step: int, truth) -> np.ndarray:
        """truth[i] = the greedy token the i-th draft should predict."""
        out = np.empty(self.K, dtype=np.int32)
        for i in range(self.K):
            j = self._index(seq, step, i)
            u = float(uniform01(1, self.seed, TID_DRAFT_COIN, j)[0])
            if u < self.p:
                out[i] = int(truth[i])
            else:
                out[i] = int(uniform_ids(1, self.seed, TID_DRAFT_ID, self.V, j)[0])
        return out
