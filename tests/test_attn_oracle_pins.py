"""Pins of the oracle's attention (the decoder's attention sub-block, the
stack with attention): rotary embedding identities, special cases with a
closed form, a two-position worked example, causality, and the reduction to
the attention-free stack.  CPU only.

Reading (the pages give no attention shape): pre-norm multi-head attention
before each MoE block, heads of width d / n_heads, rotary embedding pairing
dims i and i + hd/2 at angle pos * theta^(-2i/hd), causal over positions
0 .. pos, scores scaled by 1/sqrt(hd), bf16 rounding of the normalised
input, of k (after the rotation) and v, and of the output before W_o.
"""
import math

import numpy as np
import pytest

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S

torch = pytest.importorskip("torch")


def bf16(x):
    """Round to the nearest bf16 (torch's conversion, independent of the oracle)."""
    return float(torch.tensor(float(x), dtype=torch.float64).to(torch.bfloat16).to(torch.float64))


# ------------------------------------------------------------------- rope

def test_rope_identity_at_position_zero():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    assert np.array_equal(O.rope(x, 0), x)


@pytest.mark.parametrize("hd,pos,i", [(4, 1, 0), (4, 1, 1), (128, 7, 0), (128, 7, 5), (128, 300, 63),
                                      (16, 3, 7)])
def test_rope_turns_each_pair_by_its_angle(hd, pos, i):
    """Unit vector e_i (i < hd/2) goes to cos(a) e_i + sin(a) e_{i+hd/2}, and
    e_{i+hd/2} to -sin(a) e_i + cos(a) e_{i+hd/2}, a = pos * theta^(-2i/hd)."""
    theta = 10000.0
    a = pos * theta ** (-2.0 * i / hd)
    e = np.zeros(hd)
    e[i] = 1.0
    r = O.rope(e, pos, theta)
    want = np.zeros(hd)
    want[i], want[i + hd // 2] = math.cos(a), math.sin(a)
    assert np.allclose(r, want, atol=1e-12, rtol=0)
    e = np.zeros(hd)
    e[i + hd // 2] = 1.0
    r = O.rope(e, pos, theta)
    want = np.zeros(hd)
    want[i], want[i + hd // 2] = -math.sin(a), math.cos(a)
    assert np.allclose(r, want, atol=1e-12, rtol=0)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for p, j, s in [(5, 2, 11), (40, 40, 3), (9, 0, 1000)]:
        a = O.rope(q, p) @ O.rope(k, j)
        b = O.rope(q, p + s) @ O.rope(k, j + s)
        assert abs(a - b) <= 1e-9 * (abs(a) + 1.0)
        assert abs(np.linalg.norm(O.rope(q, p)) - np.linalg.norm(q)) <= 1e-12 * np.linalg.norm(q)


# --------------------------------------------------- one attention block

class _Cfg:
    """A custom shape for hand-built weights."""
    def __init__(self, d, heads, theta, eps):
        self.n_layers, self.hidden, self.n_experts, self.top_k = 1, d, 1, 1
        self.n_shared, self.expert_inter, self.shared_inter, self.vocab = 0, 1, 1, 2
        self.rms_eps, self.n_heads, self.rope_theta = eps, heads, theta


def _one(x):
    return O.round_bf16(x)


def _block_weights(d, wq, wk, wv, wo, gain=None):
    w = {"embed": np.zeros((2, d), np.uint16), "final_norm": np.full((d,), 0x3F80, np.uint16),
         "lm_head": np.zeros((2, d), np.uint16), "norm": np.full((1, d), 0x3F80, np.uint16),
         "router": np.zeros((1, 1, d), np.uint16), "w_gate": np.zeros((1, 1, 1, d), np.uint16),
         "w_up": np.zeros((1, 1, 1, d), np.uint16), "w_down": np.zeros((1, 1, d, 1), np.uint16),
         "attn_norm": (np.full((1, d), 0x3F80, np.uint16) if gain is None
                       else np.array([[_one(g) for g in gain]], np.uint16))}
    for name, m in (("w_q", wq), ("w_k", wk), ("w_v", wv), ("w_o", wo)):
        w[name] = np.array([[[_one(v) for v in row] for row in m]], np.uint16)
    return w


def _turn(v, i, j, ang):
    """Rotate the pair (v[i], v[j]) by ang (a plane rotation written out)."""
    x, y = v[i], v[j]
    v[i], v[j] = x * math.cos(ang) - y * math.sin(ang), x * math.sin(ang) + y * math.cos(ang)


def test_worked_example_two_positions():
    """d = 8, two heads of width 4, theta = 4 (pair (0,2) of a head turns by pos
    rad, pair (1,3) by pos / 2 rad), W_q = W_k = I, W_v and W_o cyclic shifts
    (v_m = xhat_{m+1}, y_m = o_{m+1}).  The residual rows have unit RMS, so
    xhat = h exactly.
      position 0: h = (0,2,0,0 | 2,0,0,0); one key, so o = v = shift(h) and
        h += shift(o);
      position 1: h = (0,0,0,2 | 0,0,2,0); q = k = rope(h, 1) per head (head 0
        turns its (1,3) pair by 0.5, head 1 its (0,2) pair by 1.0), the cache
        keeps bf16(k); scores q.k_j / 2; o = bf16(w0 v0 + w1 v1) per head;
        h += shift(o)."""
    d = 8
    I = np.eye(d)
    shift = np.zeros((d, d))
    for m in range(d):
        shift[m, (m + 1) % d] = 1.0
    cfg = _Cfg(d, 2, 4.0, 1e-30)
    orc = O.Oracle(cfg, _block_weights(d, I, I, shift, shift))
    kc, vc = np.zeros((2, d)), np.zeros((2, d))

    def sh(v):  # y_m = v_{m+1}
        return [v[(m + 1) % d] for m in range(d)]

    h0 = [0.0, 2.0, 0.0, 0.0, 2.0, 0.0, 0.0, 0.0]
    v0 = sh(h0)
    h0n, o0 = orc.attn_block(0, np.array(h0), 0, kc, vc)
    assert np.array_equal(kc[0], np.array(h0)) and np.array_equal(vc[0], np.array(v0))
    assert np.array_equal(o0, np.array(v0))
    assert np.array_equal(h0n, np.array(h0) + np.array(sh(v0)))

    h1 = [0.0, 0.0, 0.0, 2.0, 0.0, 0.0, 2.0, 0.0]
    q = list(h1)
    for hh in range(2):
        _turn(q, 4 * hh + 0, 4 * hh + 2, 1.0)   # pair (0, 2) at angle pos * 4^0
        _turn(q, 4 * hh + 1, 4 * hh + 3, 0.5)   # pair (1, 3) at angle pos * 4^(-1/2)
    k1 = [bf16(x) for x in q]
    v1 = sh(h1)
    o = []
    for hh in range(2):
        sl = slice(4 * hh, 4 * hh + 4)
        s0 = sum(a * b for a, b in zip(q[sl], h0[sl])) / 2.0
        s1 = sum(a * b for a, b in zip(q[sl], k1[sl])) / 2.0
        m = max(s0, s1)
        e0, e1 = math.exp(s0 - m), math.exp(s1 - m)
        o += [bf16((e0 * a + e1 * b) / (e0 + e1)) for a, b in zip(v0[sl], v1[sl])]
    h1n, o1 = orc.attn_block(0, np.array(h1), 1, kc, vc)
    assert np.array_equal(kc[1], np.array(k1))
    assert np.array_equal(vc[1], np.array(v1))
    assert np.array_equal(o1, np.array(o))
    assert np.array_equal(h1n, np.array(h1) + np.array(sh(o)))


def test_sequence_runs_attention_then_the_moe_block():
    """The whole-sequence forward is, at every position and layer, the
    attention sub-block then the MoE block applied to the residual entering
    the layer (with the caches of the earlier positions)."""
    cfg = S.TINY_ATTN
    orc = O.Oracle(cfg, S.make_weights(cfg))
    ids = S.uniform_ids(5, 21, 0, cfg.vocab)
    r = orc.forward_seq(ids, caches=True, hidden=True)
    H = r["hidden"]
    for p in range(len(ids)):
        for l in range(cfg.n_layers):
            kc = np.ascontiguousarray(r["kcache"][l, :p + 1].copy())
            vc = np.ascontiguousarray(r["vcache"][l, :p + 1].copy())
            h, _ = orc.attn_block(l, H[p, l], p, kc, vc)
            h, _, _, _, _ = orc.layer(l, h)
            assert np.array_equal(h, H[p, l + 1]), (p, l)
        assert orc.head(H[p, cfg.n_layers])[0] == r["targets"][p]


def test_position_zero_ignores_queries_and_keys():
    """With one key the softmax weight is 1: the output at position 0 is
    W_o bf16(v) whatever W_q and W_k are."""
    cfg = S.TINY_ATTN
    w = S.make_weights(cfg)
    rng = np.random.default_rng(3)
    h = rng.standard_normal(cfg.hidden)
    outs = []
    for seed in (0, 1):
        w2 = dict(w)
        if seed:
            w2["w_q"] = S.normal_bf16(w["w_q"].shape, 77, 1, 0.3)
            w2["w_k"] = S.normal_bf16(w["w_k"].shape, 77, 2, 0.3)
        orc = O.Oracle(cfg, w2)
        kc, vc = np.zeros((1, cfg.hidden)), np.zeros((1, cfg.hidden))
        outs.append(orc.attn_block(0, h, 0, kc, vc)[0])
    assert np.array_equal(outs[0], outs[1])
    # at a later position the queries do matter
    outs = []
    for seed in (0, 1):
        w2 = dict(w)
        if seed:
            w2["w_q"] = S.normal_bf16(w["w_q"].shape, 77, 1, 0.3)
        orc = O.Oracle(cfg, w2)
        kc, vc = np.zeros((3, cfg.hidden)), np.zeros((3, cfg.hidden))
        for p in range(3):
            hp, _ = orc.attn_block(0, rng.standard_normal(cfg.hidden) if p < 2 else h, p, kc, vc)
        outs.append(hp)
    assert not np.array_equal(outs[0], outs[1])


def test_zero_queries_average_the_values():
    """W_q = 0 makes every score 0: the weights are uniform over positions
    0 .. pos, so o = bf16(mean of the cached v rows 0 .. pos), and every
    cached k and v is a bf16 number."""
    cfg = S.TINY_ATTN
    w = dict(S.make_weights(cfg))
    w["w_q"] = np.zeros_like(w["w_q"])
    orc = O.Oracle(cfg, w)
    rng = np.random.default_rng(4)
    n, d = 6, cfg.hidden
    kc, vc = np.zeros((n, d)), np.zeros((n, d))
    for p in range(n):
        _, o = orc.attn_block(1, rng.standard_normal(d), p, kc, vc)
        want = np.array([O.bf16_value(O.round_bf16(x)) for x in vc[:p + 1].mean(axis=0)])
        assert np.array_equal(o, want), p
    for arr in (kc, vc):
        assert all(O.bf16_value(O.round_bf16(x)) == x for x in arr.reshape(-1))


# ------------------------------------------------------- whole sequences

def test_causal_targets_do_not_see_later_tokens():
    cfg = S.TINY_ATTN
    orc = O.Oracle(cfg, S.make_weights(cfg))
    ids = S.uniform_ids(10, 5, 0, cfg.vocab)
    base = orc.forward_seq(ids)["targets"]
    for cut in (1, 4, 9):
        ids2 = ids.copy()
        ids2[cut:] = S.uniform_ids(10 - cut, 6 + cut, 0, cfg.vocab)
        t2 = orc.forward_seq(ids2)["targets"]
        assert np.array_equal(t2[:cut], base[:cut]), cut


def test_silent_attention_reduces_to_the_attention_free_stack():
    """W_o = 0: attention adds nothing, and every position's target is the
    attention-free stack's target of its own token."""
    w = dict(S.make_weights(S.TINY_ATTN))
    w["w_o"] = np.zeros_like(w["w_o"])
    orc = O.Oracle(S.TINY_ATTN, w)
    plain = O.Oracle(S.TINY, {k: v for k, v in w.items()
                              if k not in ("attn_norm", "w_q", "w_k", "w_v", "w_o")})
    ids = S.uniform_ids(12, 8, 0, 512)
    got = orc.forward_seq(ids)["targets"]
    assert np.array_equal(got, [plain.target(int(x)) for x in ids])


def test_speculative_decoding_with_attention_is_lossless():
    """Verify steps over the sequence model (targets of the prefix plus K
    drafts), with always-right, random and adversarial drafts, commit exactly
    the greedy continuation."""
    cfg = S.TINY_ATTN
    orc = O.Oracle(cfg, S.make_weights(cfg))
    rng = np.random.default_rng(9)
    prompt = [int(x) for x in S.uniform_ids(3, 12, 0, cfg.vocab)]
    n_new = 10
    greedy = list(prompt)
    while len(greedy) < len(prompt) + n_new:
        greedy.append(int(orc.forward_seq(greedy)["targets"][-1]))
    for policy in ("right", "random", "adversarial"):
        for K in (1, 3):
            seq = list(prompt)
            while len(seq) < len(prompt) + n_new:
                truth = greedy[len(seq):len(seq) + K]
                truth += [0] * (K - len(truth))
                if policy == "right":
                    drafts = truth
                elif policy == "random":
                    drafts = [int(x) for x in rng.integers(0, cfg.vocab, K)]
                else:
                    drafts = [(t + 1) % cfg.vocab for t in truth]
                tg = orc.forward_seq(seq + drafts)["targets"][len(seq) - 1:]
                com, alen, _ = O.accept(np.array([drafts]), np.array([tg]), cfg.vocab)
                seq += [int(x) for x in com[0, :alen[0] + 1]]
            n = len(prompt) + n_new
            assert seq[:n] == greedy[:n], (policy, K)
