"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes one piece with a hand-worked value, a closed form, a library
routine on a special case, a brute-force search or an invariant, chosen so
that a dropped term, a wrong sign, a wrong index or a transposed operand in
the oracle fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle as O
from moe_speculative_decoding_router_gb300 import synth as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# ------------------------------------------------------------ bf16 rounding

_BF16_SORTED = None


def _bf16_table():
    """All finite bf16 values with their bit patterns, sorted by value."""
    global _BF16_SORTED
    if _BF16_SORTED is None:
        bits = np.arange(0, 1 << 16, dtype=np.uint32)
        with np.errstate(invalid="ignore"):
            vals = (bits << 16).view(np.float32).astype(np.float64)
        keep = np.isfinite(vals) & (bits != 0x8000)   # one zero in the table
        order = np.argsort(vals[keep], kind="stable")
        _BF16_SORTED = (vals[keep][order], bits[keep][order].astype(np.uint16))
    return _BF16_SORTED


def nearest_bf16_bruteforce(x: float) -> int:
    """Search the sorted table of every finite bf16 value for the nearest one;
    ties go to the pattern with an even last bit; beyond the largest finite
    value by half an ulp or more the result is infinity."""
    vals, bits = _bf16_table()
    big = float(vals[-1])
    half_ulp_top = 2.0 ** (127 - 8)
    if x >= big + half_ulp_top:
        return 0x7F80
    if x <= -big - half_ulp_top:
        return 0xFF80
    if x == 0.0:
        return 0x8000 if math.copysign(1.0, x) < 0 else 0x0000
    i = int(np.searchsorted(vals, x))
    cands = [j for j in (i - 1, i) if 0 <= j < len(vals)]
    best = min(cands, key=lambda j: (abs(vals[j] - x), int(bits[j]) & 1))
    if vals[best] == 0.0 and x < 0:
        return 0x8000                         # a negative value that rounds to zero keeps its sign
    return int(bits[best])


def test_bf16_hand_worked_cases():
    for line in _rows("bf16_rne_cases.txt"):
        xs, hexbits = line.split()[:2]
        x = float.fromhex(xs)
        assert O.round_bf16(x) == int(hexbits, 16), (xs, hex(O.round_bf16(x)))


def test_bf16_special_values():
    assert O.round_bf16(float("inf")) == 0x7F80
    assert O.round_bf16(float("-inf")) == 0xFF80
    assert (O.round_bf16(float("nan")) & 0x7FFF) > 0x7F80


def test_bf16_matches_bruteforce_nearest():
    rng = np.random.default_rng(7)
    mags = 2.0 ** rng.uniform(-140, 128, size=4000)
    xs = mags * rng.choice([-1.0, 1.0], size=mags.size)
    # exact midpoints between neighbouring bf16 values exercise the tie rule
    vals, _ = _bf16_table()
    idx = rng.integers(1, len(vals) - 1, size=500)
    mids = (vals[idx] + vals[idx + 1]) / 2
    for x in list(xs) + list(mids):
        assert O.round_bf16(float(x)) == nearest_bf16_bruteforce(float(x)), x


def test_bf16_matches_torch_on_float32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    xs = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([O.round_bf16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_is_sign_times_gain():
    d = 64
    one = np.full(d, 0x3F80, np.uint16)
    for c, want in ((3.0, 0x3F80), (-2.0, 0xBF80), (0.25, 0x3F80)):
        out = O.rmsnorm_bf16(np.full(d, c), one, 1e-6)
        assert np.all(out == want)


def test_rmsnorm_gain_is_elementwise_and_in_order():
    d = 64
    gains = np.array([S.lib().synth_bf16_of(v) for v in
                      np.linspace(-2, 2, d)], dtype=np.uint16)
    out = O.rmsnorm_bf16(np.ones(d), gains, 1e-6)
    # h = 1 everywhere: rms = 1, so xhat_i = bf16(g_i * (1 - 5e-7)) = g_i
    assert np.array_equal(out, gains)


def test_rmsnorm_one_hot():
    d = 64
    h = np.zeros(d)
    h[5] = -1.0
    out = O.rmsnorm_bf16(h, np.full(d, 0x3F80, np.uint16), 1e-6)
    # mean(h^2) = 1/64: xhat_5 = -1/sqrt(1/64 + 1e-6) = -7.99974..., nearest bf16 -8
    assert out[5] == 0xC100
    assert np.all(np.delete(out, 5) == 0)


def test_rmsnorm_eps_matters_at_small_scale():
    d = 64
    out = O.rmsnorm_bf16(np.full(d, 1e-4), np.full(d, 0x3F80, np.uint16), 1e-6)
    closed = 1e-4 / math.sqrt(1e-8 + 1e-6)  # 0.0995037...
    assert np.all(out == nearest_bf16_bruteforce(closed))
    zero = O.rmsnorm_bf16(np.zeros(d), np.full(d, 0x3F80, np.uint16), 1e-6)
    assert np.all(zero == 0)


# ------------------------------------------------------------------ router

def _bf(v):
    b = nearest_bf16_bruteforce(float(v))
    assert O.bf16_value(b) == float(v), "test value must be bf16-exact"
    return b


def test_router_all_equal_logits():
    E, d, k = 8, 64, 3
    xhat = np.zeros(d, np.uint16)
    W = S.normal_bf16((E, d), 99, 0, 0.05)
    z, p, sel, psel, gap = O.router(xhat, W, k)
    assert np.all(z == 0) and np.all(p == 1.0 / E)
    assert list(sel) == [0, 1, 2]          # ties: lower expert index first
    assert gap == 0.0


def test_router_constructed_logits_and_tie_order():
    E, d, k = 8, 64, 3
    v = [0.5, -1.0, 2.0, 2.0, 0.25, 1.5, -3.0, 0.0]
    xhat = np.zeros(d, np.uint16)
    xhat[3] = _bf(1.0)
    W = S.normal_bf16((E, d), 98, 0, 0.05)
    W[:, 3] = [_bf(x) for x in v]
    z, p, sel, psel, gap = O.router(xhat, W, k)
    assert np.array_equal(z, v)
    assert list(sel) == [2, 3, 5]
    np.testing.assert_allclose(p, scipy.special.softmax(v), rtol=1e-14, atol=0)
    np.testing.assert_allclose(psel, scipy.special.softmax(v)[[2, 3, 5]], rtol=1e-14)
    assert psel.sum() < 1.0                 # not renormalised over the selected experts
    assert gap == 1.5 - 0.5


def test_router_bias_only():
    E, d, k = 8, 64, 2
    b = np.array([0.1, 0.7, -0.2, 0.7, 0.3, 0.0, 0.69, -1.0], np.float32)
    z, p, sel, psel, gap = O.router(np.zeros(d, np.uint16), S.normal_bf16((E, d), 97, 0, 0.05), k, b)
    assert list(sel) == [1, 3]
    np.testing.assert_allclose(z, b.astype(np.float64), rtol=0, atol=0)
    assert gap == pytest.approx(0.7 - 0.69, abs=1e-7)


def test_router_matches_bruteforce_sort_random():
    rng = np.random.default_rng(3)
    E, d, k = 16, 64, 4
    for trial in range(200):
        xhat = S.normal_bf16((d,), 50 + trial, 1, 1.0)
        W = S.normal_bf16((E, d), 50 + trial, 2, 0.05)
        if trial % 3 == 0:  # exact ties between experts
            W[rng.integers(E)] = W[rng.integers(E)]
            W[rng.integers(E)] = W[rng.integers(E)]
        bias = rng.standard_normal(E).astype(np.float32) * 0.1 if trial % 2 else None
        z, p, sel, psel, gap = O.router(xhat, W, k, bias)
        zz = S.bf16_bits_to_f32(W).astype(np.float64) @ S.bf16_bits_to_f32(xhat).astype(np.float64)
        if bias is not None:
            zz = zz + bias.astype(np.float64)
        np.testing.assert_allclose(z, zz, rtol=1e-12, atol=1e-12)
        order = sorted(range(E), key=lambda e: (-z[e], e))
        assert list(sel) == order[:k]
        np.testing.assert_allclose(p, scipy.special.softmax(z), rtol=1e-12)
        assert gap == z[order[k - 1]] - z[order[k]]


# --------------------------------------------------------- SwiGLU expert

def _silu_table():
    return {float(a): float(b) for a, b in (r.split() for r in _rows("silu_values.txt"))}


def test_expert_zero_input_gives_zero():
    d, I = 64, 32
    y = O.swiglu_expert(np.zeros(d, np.uint16), S.normal_bf16((I, d), 1, 1, 0.05),
                        S.normal_bf16((I, d), 1, 2, 0.05), S.normal_bf16((d, I), 1, 3, 0.05))
    assert np.all(y == 0)


def test_expert_one_hot_structure():
    """Each weight row has a single nonzero, at a column chosen so that any
    transposition or index slip reads a different value; d != I."""
    d, I = 64, 32
    silu = _silu_table()
    xs = [0.0, 1.0, -1.0, 2.0, 0.5, -2.0]
    xhat = np.zeros(d, np.uint16)
    for i in range(d):
        xhat[i] = _bf(xs[i % len(xs)])
    Wg = np.zeros((I, d), np.uint16)
    Wu = np.zeros((I, d), np.uint16)
    Wd = np.zeros((d, I), np.uint16)
    gate_col = [(7 * j + 3) % d for j in range(I)]
    up_col = [(5 * j + 11) % d for j in range(I)]
    up_scale = [1.0, -0.5, 2.0, 0.25]
    for j in range(I):
        Wg[j, gate_col[j]] = _bf(1.0)
        Wu[j, up_col[j]] = _bf(up_scale[j % 4])
    down_src = [(3 * m + 1) % I for m in range(d)]
    down_scale = [1.0, 2.0, -1.0, 0.5, 4.0]
    for m in range(d):
        Wd[m, down_src[m]] = _bf(down_scale[m % 5])
    y = O.swiglu_expert(xhat, Wg, Wu, Wd)
    a = []
    for j in range(I):
        g = xs[gate_col[j] % len(xs)]
        u = xs[up_col[j] % len(xs)] * up_scale[j % 4]
        a.append(O.bf16_value(nearest_bf16_bruteforce(silu[g] * u)))
    want = np.array([a[down_src[m]] * down_scale[m % 5] for m in range(d)])
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=0)
    assert np.any(want != 0)


def test_expert_dense_matches_numpy_matmul():
    """Random weights: the dot products agree with numpy's matmul in fp64, and
    a is rounded to bf16 between the two projections."""
    d, I = 64, 32
    xhat = S.normal_bf16((d,), 5, 0, 1.0)
    Wg, Wu = S.normal_bf16((I, d), 5, 1, 0.05), S.normal_bf16((I, d), 5, 2, 0.05)
    Wd = S.normal_bf16((d, I), 5, 3, 0.05)
    f = lambda b: S.bf16_bits_to_f32(b).astype(np.float64)
    g, u = f(Wg) @ f(xhat), f(Wu) @ f(xhat)
    pre = scipy.special.expit(g) * g * u
    a = np.array([O.bf16_value(nearest_bf16_bruteforce(v)) for v in pre])
    np.testing.assert_allclose(O.swiglu_expert(xhat, Wg, Wu, Wd), f(Wd) @ a, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------- layer

def _tiny_zero_down():
    w = S.make_weights(S.TINY)
    for k in ("w_down", "s_down"):
        w[k] = np.zeros_like(w[k])
    return w


def test_layer_with_zero_down_projections_is_identity():
    cfg = S.TINY
    o = O.Oracle(cfg, _tiny_zero_down())
    h = S.bf16_bits_to_f32(S.normal_bf16((cfg.hidden,), 11, 0, 0.3)).astype(np.float64)
    hn, sel, wts, gap, xh = o.layer(0, h)
    assert np.array_equal(hn, h)
    out, f64, *_ = o.layer_bf16(1, S.normal_bf16((cfg.hidden,), 12, 0, 1.0))
    assert np.array_equal(out, S.normal_bf16((cfg.hidden,), 12, 0, 1.0))


def _identifiable_layer():
    """A tiny layer whose routed expert e writes into coordinate e only, and
    whose shared expert writes into coordinate 20, each with a known SwiGLU
    value.  The input h = e_63 normalises to xhat = 8 * e_63 exactly."""
    cfg = S.TINY
    d, E, I, k = cfg.hidden, cfg.n_experts, cfg.expert_inter, cfg.top_k
    w = S.make_weights(cfg)
    L = cfg.n_layers
    z_vals = [0.5, -1.0, 2.0, 1.0, 0.25, 1.5, -0.5, 0.0]
    for l in range(L):
        w["router"][l][:] = 0
        w["router"][l][:, 63] = [_bf(v / 8) for v in z_vals]
        for e in range(E):
            w["w_gate"][l][e][:] = 0
            w["w_up"][l][e][:] = 0
            w["w_down"][l][e][:] = 0
            w["w_gate"][l][e][0, 63] = _bf(0.125)   # g_0 = 1
            w["w_up"][l][e][0, 63] = _bf(0.25)      # u_0 = 2
            w["w_down"][l][e][e, 0] = _bf(e + 1)    # y_e = a_0 (e+1) at coordinate e
        w["s_gate"][l][0][:] = 0
        w["s_up"][l][0][:] = 0
        w["s_down"][l][0][:] = 0
        w["s_gate"][l][0][1, 63] = _bf(0.25)        # g_1 = 2
        w["s_up"][l][0][1, 63] = _bf(-0.125)        # u_1 = -1
        w["s_down"][l][0][20, 1] = _bf(4.0)
    return cfg, w, z_vals


def test_layer_combine_weights_shared_and_residual():
    cfg, w, z_vals = _identifiable_layer()
    silu = _silu_table()
    o = O.Oracle(cfg, w)
    h = np.zeros(cfg.hidden)
    h[63] = 1.0
    hn, sel, wts, gap, xh = o.layer(0, h)
    assert xh[63] == 0x4100 and np.count_nonzero(xh) == 1     # xhat = 8 e_63
    assert list(sel) == [2, 5]
    p = scipy.special.softmax(z_vals)
    a_routed = O.bf16_value(nearest_bf16_bruteforce(silu[1.0] * 2.0))   # 1.4609375
    a_shared = O.bf16_value(nearest_bf16_bruteforce(silu[2.0] * -1.0))
    want = h.copy()
    want[2] += p[2] * a_routed * 3
    want[5] += p[5] * a_routed * 6
    want[20] += a_shared * 4.0
    np.testing.assert_allclose(hn, want, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(wts, p[[2, 5]], rtol=1e-14)
    assert gap == 1.5 - 1.0
    # forcing another set moves the contributions and keeps the softmax weights
    hf, self_, wf, _, _ = o.layer(0, h, force_sel=np.array([3, 0], np.int32))
    want_f = h.copy()
    want_f[3] += p[3] * a_routed * 4
    want_f[0] += p[0] * a_routed * 1
    want_f[20] += a_shared * 4.0
    np.testing.assert_allclose(hf, want_f, rtol=1e-14, atol=1e-16)


# ---------------------------------------------------- the whole token path

def test_forward_token_embedding_lm_head_and_argmax_ties():
    cfg = S.TINY
    d, V = cfg.hidden, cfg.vocab
    w = _tiny_zero_down()                     # blocks add nothing: h_L = E[x]
    w["embed"][:] = 0
    for x in range(V):
        w["embed"][x, x % d] = _bf(0.5 if x % 2 else -0.25)
    w["lm_head"][:] = 0
    for v in range(V):
        w["lm_head"][v, v % d] = _bf(1.0)     # rows v and v+64, v+128, ... tie
    w["lm_head"][d + 7, 7] = _bf(1.0078125)   # one row wins its tie group
    o = O.Oracle(cfg, w)
    r = o.forward_token(7)
    assert r["target"] == d + 7
    assert np.array_equal(r["hidden"][0], S.bf16_bits_to_f32(w["embed"][7]).astype(np.float64))
    r = o.forward_token(9)                    # xhat_f = 8 e_9: logits 8 at v = 9, 73, ...
    assert r["target"] == 9                   # lowest id among the tie
    assert r["logit_gap"] == 0.0
    r = o.forward_token(10, logits=True)      # negative entry: xhat_f = -8 e_10
    assert r["logits"][10] == -8.0 and r["logits"][0] == 0.0
    assert r["target"] == 0                   # every logit <= 0; lowest id among the zeros


def test_final_norm_uses_its_own_gain():
    """The greedy head normalises with the final RMSNorm's gain, not a block's.
    With identity blocks and an all-ones embedding row, RMSNorm(h) = h / sqrt(1
    + eps), which rounds to 1 in bf16, so xhat_f = g_f. One-hot lm_head rows
    then make logit v = g_f[v]."""
    cfg = S.TINY
    d = cfg.hidden
    w = _tiny_zero_down()                     # blocks add nothing: h_L = E[x]
    w["embed"][:] = _bf(1.0)
    w["final_norm"][:] = _bf(1.0)
    w["final_norm"][5] = _bf(3.0)             # the final gain peaks at 5
    w["norm"][:] = _bf(1.0)
    w["norm"][:, 9] = _bf(5.0)                # the blocks' gains peak at 9
    w["lm_head"][:] = 0
    for v in range(d):
        w["lm_head"][v, v] = _bf(1.0)
    r = O.Oracle(cfg, w).forward_token(3, logits=True)
    assert r["target"] == 5
    assert r["logits"][5] == 3.0 and r["logits"][9] == 1.0 and r["logits"][0] == 1.0


# -------------------------------------------------- acceptance and the loop

def _ids(s):
    return [] if s.strip() == "-" else [int(t) for t in s.split(",")]


def test_accept_hand_worked_cases():
    for line in _rows("accept_cases.txt"):
        ds, ts, cs, n = (c.strip() for c in line.split("|"))
        d, t, c = _ids(ds), _ids(ts), _ids(cs)
        K = len(t) - 1
        drafts = np.array([d], np.int32).reshape(1, K)
        committed, alen, bad = O.accept(drafts, np.array([t], np.int32), 512)
        assert committed[0].tolist() == c, line
        assert int(alen[0]) == int(n), line


def test_accept_characterisation_random():
    """n is the first index where draft and target differ (or K), and the
    committed row is exactly target[0..n]."""
    rng = np.random.default_rng(0)
    for K in range(0, 6):
        B = 300
        t = rng.integers(0, 4, size=(B, K + 1)).astype(np.int32)
        d = rng.integers(0, 4, size=(B, K)).astype(np.int32)
        committed, alen, bad = O.accept(d, t, 512)
        assert bad == 0
        for b in range(B):
            n = int(alen[b])
            assert all(d[b, i] == t[b, i] for i in range(n))
            assert n == K or d[b, n] != t[b, n]
            assert committed[b, : n + 1].tolist() == t[b, : n + 1].tolist()
            assert np.all(committed[b, n + 1:] == -1)


@pytest.fixture(scope="module")
def tiny_oracle():
    return O.Oracle(S.TINY, S.make_weights(S.TINY))


@pytest.fixture(scope="module")
def tiny_g(tiny_oracle):
    return tiny_oracle.g_table(range(S.TINY.vocab), nthreads=4)


def test_tiny_g_table_matches_golden(tiny_g):
    """Regression pin: the committed table was written by
    tests/golden/make_golden.py from this oracle on the tiny instance."""
    want = np.loadtxt(os.path.join(GOLDEN, "tiny_g_table.txt"), dtype=np.int64)
    assert np.array_equal(tiny_g, want)


def test_verify_step_targets_align_with_verify_tokens(tiny_oracle, tiny_g):
    rng = np.random.default_rng(1)
    ctx = rng.integers(0, 512, 4).astype(np.int32)
    drafts = rng.integers(0, 512, (4, 3)).astype(np.int32)
    y = tiny_oracle.verify_step(ctx, drafts)
    assert y[:, 0].tolist() == [int(tiny_g[c]) for c in ctx]
    for i in range(3):
        assert y[:, i + 1].tolist() == [int(tiny_g[x]) for x in drafts[:, i]]


def _speculative_decode(verify, accept, start, n_tokens, K, draft_fn):
    """Run the speculative loop until n_tokens are committed; returns them."""
    out = []
    last = start
    step = 0
    while len(out) < n_tokens:
        d = np.array([draft_fn(len(out), step, i) for i in range(K)], np.int32).reshape(1, K)
        y = verify(np.array([last], np.int32), d)
        committed, alen, bad = accept(d, y)
        assert bad == 0
        n = int(alen[0])
        new = committed[0, : n + 1].tolist()
        out.extend(new)
        last = new[-1]
        step += 1
    return out[:n_tokens]


def test_lossless_exhaustive_tiny(tiny_oracle, tiny_g):
    """Speculative commits equal plain greedy decoding from every start id,
    for drafts that are always right, always wrong, random, or adversarial."""
    V = S.TINY.vocab
    g = tiny_g

    def chain(s, n):
        out, x = [], s
        for _ in range(n):
            x = int(g[x])
            out.append(x)
        return out

    def verify_memo(ctx, d):
        toks = np.concatenate([ctx.reshape(-1, 1), d], axis=1)
        return g[toks].astype(np.int32)

    acc = lambda d, y: O.accept(d, y, V)
    rng = np.random.default_rng(5)
    N = 24
    for s in range(V):
        truth = chain(s, N + 8)
        policies = {
            "right": lambda c, st, i: truth[c + i],
            "wrong": lambda c, st, i: (truth[c + i] + 1) % V,
            "random": lambda c, st, i: int(rng.integers(0, V)),
            "adversarial": lambda c, st, i: truth[c + i] if (st + i) % 2 == 0 else (truth[c + i] + 7) % V,
        }
        for K in (0, 1, 3):
            for name, pol in policies.items():
                got = _speculative_decode(verify_memo, acc, s, N, K, pol)
                assert got == truth[:N], (s, K, name)
    # the same loop through the unmemoised verify step on a few start ids
    for s in (0, 17, 300):
        truth = chain(s, 12)
        got = _speculative_decode(tiny_oracle.verify_step, acc, s, 10, 3,
                                  lambda c, st, i: truth[c + i] if (c + i) % 3 else 0)
        assert got == truth[:10]


def test_commit_rate_closed_form_and_printed_value(tiny_g):
    """Monte-Carlo mean commits per step under the synthetic draft policy
    agrees with 1 + p + ... + p^K (matches within 3 sigma), and p = 0.75 at
    K = 3 reproduces the printed 2.73."""
    K_p, p_p, printed = next(_rows("commit_rate.txt")).split()
    K_p, p_p, printed = int(K_p), float(p_p), float(printed)
    assert round(sum(p_p ** i for i in range(K_p + 1)), 2) == printed
    V = S.TINY.vocab
    g = tiny_g
    for K, p in ((3, 0.75), (1, 0.576), (3, 0.576)):
        src = S.DraftSource(p, V, K, seed=11)
        totals = []
        x = 1
        for step in range(3000):
            truth, t = [], x
            for _ in range(K):
                t = int(g[t]); truth.append(t)
            d = src.drafts(0, step, truth).reshape(1, K)
            toks = np.concatenate([[x], d[0]]).astype(np.int64)
            y = g[toks].astype(np.int32).reshape(1, K + 1)
            committed, alen, _ = O.accept(d, y, V)
            n = int(alen[0])
            totals.append(n + 1)
            x = int(committed[0, n])
        q = p + (1 - p) / V          # a random replacement id can still match
        mean = sum(q ** i for i in range(K + 1))
        var = sum((2 * i + 1) * q ** i for i in range(K + 1)) - mean ** 2
        sigma = math.sqrt(var / len(totals))
        assert abs(np.mean(totals) - mean) < 3.5 * sigma, (K, p, np.mean(totals), mean)


# ------------------------------------------------------------ draft head

def _successor_draft_head(V=16, d=64):
    """A draft head whose greedy drafts are t+1, t+2, ... (mod V): identity
    block (zero down projection), embedding E[t] = 8 e_{t+1} - 8 e_t and a
    one-hot lm_head (logit v = coordinate v of the normalised state)."""
    import dataclasses
    cfg = dataclasses.replace(S.DRAFT_TINY, hidden=d, vocab=V)
    w = S.make_weights(cfg, seed=S.SEED_DRAFT_HEAD, with_embed=False, with_lm_head=False)
    w["w_down"] = np.zeros_like(w["w_down"])
    w["s_down"] = np.zeros_like(w["s_down"])
    eight, minus_eight, one = _bf(8.0), _bf(-8.0), _bf(1.0)
    emb = np.zeros((V, d), np.uint16)
    for t in range(V):
        emb[t, (t + 1) % V] = eight
        emb[t, t] = minus_eight
    lm = np.zeros((V, d), np.uint16)
    for v in range(V):
        lm[v, v] = one
    w["embed"], w["lm_head"] = emb, lm
    w["final_norm"] = np.full((d,), one, np.uint16)
    return cfg, w


def test_draft_head_successor_construction():
    """From h = 0 and token t the recursion adds E[t], keeps the running
    state and takes the greedy head at every step: drafts t+1, t+2, t+3 and
    hidden 8 e_{t+i} - 8 e_t after step i."""
    cfg, w = _successor_draft_head()
    o = O.Oracle(cfg, w)
    V, d = cfg.vocab, cfg.hidden
    for t in range(V):
        drafts, hid, gaps = o.draft(np.zeros(d), t, 3)
        assert list(drafts) == [(t + i) % V for i in (1, 2, 3)], (t, drafts)
        for i in range(3):
            want = np.zeros(d)
            want[(t + i + 1) % V] = 8.0
            want[t] = -8.0
            assert np.array_equal(hid[i], want), (t, i)
        assert np.all(gaps > 0)


def test_draft_head_composes_block_and_head_per_step():
    """Each step is h += E[t], then the (separately pinned) block and head,
    with the state carried to the next step."""
    tw = S.make_weights(S.TINY)
    dw = S.make_draft_weights(S.DRAFT_TINY, tw)
    o = O.Oracle(S.DRAFT_TINY, dw)
    emb = S.bf16_bits_to_f32(tw["embed"]).astype(np.float64)
    for t0 in (0, 5, 511):
        h0 = S.bf16_bits_to_f32(S.normal_bf16((64,), 21 + t0, 0, 0.5)).astype(np.float64)
        drafts, hid, _ = o.draft(h0, t0, 3)
        h, t = h0.copy(), t0
        for i in range(3):
            h, *_ = o.layer(0, h + emb[t])
            t, _, _ = o.head(h)
            assert drafts[i] == t and np.array_equal(hid[i], h), (t0, i)
    with pytest.raises(ValueError):
        o.draft(np.zeros(64), 512, 1)


def test_draft_block_groups_equal_one_dense_ffn():
    """The draft block held as 8 shared experts (its intermediate units in 8
    groups, weight 1 each) is the dense SwiGLU FFN of all the units: the same
    weights as one expert of width 8 x 32 (top-1 of 1, weight exactly 1) give
    the same state."""
    import dataclasses
    tw = S.make_weights(S.TINY)
    dw = S.make_draft_weights(S.DRAFT_TINY, tw)
    grouped = O.Oracle(S.DRAFT_TINY, dw)
    S8, Is, d = S.DRAFT_TINY.n_shared, S.DRAFT_TINY.shared_inter, S.DRAFT_TINY.hidden
    dense_cfg = dataclasses.replace(S.DRAFT_TINY, n_shared=0, expert_inter=S8 * Is)
    dense_w = dict(dw)
    dense_w["w_gate"] = dw["s_gate"].reshape(1, 1, S8 * Is, d)
    dense_w["w_up"] = dw["s_up"].reshape(1, 1, S8 * Is, d)
    dense_w["w_down"] = np.ascontiguousarray(
        np.concatenate([dw["s_down"][0, s] for s in range(S8)], axis=1)).reshape(1, 1, d, S8 * Is)
    for k in ("s_gate", "s_up", "s_down"):
        dense_w[k] = np.zeros((1, 0) + dw[k].shape[2:], np.uint16)
    dense = O.Oracle(dense_cfg, dense_w)
    h0 = S.bf16_bits_to_f32(S.normal_bf16((d,), 77, 0, 0.5)).astype(np.float64)
    a, ha, _ = grouped.draft(h0, 3, 3)
    b, hb, _ = dense.draft(h0, 3, 3)
    assert np.array_equal(a, b)
    assert np.max(np.abs(ha - hb)) <= 1e-12 * np.max(np.abs(hb))
