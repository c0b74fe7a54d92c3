"""The pins catch planted mistakes.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign, a wrong index, a transposed operand, a wrong tie
rule), compiles the copy on the CPU and runs the pin suite against it.  The
suite must fail for every one.
"""
import concurrent.futures as fut
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = {
    "rmsnorm drops eps": ("ss / (double)d + eps", "ss / (double)d"),
    "rmsnorm sum instead of mean": ("sqrt(ss / (double)d + eps)", "sqrt(ss + eps)"),
    "router tie picks higher index": ("if (best < 0 || z[e] > z[best]) best = e;",
                                      "if (best < 0 || z[e] >= z[best]) best = e;"),
    "softmax drops normaliser": ("p[e] = exp(z[e] - zmax) / sum;", "p[e] = exp(z[e] - zmax);"),
    "router ignores bias": ("z[e] = acc + (bias ? (double)bias[e] : 0.0);", "z[e] = acc;"),
    "router weight transposed": ("oracle_bf16_value(W[(size_t)e * d + i])",
                                 "oracle_bf16_value(W[(size_t)i * E + e])"),
    "silu sign": ("double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    "swiglu product not rounded": ("a[j] = q_bf16(silu * u);", "a[j] = silu * u;"),
    "gate and up swapped": ("double silu = g / (1.0 + exp(-g));\n    a[j] = q_bf16(silu * u);",
                            "double silu = u / (1.0 + exp(-u));\n    a[j] = q_bf16(silu * g);"),
    "down projection transposed": ("Wd[(size_t)m * I + j]", "Wd[(size_t)j * d + m]"),
    "shared experts dropped": ("for (int s = 0; s < S; ++s) {", "for (int s = 0; s < 0; ++s) {"),
    "shared weight not one": ("for (int m = 0; m < d; ++m) acc[m] += y[m];",
                              "for (int m = 0; m < d; ++m) acc[m] += 0.5 * y[m];"),
    "residual dropped": ("for (int m = 0; m < d; ++m) h[m] += acc[m];",
                         "for (int m = 0; m < d; ++m) h[m] = acc[m];"),
    "routed weights renormalised": ("psel[j] = p[force_sel[j]];\n    }\n  }",
                                    "psel[j] = p[force_sel[j]];\n    }\n  }\n"
                                    "  { double t = 0; for (int j = 0; j < k; ++j) t += psel[j];"
                                    " for (int j = 0; j < k; ++j) psel[j] /= t; }"),
    "argmax tie picks higher id": ("    if (acc > best) {\n      second = best;",
                                   "    if (acc >= best) {\n      second = best;"),
    "embedding row off by one": ("h[i] = oracle_bf16_value(w->embed[(size_t)x * d + i]);",
                                 "h[i] = oracle_bf16_value(w->embed[(size_t)((x + 1) % c->vocab) * d + i]);"),
    "drafts misaligned": ("draft_ids[(size_t)b * K + (i - 1)]", "draft_ids[(size_t)b * K + (K - i)]"),
    "accept commits one token too few": ("for (int i = 0; i <= n; ++i) out[i] = y[i];",
                                         "for (int i = 0; i < n; ++i) out[i] = y[i];"),
    "accept keeps later matches": ("while (n < K && d[n] == y[n]) ++n;",
                                   "for (int i = 0; i < K; ++i) n += (d[i] == y[i]);"),
    "bf16 ties away from zero": ("double r = nearbyint(q);", "double r = round(q);"),
    "draft skips the embedding": ("for (int m = 0; m < d; ++m) h[m] += oracle_bf16_value(erow[m]);",
                                  "(void)erow;"),
    "draft restarts from h_prev": ("    drafts[i] = t;\n",
                                   "    drafts[i] = t;\n    if (!hidden_out) memcpy(h, h_prev, sizeof(double) * (size_t)d);\n"
                                   "    else { memcpy(hidden_out + (size_t)i * d, h, sizeof(double) * (size_t)d);"
                                   " memcpy(h, h_prev, sizeof(double) * (size_t)d); continue; }\n"),
    "draft block applied once": ("    oracle_layer(c, w, 0, h, NULL, NULL, NULL, NULL, NULL);",
                                 "    if (i == 0) oracle_layer(c, w, 0, h, NULL, NULL, NULL, NULL, NULL);"),
    "rmsnorm gain ignored": ("out[i] = oracle_round_bf16(h[i] / s * oracle_bf16_value(g[i]));",
                             "out[i] = oracle_round_bf16(h[i] / s);"),
    "rmsnorm divides by d - 1": ("double s = sqrt(ss / (double)d + eps);",
                                 "double s = sqrt(ss / (double)(d - 1) + eps);"),
    "routed outputs unweighted": ("for (int m = 0; m < d; ++m) acc[m] += psel[j] * y[m];",
                                  "for (int m = 0; m < d; ++m) acc[m] += y[m];"),
    "every slot weighted like the first": ("    p_sel[j] = p[best];", "    p_sel[j] = p[sel[0]];"),
    "final norm with the first block's gain": (
        "oracle_rmsnorm_bf16(h, w->final_norm, d, c->rms_eps, xf);",
        "oracle_rmsnorm_bf16(h, w->norm[0], d, c->rms_eps, xf);"),
    "lm_head on the unnormalised state": (
        "oracle_rmsnorm_bf16(h, w->final_norm, d, c->rms_eps, xf);",
        "for (int i = 0; i < d; ++i) xf[i] = oracle_round_bf16(h[i]);"),
    "block uses the next block's router": ("oracle_router(xhat, w->router[l],",
                                           "oracle_router(xhat, w->router[(l + 1) % c->n_layers],"),
    "accept ignores bad targets": ("for (int i = 0; i <= K; ++i) bad |= (y[i] < 0 || y[i] >= V);",
                                   "(void)0;"),
    "accept takes id V as valid": ("bad |= (d[i] < 0 || d[i] >= V);", "bad |= (d[i] < 0 || d[i] > V);"),
    "draft embeds the first token every step": ("const uint16_t* erow = w->embed + (size_t)t * d;",
                                                "const uint16_t* erow = w->embed + (size_t)t_prev * d;"),
    "routed expert off by one": ("    int e = sel[j];", "    int e = (sel[j] + 1) % E;"),
    "shared experts read the routed weights": (
        "oracle_swiglu_expert(xhat, w->s_gate[l] + s * sh_in, w->s_up[l] + s * sh_in,",
        "oracle_swiglu_expert(xhat, w->w_gate[l] + s * sh_in, w->w_up[l] + s * sh_in,"),
    "gate projection rounded before SiLU": ("    double silu = g / (1.0 + exp(-g));\n",
                                            "    g = q_bf16(g);\n    double silu = g / (1.0 + exp(-g));\n"),
    "top-k selects one expert k times": ("    taken[best] = 1;", "    (void)taken;"),
    "top-k never considers the last expert": ("      if (taken[e]) continue;",
                                              "      if (taken[e] || e == E - 1) continue;"),
    "lm_head read transposed": ("const uint16_t* row = w->lm_head + (size_t)v * d;",
                                "const uint16_t* row = w->lm_head + (size_t)v;"),
    "argmax never considers the last id": ("  for (int v = 0; v < V; ++v) {\n    double acc = 0.0;",
                                           "  for (int v = 0; v < V - 1; ++v) {\n    double acc = 0.0;"),
    "gate projection transposed": ("g += x * oracle_bf16_value(Wg[(size_t)j * d + i]);",
                                   "g += x * oracle_bf16_value(Wg[(size_t)i * I + j]);"),
    "up projection transposed": ("u += x * oracle_bf16_value(Wu[(size_t)j * d + i]);",
                                 "u += x * oracle_bf16_value(Wu[(size_t)i * I + j]);"),
    "combine added twice": ("for (int m = 0; m < d; ++m) h[m] += acc[m];",
                            "for (int m = 0; m < d; ++m) h[m] += 2.0 * acc[m];"),
    "eps added after the square root": ("double s = sqrt(ss / (double)d + eps);",
                                        "double s = sqrt(ss / (double)d) + eps;"),
}


# Mistakes in the attention of the stack with attention, run against its pins.
ATTN_MUTANTS = {
    "attention drops the 1/sqrt(hd) scale": ("sc[j] = s * scale;", "sc[j] = s;"),
    "attention leaves out the current token": ("const int nk = pos + 1;", "const int nk = pos > 0 ? pos : 1;"),
    "rope pairs neighbouring dims": (
        "    const double a = x[i], b = x[i + half];\n    x[i] = a * c - b * s;\n    x[i + half] = a * s + b * c;",
        "    const double a = x[2 * i], b = x[2 * i + 1];\n    x[2 * i] = a * c - b * s;\n    x[2 * i + 1] = a * s + b * c;"),
    "rope turns the other way": ("    x[i] = a * c - b * s;\n    x[i + half] = a * s + b * c;",
                                 "    x[i] = a * c + b * s;\n    x[i + half] = -a * s + b * c;"),
    "rope frequency exponent halved": ("pow(theta, -2.0 * (double)i / (double)hd)",
                                       "pow(theta, -(double)i / (double)hd)"),
    "queries turned at the next position": ("oracle_rope(q + (size_t)hh * hd, hd, pos, a->rope_theta);",
                                            "oracle_rope(q + (size_t)hh * hd, hd, pos + 1, a->rope_theta);"),
    "keys turned at the next position": ("oracle_rope(k + (size_t)hh * hd, hd, pos, a->rope_theta);",
                                         "oracle_rope(k + (size_t)hh * hd, hd, pos + 1, a->rope_theta);"),
    "values turned like the keys": ("    oracle_rope(k + (size_t)hh * hd, hd, pos, a->rope_theta);\n  }",
                                    "    oracle_rope(k + (size_t)hh * hd, hd, pos, a->rope_theta);\n"
                                    "    oracle_rope(v + (size_t)hh * hd, hd, pos, a->rope_theta);\n  }"),
    "key cache not rounded": ("kc[(size_t)pos * d + m] = q_bf16(k[m]);", "kc[(size_t)pos * d + m] = k[m];"),
    "value cache not rounded": ("vc[(size_t)pos * d + m] = q_bf16(v[m]);", "vc[(size_t)pos * d + m] = v[m];"),
    "attention output not rounded": ("o[hh * hd + i] = q_bf16(acc / sum);", "o[hh * hd + i] = acc / sum;"),
    "softmax drops its normaliser": ("o[hh * hd + i] = q_bf16(acc / sum);", "o[hh * hd + i] = q_bf16(acc);"),
    "output projection transposed": ("o[i] * oracle_bf16_value(a->w_o[l][(size_t)m * d + i])",
                                     "o[i] * oracle_bf16_value(a->w_o[l][(size_t)i * d + m])"),
    "value projection transposed": ("av += x * oracle_bf16_value(a->w_v[l][(size_t)m * d + i]);",
                                    "av += x * oracle_bf16_value(a->w_v[l][(size_t)i * d + m]);"),
    "attention residual dropped": ("    h[m] += acc;\n  }\n  free(xa);", "    h[m] = acc;\n  }\n  free(xa);"),
    "attention attends over the other head": ("s += qh[i] * kc[(size_t)j * d + hh * hd + i];",
                                              "s += qh[i] * kc[(size_t)j * d + ((hh + 1) % H) * hd + i];"),
    "attention after the MoE block": (
        "      oracle_attn_block(c, a, l, h, p, kc + (size_t)l * n * d, vc + (size_t)l * n * d, NULL);\n"
        "      oracle_layer(c, w, l, h, NULL, NULL, NULL, route_gaps ? route_gaps + (size_t)p * L + l : NULL,\n"
        "                   NULL);",
        "      oracle_layer(c, w, l, h, NULL, NULL, NULL, route_gaps ? route_gaps + (size_t)p * L + l : NULL,\n"
        "                   NULL);\n"
        "      oracle_attn_block(c, a, l, h, p, kc + (size_t)l * n * d, vc + (size_t)l * n * d, NULL);"),
}


def _run_mutant(name, old, new, tmp, pins="test_oracle_pins.py"):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} must occur exactly once"
    tag = "".join(c if c.isalnum() else "_" for c in name)
    c_path = os.path.join(tmp, f"{tag}.c")
    so_path = os.path.join(tmp, f"{tag}.so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                           "-fvisibility=hidden", "-o", so_path, c_path, "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=so_path)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with fut.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
            results = list(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp), MUTANTS.items()))
    survivors = [n for n, rc in results if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"


def test_every_planted_attention_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with fut.ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
            results = list(ex.map(lambda kv: _run_mutant(kv[0], *kv[1], tmp,
                                                         pins="test_attn_oracle_pins.py"),
                                  ATTN_MUTANTS.items()))
    survivors = [n for n, rc in results if rc == 0]
    assert not survivors, f"attention pins did not catch: {survivors}"
