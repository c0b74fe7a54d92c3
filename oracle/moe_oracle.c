/*
 * fp64 CPU oracle of the MoE greedy-verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg call this code; the product library never
 * links it, and it shares no code with the CUDA path.
 *
 * It is plain, single-threaded and slow on purpose: every sum runs in index
 * order in double precision, with no blocking, fusion or reordering.
 *
 * What it computes, and where that comes from:
 *   - The decoder block (RMSNorm, softmax router picking the top-6 of 64
 *     routed SwiGLU experts, two always-on shared experts, weighted combine,
 *     residual): "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser
 *     With Built-In Speculative Decoding", architecture paragraph (DeepSeek-
 *     3B-MoE decoder: 12 layers, 64 routed and two shared experts, top-6).
 *     Attention is not on this path: a verify token's target depends only
 *     on the token itself, so the target stack is a fixed map g over ids.
 *   - Greedy verification and the acceptance rule: same article, FastMTP
 *     paragraph (keep the longest draft prefix matching the decoder's own
 *     greedy choices, then commit one more token of its own; all K drafts
 *     matching commits K+1 tokens), and "Jina-OCR-v1: Efficient Document
 *     Parsing with Speculative Decoding and Dense Verifiable Rewards",
 *     Abstract (greedy verification makes decoding lossless).
 *
 * Readings the pages leave open, fixed here:
 *   - bf16 rounding (round to nearest even) happens at exactly three points:
 *     each RMSNorm output, and the SwiGLU product silu(g)*u.  The residual
 *     stream, router logits, softmax, combine and logits stay in fp64.
 *   - Top-k selects on router logits z (ties: lower expert index first);
 *     the combine weights are the softmax probabilities over all experts,
 *     not renormalised over the selected ones.
 *   - Shared experts carry weight 1.
 *   - argmax ties resolve to the lowest token id.
 *   - accept_len = number of accepted drafts n; n+1 tokens are committed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

typedef struct {
  int32_t n_layers, hidden, n_experts, top_k, n_shared, expert_inter, shared_inter, vocab;
  double rms_eps;
} oracle_config;

/* Host arrays of bf16 bit patterns, PyTorch Linear layout [out, in]. */
typedef struct {
  const uint16_t* embed;           /* [V, d] */
  const uint16_t* final_norm;      /* [d] */
  const uint16_t* lm_head;         /* [V, d] */
  const uint16_t* const* norm;     /* L x [d] */
  const uint16_t* const* router;   /* L x [E, d] */
  const float* const* router_bias; /* L x [E], or NULL */
  const uint16_t* const* w_gate;   /* L x [E, I, d] */
  const uint16_t* const* w_up;     /* L x [E, I, d] */
  const uint16_t* const* w_down;   /* L x [E, d, I] */
  const uint16_t* const* s_gate;   /* L x [S, Is, d] */
  const uint16_t* const* s_up;     /* L x [S, Is, d] */
  const uint16_t* const* s_down;   /* L x [S, d, Is] */
} oracle_weights;

/* ---------------------------------------------------------------- bf16 -- */

ORACLE_API double oracle_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), straight from fp64 so
 * that there is no double rounding.  bf16 = 1 sign, 8 exponent, 7 fraction
 * bits: a finite value is m * 2^(e-7) with m an integer, |m| < 256, e >= -126. */
ORACLE_API uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e = ilogb(x); /* x = f * 2^e with 1 <= |f| < 2 */
  if (e < -126) e = -126;
  double q = ldexp(x, 7 - e); /* |q| < 256 at normal e; exact */
  double r = nearbyint(q);    /* default rounding mode: nearest, ties to even */
  double y = ldexp(r, e - 7);
  /* largest finite bf16 is (2 - 2^-7) * 2^127 */
  if (fabs(y) > 3.3895313892515355e38) return x > 0 ? 0x7F80 : 0xFF80;
  float yf = (float)y; /* exact: y has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &yf, 4);
  return (uint16_t)(u >> 16);
}

static double q_bf16(double x) { return oracle_bf16_value(oracle_round_bf16(x)); }

/* ------------------------------------------------------------- pieces -- */

/* xhat_i = bf16( h_i / sqrt(mean(h^2) + eps) * g_i ) */
ORACLE_API void oracle_rmsnorm_bf16(const double* h, const uint16_t* g, int32_t d, double eps,
                                    uint16_t* out) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += h[i] * h[i];
  double s = sqrt(ss / (double)d + eps);
  for (int i = 0; i < d; ++i) out[i] = oracle_round_bf16(h[i] / s * oracle_bf16_value(g[i]));
}

/* z_e = sum_i xhat_i W[e,i] (+ b_e);  p = softmax(z);  sel = top-k of z,
 * ordered by (z desc, e asc);  p_sel = p[sel];  gap = z_(k) - z_(k+1). */
ORACLE_API void oracle_router(const uint16_t* xhat, const uint16_t* W, const float* bias,
                              int32_t E, int32_t d, int32_t k, double* z, double* p,
                              int32_t* sel, double* p_sel, double* gap) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
      acc += oracle_bf16_value(xhat[i]) * oracle_bf16_value(W[(size_t)e * d + i]);
    z[e] = acc + (bias ? (double)bias[e] : 0.0);
  }
  double zmax = z[0];
  for (int e = 1; e < E; ++e)
    if (z[e] > zmax) zmax = z[e];
  double sum = 0.0;
  for (int e = 0; e < E; ++e) sum += exp(z[e] - zmax);
  for (int e = 0; e < E; ++e) p[e] = exp(z[e] - zmax) / sum;
  /* selection: k passes, each takes the largest remaining z (lowest e on ties) */
  char taken[1024];
  memset(taken, 0, sizeof(taken));
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || z[e] > z[best]) best = e;
    }
    taken[best] = 1;
    sel[j] = best;
    p_sel[j] = p[best];
  }
  if (gap) {
    double next = -INFINITY;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && z[e] > next) next = z[e];
    *gap = (k < E) ? z[sel[k - 1]] - next : INFINITY;
  }
}

/* One SwiGLU expert: a_j = bf16( silu(xhat . Wg[j]) * (xhat . Wu[j]) ),
 * y_m = sum_j a_j Wd[m, j], with silu(v) = v / (1 + exp(-v)). */
ORACLE_API void oracle_swiglu_expert(const uint16_t* xhat, const uint16_t* Wg, const uint16_t* Wu,
                                     const uint16_t* Wd, int32_t d, int32_t I, double* y) {
  double* a = (double*)malloc(sizeof(double) * (size_t)I);
  for (int j = 0; j < I; ++j) {
    double g = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      double x = oracle_bf16_value(xhat[i]);
      g += x * oracle_bf16_value(Wg[(size_t)j * d + i]);
      u += x * oracle_bf16_value(Wu[(size_t)j * d + i]);
    }
    double silu = g / (1.0 + exp(-g));
    a[j] = q_bf16(silu * u);
  }
  for (int m = 0; m < d; ++m) {
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += a[j] * oracle_bf16_value(Wd[(size_t)m * I + j]);
    y[m] = acc;
  }
  free(a);
}

/* One decoder block on one token, h updated in place:
 *   xhat = bf16(RMSNorm(h));  route;  h += sum_j p_sel[j] y_sel[j] + sum_s y_s
 * (routed slots in selection order, then shared experts in index order).
 * force_sel (k ids, or NULL) replaces the selected set, keeping the softmax
 * weights of the forced experts: used to follow a different but equally valid
 * choice at a near tie.  Diagnostics (each may be NULL): sel_out[k] (the
 * block's own top-k choice, before any forcing), w_out[k] (the weights
 * applied), gap_out (z_(k) - z_(k+1)), xhat_out[d]. */
ORACLE_API void oracle_layer(const oracle_config* c, const oracle_weights* w, int32_t l, double* h,
                             const int32_t* force_sel, int32_t* sel_out, double* w_out,
                             double* gap_out, uint16_t* xhat_out) {
  const int d = c->hidden, E = c->n_experts, k = c->top_k, I = c->expert_inter,
            S = c->n_shared, Is = c->shared_inter;
  uint16_t* xhat = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
  double* z = (double*)malloc(sizeof(double) * (size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* psel = (double*)malloc(sizeof(double) * (size_t)k);
  double* y = (double*)malloc(sizeof(double) * (size_t)d);
  double* acc = (double*)calloc((size_t)d, sizeof(double));
  double gap = 0.0;

  oracle_rmsnorm_bf16(h, w->norm[l], d, c->rms_eps, xhat);
  oracle_router(xhat, w->router[l], w->router_bias ? w->router_bias[l] : NULL, E, d, k, z, p, sel,
                psel, &gap);
  if (sel_out) memcpy(sel_out, sel, sizeof(int32_t) * (size_t)k); /* the block's own choice */
  if (force_sel) {
    for (int j = 0; j < k; ++j) {
      sel[j] = force_sel[j];
      psel[j] = p[force_sel[j]];
    }
  }
  const size_t ex_in = (size_t)I * d, ex_out = (size_t)d * I;
  for (int j = 0; j < k; ++j) {
    int e = sel[j];
    oracle_swiglu_expert(xhat, w->w_gate[l] + e * ex_in, w->w_up[l] + e * ex_in,
                         w->w_down[l] + e * ex_out, d, I, y);
    for (int m = 0; m < d; ++m) acc[m] += psel[j] * y[m];
  }
  const size_t sh_in = (size_t)Is * d, sh_out = (size_t)d * Is;
  for (int s = 0; s < S; ++s) {
    oracle_swiglu_expert(xhat, w->s_gate[l] + s * sh_in, w->s_up[l] + s * sh_in,
                         w->s_down[l] + s * sh_out, d, Is, y);
    for (int m = 0; m < d; ++m) acc[m] += y[m];
  }
  for (int m = 0; m < d; ++m) h[m] += acc[m];

  if (w_out) memcpy(w_out, psel, sizeof(double) * (size_t)k);
  if (gap_out) *gap_out = gap;
  if (xhat_out) memcpy(xhat_out, xhat, sizeof(uint16_t) * (size_t)d);
  free(xhat); free(z); free(p); free(sel); free(psel); free(y); free(acc);
}

/* logits_v = xhat_f . W_lm[v];  target = argmax (lowest v on ties). */
static int32_t lm_head_argmax(const oracle_config* c, const oracle_weights* w, const uint16_t* xf,
                              double* logits_out, double* top2_gap) {
  const int d = c->hidden, V = c->vocab;
  double best = -INFINITY, second = -INFINITY;
  int32_t arg = 0;
  for (int v = 0; v < V; ++v) {
    double acc = 0.0;
    const uint16_t* row = w->lm_head + (size_t)v * d;
    for (int i = 0; i < d; ++i) acc += oracle_bf16_value(xf[i]) * oracle_bf16_value(row[i]);
    if (logits_out) logits_out[v] = acc;
    if (acc > best) {
      second = best;
      best = acc;
      arg = v;
    } else if (acc > second) {
      second = acc;
    }
  }
  if (top2_gap) *top2_gap = best - second;
  return arg;
}

/* Final RMSNorm and greedy choice on a given residual stream h [d]:
 * xhat_f = bf16(RMSNorm(h) * g_f);  returns argmax_v xhat_f . W_lm[v]
 * (lowest v on ties).  logits [V] and logit_gap (top-2 gap) may be NULL. */
ORACLE_API int32_t oracle_head(const oracle_config* c, const oracle_weights* w, const double* h,
                               double* logits, double* logit_gap) {
  uint16_t* xf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)c->hidden);
  oracle_rmsnorm_bf16(h, w->final_norm, c->hidden, c->rms_eps, xf);
  int32_t y = lm_head_argmax(c, w, xf, logits, logit_gap);
  free(xf);
  return y;
}

/* Target stack on one verify token id x:
 *   h = E[x];  L decoder blocks;  xhat_f = bf16(RMSNorm(h));  argmax of logits.
 * Returns the greedy next id.  Optional outputs: force_sel [L*k] (NULL: route
 * freely), sel_out [L*k], w_out [L*k], route_gap [L], hidden_out [(L+1)*d]
 * (residual stream after the embedding and after each block), xhat_f [d],
 * logits [V], logit_gap (top-2 logit gap). */
ORACLE_API int32_t oracle_forward_token(const oracle_config* c, const oracle_weights* w, int32_t x,
                                        const int32_t* force_sel, int32_t* sel_out, double* w_out,
                                        double* route_gap, double* hidden_out, uint16_t* xhat_f,
                                        double* logits, double* logit_gap) {
  const int d = c->hidden, L = c->n_layers, k = c->top_k;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) h[i] = oracle_bf16_value(w->embed[(size_t)x * d + i]);
  if (hidden_out) memcpy(hidden_out, h, sizeof(double) * (size_t)d);
  for (int l = 0; l < L; ++l) {
    oracle_layer(c, w, l, h, force_sel ? force_sel + (size_t)l * k : NULL,
                 sel_out ? sel_out + (size_t)l * k : NULL, w_out ? w_out + (size_t)l * k : NULL,
                 route_gap ? route_gap + l : NULL, NULL);
    if (hidden_out) memcpy(hidden_out + (size_t)(l + 1) * d, h, sizeof(double) * (size_t)d);
  }
  uint16_t* xf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
  oracle_rmsnorm_bf16(h, w->final_norm, d, c->rms_eps, xf);
  if (xhat_f) memcpy(xhat_f, xf, sizeof(uint16_t) * (size_t)d);
  int32_t y = lm_head_argmax(c, w, xf, logits, logit_gap);
  free(h);
  free(xf);
  return y;
}

/* Verify step for B sequences.  Sequence b's verify tokens are
 * x_b = [context_ids[b], draft_ids[b,0], ..., draft_ids[b,K-1]];
 * target_ids[b,i] = g(x_b[i]), the greedy choice for the token after x_b[i].
 * Returns 0, or -1 if an id is outside [0, V). */
ORACLE_API int32_t oracle_verify_step(const oracle_config* c, const oracle_weights* w,
                                      const int32_t* context_ids, const int32_t* draft_ids,
                                      int32_t B, int32_t K, int32_t* target_ids) {
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i <= K; ++i) {
      int32_t x = (i == 0) ? context_ids[b] : draft_ids[(size_t)b * K + (i - 1)];
      if (x < 0 || x >= c->vocab) return -1;
      target_ids[(size_t)b * (K + 1) + i] =
          oracle_forward_token(c, w, x, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
    }
  }
  return 0;
}

/* Acceptance: n = the length of the longest prefix with draft[i] == target[i];
 * committed = target[0..n] (n+1 tokens, the rest -1); accept_len = n.
 * A sequence with any draft or target id outside [0, V) gets accept_len -1
 * and a row of -1.  Returns the number of such sequences. */
ORACLE_API int32_t oracle_accept(const int32_t* draft_ids, const int32_t* target_ids, int32_t B,
                                 int32_t K, int32_t V, int32_t* committed, int32_t* accept_len) {
  int32_t bad_rows = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t* d = draft_ids + (size_t)b * K;
    const int32_t* y = target_ids + (size_t)b * (K + 1);
    int32_t* out = committed + (size_t)b * (K + 1);
    int bad = 0;
    for (int i = 0; i < K; ++i) bad |= (d[i] < 0 || d[i] >= V);
    for (int i = 0; i <= K; ++i) bad |= (y[i] < 0 || y[i] >= V);
    for (int i = 0; i <= K; ++i) out[i] = -1;
    if (bad) {
      accept_len[b] = -1;
      ++bad_rows;
      continue;
    }
    int n = 0;
    while (n < K && d[n] == y[n]) ++n;
    for (int i = 0; i <= n; ++i) out[i] = y[i];
    accept_len[b] = n;
  }
  return bad_rows;
}

/* Single decoder block with bf16 input and output (the layer entry point):
 * h = h_in (bf16 -> fp64), one block, h_out = bf16(h).  Diagnostics as in
 * oracle_layer; h_out_f64 (may be NULL) receives the unrounded result. */
ORACLE_API void oracle_layer_bf16(const oracle_config* c, const oracle_weights* w, int32_t l,
                                  const uint16_t* h_in, const int32_t* force_sel, uint16_t* h_out,
                                  double* h_out_f64, int32_t* sel_out, double* w_out,
                                  double* gap_out) {
  const int d = c->hidden;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  for (int i = 0; i < d; ++i) h[i] = oracle_bf16_value(h_in[i]);
  oracle_layer(c, w, l, h, force_sel, sel_out, w_out, gap_out, NULL);
  for (int i = 0; i < d; ++i) h_out[i] = oracle_round_bf16(h[i]);
  if (h_out_f64) memcpy(h_out_f64, h, sizeof(double) * (size_t)d);
  free(h);
}

/* FastMTP draft head ("Jina AI Releases jina-ocr-v1, a 3.4B MoE Document
 * Parser With Built-In Speculative Decoding", FastMTP paragraph: one dense
 * draft block applied recursively for K steps with the same parameters;
 * "Jina-OCR-v1: Efficient Document Parsing with Speculative Decoding and
 * Dense Verifiable Rewards", Abstract: a single draft block shared across the
 * K prediction steps).  The pages leave the block's inputs open; reading
 * taken: step i adds the embedding of the previous token to the running
 * hidden state, applies the block (config c with one expert of weight 1, no
 * attention), and takes the verifier's greedy head:
 *   h = h_prev;  t = t_prev;
 *   for i < K:  h += E[t];  h = block(h);  t = argmax(lm_head . bf16(RMSNorm_f(h)));  drafts[i] = t.
 * hidden_out [K*d] (h after each step) and gaps [K] (top-2 logit gaps) may be
 * NULL.  Returns 0, or -1 if an id falls outside [0, V). */
ORACLE_API int32_t oracle_draft(const oracle_config* c, const oracle_weights* w,
                                const double* h_prev, int32_t t_prev, int32_t K, int32_t* drafts,
                                double* hidden_out, double* gaps) {
  const int d = c->hidden;
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  memcpy(h, h_prev, sizeof(double) * (size_t)d);
  int32_t t = t_prev;
  int32_t rc = 0;
  for (int i = 0; i < K; ++i) {
    if (t < 0 || t >= c->vocab) {
      rc = -1;
      break;
    }
    const uint16_t* erow = w->embed + (size_t)t * d;
    for (int m = 0; m < d; ++m) h[m] += oracle_bf16_value(erow[m]);
    oracle_layer(c, w, 0, h, NULL, NULL, NULL, NULL, NULL);
    t = oracle_head(c, w, h, NULL, gaps ? gaps + i : NULL);
    drafts[i] = t;
    if (hidden_out) memcpy(hidden_out + (size_t)i * d, h, sizeof(double) * (size_t)d);
  }
  free(h);
  return rc;
}

/* ------------------------------------------------------- attention (NEXT) --
 * The decoder's attention, which the verify step above leaves out.  The
 * pages name the decoder (DeepSeek-3B-MoE, 12 layers, position limit 32,768:
 * "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser With Built-In
 * Speculative Decoding", architecture paragraph) but give no attention shape.
 * Reading taken:
 *   - each block is pre-norm attention then the MoE block above:
 *       h += W_o . attn(bf16(RMSNorm_a(h) * g_a));   then oracle_layer;
 *   - multi-head attention, n_heads heads of width hd = d / n_heads, no
 *     biases; rotary position embedding on q and k over the whole head, the
 *     two halves of a head paired (dims i and i + hd/2), angle pos *
 *     theta^(-2i/hd), pos = the token's 0-based index in its sequence;
 *   - causal: the token at pos attends to positions 0 .. pos (itself
 *     included), scores q . k_j / sqrt(hd), softmax over them;
 *   - rounding to bf16 (nearest even) at: the attention RMSNorm output, k
 *     after the rotation and v (the key/value cache holds bf16), and the
 *     attention output o before W_o.  q, scores, softmax and W_o's sum stay
 *     fp64 here.
 */

typedef struct {
  int32_t n_heads;
  double rope_theta;
  const uint16_t* const* attn_norm; /* L x [d] */
  const uint16_t* const* w_q;       /* L x [d, d] */
  const uint16_t* const* w_k;       /* L x [d, d] */
  const uint16_t* const* w_v;       /* L x [d, d] */
  const uint16_t* const* w_o;       /* L x [d, d] */
} oracle_attn_weights;

/* Rotary embedding of one head vector x [hd] at position pos, in place:
 * for i < hd/2, (x_i, x_{i+hd/2}) is turned by the angle pos * theta^(-2i/hd). */
ORACLE_API void oracle_rope(double* x, int32_t hd, int32_t pos, double theta) {
  const int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    const double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)hd);
    const double c = cos(ang), s = sin(ang);
    const double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = a * s + b * c;
  }
}

/* The attention sub-block of layer l on one token at position pos, h [d]
 * updated in place.  kc, vc: this layer's key and value cache of the token's
 * sequence, [pos + 1, d] values of bf16 numbers; rows 0 .. pos-1 are read (the
 * earlier tokens), row pos is written with this token's k and v.  o_out [d]
 * (may be NULL) receives the bf16 attention output before W_o. */
ORACLE_API void oracle_attn_block(const oracle_config* c, const oracle_attn_weights* a, int32_t l,
                                  double* h, int32_t pos, double* kc, double* vc, double* o_out) {
  const int d = c->hidden, H = a->n_heads, hd = d / H;
  uint16_t* xa = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
  double* q = (double*)malloc(sizeof(double) * (size_t)d);
  double* k = (double*)malloc(sizeof(double) * (size_t)d);
  double* v = (double*)malloc(sizeof(double) * (size_t)d);
  double* o = (double*)malloc(sizeof(double) * (size_t)d);
  double* sc = (double*)malloc(sizeof(double) * (size_t)(pos + 1));
  oracle_rmsnorm_bf16(h, a->attn_norm[l], d, c->rms_eps, xa);
  for (int m = 0; m < d; ++m) {
    double aq = 0.0, ak = 0.0, av = 0.0;
    for (int i = 0; i < d; ++i) {
      const double x = oracle_bf16_value(xa[i]);
      aq += x * oracle_bf16_value(a->w_q[l][(size_t)m * d + i]);
      ak += x * oracle_bf16_value(a->w_k[l][(size_t)m * d + i]);
      av += x * oracle_bf16_value(a->w_v[l][(size_t)m * d + i]);
    }
    q[m] = aq;
    k[m] = ak;
    v[m] = av;
  }
  for (int hh = 0; hh < H; ++hh) {
    oracle_rope(q + (size_t)hh * hd, hd, pos, a->rope_theta);
    oracle_rope(k + (size_t)hh * hd, hd, pos, a->rope_theta);
  }
  for (int m = 0; m < d; ++m) {
    kc[(size_t)pos * d + m] = q_bf16(k[m]);
    vc[(size_t)pos * d + m] = q_bf16(v[m]);
  }
  const double scale = 1.0 / sqrt((double)hd);
  const int nk = pos + 1; /* keys 0 .. pos: the earlier tokens and this one */
  for (int hh = 0; hh < H; ++hh) {
    const double* qh = q + (size_t)hh * hd;
    double mx = -INFINITY;
    for (int j = 0; j < nk; ++j) {
      double s = 0.0;
      for (int i = 0; i < hd; ++i) s += qh[i] * kc[(size_t)j * d + hh * hd + i];
      sc[j] = s * scale;
      if (sc[j] > mx) mx = sc[j];
    }
    double sum = 0.0;
    for (int j = 0; j < nk; ++j) {
      sc[j] = exp(sc[j] - mx);
      sum += sc[j];
    }
    for (int i = 0; i < hd; ++i) {
      double acc = 0.0;
      for (int j = 0; j < nk; ++j) acc += sc[j] * vc[(size_t)j * d + hh * hd + i];
      o[hh * hd + i] = q_bf16(acc / sum);
    }
  }
  if (o_out) memcpy(o_out, o, sizeof(double) * (size_t)d);
  for (int m = 0; m < d; ++m) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += o[i] * oracle_bf16_value(a->w_o[l][(size_t)m * d + i]);
    h[m] += acc;
  }
  free(xa); free(q); free(k); free(v); free(o); free(sc);
}

/* A whole sequence through the stack with attention, in order: for pos =
 * 0 .. n-1, h = E[ids[pos]]; for each layer, the attention sub-block (with
 * this sequence's caches) then the MoE block; targets[pos] = the greedy next
 * id after ids[0..pos].  Optional outputs: logit_gaps [n] (top-2 gap),
 * route_gaps [n * L] (each block's selection gap), kcache / vcache
 * [L, n, d] (the caches after the last position; NULL: kept internally),
 * hidden_out [n, L+1, d] (residual stream entering each block's attention,
 * and after the last block).  Returns 0, or -1 if an id is outside [0, V). */
ORACLE_API int32_t oracle_forward_seq(const oracle_config* c, const oracle_weights* w,
                                      const oracle_attn_weights* a, const int32_t* ids, int32_t n,
                                      int32_t* targets, double* logit_gaps, double* route_gaps,
                                      double* kcache, double* vcache, double* hidden_out) {
  const int d = c->hidden, L = c->n_layers;
  for (int p = 0; p < n; ++p)
    if (ids[p] < 0 || ids[p] >= c->vocab) return -1;
  const size_t csz = (size_t)L * n * d;
  double* kc = kcache ? kcache : (double*)malloc(sizeof(double) * csz);
  double* vc = vcache ? vcache : (double*)malloc(sizeof(double) * csz);
  double* h = (double*)malloc(sizeof(double) * (size_t)d);
  for (int p = 0; p < n; ++p) {
    for (int i = 0; i < d; ++i) h[i] = oracle_bf16_value(w->embed[(size_t)ids[p] * d + i]);
    for (int l = 0; l < L; ++l) {
      if (hidden_out) memcpy(hidden_out + ((size_t)p * (L + 1) + l) * d, h, sizeof(double) * (size_t)d);
      oracle_attn_block(c, a, l, h, p, kc + (size_t)l * n * d, vc + (size_t)l * n * d, NULL);
      oracle_layer(c, w, l, h, NULL, NULL, NULL, route_gaps ? route_gaps + (size_t)p * L + l : NULL,
                   NULL);
    }
    if (hidden_out) memcpy(hidden_out + ((size_t)p * (L + 1) + L) * d, h, sizeof(double) * (size_t)d);
    targets[p] = oracle_head(c, w, h, NULL, logit_gaps ? logit_gaps + p : NULL);
  }
  free(h);
  if (!kcache) free(kc);
  if (!vcache) free(vc);
  return 0;
}
