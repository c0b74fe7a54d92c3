/*
 * moe_verify.h - C ABI of the GB300 (sm_103a) MoE greedy-verify library.
 *
 * The library runs the batched greedy verification step of a FastMTP-style
 * speculative decoder over a DeepSeek-3B-MoE-style target stack, and the
 * acceptance rule that follows it.
 *
 *   Architecture: "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser
 *   With Built-In Speculative Decoding", architecture paragraph (12 decoder
 *   layers, 64 routed experts, two shared experts, top-6 routing).
 *   Verification and acceptance: the same article, FastMTP paragraph (the
 *   decoder checks K drafts greedily, keeps the longest prefix equal to its
 *   own choices and commits one more token of its own, K+1 tokens when all
 *   drafts match), and "Jina-OCR-v1: Efficient Document Parsing with
 *   Speculative Decoding and Dense Verifiable Rewards", Abstract (greedy
 *   verification makes decoding lossless).
 *
 * Per verify token x the step computes
 *   h = E[x]
 *   for each layer l:  xhat = bf16(RMSNorm(h) * g_l)
 *                      z = xhat W_r^T (+ b);  p = softmax(z);  S = top-k of z
 *                      a_e = bf16(silu(xhat W_g,e^T) * (xhat W_u,e^T))
 *                      h += sum_{e in S} p_e a_e W_d,e^T + sum_shared a_s W_d,s^T
 *   target = argmax_v bf16(RMSNorm(h) * g_f) . W_lm[v]   (lowest v on ties)
 * The target stack has no attention on this path, so a verify token's target
 * depends on that token alone.
 *
 * Conventions
 *   - Every pointer argument is device memory unless its comment says host.
 *     The caller owns all of it; the library never frees caller memory.
 *   - bf16 tensors are passed as raw 16-bit patterns (void*), PyTorch Linear
 *     layout [out_features, in_features], row-major, contiguous.
 *   - Calls that take a cuda_stream (a cudaStream_t, NULL = legacy default
 *     stream) only enqueue work on it and return without synchronising,
 *     except where noted.  moe_verify_step, moe_verify_accept and
 *     moe_verify_layer allocate nothing, do no host-device copies and may be
 *     captured into a CUDA graph.
 *   - Argument errors are found on the host and returned at once; nothing is
 *     enqueued then.  Errors found on the device (an id outside [0, V), a
 *     bounded wait that ran out) set a sticky flag in the context; the next
 *     moe_verify_sync_status reports and clears it.  No device code traps.
 *   - A context is not thread safe: calls on one context must not overlap on
 *     the host, and work enqueued on different streams for one context must
 *     not overlap on the device (it shares one workspace).
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_VERIFY_API __attribute__((visibility("default")))
#else
#define MOE_VERIFY_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_verify_ctx moe_verify_ctx; /* opaque */

typedef enum {
  MOE_VERIFY_OK = 0,
  MOE_VERIFY_ERR_ARG = -1,         /* bad argument (NULL, size out of range) */
  MOE_VERIFY_ERR_CUDA = -2,        /* a CUDA runtime or driver call failed */
  MOE_VERIFY_ERR_OOM = -3,         /* device memory allocation failed */
  MOE_VERIFY_ERR_ID_RANGE = -4,    /* a token id was outside [0, vocab) */
  MOE_VERIFY_ERR_TIMEOUT = -5,     /* a bounded device wait ran out */
  MOE_VERIFY_ERR_UNSUPPORTED = -6  /* shape or device this build does not run */
} moe_verify_status;

/* Shape of the target stack and the workspace bounds. */
typedef struct {
  int32_t n_layers;     /* L: 1..256 (the decoder: 12) */
  int32_t hidden;       /* d: multiple of 64, <= 8192 (1280) */
  int32_t n_experts;    /* E routed experts: 1..256 (64) */
  int32_t top_k;        /* k: 1..min(E, 16) (6) */
  int32_t n_shared;     /* S shared experts, weight 1: 0..8 (2) */
  int32_t expert_inter; /* I of a routed expert: 1..8192 (896) */
  int32_t shared_inter; /* I of a shared expert: 1..8192 (896) */
  int32_t vocab;        /* V: 2..2^30 (129280) */
  float rms_eps;        /* RMSNorm epsilon, in (0, 1) (1e-6) */
  int32_t max_batch;    /* largest B a step may be given, >= 1 */
  int32_t max_k;        /* largest K (drafts per sequence), 0..15;
                           max_batch * (max_k + 1) <= 4096 (UNSUPPORTED above) */
} moe_verify_config;

/* Weights, all device pointers of bf16 patterns unless noted.  The per-layer
 * members are HOST arrays of n_layers device pointers. */
typedef struct {
  const void* embed;                /* [V, d] token embedding */
  const void* final_norm;           /* [d] gain of the final RMSNorm */
  const void* lm_head;              /* [V, d] */
  const void* const* norm;          /* L x [d] gain of the pre-MoE RMSNorm */
  const void* const* router;        /* L x [E, d] */
  const float* const* router_bias;  /* L x [E] fp32 added to router logits, or NULL */
  const void* const* w_gate;        /* L x [E, I, d] */
  const void* const* w_up;          /* L x [E, I, d] */
  const void* const* w_down;        /* L x [E, d, I] */
  const void* const* s_gate;        /* L x [S, Is, d]  (NULL when S == 0) */
  const void* const* s_up;          /* L x [S, Is, d] */
  const void* const* s_down;        /* L x [S, d, Is] */
} moe_verify_weights;

/* Optional device outputs for tests and diagnostics (caller-owned; any member
 * may be NULL; pass NULL for the whole struct in timed runs).  T = B*(K+1)
 * verify tokens in sequence-major order. */
typedef struct {
  int32_t* topk_idx; /* [L, T, k] selected experts, in selection order */
  float* topk_w;     /* [L, T, k] their softmax weights */
  float* hidden;     /* [L+1, T, d] residual stream entering layer l (l = L: after the last) */
  float* logits;     /* [T, V] lm_head logits (step only) */
} moe_verify_probe;

/* Initialise a context: validates the config, allocates the library-owned
 * weights and workspace (sized for max_batch and max_k), copies and repacks
 * the weights into them (the caller may free its weights afterwards) and
 * prepares the TMA descriptors.  Synchronous: returns after the copies on
 * cuda_stream are complete.  Needs a device of compute capability 10.3
 * (sm_103a); other devices give MOE_VERIFY_ERR_UNSUPPORTED.  On error *out is
 * NULL and nothing stays allocated. */
MOE_VERIFY_API int moe_verify_init(const moe_verify_config* config, const moe_verify_weights* weights,
                    void* cuda_stream, moe_verify_ctx** out);

/* Greedy verification of B sequences with K drafts each (the FastMTP
 * paragraph's verify step).  Sequence b's verify tokens are
 *   x_b = [context_ids[b], draft_ids[b*K + 0], ..., draft_ids[b*K + K-1]]
 * and target_ids[b*(K+1) + i] receives the target stack's greedy choice for
 * the token that follows x_b[i].
 *   context_ids  [B] int32: each sequence's last committed token
 *   draft_ids    [B, K] int32 (may be NULL when K == 0)
 *   target_ids   [B, K+1] int32, written
 *   probe        NULL or diagnostics (see moe_verify_probe)
 * 1 <= B <= max_batch, 0 <= K <= max_k.  A verify token outside [0, V) sets
 * the sticky MOE_VERIFY_ERR_ID_RANGE flag and its target is -1.  If a bounded
 * wait of the lm_head launch runs out, every target of the step is -1 (its
 * argmax is incomplete) and the sticky MOE_VERIFY_ERR_TIMEOUT flag is set; a
 * wait of an earlier kernel of the step that runs out sets that flag only. */
MOE_VERIFY_API int moe_verify_step(moe_verify_ctx* ctx, const int32_t* context_ids, const int32_t* draft_ids,
                    int32_t B, int32_t K, int32_t* target_ids, const moe_verify_probe* probe,
                    void* cuda_stream);

/* The acceptance rule (FastMTP paragraph): for each sequence,
 *   n = the length of the longest prefix with draft_ids[b,i] == target_ids[b,i]
 *   committed[b, 0..n] = target_ids[b, 0..n], committed[b, n+1..K] = -1
 *   accept_len[b] = n  (accepted drafts; n+1 tokens are committed)
 * A sequence with a draft or target id outside [0, V) gets accept_len -1 and
 * a row of -1, and sets the sticky MOE_VERIFY_ERR_ID_RANGE flag.
 *   draft_ids [B, K] int32 (may be NULL when K == 0), target_ids [B, K+1]
 *   int32, committed [B, K+1] int32 written, accept_len [B] int32 written.
 * 1 <= B, 0 <= K <= 15 (B is not bounded by max_batch). */
MOE_VERIFY_API int moe_verify_accept(moe_verify_ctx* ctx, const int32_t* draft_ids, const int32_t* target_ids,
                      int32_t B, int32_t K, int32_t* committed, int32_t* accept_len,
                      void* cuda_stream);

/* One decoder block on T tokens with bf16 input and output:
 *   h = h_in;  one block of layer `layer`;  h_out = bf16(h)  (nearest even).
 *   h_in, h_out [T, d] bf16 patterns (may not overlap), 1 <= T <= max_batch *
 *   (max_k + 1).  probe members topk_idx/topk_w/hidden use L = 1 (the hidden
 *   probe gets [2, T, d]: the input and the fp32 output before rounding). */
MOE_VERIFY_API int moe_verify_layer(moe_verify_ctx* ctx, int32_t layer, const void* h_in, int32_t T, void* h_out,
                     const moe_verify_probe* probe, void* cuda_stream);

/* Convenience form of one decode iteration on HOST buffers: packs
 * context_ids [B] and draft_ids [B, K] (any host memory) into a
 * context-owned pinned staging buffer, then on cuda_stream copies them to the
 * device in one copy, runs moe_verify_step and moe_verify_accept, copies
 * accept_len and committed back in one copy, waits for the stream, and
 * unpacks committed [B, K+1] and accept_len [B] into the caller's buffers
 * (the targets stay in a context-owned device buffer).  1 <= B <= max_batch,
 * 0 <= K <= max_k.  Not capturable.  The first call for a given (B, K)
 * captures the device part (both copies, step and accept on the context's
 * own buffers) into a CUDA graph on a library-owned stream; later calls with
 * that shape launch the graph on cuda_stream (up to 16 shapes are kept;
 * others, and calls while per-launch timing is on, enqueue it directly).
 * Calls on one context must not run concurrently. */
MOE_VERIFY_API int moe_verify_decode_host(moe_verify_ctx* ctx, const int32_t* host_context_ids,
                           const int32_t* host_draft_ids, int32_t B, int32_t K,
                           int32_t* host_committed, int32_t* host_accept_len,
                           void* cuda_stream);

/* FastMTP draft head ("Jina AI Releases jina-ocr-v1, a 3.4B MoE Document
 * Parser With Built-In Speculative Decoding", FastMTP paragraph: one dense
 * draft block applied recursively for K steps with constant parameters;
 * "Jina-OCR-v1: ...", Abstract: one draft block shared across the K steps).
 * The pages leave the block's inputs open; reading taken here: from the
 * verifier's final residual h_prev of a sequence's last accepted position and
 * the token t_prev committed there, each step does
 *   h += E[t];  h = block(h);  t = argmax(lm_head . bf16(RMSNorm_f(h)));
 * and emits t.  `ctx` is a context initialised with n_layers = 1 whose
 * layer is the draft block (a dense block is one expert with top_k = 1 and
 * no shared experts: its softmax weight is exactly 1) and whose embed,
 * final_norm and lm_head are the verifier's.
 *   h_prev [B, d] fp32 (16-byte aligned), t_prev [B] int32 (device; ids
 *   outside [0, V) set the sticky MOE_VERIFY_ERR_ID_RANGE flag and give -1
 *   drafts), drafts [B, K] int32 written, hidden_out [K, B, d] fp32 (h after
 *   each step) or NULL.  1 <= B <= max_batch * (max_k + 1), 1 <= K <= 15.
 * Asynchronous on cuda_stream; capturable. */
MOE_VERIFY_API int moe_verify_draft(moe_verify_ctx* ctx, const float* h_prev, const int32_t* t_prev,
                                    int32_t B, int32_t K, int32_t* drafts, float* hidden_out,
                                    void* cuda_stream);

/* The draft head's inputs after moe_verify_step + moe_verify_accept on the
 * verifier's context: for each sequence b, with n = max(accept_len[b], 0),
 *   h_out[b] = the final residual (fp32, before the final RMSNorm) of verify
 *              token b*(K+1) + n of the last step;
 *   t_out[b] = committed[b*(K+1) + n]  (the last committed token).
 * committed [B, K+1], accept_len [B] as written by moe_verify_accept (device);
 * h_out [B, d] fp32 (16-byte aligned), t_out [B] int32 written.  B and K are
 * those of the last step.  Asynchronous on cuda_stream; capturable. */
MOE_VERIFY_API int moe_verify_draft_inputs(moe_verify_ctx* ctx, const int32_t* committed,
                                           const int32_t* accept_len, int32_t B, int32_t K,
                                           float* h_out, int32_t* t_out, void* cuda_stream);

/* Diagnostic (no counterpart in the method): checks the bounded waits that
 * every step kernel uses, without a context.  One thread waits on an
 * mbarrier phase that nothing completes, then on a device flag that nothing
 * sets, each for limit_ns nanoseconds (1e3 <= limit_ns <= 1e9), using the same
 * bounded-wait code as the kernels; nothing faults or traps, the kernel
 * returns when both waits have given up.  On return, elapsed_ns (host, may be
 * NULL) holds the device time of the two waits.  Returns MOE_VERIFY_OK when
 * both waits gave up and raised the timeout bit, MOE_VERIFY_ERR_TIMEOUT
 * never, MOE_VERIFY_ERR_CUDA when a wait did not report (or on a CUDA error),
 * MOE_VERIFY_ERR_ARG for a limit out of range.  Synchronises cuda_stream.
 * Uses a few bytes of file-scope device memory: calls must not overlap. */
MOE_VERIFY_API int moe_verify_check_bounded_wait(int64_t limit_ns, int64_t* elapsed_ns,
                                                 void* cuda_stream);

/* ----------------------------------------------------------------------
 * The stack with attention (NEXT step after the verify path above).  The
 * pages name the decoder ("Jina AI Releases jina-ocr-v1, a 3.4B MoE Document
 * Parser With Built-In Speculative Decoding", architecture paragraph: 12
 * layers, position limit 32,768) but give no attention shape; the reading
 * implemented here: each block is pre-norm multi-head attention, then the MoE
 * block,
 *   h += W_o . attn(bf16(RMSNorm_a(h) * g_a));   then the MoE block above,
 * with n_heads heads of width hd = d / n_heads, no biases, rotary position
 * embedding on q and k (dims i and i + hd/2 of a head turned by the angle
 * pos * theta^(-2i/hd), pos = the token's 0-based index in its sequence),
 * causal attention over positions 0 .. pos with scores q . k / sqrt(hd), and
 * bf16 (nearest even) at the attention RMSNorm output, at k (after the
 * rotation) and v (the key/value cache is bf16), and at the attention output
 * before W_o.  With attention a target depends on the sequence's prefix: the
 * library keeps, per sequence slot b < max_batch, the keys and values of
 * positions 0 .. max_pos-1 of every layer, head-major: element (l, b, head,
 * pos, i) of the key (value) cache at (((l * max_batch + b) * n_heads + head)
 * * max_pos + pos) * hd + i.
 * -------------------------------------------------------------------- */
typedef struct {
  int32_t n_heads;  /* >= 1, hd = d / n_heads one of 16, 32, 64, 128 */
  int32_t max_pos;  /* positions held per sequence slot: 1..32768 */
  float rope_theta; /* > 1 (10000) */
} moe_verify_attn_config;

typedef struct {                  /* HOST arrays of n_layers device pointers, bf16 */
  const void* const* attn_norm;   /* L x [d] gain of the attention RMSNorm */
  const void* const* w_q;         /* L x [d, d] */
  const void* const* w_k;         /* L x [d, d] */
  const void* const* w_v;         /* L x [d, d] */
  const void* const* w_o;         /* L x [d, d] */
} moe_verify_attn_weights;

/* moe_verify_init for the stack with attention: the same config and MoE
 * weights, plus the attention's shape and weights (copied and repacked: the
 * caller's buffers may be freed after the call); allocates the key/value cache
 * of max_batch sequence slots x max_pos positions x n_layers (bf16, 2 x L x
 * max_batch x max_pos x d x 2 bytes, zeroed) and a rotary table (max_pos x
 * hd/2 x 8 bytes).  Returns MOE_VERIFY_ERR_UNSUPPORTED for a head width other
 * than 16, 32, 64 or 128, or for L x max_batch x n_heads x max_pos >= 2^31.  The context then runs moe_verify_step_attn
 * (moe_verify_step, moe_verify_layer, moe_verify_decode_host and
 * moe_verify_draft refuse it with MOE_VERIFY_ERR_ARG); moe_verify_accept,
 * moe_verify_sync_status, the timing calls, moe_verify_set_grid and
 * moe_verify_destroy work as for any context. */
MOE_VERIFY_API int moe_verify_init_attn(const moe_verify_config* config,
                                        const moe_verify_weights* weights,
                                        const moe_verify_attn_config* attn,
                                        const moe_verify_attn_weights* attn_weights,
                                        void* cuda_stream, moe_verify_ctx** out);

/* Greedy verification with attention.  Sequence b (slot b of the cache) has
 * its last committed token at position positions[b] (device int32, >= 0): its
 * verify tokens [context_ids[b], draft_ids[b, 0..K-1]] take positions
 * positions[b] .. positions[b] + K, their keys and values are written there,
 * and each attends to positions 0 .. its own.  Positions below positions[b]
 * must hold the sequence's earlier tokens' keys and values (written by earlier
 * calls; a first call at position 0 needs none).  After moe_verify_accept with
 * n accepted drafts the cache is valid through position positions[b] + n, and
 * the next call for the sequence passes positions[b] + n + 1 (its context id
 * the committed bonus token).  A prompt is taken in by calls whose drafts are
 * the prompt's next tokens: the cache then holds the prompt's tokens through
 * positions[b] + K whatever the targets.  Outputs and limits as
 * moe_verify_step (probe->hidden, when given, receives [2L + 1, T, d]: row 2l
 * the residual stream entering block l's attention, row 2l + 1 entering its
 * MoE part, row 2L after the last block).
 * A sequence with positions[b] < 0 or positions[b] + K >= max_pos sets the
 * sticky MOE_VERIFY_ERR_ID_RANGE flag, writes nothing to the cache and gets
 * targets -1.  Asynchronous on cuda_stream; capturable. */
MOE_VERIFY_API int moe_verify_step_attn(moe_verify_ctx* ctx, const int32_t* context_ids,
                                        const int32_t* draft_ids, const int32_t* positions,
                                        int32_t B, int32_t K, int32_t* target_ids,
                                        const moe_verify_probe* probe, void* cuda_stream);

/* Diagnostic: the device address of the key/value cache of a context with
 * attention, for reading it: *k_cache and *v_cache receive bf16 arrays
 * [L, max_batch, n_heads, max_pos, hd] in the layout above.  The memory belongs
 * to the context.  Returns MOE_VERIFY_ERR_ARG for a context without attention. */
MOE_VERIFY_API int moe_verify_kv_cache(moe_verify_ctx* ctx, const void** k_cache,
                                       const void** v_cache);

/* Waits for the device, then returns and clears the sticky device error:
 * MOE_VERIFY_OK, MOE_VERIFY_ERR_ID_RANGE, MOE_VERIFY_ERR_TIMEOUT or
 * MOE_VERIFY_ERR_CUDA. */
MOE_VERIFY_API int moe_verify_sync_status(moe_verify_ctx* ctx);

/* Frees everything the context owns (synchronises the device first).  NULL
 * is allowed. */
MOE_VERIFY_API void moe_verify_destroy(moe_verify_ctx* ctx);

/* Static description of a status code; never NULL. */
MOE_VERIFY_API const char* moe_verify_strerror(int status);

/* Host-only checks, usable without a GPU. */

/* MOE_VERIFY_OK when the config is one this build runs, else an error code
 * (ARG for out-of-range fields, UNSUPPORTED for shapes the kernels do not
 * tile). */
MOE_VERIFY_API int moe_verify_check_config(const moe_verify_config* config);

/* Bytes of device memory moe_verify_init allocates for this config (weights
 * plus workspace), or 0 for an invalid config. */
MOE_VERIFY_API uint64_t moe_verify_device_bytes(const moe_verify_config* config);

/* Per-launch time of the library's kernel families, for profiling.
 * moe_verify_set_timing(ctx, 1) makes later steps record CUDA events around
 * each launch of the library's kernels on the step's stream (this breaks
 * graph capture and the overlap of consecutive kernels: use it outside
 * capture, for per-kernel times only).  moe_verify_get_timing synchronises
 * and reports the sums since the last reset, in milliseconds, and the launch
 * counts:
 *   ms[0], n[0]: expert FFN (gate/up + SwiGLU + down + weighted combine)
 *   ms[1], n[1]: attention sub-block (attention RMSNorm, q/k/v and output
 *                projections, attention; contexts with attention only)
 *   ms[2], n[2]: lm_head + argmax        ms[3], n[3]: routing + final RMSNorm
 * (a step run by the single-kernel layer counts its layers' routing with the
 * expert FFN).  reset != 0 clears the sums afterwards. */
MOE_VERIFY_API int moe_verify_set_timing(moe_verify_ctx* ctx, int32_t enable);
MOE_VERIFY_API int moe_verify_get_timing(moe_verify_ctx* ctx, double* ms /*[4] host*/, int64_t* n /*[4] host*/,
                          int32_t reset);

/* Diagnostic (no counterpart in the method): the number of CTAs that later
 * calls give the persistent kernels (the expert FFN and the lm_head); 0, the
 * initial value, means one per SM.  0 <= ctas <= 8 x the SM count.  Results do
 * not depend on it, bit for bit: fewer CTAs than SMs is what a context that
 * holds only part of the GPU runs with, and more CTAs than fit on the GPU at
 * once shows that no CTA waits for one that has not started (every expert-FFN
 * work item is claimed in order by a running CTA).  With attention it also
 * sets the CTAs of the projections (at most one per work item) and of the
 * attention (default one per SM).  Host-buffer decode graphs
 * already captured keep the grid they were captured with. */
MOE_VERIFY_API int moe_verify_set_grid(moe_verify_ctx* ctx, int32_t ctas);

/* The single-kernel layer for the batch-1 operating point (throughput
 * paragraph of "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser With
 * Built-In Speculative Decoding": at batch 1 on an L4, CUDA graphs take greedy
 * decoding from 42.7 to 158.3 tokens/s, so launches bound that point).
 * moe_verify_step and moe_verify_decode_host calls of at most max_tokens
 * verify tokens (B x (K + 1)) run each layer as one launch of the persistent
 * expert-FFN kernel: its first work items route one token each (the routing
 * kernel's arithmetic in the same order, so results are the same bit for bit)
 * while the other CTAs stream their first weight tiles; every CTA then takes
 * expert items.  Each wait in it is for a lower work item, claimed by a
 * running CTA, and gives up after 2 s like the others (timeout status).
 * 0 <= max_tokens <= 8; 0, the initial value, turns it off (a routing
 * launch and an expert-FFN launch per layer): on one GB300 the two launches
 * are faster (0.548 against 0.577 ms for the 12-layer step at B = 1, K = 3).  It applies where the router
 * weights (E x d bf16) fit in the kernel's shared-memory ring and d <= 2048;
 * moe_verify_layer, moe_verify_draft and moe_verify_step_attn always run the
 * two launches.  Host-buffer decode graphs already captured keep the setting
 * they were captured with.  MOE_VERIFY_ERR_ARG for max_tokens outside 0..8. */
MOE_VERIFY_API int moe_verify_set_layer_kernel(moe_verify_ctx* ctx, int32_t max_tokens);

/* Profiling (no counterpart in the method): launch timestamps inside later
 * moe_verify_step (moe_verify_step_attn) calls, for timing kernels in a
 * graph-replayed step without breaking the overlap of consecutive launches.
 * stamps is a device array of (2 L + 1) x 4 uint64 ((6 L + 1) x 4 for a context
 * with attention; 8-byte aligned, caller-owned), or NULL to stop.  Launch j of
 * a step (routing of layer l: j = 2l; expert FFN of layer l: j = 2l + 1;
 * lm_head: j = 2L; with attention: attention RMSNorm 6l, q/k/v projection
 * 6l + 1, attention 6l + 2, output projection 6l + 3, routing 6l + 4, expert
 * FFN 6l + 5, lm_head 6L) updates stamps[4j + 0] = min over its CTAs of
 * the start time, stamps[4j + 1] = max of the time its wait for the
 * preceding launch returned, stamps[4j + 2] = max of the end time (global
 * timer, ns); stamps[4j + 3] is unused.  The caller sets stamps[4j] to
 * UINT64_MAX and the others to 0 before each step it wants to read.  The
 * pointer is recorded in graphs captured while it is set. */
MOE_VERIFY_API int moe_verify_set_stamps(moe_verify_ctx* ctx, uint64_t* stamps);

/* ----------------------------------------------------------------------
 * Greedy head without allocation.  The pages have no counterpart of this
 * entry point: it exists for callers that cannot allocate device memory,
 * such as code whose device memory belongs to another allocator with a fixed
 * budget, code that must not stall other streams (cudaMalloc and cudaFree
 * can synchronise the device), or code running where CUDA allocation calls
 * are not allowed.
 *
 * It computes, for T residual-stream rows h [T, d] (fp32, device):
 *   target_ids[t] = argmax_v bf16(RMSNorm(h[t]) * g) . W_lm[v]   (lowest v on ties)
 * with final_norm g [d] and lm_head W_lm [V, d] as bf16 device arrays
 * (h and lm_head 16-byte aligned), the same kernels as moe_verify_step's
 * last stage.
 * target_ids [T] int32 (device) is written.  If any part of the call's
 * lm_head gives up a bounded wait, every row of that call is -1: this entry
 * point has no context and no sticky status, so the -1 rows are the report.
 * The next call starts afresh (the call clears its status before it runs).
 *
 * Its scratch (normalised rows, argmax keys, a completion counter) is a
 * fixed array of about 1 MB in the library's device memory; every GPU that
 * loads the library holds it until the process exits.  The call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine) and
 * enqueues two kernels on cuda_stream.  Limits: 1 <= T <= 256 and
 * 64 <= d <= 2048 with d a multiple of 64; larger sizes are rejected with
 * MOE_VERIFY_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     the call clears what must start at zero.  Calls that overlap on the GPU
 *     (other streams, other host threads) race on it and give wrong results.
 * -------------------------------------------------------------------- */
#define MOE_VERIFY_NOALLOC_MAX_TOKENS 256
#define MOE_VERIFY_NOALLOC_MAX_HIDDEN 2048
MOE_VERIFY_API int moe_verify_greedy_head_noalloc(const float* h, const void* final_norm,
                                                  const void* lm_head, int32_t T, int32_t d,
                                                  int32_t V, float rms_eps, int32_t* target_ids,
                                                  void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
