// Internal interface between the host API (api.cu) and the kernels
// (route.cu, gemm.cu, misc.cu).  Not part of the C ABI.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mv {

// Launch timestamps for profiling inside a graph-replayed step (global timer,
// ns): slot[0] = earliest CTA start (atomicMin), slot[1] = latest return from
// the wait for the preceding kernel (atomicMax), slot[2] = latest CTA end
// (atomicMax).  The caller initialises slot[0] to ~0 and the others to 0.
constexpr int kStampSlots = 4;

// Bits of the device status word.
constexpr uint32_t kErrIdRange = 1u;
constexpr uint32_t kErrTimeout = 2u;
constexpr uint32_t kErrInternal = 4u;

// Sources of the residual stream entering a routing kernel.
// kSrcEmbedAdd: the running state h (written by the previous launch) plus
// the embedding of each sequence's token (the draft head's step input).
// kSrcH: h as it stands (the stack with attention: the attention sub-block
// has already added its output to h).
enum RouteSrc : int { kSrcEmbed = 0, kSrcBf16 = 1, kSrcCombine = 2, kSrcEmbedAdd = 3, kSrcH = 4 };

struct RouteParams {
  int T, B, K;          // verify tokens, sequences, drafts per sequence
  int d, E, k, S, V;
  int tpb;              // tokens per block: 1, 2, 4 or 8
  int wr_smem;          // 1: router weights staged in shared memory
  float eps;
  int src;              // RouteSrc
  const int32_t* context_ids;
  const int32_t* draft_ids;
  const __nv_bfloat16* embed;  // [V, d]
  const __nv_bfloat16* h_in;   // [T, d] (kSrcBf16)
  float* h;                    // [T, d] residual stream (fp32)
  const float* y;              // [T, k+S, d] expert outputs of the previous block
  const float* gain;           // [d]
  const __nv_bfloat16* Wr;     // [E, d]
  int wr_row;                  // first row of this layer's router in the router tensor map
  const float* bias;           // [E] or nullptr
  int32_t* bad;                // [T]
  uint32_t* status;
  int32_t* probe_idx;          // [T, k] or nullptr
  float* probe_w;              // [T, k] or nullptr
  float* probe_hidden;         // [T, d] or nullptr
  // expert-major rows: expert e owns rows [e*T, e*T + cnt[e])
  int32_t* cnt;                // [E] rows claimed per routed expert (zero on entry)
  // cleared after the wait (the kernels that used them are complete): the
  // other parity's expert counters, the previous expert-FFN launch's
  // dependency counters, and the other parity's item counter (the next
  // expert-FFN launch claims from it, before its own wait)
  int32_t* cnt_other;          // [E]
  int32_t* dep_clear;          // [n_dep_clear]
  int n_dep_clear;
  int32_t* next_item_clear;
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
  __nv_bfloat16* xperm;        // [(E+S)*T, d] normalised inputs
  int32_t* perm_token;         // [(E+S)*T] token of each row
  int32_t* perm_slot;          // [(E+S)*T] its slot: routed rank, or k + s
  float* perm_w;               // [(E+S)*T] combine weight (1 for shared)
};

// The layer's expert FFN in one persistent kernel: gate/up + SwiGLU items for
// every (expert, 128-row tile, chunk of <= nch rows), then the down items.
struct FfnParams {
  const int32_t* cnt;          // [E] routed rows per expert (shared experts: T)
  int32_t* dep;                // [chunks] finished gate/up halves per chunk (zero on entry)
  int E, S, T, nch;
  int mt_gu, mt_dn;            // items per chunk: gate/up, down (the weight-major form: the
                               // expert's 128-row weight tiles; token-major: 256-row tiles)
  int tile_gu, tile_dn;        // 128-row weight tiles per expert in the tensor maps
  int kb_gu, kb_dn;            // 64-wide K blocks: d/64 and I_pad/64
  int a_base_gu, a_base_dn;    // first weight row of this layer in the tensor maps
  int stages, tmem_cols;
  __nv_bfloat16* a_out;        // [(E+S)*T, I_pad] SwiGLU rows
  int I_pad;
  const int32_t* perm_token;
  const int32_t* perm_slot;
  const float* perm_w;
  float* y;                    // [T, kS, d]
  int d, kS;
  uint32_t* status;
  int* next_item;              // items claimed so far, every CTA's first included (zero on entry)
  // L2 prefetch of the next kernel's first weight item of this CTA index c,
  // issued once this CTA has no items left, for c < pf_limit, pf_kb 64-column
  // boxes of the prefetch tensor map: pf_items = 1, the next layer's gate/up
  // item c as guessed for the first items (pf_base = that layer's first
  // gate/up row); pf_items = 0, rows pf_base + (c / pf_div) * 128
  int pf_base, pf_div, pf_limit, pf_kb, pf_items;
  int pf_pair;                 // 1: the next kernel is the lm_head on CTA pairs (rows per pair item)
  // Items run shared experts first, so the first items' weights are known
  // before the routing for the shared experts always, and for the routed
  // experts when each holds one chunk: spec = 2 guesses both, 1 the shared
  // experts' items only, 0 none.
  int spec;
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
  // The single-kernel layer (a few verify tokens): n_route > 0 makes the
  // first n_route tickets route one token each (rt, with rt.stamps the
  // routing's timer slots) before any expert item runs; next_item is then the
  // layer's own ticket counter (cleared by the step's final kernel), and
  // route_done counts the tokens routed (zero on entry; the first routing
  // task clears route_done_clear, the other parity's).
  int n_route;
  RouteParams rt;
  int32_t* route_done;
  int32_t* route_done_clear;
};

struct FinalParams {
  int T, d, kS;                // kS = k + S slots per token
  float eps;
  int mode;                    // 0: final RMSNorm -> xf;  1: h_out = bf16(h)
  float* h;                    // [T, d]
  const float* y;              // [T, kS, d]
  const float* gain;           // [d]
  __nv_bfloat16* out;          // mode 0: xf [T, d]; mode 1: h_out [T, d]
  float* probe_hidden;         // [T, d] or nullptr
  unsigned long long* keys;    // [T] argmax keys, cleared in mode 0
  int32_t* cnt_clear;          // [n_cnt_clear] expert counters of the last layer, cleared
  int n_cnt_clear;
  int32_t* item_clear;         // item counter of the last layer's expert FFN, cleared
  int32_t* route_done_clear;   // routed-token counter of the last layer, cleared (or nullptr)
  int32_t* layer_items_clear;  // [n_layer_items] the single-kernel layers' ticket counters, cleared
  int n_layer_items;
};

// The lm_head GEMM with its argmax epilogue.
struct GemmParams {
  int n_items_static;          // vocabulary tiles (of 128) x token chunks
  int kblocks;                 // d / 64
  int nch;                     // token rows loaded per stage (multiple of 16)
  int stages;
  int tmem_cols;
  uint32_t* status;
  int T, V, n_chunks, nch_lm;  // token chunks of nch_lm (= nch) rows
  unsigned long long* keys;    // [T]
  float* logits;               // [T, V] or nullptr
  int32_t* targets;            // [T]
  const int32_t* bad;          // [T]
  unsigned int* done;          // CTAs finished with this launch (the last one resets it)
  unsigned int* aborted;       // CTAs of this launch whose bounded wait ran out (reset with done)
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
};

// ------------------------------------------------ the stack with attention
//
// Per block: attn_norm (residual update + attention RMSNorm), the q/k/v
// projection (RoPE and the key/value cache write in its epilogue), the
// attention over the cache, the output projection added into h, then the
// routing (source kSrcH) and the expert FFN as without attention.

// Residual stream entering block l's attention and its normalised bf16 row.
// Layer 0 also checks the ids and the positions (bad[t] = 1 and the status
// bit for a token outside [0, V) or a sequence outside [0, max_pos - K)) and
// lays out the attention's work items for the step.
struct AttnNormParams {
  int T, B, K, d, kS, V, H, max_pos;
  int first;                   // 1: layer 0 (h = embedding of the token), 0: h += combine(y)
  float eps;
  const int32_t* context_ids;
  const int32_t* draft_ids;
  const int32_t* positions;    // [B]
  const __nv_bfloat16* embed;  // [V, d]
  float* h;                    // [T, d]
  const float* y;              // [T, kS, d] expert outputs of the previous block
  const float* gain;           // [d]
  __nv_bfloat16* xa;           // [T, d] bf16(RMSNorm_a(h) * g_a)
  float* probe_hidden;         // [T, d] or nullptr
  int32_t* bad;                // [T]
  uint32_t* status;
  // work items of the attention (written by layer 0's block 0): plan[0] =
  // keys per split, plan[1] = (sequence, split) pairs, then the pairs in claim
  // order as plan[2 + 2i] = sequence, plan[3 + 2i] = split, then from plan[2 +
  // 2 cap_pairs] each sequence's first split slot (the splits before it)
  int32_t* plan;
  int target_items;            // wanted (sequence, split, head) items
  int max_split;               // attn_max_split(hd): keys per chunk
  int cap_pairs;               // room in plan for pairs
  int32_t* item_ctr;           // [n_item_ctr] the attention's item counters (one per layer), cleared
  int n_item_ctr;
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
};

// Weight-major projection on the tensor cores: items are (128 weight rows,
// chunk of <= nch tokens); mode 0 is the packed q/k/v projection (rows
// [q | k | v], q and k rows of a head ordered (0, hd/2, 1, hd/2 + 1, ...) so
// that each rotary pair sits in neighbouring lanes), mode 1 W_o added into h.
struct ProjParams {
  int mode;
  int n_items, n_chunks, nch;  // weight tiles x token chunks; tokens per chunk
  int a_row0;                  // first weight row of this layer in the tensor map
  int kblocks, stages, tmem_cols;
  int T, d, K, H, hd, max_pos, Bmax;
  uint32_t* status;
  const int32_t* positions;    // [B] (mode 0)
  const float2* rope;          // [max_pos, hd/2] (cos, sin) (mode 0)
  float* q;                    // [T, d] rotated q (mode 0)
  __nv_bfloat16* kc;           // this layer's key cache [Bmax, H, max_pos, hd] (mode 0)
  __nv_bfloat16* vc;           // this layer's value cache (mode 0)
  float* h;                    // [T, d] (mode 1)
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
};

// Causal attention of the step's tokens over their sequences' caches.  Items
// (sequence, split of <= plan[0] keys, head); a sequence's keys 0 .. pos + K
// in splits, each split's unnormalised result merged by the last of its
// sequence's and head's items to finish.
struct AttnParams {
  int B, K, H, hd, d, max_pos, Bmax;
  int row0;                    // this layer's first row in the cache tensor maps
  int max_split;               // attn_max_split(hd): keys per chunk (shared-memory buffer)
  float scale_log2;            // log2(e) / sqrt(hd)
  const int32_t* positions;    // [B]
  const int32_t* plan;
  const float* q;              // [T, d]
  const __nv_bfloat16* kc;     // this layer's caches [Bmax, H, max_pos, hd]
  const __nv_bfloat16* vc;
  __nv_bfloat16* o;            // [T, d] bf16 attention output
  float* part;                 // [cap items, K+1, hd + 2] split results (m, l, acc)
  int32_t* arrive;             // [Bmax, H] finished splits (zero on entry; the merger resets)
  int32_t* item_ctr;           // items claimed so far (zero on entry: cleared by layer 0's attn_norm)
  int cap_pairs;               // room in plan for pairs (the per-sequence slots follow them)
  uint32_t* status;
  unsigned long long* stamps;  // nullptr, or this launch's [start, ready, end] timer slots
};
constexpr int kAttnMinSplit = 64;    // keys per split: at least
constexpr int kAttnMaxSplit = 1024;  // and at most
constexpr int kAttnMaxSplits = 64;   // splits of one sequence: at most (32,768 / 64 <= 1,024)
// keys per chunk (the attention kernel's shared-memory buffer holds at most
// 16,384 key elements, 32 KB of keys and as much of values, in TMA boxes of
// at most 256 rows): 128 keys of 128 dims, 256 keys of 64 or fewer
__host__ __device__ inline int attn_max_split(int hd) {
  const int c = 16384 / hd;
  return c > 256 ? 256 : c;
}

struct AcceptParams {
  int B, K, V;
  const int32_t* drafts;
  const int32_t* targets;
  int32_t* committed;
  int32_t* accept_len;
  uint32_t* status;
};

// Shared memory the GEMM kernels need for a given item width and stage count.
size_t gemm_smem_bytes(int nch, int stages);
int gemm_max_stages(int nch);
size_t ffn_tokm_smem_bytes(int stages);
int ffn_tokm_max_stages();
size_t route_smem_bytes(int tpb, int d, int E, int k, int S, bool wr_smem);
bool route_wr_fits(int tpb, int d, int E, int k, int S);

// Launchers (enqueue only).  `pdl` requests programmatic dependent launch.
cudaError_t launch_route(const CUtensorMap& map_wr, const RouteParams& p, int grid, size_t smem,
                         cudaStream_t s, bool pdl);
// Steps of at most this many verify tokens may route inside the expert-FFN
// kernel (the single-kernel layer; off unless the caller sets it).
constexpr int kFuseMaxT = 8;

// p.n_route > 0: the single-kernel layer, routing with the router map map_wr
// (64-column boxes of E rows, 128-byte swizzle) in the shared memory of the
// ring (ffn_route_fits).
cudaError_t launch_ffn(const CUtensorMap& map_gu, const CUtensorMap& map_x,
                       const CUtensorMap& map_dn, const CUtensorMap& map_a,
                       const CUtensorMap& map_pf, const CUtensorMap& map_wr, const FfnParams& p,
                       int grid, cudaStream_t s, bool pdl);
// Whether a routing task of the single-kernel layer (router weights, gain,
// one normalised row, logits) fits in the ring of `stages` stages of nch rows.
bool ffn_route_fits(int nch, int stages, int d, int E, int k, int S);
// The token-major form of the layer's expert FFN (large T): 128 of an
// expert's rows on the MMA's M side, 256 weight rows on N.  map_gu256 and
// map_dn256 are the weight maps with 256-row boxes, map_x and map_a the
// activation maps with 128-row boxes.  Needs tile_gu even.
constexpr int kTokmChunk = 128;
cudaError_t launch_ffn_tokm(const CUtensorMap& map_gu256, const CUtensorMap& map_x,
                            const CUtensorMap& map_dn256, const CUtensorMap& map_a,
                            const FfnParams& p, int grid, cudaStream_t s, bool pdl);
// The lm_head launch for T tokens: tokens on the MMA's M side for 65..128
// tokens (one chunk); above kLmPairMinT tokens on CTA pairs (256 vocabulary
// rows x chunks of 256 tokens, each CTA loading half of each); else
// vocabulary rows on M with chunks of <= 256 tokens.  Pairs measured faster
// from 136 tokens on (136: 59.5 -> 57.4 us, 192: 67.4 -> 59.6 us, 256: 86.3
// -> 60.6 us per launch).
constexpr int kLmPairMinT = 128;
struct LmLayout {
  bool tokens_on_m, pair;
  int nch, n_chunks, tmem_cols, stages;
};
LmLayout lm_layout(int T);
// The single-CTA layout for T tokens (whatever T; the form lm_layout picks
// for T <= kLmPairMinT, and the fallback when no CTA pair fits).
LmLayout lm_layout_single(int T);
// CTA pairs of the lm_head that fit on the GPU at once (0: none).
int lmhead_pair_max_clusters(int stages);
// map_x128: the final normalised rows with 128-row boxes; grid = 2 * pairs.
cudaError_t launch_lmhead_pair(const CUtensorMap& map_w, const CUtensorMap& map_x128,
                               const GemmParams& p, int pairs, cudaStream_t s, bool pdl);
cudaError_t launch_lmhead(const CUtensorMap& map_w, const CUtensorMap& map_x, const GemmParams& p,
                          bool tokens_on_m, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t s);

// Draft head plumbing: h_out[b] = h[b*(K+1) + n_b], t_out[b] =
// committed[b*(K+1) + n_b] with n_b = max(accept_len[b], 0).
cudaError_t launch_draft_inputs(const float* h, const int32_t* committed, const int32_t* accept_len,
                                int B, int K, int d, float* h_out, int32_t* t_out, cudaStream_t s);
// dst[b * stride + col] = src[b], b < B.
cudaError_t launch_scatter_column(const int32_t* src, int B, int32_t* dst, int stride, int col,
                                  cudaStream_t s);

// The stack with attention.
cudaError_t launch_attn_norm(const AttnNormParams& p, cudaStream_t s, bool pdl);
size_t proj_smem_bytes(int nch, int stages);
cudaError_t launch_proj(const CUtensorMap& map_w, const CUtensorMap& map_x, const ProjParams& p,
                        int grid, cudaStream_t s, bool pdl);
size_t attn_smem_bytes(int hd, int nq);
// map_k, map_v: the key and value caches as 2-D bf16 tensors [L * Bmax * H *
// max_pos rows, hd], boxes of min(hd, 64) x attn_max_split(hd) with the swizzle
// of the box's row bytes (128, 64 or 32).  hd is 16, 32, 64 or 128.
cudaError_t launch_attn(const CUtensorMap& map_k, const CUtensorMap& map_v, const AttnParams& p,
                        int grid, cudaStream_t s, bool pdl);
// dst [rows_pad, d] = the packed q/k/v rows of one layer (zero past 3d).
cudaError_t launch_repack_qkv(__nv_bfloat16* dst, const __nv_bfloat16* wq,
                              const __nv_bfloat16* wk, const __nv_bfloat16* wv, int d, int hd,
                              int rows_pad, cudaStream_t s);

// Self-check of the bounded waits (see moe_verify_check_bounded_wait).
cudaError_t run_bounded_wait_check(uint64_t limit_ns, cudaStream_t s, unsigned long long* host_out,
                                   uint32_t* host_status);

// Weight repacking (init only).
cudaError_t launch_repack_gateup(__nv_bfloat16* dst, const __nv_bfloat16* gate,
                                 const __nv_bfloat16* up, const __nv_bfloat16* s_gate,
                                 const __nv_bfloat16* s_up, int E, int S, int I, int Is, int d,
                                 int mt_gu, cudaStream_t s);
cudaError_t launch_repack_down(__nv_bfloat16* dst, const __nv_bfloat16* down,
                               const __nv_bfloat16* s_down, int E, int S, int I, int Is, int d,
                               int I_pad, int mt_dn, cudaStream_t s);
cudaError_t launch_bf16_to_f32(float* dst, const __nv_bfloat16* src, int64_t n, cudaStream_t s);

}  // namespace mv
