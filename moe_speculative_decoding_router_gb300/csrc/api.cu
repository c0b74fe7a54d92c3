// Host side of the C ABI declared in include/moe_verify.h: argument checks,
// library-owned weights and workspace, TMA descriptors and the launch order
// of one verify step.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <cstring>
#include <vector>

#include "moe_verify.h"
#include "internal.h"


struct TimingPair {
  int family;
  cudaEvent_t a, b;
};

struct moe_verify_ctx {
  moe_verify_config cfg;
  int device = 0, num_sms = 0;
  int L = 0, d = 0, E = 0, k = 0, S = 0, I = 0, Is = 0, V = 0;
  int nE = 0, kS = 0, I_pad = 0, d_pad = 0, V_pad = 0, mt_gu = 0, mt_dn = 0;
  int T_max = 0, rows_max = 0, chunks_cap = 0;
  // library-owned weights
  __nv_bfloat16 *w_gu = nullptr, *w_dn = nullptr, *w_lm = nullptr, *embed = nullptr,
                *router = nullptr;
  float *gain = nullptr, *final_gain = nullptr, *bias = nullptr;
  bool has_bias = false;
  // workspace
  float* h = nullptr;
  float* y = nullptr;
  __nv_bfloat16 *xperm = nullptr, *abuf = nullptr, *xf = nullptr;
  int32_t *bad = nullptr, *perm_token = nullptr, *perm_slot = nullptr, *cnt = nullptr,
          *dep = nullptr;
  float* perm_w = nullptr;
  unsigned int *done_ffn = nullptr, *done_lm = nullptr;
  // the single-kernel layer: routed tokens [2] by parity, and each layer's
  // ticket counter [L] (cleared by the step's final kernel)
  int32_t* route_ctr = nullptr;
  int32_t* layer_items = nullptr;
  unsigned long long* keys = nullptr;
  uint32_t* status = nullptr;
  int32_t *io_ctx = nullptr, *io_drafts = nullptr, *io_targets = nullptr, *io_committed = nullptr,
          *io_alen = nullptr;
  // host-buffer decode: ids in [B + B K] and accept_len + committed out
  // [B + B (K + 1)], on the device and in a pinned host staging buffer
  // (stage: T_max ints in, then T_max + max_batch out)
  int32_t* io_out = nullptr;
  int32_t* stage = nullptr;
  CUtensorMap map_gu, map_dn, map_lm, map_wr;
  // the expert weights with 256-row boxes (the token-major expert FFN)
  CUtensorMap map_gu256, map_dn256;
  std::vector<void*> allocs;
  // host-buffer decode: one captured graph (step + accept) per (B, K)
  struct DecodeGraph {
    int B, K;
    cudaGraphExec_t exec;
  };
  std::vector<DecodeGraph> decode_graphs;
  cudaStream_t capture_stream = nullptr;
  // CTAs of the persistent kernels (expert FFN, lm_head); 0: one per SM
  int grid_ctas = 0;
  // steps of at most this many verify tokens route inside the expert-FFN
  // kernel (one launch per layer); 0: off.  Off by default: measured on the
  // 12-layer step at B = 1, K = 3, 0.577 ms per step against 0.548 ms with a
  // routing launch per layer (its routing tasks and expert phase each take
  // ~1.5 us longer than in the two launches, more than the handoff it saves)
  int fuse_max_T = 0;
  int lm_pair_max = 0;  // lm_head CTA pairs that fit on the GPU at once
  // the stack with attention (moe_verify_init_attn)
  bool attn = false;
  int H = 0, hd = 0, max_pos = 0, rows_qkv = 0, cap_pairs = 0, attn_target = 0;
  __nv_bfloat16 *w_qkv = nullptr, *w_o = nullptr, *kcache = nullptr, *vcache = nullptr,
                *xa = nullptr, *obuf = nullptr;
  float *attn_gain = nullptr, *qbuf = nullptr, *part = nullptr;
  float2* rope = nullptr;
  int32_t *arrive = nullptr, *plan = nullptr, *attn_ctr = nullptr;
  CUtensorMap map_qkv, map_wo, map_kc, map_vc;
  // profiling
  unsigned long long* stamps = nullptr;  // caller-owned [2L + 1][kStampSlots] or nullptr
  bool timing = false;
  std::vector<TimingPair> pending;
  std::vector<cudaEvent_t> event_pool;
  double ms[4] = {0, 0, 0, 0};
  int64_t launches[4] = {0, 0, 0, 0};
};

namespace {

#define CK(x)                                   \
  do {                                          \
    cudaError_t _e = (x);                       \
    if (_e != cudaSuccess) return MOE_VERIFY_ERR_CUDA; \
  } while (0)

int round_up(int x, int m) { return (x + m - 1) / m * m; }

int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

struct Derived {
  int nE, kS, I_pad, d_pad, V_pad, mt_gu, mt_dn, T_max, rows_max, chunks_cap;
};

int check(const moe_verify_config* c) {
  if (!c) return MOE_VERIFY_ERR_ARG;
  if (c->n_layers < 1 || c->n_layers > 256) return MOE_VERIFY_ERR_ARG;
  if (c->hidden < 64 || c->hidden > 8192) return MOE_VERIFY_ERR_ARG;
  if (c->n_experts < 1 || c->n_experts > 256) return MOE_VERIFY_ERR_ARG;
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts) return MOE_VERIFY_ERR_ARG;
  if (c->n_shared < 0 || c->n_shared > 8) return MOE_VERIFY_ERR_ARG;
  if (c->expert_inter < 1 || c->expert_inter > 8192) return MOE_VERIFY_ERR_ARG;
  if (c->shared_inter < 1 || c->shared_inter > 8192) return MOE_VERIFY_ERR_ARG;
  if (c->vocab < 2 || c->vocab > (1 << 30)) return MOE_VERIFY_ERR_ARG;
  if (!(c->rms_eps > 0.f) || !(c->rms_eps < 1.f)) return MOE_VERIFY_ERR_ARG;
  if (c->max_batch < 1 || c->max_k < 0 || c->max_k > 15) return MOE_VERIFY_ERR_ARG;
  if (c->hidden % 64 != 0) return MOE_VERIFY_ERR_UNSUPPORTED;
  const int64_t T_max = (int64_t)c->max_batch * (c->max_k + 1);
  if (T_max > 4096) return MOE_VERIFY_ERR_UNSUPPORTED;
  // a routing block must hold eight tokens' rows when the router weights do
  // not fit in shared memory
  if (mv::route_smem_bytes(8, c->hidden, c->n_experts, c->top_k, c->n_shared, false) >
      227 * 1024)
    return MOE_VERIFY_ERR_UNSUPPORTED;
  return MOE_VERIFY_OK;
}

Derived derive(const moe_verify_config* c) {
  Derived r;
  r.nE = c->n_experts + c->n_shared;
  r.kS = c->top_k + c->n_shared;
  const int Imax = c->expert_inter > c->shared_inter ? c->expert_inter : c->shared_inter;
  r.I_pad = round_up(Imax, 64);
  r.d_pad = round_up(c->hidden, 128);
  r.V_pad = round_up(c->vocab, 128);
  r.mt_gu = r.I_pad / 64;
  r.mt_dn = r.d_pad / 128;
  r.T_max = c->max_batch * (c->max_k + 1);
  r.rows_max = r.T_max * r.nE;  // expert e owns rows [e*T, e*T + count_e)
  // chunks per layer are at most T*k/16 + E (routed) plus S*(T/16 + 1) (shared)
  const int chunks = r.T_max * c->top_k / 16 + c->n_experts + c->n_shared * (r.T_max / 16 + 1);
  r.chunks_cap = chunks;
  return r;
}

struct Sizes {
  uint64_t w_gu, w_dn, w_lm, embed, router, gain, final_gain, bias;
  uint64_t h, y, xperm, abuf, xf, bad, perm, cnt, dep, keys, io;
};

Sizes sizes(const moe_verify_config* c, const Derived& r) {
  Sizes s;
  const uint64_t L = c->n_layers, d = c->hidden, E = c->n_experts, V = c->vocab;
  s.w_gu = L * r.nE * r.mt_gu * 128ull * d * 2;
  s.w_dn = L * r.nE * r.mt_dn * 128ull * r.I_pad * 2;
  s.w_lm = (uint64_t)r.V_pad * d * 2;
  s.embed = V * d * 2;
  s.router = L * E * d * 2;
  s.gain = L * d * 4;
  s.final_gain = d * 4;
  s.bias = L * E * 4;
  s.h = (uint64_t)r.T_max * d * 4;
  s.y = (uint64_t)r.T_max * r.kS * d * 4;
  s.xperm = (uint64_t)r.rows_max * d * 2;
  s.abuf = (uint64_t)r.rows_max * r.I_pad * 2;
  s.xf = (uint64_t)round_up(r.T_max, 16) * d * 2;
  s.bad = (uint64_t)r.T_max * 4;
  s.perm = (uint64_t)r.rows_max * 4;
  s.cnt = (uint64_t)c->n_experts * 4 * 2;  // two parities
  s.dep = (uint64_t)r.chunks_cap * 4;
  s.keys = (uint64_t)r.T_max * 8;
  s.io = (uint64_t)r.T_max * 4;
  return s;
}

uint64_t total_bytes(const Sizes& s) {
  return s.w_gu + s.w_dn + s.w_lm + s.embed + s.router + s.gain + s.final_gain + s.bias + s.h +
         s.y + s.xperm + s.abuf + s.xf + s.bad + 3 * s.perm + s.cnt + s.dep + s.keys + 5 * s.io +
         64;
}

template <typename T>
int dalloc(moe_verify_ctx* c, T** p, uint64_t bytes) {
  void* v = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&v, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? MOE_VERIFY_ERR_OOM : MOE_VERIFY_ERR_CUDA;
  }
  c->allocs.push_back(v);
  *p = static_cast<T*>(v);
  return MOE_VERIFY_OK;
}

// The CUDA driver API's tensor-map encoder, looked up once (a function-local static's
// initialisation is thread safe).
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

// 2-D bf16 tensor [rows, inner] (row-major), boxes of 64 x box_rows with the
// 128-byte swizzle that the tcgen05 shared-memory descriptors expect.
int encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = get_encode();
  if (!fn) return MOE_VERIFY_ERR_CUDA;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_VERIFY_OK : MOE_VERIFY_ERR_CUDA;
}

// 2-D bf16 tensor [rows, inner] read in boxes of box_inner x box_rows with
// the swizzle that matches the box's row bytes (128, 64 or 32).
int encode_map_box(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                   uint32_t box_inner, uint32_t box_rows) {
  auto fn = get_encode();
  if (!fn) return MOE_VERIFY_ERR_CUDA;
  const uint32_t rb = box_inner * 2;
  const CUtensorMapSwizzle sw = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_32B;
  if (rb != 128 && rb != 64 && rb != 32) return MOE_VERIFY_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_VERIFY_OK : MOE_VERIFY_ERR_CUDA;
}

void free_all(moe_verify_ctx* c) {
  for (void* p : c->allocs) cudaFree(p);
  c->allocs.clear();
  if (c->stage) cudaFreeHost(c->stage);
  c->stage = nullptr;
  // timing pairs not yet read back by moe_verify_get_timing are outside the pool
  for (auto& tp : c->pending) {
    cudaEventDestroy(tp.a);
    cudaEventDestroy(tp.b);
  }
  for (cudaEvent_t e : c->event_pool) cudaEventDestroy(e);
  c->event_pool.clear();
  c->pending.clear();
}

// ------------------------------------------------------------- profiling

cudaEvent_t take_event(moe_verify_ctx* c) {
  if (!c->event_pool.empty()) {
    cudaEvent_t e = c->event_pool.back();
    c->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct Timed {
  moe_verify_ctx* c;
  int family;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  Timed(moe_verify_ctx* c_, int f, cudaStream_t s_) : c(c_), family(f), s(s_) {
    if (c->timing) {
      a = take_event(c);
      cudaEventRecord(a, s);
    }
  }
  ~Timed() {
    if (c->timing && a) {
      cudaEvent_t b = take_event(c);
      cudaEventRecord(b, s);
      c->pending.push_back({family, a, b});
    }
  }
};

// --------------------------------------------------------------- launches

// The expert FFN runs token-major (the chunk's rows on the MMA's M side) from
// this many verify tokens on: there each expert holds many rows, and the
// weight-major form's epilogue (columns = rows, gate and up in different
// warps) bounds it.  Measured on the 12-layer step: weight-major is ahead by
// ~1.5% at 256 tokens, token-major by 4.5% at 384 and 10% at 512.
constexpr int kTokmMinT = 320;

struct StepShape {
  int T, tpb, grid_route, nch, stages, tmem_cols, nch_lm, n_chunks_lm;
  bool tokm;
  bool fused;  // the verify step's layers route inside the expert-FFN kernel
  mv::LmLayout lm;
  bool wr_smem;
  size_t route_smem;
  // activation tiles of the expert FFN and the lm_head: one TMA box per stage,
  // as wide as the item's chunk of rows (rows past the buffers read as zeros;
  // rows past an item's own are loaded but never used)
  CUtensorMap map_x, map_a, map_f;
  CUtensorMap map_f128;  // the final rows with 128-row boxes (the lm_head on CTA pairs)
};

// CTA pairs of the lm_head at large T: as many as fit at once (measured once
// per context), at most half the persistent grid.
int lm_pairs(const moe_verify_ctx* c);

int shape_for(const moe_verify_ctx* c, int T, StepShape* out) {
  StepShape& s = *out;
  s.T = T;
  // tokens per routing block: 1, 2 or 4, enough blocks to cover the SMs; past
  // 4 * SMs tokens, two waves of 4-token blocks (whose router weights fit in
  // shared memory) beat one wave of 8-token blocks reading them through L1
  // (1.84 vs 1.90 ms per step at 1,024 tokens)
  const int want = (T + c->num_sms - 1) / c->num_sms;
  s.tpb = want <= 1 ? 1 : want <= 2 ? 2 : 4;
  s.grid_route = (T + s.tpb - 1) / s.tpb;
  // routed experts see about T*k/E rows each; leave headroom for uneven load.
  // Shared experts (every token) are cut into chunks of the same width, so
  // that the shared-memory stages stay small and many of them fit (bytes in
  // flight per SM are what keep HBM busy).
  int avg = (int)((3LL * T * c->k + 2LL * c->E - 1) / (2LL * c->E));
  s.tokm = T >= kTokmMinT && c->mt_gu % 2 == 0;
  s.nch = s.tokm ? mv::kTokmChunk : round_up(avg < 16 ? 16 : avg, 16);
  if (s.nch > 256) s.nch = 256;
  s.stages = s.tokm ? mv::ffn_tokm_max_stages() : mv::gemm_max_stages(s.nch);
  s.lm = mv::lm_layout(T);
  s.n_chunks_lm = s.lm.n_chunks;
  s.nch_lm = s.lm.nch;
  s.tmem_cols = s.tokm ? 512 : pow2_at_least(2 * (s.nch > s.nch_lm ? s.nch : s.nch_lm));
  s.fused = T <= c->fuse_max_T && !s.tokm &&
            mv::ffn_route_fits(s.nch, s.stages, c->d, c->E, c->k, c->S);
  s.wr_smem = mv::route_wr_fits(s.tpb, c->d, c->E, c->k, c->S);
  s.route_smem = mv::route_smem_bytes(s.tpb, c->d, c->E, c->k, c->S, s.wr_smem);
  if (encode_map(&s.map_x, c->xperm, c->d, c->rows_max, (uint32_t)s.nch) ||
      encode_map(&s.map_a, c->abuf, c->I_pad, c->rows_max, (uint32_t)s.nch) ||
      encode_map(&s.map_f, c->xf, c->d, round_up(c->T_max, 16), (uint32_t)s.nch_lm))
    return MOE_VERIFY_ERR_CUDA;
  if (s.lm.pair) {
    // the pair form needs at least one pair that fits; else the single-CTA form
    const int pairs = lm_pairs(c);
    if (pairs < 1) {
      s.lm = mv::lm_layout_single(T);
      s.n_chunks_lm = s.lm.n_chunks;
      s.nch_lm = s.lm.nch;
      s.tmem_cols = s.tokm ? 512 : pow2_at_least(2 * (s.nch > s.nch_lm ? s.nch : s.nch_lm));
      if (encode_map(&s.map_f, c->xf, c->d, round_up(c->T_max, 16), (uint32_t)s.nch_lm))
        return MOE_VERIFY_ERR_CUDA;
    } else if (encode_map(&s.map_f128, c->xf, c->d, round_up(c->T_max, 16), 128)) {
      return MOE_VERIFY_ERR_CUDA;
    }
  }
  return MOE_VERIFY_OK;
}

// Expert counters alternate between two buffers by position in the launch
// sequence (parity): routing kernel n claims rows on buffer n % 2 and clears
// buffer (n + 1) % 2, whose users are complete by then; the final kernel
// clears the buffer of the last layer.  The expert FFN's item counters
// alternate the same way: expert-FFN launch n claims on counter n % 2 from
// its first instruction, routing kernel n clears counter (n + 1) % 2 (last
// used by launch n - 1, complete by then, and next used by launch n + 1,
// which starts only after routing kernel n + 1 is past its wait), and the
// final kernel clears the last layer's.
int32_t* item_counter(moe_verify_ctx* c, int parity) {
  return reinterpret_cast<int32_t*>(c->done_ffn + 1 + parity);
}

int persistent_grid(const moe_verify_ctx* c) { return c->grid_ctas > 0 ? c->grid_ctas : c->num_sms; }

int lm_pairs(const moe_verify_ctx* c) {
  const int want = persistent_grid(c) / 2;
  return want < c->lm_pair_max ? want : c->lm_pair_max;
}

// Timer slots of launch `slot` of a step (routing of layer l: 2l, expert FFN
// of layer l: 2l + 1, lm_head: 2L; with attention: attention RMSNorm 6l,
// q/k/v projection 6l + 1, attention 6l + 2, output projection 6l + 3,
// routing 6l + 4, expert FFN 6l + 5, lm_head 6L), or nullptr when stamps are
// off or the launch is not part of a step (slot < 0).
unsigned long long* stamp_slot(const moe_verify_ctx* c, int slot) {
  return (c->stamps && slot >= 0) ? c->stamps + (size_t)slot * mv::kStampSlots : nullptr;
}

// next_head: the lm_head follows this layer (its first items are prefetched
// into L2 at the end of the expert FFN, as the next layer's are otherwise).
int run_layer(moe_verify_ctx* c, int l, int parity, int src, const StepShape& sh,
              const int32_t* context_ids, const int32_t* draft_ids, int B, int K,
              const void* h_in, const moe_verify_probe* probe, int probe_layer, cudaStream_t s,
              bool pdl, bool next_head, int stamp_base = -1) {
  const int T = sh.T;
  mv::RouteParams rp = {};
  rp.T = T;
  rp.B = B;
  rp.K = K;
  rp.d = c->d;
  rp.E = c->E;
  rp.k = c->k;
  rp.S = c->S;
  rp.V = c->V;
  rp.tpb = sh.tpb;
  rp.wr_smem = sh.wr_smem ? 1 : 0;
  rp.eps = c->cfg.rms_eps;
  rp.src = src;
  rp.context_ids = context_ids;
  rp.draft_ids = draft_ids;
  rp.embed = c->embed;
  rp.h_in = static_cast<const __nv_bfloat16*>(h_in);
  rp.h = c->h;
  rp.y = c->y;
  rp.gain = c->gain + (size_t)l * c->d;
  rp.Wr = c->router + (size_t)l * c->E * c->d;
  rp.wr_row = l * c->E;
  rp.bias = c->has_bias ? c->bias + (size_t)l * c->E : nullptr;
  rp.bad = c->bad;
  rp.status = c->status;
  if (probe) {
    if (probe->topk_idx) rp.probe_idx = probe->topk_idx + (size_t)probe_layer * T * c->k;
    if (probe->topk_w) rp.probe_w = probe->topk_w + (size_t)probe_layer * T * c->k;
    if (probe->hidden) rp.probe_hidden = probe->hidden + (size_t)probe_layer * T * c->d;
  }
  rp.cnt = c->cnt + (size_t)parity * c->E;
  rp.cnt_other = c->cnt + (size_t)(1 - parity) * c->E;
  rp.dep_clear = c->dep;
  rp.n_dep_clear = c->chunks_cap;
  rp.next_item_clear = item_counter(c, 1 - parity);
  rp.xperm = c->xperm;
  rp.perm_token = c->perm_token;
  rp.perm_slot = c->perm_slot;
  rp.perm_w = c->perm_w;
  rp.stamps = stamp_slot(c, stamp_base);
  // the verify step's few-token layers: the routing inside the expert FFN
  const bool fused = sh.fused && (src == mv::kSrcEmbed || src == mv::kSrcCombine);
  if (!fused) {
    Timed tm(c, 3, s);
    CK(mv::launch_route(c->map_wr, rp, sh.grid_route, sh.route_smem, s, pdl));
  }
  mv::FfnParams fp = {};
  fp.cnt = c->cnt + (size_t)parity * c->E;
  fp.dep = c->dep;
  fp.E = c->E;
  fp.S = c->S;
  fp.T = T;
  fp.nch = sh.nch;
  fp.tile_gu = c->mt_gu;
  fp.tile_dn = c->mt_dn;
  // items per chunk: one per 128-row weight tile (weight-major) or per
  // 256-row pair of tiles (token-major)
  fp.mt_gu = sh.tokm ? c->mt_gu / 2 : c->mt_gu;
  fp.mt_dn = sh.tokm ? (c->mt_dn + 1) / 2 : c->mt_dn;
  fp.kb_gu = c->d / 64;
  fp.kb_dn = c->I_pad / 64;
  fp.a_base_gu = l * c->nE * c->mt_gu * 128;
  fp.a_base_dn = l * c->nE * c->mt_dn * 128;
  fp.stages = sh.stages;
  fp.tmem_cols = sh.tmem_cols;
  fp.a_out = c->abuf;
  fp.I_pad = c->I_pad;
  fp.perm_token = c->perm_token;
  fp.perm_slot = c->perm_slot;
  fp.perm_w = c->perm_w;
  fp.y = c->y;
  fp.d = c->d;
  fp.kS = c->kS;
  fp.status = c->status;
  fp.next_item = item_counter(c, parity);
  // The first items run the shared experts, then (when every routed expert
  // holds one chunk) routed expert c / mt_gu's tile c % mt_gu.  Guessing the
  // routed ones costs little when a guess misses (the loads overlap the
  // routing), so it is on from one expected row per expert; the shared
  // experts' items are always right, and loading them early pays from a
  // quarter of a row per routed expert (measured on the 12-layer step: T = 4
  // 0.556 -> 0.549 ms, T = 2 0.467 -> 0.508 ms, so off there).  The L2 pull
  // of the next layer's first items competes with this layer's streaming:
  // the routed guesses are pulled from six expected rows per expert, the
  // shared experts' items whenever they are guessed.
  const int64_t rows_x_E = (int64_t)T * c->k;
  fp.spec = rows_x_E >= c->E ? 2 : 4 * rows_x_E >= c->E ? 1 : 0;
  const bool pull_routed = rows_x_E >= 6LL * c->E;
  const CUtensorMap* map_pf = &c->map_gu;
  fp.pf_kb = c->d / 64;
  if (next_head) {
    map_pf = &c->map_lm;
    fp.pf_base = 0;
    fp.pf_div = sh.n_chunks_lm;
    fp.pf_limit = (c->V_pad / 128) * sh.n_chunks_lm;
    if (sh.lm.pair) {
      fp.pf_pair = 1;
      fp.pf_limit = 2 * lm_pairs(c);
    }
  } else if (l + 1 < c->L && src == mv::kSrcH) {
    // the stack with attention: the next layer starts with its q/k/v
    // projection, whose 128-row tiles each CTA c < tiles pulls once
    map_pf = &c->map_qkv;
    fp.pf_base = (l + 1) * c->rows_qkv;
    fp.pf_div = 1;
    fp.pf_limit = c->rows_qkv / 128;
  } else if (l + 1 < c->L && src != mv::kSrcBf16 && fp.spec > 0) {
    fp.pf_items = 1;
    fp.pf_base = (l + 1) * c->nE * c->mt_gu * 128;
    fp.pf_div = 1;
    fp.pf_limit = pull_routed ? c->nE * c->mt_gu
                              : c->S * ((T + sh.nch - 1) / sh.nch) * c->mt_gu;
  }
  fp.stamps = stamp_slot(c, stamp_base >= 0 ? stamp_base + 1 : -1);
  if (fused) {
    fp.n_route = T;
    fp.rt = rp;
    fp.route_done = c->route_ctr + parity;
    fp.route_done_clear = c->route_ctr + (1 - parity);
    // the layer's own ticket counter: the launch claims on it from its first
    // instruction, and nothing else uses it before the final kernel clears it
    fp.next_item = c->layer_items + l;
  }
  if (sh.tokm) {
    fp.spec = 0;
    fp.pf_limit = 0;
    Timed tm(c, 0, s);
    CK(mv::launch_ffn_tokm(c->map_gu256, sh.map_x, c->map_dn256, sh.map_a, fp, persistent_grid(c),
                           s, pdl));
  } else {
    Timed tm(c, 0, s);
    CK(mv::launch_ffn(c->map_gu, sh.map_x, c->map_dn, sh.map_a, *map_pf, c->map_wr, fp,
                      persistent_grid(c), s, pdl));
  }
  return MOE_VERIFY_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

const char* moe_verify_strerror(int status) {
  switch (status) {
    case MOE_VERIFY_OK: return "ok";
    case MOE_VERIFY_ERR_ARG: return "invalid argument";
    case MOE_VERIFY_ERR_CUDA: return "CUDA call failed";
    case MOE_VERIFY_ERR_OOM: return "out of device memory";
    case MOE_VERIFY_ERR_ID_RANGE: return "token id outside [0, vocab)";
    case MOE_VERIFY_ERR_TIMEOUT: return "bounded device wait ran out";
    case MOE_VERIFY_ERR_UNSUPPORTED: return "unsupported shape or device";
    default: return "unknown status";
  }
}

int moe_verify_check_config(const moe_verify_config* config) { return check(config); }

uint64_t moe_verify_device_bytes(const moe_verify_config* config) {
  if (check(config) != MOE_VERIFY_OK) return 0;
  Derived r = derive(config);
  return total_bytes(sizes(config, r));
}

int moe_verify_init(const moe_verify_config* config, const moe_verify_weights* w,
                    void* cuda_stream, moe_verify_ctx** out) {
  if (!out) return MOE_VERIFY_ERR_ARG;
  *out = nullptr;
  int rc = check(config);
  if (rc != MOE_VERIFY_OK) return rc;
  if (!w || !w->embed || !w->final_norm || !w->lm_head || !w->norm || !w->router || !w->w_gate ||
      !w->w_up || !w->w_down)
    return MOE_VERIFY_ERR_ARG;
  if (config->n_shared > 0 && (!w->s_gate || !w->s_up || !w->s_down)) return MOE_VERIFY_ERR_ARG;
  for (int l = 0; l < config->n_layers; ++l) {
    if (!w->norm[l] || !w->router[l] || !w->w_gate[l] || !w->w_up[l] || !w->w_down[l])
      return MOE_VERIFY_ERR_ARG;
    if (config->n_shared > 0 && (!w->s_gate[l] || !w->s_up[l] || !w->s_down[l]))
      return MOE_VERIFY_ERR_ARG;
  }
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_VERIFY_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_VERIFY_ERR_UNSUPPORTED;
  if (!get_encode()) return MOE_VERIFY_ERR_CUDA;

  moe_verify_ctx* c = new (std::nothrow) moe_verify_ctx();
  if (!c) return MOE_VERIFY_ERR_OOM;
  c->cfg = *config;
  c->device = dev;
  c->num_sms = sms;
  c->L = config->n_layers;
  c->d = config->hidden;
  c->E = config->n_experts;
  c->k = config->top_k;
  c->S = config->n_shared;
  c->I = config->expert_inter;
  c->Is = config->shared_inter;
  c->V = config->vocab;
  Derived r = derive(config);
  c->nE = r.nE;
  c->kS = r.kS;
  c->I_pad = r.I_pad;
  c->d_pad = r.d_pad;
  c->V_pad = r.V_pad;
  c->mt_gu = r.mt_gu;
  c->mt_dn = r.mt_dn;
  c->T_max = r.T_max;
  c->rows_max = r.rows_max;
  c->chunks_cap = r.chunks_cap;
  Sizes z = sizes(config, r);
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);

  auto fail = [&](int code) {
    cudaStreamSynchronize(s);
    free_all(c);
    delete c;
    return code;
  };
#define AL(ptr, bytes)                       \
  do {                                       \
    int _r = dalloc(c, &(ptr), (bytes));     \
    if (_r != MOE_VERIFY_OK) return fail(_r); \
  } while (0)
#define CKF(x)                                                 \
  do {                                                         \
    if ((x) != cudaSuccess) return fail(MOE_VERIFY_ERR_CUDA);  \
  } while (0)

  AL(c->w_gu, z.w_gu);
  AL(c->w_dn, z.w_dn);
  AL(c->w_lm, z.w_lm);
  AL(c->embed, z.embed);
  AL(c->router, z.router);
  AL(c->gain, z.gain);
  AL(c->final_gain, z.final_gain);
  AL(c->bias, z.bias);
  AL(c->h, z.h);
  AL(c->y, z.y);
  AL(c->xperm, z.xperm);
  AL(c->abuf, z.abuf);
  AL(c->xf, z.xf);
  AL(c->bad, z.bad);
  AL(c->perm_token, z.perm);
  AL(c->perm_slot, z.perm);
  AL(c->perm_w, z.perm);
  AL(c->cnt, z.cnt);
  AL(c->dep, z.dep);
  AL(c->done_ffn, 16);
  AL(c->done_lm, 16);
  AL(c->route_ctr, 16);
  AL(c->layer_items, (size_t)c->L * 4);
  AL(c->keys, z.keys);
  AL(c->status, 16);
  AL(c->io_ctx, z.io);
  AL(c->io_drafts, z.io);
  AL(c->io_targets, z.io);
  AL(c->io_committed, z.io);
  AL(c->io_alen, z.io);
  AL(c->io_out, z.io + (size_t)config->max_batch * 4);
  if (cudaHostAlloc(reinterpret_cast<void**>(&c->stage),
                    2 * z.io + (size_t)config->max_batch * 4, cudaHostAllocDefault) != cudaSuccess) {
    c->stage = nullptr;
    return fail(MOE_VERIFY_ERR_OOM);
  }

  // zero the workspace so that padding rows read by the MMAs are finite
  CKF(cudaMemsetAsync(c->y, 0, z.y, s));
  CKF(cudaMemsetAsync(c->xperm, 0, z.xperm, s));
  CKF(cudaMemsetAsync(c->abuf, 0, z.abuf, s));
  CKF(cudaMemsetAsync(c->xf, 0, z.xf, s));
  CKF(cudaMemsetAsync(c->cnt, 0, z.cnt, s));
  CKF(cudaMemsetAsync(c->dep, 0, z.dep, s));
  CKF(cudaMemsetAsync(c->done_ffn, 0, 16, s));
  CKF(cudaMemsetAsync(c->done_lm, 0, 16, s));
  CKF(cudaMemsetAsync(c->route_ctr, 0, 16, s));
  CKF(cudaMemsetAsync(c->layer_items, 0, (size_t)c->L * 4, s));
  CKF(cudaMemsetAsync(c->status, 0, 16, s));
  CKF(cudaMemsetAsync(c->bias, 0, z.bias, s));

  // weights: copy and repack
  const int d = c->d, E = c->E, L = c->L;
  CKF(cudaMemcpyAsync(c->embed, w->embed, z.embed, cudaMemcpyDeviceToDevice, s));
  CKF(cudaMemsetAsync(c->w_lm, 0, z.w_lm, s));
  CKF(cudaMemcpyAsync(c->w_lm, w->lm_head, (size_t)c->V * d * 2, cudaMemcpyDeviceToDevice, s));
  CKF(mv::launch_bf16_to_f32(c->final_gain, static_cast<const __nv_bfloat16*>(w->final_norm), d, s));
  const size_t gu_layer = (size_t)c->nE * c->mt_gu * 128 * d;
  const size_t dn_layer = (size_t)c->nE * c->mt_dn * 128 * c->I_pad;
  for (int l = 0; l < L; ++l) {
    CKF(cudaMemcpyAsync(c->router + (size_t)l * E * d, w->router[l], (size_t)E * d * 2,
                        cudaMemcpyDeviceToDevice, s));
    CKF(mv::launch_bf16_to_f32(c->gain + (size_t)l * d,
                               static_cast<const __nv_bfloat16*>(w->norm[l]), d, s));
    if (w->router_bias && w->router_bias[l]) {
      c->has_bias = true;
      CKF(cudaMemcpyAsync(c->bias + (size_t)l * E, w->router_bias[l], (size_t)E * 4,
                          cudaMemcpyDeviceToDevice, s));
    }
    const __nv_bfloat16* sg = c->S ? static_cast<const __nv_bfloat16*>(w->s_gate[l]) : nullptr;
    const __nv_bfloat16* su = c->S ? static_cast<const __nv_bfloat16*>(w->s_up[l]) : nullptr;
    const __nv_bfloat16* sd = c->S ? static_cast<const __nv_bfloat16*>(w->s_down[l]) : nullptr;
    CKF(mv::launch_repack_gateup(c->w_gu + gu_layer * l,
                                 static_cast<const __nv_bfloat16*>(w->w_gate[l]),
                                 static_cast<const __nv_bfloat16*>(w->w_up[l]), sg, su, E, c->S,
                                 c->I, c->Is, d, c->mt_gu, s));
    CKF(mv::launch_repack_down(c->w_dn + dn_layer * l,
                               static_cast<const __nv_bfloat16*>(w->w_down[l]), sd, E, c->S, c->I,
                               c->Is, d, c->I_pad, c->mt_dn, s));
  }
  CKF(cudaStreamSynchronize(s));

  int e1 = encode_map(&c->map_gu, c->w_gu, d, (uint64_t)L * c->nE * c->mt_gu * 128, 128);
  int e2 = encode_map(&c->map_dn, c->w_dn, c->I_pad, (uint64_t)L * c->nE * c->mt_dn * 128, 128);
  int e3 = encode_map(&c->map_lm, c->w_lm, d, c->V_pad, 128);
  c->lm_pair_max = mv::lmhead_pair_max_clusters(mv::lm_layout(mv::kLmPairMinT + 1).stages);
  int e5 = encode_map(&c->map_gu256, c->w_gu, d, (uint64_t)L * c->nE * c->mt_gu * 128, 256);
  int e6 = encode_map(&c->map_dn256, c->w_dn, c->I_pad, (uint64_t)L * c->nE * c->mt_dn * 128, 256);
  // router weights of all layers: boxes of 64 columns x E rows
  int e4 = encode_map(&c->map_wr, c->router, d, (uint64_t)L * E, (uint32_t)E);
  if (e1 || e2 || e3 || e4 || e5 || e6) return fail(MOE_VERIFY_ERR_CUDA);
#undef AL
#undef CKF
  *out = c;
  return MOE_VERIFY_OK;
}

// Final RMSNorm (after the residual update of the last block) and the
// greedy lm_head for T rows; clears the expert counters of the last block
// (parity `last_parity`).  probe_hidden [T, d] and logits [T, V] may be NULL.
static int enqueue_head(moe_verify_ctx* ctx, int T, const StepShape& sh, int last_parity,
                        int32_t* target_ids, float* probe_hidden, float* logits, cudaStream_t s,
                        bool pdl, int stamp_slot_lm = -1) {
  mv::FinalParams fp = {};
  fp.T = T;
  fp.d = ctx->d;
  fp.kS = ctx->kS;
  fp.eps = ctx->cfg.rms_eps;
  fp.mode = 0;
  fp.h = ctx->h;
  fp.y = ctx->y;
  fp.gain = ctx->final_gain;
  fp.out = ctx->xf;
  fp.probe_hidden = probe_hidden;
  fp.keys = ctx->keys;
  fp.cnt_clear = ctx->cnt + (size_t)last_parity * ctx->E;
  fp.n_cnt_clear = ctx->E;
  fp.item_clear = item_counter(ctx, last_parity);
  fp.route_done_clear = ctx->route_ctr + last_parity;
  fp.layer_items_clear = ctx->layer_items;
  fp.n_layer_items = ctx->L;
  {
    Timed tm(ctx, 3, s);
    CK(mv::launch_final(fp, s, pdl));
  }
  mv::GemmParams gp = {};
  gp.n_items_static = sh.lm.pair ? ((ctx->V_pad + 255) / 256) * sh.n_chunks_lm
                                 : (ctx->V_pad / 128) * sh.n_chunks_lm;
  gp.kblocks = ctx->d / 64;
  gp.nch = sh.nch_lm;
  gp.stages = sh.lm.stages;
  gp.tmem_cols = sh.lm.tmem_cols;
  gp.status = ctx->status;
  gp.T = T;
  gp.V = ctx->V;
  gp.n_chunks = sh.n_chunks_lm;
  gp.nch_lm = sh.nch_lm;
  gp.keys = ctx->keys;
  gp.logits = logits;
  gp.targets = target_ids;
  gp.bad = ctx->bad;
  gp.done = ctx->done_lm;
  gp.aborted = ctx->done_lm + 1;
  gp.stamps = stamp_slot(ctx, stamp_slot_lm);
  {
    Timed tm(ctx, 2, s);
    if (sh.lm.pair)
      CK(mv::launch_lmhead_pair(ctx->map_lm, sh.map_f128, gp, lm_pairs(ctx), s, pdl));
    else
      CK(mv::launch_lmhead(ctx->map_lm, sh.map_f, gp, sh.lm.tokens_on_m, persistent_grid(ctx), s,
                           pdl));
  }
  return MOE_VERIFY_OK;
}

static int enqueue_step(moe_verify_ctx* ctx, const int32_t* context_ids, const int32_t* draft_ids,
                        int32_t B, int32_t K, int32_t* target_ids, const moe_verify_probe* probe,
                        cudaStream_t s) {
  const int T = B * (K + 1);
  StepShape sh;
  if (shape_for(ctx, T, &sh) != MOE_VERIFY_OK) return MOE_VERIFY_ERR_CUDA;
  const bool pdl = true;
  for (int l = 0; l < ctx->L; ++l) {
    int rc = run_layer(ctx, l, l & 1, l == 0 ? mv::kSrcEmbed : mv::kSrcCombine, sh, context_ids,
                       draft_ids, B, K, nullptr, probe, l, s, pdl, l == ctx->L - 1, 2 * l);
    if (rc != MOE_VERIFY_OK) return rc;
  }
  float* ph = (probe && probe->hidden) ? probe->hidden + (size_t)ctx->L * T * ctx->d : nullptr;
  return enqueue_head(ctx, T, sh, (ctx->L - 1) & 1, target_ids, ph, probe ? probe->logits : nullptr,
                      s, pdl, 2 * ctx->L);
}

int moe_verify_step(moe_verify_ctx* ctx, const int32_t* context_ids, const int32_t* draft_ids,
                    int32_t B, int32_t K, int32_t* target_ids, const moe_verify_probe* probe,
                    void* cuda_stream) {
  if (!ctx || !context_ids || !target_ids || ctx->attn) return MOE_VERIFY_ERR_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k) return MOE_VERIFY_ERR_ARG;
  if (K > 0 && !draft_ids) return MOE_VERIFY_ERR_ARG;
  return enqueue_step(ctx, context_ids, draft_ids, B, K, target_ids, probe,
                      static_cast<cudaStream_t>(cuda_stream));
}

int moe_verify_accept(moe_verify_ctx* ctx, const int32_t* draft_ids, const int32_t* target_ids,
                      int32_t B, int32_t K, int32_t* committed, int32_t* accept_len,
                      void* cuda_stream) {
  if (!ctx || !target_ids || !committed || !accept_len) return MOE_VERIFY_ERR_ARG;
  if (B < 1 || K < 0 || K > 15) return MOE_VERIFY_ERR_ARG;
  if (K > 0 && !draft_ids) return MOE_VERIFY_ERR_ARG;
  mv::AcceptParams ap;
  ap.B = B;
  ap.K = K;
  ap.V = ctx->V;
  ap.drafts = draft_ids;
  ap.targets = target_ids;
  ap.committed = committed;
  ap.accept_len = accept_len;
  ap.status = ctx->status;
  CK(mv::launch_accept(ap, static_cast<cudaStream_t>(cuda_stream)));
  return MOE_VERIFY_OK;
}

int moe_verify_layer(moe_verify_ctx* ctx, int32_t layer, const void* h_in, int32_t T, void* h_out,
                     const moe_verify_probe* probe, void* cuda_stream) {
  if (!ctx || !h_in || !h_out || ctx->attn) return MOE_VERIFY_ERR_ARG;
  if (layer < 0 || layer >= ctx->L || T < 1 || T > ctx->T_max) return MOE_VERIFY_ERR_ARG;
  if (!aligned16(h_in) || !aligned16(h_out)) return MOE_VERIFY_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  StepShape sh;
  if (shape_for(ctx, T, &sh) != MOE_VERIFY_OK) return MOE_VERIFY_ERR_CUDA;
  int rc = run_layer(ctx, layer, 0, mv::kSrcBf16, sh, nullptr, nullptr, T, 0, h_in, probe, 0, s,
                     true, false);
  if (rc != MOE_VERIFY_OK) return rc;
  mv::FinalParams fp = {};
  fp.T = T;
  fp.d = ctx->d;
  fp.kS = ctx->kS;
  fp.eps = ctx->cfg.rms_eps;
  fp.mode = 1;
  fp.h = ctx->h;
  fp.y = ctx->y;
  fp.gain = ctx->final_gain;
  fp.out = static_cast<__nv_bfloat16*>(h_out);
  fp.probe_hidden = (probe && probe->hidden) ? probe->hidden + (size_t)T * ctx->d : nullptr;
  fp.keys = ctx->keys;
  fp.cnt_clear = ctx->cnt;
  fp.n_cnt_clear = ctx->E;
  fp.item_clear = item_counter(ctx, 0);
  {
    Timed tm(ctx, 3, s);
    CK(mv::launch_final(fp, s, true));
  }
  return MOE_VERIFY_OK;
}

namespace {

// The device part of a host-buffer decode call: step + accept on the
// context's own io buffers.
// One host-buffer decode iteration on the device: the ids in from the pinned
// stage (one copy: [B context ids][B K drafts]), step + accept, and
// accept_len and committed out to the stage (one copy: [B][B (K + 1)]).
int enqueue_decode(moe_verify_ctx* ctx, int B, int K, cudaStream_t s) {
  const int32_t* stage_in = ctx->stage;
  int32_t* stage_out = ctx->stage + ctx->T_max;
  int32_t* drafts = ctx->io_ctx + B;
  CK(cudaMemcpyAsync(ctx->io_ctx, stage_in, (size_t)B * (K + 1) * 4, cudaMemcpyHostToDevice, s));
  int rc = enqueue_step(ctx, ctx->io_ctx, drafts, B, K, ctx->io_targets, nullptr, s);
  if (rc != MOE_VERIFY_OK) return rc;
  rc = moe_verify_accept(ctx, drafts, ctx->io_targets, B, K, ctx->io_out + B, ctx->io_out, s);
  if (rc != MOE_VERIFY_OK) return rc;
  CK(cudaMemcpyAsync(stage_out, ctx->io_out, (size_t)B * (K + 2) * 4, cudaMemcpyDeviceToHost, s));
  return MOE_VERIFY_OK;
}

// The captured graph of enqueue_decode for (B, K), built on first use
// (captured on a library-owned stream, launched on the caller's).  Returns
// nullptr when it cannot be built (the caller then enqueues directly).
cudaGraphExec_t decode_graph(moe_verify_ctx* ctx, int B, int K) {
  constexpr size_t kMaxGraphs = 16;
  for (const auto& g : ctx->decode_graphs)
    if (g.B == B && g.K == K) return g.exec;
  if (ctx->decode_graphs.size() >= kMaxGraphs) return nullptr;
  if (!ctx->capture_stream &&
      cudaStreamCreateWithFlags(&ctx->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    ctx->capture_stream = nullptr;
    return nullptr;
  }
  cudaStream_t cs = ctx->capture_stream;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return nullptr;
  const int rc = enqueue_decode(ctx, B, K, cs);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cs, &graph);
  cudaGraphExec_t exec = nullptr;
  if (rc == MOE_VERIFY_OK && ec == cudaSuccess && graph &&
      cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
    exec = nullptr;
  if (graph) cudaGraphDestroy(graph);
  if (!exec) {
    cudaGetLastError();
    return nullptr;
  }
  ctx->decode_graphs.push_back({B, K, exec});
  return exec;
}

}  // namespace

int moe_verify_decode_host(moe_verify_ctx* ctx, const int32_t* host_context_ids,
                           const int32_t* host_draft_ids, int32_t B, int32_t K,
                           int32_t* host_committed, int32_t* host_accept_len, void* cuda_stream) {
  if (!ctx || !host_context_ids || !host_committed || !host_accept_len || ctx->attn)
    return MOE_VERIFY_ERR_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k) return MOE_VERIFY_ERR_ARG;
  if (K > 0 && !host_draft_ids) return MOE_VERIFY_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // the previous call has synchronised: the stage is free
  std::memcpy(ctx->stage, host_context_ids, (size_t)B * 4);
  if (K > 0) std::memcpy(ctx->stage + B, host_draft_ids, (size_t)B * K * 4);
  cudaGraphExec_t exec = ctx->timing ? nullptr : decode_graph(ctx, B, K);
  if (exec) {
    CK(cudaGraphLaunch(exec, s));
  } else {
    int rc = enqueue_decode(ctx, B, K, s);
    if (rc != MOE_VERIFY_OK) return rc;
  }
  CK(cudaStreamSynchronize(s));
  const int32_t* out = ctx->stage + ctx->T_max;
  std::memcpy(host_accept_len, out, (size_t)B * 4);
  std::memcpy(host_committed, out + B, (size_t)B * (K + 1) * 4);
  return MOE_VERIFY_OK;
}

int moe_verify_draft_inputs(moe_verify_ctx* ctx, const int32_t* committed,
                            const int32_t* accept_len, int32_t B, int32_t K, float* h_out,
                            int32_t* t_out, void* cuda_stream) {
  if (!ctx || !committed || !accept_len || !h_out || !t_out) return MOE_VERIFY_ERR_ARG;
  if (B < 1 || K < 0 || (int64_t)B * (K + 1) > ctx->T_max) return MOE_VERIFY_ERR_ARG;
  if (!aligned16(h_out)) return MOE_VERIFY_ERR_ARG;
  CK(mv::launch_draft_inputs(ctx->h, committed, accept_len, B, K, ctx->d, h_out, t_out,
                             static_cast<cudaStream_t>(cuda_stream)));
  return MOE_VERIFY_OK;
}

int moe_verify_draft(moe_verify_ctx* ctx, const float* h_prev, const int32_t* t_prev, int32_t B,
                     int32_t K, int32_t* drafts, float* hidden_out, void* cuda_stream) {
  if (!ctx || !h_prev || !t_prev || !drafts || ctx->attn) return MOE_VERIFY_ERR_ARG;
  if (ctx->L != 1) return MOE_VERIFY_ERR_ARG;
  if (B < 1 || B > ctx->T_max || K < 1 || K > 15) return MOE_VERIFY_ERR_ARG;
  if (!aligned16(h_prev) || (hidden_out && !aligned16(hidden_out))) return MOE_VERIFY_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const int T = B;
  StepShape sh;
  if (shape_for(ctx, T, &sh) != MOE_VERIFY_OK) return MOE_VERIFY_ERR_CUDA;
  const size_t hb = (size_t)T * ctx->d * sizeof(float);
  CK(cudaMemcpyAsync(ctx->h, h_prev, hb, cudaMemcpyDeviceToDevice, s));
  const int32_t* ids = t_prev;
  for (int i = 0; i < K; ++i) {
    // h += E[t];  the block;  t = greedy head of h
    int rc = run_layer(ctx, 0, 0, mv::kSrcEmbedAdd, sh, ids, nullptr, B, 0, nullptr, nullptr, 0, s,
                       true, true);
    if (rc != MOE_VERIFY_OK) return rc;
    rc = enqueue_head(ctx, T, sh, 0, ctx->io_targets, nullptr, nullptr, s, true);
    if (rc != MOE_VERIFY_OK) return rc;
    CK(mv::launch_scatter_column(ctx->io_targets, B, drafts, K, i, s));
    if (hidden_out)
      CK(cudaMemcpyAsync(hidden_out + (size_t)i * T * ctx->d, ctx->h, hb, cudaMemcpyDeviceToDevice,
                         s));
    ids = ctx->io_targets;
  }
  return MOE_VERIFY_OK;
}

int moe_verify_init_attn(const moe_verify_config* config, const moe_verify_weights* weights,
                         const moe_verify_attn_config* attn,
                         const moe_verify_attn_weights* aw, void* cuda_stream,
                         moe_verify_ctx** out) {
  if (!out) return MOE_VERIFY_ERR_ARG;
  *out = nullptr;
  if (!attn || !aw) return MOE_VERIFY_ERR_ARG;
  int rc = check(config);
  if (rc != MOE_VERIFY_OK) return rc;
  const int d = config->hidden, L = config->n_layers;
  if (attn->n_heads < 1 || d % attn->n_heads != 0) return MOE_VERIFY_ERR_ARG;
  const int hd = d / attn->n_heads;
  if (attn->max_pos < 1 || attn->max_pos > 32768) return MOE_VERIFY_ERR_ARG;
  if (!(attn->rope_theta > 1.f) || !(attn->rope_theta < 1e30f)) return MOE_VERIFY_ERR_ARG;
  if (!aw->attn_norm || !aw->w_q || !aw->w_k || !aw->w_v || !aw->w_o) return MOE_VERIFY_ERR_ARG;
  for (int l = 0; l < L; ++l)
    if (!aw->attn_norm[l] || !aw->w_q[l] || !aw->w_k[l] || !aw->w_v[l] || !aw->w_o[l])
      return MOE_VERIFY_ERR_ARG;
  if (hd != 16 && hd != 32 && hd != 64 && hd != 128) return MOE_VERIFY_ERR_UNSUPPORTED;
  // cache rows (layers x slots x heads x positions) are addressed with 32-bit
  // tensor-map coordinates
  if ((uint64_t)L * config->max_batch * attn->n_heads * attn->max_pos >= (1ull << 31))
    return MOE_VERIFY_ERR_UNSUPPORTED;
  rc = moe_verify_init(config, weights, cuda_stream, out);
  if (rc != MOE_VERIFY_OK) return rc;
  moe_verify_ctx* c = *out;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  auto fail = [&](int code) {
    moe_verify_destroy(c);
    *out = nullptr;
    return code;
  };
  c->attn = true;
  c->H = attn->n_heads;
  c->hd = hd;
  c->max_pos = attn->max_pos;
  c->rows_qkv = round_up(3 * d, 128);
  const int Bmax = config->max_batch, K1max = config->max_k + 1;
  // about four items per SM: measured at 32 sequences of ~1,900 positions,
  // 8 per SM gave 88 us per attention launch and 2 or 4 per SM 72 us (fewer,
  // longer items: fewer item ends and split merges)
  c->attn_target = 4 * c->num_sms;
  // (sequence, split) pairs: at most B + total keys / split width, the width
  // either >= total keys x H / target or 1024
  c->cap_pairs = Bmax + (c->attn_target + c->H - 1) / c->H +
                 Bmax * ((c->max_pos + mv::kAttnMaxSplit - 1) / mv::kAttnMaxSplit) + 1;
  const uint64_t cache = (uint64_t)L * Bmax * c->max_pos * d * 2;
  const uint64_t act16 = (uint64_t)round_up(c->T_max, 16) * d * 2;
  int e = 0;
  if ((e = dalloc(c, &c->w_qkv, (uint64_t)L * c->rows_qkv * d * 2)) ||
      (e = dalloc(c, &c->w_o, (uint64_t)L * c->d_pad * d * 2)) ||
      (e = dalloc(c, &c->attn_gain, (uint64_t)L * d * 4)) ||
      (e = dalloc(c, &c->rope, (uint64_t)c->max_pos * (hd / 2) * sizeof(float2))) ||
      (e = dalloc(c, &c->kcache, cache)) || (e = dalloc(c, &c->vcache, cache)) ||
      (e = dalloc(c, &c->xa, act16)) || (e = dalloc(c, &c->obuf, act16)) ||
      (e = dalloc(c, &c->qbuf, (uint64_t)c->T_max * d * 4)) ||
      (e = dalloc(c, &c->part, (uint64_t)c->cap_pairs * c->H * K1max * (hd + 2) * 4)) ||
      (e = dalloc(c, &c->arrive, (uint64_t)Bmax * c->H * 4)) ||
      (e = dalloc(c, &c->plan, (uint64_t)(2 + 2 * c->cap_pairs + Bmax) * 4)) ||
      (e = dalloc(c, &c->attn_ctr, (uint64_t)L * 4)))
    return fail(e);
#define CKA(x)                                               \
  do {                                                       \
    if ((x) != cudaSuccess) return fail(MOE_VERIFY_ERR_CUDA); \
  } while (0)
  CKA(cudaMemsetAsync(c->kcache, 0, cache, s));
  CKA(cudaMemsetAsync(c->vcache, 0, cache, s));
  CKA(cudaMemsetAsync(c->xa, 0, act16, s));
  CKA(cudaMemsetAsync(c->obuf, 0, act16, s));
  CKA(cudaMemsetAsync(c->arrive, 0, (size_t)Bmax * c->H * 4, s));
  CKA(cudaMemsetAsync(c->plan, 0, (size_t)(2 + 2 * c->cap_pairs + Bmax) * 4, s));
  CKA(cudaMemsetAsync(c->attn_ctr, 0, (size_t)L * 4, s));
  CKA(cudaMemsetAsync(c->w_o, 0, (size_t)L * c->d_pad * d * 2, s));
  for (int l = 0; l < L; ++l) {
    CKA(mv::launch_repack_qkv(c->w_qkv + (size_t)l * c->rows_qkv * d,
                              static_cast<const __nv_bfloat16*>(aw->w_q[l]),
                              static_cast<const __nv_bfloat16*>(aw->w_k[l]),
                              static_cast<const __nv_bfloat16*>(aw->w_v[l]), d, hd, c->rows_qkv,
                              s));
    CKA(cudaMemcpyAsync(c->w_o + (size_t)l * c->d_pad * d, aw->w_o[l], (size_t)d * d * 2,
                        cudaMemcpyDeviceToDevice, s));
    CKA(mv::launch_bf16_to_f32(c->attn_gain + (size_t)l * d,
                               static_cast<const __nv_bfloat16*>(aw->attn_norm[l]), d, s));
  }
  // rotary table: (cos, sin) of pos * theta^(-2i/hd), computed in double
  {
    const int half = hd / 2;
    std::vector<float2> tab((size_t)c->max_pos * half);
    for (int i = 0; i < half; ++i) {
      const double f = pow((double)attn->rope_theta, -2.0 * i / (double)hd);
      for (int pos = 0; pos < c->max_pos; ++pos) {
        const double a = (double)pos * f;
        tab[(size_t)pos * half + i] = make_float2((float)cos(a), (float)sin(a));
      }
    }
    CKA(cudaMemcpyAsync(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice,
                        s));
    CKA(cudaStreamSynchronize(s));
  }
#undef CKA
  const uint64_t cache_rows = (uint64_t)L * Bmax * c->H * c->max_pos;
  const uint32_t bw = hd < 64 ? (uint32_t)hd : 64u;
  if (encode_map(&c->map_qkv, c->w_qkv, d, (uint64_t)L * c->rows_qkv, 128) ||
      encode_map(&c->map_wo, c->w_o, d, (uint64_t)L * c->d_pad, 128) ||
      encode_map_box(&c->map_kc, c->kcache, hd, cache_rows, bw, mv::attn_max_split(hd)) ||
      encode_map_box(&c->map_vc, c->vcache, hd, cache_rows, bw, mv::attn_max_split(hd)))
    return fail(MOE_VERIFY_ERR_CUDA);
  return MOE_VERIFY_OK;
}

int moe_verify_kv_cache(moe_verify_ctx* ctx, const void** k_cache, const void** v_cache) {
  if (!ctx || !ctx->attn || !k_cache || !v_cache) return MOE_VERIFY_ERR_ARG;
  *k_cache = ctx->kcache;
  *v_cache = ctx->vcache;
  return MOE_VERIFY_OK;
}

int moe_verify_step_attn(moe_verify_ctx* ctx, const int32_t* context_ids, const int32_t* draft_ids,
                         const int32_t* positions, int32_t B, int32_t K, int32_t* target_ids,
                         const moe_verify_probe* probe, void* cuda_stream) {
  if (!ctx || !ctx->attn || !context_ids || !positions || !target_ids) return MOE_VERIFY_ERR_ARG;
  if (B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k) return MOE_VERIFY_ERR_ARG;
  if (K > 0 && !draft_ids) return MOE_VERIFY_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const int T = B * (K + 1), d = ctx->d, L = ctx->L;
  StepShape sh;
  if (shape_for(ctx, T, &sh) != MOE_VERIFY_OK) return MOE_VERIFY_ERR_CUDA;
  // projections: token chunks of <= 256 rows, as many as it takes for the
  // (weight tile, chunk) items to cover the SMs (the chunks of one tile run
  // side by side and share its weights through L2)
  auto proj_shape = [&](int tiles, mv::ProjParams* pp, CUtensorMap* map, void* act) {
    int chunks = (ctx->num_sms + tiles - 1) / tiles;
    const int most = (T + 15) / 16;
    if (chunks > most) chunks = most;
    if (chunks < (T + 255) / 256) chunks = (T + 255) / 256;
    const int nch = round_up((T + chunks - 1) / chunks, 16);
    pp->nch = nch;
    pp->n_chunks = (T + nch - 1) / nch;
    pp->n_items = tiles * pp->n_chunks;
    int stages = 16;
    while (stages > 2 && mv::proj_smem_bytes(nch, stages) > 227 * 1024) --stages;
    pp->stages = stages;
    pp->tmem_cols = pow2_at_least(2 * nch);
    return encode_map(map, act, d, round_up(ctx->T_max, 16), (uint32_t)nch);
  };
  mv::ProjParams pb = {};
  pb.kblocks = d / 64;
  pb.T = T;
  pb.d = d;
  pb.K = K;
  pb.H = ctx->H;
  pb.hd = ctx->hd;
  pb.max_pos = ctx->max_pos;
  pb.Bmax = ctx->cfg.max_batch;
  pb.status = ctx->status;
  pb.positions = positions;
  pb.rope = ctx->rope;
  mv::ProjParams pq = pb, po = pb;
  CUtensorMap map_xa, map_o;
  if (proj_shape(ctx->rows_qkv / 128, &pq, &map_xa, ctx->xa) ||
      proj_shape(ctx->d_pad / 128, &po, &map_o, ctx->obuf))
    return MOE_VERIFY_ERR_CUDA;
  const size_t cache_layer = (size_t)ctx->cfg.max_batch * ctx->max_pos * d;
  const int attn_grid = ctx->grid_ctas > 0 ? ctx->grid_ctas : ctx->num_sms;
  // probe->hidden [2L + 1, T, d]: row 2l the residual entering block l's
  // attention (written by its RMSNorm kernel), row 2l + 1 the residual
  // entering its MoE part (written by the routing kernel, which indexes the
  // probe by layer: its pointer is offset so that layer l lands on row 2l + 1)
  moe_verify_probe route_probe = {};
  if (probe) route_probe = *probe;
  const bool pdl = true;
  for (int l = 0; l < L; ++l) {
    {
      Timed tm(ctx, 1, s);
      mv::AttnNormParams ap = {};
      ap.T = T;
      ap.B = B;
      ap.K = K;
      ap.d = d;
      ap.kS = ctx->kS;
      ap.V = ctx->V;
      ap.H = ctx->H;
      ap.max_pos = ctx->max_pos;
      ap.first = l == 0 ? 1 : 0;
      ap.eps = ctx->cfg.rms_eps;
      ap.context_ids = context_ids;
      ap.draft_ids = draft_ids;
      ap.positions = positions;
      ap.embed = ctx->embed;
      ap.h = ctx->h;
      ap.y = ctx->y;
      ap.gain = ctx->attn_gain + (size_t)l * d;
      ap.xa = ctx->xa;
      ap.probe_hidden = (probe && probe->hidden) ? probe->hidden + (size_t)(2 * l) * T * d : nullptr;
      ap.bad = ctx->bad;
      ap.status = ctx->status;
      ap.plan = ctx->plan;
      ap.target_items = ctx->attn_target;
      ap.max_split = mv::attn_max_split(ctx->hd);
      ap.item_ctr = ctx->attn_ctr;
      ap.n_item_ctr = L;
      ap.cap_pairs = ctx->cap_pairs;
      ap.stamps = stamp_slot(ctx, 6 * l);
      CK(mv::launch_attn_norm(ap, s, pdl));
    }
    {
      Timed tm(ctx, 1, s);
      mv::ProjParams qp = pq;
      qp.mode = 0;
      qp.a_row0 = l * ctx->rows_qkv;
      qp.q = ctx->qbuf;
      qp.kc = ctx->kcache + cache_layer * l;
      qp.vc = ctx->vcache + cache_layer * l;
      qp.stamps = stamp_slot(ctx, 6 * l + 1);
      const int g = persistent_grid(ctx) < qp.n_items ? persistent_grid(ctx) : qp.n_items;
      CK(mv::launch_proj(ctx->map_qkv, map_xa, qp, g, s, pdl));
    }
    {
      Timed tm(ctx, 1, s);
      mv::AttnParams at = {};
      at.B = B;
      at.K = K;
      at.H = ctx->H;
      at.hd = ctx->hd;
      at.d = d;
      at.max_pos = ctx->max_pos;
      at.Bmax = ctx->cfg.max_batch;
      at.max_split = mv::attn_max_split(ctx->hd);
      at.row0 = l * ctx->cfg.max_batch * ctx->H * ctx->max_pos;
      at.item_ctr = ctx->attn_ctr + l;
      at.cap_pairs = ctx->cap_pairs;
      at.scale_log2 = (float)(1.4426950408889634 / sqrt((double)ctx->hd));
      at.positions = positions;
      at.plan = ctx->plan;
      at.q = ctx->qbuf;
      at.kc = ctx->kcache + cache_layer * l;
      at.vc = ctx->vcache + cache_layer * l;
      at.o = ctx->obuf;
      at.part = ctx->part;
      at.arrive = ctx->arrive;
      at.status = ctx->status;
      at.stamps = stamp_slot(ctx, 6 * l + 2);
      CK(mv::launch_attn(ctx->map_kc, ctx->map_vc, at, attn_grid, s, pdl));
    }
    {
      Timed tm(ctx, 1, s);
      mv::ProjParams op = po;
      op.mode = 1;
      op.a_row0 = l * ctx->d_pad;
      op.h = ctx->h;
      op.stamps = stamp_slot(ctx, 6 * l + 3);
      const int g = persistent_grid(ctx) < op.n_items ? persistent_grid(ctx) : op.n_items;
      CK(mv::launch_proj(ctx->map_wo, map_o, op, g, s, pdl));
    }
    if (probe && probe->hidden) route_probe.hidden = probe->hidden + (size_t)(l + 1) * T * d;
    int rc = run_layer(ctx, l, l & 1, mv::kSrcH, sh, context_ids, draft_ids, B, K, nullptr,
                       probe ? &route_probe : nullptr, l, s, pdl, l == L - 1, 6 * l + 4);
    if (rc != MOE_VERIFY_OK) return rc;
  }
  float* ph = (probe && probe->hidden) ? probe->hidden + (size_t)(2 * L) * T * d : nullptr;
  return enqueue_head(ctx, T, sh, (L - 1) & 1, target_ids, ph, probe ? probe->logits : nullptr, s,
                      pdl, 6 * L);
}

int moe_verify_check_bounded_wait(int64_t limit_ns, int64_t* elapsed_ns, void* cuda_stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return MOE_VERIFY_ERR_ARG;
  unsigned long long out[3] = {0, 0, 0};
  uint32_t st = 0;
  if (mv::run_bounded_wait_check((uint64_t)limit_ns, static_cast<cudaStream_t>(cuda_stream), out,
                                 &st) != cudaSuccess)
    return MOE_VERIFY_ERR_CUDA;
  if (elapsed_ns) *elapsed_ns = (int64_t)out[0];
  return (out[1] == 1 && out[2] == 1 && (st & mv::kErrTimeout)) ? MOE_VERIFY_OK
                                                                : MOE_VERIFY_ERR_CUDA;
}

int moe_verify_sync_status(moe_verify_ctx* ctx) {
  if (!ctx) return MOE_VERIFY_ERR_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
  uint32_t st = 0;
  if (cudaMemcpy(&st, ctx->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_VERIFY_ERR_CUDA;
  if (cudaMemset(ctx->status, 0, 4) != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
  if (st & mv::kErrTimeout) return MOE_VERIFY_ERR_TIMEOUT;
  if (st & mv::kErrIdRange) return MOE_VERIFY_ERR_ID_RANGE;
  if (st) return MOE_VERIFY_ERR_CUDA;
  return MOE_VERIFY_OK;
}

void moe_verify_destroy(moe_verify_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  for (auto& g : ctx->decode_graphs) cudaGraphExecDestroy(g.exec);
  ctx->decode_graphs.clear();
  if (ctx->capture_stream) cudaStreamDestroy(ctx->capture_stream);
  free_all(ctx);
  delete ctx;
}

int moe_verify_set_grid(moe_verify_ctx* ctx, int32_t ctas) {
  if (!ctx || ctas < 0 || ctas > 8 * ctx->num_sms) return MOE_VERIFY_ERR_ARG;
  ctx->grid_ctas = ctas;
  return MOE_VERIFY_OK;
}

int moe_verify_set_layer_kernel(moe_verify_ctx* ctx, int32_t max_tokens) {
  if (!ctx || max_tokens < 0 || max_tokens > mv::kFuseMaxT) return MOE_VERIFY_ERR_ARG;
  ctx->fuse_max_T = max_tokens;
  return MOE_VERIFY_OK;
}

int moe_verify_set_stamps(moe_verify_ctx* ctx, uint64_t* stamps) {
  if (!ctx) return MOE_VERIFY_ERR_ARG;
  if (stamps && (reinterpret_cast<uintptr_t>(stamps) & 7u) != 0) return MOE_VERIFY_ERR_ARG;
  ctx->stamps = reinterpret_cast<unsigned long long*>(stamps);
  return MOE_VERIFY_OK;
}

int moe_verify_set_timing(moe_verify_ctx* ctx, int32_t enable) {
  if (!ctx) return MOE_VERIFY_ERR_ARG;
  ctx->timing = enable != 0;
  return MOE_VERIFY_OK;
}

int moe_verify_get_timing(moe_verify_ctx* ctx, double* ms, int64_t* n, int32_t reset) {
  if (!ctx || !ms || !n) return MOE_VERIFY_ERR_ARG;
  for (auto& tp : ctx->pending) {
    if (cudaEventSynchronize(tp.b) != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, tp.a, tp.b) != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
    ctx->ms[tp.family] += t;
    ctx->launches[tp.family] += 1;
    ctx->event_pool.push_back(tp.a);
    ctx->event_pool.push_back(tp.b);
  }
  ctx->pending.clear();
  for (int i = 0; i < 4; ++i) {
    ms[i] = ctx->ms[i];
    n[i] = ctx->launches[i];
    if (reset) {
      ctx->ms[i] = 0;
      ctx->launches[i] = 0;
    }
  }
  return MOE_VERIFY_OK;
}

}  // extern "C"
