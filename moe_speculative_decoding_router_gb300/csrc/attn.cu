// The attention sub-block of the stack with attention: the residual update
// and attention RMSNorm (with the step's work plan), the causal attention of
// the verify tokens over their sequences' key/value caches, and the repacking
// of the q/k/v weights.  The q/k/v and output projections are tcgen05 GEMMs
// (gemm.cu).
//
// The pages ("Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser With
// Built-In Speculative Decoding", architecture paragraph) name a 12-layer
// decoder with a 32,768-position limit but give no attention shape.  This
// library's reading: pre-norm multi-head attention before each MoE block,
//   h += W_o . attn(bf16(RMSNorm_a(h) * g_a)),
// rotary positions on q and k (dims i and i + hd/2 of a head turned by
// pos * theta^(-2i/hd)), causal over positions 0 .. pos with scores
// q . k / sqrt(hd), bf16 keys, values and attention output.
//
// Attention at decode time reads each sequence's whole cache once per layer
// for only K + 1 queries: it is bound by HBM, so it runs on the CUDA cores,
// streaming keys and values with 16-byte loads.  A sequence's keys are cut
// into splits of plan[0] keys (chosen per step from the total so that the
// (sequence, split, head) items fill the grid about four times); each item
// computes its scores into shared memory, the softmax numerators in place, and
// the weighted sum of its values, and the last of a (sequence, head)'s items
// to finish merges the splits' results in split order.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace mv {

namespace {

constexpr int kNormThreads = 256;
constexpr int kAttnThreads = 256;  // compute threads of the attention kernel (plus a loading warp)
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnStages = 3;  // chunk buffers of the attention kernel's ring

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ bool seq_in_range(int p0, int K, int max_pos) {
  return p0 >= 0 && p0 <= max_pos - 1 - K;
}

// Exclusive scan over the block of one value per thread; returns the
// thread's prefix and sets *total.
__device__ __forceinline__ int block_excl_scan(int v, int* s_scan, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  __syncthreads();  // s_scan is free
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int w = 0; w < kNormThreads / 32; ++w) {
    if (w < warp) base += s_scan[w];
    all += s_scan[w];
  }
  *total = all;
  return base + incl - v;
}

// Layer 0, block 0: the attention's (sequence, split) pairs for this step.
// keys_b = pos_b + K + 1 (0 for a sequence out of range); the split width is
// the larger of the total keys x heads over the wanted items and the longest
// sequence over kAttnMaxSplits, rounded up to a whole number of chunks
// (max_split keys, or 64 below one chunk) and kept in [64, 1024].  The pairs
// are laid out longest first (by chunks, then sequence and split), so that
// the CTAs that claim them in order end together; seqbase[b] (the splits of
// the sequences before b) places each split's partial result.
__device__ void build_plan(const AttnNormParams& p) {
  __shared__ long long s_tot[kNormThreads / 32];
  __shared__ int s_max[kNormThreads / 32];
  __shared__ int s_scan[kNormThreads / 32];
  __shared__ int s_width;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long tot = 0;
  int most = 0;
  for (int b = tid; b < p.B; b += kNormThreads) {
    const int p0 = p.positions[b];
    if (seq_in_range(p0, p.K, p.max_pos)) {
      tot += p0 + p.K + 1;
      most = max(most, p0 + p.K + 1);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    most = max(most, __shfl_xor_sync(0xffffffffu, most, o));
  }
  if (lane == 0) {
    s_tot[warp] = tot;
    s_max[warp] = most;
  }
  __syncthreads();
  if (tid == 0) {
    long long all = 0;
    int mx = 0;
    for (int w = 0; w < kNormThreads / 32; ++w) {
      all += s_tot[w];
      mx = max(mx, s_max[w]);
    }
    // and at most kAttnMaxSplits splits per sequence (the merge's scratch)
    long long want = (all * p.H + p.target_items - 1) / p.target_items;
    want = max(want, (long long)((mx + kAttnMaxSplits - 1) / kAttnMaxSplits));
    const long long g = want <= p.max_split ? kAttnMinSplit : p.max_split;
    long long c = (want + g - 1) / g * g;
    if (c < kAttnMinSplit) c = kAttnMinSplit;
    if (c > kAttnMaxSplit) c = kAttnMaxSplit;
    s_width = (int)c;
  }
  __syncthreads();
  const int C = s_width, Cm = p.max_split;
  const int maxc = (C + Cm - 1) / Cm;  // chunks of a full split
  // contiguous runs of sequences per thread
  const int per = (p.B + kNormThreads - 1) / kNormThreads;
  const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
  auto splits = [&](int b, int* last_chunks) {
    const int p0 = p.positions[b];
    if (!seq_in_range(p0, p.K, p.max_pos)) return 0;
    const int keys = p0 + p.K + 1, n = (keys + C - 1) / C;
    *last_chunks = (keys - (n - 1) * C + Cm - 1) / Cm;
    return n;
  };
  int* seqbase = p.plan + 2 + 2 * p.cap_pairs;
  int mine = 0, total = 0, lc = 0;
  for (int b = b0; b < b1; ++b) mine += splits(b, &lc);
  int at = block_excl_scan(mine, s_scan, &total);
  for (int b = b0; b < b1; ++b) {
    seqbase[b] = at;
    at += splits(b, &lc);
  }
  // the pairs, by chunks from maxc down to 1
  int placed = 0;
  for (int nb = maxc; nb >= 1; --nb) {
    int cnt = 0;
    for (int b = b0; b < b1; ++b) {
      const int n = splits(b, &lc);
      if (n == 0) continue;
      cnt += (nb == maxc ? n - 1 : 0) + (lc == nb ? 1 : 0);
    }
    int bucket = 0;
    int w = placed + block_excl_scan(cnt, s_scan, &bucket);
    for (int b = b0; b < b1; ++b) {
      const int n = splits(b, &lc);
      if (n == 0) continue;
      for (int s = 0; s < n; ++s) {
        const int ch = s + 1 < n ? maxc : lc;
        if (ch != nb) continue;
        if (w < p.cap_pairs) {
          p.plan[2 + 2 * w] = b;
          p.plan[3 + 2 * w] = s;
        }
        ++w;
      }
    }
    placed += bucket;
  }
  for (int l = tid; l < p.n_item_ctr; l += kNormThreads) p.item_ctr[l] = 0;
  if (tid == 0) {
    if (total > p.cap_pairs) atomicOr(p.status, kErrInternal);  // not reachable by the sizing
    p.plan[0] = C;
    p.plan[1] = min(total, p.cap_pairs);
  }
}

// One token per block: h = embedding (layer 0) or h + the previous block's
// expert outputs summed in slot order; xa = bf16(RMSNorm(h) * g_a).  The sum
// of squares is reduced per thread, per warp, then over the warps in order.
__global__ void __launch_bounds__(kNormThreads) attn_norm_kernel(AttnNormParams p) {
  if (threadIdx.x == 0) stamp_min(p.stamps);
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
  __shared__ float red[kNormThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x, d = p.d, nc = d / 4;
  float4* hrow = reinterpret_cast<float4*>(p.h + (size_t)t * d);
  float4* hp = p.probe_hidden ? reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d) : nullptr;
  float ss = 0.f;
  if (p.first) {
    const int K1 = p.K + 1, b = t / K1, j = t - b * K1;
    const int id = j == 0 ? p.context_ids[b] : p.draft_ids[(size_t)b * p.K + (j - 1)];
    const bool ok = id >= 0 && id < p.V && seq_in_range(p.positions[b], p.K, p.max_pos);
    if (tid == 0) {
      p.bad[t] = ok ? 0 : 1;
      if (!ok) atomicOr(p.status, kErrIdRange);
    }
    const uint2* src = reinterpret_cast<const uint2*>(p.embed + (size_t)((id >= 0 && id < p.V) ? id : 0) * d);
    for (int c = tid; c < nc; c += kNormThreads) {
      const uint2 u = __ldg(src + c);
      const __nv_bfloat162* bb = reinterpret_cast<const __nv_bfloat162*>(&u);
      const float2 a = __bfloat1622float2(bb[0]), e = __bfloat1622float2(bb[1]);
      const float4 v = make_float4(a.x, a.y, e.x, e.y);
      hrow[c] = v;
      if (hp) hp[c] = v;
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  } else {
    const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * p.kS * d);
    for (int c = tid; c < nc; c += kNormThreads) {
      float4 v = hrow[c];
      float4 acc = __ldcg(yr + c);
      for (int s = 1; s < p.kS; ++s) {
        const float4 u = __ldcg(yr + (size_t)s * nc + c);
        acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
      }
      v.x += acc.x; v.y += acc.y; v.z += acc.z; v.w += acc.w;
      hrow[c] = v;
      if (hp) hp[c] = v;
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  }
  ss = warp_sum_f(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)d + p.eps);
  for (int c = tid; c < nc; c += kNormThreads) {
    const float4 v = hrow[c];
    const float4 g = __ldg(reinterpret_cast<const float4*>(p.gain) + c);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.xa + (size_t)t * d)[c] = packed;
  }
  if (p.first && blockIdx.x == 0) {
    __syncthreads();
    build_plan(p);
  }
  if (p.stamps) {
    __syncthreads();
    if (threadIdx.x == 0) stamp_max(p.stamps + 2);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// (x, y) as the sum of two bf16 pairs: hi = bf16(x, y), lo = bf16 of the rest.
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(x - hf.x, y - hf.y);
}

// An item: split s (keys k0 .. k0 + n - 1, `chunks` chunks) of sequence b,
// head hh; its partial result's slot among the step's splits, and the slot of
// its sequence's split 0 (the splits of a sequence have consecutive slots).
struct AttnItem {
  int b, s, hh, k0, n, keys, nsplit, chunks, slot0;
};

__device__ __forceinline__ AttnItem attn_item(const AttnParams& p, int C, int item) {
  AttnItem it;
  const int pair = item / p.H;
  it.hh = item - pair * p.H;
  it.b = p.plan[2 + 2 * pair];
  it.s = p.plan[3 + 2 * pair];
  it.keys = p.positions[it.b] + p.K + 1;
  it.k0 = it.s * C;
  it.n = min(it.keys, it.k0 + C) - it.k0;
  it.nsplit = (it.keys + C - 1) / C;
  it.chunks = (it.n + p.max_split - 1) / p.max_split;
  it.slot0 = p.plan[2 + 2 * p.cap_pairs + it.b];
  return it;
}

// One thread: chunk c of an item, max_split keys and values (boxes of BW dims
// x max_split rows of the head-major caches, rows past the item's keys are
// loaded but never used), into buffer `buf`, completing on full[buf].
template <int HD>
__device__ __forceinline__ void attn_issue(const CUtensorMap* map_k, const CUtensorMap* map_v,
                                           const AttnParams& p, uint8_t* kv, uint64_t* full,
                                           const AttnItem& it, int c, int buf, uint64_t pol) {
  // buffer `buf` of kAttnStages, completing on full[buf]
  constexpr int BW = HD < 64 ? HD : 64, NB = HD / BW;
  const uint32_t box = (uint32_t)p.max_split * BW * 2, tile = NB * box;
  const int row = p.row0 + ((it.b * p.H + it.hh) * p.max_pos + it.k0 + c * p.max_split);
  mbar_arrive_expect_tx(&full[buf], 2 * tile);
  uint8_t* dst = kv + (size_t)buf * 2 * tile;
#pragma unroll
  for (int x = 0; x < NB; ++x) {
    tma_load_2d(dst + x * box, map_k, &full[buf], x * BW, row, pol);
    tma_load_2d(dst + tile + x * box, map_v, &full[buf], x * BW, row, pol);
  }
}

// Persistent, one CTA per SM: 8 compute warps and one loading warp.  The
// loading warp claims items (sequence, split, head) in order from a per-layer
// counter, one item ahead, so CTAs that stream faster take more of them, and
// streams each item's keys and values through a ring of kAttnStages
// shared-memory buffers in chunks of max_split keys (2-D TMA boxes with the
// hardware swizzle), tagging each buffer with its (item, chunk); a buffer is
// refilled once the eight compute warps have released it.  It also publishes
// each claimed item's (sequence, head) one item ahead, so that the compute
// warps copy the next item's queries into shared memory while they work on
// the current one.  (Pulling chunks into L2 ahead of the ring measured slower:
// 74 against 67 us per launch.)  Each compute warp
// takes its share of a chunk's keys, 16 at a time, on the tensor cores
// (mma.sync m16n8k16) with the keys and the head's dims on the 16-row side and
// the item's queries (8 per tile, NQT tiles) as the columns:
//   S^T = K Q^T     K bf16 (exact), Q fp32 as the sum of two bf16 parts
//   online softmax per query column in the log2 domain (running max and sum)
//   O^T += V^T P^T  V bf16 (exact), P fp32 as two bf16 parts, moved from the
//                   accumulator layout to the operand layout by an 8x8
//                   transpose in registers
// so the products are those of fp32 operands to ~2^-16, accumulated in fp32.
// At the end of an item the warps' (max, sum, O) are merged in warp order
// (their O staged in the buffer of the item's last chunk, released only
// afterwards); a split's result is merged with its sequence's other splits by
// the last of them to finish, in split order.
template <int HD, int NQT>
__global__ void __launch_bounds__(kAttnThreads + 32, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const AttnParams p) {
  constexpr int KS = HD / 16;                 // k-steps of K Q^T, m-tiles of V^T P^T
  constexpr int NQ = 8 * NQT;                 // query columns
  constexpr int BW = HD < 64 ? HD : 64;       // box width (elements)
  constexpr uint32_t RB = BW * 2;             // box row bytes
  extern __shared__ uint8_t attn_raw[];
  __shared__ int s_last;
  __shared__ int s_abort;
  __shared__ int2 s_tag[kAttnStages];         // (item, chunk) of each buffer; item < 0: end
  constexpr int kClaims = 8;
  __shared__ AttnItem s_claim[kClaims];       // claimed item k (b < 0: none)
  uint8_t* kv = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K1 = p.K + 1, Cm = p.max_split;
  const uint32_t box = (uint32_t)Cm * RB, tile = (HD / BW) * box;
  float* qs = reinterpret_cast<float*>(kv + 2 * kAttnStages * (size_t)tile);  // [2][NQ][HD]
  float* mst = qs + 2 * NQ * HD;                                 // [8][NQ]
  float* lst = mst + kAttnWarps * NQ;                            // [8][NQ]
  float* wst = lst + kAttnWarps * NQ;                            // [8][NQ] warp weights
  float* wsp = wst + kAttnWarps * NQ;                            // [16][kAttnMaxSplits]
  float* tot = wsp + 16 * kAttnMaxSplits;                        // [16]
  uint64_t* full = reinterpret_cast<uint64_t*>(tot + 16);        // [kAttnStages]
  uint64_t* empty = full + kAttnStages;                          // [kAttnStages]
  if (tid == 0) {
    stamp_min(p.stamps);
    s_abort = 0;
    for (int b = 0; b < kAttnStages; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kAttnWarps);
    }
    fence_mbar_init();
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0 && p.stamps) stamp_max(p.stamps + 1);
  const int C = p.plan[0], n_items = p.plan[1] * p.H;

  if (warp == kAttnWarps) {
    // ------------------------------------------------ loading warp
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0, k = 0;
      bool ok = true;
      // the claimed item and the one claimed after it (published before the
      // first one's chunks are loaded)
      int cur = atomicAdd(p.item_ctr, 1);
      int nxt = cur < n_items ? atomicAdd(p.item_ctr, 1) : n_items;
      AttnItem it = {};
      if (cur < n_items) it = attn_item(p, C, cur);
      if (cur >= n_items) it.b = -1;
      s_claim[0] = it;
      while (ok && cur < n_items) {
        AttnItem itn = {};
        itn.b = -1;
        if (nxt < n_items) itn = attn_item(p, C, nxt);
        ++k;
        s_claim[k % kClaims] = itn;
        for (int c = 0; c < it.chunks; ++c, ++issued) {
          const int b = issued % kAttnStages;
          if (!mbar_wait(&empty[b], (uint32_t)(((issued / kAttnStages) & 1) ^ 1), &s_abort,
                         p.status)) {
            ok = false;
            break;
          }
          s_tag[b] = make_int2(cur, c);
          attn_issue<HD>(&map_k, &map_v, p, kv, full, it, c, b, pol);
        }
        cur = nxt;
        it = itn;
        if (cur < n_items) nxt = atomicAdd(p.item_ctr, 1);
      }
      if (ok) {
        // the end: a buffer tagged with no item, completed by a plain arrival
        const int b = issued % kAttnStages;
        if (mbar_wait(&empty[b], (uint32_t)(((issued / kAttnStages) & 1) ^ 1), &s_abort,
                      p.status)) {
          s_tag[b] = make_int2(-1, 0);
          mbar_arrive(&full[b]);
        }
      } else {
        // let the loads already issued land before the CTA exits
        for (int v = issued - kAttnStages; v < issued; ++v) {
          if (v < 0) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&full[v % kAttnStages], (uint32_t)((v / kAttnStages) & 1)) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else {
    // ------------------------------------------------ compute warps 0..7
    const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
    const int kpw = Cm / kAttnWarps;  // keys per warp and chunk (a multiple of 16)
    // ldmatrix row addresses within a 16-key group (which starts on a
    // multiple of 16 rows, so the swizzle's row bits are the lane's own): the
    // row's offset, and the value XORed into the 16-byte chunk index, which
    // for chunk 2 k + d (d the lane's half) is (2 k) ^ (d ^ row bits)
    auto row_x = [](int key) {
      return RB == 128 ? (key & 7) : RB == 64 ? ((key >> 1) & 3) : ((key >> 2) & 1);
    };
    const int k_key = r8 + (mi & 1) * 8, v_key = r8 + (mi >> 1) * 8;
    const uint32_t k_row = (uint32_t)k_key * RB, v_row = (uint32_t)v_key * RB;
    const int k_x = (mi >> 1) ^ row_x(k_key), v_x = (mi & 1) ^ row_x(v_key);
    auto bar = [] { named_bar_sync(1, kAttnThreads); };
    uint32_t qh[NQT][KS][2], ql[NQT][KS][2];
    float O[KS][NQT][4];
    float mq[NQT][2], lq[NQT][2];
    AttnItem it = {};
    int item = -1, p0 = 0, m = -1;
    // rows K + 1 .. NQ - 1 of both query buffers stay zero
    for (int i = tid; i < 2 * NQ * HD; i += kAttnThreads) qs[i] = 0.f;
    // the queries of an item (sequence b, head hh) into query buffer qb, one
    // 16-byte copy per thread and pass
    auto fetch_q = [&](int b, int hh, float* qb) {
      const float* src = p.q + (size_t)(b * K1) * p.d + hh * HD;
      for (int i = tid; i < K1 * HD / 4; i += kAttnThreads) {
        const int row = i / (HD / 4), c4 = i - row * (HD / 4);
        cp_async16(qb + row * HD + 4 * c4, src + (size_t)row * p.d + 4 * c4);
      }
      cp_async_commit();
    };
    for (int u = 0;; ++u) {
      const int buf = u % kAttnStages;
      // a wait that gives up raises s_abort; the barrier makes the warps leave together
      mbar_wait(&full[buf], (uint32_t)((u / kAttnStages) & 1), &s_abort, p.status);
      bar();
      if (s_abort) break;
      const int2 tag = s_tag[buf];
      if (tag.x < 0) break;
      const int c = tag.y;
      if (c == 0) {
        // a new item (the CTA's m-th): its queries are in query buffer m % 2
        // (copied while the previous item ran; the first item's now), and
        // the next item's are copied into the other buffer meanwhile; then as
        // B fragments (pre-scaled to the log2 domain), hi and lo bf16 parts
        item = tag.x;
        ++m;
        it = s_claim[m % kClaims];  // published before the item's first chunk
        p0 = it.keys - K1;
        float* qcur = qs + (m & 1) * NQ * HD;
        if (m == 0) fetch_q(it.b, it.hh, qcur);
        cp_async_wait_all();
        bar();
        const AttnItem& nx = s_claim[(m + 1) % kClaims];
        if (nx.b >= 0) fetch_q(nx.b, nx.hh, qs + ((m + 1) & 1) * NQ * HD);
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
          for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const float2 v = *reinterpret_cast<const float2*>(qcur + (nq * 8 + g) * HD + ks * 16 +
                                                                r * 8 + 2 * t4);
              split_bf16(v.x * p.scale_log2, v.y * p.scale_log2, qh[nq][ks][r], ql[nq][ks][r]);
            }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq)
            O[mt][nq][0] = O[mt][nq][1] = O[mt][nq][2] = O[mt][nq][3] = 0.f;
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq) {
          mq[nq][0] = mq[nq][1] = -INFINITY;
          lq[nq][0] = lq[nq][1] = 0.f;
        }
      }
      const uint8_t* Kt = kv + (size_t)buf * 2 * tile;
      const uint8_t* Vt = Kt + tile;
      const int n = min(Cm, it.n - c * Cm);  // keys of this chunk
      const int kc0 = it.k0 + c * Cm;        // position of its first key
      for (int kg = warp * kpw; kg < min(n, (warp + 1) * kpw); kg += 16) {
        const uint8_t* Kg = Kt + kg * RB;
        const uint8_t* Vg = Vt + kg * RB;
        // ---- S^T = K Q^T for keys kg .. kg + 15; the hi and lo parts'
        // products in separate accumulators (independent chains)
        float S[NQT][4], Sl[NQT][4];
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[nq][e] = Sl[nq][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          // A = K: matrices (keys kg.., dims ks*16..), (kg+8.., ks*16..),
          // (kg.., ks*16+8..), (kg+8.., ks*16+8..)
          constexpr int CPB = BW / 8;  // 16-byte chunks per box row
          uint32_t a[4];
          ldmatrix_x4(a, Kg + (2 * ks / CPB) * box + k_row + (((2 * ks % CPB) ^ k_x) << 4));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            mma_16816_bf16(S[nq], a, qh[nq][ks][0], qh[nq][ks][1]);
            mma_16816_bf16(Sl[nq], a, ql[nq][ks][0], ql[nq][ks][1]);
          }
        }
        // ---- causal mask, running max per query column, numerators; this
        // lane holds keys kg + g (e = 0, 1) and kg + g + 8 (e = 2, 3) of query
        // columns 2 t4 + (e & 1).  Keys past the chunk or past a query's own
        // position are masked; below the sequence's first verify position and
        // inside the chunk every key is visible to every query.
        const bool inner = kg + 16 <= n && kc0 + kg + 15 <= p0;
        uint32_t bh[NQT][2], bl[NQT][2];
        bool moved = false;
        float f[NQT][2];
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq) {
          float sv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = nq * 8 + 2 * t4 + (e & 1);
            const int kl = kg + g + ((e & 2) ? 8 : 0);
            const bool vis = q < K1 && (inner || (kl < n && kc0 + kl <= p0 + q));
            sv[e] = vis ? S[nq][e] + Sl[nq][e] : -INFINITY;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float mx = fmaxf(sv[h], sv[h + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(mq[nq][h], mx);
            moved |= mn != mq[nq][h];
            f[nq][h] = mq[nq][h] == -INFINITY ? 0.f : exp2f(mq[nq][h] - mn);
            mq[nq][h] = mn;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mn = mq[nq][e & 1];
            sv[e] = sv[e] == -INFINITY ? 0.f : exp2f(sv[e] - mn);
          }
          lq[nq][0] = lq[nq][0] * f[nq][0] + sv[0] + sv[2];
          lq[nq][1] = lq[nq][1] * f[nq][1] + sv[1] + sv[3];
          // P^T blocks (keys 0-7 and 8-15 of the group x this query tile) in
          // the accumulator layout, transposed into B fragments
          uint32_t h0, l0, h1, l1;
          split_bf16(sv[0], sv[1], h0, l0);
          split_bf16(sv[2], sv[3], h1, l1);
          bh[nq][0] = movmatrix_trans(h0);
          bh[nq][1] = movmatrix_trans(h1);
          bl[nq][0] = movmatrix_trans(l0);
          bl[nq][1] = movmatrix_trans(l1);
        }
        // what was accumulated is rescaled only when a running max moved
        if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int nq = 0; nq < NQT; ++nq) {
              O[mt][nq][0] *= f[nq][0]; O[mt][nq][1] *= f[nq][1];
              O[mt][nq][2] *= f[nq][0]; O[mt][nq][3] *= f[nq][1];
            }
        }
        // ---- O^T += V^T P^T: A = V^T (16 dims x 16 keys) per m-tile
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          // matrices (transposed): (keys kg.., dims mt*16..), (kg.., mt*16+8..),
          // (kg+8.., mt*16..), (kg+8.., mt*16+8..)
          constexpr int CPB = BW / 8;
          uint32_t a[4];
          ldmatrix_x4_trans(a, Vg + (2 * mt / CPB) * box + v_row + (((2 * mt % CPB) ^ v_x) << 4));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            mma_16816_bf16(O[mt][nq], a, bh[nq][0], bh[nq][1]);
            mma_16816_bf16(O[mt][nq], a, bl[nq][0], bl[nq][1]);
          }
        }
      }
      if (c + 1 < it.chunks) {
        // release the buffer to the loading warp
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[buf]);
        continue;
      }

      // ---- end of the item: the warps' states, then merged in warp order;
      // O^T goes to this (last) chunk's buffer as [8][NQ][HD], released after
      float* ost = reinterpret_cast<float*>(kv + (size_t)buf * 2 * tile);
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          lq[nq][h] += __shfl_xor_sync(0xffffffffu, lq[nq][h], 4);
          lq[nq][h] += __shfl_xor_sync(0xffffffffu, lq[nq][h], 8);
          lq[nq][h] += __shfl_xor_sync(0xffffffffu, lq[nq][h], 16);
          if (g == 0) {
            mst[warp * NQ + nq * 8 + 2 * t4 + h] = mq[nq][h];
            lst[warp * NQ + nq * 8 + 2 * t4 + h] = lq[nq][h];
          }
        }
      bar();  // every warp is done with the buffer's keys and values
      float* ow = ost + (size_t)warp * NQ * HD;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ow[(nq * 8 + 2 * t4 + (e & 1)) * HD + mt * 16 + g + ((e & 2) ? 8 : 0)] = O[mt][nq][e];
      bar();
      if (tid < NQ) {
        // per query: the merged max and sum, and each warp's weight
        float M = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mst[w * NQ + tid]);
        float L = 0.f;
        for (int w = 0; w < kAttnWarps; ++w) {
          const float mw = mst[w * NQ + tid];
          const float ww = mw == -INFINITY ? 0.f : exp2f(mw - M);
          wst[w * NQ + tid] = ww;
          L = fmaf(lst[w * NQ + tid], ww, L);
        }
        mst[tid] = M;  // warp 0's slots now hold the merged values
        lst[tid] = L;
      }
      bar();
      const int outs = K1 * HD;
      if (it.nsplit == 1) {
        for (int i = tid; i < outs; i += kAttnThreads) {
          const int j = i / HD, dim = i - j * HD;
          float a = 0.f;
          for (int w = 0; w < kAttnWarps; ++w)
            a = fmaf(ost[((size_t)w * NQ + j) * HD + dim], wst[w * NQ + j], a);
          p.o[(size_t)(it.b * K1 + j) * p.d + it.hh * HD + dim] = __float2bfloat16_rn(a / lst[j]);
        }
      } else {
        // this split's (max, sum, unnormalised output) per query
        const int pitch = HD + 2;
        float* mine = p.part + ((size_t)(it.slot0 + it.s) * p.H + it.hh) * K1 * pitch;
        for (int i = tid; i < outs; i += kAttnThreads) {
          const int j = i / HD, dim = i - j * HD;
          float a = 0.f;
          for (int w = 0; w < kAttnWarps; ++w)
            a = fmaf(ost[((size_t)w * NQ + j) * HD + dim], wst[w * NQ + j], a);
          mine[j * pitch + 2 + dim] = a;
        }
        for (int j = tid; j < K1; j += kAttnThreads) {
          mine[j * pitch] = mst[j];
          mine[j * pitch + 1] = lst[j];
        }
        // the warps' writes, ordered by the barrier, released by one fence
        bar();
        if (tid == 0) {
          __threadfence();
          s_last = atomicAdd(p.arrive + it.b * p.H + it.hh, 1) == it.nsplit - 1;
        }
        bar();
        if (s_last) {
          __threadfence();
          // merge the splits in order: split s' in slot (slot0 + s') * H + hh
          const int first = it.slot0 * p.H + it.hh;
          for (int j = warp; j < K1; j += kAttnWarps) {
            float M = -INFINITY;
            for (int q = lane; q < it.nsplit; q += 32) {
              const float* pq = p.part + (size_t)(first + q * p.H) * K1 * pitch + j * pitch;
              if (__ldcg(pq + 1) > 0.f) M = fmaxf(M, __ldcg(pq));
            }
            M = warp_max_f(M);
            float Ls = 0.f;
            for (int q = lane; q < it.nsplit; q += 32) {
              const float* pq = p.part + (size_t)(first + q * p.H) * K1 * pitch + j * pitch;
              const float lsp = __ldcg(pq + 1);
              const float wq = lsp > 0.f ? exp2f(__ldcg(pq) - M) : 0.f;
              wsp[j * kAttnMaxSplits + q] = wq;
              Ls = fmaf(lsp, wq, Ls);
            }
            Ls = warp_sum_f(Ls);
            if (lane == 0) tot[j] = Ls;
          }
          bar();
          for (int i = tid; i < outs; i += kAttnThreads) {
            const int j = i / HD, dim = i - j * HD;
            float A = 0.f;
#pragma unroll 4
            for (int q = 0; q < it.nsplit; ++q)
              A = fmaf(
                  __ldcg(p.part + (size_t)(first + q * p.H) * K1 * pitch + j * pitch + 2 + dim),
                  wsp[j * kAttnMaxSplits + q], A);
            p.o[(size_t)(it.b * K1 + j) * p.d + it.hh * HD + dim] =
                __float2bfloat16_rn(A / tot[j]);
          }
          if (tid == 0) p.arrive[it.b * p.H + it.hh] = 0;
        }
      }
      bar();  // the warps' states, Q and the merge scratch are reused
      if (lane == 0) mbar_arrive(&empty[buf]);
    }
  }
  __syncthreads();
  if (tid == 0 && p.stamps) stamp_max(p.stamps + 2);
}

// Packed q/k/v rows of one layer: rows [0, d) q and [d, 2d) k with each head's
// dims ordered (0, hd/2, 1, hd/2 + 1, ...), rows [2d, 3d) v as given, zero
// rows up to rows_pad.  One block per row.
__global__ void repack_qkv_kernel(__nv_bfloat16* dst, const __nv_bfloat16* wq,
                                  const __nv_bfloat16* wk, const __nv_bfloat16* wv, int d, int hd,
                                  int rows_pad) {
  const int r = blockIdx.x;
  if (r >= rows_pad) return;
  uint4* out = reinterpret_cast<uint4*>(dst + (size_t)r * d);
  const int part = r / d;
  const uint4* src = nullptr;
  if (part < 3) {
    const int f = r - part * d;
    int row = f;
    if (part < 2) {
      const int head = f / hd, w = f - head * hd;
      row = head * hd + (w >> 1) + ((w & 1) ? hd / 2 : 0);
    }
    const __nv_bfloat16* w = part == 0 ? wq : part == 1 ? wk : wv;
    src = reinterpret_cast<const uint4*>(w + (size_t)row * d);
  }
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x)
    out[c] = src ? src[c] : make_uint4(0u, 0u, 0u, 0u);
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int HD, int NQT>
cudaError_t launch_attn_t(const CUtensorMap& map_k, const CUtensorMap& map_v, const AttnParams& p,
                          int grid, cudaStream_t s, bool pdl) {
  const size_t smem = attn_smem_bytes(HD, 8 * NQT);
  auto kern = attn_kernel<HD, NQT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kAttnThreads + 32), smem, s, pdl, map_k, map_v, p);
}

template <int HD>
cudaError_t launch_attn_hd(const CUtensorMap& map_k, const CUtensorMap& map_v, const AttnParams& p,
                           int grid, cudaStream_t s, bool pdl) {
  return p.K + 1 <= 8 ? launch_attn_t<HD, 1>(map_k, map_v, p, grid, s, pdl)
                      : launch_attn_t<HD, 2>(map_k, map_v, p, grid, s, pdl);
}

}  // namespace

size_t attn_smem_bytes(int hd, int nq) {
  const size_t cm = (size_t)attn_max_split(hd);
  return 1024 /* alignment */ + 2 * kAttnStages * cm * hd * 2 +
         ((size_t)2 * nq * hd + 3 * kAttnWarps * nq + 16 * kAttnMaxSplits + 16) * sizeof(float) +
         2 * kAttnStages * sizeof(uint64_t);
}

cudaError_t launch_attn_norm(const AttnNormParams& p, cudaStream_t s, bool pdl) {
  return launch_pdl(attn_norm_kernel, dim3(p.T), dim3(kNormThreads), 0, s, pdl, p);
}

cudaError_t launch_attn(const CUtensorMap& map_k, const CUtensorMap& map_v, const AttnParams& p,
                        int grid, cudaStream_t s, bool pdl) {
  switch (p.hd) {
    case 16: return launch_attn_hd<16>(map_k, map_v, p, grid, s, pdl);
    case 32: return launch_attn_hd<32>(map_k, map_v, p, grid, s, pdl);
    case 64: return launch_attn_hd<64>(map_k, map_v, p, grid, s, pdl);
    case 128: return launch_attn_hd<128>(map_k, map_v, p, grid, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_repack_qkv(__nv_bfloat16* dst, const __nv_bfloat16* wq,
                              const __nv_bfloat16* wk, const __nv_bfloat16* wv, int d, int hd,
                              int rows_pad, cudaStream_t s) {
  repack_qkv_kernel<<<rows_pad, 128, 0, s>>>(dst, wq, wk, wv, d, hd, rows_pad);
  return cudaGetLastError();
}

}  // namespace mv
