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
constexpr int kAttnThreads = 256;
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

__device__ __forceinline__ void bf16x8_to_f(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(b[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ bool seq_in_range(int p0, int K, int max_pos) {
  return p0 >= 0 && p0 <= max_pos - 1 - K;
}

// Layer 0, block 0: the attention's (sequence, split) pairs for this step.
// keys_b = pos_b + K + 1 (0 for a sequence out of range); the split width is
// the larger of the total keys x heads over the wanted items and the longest
// sequence over kAttnMaxSplits, rounded up to a whole number of chunks
// (max_split keys, or 64 below one chunk) and kept in [64, 1024]; a
// sequence's pairs are consecutive, in split order.
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
  const int C = s_width;
  // contiguous runs of sequences per thread, then an exclusive scan of the
  // runs' pair counts over the block
  const int per = (p.B + kNormThreads - 1) / kNormThreads;
  const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
  int mine = 0;
  for (int b = b0; b < b1; ++b) {
    const int p0 = p.positions[b];
    if (seq_in_range(p0, p.K, p.max_pos)) mine += (p0 + p.K + 1 + C - 1) / C;
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += s_scan[w];
  int at = base + incl - mine;
  for (int b = b0; b < b1; ++b) {
    const int p0 = p.positions[b];
    if (!seq_in_range(p0, p.K, p.max_pos)) continue;
    const int n = (p0 + p.K + 1 + C - 1) / C;
    for (int s = 0; s < n; ++s, ++at) {
      if (at < p.cap_pairs) {
        p.plan[2 + 2 * at] = b;
        p.plan[3 + 2 * at] = s;
      }
    }
  }
  for (int l = tid; l < p.n_item_ctr; l += kNormThreads) p.item_ctr[l] = 0;
  if (tid == kNormThreads - 1) {
    const int total = base + incl;
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

// Byte offset of 16-byte chunk cb of row r in a TMA box whose rows are rb
// bytes (128, 64 or 32) and which was written with the matching swizzle: the
// offset's bits 4.. are XORed with its bits 7.. (3, 2 or 1 of them).
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t cb, uint32_t rb) {
  const uint32_t o = r * rb + cb * 16;
  const uint32_t mask = rb == 128 ? 7u : rb == 64 ? 3u : 1u;
  return o ^ (((o >> 7) & mask) << 4);
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

struct AttnItem {
  int b, s, hh, k0, n, keys, nsplit, pair, chunks;
};

__device__ __forceinline__ AttnItem attn_item(const AttnParams& p, int C, int item) {
  AttnItem it;
  it.pair = item / p.H;
  it.hh = item - it.pair * p.H;
  it.b = p.plan[2 + 2 * it.pair];
  it.s = p.plan[3 + 2 * it.pair];
  it.keys = p.positions[it.b] + p.K + 1;
  it.k0 = it.s * C;
  it.n = min(it.keys, it.k0 + C) - it.k0;
  it.nsplit = (it.keys + C - 1) / C;
  it.chunks = (it.n + p.max_split - 1) / p.max_split;
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

// Persistent, one CTA per SM, 8 warps.  Items (sequence, split, head) are
// claimed in order from a per-layer counter, one item ahead of use, so CTAs
// that stream faster take more of them.  An item's keys and values stream
// through a ring of kAttnStages shared-memory buffers in chunks of max_split
// keys (2-D TMA boxes with the hardware swizzle), one thread keeping the next
// chunks in flight while the CTA works on the current one.  Each warp takes its
// share of a chunk's keys, 16 at a time, on the tensor cores (mma.sync
// m16n8k16) with the keys and the head's dims on the 16-row side and the
// item's queries (8 per tile, NQT tiles) as the columns:
//   S^T = K Q^T     K bf16 (exact), Q fp32 as the sum of two bf16 parts
//   online softmax per query column in the log2 domain (running max and sum)
//   O^T += V^T P^T  V bf16 (exact), P fp32 as two bf16 parts, moved from the
//                   accumulator layout to the operand layout by an 8x8
//                   transpose in registers
// so the products are those of fp32 operands to ~2^-16, accumulated in fp32.
// At the end of an item the warps' (max, sum, O) are merged in warp order
// (their O staged in the buffer of the item's last chunk, free until the ring
// comes round to it); a split's result is merged with its sequence's other
// splits by the last of them to finish, in split order.
template <int HD, int NQT>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v, const AttnParams p) {
  constexpr int KS = HD / 16;                 // k-steps of K Q^T, m-tiles of V^T P^T
  constexpr int NQ = 8 * NQT;                 // query columns
  constexpr int BW = HD < 64 ? HD : 64;       // box width (elements)
  constexpr uint32_t RB = BW * 2;             // box row bytes
  constexpr int kRing = kAttnStages + 1;      // items between claim and use
  extern __shared__ uint8_t attn_raw[];
  __shared__ int s_last;
  __shared__ int s_abort;
  __shared__ int s_item[kRing];
  uint8_t* kv = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_raw) + 1023) &
                                           ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
  const int K1 = p.K + 1, Cm = p.max_split;
  const uint32_t box = (uint32_t)Cm * RB, tile = (HD / BW) * box;
  float* qs = reinterpret_cast<float*>(kv + 2 * kAttnStages * (size_t)tile);  // [NQ][HD]
  float* mst = qs + NQ * HD;                                     // [8][NQ]
  float* lst = mst + kAttnWarps * NQ;                            // [8][NQ]
  float* wst = lst + kAttnWarps * NQ;                            // [8][NQ] warp weights
  float* wsp = wst + kAttnWarps * NQ;                            // [16][kAttnMaxSplits]
  float* tot = wsp + 16 * kAttnMaxSplits;                        // [16]
  uint64_t* full = reinterpret_cast<uint64_t*>(tot + 16);
  if (tid == 0) {
    stamp_min(p.stamps);
    s_abort = 0;
    for (int b = 0; b < kAttnStages; ++b) mbar_init(&full[b], 1);
    fence_mbar_init();
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0 && p.stamps) stamp_max(p.stamps + 1);
  const int C = p.plan[0], n_items = p.plan[1] * p.H;
  const int kpw = Cm / kAttnWarps;  // keys per warp and chunk (a multiple of 16)
  const uint64_t pol = policy_evict_first();
  // thread 0: the item whose chunks are being loaded (< 0: none left), its
  // next chunk, the items claimed and the loads issued so far, and the buffers
  // with a load not yet waited for (bit b)
  int nx_item = -1, nx_chunk = 0, claimed = 0, issued = 0;
  uint32_t pending = 0;
  AttnItem nx;
  auto claim = [&]() {
    const int it = atomicAdd(p.item_ctr, 1);
    nx_item = it < n_items ? it : -1;
    s_item[claimed % kRing] = nx_item;
    ++claimed;
    if (nx_item >= 0) nx = attn_item(p, C, nx_item);
    nx_chunk = 0;
  };
  auto issue_next = [&]() {
    attn_issue<HD>(&map_k, &map_v, p, kv, full, nx, nx_chunk, issued % kAttnStages, pol);
    pending |= 1u << (issued % kAttnStages);
    ++issued;
    if (++nx_chunk == nx.chunks) claim();
  };
  if (tid == 0) {
    claim();
    for (int k = 0; k < kAttnStages - 1 && nx_item >= 0; ++k) issue_next();
  }
  __syncthreads();
  int u = 0;  // chunks consumed so far by this CTA
  bool aborted = false;
  for (int m = 0; !aborted; ++m) {
    const int item = s_item[m % kRing];
    if (item < 0) break;
    const AttnItem it = attn_item(p, C, item);
    const int p0 = it.keys - K1;
    // Q of the item's queries into shared memory (rows >= K + 1 zero), then
    // as B fragments (pre-scaled to the log2 domain), hi and lo bf16 parts
    {
      const float* qb = p.q + (size_t)(it.b * K1) * p.d + it.hh * HD;
      for (int i = tid; i < NQ * HD / 4; i += kAttnThreads) {
        const int row = i / (HD / 4), c4 = i - row * (HD / 4);
        reinterpret_cast<float4*>(qs)[i] =
            row < K1 ? __ldcg(reinterpret_cast<const float4*>(qb + (size_t)row * p.d) + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncthreads();
    uint32_t qh[NQT][KS][2], ql[NQT][KS][2];
#pragma unroll
    for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float2 v =
              *reinterpret_cast<const float2*>(qs + (nq * 8 + g) * HD + ks * 16 + r * 8 + 2 * t4);
          split_bf16(v.x * p.scale_log2, v.y * p.scale_log2, qh[nq][ks][r], ql[nq][ks][r]);
        }
    // O^T [dims x queries] fragments; per query column of this lane (2 t4 + e
    // of each query tile) the running max and this lane's part of the sum
    float O[KS][NQT][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq) O[mt][nq][0] = O[mt][nq][1] = O[mt][nq][2] = O[mt][nq][3] = 0.f;
    float mq[NQT][2], lq[NQT][2];
#pragma unroll
    for (int nq = 0; nq < NQT; ++nq) {
      mq[nq][0] = mq[nq][1] = -INFINITY;
      lq[nq][0] = lq[nq][1] = 0.f;
    }

    int last_buf = 0;
    for (int c = 0; c < it.chunks; ++c, ++u) {
      const int buf = u % kAttnStages;
      last_buf = buf;
      // the buffer of chunk u - 1 (finished by every thread) takes the next load
      if (tid == 0 && nx_item >= 0) issue_next();
      // a wait that gives up raises s_abort; the barrier makes the CTA leave together
      mbar_wait(&full[buf], (uint32_t)((u / kAttnStages) & 1), &s_abort, p.status);
      __syncthreads();
      if (s_abort) {
        aborted = true;
        break;
      }
      if (tid == 0) pending &= ~(1u << buf);
      const uint8_t* Kt = kv + (size_t)buf * 2 * tile;
      const uint8_t* Vt = Kt + tile;
      const int n = min(Cm, it.n - c * Cm);  // keys of this chunk
      const int kc0 = it.k0 + c * Cm;        // position of its first key
      for (int kg = warp * kpw; kg < min(n, (warp + 1) * kpw); kg += 16) {
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
          const int key = kg + r8 + (mi & 1) * 8;
          const int dc = ks * 2 + (mi >> 1);  // 16-byte chunk of the head's dims
          uint32_t a[4];
          ldmatrix_x4(a, Kt + (dc * 8 / BW) * box + swz(key, dc % (BW / 8), RB));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            mma_16816_bf16(S[nq], a, qh[nq][ks][0], qh[nq][ks][1]);
            mma_16816_bf16(Sl[nq], a, ql[nq][ks][0], ql[nq][ks][1]);
          }
        }
        // ---- causal mask, running max per query column, numerators; this
        // lane holds keys kg + g (e = 0, 1) and kg + g + 8 (e = 2, 3) of query
        // columns 2 t4 + (e & 1)
        uint32_t bh[NQT][2], bl[NQT][2];
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq) {
          float sv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = nq * 8 + 2 * t4 + (e & 1);
            const int kl = kg + g + ((e & 2) ? 8 : 0);
            const bool vis = q < K1 && kl < n && kc0 + kl <= p0 + q;
            sv[e] = vis ? S[nq][e] + Sl[nq][e] : -INFINITY;
          }
          float f[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float mx = fmaxf(sv[h], sv[h + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(mq[nq][h], mx);
            f[h] = mq[nq][h] == -INFINITY ? 0.f : exp2f(mq[nq][h] - mn);
            mq[nq][h] = mn;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float mn = mq[nq][e & 1];
            sv[e] = sv[e] == -INFINITY ? 0.f : exp2f(sv[e] - mn);
          }
          lq[nq][0] = lq[nq][0] * f[0] + sv[0] + sv[2];
          lq[nq][1] = lq[nq][1] * f[1] + sv[1] + sv[3];
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            O[mt][nq][0] *= f[0]; O[mt][nq][1] *= f[1];
            O[mt][nq][2] *= f[0]; O[mt][nq][3] *= f[1];
          }
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
        // ---- O^T += V^T P^T: A = V^T (16 dims x 16 keys) per m-tile
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          // matrices (transposed): (keys kg.., dims mt*16..), (kg.., mt*16+8..),
          // (kg+8.., mt*16..), (kg+8.., mt*16+8..)
          const int key = kg + r8 + (mi >> 1) * 8;
          const int dc = mt * 2 + (mi & 1);
          uint32_t a[4];
          ldmatrix_x4_trans(a, Vt + (dc * 8 / BW) * box + swz(key, dc % (BW / 8), RB));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            mma_16816_bf16(O[mt][nq], a, bh[nq][0], bh[nq][1]);
            mma_16816_bf16(O[mt][nq], a, bl[nq][0], bl[nq][1]);
          }
        }
      }
      __syncthreads();  // the buffer is reloaded kAttnStages - 1 chunks on
    }
    if (aborted) break;

    // ---- the warps' states, then merged in warp order; O^T goes to the
    // buffer of the item's last chunk (the next load into it is issued at the
    // start of the next chunk, after this item) as [8][NQ][HD]
    float* ost = reinterpret_cast<float*>(kv + (size_t)last_buf * 2 * tile);
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
    float* ow = ost + (size_t)warp * NQ * HD;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          ow[(nq * 8 + 2 * t4 + (e & 1)) * HD + mt * 16 + g + ((e & 2) ? 8 : 0)] = O[mt][nq][e];
    __syncthreads();
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
    __syncthreads();
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
      float* mine = p.part + (size_t)item * K1 * pitch;
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
      // the CTA's writes, ordered by the barrier, released by one fence
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.arrive + it.b * p.H + it.hh, 1) == it.nsplit - 1;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        // merge the splits in order: item of split s' = (pair - s + s') * H + hh
        const int first = (it.pair - it.s) * p.H + it.hh;
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
        __syncthreads();
        for (int i = tid; i < outs; i += kAttnThreads) {
          const int j = i / HD, dim = i - j * HD;
          float A = 0.f;
#pragma unroll 4
          for (int q = 0; q < it.nsplit; ++q)
            A = fmaf(__ldcg(p.part + (size_t)(first + q * p.H) * K1 * pitch + j * pitch + 2 + dim),
                     wsp[j * kAttnMaxSplits + q], A);
          p.o[(size_t)(it.b * K1 + j) * p.d + it.hh * HD + dim] = __float2bfloat16_rn(A / tot[j]);
        }
        if (tid == 0) p.arrive[it.b * p.H + it.hh] = 0;
      }
    }
    __syncthreads();  // the warps' states, Q and the merge scratch are reused
  }
  // a wait that gave up: let the loads already issued land before the CTA
  // exits (chunk v went to buffer v % kAttnStages; the loads of chunks u ..
  // issued - 1 were not waited for)
  if (tid == 0) {
    for (int v = u; v < issued; ++v) {
      const int b = v % kAttnStages;
      if (!(pending & (1u << b))) continue;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&full[b], (uint32_t)((v / kAttnStages) & 1)) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
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
  return launch_pdl(kern, dim3(grid), dim3(kAttnThreads), smem, s, pdl, map_k, map_v, p);
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
         ((size_t)nq * hd + 3 * kAttnWarps * nq + 16 * kAttnMaxSplits + 16) * sizeof(float) +
         kAttnStages * sizeof(uint64_t);
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
