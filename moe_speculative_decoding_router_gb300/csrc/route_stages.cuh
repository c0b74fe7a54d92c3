// The routing's stages for one token, as device functions shared by the
// routing kernel (one block per token) and the expert-FFN kernel's routing
// tasks (the single-kernel layer for a few verify tokens), so that a token's
// residual stream, normalised row, router logits and selection have the same
// bits whichever kernel routes it.
//
// Decoder block of "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser
// With Built-In Speculative Decoding", architecture paragraph: RMSNorm before
// the MoE block, a softmax router over 64 experts with top-6 selection, two
// shared experts; the block's output is added to the residual stream.
#pragma once

#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace mv {
namespace rs {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 u) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
  float2 a = __bfloat1622float2(b[0]), c = __bfloat1622float2(b[1]);
  return make_float4(a.x, a.y, c.x, c.y);
}

// Sum of squares of a float4 chunk (x*x, then y, z, w by fused multiply-adds),
// the RMSNorm scale 1 / sqrt(ss / d + eps), and the bf16 of v * r * g: one
// definition for every norm path, so a token's norm has the same bits in every
// block shape.
__device__ __forceinline__ float sumsq4(float4 v) {
  float q = __fmul_rn(v.x, v.x);
  q = __fmaf_rn(v.y, v.y, q);
  q = __fmaf_rn(v.z, v.z, q);
  return __fmaf_rn(v.w, v.w, q);
}

__device__ __forceinline__ float norm_scale(float tot, int d, float eps) {
  return rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)d), eps));
}

__device__ __forceinline__ uint2 norm_pack(float4 v, float r, float4 g) {
  __nv_bfloat162 lo = __halves2bfloat162(__float2bfloat16_rn(__fmul_rn(__fmul_rn(v.x, r), g.x)),
                                         __float2bfloat16_rn(__fmul_rn(__fmul_rn(v.y, r), g.y)));
  __nv_bfloat162 hi = __halves2bfloat162(__float2bfloat16_rn(__fmul_rn(__fmul_rn(v.z, r), g.z)),
                                         __float2bfloat16_rn(__fmul_rn(__fmul_rn(v.w, r), g.w)));
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  return packed;
}

// acc[j] = y[0][c_j] + y[1][c_j] + ... + y[kS-1][c_j] (fp32, slot order) for
// NC float4 chunks c_j of tokens' expert outputs y [kS, nc] at yr[j] (chunks
// c_j >= nc are skipped).  Slots go in fixed groups of 8 whose loads are all
// issued before the first add, so the NC chunks cost one memory round trip
// per 8 slots.
template <int NC>
__device__ __forceinline__ void sum_slots(const float4* const (&yr)[NC], int nc, int kS,
                                          const int (&c)[NC], float4 (&acc)[NC]) {
  for (int s0 = 0; s0 < kS; s0 += 8) {
    float4 u[8][NC];
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
      for (int j = 0; j < NC; ++j)
        u[q][j] = (s0 + q < kS && c[j] < nc) ? __ldcg(yr[j] + (size_t)(s0 + q) * nc + c[j])
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        if (s0 + q == 0) {
          acc[j] = u[q][j];
        } else if (s0 + q < kS) {
          acc[j].x += u[q][j].x; acc[j].y += u[q][j].y;
          acc[j].z += u[q][j].z; acc[j].w += u[q][j].w;
        }
      }
  }
}

// Router-logit partition over the warps: 16-expert tiles x K splits.
__host__ __device__ inline int route_ksplit(int E) {
  const int n_mt = (E + 15) / 16;
  return n_mt >= 16 ? 1 : 16 / n_mt;
}

// Shared-memory bytes of the staged router weights: d/64 panels of E rows x
// 128 bytes (64 bf16), 128-byte swizzled, each panel 1024-byte aligned.
__host__ __device__ inline size_t route_wr_panel(int E) { return (size_t)((E + 7) / 8) * 1024; }

// Residual stream, RMSNorm and normalised bf16 row xb of one token t, all
// threads of a block of NW warps, after the wait for the previous kernel.
// The row's d / 4 float4 chunks form groups of 32; warp w takes groups w,
// w + NW, ... (lane l chunk 32 * group + l), NB groups' loads issued
// together.  The source: the embedding row of the token's id (ids outside
// [0, V) flag the token and read row 0), the bf16 input row, h plus the
// embedding row, h as it stands, or (combine) h plus the previous block's
// expert outputs summed in slot order (routed slots in selection order, then
// the shared experts).  h is written back (not for source kSrcH), and the
// hidden probe.  The sum of squares is reduced per group over the lanes, then
// over the groups in order, whatever NW is.  gs: the gain [d] in shared
// memory; red: MAXG floats of shared memory (rows of up to 128 MAXG).
template <int SRC, int NW, int MAXG = 64>
__device__ void norm_token(const RouteParams& p, int t, const float* gs, __nv_bfloat16* xb,
                           float* red) {
  constexpr int NT = (MAXG + NW - 1) / NW;  // groups per warp at most
  constexpr int NB = NW >= 16 ? 1 : 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, nc = d / 4, ng = (nc + 31) / 32, kS = p.k + p.S;
  float4* hg = reinterpret_cast<float4*>(p.h + (size_t)t * d);
  auto chunk = [&](int i) {
    const int g = warp + NW * i;
    return g < ng ? min(g * 32 + lane, nc) : nc;
  };
  float4 v[NT];
  if (SRC == kSrcCombine) {
    const float4* y0 = reinterpret_cast<const float4*>(p.y + (size_t)t * kS * d);
#pragma unroll
    for (int i0 = 0; i0 < NT; i0 += NB) {
      if (warp + NW * i0 >= ng) break;
      const float4* yr[NB];
      int cj[NB];
      float4 hh[NB], acc[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        yr[j] = y0;
        cj[j] = i0 + j < NT ? chunk(i0 + j) : nc;
        hh[j] = cj[j] < nc ? __ldcg(hg + cj[j]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      sum_slots<NB>(yr, nc, kS, cj, acc);
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (i0 + j < NT)
          v[i0 + j] = make_float4(hh[j].x + acc[j].x, hh[j].y + acc[j].y, hh[j].z + acc[j].z,
                                  hh[j].w + acc[j].w);
    }
  } else {
    const uint2* src = nullptr;
    if (SRC == kSrcEmbed || SRC == kSrcEmbedAdd) {
      const int b = t / (p.K + 1), i = t % (p.K + 1);
      const int id = (i == 0) ? p.context_ids[b] : p.draft_ids[(size_t)b * p.K + (i - 1)];
      const bool ok = (id >= 0 && id < p.V);
      if (threadIdx.x == 0) {
        p.bad[t] = ok ? 0 : 1;
        if (!ok) atomicOr(p.status, kErrIdRange);
      }
      src = reinterpret_cast<const uint2*>(p.embed + (size_t)(ok ? id : 0) * d);
    } else if (SRC == kSrcBf16) {
      src = reinterpret_cast<const uint2*>(p.h_in + (size_t)t * d);
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) {
      if (warp + NW * i >= ng) break;
      const int c = chunk(i);
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < nc) {
        if (SRC == kSrcH) {
          // h as the previous launch (the attention's output projection) left it
          x = __ldcg(hg + c);
        } else {
          x = bf16x4_to_f4(__ldg(src + c));
          if (SRC == kSrcEmbedAdd) {
            // the running state, written by the previous launch: read after the wait
            const float4 h0 = __ldcg(hg + c);
            x = make_float4(h0.x + x.x, h0.y + x.y, h0.z + x.z, h0.w + x.w);
          }
        }
      }
      v[i] = x;
    }
  }
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int g = warp + NW * i;
    if (g >= ng) break;
    const int c = chunk(i);
    float sq = 0.f;
    if (c < nc) {
      if (SRC != kSrcH) hg[c] = v[i];
      if (p.probe_hidden) reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d)[c] = v[i];
      sq = sumsq4(v[i]);
    }
    sq = warp_sum(sq);
    if (lane == 0) red[g] = sq;
  }
  __syncthreads();
  float tot = 0.f;
  for (int g = 0; g < ng; ++g) tot += red[g];
  const float r = norm_scale(tot, d, p.eps);
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    if (warp + NW * i >= ng) break;
    const int c = chunk(i);
    if (c < nc)
      reinterpret_cast<uint2*>(xb)[c] = norm_pack(v[i], r, reinterpret_cast<const float4*>(gs)[c]);
  }
}

// Router logits z [ntok, E] (shared memory) of the block's <= 8 normalised
// rows xb (row pitch `pitch`), all threads of a block of `nwarps` warps, on
// the tensor cores: z^T = W_r xhat^T as 16x8x16 tiles, rows = experts,
// columns = the block's tokens (columns >= ntok are not used), fp32
// accumulation.  Unit u covers expert tile u % n_mt and the u / n_mt-th share
// of the 64-column panels; a panel is four MMA steps on two alternating
// accumulators, and the next panel's fragments load while the current
// panel's MMAs issue.  The partial sums (part: ksplit x 16 n_mt x 8 floats)
// are added in K-split order, then the bias.  WR: the router weights are
// staged in shared memory (wr_s, d / 64 swizzled panels), else read through
// L1.  TPB bounds the token rows read.  Ends with the block synchronised.
template <int TPB, bool WR>
__device__ void router_logits(const RouteParams& p, const uint8_t* wr_s, const __nv_bfloat16* xb,
                              int pitch, float* part, float* zs, int ntok, int nwarps, bool ok) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nthreads = nwarps * 32;
  const int d = p.d, E = p.E;
  const int n_mt = (E + 15) / 16, ksplit = route_ksplit(E);
  const size_t panel = route_wr_panel(E);
  if (ok) {
    const int npan = d / 64;
    const int pper = (npan + ksplit - 1) / ksplit;
    const int g = lane >> 2, t4 = lane & 3;
    const __nv_bfloat16* xrow = xb + (size_t)min(g, TPB - 1) * pitch + 2 * t4;
    for (int u = warp; u < n_mt * ksplit; u += nwarps) {
      const int m0 = (u % n_mt) * 16, ks = u / n_mt;
      const int pb = ks * pper, pe = min(npan, pb + pper);
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // WR: this lane's ldmatrix row ar and the byte offsets of its four
      // 16-byte chunks in a panel (chunk c of row r sits at r * 128 +
      // ((c ^ (r % 8)) * 16)); otherwise the rows of its direct loads
      const int mi = lane >> 3;
      const int ar = min(m0 + (lane & 7) + (mi & 1) * 8, E - 1);
      uint32_t off[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        off[j] = (uint32_t)ar * 128u + ((uint32_t)(((j << 1) | (mi >> 1)) ^ (ar & 7)) << 4);
      const __nv_bfloat16* r0 = p.Wr + (size_t)min(m0 + g, E - 1) * d + 2 * t4;
      const __nv_bfloat16* r1 = p.Wr + (size_t)min(m0 + g + 8, E - 1) * d + 2 * t4;
      auto load_panel = [&](int pn, uint32_t(&a)[4][4], uint32_t(&b)[4][2]) {
        const uint8_t* pbase = wr_s + (size_t)pn * panel;
        const __nv_bfloat16* xp = xrow + pn * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (WR) {
            ldmatrix_x4(a[j], pbase + off[j]);
          } else {
            const int k0 = pn * 64 + j * 16;
            a[j][0] = __ldg(reinterpret_cast<const uint32_t*>(r0 + k0));
            a[j][1] = __ldg(reinterpret_cast<const uint32_t*>(r1 + k0));
            a[j][2] = __ldg(reinterpret_cast<const uint32_t*>(r0 + k0 + 8));
            a[j][3] = __ldg(reinterpret_cast<const uint32_t*>(r1 + k0 + 8));
          }
          b[j][0] = *reinterpret_cast<const uint32_t*>(xp + j * 16);
          b[j][1] = *reinterpret_cast<const uint32_t*>(xp + j * 16 + 8);
        }
      };
      auto mma_panel = [&](const uint32_t(&a)[4][4], const uint32_t(&b)[4][2]) {
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_16816_bf16(acc[j & 1], a[j], b[j][0], b[j][1]);
      };
      uint32_t fa[2][4][4], fb[2][4][2];
      if (pb < pe) load_panel(pb, fa[0], fb[0]);
      for (int pn = pb; pn < pe; pn += 2) {
        if (pn + 1 < pe) load_panel(pn + 1, fa[1], fb[1]);
        mma_panel(fa[0], fb[0]);
        if (pn + 2 < pe) load_panel(pn + 2, fa[0], fb[0]);
        if (pn + 1 < pe) mma_panel(fa[1], fb[1]);
      }
      float* pt = part + ((size_t)ks * n_mt * 16 + m0) * 8;
      pt[g * 8 + 2 * t4] = acc[0][0] + acc[1][0];
      pt[g * 8 + 2 * t4 + 1] = acc[0][1] + acc[1][1];
      pt[(g + 8) * 8 + 2 * t4] = acc[0][2] + acc[1][2];
      pt[(g + 8) * 8 + 2 * t4 + 1] = acc[0][3] + acc[1][3];
    }
  }
  __syncthreads();
  if (ok) {
    for (int i = tid; i < ntok * E; i += nthreads) {
      const int tt = i / E, e = i - tt * E;
      float z = part[e * 8 + tt];
      for (int ks = 1; ks < ksplit; ++ks) z += part[((size_t)ks * n_mt * 16 + e) * 8 + tt];
      zs[tt * E + e] = z + (p.bias ? __ldg(p.bias + e) : 0.f);
    }
  }
  __syncthreads();
}

// Softmax over the E router logits z of token t and its top-k selection, one
// warp; lane l holds experts l, l + 32, ... (PER of them, E <= 32 * PER).
// Rank of expert e = number of experts ordered before it by (z desc, index
// asc); the experts of rank < k are the selection, in rank order.  Each
// selected expert's row is claimed with its counter (all claims of a lane
// issued together); shared experts take the token's own row.  Writes the
// token's k routed expert rows into rows[] and the row metadata of all k + S.
template <int PER>
__device__ __forceinline__ void select_experts(const RouteParams& p, const float* z, int t,
                                               int* rows) {
  const int lane = threadIdx.x & 31, E = p.E, k = p.k, S = p.S;
  float ze[PER];
  int rank[PER];
  float m = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    ze[j] = e < E ? z[e] : -FLT_MAX;
    m = fmaxf(m, ze[j]);
    rank[j] = 0;
  }
  m = warp_max(m);
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < PER; ++j)
    if (lane + 32 * j < E) sum += __expf(ze[j] - m);
  sum = warp_sum(sum);
#pragma unroll 4
  for (int f = 0; f < E; ++f) {
    const float zf = z[f];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int e = lane + 32 * j;
      rank[j] += (zf > ze[j] || (zf == ze[j] && f < e)) ? 1 : 0;
    }
  }
  int slot[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j)
    slot[j] = (lane + 32 * j < E && rank[j] < k) ? atomicAdd(p.cnt + lane + 32 * j, 1) : 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    if (e < E && rank[j] < k) {
      const float w = __expf(ze[j] - m) / sum;
      int sl = slot[j];
      if (sl >= p.T) {  // only reachable if the counters were not cleared
        atomicOr(p.status, kErrInternal);
        sl = p.T - 1;
      }
      const int row = e * p.T + sl;
      rows[rank[j]] = row;
      p.perm_token[row] = t;
      p.perm_slot[row] = rank[j];
      p.perm_w[row] = w;
      if (p.probe_idx) p.probe_idx[(size_t)t * k + rank[j]] = e;
      if (p.probe_w) p.probe_w[(size_t)t * k + rank[j]] = w;
    }
  }
  // shared experts: their rows are copied right after the RMSNorm
  for (int s = lane; s < S; s += 32) {
    const int row = (E + s) * p.T + t;
    p.perm_token[row] = t;
    p.perm_slot[row] = k + s;
    p.perm_w[row] = 1.0f;
  }
}

}  // namespace rs
}  // namespace mv
