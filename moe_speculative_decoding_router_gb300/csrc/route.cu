// Per-layer routing: residual update, RMSNorm, softmax router with top-k
// selection, and the grouping of (token, slot) pairs by expert.
//
// Decoder block of "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser
// With Built-In Speculative Decoding", architecture paragraph: 64 routed
// experts, top-6 routing, two shared experts.  Top-k is taken on the router
// logits (ties: lower expert index); the weights are the softmax over all
// experts, not renormalised.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace mv {

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;

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

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 v = __bfloat1622float2(b[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 u) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
  float2 a = __bfloat1622float2(b[0]), c = __bfloat1622float2(b[1]);
  return make_float4(a.x, a.y, c.x, c.y);
}

// Stage 1 for one token (one warp): build h, normalise, write xhat.
template <int SRC>
__device__ void token_norm(const RouteParams& p, int t, float* xs) {
  const int lane = threadIdx.x & 31;
  const int d = p.d;
  const int nc = d / 4;
  float* hrow = p.h + (size_t)t * d;
  const __nv_bfloat16* erow = nullptr;
  if (SRC == kSrcEmbed) {
    const int b = t / (p.K + 1), i = t % (p.K + 1);
    int id = (i == 0) ? p.context_ids[b] : p.draft_ids[(size_t)b * p.K + (i - 1)];
    const bool ok = (id >= 0 && id < p.V);
    if (lane == 0) {
      p.bad[t] = ok ? 0 : 1;
      if (!ok) atomicOr(p.status, kErrIdRange);
    }
    erow = p.embed + (size_t)(ok ? id : 0) * d;
  }
  float ss = 0.f;
  for (int c = lane; c < nc; c += 32) {
    float4 v;
    if (SRC == kSrcEmbed) {
      v = bf16x4_to_f4(__ldg(reinterpret_cast<const uint2*>(erow) + c));
    } else if (SRC == kSrcBf16) {
      v = bf16x4_to_f4(__ldg(reinterpret_cast<const uint2*>(p.h_in + (size_t)t * d) + c));
    } else {
      v = reinterpret_cast<const float4*>(hrow)[c];
      const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * (p.k + p.S) * d);
      float4 acc = yr[c];
      for (int s = 1; s < p.k + p.S; ++s) {
        float4 u = yr[(size_t)s * nc + c];
        acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
      }
      v.x += acc.x; v.y += acc.y; v.z += acc.z; v.w += acc.w;
    }
    reinterpret_cast<float4*>(hrow)[c] = v;
    if (p.probe_hidden) reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d)[c] = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)d + p.eps);
  for (int c = lane; c < nc; c += 32) {
    float4 v = reinterpret_cast<const float4*>(hrow)[c];
    float4 g = __ldg(reinterpret_cast<const float4*>(p.gain) + c);
    __nv_bfloat16 q0 = __float2bfloat16_rn(v.x * r * g.x);
    __nv_bfloat16 q1 = __float2bfloat16_rn(v.y * r * g.y);
    __nv_bfloat16 q2 = __float2bfloat16_rn(v.z * r * g.z);
    __nv_bfloat16 q3 = __float2bfloat16_rn(v.w * r * g.w);
    __nv_bfloat162 lo = __halves2bfloat162(q0, q1), hi = __halves2bfloat162(q2, q3);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.xhat + (size_t)t * d)[c] = packed;
    float4 f = make_float4(__bfloat162float(q0), __bfloat162float(q1), __bfloat162float(q2),
                           __bfloat162float(q3));
    reinterpret_cast<float4*>(xs)[c] = f;
  }
}

// Grouping by expert, run by the last block of the grid.  Expert-major rows:
// routed expert e owns rows [off[e], off[e+1]) with its tokens in increasing
// token order; shared expert s owns rows off[E+s] + t for every token t.
__device__ void group_by_expert(const RouteParams& p, int* sm) {
  const int T = p.T, k = p.k, E = p.E, S = p.S, nE = E + S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* idx_s = sm;              // [T*k]
  int* cnt_s = idx_s + T * k;   // [nE]
  int* off_s = cnt_s + nE;      // [nE+1]
  int* igu_s = off_s + nE + 1;  // [nE+1] item offsets, gate/up
  int* idn_s = igu_s + nE + 1;  // [nE+1] item offsets, down

  for (int i = tid; i < T * k; i += kRouteThreads) {
    const int e = __ldcg(p.topk_idx + i);
    idx_s[i] = (e >= 0 && e < E) ? e : 0;
  }
  for (int e = tid; e < nE; e += kRouteThreads) cnt_s[e] = (e < E) ? 0 : T;
  __syncthreads();
  for (int i = tid; i < T * k; i += kRouteThreads) atomicAdd(&cnt_s[idx_s[i]], 1);
  __syncthreads();
  if (tid == 0) {
    int o = 0, ig = 0, id = 0;
    for (int e = 0; e < nE; ++e) {
      off_s[e] = o;
      igu_s[e] = ig;
      idn_s[e] = id;
      const int c = cnt_s[e];
      const int nch = (e < E) ? p.nch_r : p.nch_s;
      const int chunks = (c + nch - 1) / nch;
      o += c;
      ig += chunks * p.mt_gu;
      id += chunks * p.mt_dn;
    }
    off_s[nE] = o;
    igu_s[nE] = ig;
    idn_s[nE] = id;
    p.n_items[0] = ig;
    p.n_items[1] = id;
  }
  __syncthreads();
  for (int e = tid; e <= nE; e += kRouteThreads) p.expert_off[e] = off_s[e];

  // stable positions of routed (token, slot) pairs
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int e = warp; e < E; e += kRouteWarps) {
    int running = off_s[e];
    for (int c0 = 0; c0 < T; c0 += 32) {
      const int t = c0 + lane;
      int jf = -1;
      if (t < T) {
        for (int j = 0; j < k; ++j)
          if (idx_s[t * k + j] == e) jf = j;
      }
      const unsigned ballot = __ballot_sync(0xffffffffu, jf >= 0);
      if (jf >= 0) {
        const int pos = running + __popc(ballot & lt_mask);
        p.perm_token[pos] = t;
        p.perm_slot[pos] = jf;
        p.perm_w[pos] = __ldcg(p.topk_w + (size_t)t * k + jf);
      }
      running += __popc(ballot);
    }
  }
  for (int i = tid; i < S * T; i += kRouteThreads) {
    const int s = i / T, t = i % T;
    const int pos = off_s[E + s] + t;
    p.perm_token[pos] = t;
    p.perm_slot[pos] = k + s;
    p.perm_w[pos] = 1.0f;
  }
  // work items, expert-major; the tiles of one expert sit next to each other
  for (int e = tid; e < nE; e += kRouteThreads) {
    const int c = cnt_s[e];
    const int nch = (e < E) ? p.nch_r : p.nch_s;
    const int chunks = (c + nch - 1) / nch;
    for (int ch = 0; ch < chunks; ++ch) {
      const int n = min(nch, c - ch * nch);
      const int brow = off_s[e] + ch * nch;
      for (int mt = 0; mt < p.mt_gu; ++mt) {
        Item it;
        it.a_row = p.a_base_gu + (e * p.mt_gu + mt) * 128;
        it.b_row = brow;
        it.n = n;
        it.aux = mt;
        p.items_gu[igu_s[e] + ch * p.mt_gu + mt] = it;
      }
      for (int mt = 0; mt < p.mt_dn; ++mt) {
        Item it;
        it.a_row = p.a_base_dn + (e * p.mt_dn + mt) * 128;
        it.b_row = brow;
        it.n = n;
        it.aux = mt;
        p.items_dn[idn_s[e] + ch * p.mt_dn + mt] = it;
      }
    }
  }
}

template <int SRC>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  extern __shared__ __align__(16) float rsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d, E = p.E, tpb = p.tpb;
  const int t0 = blockIdx.x * tpb;
  float* xs = rsm;              // [tpb, d]  normalised input, bf16 values widened
  float* zs = rsm + tpb * d;    // [tpb, E]  router logits

  pdl_wait();
  if (warp < tpb && t0 + warp < p.T) token_norm<SRC>(p, t0 + warp, xs + warp * d);
  __syncthreads();

  // router logits: warp w computes experts w, w+8, ... for every token of the block
  for (int e = warp; e < E; e += kRouteWarps) {
    const uint4* wrow = reinterpret_cast<const uint4*>(p.Wr + (size_t)e * d);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int c = lane; c < d / 8; c += 32) {
      float w8[8];
      unpack8(__ldg(wrow + c), w8);
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        if (tt < tpb) {
          const float4* x4 = reinterpret_cast<const float4*>(xs + tt * d + c * 8);
          const float4 xa = x4[0], xb = x4[1];
          float a = acc[tt];
          a = fmaf(w8[0], xa.x, a);
          a = fmaf(w8[1], xa.y, a);
          a = fmaf(w8[2], xa.z, a);
          a = fmaf(w8[3], xa.w, a);
          a = fmaf(w8[4], xb.x, a);
          a = fmaf(w8[5], xb.y, a);
          a = fmaf(w8[6], xb.z, a);
          a = fmaf(w8[7], xb.w, a);
          acc[tt] = a;
        }
      }
    }
    const float b = p.bias ? __ldg(p.bias + e) : 0.f;
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
      if (tt < tpb) {
        const float z = warp_sum(acc[tt]);
        if (lane == 0) zs[tt * E + e] = z + b;
      }
    }
  }
  __syncthreads();

  // softmax and top-k: one warp per token, lane holds experts lane + 32 j
  if (warp < tpb && t0 + warp < p.T) {
    const int t = t0 + warp;
    const float* z = zs + warp * E;
    float zl[8];
    float m = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      zl[j] = (e < E) ? z[e] : -FLT_MAX;
      m = fmaxf(m, zl[j]);
    }
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (lane + 32 * j < E) s += __expf(zl[j] - m);
    s = warp_sum(s);
    unsigned taken = 0;
    for (int r = 0; r < p.k; ++r) {
      float bv = -FLT_MAX;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && (zl[j] > bv || (zl[j] == bv && e < be))) {
          bv = zl[j];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (be < 0 || be >= E) {  // only reachable with non-finite logits
        if (lane == 0) atomicOr(p.status, kErrInternal);
        be = r;
        bv = zl[0];
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == 0) {
        const float w = __expf(bv - m) / s;
        p.topk_idx[(size_t)t * p.k + r] = be;
        p.topk_w[(size_t)t * p.k + r] = w;
        if (p.probe_idx) p.probe_idx[(size_t)t * p.k + r] = be;
        if (p.probe_w) p.probe_w[(size_t)t * p.k + r] = w;
      }
    }
  }

  // the last block to finish groups the whole batch by expert
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = (atomicAdd(p.done, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  group_by_expert(p, reinterpret_cast<int*>(rsm));
  if (threadIdx.x == 0) *p.done = 0u;
}

__global__ void __launch_bounds__(256) scatter_kernel(const int32_t* __restrict__ perm_token,
                                                      const __nv_bfloat16* __restrict__ xhat,
                                                      __nv_bfloat16* __restrict__ xperm, int rows,
                                                      int d) {
  pdl_wait();
  const int cpr = d / 8;  // 16-byte chunks per row
  const int64_t total = (int64_t)rows * cpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / cpr), c = (int)(i % cpr);
    const int t = __ldg(perm_token + r);
    reinterpret_cast<uint4*>(xperm + (size_t)r * d)[c] =
        __ldg(reinterpret_cast<const uint4*>(xhat + (size_t)t * d) + c);
  }
}

// Residual update after the last block, then either the final RMSNorm (the
// lm_head input) or the bf16 output of the single-block entry point.
__global__ void __launch_bounds__(256) final_kernel(FinalParams p) {
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= p.T) return;
  const int d = p.d, nc = d / 4;
  float* hrow = p.h + (size_t)t * d;
  const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * p.kS * d);
  float ss = 0.f;
  for (int c = lane; c < nc; c += 32) {
    float4 v = reinterpret_cast<const float4*>(hrow)[c];
    float4 acc = yr[c];
    for (int s = 1; s < p.kS; ++s) {
      float4 u = yr[(size_t)s * nc + c];
      acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
    }
    v.x += acc.x; v.y += acc.y; v.z += acc.z; v.w += acc.w;
    reinterpret_cast<float4*>(hrow)[c] = v;
    if (p.probe_hidden) reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d)[c] = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    if (p.mode == 1) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(p.out + (size_t)t * d)[c] = packed;
    }
  }
  if (p.mode == 1) return;
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)d + p.eps);
  for (int c = lane; c < nc; c += 32) {
    float4 v = reinterpret_cast<const float4*>(hrow)[c];
    float4 g = __ldg(reinterpret_cast<const float4*>(p.gain) + c);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out + (size_t)t * d)[c] = packed;
  }
  if (lane == 0) p.keys[t] = 0ull;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
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

}  // namespace

size_t route_smem_bytes(int tpb, int d, int E, int T, int k) {
  const size_t a = (size_t)tpb * (d + E) * sizeof(float);
  const size_t b = ((size_t)T * k + 4 * 300) * sizeof(int);
  return a > b ? a : b;
}

cudaError_t launch_route(const RouteParams& p, int grid, size_t smem, cudaStream_t s, bool pdl) {
  switch (p.src) {
    case kSrcEmbed: {
      auto k = route_kernel<kSrcEmbed>;
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(k, dim3(grid), dim3(kRouteThreads), smem, s, pdl, p);
    }
    case kSrcBf16: {
      auto k = route_kernel<kSrcBf16>;
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(k, dim3(grid), dim3(kRouteThreads), smem, s, pdl, p);
    }
    default: {
      auto k = route_kernel<kSrcCombine>;
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(k, dim3(grid), dim3(kRouteThreads), smem, s, pdl, p);
    }
  }
}

cudaError_t launch_scatter(const int32_t* perm_token, const __nv_bfloat16* xhat,
                           __nv_bfloat16* xperm, int rows, int d, cudaStream_t s, bool pdl) {
  const int64_t total = (int64_t)rows * (d / 8);
  int grid = (int)((total + 255) / 256);
  if (grid > 4096) grid = 4096;
  if (grid < 1) grid = 1;
  return launch_ex(scatter_kernel, dim3(grid), dim3(256), 0, s, pdl, perm_token, xhat, xperm, rows,
                   d);
}

cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl) {
  const int grid = (p.T + 7) / 8;
  return launch_ex(final_kernel, dim3(grid), dim3(256), 0, s, pdl, p);
}

}  // namespace mv
