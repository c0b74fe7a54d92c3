// Per-layer routing: residual update, RMSNorm, softmax router with top-k
// selection, and the placement of each token's normalised row in the rows of
// the experts it selected.
//
// Decoder block of "Jina AI Releases jina-ocr-v1, a 3.4B MoE Document Parser
// With Built-In Speculative Decoding", architecture paragraph: 64 routed
// experts, top-6 routing, two shared experts.  Top-k is taken on the router
// logits (ties: lower expert index); the weights are the softmax over all
// experts, not renormalised.
//
// Expert-major rows: expert e (shared experts are E .. E+S-1) owns rows
// [e*T, e*T + count_e) of the normalised-input and SwiGLU buffers.  A routed
// token claims its row in expert e with an atomic counter, so the order of
// tokens inside an expert varies from run to run; every token's result is
// independent of its row (each row is a separate column of the expert's GEMM,
// reduced in a fixed order), so the outputs do not.  Shared expert s holds
// token t in row (E+s)*T + t.
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

// Residual stream entering the block for chunk c (4 floats) of token t.
template <int SRC>
__device__ __forceinline__ float4 residual_chunk(const RouteParams& p, int t, int c,
                                                 const __nv_bfloat16* erow) {
  const int d = p.d, nc = d / 4;
  if (SRC == kSrcEmbed) return bf16x4_to_f4(__ldg(reinterpret_cast<const uint2*>(erow) + c));
  if (SRC == kSrcBf16)
    return bf16x4_to_f4(__ldg(reinterpret_cast<const uint2*>(p.h_in + (size_t)t * d) + c));
  const int kS = p.k + p.S;
  float4 v = reinterpret_cast<const float4*>(p.h + (size_t)t * d)[c];
  const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * kS * d) + c;
  // routed slots in selection order, then shared experts, summed first
  float4 acc = yr[0];
#pragma unroll 8
  for (int s = 1; s < kS; ++s) {
    const float4 u = yr[(size_t)s * nc];
    acc.x += u.x; acc.y += u.y; acc.z += u.z; acc.w += u.w;
  }
  v.x += acc.x; v.y += acc.y; v.z += acc.z; v.w += acc.w;
  return v;
}

// Stage 1 for the block's tokens t0 .. t0+ntok-1, all threads: build h (and
// write it back), RMSNorm; the normalised row goes to xs [TPB, d] (widened
// bf16 values, for the router) and xb [TPB, d] (bf16, for the expert rows).
template <int SRC, int TPB>
__device__ void block_norm(const RouteParams& p, int t0, int ntok, float* xs,
                           __nv_bfloat16* xb, float* red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, nc = d / 4;
  float ss[TPB];
#pragma unroll
  for (int i = 0; i < TPB; ++i) ss[i] = 0.f;
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt) {
    if (tt >= ntok) break;
    const int t = t0 + tt;
    const __nv_bfloat16* erow = nullptr;
    if (SRC == kSrcEmbed) {
      const int b = t / (p.K + 1), i = t % (p.K + 1);
      const int id = (i == 0) ? p.context_ids[b] : p.draft_ids[(size_t)b * p.K + (i - 1)];
      const bool ok = (id >= 0 && id < p.V);
      if (tid == 0) {
        p.bad[t] = ok ? 0 : 1;
        if (!ok) atomicOr(p.status, kErrIdRange);
      }
      erow = p.embed + (size_t)(ok ? id : 0) * d;
    }
    for (int c = tid; c < nc; c += kRouteThreads) {
      const float4 v = residual_chunk<SRC>(p, t, c, erow);
      reinterpret_cast<float4*>(p.h + (size_t)t * d)[c] = v;
      if (p.probe_hidden) reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d)[c] = v;
      reinterpret_cast<float4*>(xs + tt * d)[c] = v;
      ss[tt] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  }
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt) {
    if (tt >= ntok) break;
    const float w = warp_sum(ss[tt]);
    if (lane == 0) red[warp * 8 + tt] = w;
  }
  __syncthreads();
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt) {
    if (tt >= ntok) break;
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) tot += red[w * 8 + tt];
    const float r = rsqrtf(tot / (float)d + p.eps);
    for (int c = tid; c < nc; c += kRouteThreads) {
      float4 v = reinterpret_cast<const float4*>(xs + tt * d)[c];
      const float4 g = __ldg(reinterpret_cast<const float4*>(p.gain) + c);
      __nv_bfloat16 q0 = __float2bfloat16_rn(v.x * r * g.x);
      __nv_bfloat16 q1 = __float2bfloat16_rn(v.y * r * g.y);
      __nv_bfloat16 q2 = __float2bfloat16_rn(v.z * r * g.z);
      __nv_bfloat16 q3 = __float2bfloat16_rn(v.w * r * g.w);
      __nv_bfloat162 lo = __halves2bfloat162(q0, q1), hi = __halves2bfloat162(q2, q3);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo);
      packed.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(xb + tt * d)[c] = packed;
      v = make_float4(__bfloat162float(q0), __bfloat162float(q1), __bfloat162float(q2),
                      __bfloat162float(q3));
      reinterpret_cast<float4*>(xs + tt * d)[c] = v;
    }
  }
}

template <int SRC, int TPB>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  extern __shared__ __align__(128) float rsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, E = p.E, k = p.k, S = p.S;
  const int t0 = blockIdx.x * TPB;
  const int ntok = min(TPB, p.T - t0);
  // shared memory: [router weights E x d bf16, when staged] [xs TPB x d fp32]
  // [xb TPB x d bf16] [zs TPB x E] [red 64] [rows TPB x (k+S) ints]
  const size_t wr_bytes = p.wr_smem ? (size_t)E * d * 2 : 0;
  __nv_bfloat16* wr_s = reinterpret_cast<__nv_bfloat16*>(rsm);
  float* xs = reinterpret_cast<float*>(reinterpret_cast<char*>(rsm) + wr_bytes);
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(xs + TPB * d);
  float* zs = reinterpret_cast<float*>(xb + TPB * d);
  float* red = zs + TPB * E;
  int* rows = reinterpret_cast<int*>(red + 64);
  __shared__ __align__(8) uint64_t wr_bar;
  __shared__ int abort_flag;

  // The router weights do not depend on earlier kernels: start their copy
  // into shared memory before waiting for the previous kernel.
  if (p.wr_smem && tid == 0) {
    abort_flag = 0;
    mbar_init(&wr_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&wr_bar, (uint32_t)wr_bytes);
    const char* src = reinterpret_cast<const char*>(p.Wr);
    char* dst = reinterpret_cast<char*>(wr_s);
    for (size_t off = 0; off < wr_bytes; off += 16384) {
      const uint32_t n = (uint32_t)min((size_t)16384, wr_bytes - off);
      bulk_load(dst + off, src + off, n, &wr_bar);
    }
  }
  // Wait for the previous kernel, then let dependents start: a kernel two
  // launches later may then read what the kernel before this one wrote.
  pdl_wait();
  pdl_launch_dependents();
  block_norm<SRC, TPB>(p, t0, ntok, xs, xb, red);
  __syncthreads();
  bool wr_ok = true;
  if (p.wr_smem) wr_ok = mbar_wait(&wr_bar, 0, &abort_flag, p.status);
  for (int i = tid; i < TPB * (k + S); i += kRouteThreads) rows[i] = -1;

  // router logits: warp w computes experts 8w .. 8w+7 (then + 64, ...) for
  // every token of the block, eight independent accumulation chains per lane
  const __nv_bfloat16* wsrc = p.wr_smem ? wr_s : p.Wr;
  for (int e0 = warp * 8; e0 < E && wr_ok; e0 += kRouteWarps * 8) {
    float acc[8][TPB];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int tt = 0; tt < TPB; ++tt) acc[j][tt] = 0.f;
    for (int c = lane; c < d / 8; c += 32) {
      float4 xa[TPB], xv[TPB];
#pragma unroll
      for (int tt = 0; tt < TPB; ++tt) {
        const float4* x4 = reinterpret_cast<const float4*>(xs + tt * d + c * 8);
        xa[tt] = x4[0];
        xv[tt] = x4[1];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = min(e0 + j, E - 1);
        const uint4* wrow = reinterpret_cast<const uint4*>(wsrc + (size_t)e * d);
        float w8[8];
        unpack8(p.wr_smem ? wrow[c] : __ldg(wrow + c), w8);
#pragma unroll
        for (int tt = 0; tt < TPB; ++tt) {
          float a = acc[j][tt];
          a = fmaf(w8[0], xa[tt].x, a);
          a = fmaf(w8[1], xa[tt].y, a);
          a = fmaf(w8[2], xa[tt].z, a);
          a = fmaf(w8[3], xa[tt].w, a);
          a = fmaf(w8[4], xv[tt].x, a);
          a = fmaf(w8[5], xv[tt].y, a);
          a = fmaf(w8[6], xv[tt].z, a);
          a = fmaf(w8[7], xv[tt].w, a);
          acc[j][tt] = a;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + j;
#pragma unroll
      for (int tt = 0; tt < TPB; ++tt) {
        const float z = warp_sum(acc[j][tt]);
        if (lane == 0 && e < E) zs[tt * E + e] = z + (p.bias ? __ldg(p.bias + e) : 0.f);
      }
    }
  }
  __syncthreads();

  // softmax and top-k, one warp per token.  Rank of expert e = number of
  // experts ordered before it by (z desc, index asc); the experts of rank < k
  // are the selection, in rank order.  Each selected expert's row is claimed
  // with its counter; shared experts take the token's own row.
  if (warp < ntok && wr_ok) {
    const int tt = warp, t = t0 + tt;
    const float* z = zs + tt * E;
    float m = -FLT_MAX;
    for (int e = lane; e < E; e += 32) m = fmaxf(m, z[e]);
    m = warp_max(m);
    float sum = 0.f;
    for (int e = lane; e < E; e += 32) sum += __expf(z[e] - m);
    sum = warp_sum(sum);
    for (int e = lane; e < E; e += 32) {
      const float ze = z[e];
      int rank = 0;
      for (int f = 0; f < E; ++f) {
        const float zf = z[f];
        rank += (zf > ze || (zf == ze && f < e)) ? 1 : 0;
      }
      if (rank < k) {
        const float w = __expf(ze - m) / sum;
        int slot = atomicAdd(p.cnt + e, 1);
        if (slot >= p.T) {  // only reachable if the counters were not cleared
          atomicOr(p.status, kErrInternal);
          slot = p.T - 1;
        }
        const int row = e * p.T + slot;
        rows[tt * (k + S) + rank] = row;
        p.perm_token[row] = t;
        p.perm_slot[row] = rank;
        p.perm_w[row] = w;
        if (p.probe_idx) p.probe_idx[(size_t)t * k + rank] = e;
        if (p.probe_w) p.probe_w[(size_t)t * k + rank] = w;
      }
    }
    for (int s = lane; s < S; s += 32) {
      const int row = (E + s) * p.T + t;
      rows[tt * (k + S) + k + s] = row;
      p.perm_token[row] = t;
      p.perm_slot[row] = k + s;
      p.perm_w[row] = 1.0f;
    }
  }
  __syncthreads();

  // copy each token's normalised row into its k + S expert rows
  if (wr_ok) {
    const int cpr = d / 8;  // 16-byte chunks per row
    const int nslots = ntok * (k + S);
    for (int i = tid; i < nslots * cpr; i += kRouteThreads) {
      const int q = i / cpr, c = i - q * cpr;
      const int tt = q / (k + S);
      const int row = rows[q];
      if (row >= 0)
        reinterpret_cast<uint4*>(p.xperm + (size_t)row * d)[c] =
            reinterpret_cast<const uint4*>(xb + tt * d)[c];
    }
  }
}

// Residual update after the last block, then either the final RMSNorm (the
// lm_head input) or the bf16 output of the single-block entry point.  One
// token per block; the sum of squares is reduced per thread over its 4-float
// chunks (c = tid, tid + 256, ...), then per warp, then over the warps in
// order (the allocation-free greedy head reduces in the same order).
__global__ void __launch_bounds__(256) final_kernel(FinalParams p) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int d = p.d, nc = d / 4;
  float* hrow = p.h + (size_t)t * d;
  const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * p.kS * d);
  float ss = 0.f;
  for (int c = tid; c < nc; c += 256) {
    float4 v = reinterpret_cast<const float4*>(hrow)[c];
    float4 acc = yr[c];
#pragma unroll 8
    for (int s = 1; s < p.kS; ++s) {
      const float4 u = yr[(size_t)s * nc + c];
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
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)d + p.eps);
  for (int c = tid; c < nc; c += 256) {
    const float4 v = reinterpret_cast<const float4*>(hrow)[c];
    const float4 g = __ldg(reinterpret_cast<const float4*>(p.gain) + c);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out + (size_t)t * d)[c] = packed;
  }
  if (tid == 0) p.keys[t] = 0ull;
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

template <int SRC, int TPB>
cudaError_t launch_route_t(const RouteParams& p, int grid, size_t smem, cudaStream_t s, bool pdl) {
  auto k = route_kernel<SRC, TPB>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_ex(k, dim3(grid), dim3(kRouteThreads), smem, s, pdl, p);
}

template <int SRC>
cudaError_t launch_route_src(const RouteParams& p, int grid, size_t smem, cudaStream_t s,
                             bool pdl) {
  switch (p.tpb) {
    case 1: return launch_route_t<SRC, 1>(p, grid, smem, s, pdl);
    case 2: return launch_route_t<SRC, 2>(p, grid, smem, s, pdl);
    case 4: return launch_route_t<SRC, 4>(p, grid, smem, s, pdl);
    default: return launch_route_t<SRC, 8>(p, grid, smem, s, pdl);
  }
}

}  // namespace

size_t route_smem_bytes(int tpb, int d, int E, int k, int S, bool wr_smem) {
  return (wr_smem ? (size_t)E * d * 2 : 0) + (size_t)tpb * d * (4 + 2) +
         ((size_t)tpb * E + 64) * sizeof(float) + (size_t)tpb * (k + S) * sizeof(int);
}

bool route_wr_fits(int tpb, int d, int E, int k, int S) {
  return route_smem_bytes(tpb, d, E, k, S, true) <= 220 * 1024;
}

cudaError_t launch_route(const RouteParams& p, int grid, size_t smem, cudaStream_t s, bool pdl) {
  switch (p.src) {
    case kSrcEmbed: return launch_route_src<kSrcEmbed>(p, grid, smem, s, pdl);
    case kSrcBf16: return launch_route_src<kSrcBf16>(p, grid, smem, s, pdl);
    default: return launch_route_src<kSrcCombine>(p, grid, smem, s, pdl);
  }
}

cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl) {
  return launch_ex(final_kernel, dim3(p.T), dim3(256), 0, s, pdl, p);
}

}  // namespace mv
