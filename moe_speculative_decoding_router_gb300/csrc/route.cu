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
//
// One block per token (up to eight at large T).  Static data and the
// residual rows are staged before the block waits for the previous kernel;
// the router logits run on the tensor cores (mma.sync m16n8k16, the block's
// tokens as the N columns).
#include <float.h>

#include "internal.h"
#include "ptx.cuh"
#include "route_stages.cuh"

namespace mv {

using rs::bf16x4_to_f4;
using rs::norm_pack;
using rs::norm_scale;
using rs::route_ksplit;
using rs::route_wr_panel;
using rs::sum_slots;
using rs::sumsq4;
using rs::warp_sum;

namespace {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;

// Bulk copy of `bytes` (16-byte aligned, multiple of 16) into shared memory,
// completing on `bar`, in pieces of at most 16 KB.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, size_t bytes, uint64_t* bar) {
  for (size_t off = 0; off < bytes; off += 16384) {
    const uint32_t n = (uint32_t)min((size_t)16384, bytes - off);
    bulk_load(static_cast<char*>(dst) + off, static_cast<const char*>(src) + off, n, bar);
  }
}

// Stage 1 for the block's tokens t0 .. t0+ntok-1 (TPB > 1; rows of at most
// 2,048, so that each thread holds at most one chunk of a row and the sum of
// squares is reduced in the order of the one-token path: per warp over its 32
// chunks, then over the warps in order), all threads: build the residual
// stream h entering the block (and write it back), RMSNorm, and the
// normalised bf16 row xb [TPB, d] (row pitch xpitch elements).  For the
// combine source xs [TPB, d] already holds the tokens' h rows and gs [d] the
// gain (bulk copies issued before the wait); the expert outputs of the
// previous block are summed in slot order (routed slots in selection order,
// then the shared experts) and added to h.
template <int SRC, int TPB>
__device__ void block_norm(const RouteParams& p, int t0, int ntok, float* xs, const float* gs,
                           __nv_bfloat16* xb, int xpitch, float* red) {
  constexpr int kPass = 2;  // float4 chunks per thread whose loads are issued together
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, nc = d / 4, kS = p.k + p.S;
  float ss[TPB];
#pragma unroll
  for (int i = 0; i < TPB; ++i) ss[i] = 0.f;
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt) {
    if (tt >= ntok) break;
    const int t = t0 + tt;
    float4* hx = reinterpret_cast<float4*>(xs + tt * d);
    float4* hg = reinterpret_cast<float4*>(p.h + (size_t)t * d);
    float4* hp = p.probe_hidden ? reinterpret_cast<float4*>(p.probe_hidden + (size_t)t * d) : nullptr;
    if (SRC == kSrcCombine) {
      const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * kS * d);
      const float4* yrs[kPass];
#pragma unroll
      for (int j = 0; j < kPass; ++j) yrs[j] = yr;
      for (int c0 = tid; c0 < nc; c0 += kPass * kRouteThreads) {
        float4 acc[kPass];
        int cj[kPass];
#pragma unroll
        for (int j = 0; j < kPass; ++j) cj[j] = c0 + j * kRouteThreads;
        sum_slots<kPass>(yrs, nc, kS, cj, acc);
#pragma unroll
        for (int j = 0; j < kPass; ++j) {
          const int c = c0 + j * kRouteThreads;
          if (c < nc) {
            float4 v = hx[c];
            v.x += acc[j].x; v.y += acc[j].y; v.z += acc[j].z; v.w += acc[j].w;
            hx[c] = v;
            hg[c] = v;
            if (hp) hp[c] = v;
            ss[tt] += sumsq4(v);
          }
        }
      }
    } else if (SRC == kSrcH) {
      // h as the previous launch (the attention's output projection) left it
      for (int c = tid; c < nc; c += kRouteThreads) {
        const float4 v = __ldcg(hg + c);
        hx[c] = v;
        if (hp) hp[c] = v;
        ss[tt] += sumsq4(v);
      }
    } else {
      const uint2* src;
      if (SRC == kSrcEmbed || SRC == kSrcEmbedAdd) {
        const int b = t / (p.K + 1), i = t % (p.K + 1);
        const int id = (i == 0) ? p.context_ids[b] : p.draft_ids[(size_t)b * p.K + (i - 1)];
        const bool ok = (id >= 0 && id < p.V);
        if (tid == 0) {
          p.bad[t] = ok ? 0 : 1;
          if (!ok) atomicOr(p.status, kErrIdRange);
        }
        src = reinterpret_cast<const uint2*>(p.embed + (size_t)(ok ? id : 0) * d);
      } else {
        src = reinterpret_cast<const uint2*>(p.h_in + (size_t)t * d);
      }
      for (int c = tid; c < nc; c += kRouteThreads) {
        float4 v = bf16x4_to_f4(__ldg(src + c));
        if (SRC == kSrcEmbedAdd) {
          // the running state, written by the previous launch: read after the wait
          const float4 hv = __ldcg(hg + c);
          v = make_float4(hv.x + v.x, hv.y + v.y, hv.z + v.z, hv.w + v.w);
        }
        hx[c] = v;
        hg[c] = v;
        if (hp) hp[c] = v;
        ss[tt] += sumsq4(v);
      }
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
    const float r = norm_scale(tot, d, p.eps);
    for (int c = tid; c < nc; c += kRouteThreads) {
      const float4 v = reinterpret_cast<const float4*>(xs + tt * d)[c];
      const float4 g = reinterpret_cast<const float4*>(gs)[c];
      reinterpret_cast<uint2*>(xb + tt * xpitch)[c] = norm_pack(v, r, g);
    }
  }
}

// WR: the router weights are staged in shared memory by TMA (else read
// through L1).
template <int SRC, int TPB, bool WR>
__global__ void __launch_bounds__(kRouteThreads, 1)
    route_kernel(const __grid_constant__ CUtensorMap map_wr, RouteParams p) {
  extern __shared__ __align__(1024) uint8_t rsm_raw[];
  uint8_t* rsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) &
                                            ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, E = p.E, k = p.k, S = p.S;
  const int t0 = blockIdx.x * TPB;
  const int ntok = min(TPB, p.T - t0);
  const int n_mt = (E + 15) / 16, ksplit = route_ksplit(E);
  // normalised bf16 rows are padded by 16 bytes so that the B-fragment loads
  // of the 8 token rows fall in distinct shared-memory banks
  const int pitch = d + 8;
  // shared memory: [router weights, when staged] [gain d fp32] [xs TPB x d
  // fp32, several tokens per block only] [xb TPB x pitch bf16] [partial
  // logits ksplit x 16n_mt x 8] [zs TPB x E] [red 128] [rows TPB x (k+S)]
  const size_t panel = route_wr_panel(E);
  const size_t wr_bytes = WR ? (size_t)(d / 64) * panel : 0;
  uint8_t* wr_s = rsm;
  float* gs = reinterpret_cast<float*>(rsm + wr_bytes);
  float* xs = gs + d;
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(xs + (TPB > 1 ? TPB * d : 0));
  float* part = reinterpret_cast<float*>(xb + TPB * pitch);
  float* zs = part + ksplit * n_mt * 16 * 8;
  float* red = zs + TPB * E;
  int* rows = reinterpret_cast<int*>(red + kRouteWarps * 8);
  __shared__ __align__(8) uint64_t hx_bar, wr_bar;
  __shared__ int abort_flag;

  // Before waiting for the previous kernel: the gain and the router weights
  // (static), and for the combine source with several tokens per block the
  // tokens' h rows, which the routing kernel two launches back wrote (a
  // kernel lets its dependents start only after its own wait, so that kernel
  // is complete here).
  if (tid == 0) {
    if (p.stamps) stamp_min(p.stamps);
    abort_flag = 0;
    mbar_init(&hx_bar, 1);
    mbar_init(&wr_bar, 1);
    fence_mbar_init();
    const size_t h_bytes = (SRC == kSrcCombine && TPB > 1) ? (size_t)ntok * d * 4 : 0;
    mbar_arrive_expect_tx(&hx_bar, (uint32_t)((size_t)d * 4 + h_bytes));
    bulk_copy(gs, p.gain, (size_t)d * 4, &hx_bar);
    if (h_bytes) bulk_copy(xs, p.h + (size_t)t0 * d, h_bytes, &hx_bar);
    if (WR) {
      const uint64_t pol = policy_evict_last();
      mbar_arrive_expect_tx(&wr_bar, (uint32_t)((size_t)E * d * 2));
      for (int pn = 0; pn < d / 64; ++pn)
        tma_load_2d(wr_s + (size_t)pn * panel, &map_wr, &wr_bar, pn * 64, p.wr_row, pol);
    }
  }
  for (int i = tid; i < TPB * (k + S); i += kRouteThreads) rows[i] = -1;
  __syncthreads();
  // Wait for the previous kernel, then let dependents start: a kernel two
  // launches later may then read what the kernel before this one wrote.
  pdl_wait();
  pdl_launch_dependents();
  if (p.stamps && tid == 0) stamp_max(p.stamps + 1);
  if (blockIdx.x == 0) {
    // counters of kernels that are complete now (the expert FFN before this
    // kernel, the routing kernel before that); the expert FFN after this
    // kernel reads them only after its own wait
    for (int i = tid; i < p.n_dep_clear; i += kRouteThreads) p.dep_clear[i] = 0;
    for (int e = tid; e < E; e += kRouteThreads) p.cnt_other[e] = 0;
    if (tid == 0) *p.next_item_clear = 0;
  }
  mbar_wait(&hx_bar, 0, &abort_flag, p.status);
  __syncthreads();
  bool ok = !abort_flag;  // the same for every thread (the norm has barriers)
  if (ok) {
    if constexpr (TPB == 1)
      rs::norm_token<SRC, kRouteWarps>(p, t0, gs, xb, red);
    else
      block_norm<SRC, TPB>(p, t0, ntok, xs, gs, xb, pitch, red);
  }
  __syncthreads();
  const int cpr = d / 8;  // 16-byte chunks per row
  if (ok) {
    // shared experts hold token t in row (E+s)*T + t: copy those rows now,
    // while the router runs
    for (int i = tid; i < ntok * S * cpr; i += kRouteThreads) {
      const int q = i / cpr, c = i - q * cpr;
      const int tt = q / S, sx = q - tt * S;
      reinterpret_cast<uint4*>(p.xperm + ((size_t)(E + sx) * p.T + t0 + tt) * d)[c] =
          reinterpret_cast<const uint4*>(xb + tt * pitch)[c];
    }
  }
  if (WR && ok) ok = mbar_wait(&wr_bar, 0, &abort_flag, p.status);

  // router logits of the block's tokens (tensor cores), then softmax and
  // top-k, one warp per token
  rs::router_logits<TPB, WR>(p, wr_s, xb, pitch, part, zs, ntok, kRouteWarps, ok);
  if (warp < ntok && ok) {
    if (E <= 64)
      rs::select_experts<2>(p, zs + warp * E, t0 + warp, rows + warp * (k + S));
    else
      rs::select_experts<8>(p, zs + warp * E, t0 + warp, rows + warp * (k + S));
  }
  __syncthreads();

  // copy each token's normalised row into its k routed expert rows
  if (ok) {
    const int nslots = ntok * (k + S);
    for (int i = tid; i < nslots * cpr; i += kRouteThreads) {
      const int q = i / cpr, c = i - q * cpr;
      const int tt = q / (k + S);
      const int row = rows[q];
      if (row >= 0)
        reinterpret_cast<uint4*>(p.xperm + (size_t)row * d)[c] =
            reinterpret_cast<const uint4*>(xb + tt * pitch)[c];
    }
  }
  if (p.stamps) {
    __syncthreads();
    if (tid == 0) stamp_max(p.stamps + 2);
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
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < p.n_cnt_clear; e += 256) p.cnt_clear[e] = 0;
    if (threadIdx.x == 0) {
      *p.item_clear = 0;
      if (p.route_done_clear) *p.route_done_clear = 0;
    }
    for (int i = threadIdx.x; i < p.n_layer_items; i += 256) p.layer_items_clear[i] = 0;
  }
  __shared__ float red[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int d = p.d, nc = d / 4;
  float* hrow = p.h + (size_t)t * d;
  const float4* yr = reinterpret_cast<const float4*>(p.y + (size_t)t * p.kS * d);
  float ss = 0.f;
  for (int c = tid; c < nc; c += 256) {
    float4 v = reinterpret_cast<const float4*>(hrow)[c];
    float4 acc[1];
    const int cj[1] = {c};
    const float4* yrs[1] = {yr};
    sum_slots<1>(yrs, nc, p.kS, cj, acc);
    v.x += acc[0].x; v.y += acc[0].y; v.z += acc[0].z; v.w += acc[0].w;
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
cudaError_t launch_route_t(const CUtensorMap& map_wr, const RouteParams& p, int grid, size_t smem,
                           cudaStream_t s, bool pdl) {
  auto k = p.wr_smem ? route_kernel<SRC, TPB, true> : route_kernel<SRC, TPB, false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_ex(k, dim3(grid), dim3(kRouteThreads), smem, s, pdl, map_wr, p);
}

template <int SRC>
cudaError_t launch_route_src(const CUtensorMap& map_wr, const RouteParams& p, int grid,
                             size_t smem, cudaStream_t s, bool pdl) {
  switch (p.tpb) {
    case 1: return launch_route_t<SRC, 1>(map_wr, p, grid, smem, s, pdl);
    case 2: return launch_route_t<SRC, 2>(map_wr, p, grid, smem, s, pdl);
    case 4: return launch_route_t<SRC, 4>(map_wr, p, grid, smem, s, pdl);
    default: return launch_route_t<SRC, 8>(map_wr, p, grid, smem, s, pdl);
  }
}

}  // namespace

size_t route_smem_bytes(int tpb, int d, int E, int k, int S, bool wr_smem) {
  const size_t pitch = (size_t)d + 8;
  const size_t part = (size_t)route_ksplit(E) * ((E + 15) / 16) * 16 * 8;
  return 1024 /* alignment slack */ + (wr_smem ? (size_t)(d / 64) * route_wr_panel(E) : 0) +
         (size_t)d * 4 + (tpb > 1 ? (size_t)tpb * d * 4 : 0) +
         (size_t)tpb * pitch * 2 + (part + (size_t)tpb * E + kRouteWarps * 8) * sizeof(float) +
         (size_t)tpb * (k + S) * sizeof(int);
}

bool route_wr_fits(int tpb, int d, int E, int k, int S) {
  return route_smem_bytes(tpb, d, E, k, S, true) <= 220 * 1024;
}

cudaError_t launch_route(const CUtensorMap& map_wr, const RouteParams& p, int grid, size_t smem,
                         cudaStream_t s, bool pdl) {
  switch (p.src) {
    case kSrcEmbed: return launch_route_src<kSrcEmbed>(map_wr, p, grid, smem, s, pdl);
    case kSrcBf16: return launch_route_src<kSrcBf16>(map_wr, p, grid, smem, s, pdl);
    case kSrcEmbedAdd: return launch_route_src<kSrcEmbedAdd>(map_wr, p, grid, smem, s, pdl);
    case kSrcH: return launch_route_src<kSrcH>(map_wr, p, grid, smem, s, pdl);
    default: return launch_route_src<kSrcCombine>(map_wr, p, grid, smem, s, pdl);
  }
}

cudaError_t launch_final(const FinalParams& p, cudaStream_t s, bool pdl) {
  return launch_ex(final_kernel, dim3(p.T), dim3(256), 0, s, pdl, p);
}

}  // namespace mv
