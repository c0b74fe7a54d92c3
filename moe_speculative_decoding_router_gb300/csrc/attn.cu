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
constexpr int kAttnThreads = 128;
constexpr int kSPitch = kAttnMaxSplit + 1;  // score row pitch (floats): no bank conflicts

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
// the total keys x heads over the wanted items, rounded up to 64 and kept in
// [64, 1024]; a sequence's pairs are consecutive, in split order.
__device__ void build_plan(const AttnNormParams& p) {
  __shared__ long long s_tot[kNormThreads / 32];
  __shared__ int s_scan[kNormThreads / 32];
  __shared__ int s_width;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long tot = 0;
  for (int b = tid; b < p.B; b += kNormThreads) {
    const int p0 = p.positions[b];
    if (seq_in_range(p0, p.K, p.max_pos)) tot += p0 + p.K + 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane == 0) s_tot[warp] = tot;
  __syncthreads();
  if (tid == 0) {
    long long all = 0;
    for (int w = 0; w < kNormThreads / 32; ++w) all += s_tot[w];
    const long long want = (all * p.H + p.target_items - 1) / p.target_items;
    long long c = (want + kAttnMinSplit - 1) / kAttnMinSplit * kAttnMinSplit;
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
  pdl_wait();
  pdl_launch_dependents();
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
}

// One (sequence, split, head) item per iteration, 4 warps.  A key is read by
// LPK = hd / 8 lanes (16 bytes each), so a warp covers 32 / LPK keys per load;
// NQ >= K + 1 queries (the step's tokens of the sequence) are held in
// registers.  Shared memory: scores [NQ][kSPitch], per-warp partial outputs
// [4][NQ][hd], per-query (max, sum) [NQ][2].
template <int NQ>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnParams p) {
  extern __shared__ float asmem[];
  float* S = asmem;
  float* red = S + NQ * kSPitch;
  float* ml = red + 4 * NQ * p.hd;
  __shared__ int s_last;
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hd = p.hd, H = p.H, K1 = p.K + 1;
  const int lpk = hd >> 3, G = 32 / lpk;
  const int sub = lane & (lpk - 1), grp = lane / lpk;
  const int C = p.plan[0], n_items = p.plan[1] * H;
  constexpr int kU = 4;  // keys per lane group in flight
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int pair = item / H, hh = item - pair * H;
    const int b = p.plan[2 + 2 * pair], s = p.plan[3 + 2 * pair];
    const int p0 = p.positions[b];
    const int keys = p0 + K1;
    const int k0 = s * C, k1 = min(keys, k0 + C), n = k1 - k0;
    const int nsplit = (keys + C - 1) / C;
    const size_t cbase = ((size_t)(b * H + hh) * p.max_pos) * hd + sub * 8;
    const uint4* kp = reinterpret_cast<const uint4*>(p.kc + cbase);
    const uint4* vp = reinterpret_cast<const uint4*>(p.vc + cbase);
    const int kstride = hd / 8;  // uint4 per key

    // ---- scores (log2 domain): S[j][key - k0] = q_j . k * scale * log2(e)
    {
      float qr[NQ][8];
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        if (j < K1) {
          const float4* qp = reinterpret_cast<const float4*>(
              p.q + (size_t)(b * K1 + j) * p.d + hh * hd + sub * 8);
          const float4 a = __ldcg(qp), c = __ldcg(qp + 1);
          qr[j][0] = a.x * p.scale_log2; qr[j][1] = a.y * p.scale_log2;
          qr[j][2] = a.z * p.scale_log2; qr[j][3] = a.w * p.scale_log2;
          qr[j][4] = c.x * p.scale_log2; qr[j][5] = c.y * p.scale_log2;
          qr[j][6] = c.z * p.scale_log2; qr[j][7] = c.w * p.scale_log2;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) qr[j][e] = 0.f;
        }
      }
      const int step = 4 * G;
      for (int base = k0 + warp * G; base < k1; base += kU * step) {
        uint4 kv[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key = base + u * step + grp;
          kv[u] = key < k1 ? __ldcs(kp + (size_t)key * kstride) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key = base + u * step + grp;
          if (base + u * step >= k1) break;  // the same for the whole warp
          float kf[8];
          bf16x8_to_f(kv[u], kf);
          float dot[NQ];
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaf(qr[j][e], kf[e], a);
            dot[j] = a;
          }
          for (int o = 1; o < lpk; o <<= 1) {
#pragma unroll
            for (int j = 0; j < NQ; ++j) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], o);
          }
          if (key < k1) {
#pragma unroll
            for (int j = 0; j < NQ; ++j)
              if ((j & (lpk - 1)) == sub && j < K1)
                S[j * kSPitch + (key - k0)] = key <= p0 + j ? dot[j] : -INFINITY;
          }
        }
      }
    }
    __syncthreads();

    // ---- per query: max, numerators in place, their sum
    for (int j = warp; j < K1; j += 4) {
      float* Sj = S + j * kSPitch;
      float m = -INFINITY;
      for (int i = lane; i < n; i += 32) m = fmaxf(m, Sj[i]);
      m = warp_max_f(m);
      float l = 0.f;
      for (int i = lane; i < n; i += 32) {
        const float e = m == -INFINITY ? 0.f : exp2f(Sj[i] - m);
        Sj[i] = e;
        l += e;
      }
      l = warp_sum_f(l);
      if (lane == 0) {
        ml[2 * j] = m;
        ml[2 * j + 1] = l;
      }
    }
    __syncthreads();

    // ---- acc_j = sum over keys of p_j(key) v(key), this lane's 8 dims
    float acc[NQ][8];
#pragma unroll
    for (int j = 0; j < NQ; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
    {
      const int step = 4 * G;
      for (int base = k0 + warp * G; base < k1; base += kU * step) {
        uint4 vv[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key = base + u * step + grp;
          vv[u] = key < k1 ? __ldcs(vp + (size_t)key * kstride) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int key = base + u * step + grp;
          if (key >= k1) continue;
          float vf[8];
          bf16x8_to_f(vv[u], vf);
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            if (j >= K1) break;
            const float pj = S[j * kSPitch + (key - k0)];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(pj, vf[e], acc[j][e]);
          }
        }
      }
    }
    // over the lane groups of the warp, then over the warps (in order)
    for (int o = lpk; o < 32; o <<= 1) {
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[j][e] += __shfl_xor_sync(0xffffffffu, acc[j][e], o);
    }
    if (grp == 0) {
#pragma unroll
      for (int j = 0; j < NQ; ++j)
        if (j < K1) {
#pragma unroll
          for (int e = 0; e < 8; ++e) red[(warp * NQ + j) * hd + sub * 8 + e] = acc[j][e];
        }
    }
    __syncthreads();
    const int outs = K1 * hd;
    if (nsplit == 1) {
      for (int i = tid; i < outs; i += kAttnThreads) {
        const int j = i / hd, dim = i - j * hd;
        float a = red[j * hd + dim];
        for (int w = 1; w < 4; ++w) a += red[(w * NQ + j) * hd + dim];
        p.o[(size_t)(b * K1 + j) * p.d + hh * hd + dim] = __float2bfloat16_rn(a / ml[2 * j + 1]);
      }
    } else {
      // this split's (max, sum, unnormalised output) per query
      const int pitch = hd + 2;
      float* mine = p.part + (size_t)item * K1 * pitch;
      for (int i = tid; i < outs; i += kAttnThreads) {
        const int j = i / hd, dim = i - j * hd;
        float a = red[j * hd + dim];
        for (int w = 1; w < 4; ++w) a += red[(w * NQ + j) * hd + dim];
        mine[j * pitch + 2 + dim] = a;
      }
      for (int j = tid; j < K1; j += kAttnThreads) {
        mine[j * pitch] = ml[2 * j];
        mine[j * pitch + 1] = ml[2 * j + 1];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int done = atomicAdd(p.arrive + b * H + hh, 1);
        s_last = done == nsplit - 1;
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        // merge the splits in order: item of split s' = (pair - s + s') * H + hh
        const int first = (pair - s) * H + hh;
        for (int i = tid; i < outs; i += kAttnThreads) {
          const int j = i / hd, dim = i - j * hd;
          float M = -INFINITY;
          for (int q = 0; q < nsplit; ++q) {
            const float* pq = p.part + (size_t)(first + q * H) * K1 * pitch + j * pitch;
            if (__ldcg(pq + 1) > 0.f) M = fmaxf(M, __ldcg(pq));
          }
          float Ls = 0.f, A = 0.f;
          for (int q = 0; q < nsplit; ++q) {
            const float* pq = p.part + (size_t)(first + q * H) * K1 * pitch + j * pitch;
            const float lq = __ldcg(pq + 1);
            if (!(lq > 0.f)) continue;
            const float w = exp2f(__ldcg(pq) - M);
            Ls = fmaf(lq, w, Ls);
            A = fmaf(__ldcg(pq + 2 + dim), w, A);
          }
          p.o[(size_t)(b * K1 + j) * p.d + hh * hd + dim] = __float2bfloat16_rn(A / Ls);
        }
        if (tid == 0) p.arrive[b * H + hh] = 0;
      }
    }
    __syncthreads();  // S, red and ml are reused by the next item
  }
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

template <int NQ>
cudaError_t launch_attn_t(const AttnParams& p, int grid, cudaStream_t s, bool pdl) {
  const size_t smem = attn_smem_bytes(NQ, p.hd);
  cudaError_t e =
      cudaFuncSetAttribute(attn_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_kernel<NQ>, dim3(grid), dim3(kAttnThreads), smem, s, pdl, p);
}

}  // namespace

size_t attn_smem_bytes(int nq, int hd) {
  return ((size_t)nq * kSPitch + 4 * (size_t)nq * hd + 2 * (size_t)nq) * sizeof(float);
}

cudaError_t launch_attn_norm(const AttnNormParams& p, cudaStream_t s, bool pdl) {
  return launch_pdl(attn_norm_kernel, dim3(p.T), dim3(kNormThreads), 0, s, pdl, p);
}

cudaError_t launch_attn(const AttnParams& p, int grid, cudaStream_t s, bool pdl) {
  const int nq = p.K + 1;
  if (nq <= 1) return launch_attn_t<1>(p, grid, s, pdl);
  if (nq <= 2) return launch_attn_t<2>(p, grid, s, pdl);
  if (nq <= 4) return launch_attn_t<4>(p, grid, s, pdl);
  if (nq <= 8) return launch_attn_t<8>(p, grid, s, pdl);
  return launch_attn_t<16>(p, grid, s, pdl);
}

cudaError_t launch_repack_qkv(__nv_bfloat16* dst, const __nv_bfloat16* wq,
                              const __nv_bfloat16* wk, const __nv_bfloat16* wv, int d, int hd,
                              int rows_pad, cudaStream_t s) {
  repack_qkv_kernel<<<rows_pad, 128, 0, s>>>(dst, wq, wk, wv, d, hd, rows_pad);
  return cudaGetLastError();
}

}  // namespace mv
