// Acceptance rule, weight repacking and small conversions.
#include "internal.h"
#include "ptx.cuh"

namespace mv {

namespace {

// Greedy acceptance, one thread per sequence ("Jina AI Releases jina-ocr-v1,
// a 3.4B MoE Document Parser With Built-In Speculative Decoding", FastMTP
// paragraph): keep the longest draft prefix equal to the target's greedy
// choices, then commit the target's own next token.
__global__ void accept_kernel(AcceptParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int K = p.K;
  const int32_t* d = p.drafts + (size_t)b * K;
  const int32_t* y = p.targets + (size_t)b * (K + 1);
  int32_t* out = p.committed + (size_t)b * (K + 1);
  bool bad = false;
  int32_t dv[16], yv[16];
  for (int i = 0; i < K; ++i) {
    dv[i] = d[i];
    bad |= (dv[i] < 0 || dv[i] >= p.V);
  }
  for (int i = 0; i <= K; ++i) {
    yv[i] = y[i];
    bad |= (yv[i] < 0 || yv[i] >= p.V);
  }
  if (bad) {
    for (int i = 0; i <= K; ++i) out[i] = -1;
    p.accept_len[b] = -1;
    atomicOr(p.status, kErrIdRange);
    return;
  }
  int n = 0;
  while (n < K && dv[n] == yv[n]) ++n;
  for (int i = 0; i <= K; ++i) out[i] = (i <= n) ? yv[i] : -1;
  p.accept_len[b] = n;
}

// Gate/up weights of all experts of one layer, as 128-row tiles: tile
// (e, mt) holds gate rows mt*64 .. mt*64+63 then up rows mt*64 .. +63.
// Experts E .. E+S-1 are the shared experts.  Rows past I are zero.
__global__ void repack_gateup_kernel(__nv_bfloat16* __restrict__ dst,
                                     const __nv_bfloat16* __restrict__ gate,
                                     const __nv_bfloat16* __restrict__ up,
                                     const __nv_bfloat16* __restrict__ s_gate,
                                     const __nv_bfloat16* __restrict__ s_up, int E, int S, int I,
                                     int Is, int d, int mt_gu) {
  const int64_t rows = (int64_t)(E + S) * mt_gu * 128;
  const int64_t total = rows * d;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t R = i / d;
    const int c = (int)(i % d);
    const int e = (int)(R / ((int64_t)mt_gu * 128));
    const int mt = (int)((R / 128) % mt_gu);
    const int r = (int)(R % 128);
    const int j = mt * 64 + (r & 63);
    const bool is_up = r >= 64;
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (e < E) {
      if (j < I) v = (is_up ? up : gate)[((size_t)e * I + j) * d + c];
    } else {
      if (j < Is) v = (is_up ? s_up : s_gate)[((size_t)(e - E) * Is + j) * d + c];
    }
    dst[i] = v;
  }
}

// Down weights of all experts of one layer as 128-row tiles of output
// dimensions, K (intermediate) padded with zeros to I_pad.
__global__ void repack_down_kernel(__nv_bfloat16* __restrict__ dst,
                                   const __nv_bfloat16* __restrict__ down,
                                   const __nv_bfloat16* __restrict__ s_down, int E, int S, int I,
                                   int Is, int d, int I_pad, int mt_dn) {
  const int64_t rows = (int64_t)(E + S) * mt_dn * 128;
  const int64_t total = rows * I_pad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t R = i / I_pad;
    const int j = (int)(i % I_pad);
    const int e = (int)(R / ((int64_t)mt_dn * 128));
    const int m = (int)(R % ((int64_t)mt_dn * 128));
    __nv_bfloat16 v = __float2bfloat16_rn(0.f);
    if (m < d) {
      if (e < E) {
        if (j < I) v = down[((size_t)e * d + m) * I + j];
      } else {
        if (j < Is) v = s_down[((size_t)(e - E) * d + m) * Is + j];
      }
    }
    dst[i] = v;
  }
}

__global__ void bf16_to_f32_kernel(float* dst, const __nv_bfloat16* src, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __bfloat162float(src[i]);
}

int grid_for(int64_t total) {
  int64_t g = (total + 255) / 256;
  if (g > 8192) g = 8192;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t s) {
  const int grid = (p.B + 127) / 128;
  accept_kernel<<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_repack_gateup(__nv_bfloat16* dst, const __nv_bfloat16* gate,
                                 const __nv_bfloat16* up, const __nv_bfloat16* s_gate,
                                 const __nv_bfloat16* s_up, int E, int S, int I, int Is, int d,
                                 int mt_gu, cudaStream_t s) {
  const int64_t total = (int64_t)(E + S) * mt_gu * 128 * d;
  repack_gateup_kernel<<<grid_for(total), 256, 0, s>>>(dst, gate, up, s_gate, s_up, E, S, I, Is, d,
                                                       mt_gu);
  return cudaGetLastError();
}

cudaError_t launch_repack_down(__nv_bfloat16* dst, const __nv_bfloat16* down,
                               const __nv_bfloat16* s_down, int E, int S, int I, int Is, int d,
                               int I_pad, int mt_dn, cudaStream_t s) {
  const int64_t total = (int64_t)(E + S) * mt_dn * 128 * I_pad;
  repack_down_kernel<<<grid_for(total), 256, 0, s>>>(dst, down, s_down, E, S, I, Is, d, I_pad,
                                                     mt_dn);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f32(float* dst, const __nv_bfloat16* src, int64_t n, cudaStream_t s) {
  bf16_to_f32_kernel<<<grid_for(n), 256, 0, s>>>(dst, src, n);
  return cudaGetLastError();
}

}  // namespace mv
