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

// Self-check of the bounded waits: one thread waits on an mbarrier phase
// that nothing completes, then spins (acquire loads, as the expert FFN's
// dependency wait does) on a flag that nothing sets, each with limit_ns.
// out[0] = elapsed ns, out[1] = 1 if the mbarrier wait gave up and raised the
// timeout bit, out[2] = 1 if the flag wait gave up.
__global__ void bounded_wait_check_kernel(const int32_t* flag, uint32_t* status, uint64_t limit_ns,
                                          unsigned long long* out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const uint64_t t0 = globaltimer_ns();
  const bool got = mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  out[1] = (!got && abort_flag && (*status & kErrTimeout)) ? 1ull : 0ull;
  abort_flag = 0;
  const uint64_t t1 = globaltimer_ns();
  bool gave_up = false;
  uint32_t n = 0;
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v > 0) break;
    if ((++n & 63u) == 0 && globaltimer_ns() - t1 > limit_ns) {
      atomicOr(status, kErrTimeout);
      gave_up = true;
      break;
    }
  }
  out[2] = gave_up ? 1ull : 0ull;
  out[0] = globaltimer_ns() - t0;
}

// The draft head's inputs from a verify step: per sequence b, the final
// residual of its accepted verify position n_b and the token committed
// there (the last committed token).  One block per sequence.
__global__ void draft_inputs_kernel(const float* __restrict__ h, const int32_t* __restrict__ committed,
                                    const int32_t* __restrict__ accept_len, int K, int d,
                                    float* __restrict__ h_out, int32_t* __restrict__ t_out) {
  const int b = blockIdx.x;
  const int n = max(accept_len[b], 0);
  const size_t row = (size_t)b * (K + 1) + n;
  const float4* src = reinterpret_cast<const float4*>(h + row * d);
  float4* dst = reinterpret_cast<float4*>(h_out + (size_t)b * d);
  for (int c = threadIdx.x; c < d / 4; c += blockDim.x) dst[c] = src[c];
  if (threadIdx.x == 0) t_out[b] = committed[row];
}

__global__ void scatter_column_kernel(const int32_t* __restrict__ src, int B, int32_t* dst, int stride,
                                      int col) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) dst[(size_t)b * stride + col] = src[b];
}

__device__ int32_t g_never_set;               // stays 0
__device__ uint32_t g_check_status;
__device__ unsigned long long g_check_out[3];

}  // namespace

cudaError_t run_bounded_wait_check(uint64_t limit_ns, cudaStream_t s, unsigned long long* host_out,
                                   uint32_t* host_status) {
  int32_t* flag = nullptr;
  uint32_t* st = nullptr;
  unsigned long long* out = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&flag), g_never_set);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st), g_check_status);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&out), g_check_out);
  if (e == cudaSuccess) e = cudaMemsetAsync(st, 0, 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(out, 0, sizeof(unsigned long long) * 3, s);
  if (e != cudaSuccess) return e;
  bounded_wait_check_kernel<<<1, 32, 0, s>>>(flag, st, limit_ns, out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaMemcpyAsync(host_out, out, sizeof(unsigned long long) * 3, cudaMemcpyDeviceToHost,
                           s)) != cudaSuccess)
    return e;
  if ((e = cudaMemcpyAsync(host_status, st, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t launch_draft_inputs(const float* h, const int32_t* committed, const int32_t* accept_len,
                                int B, int K, int d, float* h_out, int32_t* t_out, cudaStream_t s) {
  draft_inputs_kernel<<<B, 128, 0, s>>>(h, committed, accept_len, K, d, h_out, t_out);
  return cudaGetLastError();
}

cudaError_t launch_scatter_column(const int32_t* src, int B, int32_t* dst, int stride, int col,
                                  cudaStream_t s) {
  scatter_column_kernel<<<(B + 127) / 128, 128, 0, s>>>(src, B, dst, stride, col);
  return cudaGetLastError();
}

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
