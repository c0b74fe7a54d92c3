// Greedy head (final RMSNorm + lm_head + argmax) for callers that cannot
// allocate device memory.
//
// The regular entry points keep their scratch (the normalised rows and the
// argmax keys) in a context that moe_verify_init allocates with cudaMalloc.
// Some callers cannot do that: code whose device memory belongs to another
// allocator with a fixed budget (a framework's caching pool), code that must
// not stall other streams (cudaMalloc and cudaFree can synchronise the
// device), and code that runs where CUDA allocation calls are not allowed.
// This file gives them one entry point whose scratch is a fixed-size array in
// the library's own device memory, reserved when the library is loaded; the
// call itself allocates nothing.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_verify.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int kMaxTokens = MOE_VERIFY_NOALLOC_MAX_TOKENS;
constexpr int kMaxHidden = MOE_VERIFY_NOALLOC_MAX_HIDDEN;
constexpr int kMaxDevices = 64;

// Layout of the scratch array (byte offsets).
constexpr size_t kXfBytes = (size_t)kMaxTokens * kMaxHidden * 2;  // bf16 rows
constexpr size_t kKeysOff = kXfBytes;
constexpr size_t kBadOff = kKeysOff + (size_t)kMaxTokens * 8;
constexpr size_t kDoneOff = kBadOff + (size_t)kMaxTokens * 4;  // [0] done, [1] aborted
constexpr size_t kStatusOff = kDoneOff + 16;
constexpr size_t kScratchBytes = kStatusOff + 16;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;  // guarded by g_setup_mu

// Device address of g_scratch on the current device, and the CUDA driver API's
// tensor-map encoder.  In host code the name g_scratch is only a host-side
// stand-in, so the address is asked for once per device, with that device
// current.
int scratch_address(int dev, unsigned char** out, PFN_cuTensorMapEncodeTiled_v12000* encode) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_VERIFY_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
      cudaGetLastError();
      return MOE_VERIFY_ERR_CUDA;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *encode = g_encode;
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_VERIFY_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return MOE_VERIFY_OK;
}

// One block of 256 threads per token: xf = bf16(h * rsqrt(mean(h^2) + eps) * g),
// with the sum of squares reduced in the same order as the verify step's
// final RMSNorm (per thread over 4-float chunks c = tid, tid + 256, ..., then
// per warp, then over the warps in order), so both give the same bits.  Also
// clears what must start at zero: the token's argmax key and invalid flag, and
// (block 0) the lm_head's completion and abort counters and the status word.
__global__ void __launch_bounds__(256) noalloc_norm_kernel(const float* __restrict__ h,
                                                           const __nv_bfloat16* __restrict__ gain,
                                                           int T, int d, float eps,
                                                           unsigned char* scratch) {
  __shared__ float red[8];
  __nv_bfloat16* xf = reinterpret_cast<__nv_bfloat16*>(scratch);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(scratch + kKeysOff);
  int32_t* bad = reinterpret_cast<int32_t*>(scratch + kBadOff);
  unsigned int* done = reinterpret_cast<unsigned int*>(scratch + kDoneOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  if (t == 0 && tid == 0) {
    done[0] = 0u;
    done[1] = 0u;
    *reinterpret_cast<uint32_t*>(scratch + kStatusOff) = 0u;
  }
  const float4* row = reinterpret_cast<const float4*>(h + (size_t)t * d);
  const int nc = d / 4;
  float ss = 0.f;
  for (int c = tid; c < nc; c += 256) {
    const float4 v = row[c];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)d + eps);
  for (int c = tid; c < nc; c += 256) {
    const float4 v = row[c];
    const int i = 4 * c;
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * r * __bfloat162float(gain[i]),
                                              v.y * r * __bfloat162float(gain[i + 1]));
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * r * __bfloat162float(gain[i + 2]),
                                              v.w * r * __bfloat162float(gain[i + 3]));
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(xf + (size_t)t * d)[c] = packed;
  }
  if (tid == 0) {
    keys[t] = 0ull;
    bad[t] = 0;
  }
}

}  // namespace

extern "C" MOE_VERIFY_API int moe_verify_greedy_head_noalloc(const float* h,
                                                             const void* final_norm,
                                                             const void* lm_head, int32_t T,
                                                             int32_t d, int32_t V, float rms_eps,
                                                             int32_t* target_ids,
                                                             void* cuda_stream) {
  if (!h || !final_norm || !lm_head || !target_ids) return MOE_VERIFY_ERR_ARG;
  if (T < 1 || d < 64 || V < 2 || !(rms_eps > 0.f)) return MOE_VERIFY_ERR_ARG;
  if (T > kMaxTokens || d > kMaxHidden || d % 64 != 0) return MOE_VERIFY_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(lm_head) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(h) & 15u) != 0)
    return MOE_VERIFY_ERR_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_VERIFY_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_VERIFY_ERR_CUDA;
  unsigned char* scratch = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  int rc = scratch_address(dev, &scratch, &fn);
  if (rc != MOE_VERIFY_OK) return rc;

  auto encode = [fn](CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                     uint32_t box_rows) -> bool {
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  // a chunk's normalised rows arrive as one box of nch rows
  const mv::LmLayout lay = mv::lm_layout_single(T);  // the single-CTA kernel below
  const int nch = lay.nch;
  CUtensorMap map_lm, map_xf;
  // rows past V (the last vocabulary tile) and past T are read as zeros
  if (!encode(&map_lm, lm_head, (uint64_t)d, (uint64_t)V, 128) ||
      !encode(&map_xf, scratch, (uint64_t)d, (uint64_t)kMaxTokens, (uint32_t)nch))
    return MOE_VERIFY_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  noalloc_norm_kernel<<<T, 256, 0, s>>>(h, static_cast<const __nv_bfloat16*>(final_norm), T, d,
                                         rms_eps, scratch);
  if (cudaGetLastError() != cudaSuccess) return MOE_VERIFY_ERR_CUDA;

  mv::GemmParams gp = {};
  gp.n_items_static = ((V + 127) / 128) * lay.n_chunks;
  gp.kblocks = d / 64;
  gp.nch = nch;
  gp.stages = lay.stages;
  gp.tmem_cols = lay.tmem_cols;
  gp.status = reinterpret_cast<uint32_t*>(scratch + kStatusOff);
  gp.T = T;
  gp.V = V;
  gp.n_chunks = lay.n_chunks;
  gp.nch_lm = nch;
  gp.keys = reinterpret_cast<unsigned long long*>(scratch + kKeysOff);
  gp.logits = nullptr;
  gp.targets = target_ids;
  gp.bad = reinterpret_cast<const int32_t*>(scratch + kBadOff);
  gp.done = reinterpret_cast<unsigned int*>(scratch + kDoneOff);
  gp.aborted = reinterpret_cast<unsigned int*>(scratch + kDoneOff) + 1;
  if (mv::launch_lmhead(map_lm, map_xf, gp, lay.tokens_on_m, sms, s, false) != cudaSuccess)
    return MOE_VERIFY_ERR_CUDA;
  return MOE_VERIFY_OK;
}
