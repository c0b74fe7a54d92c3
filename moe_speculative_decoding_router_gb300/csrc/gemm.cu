// Grouped GEMMs of the verify step on the 5th-generation tensor cores.
//
// One persistent kernel shape serves three products:
//   kGateUp  [tile of 64 gate rows + 64 up rows of one expert] x [its tokens]
//            epilogue: a = bf16(silu(g) * u)                (SwiGLU)
//   kDown    [128 rows of one expert's down projection] x [its tokens' a]
//            epilogue: y[token, slot] = p * (a W_d^T)        (weighted combine)
//   kLmHead  [128 vocabulary rows] x [all verify tokens]
//            epilogue: running argmax over the vocabulary     (greedy choice)
// The weight rows sit on the MMA's M side (128) and the few tokens of an
// expert on its N side (16..256), so every weight byte is streamed from HBM
// once per item while the tensor pipe stays legal at small batch.
//
// Per CTA: warp 0 issues TMA loads into a ring of shared-memory stages, one
// thread of warp 1 issues tcgen05.mma into a double-buffered TMEM
// accumulator, and warps 2..5 drain TMEM through tcgen05.ld.  Items are
// taken round-robin: item i runs on CTA i mod gridDim.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace mv {

namespace {

constexpr int kGemmThreads = 192;
constexpr int kStageA = 128 * 128;  // 128 weight rows x 64 bf16
constexpr int kXbufBytes = 2 * 16 * 64 * 4;
constexpr int kBarBytes = 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int MODE>
__device__ __forceinline__ Item get_item(const GemmParams& p, int i) {
  if (MODE == kLmHead) {
    Item it;
    const int vt = i / p.n_chunks, c = i % p.n_chunks;
    it.a_row = vt * 128;
    it.b_row = c * p.nch_lm;
    it.n = min(p.nch_lm, p.T - c * p.nch_lm);
    it.aux = vt;
    return it;
  } else {
    const int4 v = __ldg(reinterpret_cast<const int4*>(p.items) + i);
    Item it;
    it.a_row = v.x;
    it.b_row = v.y;
    it.n = v.z;
    it.aux = v.w;
    return it;
  }
}

// Orderable key of (logit, vocabulary id): larger logit first, then lower id.
__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int o) {
  uint32_t lo = (uint32_t)v, hi = (uint32_t)(v >> 32);
  lo = __shfl_xor_sync(0xffffffffu, lo, o);
  hi = __shfl_xor_sync(0xffffffffu, hi, o);
  return ((unsigned long long)hi << 32) | lo;
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stage_bytes = kStageA + p.nch * 128;
  uint8_t* stages = smem;
  uint8_t* ctrl = smem + (size_t)p.stages * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + p.stages;
  uint64_t* tfull = empty + p.stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* xfull = drain + 1;   // epilogue exchange buffer filled [2]
  uint64_t* xempty = xfull + 2;  // epilogue exchange buffer free [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xbuf = reinterpret_cast<float*>(ctrl + kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    // gate/up: the two "up" warps fill, the two "gate" warps drain;
    // lm_head: all four warps fill, warp 2 drains.
    for (int b = 0; b < 2; ++b) {
      mbar_init(&xfull[b], MODE == kLmHead ? 4 : 2);
      mbar_init(&xempty[b], MODE == kLmHead ? 1 : 2);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  // everything above is independent of the previous kernel's output; all
  // global writes of this grid come after pdl_wait
  pdl_launch_dependents();
  pdl_wait();
  const int n_items = (MODE == kLmHead) ? p.n_items_static : __ldcg(p.n_items);
  const bool has_work = (int)blockIdx.x < n_items;
  if (has_work && warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = has_work ? *tmem_slot : 0u;

  if (has_work) {
    if (warp == 0) {
      // ------------------------------------------------ TMA producer
      if (lane == 0) {
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        int issued_rounds = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
          const Item it = get_item<MODE>(p, i);
          const int npad = (it.n + 15) & ~15;
          const uint32_t bytes = (uint32_t)(kStageA + npad * 128);
          for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            uint8_t* sa = stages + (size_t)stage * stage_bytes;
            uint8_t* sb = sa + kStageA;
            mbar_arrive_expect_tx(&full[stage], bytes);
            tma_load_2d(sa, &mapA, &full[stage], kb * 64, it.a_row, pol_w);
            for (int j = 0; j < npad; j += 16)
              tma_load_2d(sb + j * 128, &mapB, &full[stage], kb * 64, it.b_row + j, pol_x);
            ++issued_rounds;
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok) {
          // wind down: let every load already issued land before the CTA exits
          const int last = issued_rounds;
          for (int r = (last > p.stages ? last - p.stages : 0); r < last; ++r) {
            const int s = r % p.stages;
            const uint32_t par = (uint32_t)((r / p.stages) & 1);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&full[s], par) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x, ++local) {
          const Item it = get_item<MODE>(p, i);
          const int npad = (it.n + 15) & ~15;
          const uint32_t idesc = umma_idesc_bf16(128, (uint32_t)npad);
          const int buf = local & 1;
          const uint32_t use = (uint32_t)(local >> 1);
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tmem_d = tmem_base + (uint32_t)(buf * p.nch);
          for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(stages + (size_t)stage * stage_bytes);
            const uint32_t sb = sa + kStageA;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              umma_bf16(tmem_d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32),
                        idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&empty[stage]);
            if (++stage == p.stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) umma_commit(&tfull[buf]);
        }
        // all MMAs issued by this thread complete before TMEM is released
        umma_commit(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    } else {
      // ------------------------------------------------ epilogue warps 2..5
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const int row = q * 32 + lane;
      int local = 0;
      uint32_t chunk_seq = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const Item it = get_item<MODE>(p, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&tfull[buf], use & 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * p.nch);

        bool ok = true;
        if (MODE == kGateUp) {
          // rows 0..63: gate, rows 64..127: up, for intermediate columns aux*64 + r
          for (int c0 = 0; c0 < npad && ok; c0 += 16, ++chunk_seq) {
            uint32_t v[16];
            tmem_ld16(tb + (uint32_t)c0, v);
            tmem_ld_wait();
            const uint32_t xb = chunk_seq & 1u, xu = chunk_seq >> 1;
            float* U = xbuf + xb * (16 * 64);
            if (q >= 2) {
              ok = mbar_wait(&xempty[xb], (xu & 1u) ^ 1u, abort_flag, p.status);
              if (ok) {
#pragma unroll
                for (int j = 0; j < 16; ++j) U[j * 64 + (row - 64)] = __uint_as_float(v[j]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&xfull[xb]);
              }
            } else {
              ok = mbar_wait(&xfull[xb], xu & 1u, abort_flag, p.status);
              if (ok) {
                __nv_bfloat16* out = p.a_out + (size_t)it.aux * 64 + row;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int n = c0 + j;
                  if (n < it.n) {
                    const float g = __uint_as_float(v[j]);
                    const float u = U[j * 64 + row];
                    const float a = g / (1.0f + __expf(-g)) * u;
                    out[(size_t)(it.b_row + n) * p.I_pad] = __float2bfloat16_rn(a);
                  }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xempty[xb]);
              }
            }
          }
        } else if (MODE == kDown) {
          const int m = it.aux * 128 + row;  // output dimension
          for (int c0 = 0; c0 < npad; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tb + (uint32_t)c0, v);
            tmem_ld_wait();
            if (m < p.d) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = c0 + j;
                if (n < it.n) {
                  const int r = it.b_row + n;
                  const int tok = __ldg(p.perm_token + r);
                  const int slot = __ldg(p.perm_slot + r);
                  const float w = __ldg(p.perm_w + r);
                  p.y[((size_t)tok * p.kS + slot) * p.d + m] = w * __uint_as_float(v[j]);
                }
              }
            }
          }
        } else {
          // greedy argmax over this tile's 128 vocabulary rows, per token column
          const int vid = it.a_row + row;
          const bool valid = vid < p.V;
          unsigned long long* red = reinterpret_cast<unsigned long long*>(xbuf);
          for (int c0 = 0; c0 < npad && ok; c0 += 16, ++chunk_seq) {
            uint32_t v[16];
            tmem_ld16(tb + (uint32_t)c0, v);
            tmem_ld_wait();
            const uint32_t xb = chunk_seq & 1u, xu = chunk_seq >> 1;
            unsigned long long* R = red + xb * 64;
            unsigned long long keys[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float lv = __uint_as_float(v[j]);
              unsigned long long key = valid ? argmax_key(lv, vid) : 0ull;
              if (p.logits && valid && c0 + j < it.n)
                p.logits[(size_t)(it.b_row + c0 + j) * p.V + vid] = lv;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long other = shfl_xor_u64(key, o);
                key = other > key ? other : key;
              }
              keys[j] = key;
            }
            ok = mbar_wait(&xempty[xb], (xu & 1u) ^ 1u, abort_flag, p.status);
            if (!ok) break;
            if (lane == 0) {
#pragma unroll
              for (int j = 0; j < 16; ++j) R[(warp - 2) * 16 + j] = keys[j];
              mbar_arrive(&xfull[xb]);
            }
            if (warp == 2) {
              ok = mbar_wait(&xfull[xb], xu & 1u, abort_flag, p.status);
              if (!ok) break;
              if (lane < 16 && c0 + lane < it.n) {
                unsigned long long k0 = R[lane], k1 = R[16 + lane], k2 = R[32 + lane],
                                   k3 = R[48 + lane];
                k0 = k1 > k0 ? k1 : k0;
                k2 = k3 > k2 ? k3 : k2;
                k0 = k2 > k0 ? k2 : k0;
                atomicMax(p.keys + it.b_row + c0 + lane, k0);
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(&xempty[xb]);
            }
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
      }
    }
  }

  __syncthreads();
  if (has_work && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  if (MODE == kLmHead) {
    // the last CTA turns the argmax keys into token ids
    __threadfence();
    __syncthreads();
    __shared__ int is_last;
    if (threadIdx.x == 0) is_last = (atomicAdd(p.done, 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (is_last) {
      __threadfence();
      for (int t = threadIdx.x; t < p.T; t += blockDim.x) {
        const unsigned long long key = __ldcg(p.keys + t);
        const int id = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        p.targets[t] = (__ldg(p.bad + t) || key == 0ull) ? -1 : id;
      }
      if (threadIdx.x == 0) *p.done = 0u;
    }
  }
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p,
                        int grid, cudaStream_t s, bool pdl) {
  const size_t smem = gemm_smem_bytes(p.nch, p.stages);
  auto kern = gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, mapA, mapB, p);
}

}  // namespace

size_t gemm_smem_bytes(int nch, int stages) {
  return 1024 /* alignment slack */ + (size_t)stages * (kStageA + (size_t)nch * 128) + kBarBytes +
         kXbufBytes;
}

int gemm_max_stages(int nch) {
  const size_t budget = 227 * 1024;
  int s = 16;
  while (s > 2 && gemm_smem_bytes(nch, s) > budget) --s;
  return s;
}

cudaError_t launch_gemm(int mode, const CUtensorMap& mapA, const CUtensorMap& mapB,
                        const GemmParams& p, int grid, cudaStream_t s, bool pdl) {
  switch (mode) {
    case kGateUp: return launch_mode<kGateUp>(mapA, mapB, p, grid, s, pdl);
    case kDown: return launch_mode<kDown>(mapA, mapB, p, grid, s, pdl);
    default: return launch_mode<kLmHead>(mapA, mapB, p, grid, s, pdl);
  }
}

}  // namespace mv
