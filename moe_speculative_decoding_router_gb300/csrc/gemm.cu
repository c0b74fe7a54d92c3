// Grouped GEMMs of the verify step on the 5th-generation tensor cores.
//
// ffn_kernel: one layer's expert FFN in one persistent launch.  Work items:
//   gate/up  [64 gate rows + 64 up rows of one expert] x [<= nch of its rows]
//            epilogue a = bf16(silu(g) * u)                  (SwiGLU)
//   down     [128 rows of one expert's down projection] x [the same rows' a]
//            epilogue y[token, slot] = p * (a W_d^T)         (weighted combine)
// All gate/up items come first, then all down items.  Items are claimed in
// order from a global counter (the first as the CTA starts, the next one
// claim ahead of use), so CTAs that stream faster take more items and all
// finish within about one item of each other.  A down item waits (bounded)
// until both SwiGLU halves of every gate/up tile of its chunk of rows are
// written; the items it waits for were claimed earlier, by CTAs that are
// running, and have no waits of their own.
// Once a CTA has issued its last load it pulls into L2 the weight item its
// index starts with in the next kernel (next layer, or the lm_head).
// ffn_tokm_kernel: the same layer's work with the operands swapped, for large
// T: a chunk of <= 128 of an expert's rows on the MMA's M side, 256 weight rows
// on N, so that each epilogue thread owns one row and the SwiGLU and the
// weighted combine need no exchange between warps.
// lmhead_kernel: [128 vocabulary rows] x [a chunk of <= 256 verify tokens],
// epilogue the running greedy argmax over the vocabulary (two warp
// reductions per token column, then across the four epilogue warps).
// lmhead_tokm_kernel: the same product with the tokens on the MMA's M side
// (65..128 tokens), so each epilogue thread holds one token's logits and
// keeps its argmax in registers across the CTA's tiles.  Measured on the full
// step, the second is faster from ~96 to 128 tokens and the first at 64
// tokens or fewer and above 128 (there the vocabulary-on-M form loads each
// tile once for up to 256 tokens).  Both load a chunk's normalised rows as
// one TMA box per stage (the tensor map's box is the chunk width): many small
// boxes per stage throttled the TMA unit.
//
// The weight rows sit on the MMA's M side (128) and the few tokens of an
// expert on its N side (16..256), so every weight byte is streamed from HBM
// once per item while the tensor pipe stays legal at small batch.
//
// Per CTA: warp 0 issues TMA loads into a ring of shared-memory stages, one
// thread of warp 1 issues tcgen05.mma into a double-buffered TMEM
// accumulator, and warps 2..5 drain TMEM through tcgen05.ld.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"
#include "route_stages.cuh"

namespace mv {

namespace {

constexpr int kGemmThreads = 192;
// The single-kernel layer's CTAs: 16 warps, for its routing tasks (the
// routing kernel's block size); warps 6.. take no expert-FFN role.
constexpr int kLayerThreads = 512;
constexpr int kStageA = 128 * 128;  // 128 weight rows x 64 bf16
constexpr int kXbufBytes = 2 * 16 * 64 * 4;
constexpr int kCtrlBytes = 1024;
constexpr int kMaxExperts = 264;  // routed (<= 256) + shared (<= 8)
constexpr int kQueue = 8;         // claimed items in flight inside a CTA
constexpr int kListBytes = 6144;  // per-expert counts and prefix sums (<= 264 experts)

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Orderable 32-bit image of a float: larger float, larger unsigned value.
__device__ __forceinline__ uint32_t orderable(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Orderable key of (logit, vocabulary id): larger logit first, then lower id.
__device__ __forceinline__ unsigned long long argmax_key(float v, int id) {
  return ((unsigned long long)orderable(v) << 32) |
         (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}

// Barriers and flags at the start of the control area.
struct Ctrl {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  uint64_t* xfull;
  uint64_t* xempty;
  uint64_t* spec;      // speculative weight tiles of the first item
  uint64_t* spec_b;    // speculative activation tiles of the first item
  uint64_t* q_full;   // [kQueue] item queue: producer -> MMA issuer and epilogue
  uint64_t* q_empty;  // [kQueue]
  int* q_item;        // [kQueue]
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  uint64_t* rbar;     // single-kernel layer: router weights and gain staged
  int* ticket;        // single-kernel layer: the CTA's current ticket
};

__device__ __forceinline__ Ctrl ctrl_at(uint8_t* base, int stages) {
  Ctrl c;
  c.full = reinterpret_cast<uint64_t*>(base);
  c.empty = c.full + stages;
  c.tfull = c.empty + stages;
  c.tempty = c.tfull + 2;
  c.drain = c.tempty + 2;
  c.xfull = c.drain + 1;
  c.xempty = c.xfull + 2;
  c.spec = c.xempty + 2;
  c.spec_b = c.spec + 1;
  c.q_full = c.spec_b + 1;
  c.q_empty = c.q_full + kQueue;
  c.q_item = reinterpret_cast<int*>(c.q_empty + kQueue);
  c.tmem_slot = reinterpret_cast<uint32_t*>(c.q_item + kQueue);
  c.abort_flag = reinterpret_cast<volatile int*>(c.tmem_slot + 1);
  c.rbar = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(c.abort_flag + 2) + 7) & ~uintptr_t(7));
  c.ticket = reinterpret_cast<int*>(c.rbar + 1);
  return c;
}

__device__ __forceinline__ void init_ctrl(const Ctrl& c, int stages, uint32_t xfull_n,
                                          uint32_t xempty_n) {
  for (int s = 0; s < stages; ++s) {
    mbar_init(&c.full[s], 1);
    mbar_init(&c.empty[s], 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&c.tfull[b], 1);
    mbar_init(&c.tempty[b], 4);
    mbar_init(&c.xfull[b], xfull_n);
    mbar_init(&c.xempty[b], xempty_n);
  }
  mbar_init(c.drain, 1);
  mbar_init(c.spec, 1);
  mbar_init(c.spec_b, 1);
  for (int q = 0; q < kQueue; ++q) {
    mbar_init(&c.q_full[q], 1);
    mbar_init(&c.q_empty[q], 5);  // the MMA issuer and the four epilogue warps
  }
  *c.abort_flag = 0;
  fence_mbar_init();
}

// The MMA issuer's wind-down: everything it issued completes before TMEM is
// released.
__device__ __forceinline__ void mma_drain(const Ctrl& c) {
  umma_commit(c.drain);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(c.drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
  }
}

// The producer's wind-down after an abort: let every load already issued land.
__device__ __forceinline__ void producer_drain(const Ctrl& c, int issued, int stages) {
  for (int r = (issued > stages ? issued - stages : 0); r < issued; ++r) {
    const int s = r % stages;
    const uint32_t par = (uint32_t)((r / stages) & 1);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(&c.full[s], par) && globaltimer_ns() - t0 < kWaitLimitNs) {
    }
  }
}

// Item queue inside a CTA.  The producer pushes each item it starts (-1 when
// there are no more); the MMA issuer and every epilogue warp pop them in the
// same order.  n counts the pushes (pops) made so far.
__device__ __forceinline__ bool queue_push(const Ctrl& c, int n, int item, uint32_t* status) {
  const int q = n % kQueue;
  const uint32_t use = (uint32_t)(n / kQueue);
  if (!mbar_wait(&c.q_empty[q], (use & 1u) ^ 1u, c.abort_flag, status)) return false;
  c.q_item[q] = item;
  mbar_arrive(&c.q_full[q]);
  return true;
}

// Returns the item, or -1 at the end (also when a wait gave up).  Every lane
// of the calling warp gets the value; lane 0 releases the slot.
__device__ __forceinline__ int queue_pop(const Ctrl& c, int n, uint32_t* status, bool warp_wide) {
  const int q = n % kQueue;
  const uint32_t use = (uint32_t)(n / kQueue);
  if (!mbar_wait(&c.q_full[q], use & 1u, c.abort_flag, status)) return -1;
  const int item = c.q_item[q];
  if (warp_wide) __syncwarp();
  if (!warp_wide || (threadIdx.x & 31) == 0) mbar_arrive(&c.q_empty[q]);
  return item;
}

// Issues the MMAs of one item (kblocks stages) into TMEM columns tmem_d.
// Returns false if a wait gave up.
__device__ __forceinline__ bool mma_item(const Ctrl& c, uint8_t* stages, int stage_bytes,
                                         int n_stages, int& stage, uint32_t& phase, int kblocks,
                                         uint32_t tmem_d, uint32_t idesc, uint32_t* status) {
  for (int kb = 0; kb < kblocks; ++kb) {
    if (!mbar_wait(&c.full[stage], phase, c.abort_flag, status)) return false;
    tc_fence_after();
    const uint32_t sa = smem_u32(stages + (size_t)stage * stage_bytes);
    const uint32_t sb = sa + kStageA;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_bf16(tmem_d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), idesc,
                (kb | kk) != 0 ? 1u : 0u);
    umma_commit(&c.empty[stage]);
    if (++stage == n_stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  return true;
}

// ----------------------------------------------------------------- FFN

struct FItem {
  int down;     // 0: gate/up, 1: down
  int e, mt;    // expert, 128-row tile inside it
  int n;        // rows (tokens) of this chunk
  int row0;     // first expert-major row
  int chunk;    // global chunk id
  int a_row;    // first weight row in the tensor map
  int kblocks;
};

struct Lists {
  int* cnt;  // [nE] rows per expert
  int* cb;   // [nE+1] first chunk id per expert
  int* igu;  // [nE+1] first gate/up item per expert
  int* idn;  // [nE+1] first down item per expert
};

// Expert of list position j: the shared experts (E .. E+S-1) come first,
// then the routed experts in index order.
__device__ __forceinline__ int list_expert(const FfnParams& p, int j) {
  return j < p.S ? p.E + j : j - p.S;
}

__device__ __forceinline__ FItem decode(const FfnParams& p, const Lists& L, int nE, int n_gu,
                                        int i) {
  FItem it;
  it.down = i >= n_gu ? 1 : 0;
  const int r = it.down ? i - n_gu : i;
  const int* io = it.down ? L.idn : L.igu;
  const int mt_n = it.down ? p.mt_dn : p.mt_gu;
  // the last expert whose first item is <= r (empty experts share the start
  // of the next non-empty one and come before it)
  int lo = 0, hi = nE - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (io[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int ex = list_expert(p, lo);
  it.e = ex;
  const int q = r - io[lo];
  const int ch = q / mt_n;
  it.mt = q - ch * mt_n;
  it.n = min(p.nch, L.cnt[lo] - ch * p.nch);
  it.row0 = ex * p.T + ch * p.nch;
  it.chunk = L.cb[lo] + ch;
  it.a_row = (it.down ? p.a_base_dn : p.a_base_gu) + (ex * mt_n + it.mt) * 128;
  it.kblocks = it.down ? p.kb_dn : p.kb_gu;
  return it;
}

// Per-expert rows, chunk and item prefix sums of one expert-FFN launch, by
// one warp: 32 list positions per round, shuffle scans with a running carry,
// all counts loaded before the scans (one memory round trip).  Lists are in
// list order (shared experts first, T rows each).  An expert of c rows has
// ceil(c / nch) chunks, each with mt_gu gate/up items and mt_dn down items.
// totals: [0] gate/up items, [1] down items, [2] chunks.
__device__ __forceinline__ void build_lists(const FfnParams& p, const Lists& L, int* totals) {
  const int lane = threadIdx.x & 31, nE = p.E + p.S;
  constexpr int kMaxRounds = (kMaxExperts + 31) / 32;
  int craw[kMaxRounds];
#pragma unroll
  for (int r = 0; r < kMaxRounds; ++r) {
    const int j = r * 32 + lane;
    craw[r] = (j < p.S || j >= nE) ? p.T : __ldcg(p.cnt + (j - p.S));
  }
  int cc = 0, cg = 0, cd = 0;
#pragma unroll
  for (int r = 0; r < kMaxRounds; ++r) {
    const int e0 = r * 32;
    if (e0 >= nE) break;
    const int e = e0 + lane;
    int c = 0, ch = 0;
    if (e < nE) {
      c = min(craw[r], p.T);
      ch = (c + p.nch - 1) / p.nch;
      L.cnt[e] = c;
    }
    int ich = ch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ich, o);
      if (lane >= o) ich += a;
    }
    if (e < nE) {
      const int before = ich - ch;
      L.cb[e] = cc + before;
      L.igu[e] = cg + before * p.mt_gu;
      L.idn[e] = cd + before * p.mt_dn;
    }
    const int tot = __shfl_sync(0xffffffffu, ich, 31);
    cc += tot;
    cg += tot * p.mt_gu;
    cd += tot * p.mt_dn;
  }
  if (lane == 0) {
    L.cb[nE] = cc;
    L.igu[nE] = cg;
    L.idn[nE] = cd;
    totals[0] = cg;
    totals[1] = cd;
    totals[2] = cc;
  }
}

// Weight row (in the gate/up tensor map, layer base `base`) and first
// expert-major row of gate/up item c as the first items run: the shared
// experts' items (ceil(T / nch) chunks each) are always where this says; a
// routed expert's are when each routed expert holds one chunk (then routed
// item c is tile c % mt_gu of expert c / mt_gu).  Returns false past the
// gate/up items such a layout has, or for routed items when routed = false.
__device__ __forceinline__ bool guess_gu_item(const FfnParams& p, int c, int base, bool routed,
                                              int* a_row, int* row0) {
  const int ch_s = (p.T + p.nch - 1) / p.nch;
  const int n_sh = p.S * ch_s * p.mt_gu;
  if (c < n_sh) {
    const int s = c / (ch_s * p.mt_gu), q = c - s * ch_s * p.mt_gu;
    const int ch = q / p.mt_gu, t = q - ch * p.mt_gu;
    *a_row = base + ((p.E + s) * p.mt_gu + t) * 128;
    *row0 = (p.E + s) * p.T + ch * p.nch;
    return true;
  }
  const int cr = c - n_sh;
  if (!routed || cr >= p.E * p.mt_gu) return false;
  *a_row = base + cr * 128;
  *row0 = (cr / p.mt_gu) * p.T;
  return true;
}

// Shared memory of a routing task of the single-kernel layer, in the ring:
// [router weights: d / 64 swizzled panels] [gain d fp32] [normalised row
// d + 8 bf16] [partial logits] [logits E] [reduction 64] [rows k + S].
__host__ __device__ inline size_t route_task_bytes(int d, int E, int k, int S) {
  const int n_mt = (E + 15) / 16;
  return (size_t)(d / 64) * rs::route_wr_panel(E) + (size_t)d * 4 + ((size_t)d + 8) * 2 +
         ((size_t)rs::route_ksplit(E) * n_mt * 16 * 8 + E + 64) * 4 + (size_t)(k + S) * 4;
}

// Routing tasks of the single-kernel layer, all threads of the CTA.  Ticket
// j < n_route routes token j with the routing kernel's stages (the same bits
// as there): residual stream and RMSNorm, router logits on the tensor cores
// from the router weights staged in this CTA's ring (rbar), softmax and top-k
// with the row claims, and the token's normalised row copied into its expert
// rows.  Ticket 0 clears, after the wait, what kernels complete by then used:
// the dependency counters, the other parity's expert counters and routed-token
// counter.  Each task then publishes its token (rows, row metadata and claims
// made visible to other CTAs' loads, TMA included, then route_done) and
// claims the next ticket.  `first` is this CTA's ticket - n_route (< 0);
// returns its first expert item.
template <int SRC>
__device__ int ffn_route_tasks(const FfnParams& p, const Ctrl& C, uint8_t* ring, int first) {
  constexpr int NW = kLayerThreads / 32;
  const RouteParams& rt = p.rt;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int d = rt.d, E = rt.E, k = rt.k, S = rt.S;
  const int n_mt = (E + 15) / 16, ksplit = rs::route_ksplit(E);
  const int pitch = d + 8, cpr = d / 8;
  uint8_t* wr_s = ring;
  float* gs = reinterpret_cast<float*>(ring + (size_t)(d / 64) * rs::route_wr_panel(E));
  __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(gs + d);
  float* part = reinterpret_cast<float*>(xb + pitch);
  float* zs = part + ksplit * n_mt * 16 * 8;
  float* red = zs + E;
  int* rows = reinterpret_cast<int*>(red + 64);
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0 && rt.stamps) stamp_max(rt.stamps + 1);
  if (first == -p.n_route) {
    for (int i = tid; i < rt.n_dep_clear; i += kLayerThreads) rt.dep_clear[i] = 0;
    for (int e = tid; e < E; e += kLayerThreads) rt.cnt_other[e] = 0;
    if (tid == 0) *p.route_done_clear = 0;
  }
  mbar_wait(C.rbar, 0, C.abort_flag, rt.status);
  __syncthreads();
  const bool ok = !*C.abort_flag;  // the same for every thread (barriers below)
  while (first < 0) {
    const int t = first + p.n_route;
    for (int i = tid; i < k + S; i += kLayerThreads) rows[i] = -1;
    if (ok) rs::norm_token<SRC, NW, 16>(rt, t, gs, xb, red);  // d <= 2048
    __syncthreads();
    if (ok)
      for (int i = tid; i < S * cpr; i += kLayerThreads) {
        const int sx = i / cpr, c = i - sx * cpr;
        reinterpret_cast<uint4*>(rt.xperm + ((size_t)(E + sx) * rt.T + t) * d)[c] =
            reinterpret_cast<const uint4*>(xb)[c];
      }
    rs::router_logits<1, true>(rt, wr_s, xb, pitch, part, zs, 1, NW, ok);
    if (warp == 0 && ok) {
      if (E <= 64)
        rs::select_experts<2>(rt, zs, t, rows);
      else
        rs::select_experts<8>(rt, zs, t, rows);
    }
    __syncthreads();
    if (ok)
      for (int i = tid; i < k * cpr; i += kLayerThreads) {
        const int q = i / cpr, c = i - q * cpr;
        const int row = rows[q];
        if (row >= 0)
          reinterpret_cast<uint4*>(rt.xperm + (size_t)row * d)[c] =
              reinterpret_cast<const uint4*>(xb)[c];
      }
    __threadfence();
    fence_proxy_async_global();
    __syncthreads();
    if (tid == 0) {
      if (rt.stamps) stamp_max(rt.stamps + 2);
      atomicAdd(p.route_done, 1);
      *C.ticket = atomicAdd(p.next_item, 1) - p.n_route;
    }
    __syncthreads();
    first = *C.ticket;
  }
  // the ring goes to this CTA's TMA loads: its ordinary accesses come first
  fence_proxy_async_shared();
  __syncthreads();
  return first;
}

// kRoute: the single-kernel layer (FfnParams::n_route tokens routed here
// first, with the router map map_wr); otherwise map_wr is not read.
template <bool kRoute>
__global__ void __launch_bounds__(kRoute ? kLayerThreads : kGemmThreads, 1)
    ffn_kernel(const __grid_constant__ CUtensorMap map_gu, const __grid_constant__ CUtensorMap map_x,
               const __grid_constant__ CUtensorMap map_dn, const __grid_constant__ CUtensorMap map_a,
               const __grid_constant__ CUtensorMap map_pf, const __grid_constant__ CUtensorMap map_wr,
               const FfnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stage_bytes = kStageA + p.nch * 128;
  uint8_t* stages = smem;
  uint8_t* ctrl_base = smem + (size_t)p.stages * stage_bytes;
  const Ctrl C = ctrl_at(ctrl_base, p.stages);
  int* list_base = reinterpret_cast<int*>(ctrl_base + kCtrlBytes);
  float* xbuf = reinterpret_cast<float*>(ctrl_base + kCtrlBytes + kListBytes);
  __shared__ int s_totals[3];  // gate/up items, down items, chunks

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nE = p.E + p.S;
  Lists L;
  L.cnt = list_base;
  L.cb = L.cnt + nE;
  L.igu = L.cb + nE + 1;
  L.idn = L.igu + nE + 1;

  // Every item is claimed from one counter in increasing order, the CTA's
  // first included: its ticket, taken as the CTA starts (before the wait, the
  // counter was cleared two launches back).  So any gate/up item that a down
  // item waits for belongs to a CTA that is already running, and the kernel
  // makes progress whatever number of its CTAs the GPU runs at once.
  // Speculation: the first items run the shared experts (their rows are all
  // T tokens), then, when every routed expert holds one chunk, routed expert
  // c / mt_gu's tile c % mt_gu; so the weight tiles of the ticket's item are
  // known without the routing and start streaming before waiting for it.
  // The host guesses routed items only when every routed expert expects
  // several rows (else most of those guesses would miss and their loads
  // would only take bandwidth); shared items are always right.
  // The single-kernel layer: tickets below n_route are routing tasks, and
  // expert item i is ticket n_route + i, so every wait (an expert item's for
  // the routing, a down item's for gate/up items) is for lower tickets.
  int first = 0, guess_row = 0, guess_row0 = 0, pre = 0;
  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    first = atomicAdd(p.next_item, 1);
    if (kRoute) first -= p.n_route;
    if (first >= 0 && p.spec > 0 &&
        guess_gu_item(p, first, p.a_base_gu, p.spec > 1, &guess_row, &guess_row0))
      pre = min(p.stages, p.kb_gu);
    init_ctrl(C, p.stages, 2, 2);
    if (kRoute) {
      mbar_init(C.rbar, 1);
      fence_mbar_init();
      *C.ticket = first;
    }
    tma_prefetch_desc(&map_gu);
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_dn);
    tma_prefetch_desc(&map_a);
    if (p.pf_limit > 0) tma_prefetch_desc(&map_pf);
    if (kRoute && first < 0) {
      // a routing task: the router weights and the gain (static) into the ring
      if (p.rt.stamps) stamp_min(p.rt.stamps);
      tma_prefetch_desc(&map_wr);
      const int d = p.rt.d, E = p.rt.E;
      const size_t panel = rs::route_wr_panel(E);
      const uint64_t pol = policy_evict_last();
      mbar_arrive_expect_tx(C.rbar, (uint32_t)((size_t)E * d * 2 + (size_t)d * 4));
      for (int pn = 0; pn < d / 64; ++pn)
        tma_load_2d(stages + (size_t)pn * panel, &map_wr, C.rbar, pn * 64, p.rt.wr_row, pol);
      bulk_load(stages + (size_t)(d / 64) * panel, p.rt.gain, (uint32_t)(d * 4), C.rbar);
    }
    if (pre > 0) {
      const uint64_t pol_w = policy_evict_first();
      mbar_arrive_expect_tx(C.spec, (uint32_t)(pre * kStageA));
      for (int s = 0; s < pre; ++s)
        tma_load_2d(stages + (size_t)s * stage_bytes, &map_gu, C.spec, s * 64, guess_row, pol_w);
    }
  }
  if (warp == 1) {
    tmem_alloc(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  if constexpr (kRoute) {
    __syncthreads();
    first = *C.ticket;
    if (first < 0) {
      if (p.rt.src == kSrcEmbed)
        first = ffn_route_tasks<kSrcEmbed>(p, C, stages, first);
      else
        first = ffn_route_tasks<kSrcCombine>(p, C, stages, first);
    }
  }
  // The routing (the predecessor kernel, or this kernel's routing tasks) must
  // be complete before the counts and rows are read; dependents may start
  // once this grid is past its wait.
  pdl_wait();
  pdl_launch_dependents();
  if constexpr (kRoute) {
    if (threadIdx.x == 0) {
      const uint64_t t0 = globaltimer_ns();
      uint32_t n = 0;
      // (polled with a pause: every CTA waits here while the routing tasks'
      // own loads are in flight)
      while (ld_acquire(p.route_done) < p.n_route) {
        __nanosleep(128);
        if ((++n & 15u) == 0 && (*C.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
          if (!*C.abort_flag) {
            *C.abort_flag = 1;
            atomicOr(p.status, kErrTimeout);
          }
          break;
        }
      }
      fence_proxy_async_global();
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
  if (threadIdx.x == 0 && pre > 0) {
    // the speculated first item's activation rows load while the item lists
    // are built
    const uint64_t pol_x = policy_evict_last();
    mbar_arrive_expect_tx(C.spec_b, (uint32_t)(pre * p.nch * 128));
    for (int s = 0; s < pre; ++s)
      tma_load_2d(stages + (size_t)s * stage_bytes + kStageA, &map_x, C.spec_b, s * 64, guess_row0,
                  pol_x);
  }
  if (warp == 0) build_lists(p, L, s_totals);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *C.tmem_slot;
  const int n_gu = s_totals[0];
  const int n_items = n_gu + s_totals[1];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int i = first < n_items ? first : -1, kb = 0;
      FItem it = {};
      // announce item `item` to the MMA issuer and the epilogue, and claim
      // the item after it (the claim's result is first used when `item` is
      // fully issued, so its latency is hidden)
      int nq = 0, next_raw = 0;
      auto start_item = [&](int item) -> bool {
        if (!queue_push(C, nq++, item, p.status)) return false;
        if (item >= 0) {
          it = decode(p, L, nE, n_gu, item);
          next_raw = atomicAdd(p.next_item, 1) - (kRoute ? p.n_route : 0);
        }
        return true;
      };
      auto next_item = [&]() -> int { return next_raw < n_items ? next_raw : -1; };
      bool ok = true;
      // the speculative tiles have landed (kept on a hit, overwritten otherwise)
      if (pre > 0) ok = mbar_wait(C.spec, 0, C.abort_flag, p.status) &&
                        mbar_wait(C.spec_b, 0, C.abort_flag, p.status);
      ok = ok && start_item(i);
      const bool hit = ok && pre > 0 && i >= 0 && !it.down && it.a_row == guess_row &&
                       it.row0 == guess_row0;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      if (hit) {
        // weight and activation tiles are in place: release the stages
        for (int s = 0; s < pre; ++s) mbar_arrive(&C.full[s]);
        issued = pre;
        stage = pre;
        kb = pre;
        if (kb == it.kblocks) {
          kb = 0;
          i = next_item();
          ok = start_item(i);
        }
        if (stage == p.stages) {
          stage = 0;
          phase = 1;
        }
      }
      while (ok && i >= 0) {
        if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
          ok = false;
          break;
        }
        uint8_t* sa = stages + (size_t)stage * stage_bytes;
        uint8_t* sb = sa + kStageA;
        mbar_arrive_expect_tx(&C.full[stage], (uint32_t)(kStageA + p.nch * 128));
        tma_load_2d(sa, it.down ? &map_dn : &map_gu, &C.full[stage], kb * 64, it.a_row, pol_w);
        if (it.down && kb == 0) {
          // both SwiGLU halves of every gate/up tile of this chunk are written
          const int want = 2 * p.mt_gu;
          const uint64_t t0 = globaltimer_ns();
          uint32_t n = 0;
          while (ld_acquire(p.dep + it.chunk) < want) {
            if ((++n & 63u) == 0 && (*C.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
              if (!*C.abort_flag) {
                *C.abort_flag = 1;
                atomicOr(p.status, kErrTimeout);
              }
              ok = false;
              break;
            }
          }
          fence_proxy_async_global();
        }
        // on a failed wait the activation tiles are still loaded (stale rows),
        // so that the stage's byte count completes and the drain ends
        tma_load_2d(sb, it.down ? &map_a : &map_x, &C.full[stage], kb * 64, it.row0, pol_x);
        ++issued;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kb == it.kblocks) {
          kb = 0;
          i = next_item();
          if (!start_item(i)) ok = false;
        }
      }
      if (ok && (int)blockIdx.x < p.pf_limit) {
        // every load of this CTA is issued: pull into L2 the next kernel's
        // weight item numbered like this CTA (the first items of the next
        // kernel's CTAs together), while HBM has room (the last items of
        // other CTAs and the routing in between)
        // (the lm_head on CTA pairs: CTA c's first rows are half c % 2 of
        // the 256-row tile of item c / 2)
        const int c = (int)blockIdx.x;
        int row = p.pf_base + (p.pf_pair ? ((c >> 1) / p.pf_div) * 256 + (c & 1) * 128
                                         : (c / p.pf_div) * 128),
            row0 = 0;
        const bool known = !p.pf_items || guess_gu_item(p, (int)blockIdx.x, p.pf_base, true, &row,
                                                        &row0);
        if (known)
          for (int k = 0; k < p.pf_kb; ++k) tma_prefetch_l2_2d(&map_pf, k * 64, row);
      }
      if (!ok) producer_drain(C, issued, p.stages);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int local = 0;; ++local) {
        const int i = queue_pop(C, local, p.status, false);
        if (i < 0) break;
        const FItem it = decode(p, L, nE, n_gu, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        if (!mma_item(C, stages, stage_bytes, p.stages, stage, phase, it.kblocks,
                      tmem_base + (uint32_t)(buf * p.nch), umma_idesc_bf16(128, (uint32_t)npad),
                      p.status))
          break;
        umma_commit(&C.tfull[buf]);
      }
      mma_drain(C);
    }
  } else if (warp < 6) {
    // ------------------------------------------------ epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    uint32_t chunk_seq = 0;
    for (int local = 0;; ++local) {
      const int i = queue_pop(C, local, p.status, true);
      if (i < 0) break;
      const FItem it = decode(p, L, nE, n_gu, i);
      const int npad = (it.n + 15) & ~15;
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * p.nch);
      bool ok = true;
      if (!it.down) {
        // rows 0..63: gate, rows 64..127: up, intermediate columns mt*64 + r;
        // the "up" warps hand their values to the "gate" warps
        for (int c0 = 0; c0 < npad && ok; c0 += 16, ++chunk_seq) {
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)c0, v);
          tmem_ld_wait();
          const uint32_t xb = chunk_seq & 1u, xu = chunk_seq >> 1;
          float* U = xbuf + xb * (16 * 64);
          if (q >= 2) {
            ok = mbar_wait(&C.xempty[xb], (xu & 1u) ^ 1u, C.abort_flag, p.status);
            if (ok) {
#pragma unroll
              for (int j = 0; j < 16; ++j) U[j * 64 + (row - 64)] = __uint_as_float(v[j]);
              __syncwarp();
              if (lane == 0) mbar_arrive(&C.xfull[xb]);
            }
          } else {
            ok = mbar_wait(&C.xfull[xb], xu & 1u, C.abort_flag, p.status);
            if (ok) {
              __nv_bfloat16* out = p.a_out + (size_t)it.mt * 64 + row;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = c0 + j;
                if (n < it.n) {
                  const float g = __uint_as_float(v[j]);
                  const float u = U[j * 64 + row];
                  const float a = g / (1.0f + __expf(-g)) * u;
                  out[(size_t)(it.row0 + n) * p.I_pad] = __float2bfloat16_rn(a);
                }
              }
              __syncwarp();
              if (lane == 0) mbar_arrive(&C.xempty[xb]);
            }
          }
        }
        if (ok && q < 2) {
          // publish this half of the tile to the chunk's down items
          __threadfence();
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) atomicAdd(p.dep + it.chunk, 1);
        }
      } else {
        const int m = it.mt * 128 + row;  // output dimension
        for (int c0 = 0; c0 < npad; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)c0, v);
          tmem_ld_wait();
          if (m < p.d) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = c0 + j;
              if (n < it.n) {
                const int r = it.row0 + n;
                // (written in this launch by its routing tasks: through L2)
                const int tok = kRoute ? __ldcg(p.perm_token + r) : __ldg(p.perm_token + r);
                const int slot = kRoute ? __ldcg(p.perm_slot + r) : __ldg(p.perm_slot + r);
                const float w = kRoute ? __ldcg(p.perm_w + r) : __ldg(p.perm_w + r);
                p.y[((size_t)tok * p.kS + slot) * p.d + m] = w * __uint_as_float(v[j]);
              }
            }
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.tempty[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 2);
  // the counters this launch used are cleared by the next routing kernel (the
  // single-kernel layer: its layer's own ticket counter, by the step's final
  // kernel)
}

// End of an lm_head launch: the last CTA to finish turns the argmax keys into
// token ids.  A row is -1 when its token was invalid, when no key reached it,
// or when any CTA of this launch gave up a bounded wait (its tiles are then
// missing from the argmax, so no row of the launch can be trusted).  The last
// CTA resets the launch counters for the next launch.
__device__ __forceinline__ void lm_finish(const GemmParams& p, bool cta_aborted, int* is_last) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (cta_aborted) atomicAdd(p.aborted, 1u);
    __threadfence();
    *is_last = (atomicAdd(p.done, 1u) == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*is_last) {
    __threadfence();
    const bool any_aborted = __ldcg(p.aborted) != 0u;
    for (int t = threadIdx.x; t < p.T; t += blockDim.x) {
      const unsigned long long key = __ldcg(p.keys + t);
      const int id = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
      p.targets[t] = (any_aborted || __ldg(p.bad + t) || key == 0ull) ? -1 : id;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      *p.done = 0u;
      *p.aborted = 0u;
    }
  }
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 2);
}

// ----------------------------------------------- expert FFN, token-major
//
// The same work as ffn_kernel with the roles of the operands swapped, for
// large T (many rows per expert): a chunk of <= 128 of an expert's rows on the
// MMA's M side, 256 weight rows on N.  A gate/up item covers 128 intermediate
// units: two consecutive repacked 128-row tiles, i.e. accumulator columns
// [gate u0..u0+63 | up u0..u0+63 | gate u0+64..u0+127 | up u0+64..u0+127].  A
// down item covers 256 output dimensions.  Each epilogue thread owns one row
// (one TMEM lane), so SwiGLU pairs column c with column c + 64 in registers and
// the down epilogue looks up its row's token, slot and weight once per item:
// no exchange between warps.  Items run expert-major as in ffn_kernel and are
// claimed in the same order; a down item waits until the four epilogue warps
// of every gate/up item of its chunk have published their rows.

__device__ __forceinline__ FItem decode_tokm(const FfnParams& p, const Lists& L, int nE, int n_gu,
                                             int i) {
  FItem it;
  it.down = i >= n_gu ? 1 : 0;
  const int r = it.down ? i - n_gu : i;
  const int* io = it.down ? L.idn : L.igu;
  const int mt_n = it.down ? p.mt_dn : p.mt_gu;  // 256-row tiles per chunk
  int lo = 0, hi = nE - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (io[mid] <= r) lo = mid; else hi = mid - 1;
  }
  const int ex = list_expert(p, lo);
  it.e = ex;
  const int q = r - io[lo];
  const int ch = q / mt_n;
  it.mt = q - ch * mt_n;
  it.n = min(p.nch, L.cnt[lo] - ch * p.nch);
  it.row0 = ex * p.T + ch * p.nch;
  it.chunk = L.cb[lo] + ch;
  const int tiles = it.down ? p.tile_dn : p.tile_gu;
  it.a_row = (it.down ? p.a_base_dn : p.a_base_gu) + (ex * tiles + 2 * it.mt) * 128;
  it.kblocks = it.down ? p.kb_dn : p.kb_gu;
  return it;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    ffn_tokm_kernel(const __grid_constant__ CUtensorMap map_gu, const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_dn, const __grid_constant__ CUtensorMap map_a,
                    const FfnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr int kStageX = kTokmChunk * 128;  // 128 rows x 64 bf16
  constexpr int kStageW = 256 * 128;         // 256 weight rows x 64 bf16
  constexpr int stage_bytes = kStageX + kStageW;
  uint8_t* stages = smem;
  uint8_t* ctrl_base = smem + (size_t)p.stages * stage_bytes;
  const Ctrl C = ctrl_at(ctrl_base, p.stages);
  int* list_base = reinterpret_cast<int*>(ctrl_base + kCtrlBytes);
  __shared__ int s_totals[3];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nE = p.E + p.S;
  Lists L;
  L.cnt = list_base;
  L.cb = L.cnt + nE;
  L.igu = L.cb + nE + 1;
  L.idn = L.igu + nE + 1;

  // every item, the first included, is claimed in order (see ffn_kernel)
  int first = 0;
  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    first = atomicAdd(p.next_item, 1);
    init_ctrl(C, p.stages, 2, 2);
    tma_prefetch_desc(&map_gu);
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_dn);
    tma_prefetch_desc(&map_a);
  }
  if (warp == 1) {
    tmem_alloc(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
  if (warp == 0) build_lists(p, L, s_totals);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *C.tmem_slot;
  const int n_gu = s_totals[0];
  const int n_items = n_gu + s_totals[1];

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int i = first < n_items ? first : -1, kb = 0;
      FItem it = {};
      int nq = 0, next_raw = 0;
      auto start_item = [&](int item) -> bool {
        if (!queue_push(C, nq++, item, p.status)) return false;
        if (item >= 0) {
          it = decode_tokm(p, L, nE, n_gu, item);
          next_raw = atomicAdd(p.next_item, 1);
        }
        return true;
      };
      bool ok = start_item(i);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      while (ok && i >= 0) {
        if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
          ok = false;
          break;
        }
        uint8_t* sx = stages + (size_t)stage * stage_bytes;
        uint8_t* sw = sx + kStageX;
        mbar_arrive_expect_tx(&C.full[stage], (uint32_t)stage_bytes);
        tma_load_2d(sw, it.down ? &map_dn : &map_gu, &C.full[stage], kb * 64, it.a_row, pol_w);
        if (it.down && kb == 0) {
          // every gate/up item of this chunk is published (four warps each)
          const int want = 4 * p.mt_gu;
          const uint64_t t0 = globaltimer_ns();
          uint32_t n = 0;
          while (ld_acquire(p.dep + it.chunk) < want) {
            if ((++n & 63u) == 0 && (*C.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) {
              if (!*C.abort_flag) {
                *C.abort_flag = 1;
                atomicOr(p.status, kErrTimeout);
              }
              ok = false;
              break;
            }
          }
          fence_proxy_async_global();
        }
        // on a failed wait the rows are still loaded (stale), so that the
        // stage's byte count completes and the drain ends
        tma_load_2d(sx, it.down ? &map_a : &map_x, &C.full[stage], kb * 64, it.row0, pol_x);
        ++issued;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kb == it.kblocks) {
          kb = 0;
          i = next_raw < n_items ? next_raw : -1;
          if (!start_item(i)) ok = false;
        }
      }
      if (!ok) producer_drain(C, issued, p.stages);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const uint32_t idesc = umma_idesc_bf16(128, 256);
      for (int local = 0;; ++local) {
        const int i = queue_pop(C, local, p.status, false);
        if (i < 0) break;
        const FItem it = decode_tokm(p, L, nE, n_gu, i);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        // A = the chunk's rows (stage offset 0), B = the weight rows (kStageX on)
        if (!mma_item(C, stages, stage_bytes, p.stages, stage, phase, it.kblocks,
                      tmem_base + (uint32_t)(buf * 256), idesc, p.status))
          break;
        umma_commit(&C.tfull[buf]);
      }
      mma_drain(C);
    }
  } else {
    // ------------------------------------------------ epilogue warps 2..5
    const int q = warp & 3;      // TMEM lane quarter: rows q*32 .. q*32+31 of the chunk
    const int rr = q * 32 + lane;
    for (int local = 0;; ++local) {
      const int i = queue_pop(C, local, p.status, true);
      if (i < 0) break;
      const FItem it = decode_tokm(p, L, nE, n_gu, i);
      const int buf = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256);
      const bool valid = rr < it.n;
      const int row = it.row0 + rr;
      if (!it.down) {
        // a = bf16(silu(g) * u) for units it.mt*128 + [0, 128) of this row
        __nv_bfloat16* out = p.a_out + (size_t)row * p.I_pad + it.mt * 128;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 16) {
            uint32_t g[16], u[16];
            tmem_ld16(tb + (uint32_t)(h * 128 + c0), g);
            tmem_ld16(tb + (uint32_t)(h * 128 + 64 + c0), u);
            tmem_ld_wait();
            if (valid) {
              uint32_t pk[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
                const float a0 = g0 / (1.0f + __expf(-g0)) * __uint_as_float(u[2 * j]);
                const float a1 = g1 / (1.0f + __expf(-g1)) * __uint_as_float(u[2 * j + 1]);
                __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
                pk[j] = *reinterpret_cast<uint32_t*>(&b2);
              }
              uint4* dst = reinterpret_cast<uint4*>(out + h * 64 + c0);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
          }
        }
        // publish this warp's rows of the chunk to its down items
        __threadfence();
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) atomicAdd(p.dep + it.chunk, 1);
      } else {
        int tok = 0, slot = 0;
        float w = 0.f;
        if (valid) {
          tok = __ldg(p.perm_token + row);
          slot = __ldg(p.perm_slot + row);
          w = __ldg(p.perm_w + row);
        }
        const int m0 = it.mt * 256;  // first output dimension of this item
        float* out = p.y + ((size_t)tok * p.kS + slot) * p.d + m0;
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)c0, v);
          tmem_ld_wait();
          if (valid && m0 + c0 < p.d) {
            float4* dst = reinterpret_cast<float4*>(out + c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(w * __uint_as_float(v[4 * j]), w * __uint_as_float(v[4 * j + 1]),
                                   w * __uint_as_float(v[4 * j + 2]),
                                   w * __uint_as_float(v[4 * j + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&C.tempty[buf]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 2);
}

// ------------------------------------ lm_head, vocabulary rows on M (any T)

struct LmItem {
  int a_row, b_row, n;
};

__device__ __forceinline__ LmItem lm_item(const GemmParams& p, int i) {
  LmItem it;
  const int vt = i / p.n_chunks, c = i % p.n_chunks;
  it.a_row = vt * 128;
  it.b_row = c * p.nch_lm;
  it.n = min(p.nch_lm, p.T - c * p.nch_lm);
  return it;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap mapA,
                  const __grid_constant__ CUtensorMap mapB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stage_bytes = kStageA + p.nch * 128;
  uint8_t* stages = smem;
  uint8_t* ctrl_base = smem + (size_t)p.stages * stage_bytes;
  const Ctrl C = ctrl_at(ctrl_base, p.stages);
  float* xbuf = reinterpret_cast<float*>(ctrl_base + kCtrlBytes + kListBytes);
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_items_static;
  const bool has_work = (int)blockIdx.x < n_items;

  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    init_ctrl(C, p.stages, 4, 1);
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (has_work && warp == 1) {
    tmem_alloc(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = has_work ? *C.tmem_slot : 0u;

  if (has_work && warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    // The first ring of weight tiles does not depend on earlier kernels:
    // issue it before waiting for the final RMSNorm.
    int i = blockIdx.x, kb = 0;
    LmItem it = lm_item(p, i);
    int pre = 0;
    {
      int pi = i, pk = kb;
      LmItem pt = it;
      while (pre < p.stages && pi < n_items) {
        mbar_arrive_expect_tx(&C.full[pre], (uint32_t)(kStageA + p.nch * 128));
        tma_load_2d(stages + (size_t)pre * stage_bytes, &mapA, &C.full[pre], pk * 64, pt.a_row,
                    pol_w);
        ++pre;
        if (++pk == p.kblocks) {
          pk = 0;
          pi += gridDim.x;
          if (pi < n_items) pt = lm_item(p, pi);
        }
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (p.stamps) stamp_max(p.stamps + 1);
    for (int s = 0; s < pre; ++s) {
      tma_load_2d(stages + (size_t)s * stage_bytes + kStageA, &mapB, &C.full[s], kb * 64,
                  it.b_row, pol_x);
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = lm_item(p, i);
      }
    }
    int stage = pre, issued = pre;
    uint32_t phase = 0;
    if (stage == p.stages) {
      stage = 0;
      phase = 1;
    }
    bool ok = true;
    while (i < n_items) {
      if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + (size_t)stage * stage_bytes;
      mbar_arrive_expect_tx(&C.full[stage], (uint32_t)(kStageA + p.nch * 128));
      tma_load_2d(sa, &mapA, &C.full[stage], kb * 64, it.a_row, pol_w);
      tma_load_2d(sa + kStageA, &mapB, &C.full[stage], kb * 64, it.b_row, pol_x);
      ++issued;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = lm_item(p, i);
      }
    }
    if (!ok) producer_drain(C, issued, p.stages);
  } else {
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
    if (has_work && warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, local = 0;
      uint32_t phase = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const LmItem it = lm_item(p, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        if (!mma_item(C, stages, stage_bytes, p.stages, stage, phase, p.kblocks,
                      tmem_base + (uint32_t)(buf * p.nch), umma_idesc_bf16(128, (uint32_t)npad),
                      p.status))
          break;
        umma_commit(&C.tfull[buf]);
      }
      mma_drain(C);
    } else if (has_work && warp >= 2) {
      // ------------------------------------------------ epilogue warps 2..5
      const int q = warp & 3;
      const int row = q * 32 + lane;
      int local = 0;
      uint32_t chunk_seq = 0;
      unsigned long long* red = reinterpret_cast<unsigned long long*>(xbuf);
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const LmItem it = lm_item(p, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * p.nch);
        // greedy argmax over this tile's 128 vocabulary rows, per token column
        const int vid = it.a_row + row;
        const bool valid = vid < p.V;
        bool ok = true;
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
            if (p.logits && valid && c0 + j < it.n)
              p.logits[(size_t)(it.b_row + c0 + j) * p.V + vid] = lv;
            // warp argmax in two 32-bit reductions: the largest orderable
            // logit, then the largest inverted id among the lanes holding it
            // (= the lowest vocabulary id)
            const unsigned long long k = valid ? argmax_key(lv, vid) : 0ull;
            const uint32_t hi = (uint32_t)(k >> 32);
            const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
            const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? (uint32_t)k : 0u);
            keys[j] = ((unsigned long long)mh << 32) | ml;
          }
          ok = mbar_wait(&C.xempty[xb], (xu & 1u) ^ 1u, C.abort_flag, p.status);
          if (!ok) break;
          if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) R[(warp - 2) * 16 + j] = keys[j];
            mbar_arrive(&C.xfull[xb]);
          }
          if (warp == 2) {
            ok = mbar_wait(&C.xfull[xb], xu & 1u, C.abort_flag, p.status);
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
            if (lane == 0) mbar_arrive(&C.xempty[xb]);
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.tempty[buf]);
      }
    }
  }

  __syncthreads();
  if (has_work && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  lm_finish(p, *C.abort_flag != 0, &is_last);
}

// ------------------------------------------- lm_head, tokens on M (65..128)
//
// Tokens on the MMA's M side (a chunk of <= 128 rows; rows past the chunk's
// box are whatever the stage holds next and their accumulator lanes are never
// read), 128 vocabulary rows on N.  Each epilogue thread owns one token's TMEM
// lane, so the greedy argmax over a tile is a running maximum in registers: no
// cross-lane reduction, and one atomic per token per CTA and token chunk.
// Items run vocabulary-major (item i: tile i / n_chunks, chunk i % n_chunks),
// so the CTAs that read one vocabulary tile run side by side and share it
// through L2; when n_chunks divides the grid a CTA keeps one chunk throughout.

struct TokItem {
  int x_row, w_row, n;  // first token of the chunk, first vocabulary row, tokens in the chunk
};

__device__ __forceinline__ TokItem tok_item(const GemmParams& p, int i) {
  TokItem it;
  const int vt = i / p.n_chunks, c = i - vt * p.n_chunks;
  it.x_row = c * 128;
  it.w_row = vt * 128;
  it.n = min(128, p.T - it.x_row);
  return it;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_tokm_kernel(const __grid_constant__ CUtensorMap map_w,
                  const __grid_constant__ CUtensorMap map_x, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  // stage: [p.nch token rows x 64 columns][128 vocabulary rows x 64 columns]
  const int x_bytes = p.nch * 128;
  const int stage_bytes = x_bytes + kStageA;
  uint8_t* stages = smem;
  uint8_t* ctrl_base = smem + (size_t)p.stages * stage_bytes;
  const Ctrl C = ctrl_at(ctrl_base, p.stages);
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_items_static;
  const bool has_work = (int)blockIdx.x < n_items;

  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    init_ctrl(C, p.stages, 4, 1);
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_x);
  }
  if (has_work && warp == 1) {
    tmem_alloc(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = has_work ? *C.tmem_slot : 0u;

  if (has_work && warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    // The first ring of vocabulary tiles does not depend on earlier kernels:
    // issue it before waiting for the final RMSNorm.
    int i = blockIdx.x, kb = 0;
    TokItem it = tok_item(p, i);
    int pre = 0;
    {
      int pi = i, pk = kb;
      TokItem pt = it;
      while (pre < p.stages && pi < n_items) {
        mbar_arrive_expect_tx(&C.full[pre], (uint32_t)stage_bytes);
        tma_load_2d(stages + (size_t)pre * stage_bytes + x_bytes, &map_w, &C.full[pre], pk * 64,
                    pt.w_row, pol_w);
        ++pre;
        if (++pk == p.kblocks) {
          pk = 0;
          pi += gridDim.x;
          if (pi < n_items) pt = tok_item(p, pi);
        }
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (p.stamps) stamp_max(p.stamps + 1);
    for (int s = 0; s < pre; ++s) {
      tma_load_2d(stages + (size_t)s * stage_bytes, &map_x, &C.full[s], kb * 64, it.x_row, pol_x);
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = tok_item(p, i);
      }
    }
    int stage = pre, issued = pre;
    uint32_t phase = 0;
    if (stage == p.stages) {
      stage = 0;
      phase = 1;
    }
    bool ok = true;
    while (i < n_items) {
      if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + (size_t)stage * stage_bytes;
      mbar_arrive_expect_tx(&C.full[stage], (uint32_t)stage_bytes);
      tma_load_2d(sa + x_bytes, &map_w, &C.full[stage], kb * 64, it.w_row, pol_w);
      tma_load_2d(sa, &map_x, &C.full[stage], kb * 64, it.x_row, pol_x);
      ++issued;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = tok_item(p, i);
      }
    }
    if (!ok) producer_drain(C, issued, p.stages);
  } else {
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
    if (has_work && warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = umma_idesc_bf16(128, 128);
      int stage = 0, local = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < n_items && ok; i += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * 128);
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(&C.full[stage], phase, C.abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sx = smem_u32(stages + (size_t)stage * stage_bytes);
          const uint32_t sw = sx + (uint32_t)x_bytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem_d, umma_desc_sw128(sx + kk * 32), umma_desc_sw128(sw + kk * 32), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&C.empty[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&C.tfull[buf]);
      }
      mma_drain(C);
    } else if (has_work && warp >= 2) {
      // ------------------------------------------------ epilogue warps 2..5
      // thread = one token of the chunk (TMEM lane q*32 + lane)
      const int q = warp & 3;
      int local = 0, cur_x = -1;
      uint32_t best_u = 0u;
      int best_id = 0;
      auto flush = [&]() {
        const int tok = cur_x + q * 32 + lane;
        if (cur_x >= 0 && tok < p.T && best_u != 0u)
          atomicMax(p.keys + tok, ((unsigned long long)best_u << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (uint32_t)best_id));
        best_u = 0u;
      };
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const TokItem it = tok_item(p, i);
        if (it.x_row != cur_x) {
          flush();
          cur_x = it.x_row;
        }
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        if (q * 32 < it.n) {
          const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 128);
          const int vlim = min(128, p.V - it.w_row);  // vocabulary rows of this tile
          const int tok = it.x_row + q * 32 + lane;
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t v0[16], v1[16];
            tmem_ld16(tb + (uint32_t)c0, v0);
            tmem_ld16(tb + (uint32_t)(c0 + 16), v1);
            tmem_ld_wait();
            // increasing vocabulary order with a strict comparison keeps the
            // lowest id among equal logits
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float lv = __uint_as_float(j < 16 ? v0[j] : v1[j - 16]);
              const int col = c0 + j;
              if (col < vlim) {
                const uint32_t u = orderable(lv);
                if (u > best_u) {
                  best_u = u;
                  best_id = it.w_row + col;
                }
                if (p.logits && tok < p.T) p.logits[(size_t)tok * p.V + it.w_row + col] = lv;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.tempty[buf]);
      }
      flush();
    }
  }

  __syncthreads();
  if (has_work && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  lm_finish(p, *C.abort_flag != 0, &is_last);
}

// ------------------------------------------- lm_head on CTA pairs (T > 256)
//
// Items (a chunk of <= 256 tokens, 256 vocabulary rows), vocabulary-major
// (item i: vocabulary tile i / n_chunks, chunk i % n_chunks), in a static
// stride over the pairs (clusters of 2 CTAs), so that the pairs working at
// once share each vocabulary tile through L2.  The even CTA holds each stage's
// tokens 0..127 and vocabulary rows 0..127, the odd CTA tokens 128..255 and
// rows 128..255; one thread of the even CTA issues M = 256 (tokens), N = 256
// (vocabulary rows) MMAs (cta_group::2) over both CTAs' shared memory, and each
// CTA's TMEM receives its 128 tokens x the tile's 256 rows.  So each SM
// receives 32 KB per stage for its 128 x 256 x 64 share of the product,
// against 48 KB with one CTA per item: at large T the single-CTA form is bound
// by its SM's TMA ingest.  Each epilogue thread owns one token (one TMEM lane)
// and takes the argmax over the item's 256 rows in registers: one atomic per
// token and item, no exchange between lanes or warps.
// Handshakes: each CTA loads its halves into its own ring, and every load
// completes on the even CTA's full barrier (which expects both CTAs' bytes);
// the even CTA's commits release the stage in both CTAs (empty) and hand each
// accumulator to both CTAs' epilogues (tfull), which release it on the even
// CTA's tempty (eight arrivals).  A stage is refilled only after the commit of
// its previous use, so one use's bytes never reach the barrier's previous
// phase.  Each CTA reduces its own 128 rows per token.

struct PairItem {
  int tok_row, voc_row, v0;
};

__device__ __forceinline__ PairItem pair_item(const GemmParams& p, int i, uint32_t rank) {
  PairItem it;
  const int vt = i / p.n_chunks, c = i - vt * p.n_chunks;
  it.tok_row = c * 256 + (int)rank * 128;  // this CTA's tokens
  it.v0 = vt * 256;                        // the tile's first vocabulary row
  it.voc_row = it.v0 + (int)rank * 128;    // this CTA's half of the tile
  return it;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_pair_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr int stage_bytes = 2 * 128 * 128;  // 128 tokens + 128 vocabulary rows, x 64 bf16
  uint8_t* stages = smem;
  uint8_t* ctrl_base = smem + (size_t)p.stages * stage_bytes;
  const Ctrl C = ctrl_at(ctrl_base, p.stages);
  __shared__ int is_last;
  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int n_items = p.n_items_static;
  const bool has_work = pair < n_items;  // the same for both CTAs of a pair

  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&C.full[s], 1);
      mbar_init(&C.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&C.tfull[b], 1);
      mbar_init(&C.tempty[b], 8);  // both CTAs' four epilogue warps
    }
    mbar_init(C.drain, 1);
    *C.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (has_work && warp == 1) {
    tmem_alloc_pair(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any arrival on them
  tc_fence_after();
  const uint32_t tmem_base = has_work ? *C.tmem_slot : 0u;

  if (has_work && warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    // every load completes on the even CTA's barrier, which the even CTA's
    // producer arms with both CTAs' bytes
    const uint32_t full0 = mbar_cluster_addr(&C.full[0], 0);
    auto full_at = [&](int st) { return full0 + (uint32_t)(st * sizeof(uint64_t)); };
    // the first ring of vocabulary tiles (B, from offset 16 KB of each stage)
    // does not depend on earlier kernels
    int i = pair, kb = 0;
    PairItem it = pair_item(p, i, rank);
    int pre = 0;
    {
      int pi = i, pk = 0;
      PairItem pt = it;
      while (pre < p.stages && pi < n_items) {
        if (rank == 0) mbar_arrive_expect_tx(&C.full[pre], (uint32_t)(2 * stage_bytes));
        tma_load_2d_pair(stages + (size_t)pre * stage_bytes + kStageA, &mapA, full_at(pre),
                         pk * 64, pt.voc_row, pol_w);
        ++pre;
        if (++pk == p.kblocks) {
          pk = 0;
          pi += n_pairs;
          if (pi < n_items) pt = pair_item(p, pi, rank);
        }
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (p.stamps) stamp_max(p.stamps + 1);
    for (int s = 0; s < pre; ++s) {
      tma_load_2d_pair(stages + (size_t)s * stage_bytes, &mapB, full_at(s), kb * 64,
                       it.tok_row, pol_x);
      if (++kb == p.kblocks) {
        kb = 0;
        i += n_pairs;
        if (i < n_items) it = pair_item(p, i, rank);
      }
    }
    int stage = pre, issued = pre;
    uint32_t phase = 0;
    if (stage == p.stages) {
      stage = 0;
      phase = 1;
    }
    bool ok = true;
    while (i < n_items) {
      if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + (size_t)stage * stage_bytes;
      if (rank == 0) mbar_arrive_expect_tx(&C.full[stage], (uint32_t)(2 * stage_bytes));
      tma_load_2d_pair(sa + kStageA, &mapA, full_at(stage), kb * 64, it.voc_row, pol_w);
      tma_load_2d_pair(sa, &mapB, full_at(stage), kb * 64, it.tok_row, pol_x);
      ++issued;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++kb == p.kblocks) {
        kb = 0;
        i += n_pairs;
        if (i < n_items) it = pair_item(p, i, rank);
      }
    }
    // (the even CTA's barriers see both CTAs' loads: it alone can wait for the
    // loads in flight; the odd CTA's are covered by the even CTA's drain and
    // the cluster barrier before either exits)
    if (!ok && rank == 0) producer_drain(C, issued, p.stages);
  } else {
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
    if (has_work && warp == 1 && lane == 0 && rank == 0) {
      // ------------------------------------------------ even CTA: MMA issuer
      int stage = 0, local = 0;
      uint32_t phase = 0;
      const uint32_t idesc = umma_idesc_bf16(256, 256);
      bool ok = true;
      for (int i = pair; i < n_items && ok; i += n_pairs, ++local) {
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + (uint32_t)(buf * 256);
        for (int kb = 0; kb < p.kblocks; ++kb) {
          if (!mbar_wait(&C.full[stage], phase, C.abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + (size_t)stage * stage_bytes);
          const uint32_t sb = sa + kStageA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16_pair(tmem_d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32),
                           idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(&C.empty[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&C.tfull[buf]);
      }
      // every MMA issued completes before TMEM is released
      umma_commit_pair(C.drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(C.drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    } else if (has_work && warp >= 2) {
      // ------------------------------------------------ epilogue warps 2..5 (both CTAs)
      const int q = warp & 3;
      int local = 0;
      for (int i = pair; i < n_items; i += n_pairs, ++local) {
        const PairItem it = pair_item(p, i, rank);
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256);
        // this thread's token: the greedy argmax over the tile's 256 rows
        // (ascending ids, so a strictly larger key keeps the lowest id on ties)
        const int tok = it.tok_row + q * 32 + lane;
        uint32_t best = 0u;  // orderable image of the best logit so far
        int best_id = -1;
        const int nv = min(256, p.V - it.v0);
        for (int c0 = 0; c0 < 256; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float lv = __uint_as_float(v[j]);
            const uint32_t key = orderable(lv);
            if (c0 + j < nv && (key > best || best_id < 0)) {
              best = key;
              best_id = it.v0 + c0 + j;
            }
            if (p.logits && tok < p.T && c0 + j < nv)
              p.logits[(size_t)tok * p.V + it.v0 + c0 + j] = lv;
          }
        }
        // the key of argmax_key(): larger logit first, then lower id
        if (tok < p.T && best_id >= 0)
          atomicMax(p.keys + tok, ((unsigned long long)best << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (uint32_t)best_id));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&C.tempty[buf]);
          else
            mbar_arrive_remote(&C.tempty[buf], 0);
        }
      }
    }
  }

  __syncthreads();
  cluster_sync_all();  // the pair's MMAs, epilogues and remote arrivals are done
  if (has_work && warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
  }
  lm_finish(p, *C.abort_flag != 0, &is_last);
}

// ----------------------------------- attention projections (weight rows on M)
//
// [128 rows of one layer's packed q/k/v or W_o] x [a chunk of <= nch tokens],
// K = d.  Items run tile-major (item i: tile i / n_chunks, chunk i %
// n_chunks) in a static stride over the grid; the first ring of weight tiles
// is loaded before the wait for the previous kernel.  Each epilogue thread
// owns one weight row (one output feature) for all of the chunk's tokens.
// Mode 0: rows [q | k | v]; in q and k the two dims of a rotary pair sit in
// neighbouring rows, so the rotation of a token's pair takes one lane
// exchange; q is stored fp32, the rotated k and v as bf16 in the cache at the
// token's position.  Mode 1: h[t, row] += acc.

struct ProjItem {
  int tile, a_row, b_row, n;
};

__device__ __forceinline__ ProjItem proj_item(const ProjParams& p, int i) {
  ProjItem it;
  it.tile = i / p.n_chunks;
  const int c = i - it.tile * p.n_chunks;
  it.a_row = p.a_row0 + it.tile * 128;
  it.b_row = c * p.nch;
  it.n = min(p.nch, p.T - it.b_row);
  return it;
}

// Rows [row0, row0 + 32) of the packed q/k/v block of one warp's epilogue:
// the rows' part (0 q, 1 k, 2 v, 3 padding; the same for the whole warp since
// d is a multiple of 64), and this lane's head, head dim and rotary index.
struct QkvRow {
  int part, head, dim, freq;
  bool odd;
};

__device__ __forceinline__ QkvRow qkv_row(const ProjParams& p, int prow) {
  QkvRow r;
  r.part = prow / p.d;
  const int f = prow - r.part * p.d;
  r.head = f / p.hd;
  const int w = f - r.head * p.hd;
  r.freq = w >> 1;
  r.odd = (w & 1) != 0;
  r.dim = r.part < 2 ? r.freq + (r.odd ? (p.hd >> 1) : 0) : w;
  return r;
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    proj_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stage_bytes = kStageA + p.nch * 128;
  uint8_t* stages = smem;
  const Ctrl C = ctrl_at(smem + (size_t)p.stages * stage_bytes, p.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_items;
  const bool has_work = (int)blockIdx.x < n_items;

  if (threadIdx.x == 0) {
    stamp_min(p.stamps);
    init_ctrl(C, p.stages, 4, 1);
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (has_work && warp == 1) {
    tmem_alloc(C.tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = has_work ? *C.tmem_slot : 0u;

  if (has_work && warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const uint32_t tx = (uint32_t)(kStageA + p.nch * 128);
    int i = blockIdx.x, kb = 0;
    ProjItem it = proj_item(p, i);
    int pre = 0;
    {
      int pi = i, pk = 0;
      ProjItem pt = it;
      while (pre < p.stages && pi < n_items) {
        mbar_arrive_expect_tx(&C.full[pre], tx);
        tma_load_2d(stages + (size_t)pre * stage_bytes, &mapA, &C.full[pre], pk * 64, pt.a_row,
                    pol_w);
        ++pre;
        if (++pk == p.kblocks) {
          pk = 0;
          pi += gridDim.x;
          if (pi < n_items) pt = proj_item(p, pi);
        }
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (p.stamps) stamp_max(p.stamps + 1);
    for (int s = 0; s < pre; ++s) {
      tma_load_2d(stages + (size_t)s * stage_bytes + kStageA, &mapB, &C.full[s], kb * 64,
                  it.b_row, pol_x);
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = proj_item(p, i);
      }
    }
    int stage = pre, issued = pre;
    uint32_t phase = 0;
    if (stage == p.stages) {
      stage = 0;
      phase = 1;
    }
    bool ok = true;
    while (i < n_items) {
      if (!mbar_wait(&C.empty[stage], phase ^ 1u, C.abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint8_t* sa = stages + (size_t)stage * stage_bytes;
      mbar_arrive_expect_tx(&C.full[stage], tx);
      tma_load_2d(sa, &mapA, &C.full[stage], kb * 64, it.a_row, pol_w);
      tma_load_2d(sa + kStageA, &mapB, &C.full[stage], kb * 64, it.b_row, pol_x);
      ++issued;
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (++kb == p.kblocks) {
        kb = 0;
        i += gridDim.x;
        if (i < n_items) it = proj_item(p, i);
      }
    }
    if (!ok) producer_drain(C, issued, p.stages);
  } else {
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 1);
    if (has_work && warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0, local = 0;
      uint32_t phase = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const ProjItem it = proj_item(p, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!mbar_wait(&C.tempty[buf], (use & 1u) ^ 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        if (!mma_item(C, stages, stage_bytes, p.stages, stage, phase, p.kblocks,
                      tmem_base + (uint32_t)(buf * p.nch), umma_idesc_bf16(128, (uint32_t)npad),
                      p.status))
          break;
        umma_commit(&C.tfull[buf]);
      }
      mma_drain(C);
    } else if (has_work && warp >= 2) {
      // ------------------------------------------------ epilogue warps 2..5
      const int q = warp & 3;
      const int K1 = p.K + 1, half = p.hd >> 1;
      // The global inputs of 16 token columns, loaded ahead of use (the
      // item's first 32 while its MMAs run, then each group two ahead of the
      // one being stored).  MODE 0: each column's cache row (slot * H *
      // max_pos + position; -1 for a column past the chunk or a sequence out
      // of range) and this row's rotary (cos, sin); MODE 1: h[t, row].
      struct Cols {
        int crow[MODE == 0 ? 16 : 1];
        float2 cs[MODE == 0 ? 16 : 1];
        float hv[MODE == 1 ? 16 : 1];
      };
      auto fetch = [&](const ProjItem& it, const QkvRow& r, int prow, int c0, Cols& f) {
        if constexpr (MODE == 1) {
          if (prow < p.d) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              f.hv[j] = c0 + j < it.n ? p.h[(size_t)(it.b_row + c0 + j) * p.d + prow] : 0.f;
          }
        } else {
          if (r.part >= 3) return;
          int pos[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = it.b_row + c0 + j;
            const bool valid = c0 + j < it.n;
            const int b = valid ? t / K1 : 0;
            const int p0 = valid ? __ldg(p.positions + b) : 0;
            const bool ok = valid && p0 >= 0 && p0 <= p.max_pos - K1;
            pos[j] = ok ? p0 + (t - b * K1) : 0;
            f.crow[j] = ok ? b * p.H * p.max_pos + pos[j] : -1;
          }
          if (r.part < 2) {
#pragma unroll
            for (int j = 0; j < 16; ++j) f.cs[j] = __ldg(p.rope + (size_t)pos[j] * half + r.freq);
          }
        }
      };
      int local = 0;
      for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++local) {
        const ProjItem it = proj_item(p, i);
        const int npad = (it.n + 15) & ~15;
        const int buf = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        const int prow = it.tile * 128 + q * 32 + lane;  // row within this layer's block
        const QkvRow r = qkv_row(p, prow);
        Cols cur, nxt;
        fetch(it, r, prow, 0, cur);
        if (16 < npad) fetch(it, r, prow, 16, nxt);
        if (!mbar_wait(&C.tfull[buf], use & 1u, C.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * p.nch);
        for (int c0 = 0; c0 < npad; c0 += 16) {
          Cols nn;
          if (c0 + 32 < npad) fetch(it, r, prow, c0 + 32, nn);
          uint32_t v[16];
          tmem_ld16(tb + (uint32_t)c0, v);
          tmem_ld_wait();
          if constexpr (MODE == 1) {
            if (prow < p.d) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < it.n)
                  p.h[(size_t)(it.b_row + c0 + j) * p.d + prow] = cur.hv[j] + __uint_as_float(v[j]);
            }
          } else if (r.part < 2) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              // rotary pair (dim i, dim i + hd/2) in lanes (2i, 2i + 1)
              const float x = __uint_as_float(v[j]);
              const float y = __shfl_xor_sync(0xffffffffu, x, 1);
              const float2 cs = cur.cs[j];
              const float rot = r.odd ? y * cs.y + x * cs.x : x * cs.x - y * cs.y;
              if (c0 + j >= it.n) continue;
              const int t = it.b_row + c0 + j;
              if (r.part == 0)
                p.q[(size_t)t * p.d + r.head * p.hd + r.dim] = rot;
              else if (cur.crow[j] >= 0)
                p.kc[((size_t)cur.crow[j] + (size_t)r.head * p.max_pos) * p.hd + r.dim] =
                    __float2bfloat16_rn(rot);
            }
          } else if (r.part == 2) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (cur.crow[j] >= 0)
                p.vc[((size_t)cur.crow[j] + (size_t)r.head * p.max_pos) * p.hd + r.dim] =
                    __float2bfloat16_rn(__uint_as_float(v[j]));
          }
          cur = nxt;
          nxt = nn;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&C.tempty[buf]);
      }
    }
  }

  __syncthreads();
  if (has_work && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
  }
  if (threadIdx.x == 0 && p.stamps) stamp_max(p.stamps + 2);
}

template <typename Kern, typename... Args>
cudaError_t launch_gemm_threads(Kern kern, int grid, int threads, size_t smem, cudaStream_t s,
                                bool pdl, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
cudaError_t launch_gemm_ex(Kern kern, int grid, size_t smem, cudaStream_t s, bool pdl,
                           Args... args) {
  return launch_gemm_threads(kern, grid, kGemmThreads, smem, s, pdl, args...);
}

}  // namespace

size_t gemm_smem_bytes(int nch, int stages) {
  return 1024 /* alignment slack */ + (size_t)stages * (kStageA + (size_t)nch * 128) + kCtrlBytes +
         kListBytes + kXbufBytes;
}

int gemm_max_stages(int nch) {
  const size_t budget = 227 * 1024;
  int s = 16;
  while (s > 2 && gemm_smem_bytes(nch, s) > budget) --s;
  return s;
}

cudaError_t launch_ffn(const CUtensorMap& map_gu, const CUtensorMap& map_x,
                       const CUtensorMap& map_dn, const CUtensorMap& map_a,
                       const CUtensorMap& map_pf, const CUtensorMap& map_wr, const FfnParams& p,
                       int grid, cudaStream_t s, bool pdl) {
  if (p.n_route > 0)
    return launch_gemm_threads(ffn_kernel<true>, grid, kLayerThreads,
                               gemm_smem_bytes(p.nch, p.stages), s, pdl, map_gu, map_x, map_dn,
                               map_a, map_pf, map_wr, p);
  return launch_gemm_ex(ffn_kernel<false>, grid, gemm_smem_bytes(p.nch, p.stages), s, pdl, map_gu,
                        map_x, map_dn, map_a, map_pf, map_wr, p);
}

bool ffn_route_fits(int nch, int stages, int d, int E, int k, int S) {
  return d <= 2048 && route_task_bytes(d, E, k, S) <= (size_t)stages * (kStageA + (size_t)nch * 128);
}

size_t ffn_tokm_smem_bytes(int stages) {
  return 1024 /* alignment slack */ + (size_t)stages * (kTokmChunk * 128 + 256 * 128) +
         kCtrlBytes + kListBytes;
}

int ffn_tokm_max_stages() {
  int s = 8;
  while (s > 2 && ffn_tokm_smem_bytes(s) > 227 * 1024) --s;
  return s;
}

cudaError_t launch_ffn_tokm(const CUtensorMap& map_gu256, const CUtensorMap& map_x,
                            const CUtensorMap& map_dn256, const CUtensorMap& map_a,
                            const FfnParams& p, int grid, cudaStream_t s, bool pdl) {
  return launch_gemm_ex(ffn_tokm_kernel, grid, ffn_tokm_smem_bytes(p.stages), s, pdl, map_gu256,
                        map_x, map_dn256, map_a, p);
}

size_t proj_smem_bytes(int nch, int stages) {
  return 1024 /* alignment slack */ + (size_t)stages * (kStageA + (size_t)nch * 128) + kCtrlBytes;
}

cudaError_t launch_proj(const CUtensorMap& map_w, const CUtensorMap& map_x, const ProjParams& p,
                        int grid, cudaStream_t s, bool pdl) {
  if (p.mode == 1)
    return launch_gemm_ex(proj_kernel<1>, grid, proj_smem_bytes(p.nch, p.stages), s, pdl, map_w,
                          map_x, p);
  return launch_gemm_ex(proj_kernel<0>, grid, proj_smem_bytes(p.nch, p.stages), s, pdl, map_w,
                        map_x, p);
}

LmLayout lm_layout(int T) {
  if (T <= kLmPairMinT) return lm_layout_single(T);
  LmLayout l;
  l.tokens_on_m = false;
  l.pair = true;
  // chunks of 256 tokens, each CTA of a pair loading 128 of them
  l.n_chunks = (T + 255) / 256;
  l.nch = 128;
  l.tmem_cols = 512;  // two accumulators of 256 token columns
  l.stages = gemm_max_stages(l.nch);
  if (l.stages > 16) l.stages = 16;
  return l;
}

LmLayout lm_layout_single(int T) {
  LmLayout l;
  l.tokens_on_m = T > 64 && T <= 128;
  l.pair = false;
  if (l.tokens_on_m) {
    l.n_chunks = 1;
    l.nch = (T + 15) / 16 * 16;
    l.tmem_cols = 256;  // two accumulators of 128 vocabulary columns
  } else {
    l.n_chunks = (T + 255) / 256;
    l.nch = ((T + l.n_chunks - 1) / l.n_chunks + 15) / 16 * 16;
    l.tmem_cols = 32;  // two accumulators of nch token columns
    while (l.tmem_cols < 2 * l.nch) l.tmem_cols <<= 1;
  }
  l.stages = gemm_max_stages(l.nch);
  return l;
}

int lmhead_pair_max_clusters(int stages) {
  const size_t smem = gemm_smem_bytes(128, stages);
  if (cudaFuncSetAttribute(lmhead_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, lmhead_pair_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_lmhead_pair(const CUtensorMap& map_w, const CUtensorMap& map_x128,
                               const GemmParams& p, int pairs, cudaStream_t s, bool pdl) {
  const size_t smem = gemm_smem_bytes(128, p.stages);
  cudaError_t e = cudaFuncSetAttribute(lmhead_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, lmhead_pair_kernel, map_w, map_x128, p);
}

cudaError_t launch_lmhead(const CUtensorMap& map_w, const CUtensorMap& map_x, const GemmParams& p,
                          bool tokens_on_m, int grid, cudaStream_t s, bool pdl) {
  if (tokens_on_m)
    return launch_gemm_ex(lmhead_tokm_kernel, grid, gemm_smem_bytes(p.nch, p.stages), s, pdl,
                          map_w, map_x, p);
  return launch_gemm_ex(lmhead_kernel, grid, gemm_smem_bytes(p.nch, p.stages), s, pdl, map_w,
                        map_x, p);
}

}  // namespace mv
