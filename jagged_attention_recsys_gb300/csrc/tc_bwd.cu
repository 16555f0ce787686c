// Tensor-core jagged attention backward for sm_103a: TMA + tcgen05 + TMEM, no atomics.
//
// Method: Jagged Flash Attention bullet of the Meta GEM MFU write-up
// (piletech.kr/articles/112134, details): the backward is parallelised
// without atomic operations.  Every gradient element is produced by exactly
// one CTA in one store:
//   * row pass      rowstat[h][t] = (lse * log2 e, D = <dO, O>), head-major so
//                   a 64-row block of one head is contiguous;
//   * dK/dV pass    one item = (sequence, head, 128-key tile).  TMEM holds
//                   dK, dV and two 128-column step buffers that take, in turn,
//                   S^T = K Q^T, dP^T = V dO^T and the packed bf16 P^T and
//                   dS^T = P^T (dP^T - D) for 128-row query steps; the compute
//                   warpgroups (one key per thread) form P^T and dS^T and two
//                   issuer warps add dV += P^T dO and dK += dS^T Q with the
//                   left operand in TMEM (Q and dO read MN-major from the
//                   tiles S^T and dP^T were read K-major from);
//   * dQ pass       one item = (sequence, head, 128-row query tile).  TMEM holds
//                   dQ, two buffers of S = Q K^T and one of dP = dO V^T over
//                   128-key steps; the compute warpgroups (one row per thread)
//                   form dS into TMEM and dQ += dS K reads it from there.
// The SiLU/L variant has no lse and no D: P = SiLU(u)/L and
// dS = dP SiLU'(u)/L with u = scale s.  Masking is by subtraction as in the
// forward; masked (query, key) pairs contribute exact zeros.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "tc.h"
#include "tc_host.h"
#include "tc_ptx.cuh"
#include "feed.cuh"

namespace jfa {
namespace {
using namespace tc;

// Both passes: producer warp 0, MMA issuer warp 1, G compute warpgroups (warps
// 2 .. 4G+1), MMA issuer warp 4G+2 and, with P2 = 1, a second producer warp 4G+3.
template <int G_, int P2 = 0>
struct Groups {
  static constexpr int G = G_;
  static constexpr int kThreads = 32 * (3 + 4 * G + P2);
  static constexpr int kIssuerB = 2 + 4 * G;
  static constexpr int kProducer2 = P2 ? 3 + 4 * G : 0;
  static constexpr int HC = 128 / G;  // query columns of a step per compute warpgroup
};
constexpr int TILE = 128;  // keys per dK/dV item, rows per dQ item (MMA M)
constexpr int STEP = 128;  // query rows per dK/dV step, keys per dQ step (MMA N)
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ row pass
// rowstat[h * T + t] = (lse[t, h] * log2 e, sum_c dO[t, h, c] * O[t, h, c]).
//
// DV/8 consecutive threads own one (row, head) slice, 16 bytes of O and of dO each.
// The grid covers every slice in one pass of small CTAs, not one wave with a fixed share
// per CTA: in the backward this pass runs beside the scheduler, whose CTAs hold two SMs,
// and a fixed share per CTA then waits for those SMs (measured 0.286 against 0.218 ms
// for the causal workload's 1.33 GB).  The loop bound is CTA-uniform, so the
// width-limited shuffles always see whole warps; threads past the end load nothing and
// store nothing.
template <int DV>
__global__ void __launch_bounds__(256)
rowstat_kernel(int64_t total, int heads, const __nv_bfloat16* __restrict__ o,
               const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
               float2* __restrict__ rowstat) {
  constexpr int TPR = DV / 8;  // threads per (row, head), 8 elements each
  const int64_t rows = total * heads;
  const int64_t n = rows * TPR;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < n; base += (int64_t)gridDim.x * blockDim.x) {
    const int64_t idx = base + threadIdx.x;
    const bool valid = idx < n;
    const int64_t row = idx / TPR;
    const int part = (int)(idx % TPR);
    uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
    if (valid) {
      a = reinterpret_cast<const uint4*>(o + row * DV)[part];
      b = reinterpret_cast<const uint4*>(dout + row * DV)[part];
    }
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 x = __bfloat1622float2(pa[t]);
      const float2 y = __bfloat1622float2(pb[t]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
    if (valid && part == 0) {
      const int64_t t = row / heads;
      const int h = (int)(row - t * heads);
      rowstat[(int64_t)h * total + t] = make_float2(lse[row] * kLog2e, acc);
    }
  }
}

// Shared pieces ---------------------------------------------------------------
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* x, float f) {
  store32_bf16(dst, x, f);
}
// 32 fp32 values times f (dst 16-byte aligned)
__device__ __forceinline__ void store_row_f32(float* dst, const float* x, float f) {
#pragma unroll
  for (int t = 0; t < 32; t += 4)
    *reinterpret_cast<float4*>(dst + t) = make_float4(x[t] * f, x[t + 1] * f, x[t + 2] * f, x[t + 3] * f);
}

// =============================================================================
// dK / dV pass
// =============================================================================
// One item = (sequence, head, 128-key tile); the inner loop steps over 128 query
// rows.  TMEM holds the dK and dV accumulators and two 128-column buffers; step g
// (counted over the CTA's whole list) uses buffer X[g & 1] three times over:
//   S^T = K Q^T  ->  loaded by the compute warps  ->  dP^T = V dO^T over it  ->
//   loaded  ->  P^T and dS^T packed over it (each compute warpgroup in its own
//   HC columns: P^T in the first HC/2, dS^T in the next HC/2)  ->  read by dV
//   and dK.
// Step g+1 uses the other buffer, so nothing of step g waits for it:
//   issuer A (warp 1):        S^T(g+1) once dK(g-1) has read X[(g+1) & 1], then
//                             dV += P^T(g) dO(g)
//   issuer B (the last warp): dP^T(g+1) once S^T(g+1) has been loaded, then
//                             dK += dS^T(g) Q(g)
// The compute warps compute P^T(g) while dP^T(g) runs and find S^T(g+1) ready
// when they finish step g.  Only the step's valid query rows (rounded up to 16)
// enter the MMAs.  K and V have separate slots, so the next item's K loads as
// soon as its last S^T has been issued and its V after the last dP^T.
constexpr int KSTEP = 128;  // query rows per dK/dV step

template <int DQK, int DV>
struct KvLayout {
  static constexpr int NQ = DQK == 128 ? 3 : 4;             // Q stages
  static constexpr int NO = DQK == 64 && DV == 64 ? 4 : 2;  // dO stages, with the row terms
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;  // 128 keys
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;  // 128 rows
  static constexpr uint32_t O_BYTES = DV / 64 * 16384;
  static constexpr uint32_t RS_BYTES = 2 * KSTEP * 4;    // -lse log2 e and -D of 128 rows
  // in front of the tiles: mbarriers, TMEM slot, abort flag (640 bytes), the work item
  // ring, row terms
  static constexpr uint32_t FEED_OFF = 640;
  static constexpr uint32_t RS_OFF = FEED_OFF + kFeedSlots * sizeof(WorkItem);
  static constexpr uint32_t SMALL = RS_OFF + NO * RS_BYTES;
  static constexpr uint32_t TILE0 = (SMALL + 1023) / 1024 * 1024;  // for a 1 KB-aligned base
  static constexpr uint32_t K_OFF = 0;  // offsets from the 1 KB-aligned tile base
  static constexpr uint32_t V_OFF = K_OFF + K_BYTES;
  static constexpr uint32_t Q_OFF = V_OFF + V_BYTES;
  static constexpr uint32_t O_OFF = Q_OFF + NQ * Q_BYTES;
  static constexpr uint32_t TILES = O_OFF + NO * O_BYTES;
  static constexpr uint32_t SMEM = TILE0 + TILES;
  static_assert(SMEM <= 232448u && SMEM >= 122880u, "one CTA per SM within its shared memory");
};

enum : uint32_t {
  KV_KFULL = 0, KV_KEMPTY = 1, KV_VFULL = 2, KV_VEMPTY = 3, KV_QFULL = 4, KV_QEMPTY = 8,
  KV_OFULL = 12, KV_OEMPTY = 16, KV_RSFULL = 20, KV_SFULL = 24, KV_SEMPTY = 26, KV_DPFULL = 28,
  KV_PDSFULL = 30, KV_KDONE = 32, KV_ACCFULL = 34, KV_ACCEMPTY = 35, KV_DRAIN = 36, KV_KREADY = 38,
  KV_QREADY = 39, KV_FEEDFULL = 43, KV_FEEDEMPTY = 51, KV_COUNT = 59
};
static_assert(8 * KV_COUNT + 8 <= 640, "mbarriers, TMEM slot and abort flag in front of the item ring");

// bf16 pair (low, high) of a packed word to two floats, exactly
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// Walks the steps of a CTA's items in order (items without steps are skipped):
// item w, local step j, global step g, Q/dO stage counter q, item counter kv.  The
// items come from the CTA's feed; `arrive` marks the cursor that releases each feed
// slot (an issuer's lagging cursor).  Becomes invalid at the end of the list or when a
// bounded wait gave up.
template <bool DYN>
struct StepCursor {
  Feed<DYN> feed;
  volatile int* abort;
  int* status;
  WorkItem w;
  int j;
  uint32_t g, q, kv;
  bool valid, arrive;
  __device__ void next_item() { valid = feed.take(w, true, arrive, abort, status); }
  __device__ void skip_empty() {
    while (valid && w.cost == 0) next_item();
  }
  __device__ void init(const FeedRing& r, const WorkItem* l, const int* ctr, int n, bool arr,
                       volatile int* ab, int* st) {
    feed.init(r, l, ctr, n);
    abort = ab;
    status = st;
    arrive = arr;
    j = 0;
    g = q = kv = 0;
    next_item();
    skip_empty();
  }
  __device__ void advance() {
    ++g;
    ++q;
    if (++j < w.cost) return;
    j = 0;
    ++kv;
    next_item();
    skip_empty();
  }
  __device__ bool last() const { return j == w.cost - 1; }
  // valid query rows of this step, rounded up to 16 (MMA N of S^T / dP^T)
  template <bool CAUSAL>
  __device__ int n16() const {
    const int qs0 = CAUSAL ? (w.tile * TILE) / KSTEP : 0;
    const int v = min(KSTEP, w.lq - (qs0 + j) * KSTEP);
    return (max(v, 1) + 15) & ~15;
  }
};

// dK/dV: the SiLU/L variant has about three times the per-element work of the softmax
// one (two MUFU operations and twice the FMAs per key and query), and its compute
// warps, not the tensor pipe, set the pace; four groups of 32 query columns hide that
// work's latencies with twice the warps.  Softmax keeps two groups of 64 columns,
// which leave its issuers' warp schedulers less busy.
template <int ACT>
using KvGroups = Groups<ACT == kActSoftmax ? 2 : 4, 1>;
// dQ: two groups of 64 key columns for softmax, four of 32 for SiLU/L (its compute
// warps set the pace once the issuers run converged: 3.95 -> 3.80 ms on the GDPA
// workload), and two producers: Q and K in warp 0, dO and V in the last warp, so that
// a V load never queues behind a K load that waits for its slot (K(j+2) takes the slot
// of K(j-1), which dQ(j-1) frees late in the step, while dP(j+1) wants V(j+1) early).
template <int ACT>
using QGroups = Groups<ACT == kActSoftmax ? 2 : 4, 1>;

// Rotary embedding (BlockAttention), done by the compute warps: the next non-empty item
// of the CTA's list (index rot_next, advanced) has its tiles rotated once they have
// landed, and signalled ready (one arrival per compute warp).  rot_cnt counts the items
// rotated, which fixes their ring stages (every item of the rotary kernels has one step).
// Warp wi of the nw compute warps takes its share of the rows.  False if a wait gave up.
template <int DQK, int NQ, bool CAUSAL, class L>
__device__ __forceinline__ bool kv_rotate_next(int& rot_next, uint32_t& rot_cnt, const WorkItem* list,
                                               int n_items, uint32_t raw, uint32_t sb, const Problem& p,
                                               int wi, int nw, int lane, volatile int* abort,
                                               int* status) {
  auto bar = [&](uint32_t i) { return raw + 8u * i; };
  while (rot_next < n_items && load_item(list, rot_next).cost == 0) rot_next += gridDim.x;
  if (rot_next >= n_items) return true;
  const WorkItem x = load_item(list, rot_next);
  rot_next += gridDim.x;
  const int key0 = x.tile * TILE, row0 = (CAUSAL ? key0 / KSTEP : 0) * KSTEP;
  const uint32_t qs = rot_cnt % NQ;
  if (!mbar_wait(bar(KV_KFULL), rot_cnt & 1, abort, status) ||
      !mbar_wait(bar(KV_QFULL + qs), (rot_cnt / NQ) & 1, abort, status))
    return false;
  if (key0 == row0) {  // one step: the K and Q tiles start at the same position
    rope_rotate_pair_share<DQK>(sb + L::K_OFF, rope_rows(key0, x.lk, p.rope_npos), sb + L::Q_OFF + qs * L::Q_BYTES,
                                rope_rows(row0, x.lq, p.rope_npos), key0, p.rope, wi, nw, lane);
  } else {
    rope_rotate_pair_share<DQK>(sb + L::K_OFF, rope_rows(key0, x.lk, p.rope_npos), 0, 0, key0, p.rope, wi, nw,
                                lane);
    rope_rotate_pair_share<DQK>(sb + L::Q_OFF + qs * L::Q_BYTES, rope_rows(row0, x.lq, p.rope_npos), 0, 0, row0,
                                p.rope, wi, nw, lane);
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(bar(KV_KREADY));
    mbar_arrive(bar(KV_QREADY + qs));
  }
  ++rot_cnt;
  return true;
}

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE>
__global__ void __launch_bounds__(KvGroups<ACT>::kThreads, 1)
tc_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
               const Problem p, const float2* __restrict__ rowstat,
               __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, WsHeader* hdr,
               const WorkItem* __restrict__ list) {
  using L = KvLayout<DQK, DV>;
  using Gr = KvGroups<ACT>;
  constexpr int NQ = L::NQ, NO = L::NO;
  constexpr int HC = Gr::HC;  // query columns per compute warpgroup
  static_assert(HC * Gr::G == KSTEP && HC % 32 == 0, "the compute warpgroups split a step's query rows");
  constexpr uint32_t kCompute = 32 * 4 * Gr::G;  // compute threads
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + L::SMALL + 1023u) & ~1023u;  // 128-byte swizzled tiles: 1 KB aligned
  int* status = &hdr->status;
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  if (sb - raw + L::TILES > dyn_bytes) {  // same for every thread: nothing has started yet
    if (threadIdx.x == 0) atomicExch(status, (int)JFA_ERR_CUDA);
    return;
  }
  auto bar = [&](uint32_t i) { return raw + 8u * i; };
  uint32_t* tmem_slot = (uint32_t*)(smem_raw + 8 * KV_COUNT);
  volatile int* abort = (volatile int*)(smem_raw + 8 * KV_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_k;

  if (threadIdx.x == 0) {
    mbar_init(bar(KV_KFULL), 1);
    mbar_init(bar(KV_KEMPTY), 1);
    mbar_init(bar(KV_VFULL), 1);
    mbar_init(bar(KV_VEMPTY), 1);
    // Q / dO stages and the accumulators are released by both issuers
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar(KV_QFULL + s), 1);
      mbar_init(bar(KV_QEMPTY + s), 1);  // dK's commit (see the issuers)
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(bar(KV_OFULL + s), 1);
      mbar_init(bar(KV_OEMPTY + s), 1);  // dV's commit
      mbar_init(bar(KV_RSFULL + s), 32);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(KV_SFULL + s), 1);
      mbar_init(bar(KV_SEMPTY + s), kCompute);
      mbar_init(bar(KV_DPFULL + s), 1);
      mbar_init(bar(KV_PDSFULL + s), kCompute);
      mbar_init(bar(KV_KDONE + s), 1);
    }
    mbar_init(bar(KV_ACCFULL), 2);
    mbar_init(bar(KV_ACCEMPTY), kCompute);
    mbar_init(bar(KV_DRAIN), 1);      // issuer A's exit drain
    mbar_init(bar(KV_DRAIN + 1), 1);  // issuer B's exit drain
    // rotated K and Q tiles (rotary embedding): one arrival per compute warp
    mbar_init(bar(KV_KREADY), kCompute / 32);
    for (int s = 0; s < NQ; ++s) mbar_init(bar(KV_QREADY + s), kCompute / 32);
    // work item ring: warp 0 claims; the second producer, both issuers and every
    // compute warp read
    for (int s = 0; s < kFeedSlots; ++s) {
      mbar_init(bar(KV_FEEDFULL + s), 1);
      mbar_init(bar(KV_FEEDEMPTY + s), 3 + kCompute / 32);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: dK [0,128), dV [128,256), step buffers X0 [256,384), X1 [384,512)
  constexpr uint32_t T_DK = 0, T_DV = 128, T_X = 256;
  // SiLU/L items may be claimed from the launch's counter as CTAs become free (the
  // scheduler decides per list).  The softmax kernels keep the fixed assignment: their
  // workloads' items are short, and the feed's registers would cost them spills; so do
  // the rotary kernels, whose compute warps look ahead in the list.
  constexpr bool kDyn = !ROPE && ACT != kActSoftmax;
  static_assert(KV_FEEDEMPTY == KV_FEEDFULL + kFeedSlots, "feed ring barriers");
  const FeedRing ring{bar(KV_FEEDFULL), raw + L::FEED_OFF};
  int* const claim_ctr = &hdr->claim[kClaimDkdv];

  // Rotary embedding of Q and K (BlockAttention): the compute warps rotate each item's K
  // and Q tiles in shared memory once they have landed and signal them ready; issuer A
  // waits for that instead of the loads.  Its items are blocks of at most 64 rows, so
  // each has exactly one step; the compute warps rotate the next item's tiles right after
  // the current item's step, while its gradient products run.
  constexpr bool rope = ROPE;
  if (warp == 0) {
    // ------------------------------------------------------------ producer: K and Q
    // Two producers, so that neither ring waits behind a load of the other: warp 0
    // loads each item's K and every step's Q, the last warp its V and every step's
    // dO with the step's row terms.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
      uint32_t kv_it = 0, q_it = 0;
      bool ok = true;
      FeedClaimer<kDyn> claimer;
      claimer.init(ring, list, claim_ctr, n_items);
      WorkItem w;
      while (ok && claimer.claim(w, abort, status)) {
        const int n = w.cost;
        if (n == 0) continue;
        const int h = w.h, key0 = w.tile * TILE;
        const int64_t q0 = w.q0, k0 = w.k0;
        const int qs0 = CAUSAL ? key0 / KSTEP : 0;
        if (!mbar_wait(bar(KV_KEMPTY), (kv_it & 1) ^ 1, abort, status)) break;
        ++kv_it;
        mbar_expect_tx(bar(KV_KFULL), L::K_BYTES);
#pragma unroll
        for (int a = 0; a < DQK / 64; ++a)
          tma_load_2d(sb + L::K_OFF + a * 16384, &tm_k, h * DQK + a * 64, (int32_t)(k0 + key0), bar(KV_KFULL));
        for (int j = 0; j < n; ++j, ++q_it) {
          const uint32_t st = q_it % NQ;
          if (!mbar_wait(bar(KV_QEMPTY + st), ((q_it / NQ) & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(KV_QFULL + st), L::Q_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::Q_OFF + st * L::Q_BYTES + a * 16384, &tm_q, h * DQK + a * 64,
                        (int32_t)(q0 + (qs0 + j) * KSTEP), bar(KV_QFULL + st));
        }
      }
      // every load issued has landed before the CTA leaves (also after giving up)
      drain_ring(bar(KV_KFULL), 1, kv_it, status);
      drain_ring(bar(KV_QFULL), NQ, q_it, status);
    }
    __syncwarp();
  } else if (warp == Gr::kProducer2) {
    // ------------------------------------------------------------ producer: V, dO, row terms
    if (lane == 0) {
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
    }
    uint32_t kv_it = 0, q_it = 0;
    bool ok = true;
    Feed<kDyn> feed;
    feed.init(ring, list, claim_ctr, n_items);
    WorkItem w;
    while (ok && feed.take(w, true, true, abort, status)) {
      const int n = w.cost;
      if (n == 0) continue;
      const int h = w.h, key0 = w.tile * TILE;
      const int64_t q0 = w.q0, k0 = w.k0;
      const int Lq = w.lq;
      const int qs0 = CAUSAL ? key0 / KSTEP : 0;
      if (lane == 0) {
        ok = mbar_wait(bar(KV_VEMPTY), (kv_it & 1) ^ 1, abort, status);
        if (ok) {
          mbar_expect_tx(bar(KV_VFULL), L::V_BYTES);
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::V_OFF + a * 16384, &tm_v, h * DV + a * 64, (int32_t)(k0 + key0), bar(KV_VFULL));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) { ok = false; break; }
      ++kv_it;
      for (int j = 0; j < n && ok; ++j, ++q_it) {
        const int i0 = (qs0 + j) * KSTEP;
        // row terms of this step: issue the global loads before waiting for the stage
        float2 rv[KSTEP / 32];
#pragma unroll
        for (int t = 0; t < KSTEP / 32; ++t) {
          const int c = lane + 32 * t;
          rv[t] = make_float2(0.f, 0.f);
          if (ACT == kActSoftmax && i0 + c < Lq) rv[t] = rowstat[(int64_t)h * p.total_q + q0 + i0 + c];
        }
        const uint32_t so = q_it % NO;
        ok = mbar_wait(bar(KV_OEMPTY + so), ((q_it / NO) & 1) ^ 1, abort, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(bar(KV_OFULL + so), L::O_BYTES);
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::O_OFF + so * L::O_BYTES + a * 16384, &tm_do, h * DV + a * 64,
                        (int32_t)(q0 + i0), bar(KV_OFULL + so));
        }
        // the row terms share the dO stage: it is released by dV(g), which waits for
        // the compute warps to finish dS^T(g)
        float* rs = reinterpret_cast<float*>(smem_raw + L::RS_OFF + so * L::RS_BYTES);
#pragma unroll
        for (int t = 0; t < KSTEP / 32; ++t) {
          rs[lane + 32 * t] = -rv[t].x;
          rs[KSTEP + lane + 32 * t] = -rv[t].y;
        }
        mbar_arrive(bar(KV_RSFULL + so));
      }
    }
    if (lane == 0) {  // every load issued has landed before the CTA leaves
      drain_ring(bar(KV_VFULL), 1, kv_it, status);
      drain_ring(bar(KV_OFULL), NO, q_it, status);
    }
    __syncwarp();
  } else if (warp == 1 || warp == Gr::kIssuerB) {
    // ------------------------------------------------------------ MMA issuers
    // An MMA issue occupies the issuing thread for most of the MMA's duration and
    // the tensor pipe queues only a few, so the products come from two threads.
    // Each commit covers only its own thread's MMAs.  The accumulators, read by both
    // chains, take one commit from each.  A Q stage is read by S^T(g) (issuer A) and
    // dK(g) (issuer B), a dO stage by dP^T(g) (B) and dV(g) (A); each is released by
    // the later product's commit alone: dK(g) is issued only after the compute warps
    // formed dS^T(g), which they do after loading S^T(g) (so S^T(g) has completed), and
    // dV(g) likewise after dP^T(g).
    {  // the whole warp runs the issuer loop; one elected lane issues
      const bool chain_p = warp == 1;
      constexpr uint32_t idesc_dv = idesc_bf16(TILE, DV, 0, 1);
      constexpr uint32_t idesc_dk = idesc_bf16(TILE, DQK, 0, 1);
      uint32_t a_it = 0;
      bool ok = true;
      // Score product of step c into X[g & 1]: S^T (chain P) once dK(g-2) has read
      // the buffer (dV(g-2) was issued earlier by this thread); dP^T (chain dS)
      // once the compute warps have loaded S^T(g) from it.
      auto issue_score = [&](const StepCursor<kDyn>& c) {
        const uint32_t b = c.g & 1;
        const uint32_t st = chain_p ? c.q % NQ : c.q % NO;
        const uint32_t ph = chain_p ? (c.q / NQ) & 1 : (c.q / NO) & 1;
        const uint32_t kbar = chain_p ? (rope ? KV_KREADY : KV_KFULL) : KV_VFULL;
        const uint32_t qbar = chain_p ? (rope ? KV_QREADY : KV_QFULL) : KV_OFULL;
        if ((c.j == 0 && !mbar_wait(bar(kbar), c.kv & 1, abort, status)) ||
            !mbar_wait(bar(qbar + st), ph, abort, status) ||
            (chain_p && !mbar_wait(bar(KV_KDONE + b), ((c.g >> 1) & 1) ^ 1, abort, status)) ||
            (!chain_p && !mbar_wait(bar(KV_SEMPTY + b), (c.g >> 1) & 1, abort, status)))
          return false;
        __syncwarp();  // converged for elect.sync
        tc_fence_after();
        const uint32_t a_tile = sb + (chain_p ? L::K_OFF : L::V_OFF);
        const uint32_t b_tile = chain_p ? sb + L::Q_OFF + st * L::Q_BYTES : sb + L::O_OFF + st * L::O_BYTES;
        const uint64_t da = sw128_desc(a_tile, 16, 1024), db = sw128_desc(b_tile, 16, 1024);
        const uint32_t idesc = idesc_bf16(TILE, c.template n16<CAUSAL>(), 0, 0);
        const uint32_t d_tm = tmem + T_X + b * 128;
#pragma unroll
        for (int kk = 0; kk < (chain_p ? DQK : DV) / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;  // descriptor units
          mma_bf16(d_tm, da + off, db + off, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar((chain_p ? KV_SFULL : KV_DPFULL) + b));
        if (c.last()) mma_commit(bar(chain_p ? KV_KEMPTY : KV_VEMPTY));  // last use of this tile
        return true;
      };
      StepCursor<kDyn> cs, cg;  // cs: next score product (one step ahead); cg: gradient product
      cs.init(ring, list, claim_ctr, n_items, false, abort, status);
      cg.init(ring, list, claim_ctr, n_items, true, abort, status);
      if (cs.valid) {
        ok = issue_score(cs);
        cs.advance();
      }
      while (ok && cg.valid) {
        // Issuer A issues S^T(g+1) before dV(g): the compute warps want it next.
        // Issuer B issues dK(g) before dP^T(g+1) (dP^T(g+1) waits for S^T(g+1) to be
        // loaded, and S^T(g+1) waits for dK(g-1)), except at an item's first step:
        // there dK(g) waits for the previous item's epilogue, which the compute warps
        // run after this step, so dP^T(g+1) goes first.
        const bool score_first = chain_p || cg.j == 0;
        if (score_first && cs.valid) {
          if (!(ok = issue_score(cs))) break;
          cs.advance();
        }
        // chain P: dV += P^T(g) dO(g); chain dS: dK += dS^T(g) Q(g)
        const uint32_t b = cg.g & 1;
        const uint32_t sq = cg.q % NQ, so = cg.q % NO;
        if (!mbar_wait(bar(KV_PDSFULL + b), (cg.g >> 1) & 1, abort, status) ||
            (cg.j == 0 && !mbar_wait(bar(KV_ACCEMPTY), (a_it & 1) ^ 1, abort, status))) {
          ok = false;
          break;
        }
        __syncwarp();  // converged for elect.sync
        tc_fence_after();
        const int ksteps = cg.template n16<CAUSAL>() >> 4;
        // P^T or dS^T: each group's HC columns hold P^T of its HC queries in the first
        // HC/2 (16-query K-steps of 8 columns) and dS^T in the next HC/2
        const uint32_t xb = tmem + T_X + b * 128 + (chain_p ? 0 : HC / 2);
        const uint64_t db = sw128_desc(chain_p ? sb + L::O_OFF + so * L::O_BYTES : sb + L::Q_OFF + sq * L::Q_BYTES,
                                       16384, 1024);
#pragma unroll
        for (int kk = 0; kk < KSTEP / 16; ++kk)
          if (kk < ksteps)
            mma_bf16_tmem_a(tmem + (chain_p ? T_DV : T_DK), xb + (kk / (HC / 16)) * HC + (kk % (HC / 16)) * 8,
                            db + ((kk * 2048) >> 4), chain_p ? idesc_dv : idesc_dk,
                            (cg.j > 0 || kk > 0) ? 1u : 0u);
        if (chain_p) {
          mma_commit(bar(KV_OEMPTY + so));
        } else {
          mma_commit(bar(KV_KDONE + b));
          mma_commit(bar(KV_QEMPTY + sq));
        }
        if (cg.last()) {
          mma_commit(bar(KV_ACCFULL));
          ++a_it;
        }
        if (!score_first && cs.valid) {
          if (!(ok = issue_score(cs))) break;
          cs.advance();
        }
        cg.advance();
      }
      __syncwarp();
      mma_drain(bar(KV_DRAIN + (chain_p ? 0 : 1)), status);  // every MMA issued has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warpgroups
    // Each group of four consecutive warps covers all 128 keys (TMEM lanes) and
    // handles query columns [HC grp, HC grp + HC) of every step.  In the epilogue
    // two groups store the two halves of dK and of dV each; four groups store one
    // half of dK (groups 0, 1) or of dV (groups 2, 3) each.  Each group reads and
    // writes only inside its own columns.
    const int grp = (warp - 2) >> 2;
    const int r = 32 * (warp & 3) + lane;  // key of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    const float2 cc = make_float2(c_score, c_score);
    const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
    const float2 one = make_float2(1.f, 1.f);
    uint32_t q_it = 0, s_it = 0, a_it = 0;
    bool ok = true;
    // The epilogue of an item (dK, dV from TMEM to HBM) runs after the next item's
    // first step, when its last dV / dK products have long completed; the next
    // item's first dV / dK wait for it (ACCEMPTY).
    bool pend = false, pend_key_ok = false;
    int64_t pend_krow = 0;
    int pend_kpos = 0;  // key index inside its sequence: the rotary embedding's position
    auto epilogue = [&]() -> bool {
      if (!mbar_wait(bar(KV_ACCFULL), a_it & 1, abort, status)) return false;
      ++a_it;
      tc_fence_after();
      if constexpr (Gr::G == 4) {
        // one half of dK or of dV, through an array of exactly its columns
        // (four groups serve SiLU/L only, which has no rotary variant)
        auto drain = [&](auto cols, uint32_t t_acc, __nv_bfloat16* dst, float f) {
          constexpr int NC = decltype(cols)::value;
          float x[NC];
#pragma unroll
          for (int c = 0; c < NC / 32; ++c) tmem_ld32(t_acc + 32 * c, x + 32 * c);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(KV_ACCEMPTY));
          if (pend_key_ok) {
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) store_row_bf16(dst + 32 * c, x + 32 * c, f);
          }
        };
        if (grp >= 2)
          drain(std::integral_constant<int, DV / 2>{}, tmem + lane_base + T_DV + (grp & 1) * (DV / 2),
                dv + pend_krow * DV + (grp & 1) * (DV / 2), 1.f);
        else
          drain(std::integral_constant<int, DQK / 2>{}, tmem + lane_base + T_DK + (grp & 1) * (DQK / 2),
                dk + pend_krow * DQK + (grp & 1) * (DQK / 2),
                ACT == kActSoftmax ? p.scale : 0.5f * p.scale);  // SiLU/L: dS^T was doubled
      } else {
        // half grp of dK and half grp of dV
        float x[DQK / 2], y[DV / 2];
#pragma unroll
        for (int c = 0; c < DQK / 64; ++c) tmem_ld32(tmem + lane_base + T_DK + grp * (DQK / 2) + 32 * c, x + 32 * c);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c) tmem_ld32(tmem + lane_base + T_DV + grp * (DV / 2) + 32 * c, y + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(KV_ACCEMPTY));
        // dK with the rotary embedding: the gradient of the rotated keys turned back
        if (rope && pend_key_ok && pend_kpos < p.rope_npos)
          rope_unrotate_row<DQK / 2>(x, grp * (DQK / 2), pend_kpos, DQK, p.rope);
        if (pend_key_ok) {
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c)
            store_row_bf16(dk + pend_krow * DQK + grp * (DQK / 2) + 32 * c, x + 32 * c, p.scale);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            store_row_bf16(dv + pend_krow * DV + grp * (DV / 2) + 32 * c, y + 32 * c, 1.f);
        }
      }
      pend = false;
      return true;
    };
    // rotary embedding: the next non-empty item to rotate (list index) and the count of
    // items rotated so far (which fixes its K and Q stages)
    int rot_next = blockIdx.x;
    uint32_t rot_cnt = 0;
    if constexpr (ROPE) {
      if (!kv_rotate_next<DQK, NQ, CAUSAL, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp - 2,
                                               kCompute / 32, lane, abort, status))
        ok = false;
    }
    Feed<kDyn> feed;
    feed.init(ring, list, claim_ctr, n_items);
    WorkItem w;
    while (ok && feed.take(w, true, true, abort, status)) {
      const int n = w.cost;
      const int h = w.h, key0 = w.tile * TILE;
      const int64_t k0 = w.k0;
      const int Lq = w.lq, Lk = w.lk;
      const int j = key0 + r;  // key index inside the sequence
      if (rope && n > 1) {  // the rotary kernels take items of one step only
        if (lane == 0) atomicExch(status, (int)JFA_ERR_UNSUPPORTED);
        *abort = 1;
        ok = false;
        break;
      }
      const float inv_len = 1.0f / (float)max(Lq, 1);
      const float2 il = make_float2(inv_len, inv_len);
      const int qs0 = CAUSAL ? key0 / KSTEP : 0;
      for (int step = 0; step < n; ++step, ++q_it, ++s_it) {
        const uint32_t b = s_it & 1;
        const uint32_t x_tm = tmem + lane_base + T_X + b * 128 + grp * HC;  // this group's columns
        const int i0 = (qs0 + step) * KSTEP + grp * HC;
        if (!mbar_wait(bar(KV_SFULL + b), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        if (Lq - i0 <= 0) {
          // No valid query among this group's columns: the step's MMAs stop before
          // them (N and K are trimmed to the valid rows), so only the arrivals remain.
          mbar_arrive(bar(KV_SEMPTY + b));
          if (!mbar_wait(bar(KV_DPFULL + b), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
          mbar_arrive(bar(KV_PDSFULL + b));
          if (pend && !epilogue()) { ok = false; break; }
          if constexpr (ROPE) {  // the next item's K and Q tiles
            if (!kv_rotate_next<DQK, NQ, CAUSAL, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp - 2,
                                                     kCompute / 32, lane, abort, status)) {
              ok = false;
              break;
            }
          }
          continue;
        }
        float sv[HC];
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld32(x_tm + 32 * c, sv + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(KV_SEMPTY + b));  // dP^T(s_it) may overwrite the buffer
        const uint32_t st = q_it % NO;
        if (!mbar_wait(bar(KV_RSFULL + st), (q_it / NO) & 1, abort, status)) { ok = false; break; }
        const float* rs = reinterpret_cast<const float*>(smem_raw + L::RS_OFF + st * L::RS_BYTES) + grp * HC;
        // valid queries of this group's columns for key j: i < Lq and (causal) i >= j
        const int lo = CAUSAL ? j - i0 : 0;
        int hi = j < Lk ? Lq - i0 : 0;
        if (p.block_mask > 0 && (j ^ i0) >= p.block_mask) hi = 0;  // another block's queries
        if (lo > 0 || hi < HC) {
#pragma unroll
          for (int c = 0; c < HC; ++c) sv[c] -= (c >= lo && c < hi) ? 0.f : shift_raw;
        }
        // P^T (and, for SiLU/L, the factor SiLU'(u)/L used by dS^T), packed bf16
        uint32_t pk[HC / 2], fk[ACT == kActSoftmax ? 1 : HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          const float2 x = make_float2(sv[c], sv[c + 1]);
          float2 pv;
          if (ACT == kActSoftmax) {
            const float2 e = ffma2(x, cc, *reinterpret_cast<const float2*>(rs + c));
            pv = make_float2(ex2(e.x), ex2(e.y));
          } else {
            // u = s c, h = u/2, t = tanh h: P = h (1+t)/L, SiLU'(u)/L = (1+t)/(2L) (1 + h - h t).
            // The factor formed here is twice SiLU'(u)/L, sharing (1+t)/L with P; dS^T and dK
            // come out doubled, exactly, and the dK epilogue halves its scale.
            const float2 hh = fmul2(x, hc);
            const float2 t = make_float2(tanh_approx(hh.x), tanh_approx(hh.y));
            const float2 ti = ffma2(t, il, il);
            pv = fmul2(hh, ti);
            const float2 f = fmul2(ti, ffma2(make_float2(-hh.x, -hh.y), t, fadd2(hh, one)));
            fk[c / 2] = pack_bf16(f.x, f.y);
          }
          pk[c / 2] = pack_bf16(pv.x, pv.y);
        }
        // dS^T = P^T (dP^T - D)  or  dP^T SiLU'(u)/L
        if (!mbar_wait(bar(KV_DPFULL + b), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        float dp[HC];
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld32(x_tm + 32 * c, dp + 32 * c);
        tmem_wait_ld();
        uint32_t dk2[HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          const float2 d = make_float2(dp[c], dp[c + 1]);
          if (ACT == kActSoftmax) {  // dP^T - D in fp32, rounded to bf16, times the bf16 P^T
            const float2 t = fadd2(d, *reinterpret_cast<const float2*>(rs + KSTEP + c));
            if constexpr (ROPE) {  // measured faster in fp32 here (register allocation)
              const float2 ds = fmul2(unpack_bf16(pk[c / 2]), t);
              dk2[c / 2] = pack_bf16(ds.x, ds.y);
            } else {
              dk2[c / 2] = mul_bf16x2(pack_bf16(t.x, t.y), pk[c / 2]);
            }
          } else {  // dP^T rounded to bf16, times the bf16 factor, rounded once
            dk2[c / 2] = mul_bf16x2(pack_bf16(d.x, d.y), fk[c / 2]);
          }
        }
        // P^T then dS^T over this group's own, already loaded columns
        if constexpr (HC == 64) {
          tmem_st32(x_tm, reinterpret_cast<const float*>(pk));
          tmem_st32(x_tm + 32, reinterpret_cast<const float*>(dk2));
        } else {
          tmem_st16(x_tm, pk);
          tmem_st16(x_tm + 16, dk2);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(KV_PDSFULL + b));
        if (pend && !epilogue()) { ok = false; break; }
        if constexpr (ROPE) {  // the next item's K and Q tiles
            if (!kv_rotate_next<DQK, NQ, CAUSAL, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp - 2,
                                                     kCompute / 32, lane, abort, status)) {
              ok = false;
              break;
            }
          }
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue (deferred)
      const bool key_ok = j < Lk;
      const int64_t krow = (k0 + j) * p.heads + h;
      if (n > 0) {
        if (pend && !epilogue()) { ok = false; break; }  // defensive: flushed after step 0
        pend = true;
        pend_key_ok = key_ok;
        pend_krow = krow;
        if constexpr (ROPE) pend_kpos = j;
      } else if (key_ok) {
        const float z[32] = {0.f};
        const bool do_k = Gr::G == 2 || grp < 2, do_v = Gr::G == 2 || grp >= 2;
        const int hk = Gr::G == 2 ? grp : (grp & 1);  // which half
        if (do_k) {
#pragma unroll
          for (int c = 0; c < DQK / 64; ++c) store_row_bf16(dk + krow * DQK + hk * (DQK / 2) + 32 * c, z, 1.f);
        }
        if (do_v) {
#pragma unroll
          for (int c = 0; c < DV / 64; ++c) store_row_bf16(dv + krow * DV + hk * (DV / 2) + 32 * c, z, 1.f);
        }
      }
    }
    if (ok && pend) ok = epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================
// dQ pass
// =============================================================================
// One item = (sequence, head, 128-row query tile); the inner loop steps over
// 128 keys.  S is double-buffered in TMEM so that S of the next step is
// computed while the compute warpgroups form dS of this one; dS goes back into
// TMEM as packed bf16 over the S columns it was formed from (each warpgroup its
// own, already loaded), so dP of the next step may start as soon as dP of this
// one is loaded, and dQ += dS K reads dS from there.
template <int DQK, int DV>
struct QLayout {
  // K(j+2) is wanted right after dQ(j) and V(j+1) right after dP(j) is loaded, so
  // the K ring is one stage deeper than the V ring: a TMA load takes about a step.
  // Q and dO tiles are double-buffered across items except at Dqk = Dv = 128, where
  // the K ring keeps its third stage instead (a two-deep K ring there was measured
  // 15-30% slower than single Q and dO tiles).
  static constexpr bool kWide = DQK + DV == 256;
  static constexpr int NQ = kWide ? 1 : 2;  // Q tiles
  static constexpr int NO = kWide ? 1 : 2;  // dO tiles
  static constexpr int NK = DQK == 128 ? 3 : (DV == 128 ? 4 : 6);
  static constexpr int NV = DQK == 64 && DV == 64 ? 4 : 2;
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;   // 128 rows
  static constexpr uint32_t O_BYTES = DV / 64 * 16384;
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;   // 128 keys
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  // in front: mbarriers, TMEM slot, abort flag (640 bytes), the work item ring
  static constexpr uint32_t FEED_OFF = 640;
  static constexpr uint32_t SMALL = FEED_OFF + kFeedSlots * sizeof(WorkItem);
  static constexpr uint32_t TILE0 = 1024;
  static_assert(SMALL <= TILE0, "the front area fits below the tiles");
  static constexpr uint32_t Q_OFF = 0;     // offsets from the 1 KB-aligned tile base
  static constexpr uint32_t O_OFF = Q_OFF + NQ * Q_BYTES;
  static constexpr uint32_t K_OFF = O_OFF + NO * O_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + NK * K_BYTES;
  static constexpr uint32_t TILES = V_OFF + NV * V_BYTES;
  static constexpr uint32_t SMEM = TILE0 + TILES;
  static_assert(SMEM <= 232448u && SMEM >= 122880u, "one CTA per SM within its shared memory");
};

// Each ring has one consumer thread: Q and K feed issuer A (S and dQ), dO and V
// feed issuer B (dP).  dS(g) is signalled on DSFULL[g & 1]: S(g+1) is issued before
// issuer A waits for dS(g), so the compute warps may finish steps g and g+1 before
// it looks, and a single barrier would then have moved on by two phases.
enum : uint32_t {
  Q_QFULL = 0, Q_QEMPTY = 2, Q_OFULL = 4, Q_OEMPTY = 6, Q_KFULL = 8, Q_KEMPTY = 14, Q_VFULL = 20,
  Q_VEMPTY = 24, Q_SFULL = 28, Q_DPFULL = 30, Q_DPEMPTY = 31, Q_DSFULL = 32, Q_ACCFULL = 34,
  Q_ACCEMPTY = 35, Q_DRAIN = 36, Q_QREADY = 38, Q_KREADY = 40, Q_FEEDFULL = 46, Q_FEEDEMPTY = 54,
  Q_COUNT = 62
};
static_assert(8 * Q_COUNT + 8 <= 640, "mbarriers, TMEM slot and abort flag in front of the item ring");

// The dQ pass's counterpart of kv_rotate_next: the item's Q tile and its one K tile.
template <int DQK, int NQ, int NK, class L>
__device__ __forceinline__ bool q_rotate_next(int& rot_next, uint32_t& rot_cnt, const WorkItem* list,
                                              int n_items, uint32_t raw, uint32_t sb, const Problem& p,
                                              int wi, int nw, int lane, volatile int* abort,
                                              int* status) {
  auto bar = [&](uint32_t i) { return raw + 8u * i; };
  while (rot_next < n_items && load_item(list, rot_next).cost == 0) rot_next += gridDim.x;
  if (rot_next >= n_items) return true;
  const WorkItem x = load_item(list, rot_next);
  rot_next += gridDim.x;
  const int row0 = x.tile * TILE;
  const uint32_t qs = rot_cnt % NQ, ks = rot_cnt % NK;
  if (!mbar_wait(bar(Q_QFULL + qs), (rot_cnt / NQ) & 1, abort, status) ||
      !mbar_wait(bar(Q_KFULL + ks), (rot_cnt / NK) & 1, abort, status))
    return false;
  if (row0 == 0) {  // the Q tile and the item's one K tile start at position 0
    rope_rotate_pair_share<DQK>(sb + L::Q_OFF + qs * L::Q_BYTES, rope_rows(0, x.lq, p.rope_npos),
                                        sb + L::K_OFF + ks * L::K_BYTES, rope_rows(0, x.lk, p.rope_npos), 0,
                                        p.rope, wi, nw, lane);
  } else {
    rope_rotate_pair_share<DQK>(sb + L::Q_OFF + qs * L::Q_BYTES, rope_rows(row0, x.lq, p.rope_npos), 0, 0, row0,
                                p.rope, wi, nw, lane);
    rope_rotate_pair_share<DQK>(sb + L::K_OFF + ks * L::K_BYTES, rope_rows(0, x.lk, p.rope_npos), 0, 0, 0, p.rope,
                                wi, nw, lane);
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(bar(Q_QREADY + qs));
    mbar_arrive(bar(Q_KREADY + ks));
  }
  ++rot_cnt;
  return true;
}

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE>
__global__ void __launch_bounds__(QGroups<ACT>::kThreads, 1)
tc_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const Problem p, const float2* __restrict__ rowstat, __nv_bfloat16* __restrict__ dq,
             WsHeader* hdr, const WorkItem* __restrict__ list) {
  using L = QLayout<DQK, DV>;
  using Gr = QGroups<ACT>;
  constexpr int NK = L::NK, NV = L::NV, NQ = L::NQ, NO = L::NO;
  constexpr int HC = Gr::HC;  // key columns per compute warpgroup
  static_assert(HC * Gr::G == STEP && HC % 32 == 0, "the compute warpgroups split a step's keys");
  constexpr uint32_t kCompute = 32 * 4 * Gr::G;  // compute threads
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + L::SMALL + 1023u) & ~1023u;  // 128-byte swizzled tiles: 1 KB aligned
  int* status = &hdr->status;
  uint32_t dyn_bytes;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn_bytes));
  if (sb - raw + L::TILES > dyn_bytes) {  // same for every thread: nothing has started yet
    if (threadIdx.x == 0) atomicExch(status, (int)JFA_ERR_CUDA);
    return;
  }
  auto bar = [&](uint32_t i) { return raw + 8u * i; };
  uint32_t* tmem_slot = (uint32_t*)(smem_raw + 8 * Q_COUNT);
  volatile int* abort = (volatile int*)(smem_raw + 8 * Q_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_q;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar(Q_QFULL + s), 1);
      mbar_init(bar(Q_QEMPTY + s), 1);
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(bar(Q_OFULL + s), 1);
      mbar_init(bar(Q_OEMPTY + s), 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(Q_KFULL + s), 1);
      mbar_init(bar(Q_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(Q_VFULL + s), 1);
      mbar_init(bar(Q_VEMPTY + s), 1);
    }
    mbar_init(bar(Q_SFULL), 1);
    mbar_init(bar(Q_SFULL + 1), 1);
    mbar_init(bar(Q_DPFULL), 1);
    mbar_init(bar(Q_DPEMPTY), kCompute);
    mbar_init(bar(Q_DSFULL), kCompute);
    mbar_init(bar(Q_DSFULL + 1), kCompute);
    mbar_init(bar(Q_ACCFULL), 1);
    mbar_init(bar(Q_ACCEMPTY), kCompute);
    mbar_init(bar(Q_DRAIN), 1);      // issuer A's exit drain
    mbar_init(bar(Q_DRAIN + 1), 1);  // issuer B's exit drain
    // rotated Q and K tiles (rotary embedding): one arrival per compute warp
    for (int s = 0; s < NQ; ++s) mbar_init(bar(Q_QREADY + s), kCompute / 32);
    for (int s = 0; s < NK; ++s) mbar_init(bar(Q_KREADY + s), kCompute / 32);
    // work item ring: warp 0 claims; the second producer, both issuers and every
    // compute warp read
    for (int s = 0; s < kFeedSlots; ++s) {
      mbar_init(bar(Q_FEEDFULL + s), 1);
      mbar_init(bar(Q_FEEDEMPTY + s), 3 + kCompute / 32);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: dQ [0,128), S buffer 0 [128,256), dP (dS) [256,384), S buffer 1 [384,512)
  constexpr uint32_t T_DQ = 0, T_DP = 256;
  auto t_s = [](uint32_t b) { return b ? 384u : 128u; };
  // SiLU/L items may be claimed from the launch's counter as CTAs become free (the
  // scheduler decides per list).  The softmax kernels keep the fixed assignment: their
  // workloads' items are short, and the feed's registers would cost them spills; so do
  // the rotary kernels, whose compute warps look ahead in the list.
  constexpr bool kDyn = !ROPE && ACT != kActSoftmax;
  static_assert(Q_FEEDEMPTY == Q_FEEDFULL + kFeedSlots, "feed ring barriers");
  const FeedRing ring{bar(Q_FEEDFULL), raw + L::FEED_OFF};
  int* const claim_ctr = &hdr->claim[kClaimDq];

  // Rotary embedding of Q and K (BlockAttention): the compute warps rotate each item's K
  // and Q tiles in shared memory once they have landed and signal them ready; issuer A
  // waits for that instead of the loads.  Its items are blocks of at most 64 rows, so
  // each has exactly one step; the compute warps rotate the next item's tiles right after
  // the current item's step, while its gradient products run.
  constexpr bool rope = ROPE;
  if (warp == 0 || warp == Gr::kProducer2) {
    // ------------------------------------------------------------ producers
    // warp 0: the item's Q tile, then K(0), K(1), ...; the second producer: its dO
    // tile, then V(0), V(1), ...  Each ring is filled in consumption order.
    if (lane == 0) {
      const bool qk = warp == 0;
      const CUtensorMap* tm_row = qk ? &tm_q : &tm_do;
      const CUtensorMap* tm_key = qk ? &tm_k : &tm_v;
      tma_prefetch_desc(tm_row);
      tma_prefetch_desc(tm_key);
      const int D = qk ? DQK : DV;
      const uint32_t row_off = qk ? L::Q_OFF : L::O_OFF, row_bytes = qk ? L::Q_BYTES : L::O_BYTES;
      const uint32_t key_off = qk ? L::K_OFF : L::V_OFF, key_bytes = qk ? L::K_BYTES : L::V_BYTES;
      const uint32_t nring = qk ? NK : NV, nrow = qk ? NQ : NO;
      const uint32_t b_rfull = qk ? Q_QFULL : Q_OFULL, b_rempty = qk ? Q_QEMPTY : Q_OEMPTY;
      const uint32_t b_kfull = qk ? Q_KFULL : Q_VFULL, b_kempty = qk ? Q_KEMPTY : Q_VEMPTY;
      uint32_t q_it = 0, t_it = 0;
      bool ok = true;
      FeedClaimer<kDyn> claimer;  // warp 0 claims, the second producer reads
      Feed<kDyn> feed;
      if (qk)
        claimer.init(ring, list, claim_ctr, n_items);
      else
        feed.init(ring, list, claim_ctr, n_items);
      WorkItem w;
      while (ok && (qk ? claimer.claim(w, abort, status) : feed.take(w, false, true, abort, status))) {
        const int n = w.cost;
        if (n == 0) continue;
        const int h = w.h, row0 = w.tile * TILE;
        const int32_t q0 = w.q0, k0 = w.k0;
        const uint32_t qs = q_it % nrow, qph = ((q_it / nrow) & 1) ^ 1;
        if (!mbar_wait(bar(b_rempty + qs), qph, abort, status)) break;
        mbar_expect_tx(bar(b_rfull + qs), row_bytes);
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(sb + row_off + qs * row_bytes + a * 16384, tm_row, h * D + a * 64, q0 + row0,
                      bar(b_rfull + qs));
        ++q_it;
        for (int j = 0; j < n; ++j, ++t_it) {
          const uint32_t st = t_it % nring;
          if (!mbar_wait(bar(b_kempty + st), ((t_it / nring) & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(bar(b_kfull + st), key_bytes);
          for (int a = 0; a < D / 64; ++a)
            tma_load_2d(sb + key_off + st * key_bytes + a * 16384, tm_key, h * D + a * 64, k0 + j * STEP,
                        bar(b_kfull + st));
        }
      }
      // every load issued has landed before the CTA leaves (also after giving up)
      drain_ring(bar(b_rfull), nrow, q_it, status);
      drain_ring(bar(b_kfull), nring, t_it, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ issuer A: S and dQ
    // dS(g) is written by the compute warpgroups over their own (already read) S(g)
    // columns, so the dP columns are free as soon as dP(g) is loaded and dP(g+1)
    // need not wait for dQ(g); S(g+2) reuses the buffer after dQ(g) has read dS(g).
    // With two Q tiles the steps are walked over the CTA's whole list, so S of the
    // next item's first two steps is issued before the last two dQ products of this
    // one.  With a single Q tile the items are walked one by one: the next Q tile
    // loads only once this item's last S has completed, and the cross-item walk was
    // measured 2-12% slower there.
    {  // the whole warp runs the issuer loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_bf16(TILE, STEP, 0, 0);
      constexpr uint32_t idesc_dq = idesc_bf16(TILE, DQK, 0, 1);
      if constexpr (NQ == 1) {
        uint32_t q_it = 0, k_it = 0, s_it = 0, d_it = 0, a_it = 0;
        bool ok = true;
        Feed<kDyn> feed;
        feed.init(ring, list, claim_ctr, n_items);
        WorkItem w;
        while (ok && feed.take(w, true, true, abort, status)) {
          const int n = w.cost;
          if (n == 0) continue;
          const uint32_t qs = q_it % NQ;
          if (!mbar_wait(bar((rope ? Q_QREADY : Q_QFULL) + qs), (q_it / NQ) & 1, abort, status)) break;
          const uint32_t q_tile = sb + L::Q_OFF + qs * L::Q_BYTES;
          const uint32_t k_base = k_it, s_base = s_it;
          auto issue_s = [&](int i) {  // S(i) = Q K(i)^T into buffer (s_base + i) & 1
            const uint32_t kk_it = k_base + i, kst = kk_it % NK;
            if (!mbar_wait(bar((rope ? Q_KREADY : Q_KFULL) + kst), (kk_it / NK) & 1, abort, status)) return false;
            __syncwarp();  // converged for elect.sync
            tc_fence_after();
            const uint32_t k_tile = sb + L::K_OFF + kst * L::K_BYTES;
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              mma_bf16(tmem + t_s((s_base + i) & 1), sw128_desc(q_tile + off, 16, 1024),
                       sw128_desc(k_tile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(Q_SFULL + ((s_base + i) & 1)));
            if (i == n - 1) mma_commit(bar(Q_QEMPTY + qs));  // last use of this Q tile
            return true;
          };
          ok = issue_s(0);
          if (ok && n > 1) ok = issue_s(1);
          for (int j = 0; j < n && ok; ++j) {
            const uint32_t kst = (k_base + j) % NK;
            // dQ += dS(j) K(j); dS packed in TMEM over the S(j) columns of each group
            if (!mbar_wait(bar(Q_DSFULL + (d_it & 1)), (d_it >> 1) & 1, abort, status) ||
                (j == 0 && !mbar_wait(bar(Q_ACCEMPTY), (a_it & 1) ^ 1, abort, status))) {
              ok = false;
              break;
            }
            __syncwarp();  // converged for elect.sync
            tc_fence_after();
            const uint32_t k_tile = sb + L::K_OFF + kst * L::K_BYTES;
            const uint32_t ds_tm = tmem + t_s((s_base + j) & 1);
#pragma unroll
            for (int kk = 0; kk < STEP / 16; ++kk)
              mma_bf16_tmem_a(tmem + T_DQ, ds_tm + (kk / (HC / 16)) * HC + (kk % (HC / 16)) * 8,
                              sw128_desc(k_tile + kk * 2048, 16384, 1024), idesc_dq,
                              (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(Q_KEMPTY + kst));
            ++d_it;
            if (j + 2 < n) ok = issue_s(j + 2);
          }
          if (!ok) break;
          mma_commit(bar(Q_ACCFULL));
          k_it += n;
          s_it += n;
          ++q_it;
          ++a_it;
        }
      } else {
        uint32_t a_it = 0;
        bool ok = true;
        // S(c.g) = Q K(c.g)^T into buffer c.g & 1; the item's Q tile is stage c.kv % NQ
        auto issue_s = [&](const StepCursor<kDyn>& c) -> bool {
          const uint32_t qs = c.kv % NQ, kst = c.g % NK;
          if ((c.j == 0 && !mbar_wait(bar((rope ? Q_QREADY : Q_QFULL) + qs), (c.kv / NQ) & 1, abort, status)) ||
              !mbar_wait(bar((rope ? Q_KREADY : Q_KFULL) + kst), (c.g / NK) & 1, abort, status))
            return false;
          __syncwarp();  // converged for elect.sync
          tc_fence_after();
          const uint32_t q_tile = sb + L::Q_OFF + qs * L::Q_BYTES;
          const uint32_t k_tile = sb + L::K_OFF + kst * L::K_BYTES;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem + t_s(c.g & 1), sw128_desc(q_tile + off, 16, 1024),
                     sw128_desc(k_tile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(Q_SFULL + (c.g & 1)));
          if (c.last()) mma_commit(bar(Q_QEMPTY + qs));  // last use of this Q tile
          return true;
        };
        StepCursor<kDyn> cs, cg;  // cs: next S (up to two steps ahead); cg: next dQ
        cs.init(ring, list, claim_ctr, n_items, false, abort, status);
        cg.init(ring, list, claim_ctr, n_items, true, abort, status);
        auto run_ahead = [&]() -> bool {  // S up to step cg.g + 1
          while (cs.valid && cg.valid && cs.g < cg.g + 2) {
            if (!issue_s(cs)) return false;
            cs.advance();
          }
          return true;
        };
        ok = run_ahead();
        while (ok && cg.valid) {
          // dQ += dS(g) K(g); dS packed in TMEM over the S(g) columns of each group
          const uint32_t kst = cg.g % NK;
          if (!mbar_wait(bar(Q_DSFULL + (cg.g & 1)), (cg.g >> 1) & 1, abort, status) ||
              (cg.j == 0 && !mbar_wait(bar(Q_ACCEMPTY), (a_it & 1) ^ 1, abort, status))) {
            ok = false;
            break;
          }
          __syncwarp();  // converged for elect.sync
          tc_fence_after();
          const uint32_t k_tile = sb + L::K_OFF + kst * L::K_BYTES;
          const uint32_t ds_tm = tmem + t_s(cg.g & 1);
#pragma unroll
          for (int kk = 0; kk < STEP / 16; ++kk)
            mma_bf16_tmem_a(tmem + T_DQ, ds_tm + (kk / (HC / 16)) * HC + (kk % (HC / 16)) * 8,
                            sw128_desc(k_tile + kk * 2048, 16384, 1024), idesc_dq,
                            (cg.j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(Q_KEMPTY + kst));
          if (cg.last()) {
            mma_commit(bar(Q_ACCFULL));
            ++a_it;
          }
          cg.advance();
          ok = run_ahead();
        }
      }
      __syncwarp();
      mma_drain(bar(Q_DRAIN), status);  // every MMA issued has completed
    }
    __syncwarp();
  } else if (warp == Gr::kIssuerB) {
    // ------------------------------------------------------------ issuer B: dP = dO V^T
    {  // the whole warp runs the issuer loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_bf16(TILE, STEP, 0, 0);
      uint32_t q_it = 0, v_it = 0, dp_it = 0;  // V ring: v_it % NV
      bool ok = true;
      Feed<kDyn> feed;
      feed.init(ring, list, claim_ctr, n_items);
      WorkItem w;
      while (ok && feed.take(w, true, true, abort, status)) {
        const int n = w.cost;
        if (n == 0) continue;
        const uint32_t qs = q_it % NO;
        if (!mbar_wait(bar(Q_OFULL + qs), (q_it / NO) & 1, abort, status)) break;
        const uint32_t o_tile = sb + L::O_OFF + qs * L::O_BYTES;
        for (int j = 0; j < n; ++j, ++v_it, ++dp_it) {
          const uint32_t vst = v_it % NV;
          // the dP columns are free once the compute warpgroups have loaded dP(j-1)
          if (!mbar_wait(bar(Q_VFULL + vst), (v_it / NV) & 1, abort, status) ||
              !mbar_wait(bar(Q_DPEMPTY), (dp_it & 1) ^ 1, abort, status)) {
            ok = false;
            break;
          }
          __syncwarp();  // converged for elect.sync
          tc_fence_after();
          const uint32_t v_tile = sb + L::V_OFF + vst * L::V_BYTES;
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem + T_DP, sw128_desc(o_tile + off, 16, 1024), sw128_desc(v_tile + off, 16, 1024),
                     idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(Q_DPFULL));
          mma_commit(bar(Q_VEMPTY + vst));
          if (j == n - 1) mma_commit(bar(Q_OEMPTY + qs));  // last use of this dO tile
        }
        if (!ok) break;
        ++q_it;
      }
      __syncwarp();
      mma_drain(bar(Q_DRAIN + 1), status);  // every MMA issued has completed
    }
    __syncwarp();
  } else {
    // Compute warpgroups: group grp (four consecutive warps, all 128 rows) takes key
    // columns [HC grp, HC grp + HC) of every step and dQ columns [CQ grp, CQ grp + CQ)
    // in the epilogue; each group writes only inside its own columns.
    const int grp = (warp - 2) >> 2;
    const int r = 32 * (warp & 3) + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    const float2 cc = make_float2(c_score, c_score);
    const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
    const float2 one = make_float2(1.f, 1.f);
    const uint32_t p_tm = tmem + lane_base + T_DP + grp * HC;
    // dQ columns drained per group, in whole 32-column loads: with four groups and
    // Dqk = 64 the last two groups drain nothing
    constexpr int CQ = DQK / Gr::G >= 32 ? DQK / Gr::G : 32;
    const bool drains = CQ * Gr::G == DQK || grp * CQ < DQK;
    uint32_t s_it = 0, d_it = 0, a_it = 0;
    bool ok = true;
    // The epilogue of an item (dQ from TMEM to HBM) runs after the next item's first
    // step, when its last dQ product has long completed; the next item's first dQ
    // product waits for it (ACCEMPTY).
    bool pend = false, pend_row_ok = false;
    int64_t pend_orow = 0;
    int pend_pos = 0;  // row index inside its sequence: the rotary embedding's position
    auto epilogue = [&]() -> bool {
      if (!mbar_wait(bar(Q_ACCFULL), a_it & 1, abort, status)) return false;
      ++a_it;
      tc_fence_after();
      if (drains) {
        float x[CQ];
#pragma unroll
        for (int c = 0; c < CQ / 32; ++c) tmem_ld32(tmem + lane_base + T_DQ + grp * CQ + 32 * c, x + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(Q_ACCEMPTY));
        // dQ with the rotary embedding: the gradient of the rotated queries turned back
        if (rope && pend_row_ok && pend_pos < p.rope_npos)
          rope_unrotate_row<CQ>(x, grp * CQ, pend_pos, DQK, p.rope);
        if (pend_row_ok) {
#pragma unroll
          for (int c = 0; c < CQ / 32; ++c) {
            if (p.dq_f32)
              store_row_f32(p.dq_f32 + pend_orow * DQK + grp * CQ + 32 * c, x + 32 * c, p.scale);
            else
              store_row_bf16(dq + pend_orow * DQK + grp * CQ + 32 * c, x + 32 * c, p.scale);
          }
        }
      } else {
        tc_fence_before();
        mbar_arrive(bar(Q_ACCEMPTY));
      }
      pend = false;
      return true;
    };
    // rotary embedding: the next non-empty item to rotate (list index) and the count of
    // items rotated so far (which fixes its Q and K stages)
    int rot_next = blockIdx.x;
    uint32_t rot_cnt = 0;
    if constexpr (ROPE) {
      if (!q_rotate_next<DQK, NQ, NK, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp - 2,
                                          kCompute / 32, lane, abort, status))
        ok = false;
    }
    Feed<kDyn> feed;
    feed.init(ring, list, claim_ctr, n_items);
    WorkItem w;
    while (ok && feed.take(w, true, true, abort, status)) {
      const int n = w.cost;
      const int h = w.h, row0 = w.tile * TILE;
      const int64_t q0 = w.q0;
      const int Lq = w.lq, Lk = w.lk;
      const int i = row0 + r;
      const bool row_ok = i < Lq;
      if (rope && n > 1) {  // the rotary kernels take items of one step only
        if (lane == 0) atomicExch(status, (int)JFA_ERR_UNSUPPORTED);
        *abort = 1;
        ok = false;
        break;
      }
      const float inv_len = 1.0f / (float)max(Lq, 1);
      const float2 hl = make_float2(0.5f * inv_len, 0.5f * inv_len);
      float2 rsv = make_float2(0.f, 0.f);
      if (ACT == kActSoftmax && row_ok && n > 0) rsv = rowstat[(int64_t)h * p.total_q + q0 + i];
      const float2 nl = make_float2(-rsv.x, -rsv.x), nd = make_float2(-rsv.y, -rsv.y);
      for (int step = 0; step < n; ++step, ++s_it, ++d_it) {
        const uint32_t sbuf = s_it & 1;
        if (!mbar_wait(bar(Q_SFULL + sbuf), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t s_tm = tmem + lane_base + t_s(sbuf) + grp * HC;
        float sv[HC];
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld32(s_tm + 32 * c, sv + 32 * c);
        tmem_wait_ld();
        const int kb = step * STEP + grp * HC;
        int nvalid = Lk - kb;
        if (CAUSAL) nvalid = min(nvalid, i - kb + 1);
        if (p.block_mask > 0 && (kb ^ i) >= p.block_mask) nvalid = 0;  // another block's keys
        if (!row_ok) nvalid = 0;
        if (nvalid < HC) {
#pragma unroll
          for (int c = 0; c < HC; ++c) sv[c] -= c < nvalid ? 0.f : shift_raw;
        }
        // P (softmax) or SiLU'(u)/L, packed bf16; both multiply dP into dS
        uint32_t fk[HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          const float2 x = make_float2(sv[c], sv[c + 1]);
          float2 f;
          if (ACT == kActSoftmax) {
            const float2 e = ffma2(x, cc, nl);
            f = make_float2(ex2(e.x), ex2(e.y));
          } else {
            const float2 hh = fmul2(x, hc);
            const float2 t = make_float2(tanh_approx(hh.x), tanh_approx(hh.y));
            f = fmul2(ffma2(t, hl, hl), ffma2(make_float2(-hh.x, -hh.y), t, fadd2(hh, one)));
          }
          fk[c / 2] = pack_bf16(f.x, f.y);
        }
        if (!mbar_wait(bar(Q_DPFULL), d_it & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        float dp[HC];
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_ld32(p_tm + 32 * c, dp + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(Q_DPEMPTY));  // dP(step + 1) may overwrite the dP columns
        uint32_t dk2[HC / 2];
#pragma unroll
        for (int c = 0; c < HC; c += 2) {
          const float2 d = make_float2(dp[c], dp[c + 1]);
          if (ACT == kActSoftmax) {  // dP - D in fp32, rounded to bf16, times the bf16 P
            const float2 t = fadd2(d, nd);
            if constexpr (ROPE) {  // measured faster in fp32 here (register allocation)
              const float2 ds = fmul2(unpack_bf16(fk[c / 2]), t);
              dk2[c / 2] = pack_bf16(ds.x, ds.y);
            } else {
              dk2[c / 2] = mul_bf16x2(pack_bf16(t.x, t.y), fk[c / 2]);
            }
          } else {  // dP rounded to bf16, times the bf16 factor, rounded once
            dk2[c / 2] = mul_bf16x2(pack_bf16(d.x, d.y), fk[c / 2]);
          }
        }
        // dS over this group's own S columns (already loaded above)
        if constexpr (HC == 64)
          tmem_st32(s_tm, reinterpret_cast<const float*>(dk2));
        else
          tmem_st16(s_tm, dk2);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(Q_DSFULL + sbuf));
        if (pend && !epilogue()) { ok = false; break; }
        if constexpr (ROPE) {  // the next item's Q and K tiles
          if (!q_rotate_next<DQK, NQ, NK, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp - 2,
                                              kCompute / 32, lane, abort, status)) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) break;
      const int64_t orow = (q0 + i) * p.heads + h;
      if (n > 0) {  // epilogue deferred to the next item's first step
        if (pend && !epilogue()) { ok = false; break; }
        pend = true;
        pend_row_ok = row_ok;
        pend_orow = orow;
        if constexpr (ROPE) pend_pos = i;
      } else if (row_ok) {
        const float z[32] = {0.f};
        if (drains) {
#pragma unroll
          for (int c = 0; c < CQ / 32; ++c) {
            if (p.dq_f32)
              store_row_f32(p.dq_f32 + orow * DQK + grp * CQ + 32 * c, z, 1.f);
            else
              store_row_bf16(dq + orow * DQK + grp * CQ + 32 * c, z, 1.f);
          }
        }
      }
    }
    if (ok && pend) ok = epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
// Every tile of both passes is 128 rows (or keys) by 64 columns.
struct Maps {
  CUtensorMap q, dout, k, v;
};

bool make_maps(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
               Maps* m) {
  const int64_t cq = (int64_t)p.heads * p.dim_qk, cv = (int64_t)p.heads * p.dim_v;
  const int64_t tk = p.total_k > 0 ? p.total_k : p.total_q;
  const void* kk = p.total_k > 0 ? k : q;
  const void* vv = p.total_k > 0 ? v : dout;
  return make_tile_map(&m->q, q, p.total_q, cq, 64, TILE) &&
         make_tile_map(&m->dout, dout, p.total_q, cv, 64, TILE) &&
         make_tile_map(&m->k, kk, tk, cq, 64, TILE) && make_tile_map(&m->v, vv, tk, cv, 64, TILE);
}

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE = false>
cudaError_t dkdv_t(const Maps& m, const Problem& p, const float2* rowstat, void* dk, void* dv,
                   const Workspace& ws, cudaStream_t s) {
  auto kern = tc_dkdv_kernel<DQK, DV, ACT, CAUSAL, ROPE>;
  constexpr uint32_t smem = KvLayout<DQK, DV>::SMEM;
  cudaError_t e = kernel_setup((const void*)kern, KvGroups<ACT>::kThreads, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), KvGroups<ACT>::kThreads, smem, s>>>(m.k, m.v, m.q, m.dout, p, rowstat,
                                         (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, ws.hdr, ws.list_k);
  return cudaGetLastError();
}

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE = false>
cudaError_t dq_t(const Maps& m, const Problem& p, const float2* rowstat, void* dq,
                 const Workspace& ws, cudaStream_t s) {
  auto kern = tc_dq_kernel<DQK, DV, ACT, CAUSAL, ROPE>;
  constexpr uint32_t smem = QLayout<DQK, DV>::SMEM;
  cudaError_t e = kernel_setup((const void*)kern, QGroups<ACT>::kThreads, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), QGroups<ACT>::kThreads, smem, s>>>(m.q, m.dout, m.k, m.v, p, rowstat,
                                         (__nv_bfloat16*)dq, ws.hdr, ws.list_q);
  return cudaGetLastError();
}

#define JFA_TC_BWD_DISPATCH(FN, ...)                                                          \
  do {                                                                                        \
    const bool sm_ = p.act == kActSoftmax, c_ = p.causal != 0;                               \
    if (p.rope != nullptr) { /* rotary embedding: softmax, Dqk = Dv */                       \
      if (!sm_ || p.dim_qk != p.dim_v) return cudaErrorInvalidValue;                         \
      if (p.dim_qk == 128) return c_ ? FN<128, 128, kActSoftmax, true, true>(__VA_ARGS__)     \
                                     : FN<128, 128, kActSoftmax, false, true>(__VA_ARGS__);   \
      if (p.dim_qk == 64) return c_ ? FN<64, 64, kActSoftmax, true, true>(__VA_ARGS__)        \
                                    : FN<64, 64, kActSoftmax, false, true>(__VA_ARGS__);      \
      return cudaErrorInvalidValue;                                                           \
    }                                                                                         \
    if (p.dim_qk == 128 && p.dim_v == 128) {                                                  \
      if (sm_) return c_ ? FN<128, 128, kActSoftmax, true>(__VA_ARGS__)                       \
                         : FN<128, 128, kActSoftmax, false>(__VA_ARGS__);                     \
      return c_ ? FN<128, 128, kActSiluOverLen, true>(__VA_ARGS__)                            \
                : FN<128, 128, kActSiluOverLen, false>(__VA_ARGS__);                          \
    }                                                                                         \
    if (p.dim_qk == 128 && p.dim_v == 64) {                                                   \
      if (sm_) return c_ ? FN<128, 64, kActSoftmax, true>(__VA_ARGS__)                        \
                         : FN<128, 64, kActSoftmax, false>(__VA_ARGS__);                      \
      return c_ ? FN<128, 64, kActSiluOverLen, true>(__VA_ARGS__)                             \
                : FN<128, 64, kActSiluOverLen, false>(__VA_ARGS__);                           \
    }                                                                                         \
    if (p.dim_qk == 64 && p.dim_v == 128) {                                                   \
      if (sm_) return c_ ? FN<64, 128, kActSoftmax, true>(__VA_ARGS__)                        \
                         : FN<64, 128, kActSoftmax, false>(__VA_ARGS__);                      \
      return c_ ? FN<64, 128, kActSiluOverLen, true>(__VA_ARGS__)                             \
                : FN<64, 128, kActSiluOverLen, false>(__VA_ARGS__);                           \
    }                                                                                         \
    if (p.dim_qk == 64 && p.dim_v == 64) {                                                    \
      if (sm_) return c_ ? FN<64, 64, kActSoftmax, true>(__VA_ARGS__)                         \
                         : FN<64, 64, kActSoftmax, false>(__VA_ARGS__);                       \
      return c_ ? FN<64, 64, kActSiluOverLen, true>(__VA_ARGS__)                              \
                : FN<64, 64, kActSiluOverLen, false>(__VA_ARGS__);                            \
    }                                                                                         \
    return cudaErrorInvalidValue;                                                             \
  } while (0)

}  // namespace

// q-list: 128-row tiles over 128-key steps (dQ); k-list: 128-key tiles over 128-row steps (dK/dV)
SchedConfig tc_bwd_sched(const Problem&) { return SchedConfig{TILE, STEP, TILE, KSTEP, 1, 1, 0}; }

cudaError_t launch_tc_rowstat(const Problem& p, const void* o, const void* dout, const float* lse,
                              const Workspace& ws, cudaStream_t s) {
  const int64_t threads = p.total_q * p.heads * (p.dim_v / 8);
  if (threads == 0) return cudaSuccess;
  int64_t blocks = (threads + 255) / 256;  // one pass; the loop covers grids past the cap
  const int64_t cap = (int64_t)1 << 30;
  if (blocks > cap) blocks = cap;
  float2* rs = reinterpret_cast<float2*>(ws.drow);
  if (p.dim_v == 128)
    rowstat_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(p.total_q, p.heads, (const __nv_bfloat16*)o,
                                                         (const __nv_bfloat16*)dout, lse, rs);
  else
    rowstat_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(p.total_q, p.heads, (const __nv_bfloat16*)o,
                                                        (const __nv_bfloat16*)dout, lse, rs);
  return cudaGetLastError();
}

cudaError_t launch_tc_dkdv(const Problem& p, const void* q, const void* k, const void* v,
                           const float* lse, const void* dout, void* dk, void* dv,
                           const Workspace& ws, cudaStream_t s) {
  (void)lse;
  Maps m;
  if (!make_maps(p, q, k, v, dout, &m)) return cudaErrorInvalidValue;
  const float2* rs = reinterpret_cast<const float2*>(ws.drow);
  JFA_TC_BWD_DISPATCH(dkdv_t, m, p, rs, dk, dv, ws, s);
}

cudaError_t launch_tc_dq(const Problem& p, const void* q, const void* k, const void* v,
                         const float* lse, const void* dout, void* dq, const Workspace& ws,
                         cudaStream_t s) {
  (void)lse;
  Maps m;
  if (!make_maps(p, q, k, v, dout, &m)) return cudaErrorInvalidValue;
  const float2* rs = reinterpret_cast<const float2*>(ws.drow);
  JFA_TC_BWD_DISPATCH(dq_t, m, p, rs, dq, ws, s);
}

}  // namespace jfa
