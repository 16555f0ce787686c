// Tensor-core jagged attention forward for sm_103a: TMA + tcgen05 + TMEM.
//
// Method: Jagged Flash Attention bullet of the Meta GEM MFU write-up
// (piletech.kr/articles/112134, details): attention computed directly on the
// jagged buffers, masked by subtraction, persistent kernel scheduling with
// specialised warps; Generalized Dot-Product Attention bullet: the same
// pipeline with a non-softmax activation (here SiLU(s)/L).
//
// One persistent CTA per SM walks the scheduler's heavy-first list of
// (sequence, head, 128-row q-tile) items.  Warp roles (G compute warpgroups: 2 for
// softmax, 4 for SiLU/L):
//   warps 0..4G-1  compute warpgroups: group g takes key columns
//                  [g*128/G, (g+1)*128/G) of every 128-key step (one query row
//                  per thread = TMEM lane).  Softmax: the two threads of a row
//                  exchange their partial row maximum through shared memory.
//                  SiLU/L has no row statistics, so its elementwise work is
//                  split four ways: twice the warps hide the latencies of the
//                  TMEM loads and of tanh.
//   warp 4G        TMA producer of Q (double-buffered across items) and of the K
//                  ring; warp 4G+3 that of the V ring.  128-key tiles come
//                  straight from the jagged [T, H*D] buffers (rows past a
//                  sequence belong to its neighbour and are masked; rows past
//                  the buffer are zero-filled by TMA)
//   warp 4G+1      TMEM owner and S = Q K^T issuer (one lane)
//   warp 4G+2      O += P V issuer (one lane)
// TMEM: S double-buffered at columns [0,128) and [128,256), O at [256, 256+Dv),
// P (packed bf16, 128 keys) double-buffered at [384, 448) and [448, 512).  S of
// step j+2 goes into the buffer of S(j) once P(j) has been written; PV(j) reads
// P buffer j & 1, which P(j+2) reuses once PV(j) has completed.
// Per step the softmax warpgroups scale to log2 units,
// subtract a finite shift from masked columns, keep an online max with lazy
// rescaling of O (only when it grows by more than 2^8), take exp2 and the row
// sum, and write P.  Epilogue: O / l -> bf16, lse = (m + log2 l) ln 2.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc.h"
#include "tc_host.h"
#include "tc_ptx.cuh"
#include "feed.cuh"

namespace jfa {
namespace {
using namespace tc;

constexpr int BM = 128;     // rows per item (MMA M)
constexpr int BN = 128;     // keys per step (MMA N of S)

// Warp roles of the forward for activation ACT (see the file comment).
template <int ACT>
struct FwdRoles {
  static constexpr int G = ACT == kActSoftmax ? 2 : 4;  // compute warpgroups
  static constexpr int HC = BN / G;                      // key columns per group
  static constexpr int kCompute = 128 * G;               // compute threads
  static constexpr int kProducerWarp = 4 * G, kSWarp = 4 * G + 1, kPvWarp = 4 * G + 2,
                       kVWarp = 4 * G + 3;
  static constexpr int kThreads = 32 * (4 * G + 4);
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

template <int DQK, int DV>
struct FwdLayout {
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;  // one 128-row tile
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;  // one 128-key tile
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  // In front of the tiles: mbarriers, TMEM slot and abort flag (640 bytes), the work
  // item ring, then the row statistics exchanged by the two softmax warpgroups
  // ([2 steps][128 rows][2]).
  static constexpr uint32_t FEED_OFF = 640;
  static constexpr uint32_t RED_OFF = FEED_OFF + kFeedSlots * sizeof(WorkItem);
  static constexpr uint32_t RED_BYTES = 2 * BM * 2 * 4;
  static constexpr uint32_t SMALL = RED_OFF + RED_BYTES;
  static constexpr uint32_t TILE0 = (SMALL + 1023) / 1024 * 1024;  // for a 1 KB-aligned base
  static constexpr uint32_t kMaxSmem = 232448;
  // Q is double-buffered, so the next item's Q tile loads during this item; the K
  // and V rings take the rest (at Dqk = Dv = 128 the V ring is the shorter one: V(j)
  // is wanted a step after K(j)).
  static constexpr int NQB = 2;
  static constexpr int NK = DQK == 64 ? (DV == 64 ? 6 : 4) : 3;
  static constexpr int NV = DV == 64 ? (DQK == 64 ? 6 : 4) : (DQK == 64 ? 4 : 2);
  static constexpr uint32_t Q_OFF = 0;  // offsets from the 1 KB-aligned tile base
  static constexpr uint32_t K_OFF = Q_OFF + NQB * Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + NK * K_BYTES;
  static constexpr uint32_t TILES = V_OFF + NV * V_BYTES;
  static constexpr uint32_t SMEM = TILE0 + TILES;
  static_assert(SMEM <= kMaxSmem, "forward tiles exceed the shared memory of one CTA");
  static_assert(SMEM >= 122880u, "one CTA per SM: it owns all of TMEM");
};

enum : uint32_t {
  B_QFULL = 0, B_QEMPTY = 2, B_KFULL = 4, B_KEMPTY = 10, B_VFULL = 16, B_VEMPTY = 22,
  B_SFULL = 28, B_PFULL = 30, B_PEMPTY = 32, B_OFULL = 34, B_OEMPTY = 35, B_RED = 36, B_REDL = 38,
  B_DRAIN = 40, B_HOLD = 42, B_QREADY = 43, B_KREADY = 45, B_FEEDFULL = 51, B_FEEDEMPTY = 59,
  B_COUNT = 67
};
static_assert(8 * B_COUNT + 8 <= FwdLayout<128, 128>::FEED_OFF, "mbarriers, TMEM slot and abort flag in front");
constexpr uint32_t T_S = 0, T_O = 256, T_P = 384;  // S: 2 x 128 columns; P: 2 x 64 columns

// Rotary embedding (BlockAttention), done by the compute warps: the next non-empty item
// of the CTA's list (index rot_next, advanced) has its Q and K tiles rotated once they
// have landed, and signalled ready (one arrival per compute warp).  rot_cnt counts the
// items rotated, which fixes their ring stages (every item of the rotary kernels has one
// step).  Warp wi of the nw compute warps takes its share of the rows.  False if a wait
// gave up.
template <int DQK, int NK, class L>
__device__ __forceinline__ bool fwd_rotate_next(int& rot_next, uint32_t& rot_cnt, const WorkItem* list,
                                                int n_items, uint32_t raw, uint32_t sb, const Problem& p,
                                                int wi, int nw, int lane, volatile int* abort,
                                                int* status) {
  auto bar = [&](uint32_t i) { return raw + 8u * i; };
  while (rot_next < n_items && load_item(list, rot_next).cost == 0) rot_next += gridDim.x;
  if (rot_next >= n_items) return true;
  const WorkItem x = load_item(list, rot_next);
  rot_next += gridDim.x;
  const uint32_t qs = rot_cnt % L::NQB, ks = rot_cnt % NK;
  if (!mbar_wait(bar(B_QFULL + qs), (rot_cnt / L::NQB) & 1, abort, status) ||
      !mbar_wait(bar(B_KFULL + ks), (rot_cnt / NK) & 1, abort, status))
    return false;
  if (x.tile == 0) {  // the Q tile and the item's one K tile start at position 0
    rope_rotate_pair_share<DQK>(sb + L::Q_OFF + qs * L::Q_BYTES, rope_rows(0, x.lq, p.rope_npos),
                                   sb + L::K_OFF + ks * L::K_BYTES, rope_rows(0, x.lk, p.rope_npos), 0, p.rope,
                                   wi, nw, lane);
  } else {
    rope_rotate_pair_share<DQK>(sb + L::Q_OFF + qs * L::Q_BYTES, rope_rows(x.tile * BM, x.lq, p.rope_npos), 0,
                                0, x.tile * BM, p.rope, wi, nw, lane);
    rope_rotate_pair_share<DQK>(sb + L::K_OFF + ks * L::K_BYTES, rope_rows(0, x.lk, p.rope_npos), 0, 0, 0,
                                p.rope, wi, nw, lane);
  }
  __syncwarp();
  if (lane == 0) {
    mbar_arrive(bar(B_QREADY + qs));
    mbar_arrive(bar(B_KREADY + ks));
  }
  ++rot_cnt;
  return true;
}

// Test hook (jfa_test_hold): while nonzero, the S issuer of every CTA first waits on
// B_HOLD, on which no role ever arrives, so that its bounded wait gives up before any
// MMA is issued and the CTA leaves through its abort path.  Zero unless a test sets it.
__device__ int g_test_hold = 0;

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE>
__global__ void __launch_bounds__(FwdRoles<ACT>::kThreads, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const Problem p,
              __nv_bfloat16* __restrict__ out, float* __restrict__ lse, WsHeader* hdr,
              const WorkItem* __restrict__ list) {
  using L = FwdLayout<DQK, DV>;
  using R = FwdRoles<ACT>;
  constexpr int NK = L::NK, NV = L::NV;
  constexpr int HC = R::HC;
  constexpr int OC = DV / R::G;  // O columns drained per compute warpgroup
  constexpr int kProducerWarp = R::kProducerWarp, kSWarp = R::kSWarp, kPvWarp = R::kPvWarp,
                kVWarp = R::kVWarp;
  static_assert(R::G == 2 || ACT != kActSoftmax, "softmax row statistics are exchanged in pairs");
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
  uint32_t* tmem_slot = (uint32_t*)(smem_raw + 8 * B_COUNT);
  volatile int* abort = (volatile int*)(smem_raw + 8 * B_COUNT + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_q;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_QFULL + s), 1);
      mbar_init(bar(B_QEMPTY + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), R::kCompute);
      mbar_init(bar(B_PEMPTY + s), 1);
      // exchanges between the two softmax warpgroups (bounded waits, never bar.sync)
      mbar_init(bar(B_RED + s), 256);
      mbar_init(bar(B_REDL + s), 256);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    mbar_init(bar(B_OFULL), 1);
    mbar_init(bar(B_OEMPTY), R::kCompute);
    mbar_init(bar(B_DRAIN), 1);      // S issuer's exit drain
    mbar_init(bar(B_DRAIN + 1), 1);  // PV issuer's exit drain
    mbar_init(bar(B_HOLD), 1);       // test hook: nothing arrives on it
    // rotated Q and K tiles (rotary embedding): one arrival per compute warp
    for (int s = 0; s < 2; ++s) mbar_init(bar(B_QREADY + s), R::kCompute / 32);
    for (int s = 0; s < NK; ++s) mbar_init(bar(B_KREADY + s), R::kCompute / 32);
    // work item ring: the Q/K producer claims; the V producer, both issuers and every
    // compute warp read
    for (int s = 0; s < kFeedSlots; ++s) {
      mbar_init(bar(B_FEEDFULL + s), 1);
      mbar_init(bar(B_FEEDEMPTY + s), 3 + R::kCompute / 32);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == kSWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // SiLU/L items may be claimed from the launch's counter as CTAs become free (the
  // scheduler decides per list).  The softmax kernels keep the fixed assignment: their
  // workloads' items are short, and the feed's registers would cost them spills; so do
  // the rotary kernels, whose compute warps look ahead in the list.
  constexpr bool kDyn = !ROPE && ACT != kActSoftmax;
  static_assert(B_FEEDEMPTY == B_FEEDFULL + kFeedSlots, "feed ring barriers");
  const FeedRing ring{bar(B_FEEDFULL), raw + L::FEED_OFF};
  Feed<kDyn> feed;
  feed.init(ring, list, &hdr->claim[kClaimFwd], n_items);

  // Rotary embedding of Q and K (BlockAttention): the compute warps rotate each item's Q
  // and K tiles in shared memory once they have landed and signal them ready; the S
  // issuer waits for that instead of the loads.  Its items are blocks of at most 64
  // rows, so each has exactly one step; the compute warps rotate the next item's tiles
  // before they turn to the current item's scores, while its S product runs.
  constexpr bool rope = ROPE;
  if (warp == kProducerWarp || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers
    // warp 8: each item's Q tile, then K(0), K(1), ...; warp 11: V(0), V(1), ...
    // Two threads, so that neither ring waits behind a load of the other.
    if (lane == 0) {
      const bool qk = warp == kProducerWarp;
      if (qk) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      } else {
        tma_prefetch_desc(&tm_v);
      }
      uint32_t t_it = 0, q_it = 0;
      bool ok = true;
      FeedClaimer<kDyn> claimer;  // the Q/K thread claims, the V thread reads
      claimer.init(ring, list, &hdr->claim[kClaimFwd], n_items);
      WorkItem w;
      while (ok && (qk ? claimer.claim(w, abort, status) : feed.take(w, false, true, abort, status))) {
        const int n = w.cost;
        if (n == 0) continue;
        if (qk) {
          const uint32_t qs = q_it % L::NQB;
          if (!mbar_wait(bar(B_QEMPTY + qs), ((q_it / L::NQB) & 1) ^ 1, abort, status)) break;
          mbar_expect_tx(bar(B_QFULL + qs), L::Q_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::Q_OFF + qs * L::Q_BYTES + a * 16384, &tm_q, w.h * DQK + a * 64,
                        w.q0 + w.tile * BM, bar(B_QFULL + qs));
          ++q_it;
        }
        for (int j = 0; j < n; ++j, ++t_it) {
          if (qk) {
            const uint32_t st = t_it % NK;
            if (!mbar_wait(bar(B_KEMPTY + st), ((t_it / NK) & 1) ^ 1, abort, status)) { ok = false; break; }
            mbar_expect_tx(bar(B_KFULL + st), L::K_BYTES);
#pragma unroll
            for (int a = 0; a < DQK / 64; ++a)
              tma_load_2d(sb + L::K_OFF + st * L::K_BYTES + a * 16384, &tm_k, w.h * DQK + a * 64,
                          w.k0 + j * BN, bar(B_KFULL + st));
          } else {
            const uint32_t st = t_it % NV;
            if (!mbar_wait(bar(B_VEMPTY + st), ((t_it / NV) & 1) ^ 1, abort, status)) { ok = false; break; }
            mbar_expect_tx(bar(B_VFULL + st), L::V_BYTES);
#pragma unroll
            for (int a = 0; a < DV / 64; ++a)
              tma_load_2d(sb + L::V_OFF + st * L::V_BYTES + a * 16384, &tm_v, w.h * DV + a * 64,
                          w.k0 + j * BN, bar(B_VFULL + st));
          }
        }
      }
      // every load issued has landed before the CTA leaves (also after giving up)
      if (qk) {
        drain_ring(bar(B_QFULL), L::NQB, q_it, status);
        drain_ring(bar(B_KFULL), NK, t_it, status);
      } else {
        drain_ring(bar(B_VFULL), NV, t_it, status);
      }
    }
    __syncwarp();
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ S = Q K^T issuer
    // An MMA issue occupies the issuing thread for most of the MMA's own duration
    // and the tensor pipe queues only a few, so the S and PV products come from two
    // threads: the waits and commits of one overlap the other's MMAs.
    {  // the whole warp runs the issuer loop; one elected lane issues
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      uint32_t k_it = 0, q_it = 0, gs = 0;
      bool ok = true;
      if (*(volatile int*)&g_test_hold) ok = mbar_wait(bar(B_HOLD), 0, abort, status);
      WorkItem w;
      while (ok && feed.take(w, true, true, abort, status)) {
        const int n = w.cost;
        if (n == 0) continue;
        const uint32_t qs = q_it % L::NQB;
        if (!mbar_wait(bar((rope ? B_QREADY : B_QFULL) + qs), (q_it / L::NQB) & 1, abort, status)) break;
        const uint32_t q_tile = sb + L::Q_OFF + qs * L::Q_BYTES;
        for (int i = 0; i < n; ++i, ++gs, ++k_it) {
          // S(gs) goes into the buffer of S(gs - 2): free once the softmax has written P(gs - 2)
          const uint32_t b = gs & 1, kst = k_it % NK;
          if (!mbar_wait(bar(B_PFULL + b), ((gs >> 1) & 1) ^ 1, abort, status) ||
              !mbar_wait(bar((rope ? B_KREADY : B_KFULL) + kst), (k_it / NK) & 1, abort, status)) {
            ok = false;
            break;
          }
          __syncwarp();  // converged for elect.sync
          tc_fence_after();
          const uint32_t k_tile = sb + L::K_OFF + kst * L::K_BYTES;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16(tmem + T_S + b * 128, sw128_desc(q_tile + off, 16, 1024),
                     sw128_desc(k_tile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL + b));
          mma_commit(bar(B_KEMPTY + kst));
          if (i == n - 1) mma_commit(bar(B_QEMPTY + qs));  // last use of this Q tile
        }
        ++q_it;
      }
      __syncwarp();
      mma_drain(bar(B_DRAIN), status);  // every MMA issued has completed
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ O += P V issuer
    {  // the whole warp runs the issuer loop; one elected lane issues
      constexpr uint32_t idesc_o = idesc_bf16(BM, DV, 0, 1);
      uint32_t v_it = 0, o_it = 0, gs = 0;
      bool ok = true;
      WorkItem w;
      while (ok && feed.take(w, true, true, abort, status)) {
        const int n = w.cost;
        if (n == 0) continue;
        for (int j = 0; j < n; ++j, ++gs, ++v_it) {
          const uint32_t b = gs & 1, vst = v_it % NV;
          if (!mbar_wait(bar(B_PFULL + b), (gs >> 1) & 1, abort, status) ||
              !mbar_wait(bar(B_VFULL + vst), (v_it / NV) & 1, abort, status) ||
              (j == 0 && !mbar_wait(bar(B_OEMPTY), (o_it & 1) ^ 1, abort, status))) {
            ok = false;
            break;
          }
          __syncwarp();  // converged for elect.sync
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bd = sw128_desc(sb + L::V_OFF + vst * L::V_BYTES + kk * 2048, 16384, 1024);
            mma_bf16_tmem_a(tmem + T_O, tmem + T_P + b * 64 + kk * 8, bd, idesc_o,
                            (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_PEMPTY + b));
          mma_commit(bar(B_VEMPTY + vst));
          if (j == n - 1) mma_commit(bar(B_OFULL));
        }
        if (!ok) break;
        ++o_it;
      }
      __syncwarp();
      mma_drain(bar(B_DRAIN + 1), status);  // every MMA issued has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int grp = warp >> 2;             // key columns [grp*HC, grp*HC+HC) of each step
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = row of the tile
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    float* red = reinterpret_cast<float*>(smem_raw + L::RED_OFF);  // [2 steps][128 rows][2]
    uint32_t p_it = 0, o_it = 0, l_it = 0;  // p_it: global step (S / P buffer p_it & 1)
    bool ok = true;
    // The output of an item (O from TMEM to HBM) is written after the next item's
    // first P, when its last PV product has long completed; the next item's first
    // PV waits for it (OEMPTY).  The row statistics are settled before that.
    bool pend = false, pend_row_ok = false;
    int64_t pend_orow = 0;
    float pend_norm = 0.f, pend_lse = 0.f;
    auto epilogue = [&]() -> bool {
      if (!mbar_wait(bar(B_OFULL), o_it & 1, abort, status)) return false;
      ++o_it;
      tc_fence_after();
      float ov[OC];
      tmem_ld<OC>(tmem + lane_base + T_O + grp * OC, ov);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_OEMPTY));
      if (pend_row_ok) {
        store_bf16<OC>(out + pend_orow * DV + grp * OC, ov, pend_norm);
        if (ACT == kActSoftmax && grp == 0 && lse != nullptr) lse[pend_orow] = pend_lse;
      }
      pend = false;
      return true;
    };
    // rotary embedding: the next non-empty item to rotate (list index) and the count of
    // items rotated so far (which fixes its Q and K stages)
    int rot_next = blockIdx.x;
    uint32_t rot_cnt = 0;
    if constexpr (ROPE) {
      if (!fwd_rotate_next<DQK, NK, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp, R::kCompute / 32,
                                        lane, abort, status))
        ok = false;
    }
    WorkItem w;
    while (ok && feed.take(w, true, true, abort, status)) {
      const int n = w.cost, h = w.h;
      const int Lq = w.lq, Lk = w.lk;
      if (rope && n > 1) {  // the rotary kernels take items of one step only
        if (lane == 0) atomicExch(status, (int)JFA_ERR_UNSUPPORTED);
        *abort = 1;
        ok = false;
        break;
      }
      // the next item's Q and K tiles, while S of this item runs (its rings are deep
      // enough that they have landed)
      if constexpr (ROPE) {
        if (n > 0 && !fwd_rotate_next<DQK, NK, L>(rot_next, rot_cnt, list, n_items, raw, sb, p, warp,
                                                  R::kCompute / 32, lane, abort, status)) {
          ok = false;
          break;
        }
      }
      const int i = w.tile * BM + r;
      const float inv_len = 1.0f / (float)max(Lq, 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++p_it) {
        const uint32_t b = p_it & 1;
        if (!mbar_wait(bar(B_SFULL + b), (p_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t s_tm = tmem + lane_base + T_S + b * 128 + grp * HC;
        float sv[HC];
        tmem_ld<HC>(s_tm, sv);
        tmem_wait_ld();
        const int kb = j * BN + grp * HC;
        int nvalid = Lk - kb;
        if (CAUSAL) nvalid = min(nvalid, i - kb + 1);
        if (p.block_mask > 0 && (kb ^ i) >= p.block_mask) nvalid = 0;  // another block's keys
        if (nvalid < HC) {
#pragma unroll
          for (int k = 0; k < HC; ++k) sv[k] -= k < nvalid ? 0.f : shift_raw;
        }
        float alpha = 1.f;
        bool rescale = false;
        if (ACT == kActSoftmax) {
          // row max of the raw scores (scale > 0): partial over this half, then exchanged
          float m0 = fmaxf(sv[0], sv[1]), m1 = fmaxf(sv[2], sv[3]);
#pragma unroll
          for (int k = 4; k < HC; k += 4) {  // HC is a multiple of 4
            m0 = fmax3(m0, sv[k], sv[k + 1]);
            m1 = fmax3(m1, sv[k + 2], sv[k + 3]);
          }
          float* rb = red + (p_it & 1) * (BM * 2);
          rb[r * 2 + grp] = fmaxf(m0, m1);
          mbar_arrive(bar(B_RED + (p_it & 1)));
          if (!mbar_wait(bar(B_RED + (p_it & 1)), (p_it >> 1) & 1, abort, status)) { ok = false; break; }
          const float mt = fmaxf(rb[r * 2], rb[r * 2 + 1]) * c_score;
          if (j == 0) {
            m = mt;
          } else {
            // lazy rescaling: move the reference max only when it grows by > 2^8
            const bool need = mt > m + kRescaleLog2;
            rescale = __any_sync(0xffffffffu, need);
            if (need) {
              alpha = ex2(m - mt);
              m = mt;
            }
          }
          l *= alpha;
        }
        // P = exp2(s c - m) or SiLU(s c)/L as packed bf16 pairs
        const float2 cc = make_float2(c_score, c_score);
        const float2 nm = make_float2(-m, -m);
        const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
        const float2 il = make_float2(inv_len, inv_len);
        float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
        uint32_t pk[HC / 2];
#pragma unroll
        for (int c = 0; c < HC / 2; ++c) {
          const float2 x = make_float2(sv[2 * c], sv[2 * c + 1]);
          float2 pv;
          if (ACT == kActSoftmax) {
            const float2 e = ffma2(x, cc, nm);
            pv = make_float2(ex2(e.x), ex2(e.y));
            if (c & 1) rs1 = fadd2(rs1, pv); else rs0 = fadd2(rs0, pv);
          } else {
            // SiLU(u)/L with u = s c: h = u/2, P = h (1 + tanh h) / L
            const float2 hh = fmul2(x, hc);
            const float2 t = make_float2(tanh_approx(hh.x), tanh_approx(hh.y));
            pv = fmul2(hh, ffma2(t, il, il));
          }
          pk[c] = pack_bf16(pv.x, pv.y);
        }
        if (ACT == kActSoftmax) {
          const float2 rr = fadd2(rs0, rs1);
          l += rr.x + rr.y;
        }
        // P buffer b is free once PV(p_it - 2) has completed; rescaling O also needs
        // PV(p_it - 1) complete.
        if (!mbar_wait(bar(B_PEMPTY + b), ((p_it >> 1) & 1) ^ 1, abort, status) ||
            (rescale && !mbar_wait(bar(B_PEMPTY + (b ^ 1)), ((p_it - 1) >> 1) & 1, abort, status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if constexpr (ACT == kActSoftmax) {
          if (rescale) {
            float ov[32];
#pragma unroll
            for (int c = 0; c < OC / 32; ++c) {
              const uint32_t o_tm = tmem + lane_base + T_O + grp * OC + 32 * c;
              tmem_ld32(o_tm, ov);
              tmem_wait_ld();
#pragma unroll
              for (int t = 0; t < 32; ++t) ov[t] *= alpha;
              tmem_st32(o_tm, ov);
            }
          }
        }
        // P of this group's keys, packed: HC/2 columns at the group's offset, so that the
        // P buffer holds the step's 128 keys in order
        if constexpr (HC == 64)
          tmem_st32(tmem + lane_base + T_P + b * 64 + grp * (HC / 2), reinterpret_cast<const float*>(pk));
        else
          tmem_st16(tmem + lane_base + T_P + b * 64 + grp * (HC / 2), pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + b));
        if (pend && !epilogue()) { ok = false; break; }
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue (deferred)
      const bool row_ok = i < Lq;
      const int64_t orow = ((int64_t)w.q0 + i) * p.heads + h;
      if (n > 0) {
        float lt = l;
        if (ACT == kActSoftmax) {
          // Row sums are exchanged through the buffer of the item's last step: first
          // every thread confirms it has read that step's maxima, then the sums go in.
          float* rl = red + ((p_it - 1) & 1) * (BM * 2);
          mbar_arrive(bar(B_REDL));
          if (!mbar_wait(bar(B_REDL), l_it & 1, abort, status)) { ok = false; break; }
          rl[r * 2 + grp] = l;
          mbar_arrive(bar(B_REDL + 1));
          if (!mbar_wait(bar(B_REDL + 1), l_it & 1, abort, status)) { ok = false; break; }
          ++l_it;
          lt = rl[r * 2] + rl[r * 2 + 1];
        }
        if (pend && !epilogue()) { ok = false; break; }  // defensive: flushed after step 0
        pend = true;
        pend_row_ok = row_ok;
        pend_orow = orow;
        pend_norm = ACT == kActSoftmax ? (lt > 0.f ? 1.f / lt : 0.f) : 1.f;
        pend_lse = lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
      } else if (row_ok) {
        const float z[OC] = {0.f};
        store_bf16<OC>(out + orow * DV + grp * OC, z, 1.f);
        if (ACT == kActSoftmax && grp == 0 && lse != nullptr) lse[orow] = -INFINITY;
      }
    }
    if (ok && pend) ok = epilogue();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, int ACT, bool CAUSAL, bool ROPE = false>
cudaError_t launch_fwd_t(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, void* o, float* lse, const Workspace& ws,
                         cudaStream_t s) {
  auto kern = tc_fwd_kernel<DQK, DV, ACT, CAUSAL, ROPE>;
  constexpr uint32_t smem = FwdLayout<DQK, DV>::SMEM;
  constexpr int threads = FwdRoles<ACT>::kThreads;
  cudaError_t e = kernel_setup((const void*)kern, threads, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), threads, smem, s>>>(mq, mk, mv, p, (__nv_bfloat16*)o, lse, ws.hdr, ws.list_q);
  return cudaGetLastError();
}

template <int DQK, int DV>
cudaError_t launch_fwd_d(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, void* o, float* lse, const Workspace& ws,
                         cudaStream_t s) {
  if (p.rope != nullptr) {  // rotary embedding: softmax self-attention with Dqk = Dv only
    if constexpr (DQK == DV) {
      if (p.act == kActSoftmax)
        return p.causal ? launch_fwd_t<DQK, DV, kActSoftmax, true, true>(p, mq, mk, mv, o, lse, ws, s)
                        : launch_fwd_t<DQK, DV, kActSoftmax, false, true>(p, mq, mk, mv, o, lse, ws, s);
    }
    return cudaErrorInvalidValue;
  }
  if (p.act == kActSoftmax)
    return p.causal ? launch_fwd_t<DQK, DV, kActSoftmax, true>(p, mq, mk, mv, o, lse, ws, s)
                    : launch_fwd_t<DQK, DV, kActSoftmax, false>(p, mq, mk, mv, o, lse, ws, s);
  return p.causal ? launch_fwd_t<DQK, DV, kActSiluOverLen, true>(p, mq, mk, mv, o, lse, ws, s)
                  : launch_fwd_t<DQK, DV, kActSiluOverLen, false>(p, mq, mk, mv, o, lse, ws, s);
}

}  // namespace

cudaError_t tc_set_test_hold(int on) {
  const int v = on != 0;
  return cudaMemcpyToSymbol(g_test_hold, &v, sizeof(int));
}

bool tc_supports(int dim_qk, int dim_v) {
  return (dim_qk == 64 || dim_qk == 128) && (dim_v == 64 || dim_v == 128);
}

// Items are 128-row q-tiles; the cost is the number of 128-key steps.
SchedConfig tc_fwd_sched(const Problem&) { return SchedConfig{BM, BN, BN, BM, 1, 0, 0}; }

cudaError_t launch_tc_fwd(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, const Workspace& ws, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const void* dummy = q;
  if (!make_tile_map(&mq, q, p.total_q, (int64_t)p.heads * p.dim_qk, 64, BM) ||
      !make_tile_map(&mk, p.total_k > 0 ? k : dummy, p.total_k > 0 ? p.total_k : p.total_q,
                     (int64_t)p.heads * p.dim_qk, 64, BN) ||
      !make_tile_map(&mv, p.total_k > 0 ? v : dummy, p.total_k > 0 ? p.total_k : p.total_q,
                     (int64_t)p.heads * (p.total_k > 0 ? p.dim_v : p.dim_qk), 64, BN))
    return cudaErrorInvalidValue;
  if (p.dim_qk == 128 && p.dim_v == 128) return launch_fwd_d<128, 128>(p, mq, mk, mv, o, lse, ws, s);
  if (p.dim_qk == 128 && p.dim_v == 64) return launch_fwd_d<128, 64>(p, mq, mk, mv, o, lse, ws, s);
  if (p.dim_qk == 64 && p.dim_v == 128) return launch_fwd_d<64, 128>(p, mq, mk, mv, o, lse, ws, s);
  if (p.dim_qk == 64 && p.dim_v == 64) return launch_fwd_d<64, 64>(p, mq, mk, mv, o, lse, ws, s);
  return cudaErrorInvalidValue;
}

}  // namespace jfa
