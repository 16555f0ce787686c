// Tensor-core jagged attention forward for sm_103a: TMA + tcgen05 + TMEM.
//
// Method: Jagged Flash Attention bullet of the Meta GEM MFU write-up
// (piletech.kr/articles/112134, details): attention computed directly on the
// jagged buffers, masked by subtraction, persistent kernel scheduling with
// specialised warps; Generalized Dot-Product Attention bullet: the same
// pipeline with a non-softmax activation (here SiLU(s)/L).
//
// One persistent CTA per SM walks the scheduler's heavy-first list of items;
// an item is a PAIR of adjacent 128-row q-tiles of one (sequence, head),
// held in two slots that share every K/V tile:
//   warps 0..3  softmax warpgroup of slot 0, one query row per thread (TMEM lane)
//   warps 4..7  softmax warpgroup of slot 1
//   warp 8      TMA producer: both Q tiles once per item, K and V tiles of 128
//               keys into an NS-stage ring, straight from the jagged [T, H*D]
//               buffers (rows past a sequence belong to its neighbour and are
//               masked; rows past the buffer are zero-filled by TMA)
//   warp 9      TMEM owner and MMA issuer (one lane).  Per key step j it issues,
//               slot by slot, O_s += P_s(j-1) V(j-1) and S_s(j) = Q_s K(j)^T, so
//               the tensor pipe works on one slot while the other slot's
//               warpgroup turns its S into P (ping-pong).
// Softmax warpgroup, per step: tcgen05.ld of its S row, scale to log2 units,
// subtract a finite shift from masked columns, online max with lazy rescaling
// of O (only when the running max grows by more than 2^8), exp2, row sum,
// and P as packed bf16 back into TMEM over the S columns; the PV product reads
// P straight from TMEM.  Epilogue: O / l -> bf16, lse = (m + log2 l) ln 2.
// TMEM per slot s: S (and P) at columns [256 s, 256 s + 128), O at
// [256 s + 128, 256 s + 128 + Dv).  MMAs issued by one thread execute in
// order, so S_s(j) overwriting P_s(j-1) is ordered after the PV that reads it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace jfa {
namespace {
using namespace tc;

constexpr int BM = 128;          // rows per slot (MMA M)
constexpr int BN = 128;          // keys per step (MMA N of S)
constexpr int kPair = 2 * BM;    // rows per item
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

template <int DQK, int DV>
struct FwdLayout {
  // K tiles are consumed one step before V tiles, so they get the deeper ring.
  static constexpr int NK = DQK == 64 ? 4 : 3;
  static constexpr int NV = DV == 64 ? 4 : (DQK == 64 ? 3 : 2);
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;  // one 128-row tile
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  static constexpr uint32_t Q_OFF = 0;                    // 2 slots
  static constexpr uint32_t K_OFF = Q_OFF + 2 * Q_BYTES;  // NK stages
  static constexpr uint32_t V_OFF = K_OFF + NK * K_BYTES; // NV stages
  static constexpr uint32_t BAR_OFF = V_OFF + NV * V_BYTES;
  // at least 120 KB so that exactly one CTA (which owns all of TMEM) fits per SM
  static constexpr uint32_t SMEM = (BAR_OFF + 512 + 1024) > 122880u ? (BAR_OFF + 512 + 1024) : 122880u;
};

// mbarrier slots (the K and V rings have up to 4 stages each)
enum : uint32_t {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = 6, B_VFULL = 10, B_VEMPTY = 14,
  B_SFULL = 18, B_PFULL = 20, B_OFULL = 22, B_OEMPTY = 24, B_COUNT = 26
};

template <int DQK, int DV, int ACT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const Problem p,
              __nv_bfloat16* __restrict__ out, float* __restrict__ lse, WsHeader* hdr,
              const WorkItem* __restrict__ list) {
  using L = FwdLayout<DQK, DV>;
  constexpr int NK = L::NK, NV = L::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + L::BAR_OFF;
  auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = (uint32_t*)(smem + L::BAR_OFF + 8 * B_COUNT);
  volatile int* abort = (volatile int*)(smem + L::BAR_OFF + 8 * B_COUNT + 4);
  int* status = &hdr->status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_q;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_PFULL + s), 128);
      mbar_init(bar(B_OFULL + s), 1);
      mbar_init(bar(B_OEMPTY + s), 128);
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      bool ok = true;
      WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = nxt;  // prefetched one item ahead
        if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
        const int n = w.cost;
        if (n == 0) continue;
        const int h = w.h, row0 = w.tile * kPair;
        const bool two = row0 + BM < w.lq;
        if (!mbar_wait(bar(B_QEMPTY), (q_it & 1) ^ 1, abort, status)) break;
        mbar_expect_tx(bar(B_QFULL), (two ? 2u : 1u) * L::Q_BYTES);
        for (int s = 0; s < (two ? 2 : 1); ++s) {
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::Q_OFF + s * L::Q_BYTES + a * 16384, &tm_q, h * DQK + a * 64,
                        w.q0 + row0 + s * BM, bar(B_QFULL));
        }
        ++q_it;
        // K(j) is needed one step before V(j): issue K(j), then V(j-1)
        for (int j = 0; j <= n && ok; ++j) {
          if (j < n) {
            const uint32_t st = k_it % NK;
            if (!mbar_wait(bar(B_KEMPTY + st), ((k_it / NK) & 1) ^ 1, abort, status)) { ok = false; break; }
            mbar_expect_tx(bar(B_KFULL + st), L::K_BYTES);
#pragma unroll
            for (int a = 0; a < DQK / 64; ++a)
              tma_load_2d(sb + L::K_OFF + st * L::K_BYTES + a * 16384, &tm_k, h * DQK + a * 64,
                          w.k0 + j * BN, bar(B_KFULL + st));
            ++k_it;
          }
          if (j > 0) {
            const uint32_t st = v_it % NV;
            if (!mbar_wait(bar(B_VEMPTY + st), ((v_it / NV) & 1) ^ 1, abort, status)) { ok = false; break; }
            mbar_expect_tx(bar(B_VFULL + st), L::V_BYTES);
#pragma unroll
            for (int a = 0; a < DV / 64; ++a)
              tma_load_2d(sb + L::V_OFF + st * L::V_BYTES + a * 16384, &tm_v, h * DV + a * 64,
                          w.k0 + (j - 1) * BN, bar(B_VFULL + st));
            ++v_it;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16(BM, DV, 0, 1);
      uint32_t k_it = 0, v_it = 0, q_it = 0;
      uint32_t s_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
      bool ok = true;
      WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = nxt;
        if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
        const int n = w.cost;
        if (n == 0) continue;
        const int row0 = w.tile * kPair;
        const bool two = row0 + BM < w.lq;
        // key steps of each slot: slot 1 needs n, slot 0 one fewer on the causal diagonal
        int ns[2];
        ns[0] = CAUSAL ? min(n, (min(w.lk, row0 + BM) + BN - 1) / BN) : n;
        ns[1] = two ? n : 0;
        if (!mbar_wait(bar(B_QFULL), q_it & 1, abort, status)) break;
        tc_fence_after();
        for (int j = 0; j <= n && ok; ++j) {
          const uint32_t kst = k_it % NK, vst = v_it % NV;
          if (j < n) {
            if (!mbar_wait(bar(B_KFULL + kst), (k_it / NK) & 1, abort, status)) { ok = false; break; }
            tc_fence_after();
          }
          if (j > 0) {
            if (!mbar_wait(bar(B_VFULL + vst), (v_it / NV) & 1, abort, status)) { ok = false; break; }
            tc_fence_after();
          }
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint32_t s_tm = tmem + s * 256;
            if (j > 0 && j - 1 < ns[s]) {
              // O_s += P_s(j-1) V(j-1), P read from TMEM
              if (!mbar_wait(bar(B_PFULL + s), (s_cnt[s] - 1) & 1, abort, status) ||
                  (j == 1 && !mbar_wait(bar(B_OEMPTY + s), (o_cnt[s] & 1) ^ 1, abort, status))) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk) {
                const uint64_t bd = sw128_desc(sb + L::V_OFF + vst * L::V_BYTES + kk * 2048, 16384, 1024);
                mma_bf16_tmem_a(s_tm + 128, s_tm + kk * 8, bd, idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
              }
              if (j == ns[s]) {
                mma_commit(bar(B_OFULL + s));
                ++o_cnt[s];
              }
            }
            if (j < ns[s]) {
              // S_s(j) = Q_s K(j)^T
#pragma unroll
              for (int kk = 0; kk < DQK / 16; ++kk) {
                const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint64_t ad = sw128_desc(sb + L::Q_OFF + s * L::Q_BYTES + off, 16, 1024);
                const uint64_t bd = sw128_desc(sb + L::K_OFF + kst * L::K_BYTES + off, 16, 1024);
                mma_bf16(s_tm, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
              }
              mma_commit(bar(B_SFULL + s));
              ++s_cnt[s];
            }
          }
          if (!ok) break;
          if (j < n) {
            mma_commit(bar(B_KEMPTY + kst));  // both slots' S(j) issued
            if (j == n - 1) mma_commit(bar(B_QEMPTY));
            ++k_it;
          }
          if (j > 0) {
            mma_commit(bar(B_VEMPTY + vst));  // both slots' PV(j-1) issued
            ++v_it;
          }
        }
        ++q_it;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int slot = warp >> 2;
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = row of the slot's tile
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t s_tm = tmem + slot * 256 + lane_base;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    uint32_t s_cnt = 0, o_cnt = 0;
    bool ok = true;
    WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const WorkItem w = nxt;
      if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
      const int n = w.cost, h = w.h;
      const int row0 = w.tile * kPair + slot * BM;  // first row of this slot's tile
      if (row0 >= w.lq) continue;                   // slot empty for this item
      const int Lq = w.lq, Lk = w.lk;
      const int ns = (slot == 0 && CAUSAL) ? min(n, (min(Lk, row0 + BM) + BN - 1) / BN) : n;
      const int i = row0 + r;
      const float inv_len = 1.0f / (float)max(Lq, 1);
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < ns; ++j) {
        if (!mbar_wait(bar(B_SFULL + slot), s_cnt & 1, abort, status)) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        float sv[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(s_tm + 32 * c, sv + 32 * c);
        tmem_wait_ld();
        const int kb = j * BN;
        int nvalid = Lk - kb;
        if (CAUSAL) nvalid = min(nvalid, i - kb + 1);
        float alpha = 1.f;  // rescale factor of O for this step (softmax only)
        bool rescale = false;
        if (nvalid < BN) {
          // partial tile: move masked raw scores down by a finite shift (in raw units,
          // so that after scaling the shift is kMaskShift)
#pragma unroll
          for (int k = 0; k < BN; ++k) sv[k] -= k < nvalid ? 0.f : shift_raw;
        }
        if (ACT == kActSoftmax) {
          // row max of the raw scores (scale > 0), two independent 3-input chains
          float m0 = fmaxf(sv[0], sv[1]), m1 = fmaxf(sv[2], sv[3]);
#pragma unroll
          for (int k = 4; k < BN; k += 4) {  // BN is a multiple of 4: last group is BN-4..BN-1
            m0 = fmax3(m0, sv[k], sv[k + 1]);
            m1 = fmax3(m1, sv[k + 2], sv[k + 3]);
          }
          const float mt = fmaxf(m0, m1) * c_score;
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
        // P = exp2(s c - m) or SiLU(s c)/L, packed bf16 pairs over the first 64 S
        // columns, written 64 values at a time so the fp32 scores die as they go.
        const float2 cc = make_float2(c_score, c_score);
        const float2 nm = make_float2(-m, -m);
        const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
        const float2 il = make_float2(inv_len, inv_len);
        float2 rs0 = make_float2(0.f, 0.f), rs1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = make_float2(sv[half * 64 + 2 * c], sv[half * 64 + 2 * c + 1]);
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
          tmem_st32(s_tm + 32 * half, reinterpret_cast<const float*>(pk));
        }
        if (ACT == kActSoftmax) {
          const float2 r = fadd2(rs0, rs1);
          l += r.x + r.y;
        }
        if (rescale) {
          // O_s already holds every PV issued before this S (in-order MMAs).
          float ov[32];
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            tmem_ld32(s_tm + 128 + 32 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) ov[t] *= alpha;
            tmem_st32(s_tm + 128 + 32 * c, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + slot));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      const bool row_ok = i < Lq;
      const int64_t orow = ((int64_t)w.q0 + i) * p.heads + h;
      if (ns > 0) {
        if (!mbar_wait(bar(B_OFULL + slot), o_cnt & 1, abort, status)) { ok = false; break; }
        ++o_cnt;
        tc_fence_after();
        const float norm = ACT == kActSoftmax ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
        float ov[32];
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          tmem_ld32(s_tm + 128 + 32 * c, ov);
          tmem_wait_ld();
          if (row_ok) store32_bf16(out + orow * DV + 32 * c, ov, norm);
        }
        tc_fence_before();
        mbar_arrive(bar(B_OEMPTY + slot));
        if (ACT == kActSoftmax && row_ok && lse != nullptr)
          lse[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(out + orow * DV);
#pragma unroll
        for (int t = 0; t < DV / 8; ++t) dst[t] = make_uint4(0, 0, 0, 0);
        if (ACT == kActSoftmax && lse != nullptr) lse[orow] = -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, int ACT, bool CAUSAL>
cudaError_t launch_fwd_t(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, void* o, float* lse, const Workspace& ws,
                         cudaStream_t s) {
  auto kern = tc_fwd_kernel<DQK, DV, ACT, CAUSAL>;
  constexpr uint32_t smem = FwdLayout<DQK, DV>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreads, smem, s>>>(mq, mk, mv, p, (__nv_bfloat16*)o, lse, ws.hdr, ws.list_q);
  return cudaGetLastError();
}

template <int DQK, int DV>
cudaError_t launch_fwd_d(const Problem& p, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, void* o, float* lse, const Workspace& ws,
                         cudaStream_t s) {
  if (p.act == kActSoftmax)
    return p.causal ? launch_fwd_t<DQK, DV, kActSoftmax, true>(p, mq, mk, mv, o, lse, ws, s)
                    : launch_fwd_t<DQK, DV, kActSoftmax, false>(p, mq, mk, mv, o, lse, ws, s);
  return p.causal ? launch_fwd_t<DQK, DV, kActSiluOverLen, true>(p, mq, mk, mv, o, lse, ws, s)
                  : launch_fwd_t<DQK, DV, kActSiluOverLen, false>(p, mq, mk, mv, o, lse, ws, s);
}

}  // namespace

bool tc_supports(int dim_qk, int dim_v) {
  return (dim_qk == 64 || dim_qk == 128) && (dim_v == 64 || dim_v == 128);
}

// Items are pairs of 128-row q-tiles; the cost is the number of 128-key steps.
SchedConfig tc_fwd_sched(const Problem&) { return SchedConfig{kPair, BN, BN, BM, 1, 0, 0}; }

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
