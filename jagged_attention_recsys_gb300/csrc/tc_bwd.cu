// Tensor-core jagged attention backward for sm_103a: TMA + tcgen05 + TMEM, no atomics.
//
// Method: Jagged Flash Attention bullet of the Meta GEM MFU write-up
// (piletech.kr/articles/112134, details): the backward is parallelised
// without atomic operations.  Every gradient element is produced by exactly
// one CTA in one store:
//   * row pass      rowstat[h][t] = (lse * log2 e, D = <dO, O>), head-major so
//                   a 64-row block of one head is contiguous;
//   * dK/dV pass    one item = (sequence, head, 128-key tile).  TMEM holds
//                   dK, dV and two buffers of S^T = K Q^T and dP^T = V dO^T
//                   for 64-row query steps; per step the compute warpgroup
//                   (one key per thread) forms P^T and dS^T = P^T (dP^T - D)
//                   into swizzled smem and the MMA lane issues dV += P^T dO and
//                   dK += dS^T Q (Q and dO read MN-major from the same tiles);
//   * dQ pass       one item = (sequence, head, 128-row query tile).  TMEM holds
//                   dQ and two buffers of S = Q K^T, dP = dO V^T over 64-key
//                   steps; the compute warpgroup (one row per thread) forms dS
//                   and the MMA lane issues dQ += dS K.
// The SiLU/L variant has no lse and no D: P = SiLU(u)/L and
// dS = dP SiLU'(u)/L with u = scale s.  Masking is by subtraction as in the
// forward; masked (query, key) pairs contribute exact zeros.
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

constexpr int kThreads = 192;
constexpr int TILE = 128;  // keys per dK/dV item, rows per dQ item (MMA M)
constexpr int STEP = 64;   // query rows per dK/dV step, keys per dQ step (MMA N)
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ row pass
// rowstat[h * T + t] = (lse[t, h] * log2 e, sum_c dO[t, h, c] * O[t, h, c]).
template <int DV>
__global__ void __launch_bounds__(256)
rowstat_kernel(int64_t total, int heads, const __nv_bfloat16* __restrict__ o,
               const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
               float2* __restrict__ rowstat) {
  constexpr int TPR = DV / 8;  // threads per (row, head), 8 elements each
  const int64_t rows = total * heads;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = gid; idx < rows * TPR; idx += stride) {
    const int64_t row = idx / TPR;
    const int part = (int)(idx % TPR);
    const uint4 a = reinterpret_cast<const uint4*>(o + row * DV)[part];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * DV)[part];
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
    if (part == 0) {
      const int64_t t = row / heads;
      const int h = (int)(row % heads);
      rowstat[(int64_t)h * total + t] = make_float2(lse[row] * kLog2e, acc);
    }
  }
}

// Shared pieces ---------------------------------------------------------------
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* x, float f) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float* y = x + 8 * t;
    d[t] = make_uint4(pack_bf16(y[0] * f, y[1] * f), pack_bf16(y[2] * f, y[3] * f),
                      pack_bf16(y[4] * f, y[5] * f), pack_bf16(y[6] * f, y[7] * f));
  }
}

// =============================================================================
// dK / dV pass
// =============================================================================
// Q/dO steps are staged in an NQ-deep ring so the loads of later query steps
// are in flight while the current ones are computed.  P^T and dS^T are written
// back into TMEM as packed bf16 over the first 32 columns of the S^T and dP^T
// buffers they were computed from, and the dV / dK products read them from
// there (A operand in TMEM).
template <int DQK, int DV>
struct KvLayout {
  static constexpr int NKV = 2;                           // K/V tiles: current and next item
  static constexpr int NQ = DQK + DV > 192 ? 3 : (DQK + DV > 128 ? 4 : 8);  // Q/dO ring stages
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;   // 128 keys
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  static constexpr uint32_t Q_BYTES = DQK / 64 * 8192;    // 64 rows
  static constexpr uint32_t O_BYTES = DV / 64 * 8192;
  static constexpr uint32_t K_OFF = 0;                     // NKV stages
  static constexpr uint32_t V_OFF = K_OFF + NKV * K_BYTES; // NKV stages
  static constexpr uint32_t Q_OFF = V_OFF + NKV * V_BYTES; // NQ stages
  static constexpr uint32_t O_OFF = Q_OFF + NQ * Q_BYTES;  // NQ stages (dO)
  static constexpr uint32_t RS_OFF = O_OFF + NQ * O_BYTES; // NQ stages x 64 float2
  static constexpr uint32_t BAR_OFF = RS_OFF + NQ * STEP * 8;
  // at least 120 KB so that exactly one CTA (which owns all of TMEM) fits per SM
  static constexpr uint32_t SMEM = (BAR_OFF + 512 + 1024) > 122880u ? (BAR_OFF + 512 + 1024) : 122880u;
};

enum : uint32_t {
  KV_KVFULL = 0, KV_KVEMPTY = 2, KV_QFULL = 4, KV_RSFULL = 12, KV_QEMPTY = 20, KV_SFULL = 28,
  KV_PFULL = 30, KV_ACCFULL = 32, KV_ACCEMPTY = 33, KV_COUNT = 34
};

template <int DQK, int DV, int ACT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
tc_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
               const Problem p, const float2* __restrict__ rowstat,
               __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, WsHeader* hdr,
               const WorkItem* __restrict__ list) {
  using L = KvLayout<DQK, DV>;
  constexpr int NQ = L::NQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + L::BAR_OFF;
  auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = (uint32_t*)(smem + L::BAR_OFF + 8 * KV_COUNT);
  volatile int* abort = (volatile int*)(smem + L::BAR_OFF + 8 * KV_COUNT + 4);
  int* status = &hdr->status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NKV; ++s) {
      mbar_init(bar(KV_KVFULL + s), 1);
      mbar_init(bar(KV_KVEMPTY + s), 1);
    }
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar(KV_QFULL + s), 1);
      mbar_init(bar(KV_RSFULL + s), 32);
      mbar_init(bar(KV_QEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(KV_SFULL + s), 1);
      mbar_init(bar(KV_PFULL + s), 128);
    }
    mbar_init(bar(KV_ACCFULL), 1);
    mbar_init(bar(KV_ACCEMPTY), 128);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: dK [0,128), dV [128,256), S^T/P^T [256 + 64 b), dP^T/dS^T [384 + 64 b)
  constexpr uint32_t T_DK = 0, T_DV = 128, T_S = 256, T_DP = 384;

  if (warp == 0) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
    }
    uint32_t kv_it = 0, q_it = 0;
    bool ok = true;
    WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const WorkItem w = nxt;  // prefetched one item ahead
      if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
      const int n = w.cost;
      if (n == 0) continue;
      const int h = w.h, key0 = w.tile * TILE;
      const int64_t q0 = w.q0, k0 = w.k0;
      const int Lq = w.lq;
      if (lane == 0) {
        const uint32_t ks = kv_it % L::NKV;
        ok = mbar_wait(bar(KV_KVEMPTY + ks), ((kv_it / L::NKV) & 1) ^ 1, abort, status);
        if (ok) {
          mbar_expect_tx(bar(KV_KVFULL + ks), L::K_BYTES + L::V_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::K_OFF + ks * L::K_BYTES + a * 16384, &tm_k, h * DQK + a * 64,
                        (int32_t)(k0 + key0), bar(KV_KVFULL + ks));
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::V_OFF + ks * L::V_BYTES + a * 16384, &tm_v, h * DV + a * 64,
                        (int32_t)(k0 + key0), bar(KV_KVFULL + ks));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      ++kv_it;
      const int qs0 = CAUSAL ? key0 / STEP : 0;
      for (int j = 0; j < n; ++j, ++q_it) {
        const int i0 = (qs0 + j) * STEP;
        const uint32_t st = q_it % NQ, ph = (q_it / NQ) & 1;
        // row terms of this step: issue the global loads before waiting for the stage
        float2 rv[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int c = lane + 32 * t;
          rv[t] = make_float2(0.f, 0.f);
          if (ACT == kActSoftmax && i0 + c < Lq) rv[t] = rowstat[(int64_t)h * p.total_q + q0 + i0 + c];
        }
        ok = mbar_wait(bar(KV_QEMPTY + st), ph ^ 1, abort, status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        if (lane == 0) {
          mbar_expect_tx(bar(KV_QFULL + st), L::Q_BYTES + L::O_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::Q_OFF + st * L::Q_BYTES + a * 8192, &tm_q, h * DQK + a * 64,
                        (int32_t)(q0 + i0), bar(KV_QFULL + st));
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::O_OFF + st * L::O_BYTES + a * 8192, &tm_do, h * DV + a * 64,
                        (int32_t)(q0 + i0), bar(KV_QFULL + st));
        }
        // stage layout: 64 x (-lse * log2 e), then 64 x (-D)
        float* rs = reinterpret_cast<float*>(smem + L::RS_OFF + st * STEP * 8);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          rs[lane + 32 * t] = -rv[t].x;
          rs[STEP + lane + 32 * t] = -rv[t].y;
        }
        mbar_arrive(bar(KV_RSFULL + st));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(TILE, STEP, 0, 0);
      constexpr uint32_t idesc_dv = idesc_bf16(TILE, DV, 0, 1);
      constexpr uint32_t idesc_dk = idesc_bf16(TILE, DQK, 0, 1);
      uint32_t kv_it = 0, q_it = 0, s_it = 0, a_it = 0;
      bool ok = true;
      WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = nxt;
        if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
        const int n = w.cost;
        if (n == 0) continue;
        const uint32_t ks = kv_it % L::NKV;
        if (!mbar_wait(bar(KV_KVFULL + ks), (kv_it / L::NKV) & 1, abort, status)) break;
        tc_fence_after();
        const uint32_t k_tile = sb + L::K_OFF + ks * L::K_BYTES;
        const uint32_t v_tile = sb + L::V_OFF + ks * L::V_BYTES;
        uint32_t prev_stage = 0;
        for (int j = 0; j <= n && ok; ++j) {
          uint32_t cur_stage = 0;
          if (j < n) {
            // S^T(j) = K Q(j)^T and dP^T(j) = V dO(j)^T into buffer j % 2.  The buffer
            // held step j-2, whose P^T / dS^T were consumed by the dV / dK products
            // issued (in order) before this point.
            cur_stage = q_it % NQ;
            const uint32_t sbuf = s_it & 1;
            if (!mbar_wait(bar(KV_QFULL + cur_stage), (q_it / NQ) & 1, abort, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint64_t ad = sw128_desc(k_tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::Q_OFF + cur_stage * L::Q_BYTES + (kk >> 2) * 8192 +
                                                 (kk & 3) * 32, 16, 1024);
              mma_bf16(tmem + T_S + sbuf * STEP, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < DV / 16; ++kk) {
              const uint64_t ad = sw128_desc(v_tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::O_OFF + cur_stage * L::O_BYTES + (kk >> 2) * 8192 +
                                                 (kk & 3) * 32, 16, 1024);
              mma_bf16(tmem + T_DP + sbuf * STEP, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(KV_SFULL + sbuf));
            if (j == n - 1) mma_commit(bar(KV_KVEMPTY + ks));
            ++s_it;
            ++q_it;
          }
          if (j > 0) {
            // dV += P^T(j-1) dO(j-1), dK += dS^T(j-1) Q(j-1); A operands from TMEM
            const uint32_t pbuf = (s_it - (j < n ? 2 : 1)) & 1;
            const uint32_t pidx = s_it - (j < n ? 2 : 1);
            if (!mbar_wait(bar(KV_PFULL + pbuf), (pidx >> 1) & 1, abort, status) ||
                (j == 1 && !mbar_wait(bar(KV_ACCEMPTY), (a_it & 1) ^ 1, abort, status))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t acc = j > 1 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < STEP / 16; ++kk) {
              const uint64_t bd = sw128_desc(sb + L::O_OFF + prev_stage * L::O_BYTES + kk * 2048, 8192, 1024);
              mma_bf16_tmem_a(tmem + T_DV, tmem + T_S + pbuf * STEP + kk * 8, bd, idesc_dv,
                              (acc | (kk > 0)) ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < STEP / 16; ++kk) {
              const uint64_t bd = sw128_desc(sb + L::Q_OFF + prev_stage * L::Q_BYTES + kk * 2048, 8192, 1024);
              mma_bf16_tmem_a(tmem + T_DK, tmem + T_DP + pbuf * STEP + kk * 8, bd, idesc_dk,
                              (acc | (kk > 0)) ? 1u : 0u);
            }
            mma_commit(bar(KV_QEMPTY + prev_stage));
            if (j == n) mma_commit(bar(KV_ACCFULL));
          }
          prev_stage = cur_stage;
        }
        ++kv_it;
        ++a_it;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warpgroup
    const int r = 32 * (warp & 3) + lane;  // key of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
    const float2 one = make_float2(1.f, 1.f), half = make_float2(0.5f, 0.5f);
    uint32_t q_it = 0, s_it = 0, a_it = 0;
    bool ok = true;
    WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const WorkItem w = nxt;
      if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
      const int n = w.cost;
      const int h = w.h, key0 = w.tile * TILE;
      const int64_t k0 = w.k0;
      const int Lq = w.lq, Lk = w.lk;
      const int j = key0 + r;  // key index inside the sequence
      const float inv_len = 1.0f / (float)max(Lq, 1);
      const float2 il = make_float2(inv_len, inv_len);
      const int qs0 = CAUSAL ? key0 / STEP : 0;
      for (int step = 0; step < n; ++step, ++q_it) {
        const uint32_t sbuf = s_it & 1;
        if (!mbar_wait(bar(KV_SFULL + sbuf), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        float sv[STEP], dp[STEP];
        const uint32_t s_tm = tmem + lane_base + T_S + sbuf * STEP;
        const uint32_t p_tm = tmem + lane_base + T_DP + sbuf * STEP;
        tmem_ld32(s_tm, sv);
        tmem_ld32(s_tm + 32, sv + 32);
        tmem_ld32(p_tm, dp);
        tmem_ld32(p_tm + 32, dp + 32);
        tmem_wait_ld();
        const uint32_t st = q_it % NQ;
        if (!mbar_wait(bar(KV_RSFULL + st), (q_it / NQ) & 1, abort, status)) { ok = false; break; }
        const float* rs = reinterpret_cast<const float*>(smem + L::RS_OFF + st * STEP * 8);
        const int i0 = (qs0 + step) * STEP;
        // valid queries of this step for key j: i < Lq and (causal) i >= j
        const int lo = CAUSAL ? j - i0 : 0;
        const int hi = j < Lk ? Lq - i0 : 0;
        if (lo > 0 || hi < STEP) {
          // partial step: move masked raw scores down by a finite shift
#pragma unroll
          for (int c = 0; c < STEP; ++c) sv[c] -= (c >= lo && c < hi) ? 0.f : shift_raw;
        }
        const float2 cc = make_float2(c_score, c_score);
        uint32_t pk[STEP / 2], dk2[STEP / 2];
#pragma unroll
        for (int c = 0; c < STEP; c += 2) {
          const float2 x = make_float2(sv[c], sv[c + 1]);
          const float2 d = make_float2(dp[c], dp[c + 1]);
          float2 pv, ds;
          if (ACT == kActSoftmax) {
            const float2 nl = *reinterpret_cast<const float2*>(rs + c);        // -lse log2 e
            const float2 nd = *reinterpret_cast<const float2*>(rs + STEP + c); // -D
            const float2 e = ffma2(x, cc, nl);
            pv = make_float2(ex2(e.x), ex2(e.y));
            ds = fmul2(pv, fadd2(d, nd));
          } else {
            // u = s c, h = u/2, t = tanh h: P = h (1+t)/L, dS = dP (1+t)/L (1 + h - h t)/2
            const float2 hh = fmul2(x, hc);
            const float2 t = make_float2(tanh_approx(hh.x), tanh_approx(hh.y));
            const float2 g = ffma2(t, il, il);
            pv = fmul2(hh, g);
            const float2 b = ffma2(make_float2(-hh.x, -hh.y), t, fadd2(hh, one));
            ds = fmul2(fmul2(d, g), fmul2(b, half));
          }
          pk[c / 2] = pack_bf16(pv.x, pv.y);
          dk2[c / 2] = pack_bf16(ds.x, ds.y);
        }
        tmem_st32(s_tm, reinterpret_cast<const float*>(pk));
        tmem_st32(p_tm, reinterpret_cast<const float*>(dk2));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(KV_PFULL + sbuf));
        ++s_it;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      const bool key_ok = j < Lk;
      const int64_t krow = (k0 + j) * p.heads + h;
      if (n > 0) {
        if (!mbar_wait(bar(KV_ACCFULL), a_it & 1, abort, status)) { ok = false; break; }
        ++a_it;
        tc_fence_after();
        float x[32];
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) {
          tmem_ld32(tmem + lane_base + T_DK + 32 * c, x);
          tmem_wait_ld();
          if (key_ok) store_row_bf16(dk + krow * DQK + 32 * c, x, p.scale);
        }
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          tmem_ld32(tmem + lane_base + T_DV + 32 * c, x);
          tmem_wait_ld();
          if (key_ok) store_row_bf16(dv + krow * DV + 32 * c, x, 1.f);
        }
        tc_fence_before();
        mbar_arrive(bar(KV_ACCEMPTY));
      } else if (key_ok) {
        const float z[32] = {0.f};
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) store_row_bf16(dk + krow * DQK + 32 * c, z, 1.f);
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) store_row_bf16(dv + krow * DV + 32 * c, z, 1.f);
      }
    }
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
// K/V steps are staged in an NK-deep ring; dS is written back into TMEM as
// packed bf16 over the first 32 columns of the dP buffer and the dQ product
// reads it from there.
template <int DQK, int DV>
struct QLayout {
  // Q/dO of the next item are prefetched where shared memory allows; the K/V
  // ring depth matters more and is kept at 4 or more.
  static constexpr int NQO = DQK + DV > 192 ? 1 : 2;       // Q/dO tiles
  static constexpr int NK = DQK + DV > 128 ? 4 : 6;        // K/V ring stages
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;   // 128 rows
  static constexpr uint32_t O_BYTES = DV / 64 * 16384;
  static constexpr uint32_t K_BYTES = DQK / 64 * 8192;    // 64 keys
  static constexpr uint32_t V_BYTES = DV / 64 * 8192;
  static constexpr uint32_t Q_OFF = 0;                     // NQO stages
  static constexpr uint32_t O_OFF = Q_OFF + NQO * Q_BYTES; // NQO stages
  static constexpr uint32_t K_OFF = O_OFF + NQO * O_BYTES; // NK stages
  static constexpr uint32_t V_OFF = K_OFF + NK * K_BYTES;  // NK stages
  static constexpr uint32_t BAR_OFF = V_OFF + NK * V_BYTES;
  static constexpr uint32_t SMEM = (BAR_OFF + 512 + 1024) > 122880u ? (BAR_OFF + 512 + 1024) : 122880u;
};

enum : uint32_t {
  Q_QFULL = 0, Q_QEMPTY = 2, Q_KFULL = 4, Q_KEMPTY = 10, Q_SFULL = 16, Q_PFULL = 18,
  Q_ACCFULL = 20, Q_ACCEMPTY = 21, Q_COUNT = 22
};

template <int DQK, int DV, int ACT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
tc_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
             const Problem p, const float2* __restrict__ rowstat, __nv_bfloat16* __restrict__ dq,
             WsHeader* hdr, const WorkItem* __restrict__ list) {
  using L = QLayout<DQK, DV>;
  constexpr int NK = L::NK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + L::BAR_OFF;
  auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = (uint32_t*)(smem + L::BAR_OFF + 8 * Q_COUNT);
  volatile int* abort = (volatile int*)(smem + L::BAR_OFF + 8 * Q_COUNT + 4);
  int* status = &hdr->status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = hdr->n_q;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::NQO; ++s) {
      mbar_init(bar(Q_QFULL + s), 1);
      mbar_init(bar(Q_QEMPTY + s), 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(Q_KFULL + s), 1);
      mbar_init(bar(Q_KEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(Q_SFULL + s), 1);
      mbar_init(bar(Q_PFULL + s), 128);
    }
    mbar_init(bar(Q_ACCFULL), 1);
    mbar_init(bar(Q_ACCEMPTY), 128);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: dQ [0,128), S [128 + 64 b), dP/dS [256 + 64 b)
  constexpr uint32_t T_DQ = 0, T_S = 128, T_DP = 256;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t q_it = 0, k_it = 0;
      bool ok = true;
      WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = nxt;  // prefetched one item ahead
        if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
        const int n = w.cost;
        if (n == 0) continue;
        const int h = w.h, row0 = w.tile * TILE;
        const int32_t q0 = w.q0, k0 = w.k0;
        const uint32_t qs = q_it % L::NQO;
        if (!mbar_wait(bar(Q_QEMPTY + qs), ((q_it / L::NQO) & 1) ^ 1, abort, status)) break;
        mbar_expect_tx(bar(Q_QFULL + qs), L::Q_BYTES + L::O_BYTES);
#pragma unroll
        for (int a = 0; a < DQK / 64; ++a)
          tma_load_2d(sb + L::Q_OFF + qs * L::Q_BYTES + a * 16384, &tm_q, h * DQK + a * 64, q0 + row0,
                      bar(Q_QFULL + qs));
#pragma unroll
        for (int a = 0; a < DV / 64; ++a)
          tma_load_2d(sb + L::O_OFF + qs * L::O_BYTES + a * 16384, &tm_do, h * DV + a * 64, q0 + row0,
                      bar(Q_QFULL + qs));
        ++q_it;
        for (int j = 0; j < n; ++j, ++k_it) {
          const uint32_t st = k_it % NK, ph = (k_it / NK) & 1;
          if (!mbar_wait(bar(Q_KEMPTY + st), ph ^ 1, abort, status)) { ok = false; break; }
          mbar_expect_tx(bar(Q_KFULL + st), L::K_BYTES + L::V_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::K_OFF + st * L::K_BYTES + a * 8192, &tm_k, h * DQK + a * 64,
                        k0 + j * STEP, bar(Q_KFULL + st));
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::V_OFF + st * L::V_BYTES + a * 8192, &tm_v, h * DV + a * 64,
                        k0 + j * STEP, bar(Q_KFULL + st));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(TILE, STEP, 0, 0);
      constexpr uint32_t idesc_dq = idesc_bf16(TILE, DQK, 0, 1);
      uint32_t q_it = 0, k_it = 0, s_it = 0, a_it = 0;
      bool ok = true;
      WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = nxt;
        if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
        const int n = w.cost;
        if (n == 0) continue;
        const uint32_t qs = q_it % L::NQO;
        if (!mbar_wait(bar(Q_QFULL + qs), (q_it / L::NQO) & 1, abort, status)) break;
        tc_fence_after();
        const uint32_t q_tile = sb + L::Q_OFF + qs * L::Q_BYTES;
        const uint32_t o_tile = sb + L::O_OFF + qs * L::O_BYTES;
        uint32_t prev_stage = 0;
        for (int j = 0; j <= n && ok; ++j) {
          uint32_t cur_stage = 0;
          if (j < n) {
            cur_stage = k_it % NK;
            const uint32_t sbuf = s_it & 1;
            if (!mbar_wait(bar(Q_KFULL + cur_stage), (k_it / NK) & 1, abort, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint64_t ad = sw128_desc(q_tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::K_OFF + cur_stage * L::K_BYTES + (kk >> 2) * 8192 +
                                                 (kk & 3) * 32, 16, 1024);
              mma_bf16(tmem + T_S + sbuf * STEP, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < DV / 16; ++kk) {
              const uint64_t ad = sw128_desc(o_tile + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::V_OFF + cur_stage * L::V_BYTES + (kk >> 2) * 8192 +
                                                 (kk & 3) * 32, 16, 1024);
              mma_bf16(tmem + T_DP + sbuf * STEP, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(Q_SFULL + sbuf));
            if (j == n - 1) mma_commit(bar(Q_QEMPTY + qs));
            ++s_it;
            ++k_it;
          }
          if (j > 0) {
            // dQ += dS(j-1) K(j-1), dS from TMEM
            const uint32_t pidx = s_it - (j < n ? 2 : 1);
            const uint32_t pbuf = pidx & 1;
            if (!mbar_wait(bar(Q_PFULL + pbuf), (pidx >> 1) & 1, abort, status) ||
                (j == 1 && !mbar_wait(bar(Q_ACCEMPTY), (a_it & 1) ^ 1, abort, status))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < STEP / 16; ++kk) {
              const uint64_t bd = sw128_desc(sb + L::K_OFF + prev_stage * L::K_BYTES + kk * 2048, 8192, 1024);
              mma_bf16_tmem_a(tmem + T_DQ, tmem + T_DP + pbuf * STEP + kk * 8, bd, idesc_dq,
                              (j > 1 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(Q_KEMPTY + prev_stage));
            if (j == n) mma_commit(bar(Q_ACCFULL));
          }
          prev_stage = cur_stage;
        }
        ++q_it;
        ++a_it;
      }
    }
    __syncwarp();
  } else {
    const int r = 32 * (warp & 3) + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    const float shift_raw = kMaskShift / c_score;  // masked raw scores land kMaskShift lower
    const float2 cc = make_float2(c_score, c_score);
    const float2 hc = make_float2(0.5f * c_score, 0.5f * c_score);
    const float2 one = make_float2(1.f, 1.f), half = make_float2(0.5f, 0.5f);
    uint32_t s_it = 0, a_it = 0;
    bool ok = true;
    WorkItem nxt = blockIdx.x < (unsigned)n_items ? load_item(list, blockIdx.x) : WorkItem{};
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const WorkItem w = nxt;
      if (it + (int)gridDim.x < n_items) nxt = load_item(list, it + gridDim.x);
      const int n = w.cost;
      const int h = w.h, row0 = w.tile * TILE;
      const int64_t q0 = w.q0;
      const int Lq = w.lq, Lk = w.lk;
      const int i = row0 + r;
      const bool row_ok = i < Lq;
      const float inv_len = 1.0f / (float)max(Lq, 1);
      float2 rsv = make_float2(0.f, 0.f);
      if (ACT == kActSoftmax && row_ok && n > 0) rsv = rowstat[(int64_t)h * p.total_q + q0 + i];
      const float2 nl = make_float2(-rsv.x, -rsv.x), nd = make_float2(-rsv.y, -rsv.y);
      const float2 il = make_float2(inv_len, inv_len);
      for (int step = 0; step < n; ++step) {
        const uint32_t sbuf = s_it & 1;
        if (!mbar_wait(bar(Q_SFULL + sbuf), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        float sv[STEP], dp[STEP];
        const uint32_t s_tm = tmem + lane_base + T_S + sbuf * STEP;
        const uint32_t p_tm = tmem + lane_base + T_DP + sbuf * STEP;
        tmem_ld32(s_tm, sv);
        tmem_ld32(s_tm + 32, sv + 32);
        tmem_ld32(p_tm, dp);
        tmem_ld32(p_tm + 32, dp + 32);
        tmem_wait_ld();
        const int kb = step * STEP;
        int nvalid = Lk - kb;
        if (CAUSAL) nvalid = min(nvalid, i - kb + 1);
        if (!row_ok) nvalid = 0;
        if (nvalid < STEP) {
          // partial step: move masked raw scores down by a finite shift
#pragma unroll
          for (int c = 0; c < STEP; ++c) sv[c] -= c < nvalid ? 0.f : shift_raw;
        }
        uint32_t pk[STEP / 2];
#pragma unroll
        for (int c = 0; c < STEP; c += 2) {
          const float2 x = make_float2(sv[c], sv[c + 1]);
          const float2 d = make_float2(dp[c], dp[c + 1]);
          float2 ds;
          if (ACT == kActSoftmax) {
            const float2 e = ffma2(x, cc, nl);
            ds = fmul2(make_float2(ex2(e.x), ex2(e.y)), fadd2(d, nd));
          } else {
            const float2 hh = fmul2(x, hc);
            const float2 t = make_float2(tanh_approx(hh.x), tanh_approx(hh.y));
            const float2 g = ffma2(t, il, il);
            const float2 b = ffma2(make_float2(-hh.x, -hh.y), t, fadd2(hh, one));
            ds = fmul2(fmul2(d, g), fmul2(b, half));
          }
          pk[c / 2] = pack_bf16(ds.x, ds.y);
        }
        tmem_st32(p_tm, reinterpret_cast<const float*>(pk));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(Q_PFULL + sbuf));
        ++s_it;
      }
      if (!ok) break;
      const int64_t orow = (q0 + i) * p.heads + h;
      if (n > 0) {
        if (!mbar_wait(bar(Q_ACCFULL), a_it & 1, abort, status)) { ok = false; break; }
        ++a_it;
        tc_fence_after();
        float x[32];
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) {
          tmem_ld32(tmem + lane_base + T_DQ + 32 * c, x);
          tmem_wait_ld();
          if (row_ok) store_row_bf16(dq + orow * DQK + 32 * c, x, p.scale);
        }
        tc_fence_before();
        mbar_arrive(bar(Q_ACCEMPTY));
      } else if (row_ok) {
        const float z[32] = {0.f};
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) store_row_bf16(dq + orow * DQK + 32 * c, z, 1.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host side
struct Maps {
  CUtensorMap q64, do64, k128, v128;  // dK/dV pass: 64-row Q/dO boxes, 128-key K/V boxes
  CUtensorMap q128, do128, k64, v64;  // dQ pass: 128-row Q/dO boxes, 64-key K/V boxes
};

bool make_maps(const Problem& p, const void* q, const void* k, const void* v, const void* dout,
               bool kv_pass, Maps* m) {
  const int64_t cq = (int64_t)p.heads * p.dim_qk, cv = (int64_t)p.heads * p.dim_v;
  const int64_t tk = p.total_k > 0 ? p.total_k : p.total_q;
  const void* kk = p.total_k > 0 ? k : q;
  const void* vv = p.total_k > 0 ? v : dout;
  if (kv_pass)
    return make_tile_map(&m->q64, q, p.total_q, cq, 64, STEP) &&
           make_tile_map(&m->do64, dout, p.total_q, cv, 64, STEP) &&
           make_tile_map(&m->k128, kk, tk, cq, 64, TILE) && make_tile_map(&m->v128, vv, tk, cv, 64, TILE);
  return make_tile_map(&m->q128, q, p.total_q, cq, 64, TILE) &&
         make_tile_map(&m->do128, dout, p.total_q, cv, 64, TILE) &&
         make_tile_map(&m->k64, kk, tk, cq, 64, STEP) && make_tile_map(&m->v64, vv, tk, cv, 64, STEP);
}

template <int DQK, int DV, int ACT, bool CAUSAL>
cudaError_t dkdv_t(const Maps& m, const Problem& p, const float2* rowstat, void* dk, void* dv,
                   const Workspace& ws, cudaStream_t s) {
  auto kern = tc_dkdv_kernel<DQK, DV, ACT, CAUSAL>;
  constexpr uint32_t smem = KvLayout<DQK, DV>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreads, smem, s>>>(m.k128, m.v128, m.q64, m.do64, p, rowstat,
                                         (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, ws.hdr, ws.list_k);
  return cudaGetLastError();
}

template <int DQK, int DV, int ACT, bool CAUSAL>
cudaError_t dq_t(const Maps& m, const Problem& p, const float2* rowstat, void* dq,
                 const Workspace& ws, cudaStream_t s) {
  auto kern = tc_dq_kernel<DQK, DV, ACT, CAUSAL>;
  constexpr uint32_t smem = QLayout<DQK, DV>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreads, smem, s>>>(m.q128, m.do128, m.k64, m.v64, p, rowstat,
                                         (__nv_bfloat16*)dq, ws.hdr, ws.list_q);
  return cudaGetLastError();
}

#define JFA_TC_BWD_DISPATCH(FN, ...)                                                          \
  do {                                                                                        \
    const bool sm_ = p.act == kActSoftmax, c_ = p.causal != 0;                               \
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

SchedConfig tc_bwd_sched(const Problem&) { return SchedConfig{TILE, STEP, TILE, STEP, 1, 1, 0}; }

cudaError_t launch_tc_rowstat(const Problem& p, const void* o, const void* dout, const float* lse,
                              const Workspace& ws, cudaStream_t s) {
  const int64_t threads = p.total_q * p.heads * (p.dim_v / 8);
  if (threads == 0) return cudaSuccess;
  int64_t blocks = (threads + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 16;
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
  if (!make_maps(p, q, k, v, dout, true, &m)) return cudaErrorInvalidValue;
  const float2* rs = reinterpret_cast<const float2*>(ws.drow);
  JFA_TC_BWD_DISPATCH(dkdv_t, m, p, rs, dk, dv, ws, s);
}

cudaError_t launch_tc_dq(const Problem& p, const void* q, const void* k, const void* v,
                         const float* lse, const void* dout, void* dq, const Workspace& ws,
                         cudaStream_t s) {
  (void)lse;
  Maps m;
  if (!make_maps(p, q, k, v, dout, false, &m)) return cudaErrorInvalidValue;
  const float2* rs = reinterpret_cast<const float2*>(ws.drow);
  JFA_TC_BWD_DISPATCH(dq_t, m, p, rs, dq, ws, s);
}

}  // namespace jfa
