// Tensor-core jagged attention forward for sm_103a: TMA + tcgen05 + TMEM.
//
// Method: Jagged Flash Attention bullet of the Meta GEM MFU write-up
// (piletech.kr/articles/112134, details): attention computed directly on the
// jagged buffers, masked by subtraction, persistent kernel scheduling with
// specialised warps; Generalized Dot-Product Attention bullet: the same
// pipeline with a non-softmax activation (here SiLU(s)/L).
//
// One persistent CTA per SM walks the scheduler's heavy-first list of
// (sequence, head, 128-row q-tile) items.  Warp roles:
//   warp 0      TMA producer: Q tile once per item, K and V tiles of 128 keys
//               into a two-stage ring, straight from the jagged [T, H*D]
//               buffers (rows past a sequence belong to its neighbour and are
//               masked; rows past the buffer are zero-filled by TMA).
//   warp 1      TMEM owner and MMA issuer (one lane): S = Q K^T into one of two
//               TMEM S buffers, then O += P V into the TMEM O accumulator; S of
//               step j+1 is issued before PV of step j so the tensor pipe works
//               while the softmax warps process S_j.
//   warps 2..5  softmax warpgroup, one query row per thread (TMEM lane):
//               tcgen05.ld of its S row, scale to log2 units, subtract a finite
//               shift from masked columns, online max with lazy rescaling of O
//               (only when the running max grows by more than 2^8), exp2, row
//               sum, P as bf16 into a 128-byte-swizzled smem tile, and the
//               epilogue O / l -> bf16, lse = (m + log2 l) ln 2.
// TMEM: S0 cols [0,128), S1 [128,256), O [256, 256+Dv).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tc.h"
#include "tc_ptx.cuh"
#include "tc_host.h"

namespace jfa {
namespace {
using namespace tc;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

template <int DQK, int DV>
struct FwdLayout {
  static constexpr uint32_t Q_BYTES = DQK / 64 * 16384;
  static constexpr uint32_t K_BYTES = DQK / 64 * 16384;
  static constexpr uint32_t V_BYTES = DV / 64 * 16384;
  static constexpr uint32_t P_BYTES = 2 * 16384;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + 2 * K_BYTES;
  static constexpr uint32_t P_OFF = V_OFF + 2 * V_BYTES;
  static constexpr uint32_t BAR_OFF = P_OFF + 2 * P_BYTES;
  // at least 120 KB so that exactly one CTA (which owns all of TMEM) fits per SM
  static constexpr uint32_t SMEM = (BAR_OFF + 256 + 1024) > 122880u ? (BAR_OFF + 256 + 1024) : 122880u;
};

// mbarrier slots
enum : uint32_t {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_VFULL = 4, B_KVEMPTY = 6, B_SFULL = 8,
  B_SEMPTY = 10, B_PFULL = 12, B_PEMPTY = 14, B_OEMPTY = 16, B_COUNT = 17
};

template <int DQK, int DV, int ACT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const Problem p,
              __nv_bfloat16* __restrict__ out, float* __restrict__ lse, WsHeader* hdr,
              const WorkItem* __restrict__ list) {
  using L = FwdLayout<DQK, DV>;
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SEMPTY + s), 128);
      mbar_init(bar(B_PFULL + s), 128);
      mbar_init(bar(B_PEMPTY + s), 1);
    }
    mbar_init(bar(B_OEMPTY), 128);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      uint32_t kv_it = 0, q_it = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const WorkItem w = list[it];
        const int n = w.w;
        if (n == 0) continue;
        const int b = w.x, h = w.y, row0 = w.z * BM;
        const int32_t q0 = (int32_t)p.offs_q[b], k0 = (int32_t)p.offs_k[b];
        if (!mbar_wait(bar(B_QEMPTY), (q_it & 1) ^ 1, abort, status)) break;
        mbar_expect_tx(bar(B_QFULL), L::Q_BYTES);
#pragma unroll
        for (int a = 0; a < DQK / 64; ++a)
          tma_load_2d(sb + L::Q_OFF + a * 16384, &tm_q, h * DQK + a * 64, q0 + row0, bar(B_QFULL));
        ++q_it;
        bool ok = true;
        for (int j = 0; j < n; ++j, ++kv_it) {
          const uint32_t s = kv_it & 1, ph = (kv_it >> 1) & 1;
          if (!mbar_wait(bar(B_KVEMPTY + s), ph ^ 1, abort, status)) { ok = false; break; }
          mbar_expect_tx(bar(B_KFULL + s), L::K_BYTES);
#pragma unroll
          for (int a = 0; a < DQK / 64; ++a)
            tma_load_2d(sb + L::K_OFF + s * L::K_BYTES + a * 16384, &tm_k, h * DQK + a * 64,
                        k0 + j * BN, bar(B_KFULL + s));
          mbar_expect_tx(bar(B_VFULL + s), L::V_BYTES);
#pragma unroll
          for (int a = 0; a < DV / 64; ++a)
            tma_load_2d(sb + L::V_OFF + s * L::V_BYTES + a * 16384, &tm_v, h * DV + a * 64,
                        k0 + j * BN, bar(B_VFULL + s));
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16(BM, DV, 0, 1);
      uint32_t kv_it = 0, s_it = 0, p_it = 0, q_it = 0, o_it = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const WorkItem w = list[it];
        const int n = w.w;
        if (n == 0) continue;
        if (!mbar_wait(bar(B_QFULL), q_it & 1, abort, status)) break;
        tc_fence_after();
        uint32_t prev_stage = 0, prev_phase = 0;
        for (int j = 0; j <= n && ok; ++j) {
          uint32_t cur_stage = 0, cur_phase = 0;
          if (j < n) {
            cur_stage = kv_it & 1;
            cur_phase = (kv_it >> 1) & 1;
            const uint32_t sbuf = s_it & 1;
            if (!mbar_wait(bar(B_KFULL + cur_stage), cur_phase, abort, status) ||
                !mbar_wait(bar(B_SEMPTY + sbuf), ((s_it >> 1) & 1) ^ 1, abort, status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + sbuf * 128;
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              const uint64_t ad = sw128_desc(sb + L::Q_OFF + off, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::K_OFF + cur_stage * L::K_BYTES + off, 16, 1024);
              mma_bf16(d, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar(B_SFULL + sbuf));
            if (j == n - 1) mma_commit(bar(B_QEMPTY));
            ++s_it;
            ++kv_it;
          }
          if (j > 0) {
            const uint32_t pbuf = p_it & 1;
            if (!mbar_wait(bar(B_PFULL + pbuf), (p_it >> 1) & 1, abort, status) ||
                !mbar_wait(bar(B_VFULL + prev_stage), prev_phase, abort, status) ||
                (j == 1 && !mbar_wait(bar(B_OEMPTY), (o_it & 1) ^ 1, abort, status))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              const uint64_t ad = sw128_desc(sb + L::P_OFF + pbuf * L::P_BYTES + (kk >> 2) * 16384 +
                                                 (kk & 3) * 32, 16, 1024);
              const uint64_t bd = sw128_desc(sb + L::V_OFF + prev_stage * L::V_BYTES + kk * 2048,
                                             16384, 1024);
              mma_bf16(tmem + 256, ad, bd, idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(B_PEMPTY + pbuf));
            mma_commit(bar(B_KVEMPTY + prev_stage));
            ++p_it;
          }
          prev_stage = cur_stage;
          prev_phase = cur_phase;
        }
        ++q_it;
        ++o_it;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int r = 32 * (warp & 3) + lane;  // TMEM lane = row of the tile
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float c_score = ACT == kActSoftmax ? p.scale * kLog2e : p.scale;
    uint32_t s_it = 0, p_it = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const WorkItem w = list[it];
      const int n = w.w;
      const int b = w.x, h = w.y, row0 = w.z * BM;
      const int64_t q0 = p.offs_q[b], k0 = p.offs_k[b];
      const int Lq = (int)(p.offs_q[b + 1] - q0), Lk = (int)(p.offs_k[b + 1] - k0);
      const int i = row0 + r;
      const float inv_len = 1.0f / (float)max(Lq, 1);
      float m = -INFINITY, l = 0.f;
      float sv[BN];
      for (int j = 0; j < n; ++j) {
        const uint32_t sbuf = s_it & 1;
        if (!mbar_wait(bar(B_SFULL + sbuf), (s_it >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tmem + lane_base + sbuf * 128 + 32 * c, sv + 32 * c);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(B_SEMPTY + sbuf));
        ++s_it;
        const int kb = j * BN;
        int nvalid = Lk - kb;
        if (CAUSAL) nvalid = min(nvalid, i - kb + 1);
        if (ACT == kActSoftmax) {
          float mt = -INFINITY;
          if (nvalid >= BN) {
#pragma unroll
            for (int k = 0; k < BN; ++k) { sv[k] *= c_score; mt = fmaxf(mt, sv[k]); }
          } else {
#pragma unroll
            for (int k = 0; k < BN; ++k) {
              sv[k] = fmaf(sv[k], c_score, k < nvalid ? 0.f : -kMaskShift);
              mt = fmaxf(mt, sv[k]);
            }
          }
          if (j == 0) {
            m = mt;
          } else {
            const bool need = mt > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
              // O must hold PV of step j-1 before it is rescaled.
              const uint32_t pprev = p_it - 1;
              if (!mbar_wait(bar(B_PEMPTY + (pprev & 1)), (pprev >> 1) & 1, abort, status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const float alpha = need ? ex2(m - mt) : 1.f;
              float ov[32];
#pragma unroll
              for (int c = 0; c < DV / 32; ++c) {
                tmem_ld32(tmem + lane_base + 256 + 32 * c, ov);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) ov[t] *= alpha;
                tmem_st32(tmem + lane_base + 256 + 32 * c, ov);
              }
              tmem_wait_st();
              l *= alpha;
              if (need) m = mt;
            }
          }
          float rs = 0.f;
#pragma unroll
          for (int k = 0; k < BN; ++k) { sv[k] = ex2(sv[k] - m); rs += sv[k]; }
          l += rs;
        } else {
#pragma unroll
          for (int k = 0; k < BN; ++k) {
            const float u = fmaf(sv[k], c_score, k < nvalid ? 0.f : -kMaskShift);
            const float sg = rcp(1.f + ex2(-u * kLog2e));
            sv[k] = u * sg * inv_len;
          }
        }
        // P (bf16) into the swizzled smem tile of this buffer
        const uint32_t pbuf = p_it & 1;
        if (!mbar_wait(bar(B_PEMPTY + pbuf), ((p_it >> 1) & 1) ^ 1, abort, status)) { ok = false; break; }
        const uint32_t pbase = sb + L::P_OFF + pbuf * L::P_BYTES;
#pragma unroll
        for (int a = 0; a < 2; ++a) {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const float* x = sv + a * 64 + ch * 8;
            st_shared_v4(pbase + a * 16384 + sw128_offset(r, ch), pack_bf16(x[0], x[1]),
                         pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]), pack_bf16(x[6], x[7]));
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + pbuf));
        ++p_it;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      const bool row_ok = i < Lq;
      const int64_t orow = (q0 + i) * p.heads + h;
      if (n > 0) {
        const uint32_t plast = p_it - 1;
        if (!mbar_wait(bar(B_PEMPTY + (plast & 1)), (plast >> 1) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        const float norm = ACT == kActSoftmax ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
        float ov[32];
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          tmem_ld32(tmem + lane_base + 256 + 32 * c, ov);
          tmem_wait_ld();
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + orow * DV + 32 * c);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float* x = ov + 8 * t;
              dst[t] = make_uint4(pack_bf16(x[0] * norm, x[1] * norm), pack_bf16(x[2] * norm, x[3] * norm),
                                  pack_bf16(x[4] * norm, x[5] * norm), pack_bf16(x[6] * norm, x[7] * norm));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_OEMPTY));
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
  if (warp == 1) {
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
