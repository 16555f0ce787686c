// CUDA-core jagged attention kernels: fp32 arithmetic end to end.
//
// These serve fp32 inputs (where the tensor cores' bf16/tf32 kinds cannot
// meet fp32 accuracy) and any head size the tensor-core kernels do not
// cover.  They follow the same structure as the tensor-core path: persistent
// CTAs walk the scheduler's heavy-first work lists; the forward keeps an
// online softmax (running maximum and sum, exp2 of log2-scaled scores);
// masked scores are shifted down by a finite constant rather than set to
// -inf; the backward is two atomic-free passes (key-tile-major for dK/dV,
// query-tile-major for dQ) after a row-term pass D_i = <dO_i, O_i>.
//
// Method: Jagged Flash Attention and Generalized Dot-Product Attention
// bullets, Meta GEM MFU write-up (piletech.kr/articles/112134), details.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kRowsPerWarp = 8;
constexpr int kTileRows = 64;  // q rows per forward / dQ item, keys per dK/dV item
constexpr int kStep = 32;      // keys per forward / dQ step, rows per dK/dV step
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float sigmoidf_(float u) { return 1.0f / (1.0f + expf(-u)); }

// Factor folded into Q when it is staged: scores come out log2-scaled for
// softmax (so exp2 applies directly) and plainly scaled for SiLU.
__device__ __forceinline__ float q_factor(const Problem& p) {
  return p.act == kActSoftmax ? p.scale * kLog2e : p.scale;
}

template <typename T, int DQ, int DV>
struct SimtFwdSmem {
  float q[kTileRows][DQ];
  float k[kStep][DQ + 1];
  float v[kStep][DV];
};

// Forward: one item = (b, h, 64-row q-tile); 8 warps x 8 rows; key steps of 32.
template <typename T, int DQ, int DV>
__global__ void __launch_bounds__(kThreads)
simt_fwd_kernel(Problem p, const T* __restrict__ q, const T* __restrict__ k,
                const T* __restrict__ v, T* __restrict__ o, float* __restrict__ lse,
                const WsHeader* __restrict__ hdr, const WorkItem* __restrict__ list) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<SimtFwdSmem<T, DQ, DV>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.heads, Dq = p.dim_qk, Dv = p.dim_v;
  const float qf = q_factor(p);
  const int n = hdr->n_q;
  for (int it = blockIdx.x; it < n; it += gridDim.x) {
    const WorkItem w = load_item(list, it);
    const int h = w.h, row0 = w.tile * kTileRows;
    const int64_t q0 = w.q0, k0 = w.k0;
    const int Lq = w.lq, Lk = w.lk;
    const float inv_len = 1.0f / (float)max(Lq, 1);
    __syncthreads();
    for (int idx = tid; idx < kTileRows * DQ; idx += kThreads) {
      int r = idx / DQ, d = idx % DQ;
      float x = 0.f;
      if (row0 + r < Lq && d < Dq) x = ld(q, ((q0 + row0 + r) * H + h) * Dq + d) * qf;
      sm.q[r][d] = x;
    }
    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][DV / 32];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      m[rr] = -INFINITY;
      l[rr] = 0.f;
#pragma unroll
      for (int t = 0; t < DV / 32; ++t) acc[rr][t] = 0.f;
    }
    const int kend = p.causal ? min(Lk, row0 + kTileRows) : Lk;
    for (int kb = 0; kb < kend; kb += kStep) {
      __syncthreads();
      for (int idx = tid; idx < kStep * DQ; idx += kThreads) {
        int r = idx / DQ, d = idx % DQ;
        sm.k[r][d] = (kb + r < Lk && d < Dq) ? ld(k, ((k0 + kb + r) * H + h) * Dq + d) : 0.f;
      }
      for (int idx = tid; idx < kStep * DV; idx += kThreads) {
        int r = idx / DV, d = idx % DV;
        sm.v[r][d] = (kb + r < Lk && d < Dv) ? ld(v, ((k0 + kb + r) * H + h) * Dv + d) : 0.f;
      }
      __syncthreads();
      const int j = kb + lane;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = warp * kRowsPerWarp + rr, i = row0 + r;
        float s = 0.f;
#pragma unroll 8
        for (int d = 0; d < DQ; ++d) s = fmaf(sm.q[r][d], sm.k[lane][d], s);
        const bool valid = j < Lk && (!p.causal || j <= i);
        s -= valid ? 0.f : kMaskShift;
        float pj;
        if (p.act == kActSoftmax) {
          const float mn = fmaxf(m[rr], warp_max(s));
          const float alpha = exp2f(m[rr] - mn);
          pj = exp2f(s - mn);
          l[rr] = l[rr] * alpha + warp_sum(pj);
          m[rr] = mn;
#pragma unroll
          for (int t = 0; t < DV / 32; ++t) acc[rr][t] *= alpha;
        } else {
          pj = s * sigmoidf_(s) * inv_len;
        }
#pragma unroll 4
        for (int jj = 0; jj < kStep; ++jj) {
          const float pv = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
          for (int t = 0; t < DV / 32; ++t) acc[rr][t] = fmaf(pv, sm.v[jj][lane + 32 * t], acc[rr][t]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int i = row0 + warp * kRowsPerWarp + rr;
      if (i >= Lq) continue;
      const int64_t row = (q0 + i) * H + h;
      float norm = 1.f;
      if (p.act == kActSoftmax) norm = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
#pragma unroll
      for (int t = 0; t < DV / 32; ++t) {
        const int c = lane + 32 * t;
        if (c < Dv) st(o, row * Dv + c, acc[rr][t] * norm);
      }
      if (lse != nullptr && lane == 0)
        lse[row] = (p.act != kActSoftmax) ? 0.f
                   : (l[rr] > 0.f ? (m[rr] + log2f(l[rr])) * kLn2 : -INFINITY);
    }
  }
}

// D_i = <dO_i, O_i> for every (row, head): one warp per (row, head).
template <typename T>
__global__ void __launch_bounds__(kThreads)
rowterm_kernel(int64_t rows, int dv, const T* __restrict__ o, const T* __restrict__ dout,
               float* __restrict__ drow) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t r = blockIdx.x * (int64_t)(kThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    float acc = 0.f;
    for (int c = lane; c < dv; c += 32) acc = fmaf(ld(o, r * dv + c), ld(dout, r * dv + c), acc);
    acc = warp_sum(acc);
    if (lane == 0) drow[r] = acc;
  }
}

template <typename T, int DQ, int DV>
struct SimtDqSmem {
  float q[kTileRows][DQ];
  float dout[kTileRows][DV];
  float k[kStep][DQ + 1];
  float v[kStep][DV + 1];
};

// dQ pass: one item = (b, h, 64-row q-tile); loop over key steps of 32.
template <typename T, int DQ, int DV>
__global__ void __launch_bounds__(kThreads)
simt_dq_kernel(Problem p, const T* __restrict__ q, const T* __restrict__ k,
               const T* __restrict__ v, const float* __restrict__ lse,
               const float* __restrict__ drow, const T* __restrict__ dout, T* __restrict__ dq,
               const WsHeader* __restrict__ hdr, const WorkItem* __restrict__ list) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<SimtDqSmem<T, DQ, DV>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.heads, Dq = p.dim_qk, Dv = p.dim_v;
  const float qf = q_factor(p);
  const bool softmax = p.act == kActSoftmax;
  const int n = hdr->n_q;
  for (int it = blockIdx.x; it < n; it += gridDim.x) {
    const WorkItem w = load_item(list, it);
    const int h = w.h, row0 = w.tile * kTileRows;
    const int64_t q0 = w.q0, k0 = w.k0;
    const int Lq = w.lq, Lk = w.lk;
    const float inv_len = 1.0f / (float)max(Lq, 1);
    __syncthreads();
    for (int idx = tid; idx < kTileRows * DQ; idx += kThreads) {
      int r = idx / DQ, d = idx % DQ;
      sm.q[r][d] = (row0 + r < Lq && d < Dq) ? ld(q, ((q0 + row0 + r) * H + h) * Dq + d) * qf : 0.f;
    }
    for (int idx = tid; idx < kTileRows * DV; idx += kThreads) {
      int r = idx / DV, d = idx % DV;
      sm.dout[r][d] = (row0 + r < Lq && d < Dv) ? ld(dout, ((q0 + row0 + r) * H + h) * Dv + d) : 0.f;
    }
    float lse2[kRowsPerWarp], drr[kRowsPerWarp], acc[kRowsPerWarp][DQ / 32];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int i = row0 + warp * kRowsPerWarp + rr;
      const int64_t row = (q0 + i) * H + h;
      lse2[rr] = (softmax && i < Lq) ? lse[row] * kLog2e : 0.f;
      drr[rr] = (softmax && i < Lq) ? drow[row] : 0.f;
#pragma unroll
      for (int t = 0; t < DQ / 32; ++t) acc[rr][t] = 0.f;
    }
    const int kend = p.causal ? min(Lk, row0 + kTileRows) : Lk;
    for (int kb = 0; kb < kend; kb += kStep) {
      __syncthreads();
      for (int idx = tid; idx < kStep * DQ; idx += kThreads) {
        int r = idx / DQ, d = idx % DQ;
        sm.k[r][d] = (kb + r < Lk && d < Dq) ? ld(k, ((k0 + kb + r) * H + h) * Dq + d) : 0.f;
      }
      for (int idx = tid; idx < kStep * DV; idx += kThreads) {
        int r = idx / DV, d = idx % DV;
        sm.v[r][d] = (kb + r < Lk && d < Dv) ? ld(v, ((k0 + kb + r) * H + h) * Dv + d) : 0.f;
      }
      __syncthreads();
      const int j = kb + lane;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = warp * kRowsPerWarp + rr, i = row0 + r;
        float s = 0.f, dp = 0.f;
#pragma unroll 8
        for (int d = 0; d < DQ; ++d) s = fmaf(sm.q[r][d], sm.k[lane][d], s);
#pragma unroll 8
        for (int d = 0; d < DV; ++d) dp = fmaf(sm.dout[r][d], sm.v[lane][d], dp);
        const bool valid = i < Lq && j < Lk && (!p.causal || j <= i);
        s -= valid ? 0.f : kMaskShift;
        float ds;
        if (softmax) {
          const float pj = exp2f(s - lse2[rr]);
          ds = pj * (dp - drr[rr]);
        } else {
          const float sg = sigmoidf_(s);
          ds = dp * sg * (1.f + s * (1.f - sg)) * inv_len;
        }
        if (!valid) ds = 0.f;
#pragma unroll 4
        for (int jj = 0; jj < kStep; ++jj) {
          const float dsj = __shfl_sync(0xffffffffu, ds, jj);
#pragma unroll
          for (int t = 0; t < DQ / 32; ++t) acc[rr][t] = fmaf(dsj, sm.k[jj][lane + 32 * t], acc[rr][t]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int i = row0 + warp * kRowsPerWarp + rr;
      if (i >= Lq) continue;
      const int64_t row = (q0 + i) * H + h;
#pragma unroll
      for (int t = 0; t < DQ / 32; ++t) {
        const int c = lane + 32 * t;
        if (c < Dq) st(dq, row * Dq + c, acc[rr][t] * p.scale);
      }
    }
  }
}

template <typename T, int DQ, int DV>
struct SimtDkdvSmem {
  float k[kTileRows][DQ];
  float v[kTileRows][DV];
  float q[kStep][DQ + 1];
  float dout[kStep][DV + 1];
  float lse2[kStep];
  float drow[kStep];
};

// dK/dV pass: one item = (b, h, 64-key k-tile); 8 warps x 8 keys; row steps of 32.
template <typename T, int DQ, int DV>
__global__ void __launch_bounds__(kThreads)
simt_dkdv_kernel(Problem p, const T* __restrict__ q, const T* __restrict__ k,
                 const T* __restrict__ v, const float* __restrict__ lse,
                 const float* __restrict__ drow, const T* __restrict__ dout,
                 T* __restrict__ dk, T* __restrict__ dv, const WsHeader* __restrict__ hdr,
                 const WorkItem* __restrict__ list) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<SimtDkdvSmem<T, DQ, DV>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int H = p.heads, Dq = p.dim_qk, Dv = p.dim_v;
  const float qf = q_factor(p);
  const bool softmax = p.act == kActSoftmax;
  const int n = hdr->n_k;
  for (int it = blockIdx.x; it < n; it += gridDim.x) {
    const WorkItem w = load_item(list, it);
    const int h = w.h, key0 = w.tile * kTileRows;
    const int64_t q0 = w.q0, k0 = w.k0;
    const int Lq = w.lq, Lk = w.lk;
    const float inv_len = 1.0f / (float)max(Lq, 1);
    __syncthreads();
    for (int idx = tid; idx < kTileRows * DQ; idx += kThreads) {
      int r = idx / DQ, d = idx % DQ;
      sm.k[r][d] = (key0 + r < Lk && d < Dq) ? ld(k, ((k0 + key0 + r) * H + h) * Dq + d) : 0.f;
    }
    for (int idx = tid; idx < kTileRows * DV; idx += kThreads) {
      int r = idx / DV, d = idx % DV;
      sm.v[r][d] = (key0 + r < Lk && d < Dv) ? ld(v, ((k0 + key0 + r) * H + h) * Dv + d) : 0.f;
    }
    float ak[kRowsPerWarp][DQ / 32], av[kRowsPerWarp][DV / 32];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
#pragma unroll
      for (int t = 0; t < DQ / 32; ++t) ak[rr][t] = 0.f;
#pragma unroll
      for (int t = 0; t < DV / 32; ++t) av[rr][t] = 0.f;
    }
    // causal: only rows >= key0 can see this tile (start on a step boundary)
    const int qstart = p.causal ? (key0 / kStep) * kStep : 0;
    for (int qb = qstart; qb < Lq; qb += kStep) {
      __syncthreads();
      for (int idx = tid; idx < kStep * DQ; idx += kThreads) {
        int r = idx / DQ, d = idx % DQ;
        sm.q[r][d] = (qb + r < Lq && d < Dq) ? ld(q, ((q0 + qb + r) * H + h) * Dq + d) * qf : 0.f;
      }
      for (int idx = tid; idx < kStep * DV; idx += kThreads) {
        int r = idx / DV, d = idx % DV;
        sm.dout[r][d] = (qb + r < Lq && d < Dv) ? ld(dout, ((q0 + qb + r) * H + h) * Dv + d) : 0.f;
      }
      if (tid < kStep) {
        const bool ok = qb + tid < Lq && softmax;
        sm.lse2[tid] = ok ? lse[(q0 + qb + tid) * H + h] * kLog2e : 0.f;
        sm.drow[tid] = ok ? drow[(q0 + qb + tid) * H + h] : 0.f;
      }
      __syncthreads();
      const int i = qb + lane;
#pragma unroll
      for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = warp * kRowsPerWarp + rr, j = key0 + r;
        float s = 0.f, dp = 0.f;
#pragma unroll 8
        for (int d = 0; d < DQ; ++d) s = fmaf(sm.q[lane][d], sm.k[r][d], s);
#pragma unroll 8
        for (int d = 0; d < DV; ++d) dp = fmaf(sm.dout[lane][d], sm.v[r][d], dp);
        const bool valid = i < Lq && j < Lk && (!p.causal || j <= i);
        s -= valid ? 0.f : kMaskShift;
        float pi, ds;
        if (softmax) {
          pi = exp2f(s - sm.lse2[lane]);
          ds = pi * (dp - sm.drow[lane]);
        } else {
          const float sg = sigmoidf_(s);
          pi = s * sg * inv_len;
          ds = dp * sg * (1.f + s * (1.f - sg)) * inv_len;
        }
        if (!valid) { pi = 0.f; ds = 0.f; }
#pragma unroll 4
        for (int ii = 0; ii < kStep; ++ii) {
          const float pv = __shfl_sync(0xffffffffu, pi, ii);
          const float dsv = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
          for (int t = 0; t < DV / 32; ++t) av[rr][t] = fmaf(pv, sm.dout[ii][lane + 32 * t], av[rr][t]);
#pragma unroll
          for (int t = 0; t < DQ / 32; ++t) ak[rr][t] = fmaf(dsv, sm.q[ii][lane + 32 * t], ak[rr][t]);
        }
      }
    }
    // sm.q held Q * qf, so dK = scale * sum ds q = ak * (scale / qf)
    const float kf = p.scale / qf;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int j = key0 + warp * kRowsPerWarp + rr;
      if (j >= Lk) continue;
      const int64_t row = (k0 + j) * H + h;
#pragma unroll
      for (int t = 0; t < DQ / 32; ++t) {
        const int c = lane + 32 * t;
        if (c < Dq) st(dk, row * Dq + c, ak[rr][t] * kf);
      }
#pragma unroll
      for (int t = 0; t < DV / 32; ++t) {
        const int c = lane + 32 * t;
        if (c < Dv) st(dv, row * Dv + c, av[rr][t]);
      }
    }
  }
}

int padded(int d) { return d <= 32 ? 32 : (d <= 64 ? 64 : 128); }

template <typename Kern>
cudaError_t launch_persistent(Kern kern, size_t smem, cudaStream_t s, void** args) {
  int per_sm = 0;
  cudaError_t e = kernel_setup((const void*)kern, kThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  dim3 grid(num_sms() * per_sm);
  return cudaLaunchKernel((const void*)kern, grid, dim3(kThreads), args, smem, s);
}

template <typename T, int DQ, int DV>
cudaError_t fwd_t(const Problem& p, const void* q, const void* k, const void* v, void* o,
                  float* lse, const Workspace& ws, cudaStream_t s) {
  Problem pp = p;
  const T* qq = (const T*)q; const T* kk = (const T*)k; const T* vv = (const T*)v;
  T* oo = (T*)o;
  const WsHeader* hdr = ws.hdr;
  const WorkItem* list = ws.list_q;
  void* args[] = {&pp, &qq, &kk, &vv, &oo, &lse, &hdr, &list};
  return launch_persistent(simt_fwd_kernel<T, DQ, DV>, sizeof(SimtFwdSmem<T, DQ, DV>), s, args);
}

template <typename T, int DQ, int DV>
cudaError_t dq_t(const Problem& p, const void* q, const void* k, const void* v,
                 const float* lse, const void* dout, void* dq, const Workspace& ws,
                 cudaStream_t s) {
  Problem pp = p;
  const T* qq = (const T*)q; const T* kk = (const T*)k; const T* vv = (const T*)v;
  const T* dd = (const T*)dout;
  T* gq = (T*)dq;
  const float* dr = ws.drow;
  const WsHeader* hdr = ws.hdr;
  const WorkItem* list = ws.list_q;
  void* args[] = {&pp, &qq, &kk, &vv, &lse, &dr, &dd, &gq, &hdr, &list};
  return launch_persistent(simt_dq_kernel<T, DQ, DV>, sizeof(SimtDqSmem<T, DQ, DV>), s, args);
}

template <typename T, int DQ, int DV>
cudaError_t dkdv_t(const Problem& p, const void* q, const void* k, const void* v,
                   const float* lse, const void* dout, void* dk, void* dv, const Workspace& ws,
                   cudaStream_t s) {
  Problem pp = p;
  const T* qq = (const T*)q; const T* kk = (const T*)k; const T* vv = (const T*)v;
  const T* dd = (const T*)dout;
  T* gk = (T*)dk; T* gv = (T*)dv;
  const float* dr = ws.drow;
  const WsHeader* hdr = ws.hdr;
  const WorkItem* list = ws.list_k;
  void* args[] = {&pp, &qq, &kk, &vv, &lse, &dr, &dd, &gk, &gv, &hdr, &list};
  return launch_persistent(simt_dkdv_kernel<T, DQ, DV>, sizeof(SimtDkdvSmem<T, DQ, DV>), s, args);
}

// Dispatch over (dtype, padded Dqk, padded Dv).
#define JFA_SIMT_DISPATCH(FN, ...)                                                        \
  do {                                                                                    \
    const int dq_ = padded(p.dim_qk), dv_ = padded(p.dim_v);                              \
    if (dtype == JFA_F32) {                                                               \
      JFA_SIMT_DIMS(float, FN, __VA_ARGS__);                                              \
    } else {                                                                              \
      JFA_SIMT_DIMS(__nv_bfloat16, FN, __VA_ARGS__);                                      \
    }                                                                                     \
    return cudaErrorInvalidValue;                                                         \
  } while (0)
#define JFA_SIMT_ONE(T, FN, A, B, ...) \
  if (dq_ == A && dv_ == B) return FN<T, A, B>(__VA_ARGS__)
#define JFA_SIMT_DIMS(T, FN, ...)            \
  JFA_SIMT_ONE(T, FN, 32, 32, __VA_ARGS__);  \
  JFA_SIMT_ONE(T, FN, 32, 64, __VA_ARGS__);  \
  JFA_SIMT_ONE(T, FN, 32, 128, __VA_ARGS__); \
  JFA_SIMT_ONE(T, FN, 64, 32, __VA_ARGS__);  \
  JFA_SIMT_ONE(T, FN, 64, 64, __VA_ARGS__);  \
  JFA_SIMT_ONE(T, FN, 64, 128, __VA_ARGS__); \
  JFA_SIMT_ONE(T, FN, 128, 32, __VA_ARGS__); \
  JFA_SIMT_ONE(T, FN, 128, 64, __VA_ARGS__); \
  JFA_SIMT_ONE(T, FN, 128, 128, __VA_ARGS__)

}  // namespace

const SchedConfig kSimtSched = {kTileRows, kStep, kTileRows, kStep, 1, 1, 0};

cudaError_t launch_simt_fwd(const Problem& p, int dtype, const void* q, const void* k,
                            const void* v, void* o, float* lse, const Workspace& ws,
                            cudaStream_t s) {
  JFA_SIMT_DISPATCH(fwd_t, p, q, k, v, o, lse, ws, s);
}

cudaError_t launch_simt_dq(const Problem& p, int dtype, const void* q, const void* k,
                           const void* v, const float* lse, const void* dout, void* dq,
                           const Workspace& ws, cudaStream_t s) {
  JFA_SIMT_DISPATCH(dq_t, p, q, k, v, lse, dout, dq, ws, s);
}

cudaError_t launch_simt_dkdv(const Problem& p, int dtype, const void* q, const void* k,
                             const void* v, const float* lse, const void* dout, void* dk,
                             void* dv, const Workspace& ws, cudaStream_t s) {
  JFA_SIMT_DISPATCH(dkdv_t, p, q, k, v, lse, dout, dk, dv, ws, s);
}

cudaError_t launch_bwd_rowterm(const Problem& p, int dtype, const void* o, const void* dout,
                               const Workspace& ws, cudaStream_t s) {
  const int64_t rows = p.total_q * p.heads;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + (kThreads / 32) - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (dtype == JFA_F32)
    rowterm_kernel<float><<<(unsigned)blocks, kThreads, 0, s>>>(rows, p.dim_v, (const float*)o,
                                                               (const float*)dout, ws.drow);
  else
    rowterm_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, s>>>(
        rows, p.dim_v, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dout, ws.drow);
  return cudaGetLastError();
}

}  // namespace jfa
