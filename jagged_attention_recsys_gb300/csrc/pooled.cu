// Pooled multi-head attention: m learned queries per head, shared by every sequence,
// attend each jagged sequence's keys and values.
//
// Meta GEM MFU write-up (piletech.kr/articles/112134), details section, jagged-input
// bullet: pooled multi-head attention is one of the attention patterns over jagged
// sequences.  It is the asymmetric cross-attention of the main path with every
// sequence's query block equal to the same m rows, so it runs on the cross-attention
// kernels: these two kernels broadcast the shared queries into the per-sequence query
// rows (with their offsets) before them, and sum the per-sequence query gradients
// after them, in a fixed order (no atomics; bitwise reproducible).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

// offs_q[b] = b*m for b <= B; rows b*m + i of q_rep = row i of q.  W is the copied word
// (16 bytes when a sequence's block of rows is a multiple of 16 bytes, else 4).  Threads
// along x own words of the shared block; CTAs along y take the sequences.
template <typename W>
__global__ void pooled_broadcast_kernel(const W* __restrict__ q, W* __restrict__ q_rep,
                                        int64_t* __restrict__ offs_q, int64_t batch, int32_t m,
                                        int64_t per_seq_words) {
  const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nx = (int64_t)gridDim.x * blockDim.x;
  if (blockIdx.y == 0)
    for (int64_t b = x; b <= batch; b += nx) offs_q[b] = b * m;
  for (int64_t w = x; w < per_seq_words; w += nx) {
    const W v = q[w];
    for (int64_t b = blockIdx.y; b < batch; b += gridDim.y) q_rep[b * per_seq_words + w] = v;
  }
}

// dq[e] = sum over b of dq_rep[b*per_seq + e], in fp32, in a fixed order: warp w of a CTA
// sums the sequences b = w, w + kSumWarps, ... in increasing b for 32 consecutive elements,
// then the warps' partial sums are added in warp order.  The order depends only on the
// sizes, so the result is bitwise reproducible (no atomics).
constexpr int kSumWarps = 16;

template <typename TI, typename T>
__global__ void __launch_bounds__(kSumWarps * 32)
pooled_reduce_kernel(const TI* __restrict__ dq_rep, T* __restrict__ dq, int64_t batch,
                     int64_t per_seq) {
  __shared__ float part[kSumWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t e0 = (int64_t)blockIdx.x * 32; e0 < per_seq; e0 += (int64_t)gridDim.x * 32) {
    const int64_t e = e0 + lane;
    float acc = 0.f;
    if (e < per_seq) {
#pragma unroll 4
      for (int64_t b = warp; b < batch; b += kSumWarps)
        acc += static_cast<float>(dq_rep[b * per_seq + e]);
    }
    part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && e < per_seq) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kSumWarps; ++w) sum += part[w][lane];
      dq[e] = static_cast<T>(sum);
    }
    __syncthreads();
  }
}

unsigned grid_for(int64_t n, int threads) {
  int64_t blocks = (n + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return (unsigned)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_pooled_broadcast(int64_t batch, int32_t m, int64_t row_bytes, const void* q,
                                    void* q_rep, int64_t* offs_q, cudaStream_t s) {
  // row_bytes is a multiple of 4 and q, q_rep are 16-byte aligned (checked by the caller)
  const int64_t per_seq_bytes = (int64_t)m * row_bytes;
  const bool wide = per_seq_bytes % 16 == 0;
  const int64_t words = per_seq_bytes / (wide ? 16 : 4);
  const int64_t xs = (words > batch + 1 ? words : batch + 1);
  const unsigned gx = grid_for(xs, 256);
  // enough CTAs along the sequences to fill the GPU about 8 CTAs deep
  int64_t gy = ((int64_t)num_sms() * 8 + gx - 1) / gx;
  if (gy > batch) gy = batch;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  const dim3 grid(gx, (unsigned)gy);
  if (wide)
    pooled_broadcast_kernel<uint4><<<grid, 256, 0, s>>>((const uint4*)q, (uint4*)q_rep, offs_q, batch, m,
                                                         words);
  else
    pooled_broadcast_kernel<uint32_t><<<grid, 256, 0, s>>>((const uint32_t*)q, (uint32_t*)q_rep, offs_q,
                                                           batch, m, words);
  return cudaGetLastError();
}

cudaError_t launch_pooled_reduce(int dtype, bool rep_f32, int64_t batch, int64_t per_seq_elems,
                                 const void* dq_rep, void* dq, cudaStream_t s) {
  int64_t blocks = (per_seq_elems + 31) / 32;
  const int64_t cap = (int64_t)num_sms() * 4;  // 4 CTAs of 512 threads per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dtype == JFA_BF16 && rep_f32)
    pooled_reduce_kernel<float, __nv_bfloat16><<<(unsigned)blocks, kSumWarps * 32, 0, s>>>(
        (const float*)dq_rep, (__nv_bfloat16*)dq, batch, per_seq_elems);
  else if (dtype == JFA_BF16)
    pooled_reduce_kernel<__nv_bfloat16, __nv_bfloat16><<<(unsigned)blocks, kSumWarps * 32, 0, s>>>(
        (const __nv_bfloat16*)dq_rep, (__nv_bfloat16*)dq, batch, per_seq_elems);
  else
    pooled_reduce_kernel<float, float><<<(unsigned)blocks, kSumWarps * 32, 0, s>>>(
        (const float*)dq_rep, (float*)dq, batch, per_seq_elems);
  return cudaGetLastError();
}

}  // namespace jfa
