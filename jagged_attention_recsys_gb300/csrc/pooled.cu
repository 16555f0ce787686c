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

// offs_q[b] = b*m for b <= B; rows b*m + i of q_rep = row i of q (32-bit words).
__global__ void pooled_broadcast_kernel(const uint32_t* __restrict__ q, uint32_t* __restrict__ q_rep,
                                        int64_t* __restrict__ offs_q, int64_t batch, int32_t m,
                                        int64_t row_words) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = tid; b <= batch; b += stride) offs_q[b] = b * m;
  const int64_t per_seq = (int64_t)m * row_words;
  const int64_t total = batch * per_seq;
  for (int64_t e = tid; e < total; e += stride) q_rep[e] = q[e % per_seq];
}

// dq[e] = sum over b of dq_rep[b*m*row + e], accumulated in fp32 in sequence order.
template <typename T>
__global__ void pooled_reduce_kernel(const T* __restrict__ dq_rep, T* __restrict__ dq, int64_t batch,
                                     int64_t per_seq) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = tid; e < per_seq; e += stride) {
    float acc = 0.f;
    for (int64_t b = 0; b < batch; ++b) acc += static_cast<float>(dq_rep[b * per_seq + e]);
    dq[e] = static_cast<T>(acc);
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
  const int64_t row_words = row_bytes / 4;  // row_bytes is a multiple of 4 (checked by the caller)
  const int64_t n = batch * m * row_words > batch + 1 ? batch * m * row_words : batch + 1;
  pooled_broadcast_kernel<<<grid_for(n, 256), 256, 0, s>>>((const uint32_t*)q, (uint32_t*)q_rep, offs_q,
                                                           batch, m, row_words);
  return cudaGetLastError();
}

cudaError_t launch_pooled_reduce(int dtype, int64_t batch, int64_t per_seq_elems, const void* dq_rep,
                                 void* dq, cudaStream_t s) {
  const unsigned g = grid_for(per_seq_elems, 256);
  if (dtype == JFA_BF16)
    pooled_reduce_kernel<__nv_bfloat16><<<g, 256, 0, s>>>((const __nv_bfloat16*)dq_rep,
                                                          (__nv_bfloat16*)dq, batch, per_seq_elems);
  else
    pooled_reduce_kernel<float><<<g, 256, 0, s>>>((const float*)dq_rep, (float*)dq, batch, per_seq_elems);
  return cudaGetLastError();
}

}  // namespace jfa
