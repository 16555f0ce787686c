// BlockAttention: every row attends only the keys of its own fixed 64-row block.
//
// Meta GEM MFU write-up (piletech.kr/articles/112134), details section, BlockAttention
// bullet: fixed 64-token blocks turn attention from quadratic into linear in the sequence
// length.  A block is the rows 64c .. 64c+63 of a sequence, counted from its first row (the
// last block may be shorter).  Attention restricted to blocks is jagged attention over
// pieces of the sequences, so this kernel only rewrites the offsets: sequence b of length
// L becomes ceil(L/P) pieces of P rows.  On the fp32 path a piece is one block (P = 64)
// and the kernels run on the piece offsets unchanged; on the tensor-core path a piece is
// two blocks (P = 128, one MMA tile), and the kernels mask each row to its own block's
// keys, which halves the tiles and the work items.  The piece count depends on the
// lengths, which only the device holds, so the host reserves B + ceil(T/P) piece
// sequences (an upper bound) and the unused ones at the end are empty.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

constexpr int kThreads = 1024;

// Inclusive scan of one value per thread over the CTA (warp shuffles + one warp of totals).
__device__ int64_t cta_inclusive_scan(int64_t x, int64_t* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t t = warp_tot[lane];  // kThreads / 32 == 32 warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int64_t r = x + (warp > 0 ? warp_tot[warp - 1] : 0);
  __syncthreads();
  return r;
}

// out[0 .. n_out] (n_out + 1 entries): the piece offsets (pieces of `block` rows), then
// empty piece sequences up to n_out.  Offsets that are not a valid jagged layout give out[0] = -1, which the scheduler
// reports as JFA_ERR_BAD_OFFSETS (nothing is then computed).
__global__ void __launch_bounds__(kThreads, 1)
block_offsets_kernel(const int64_t* __restrict__ offs, int64_t batch, int64_t total, int block,
                     int64_t* __restrict__ out, int64_t n_out) {
  __shared__ int64_t warp_tot[32];
  __shared__ int64_t carry_sh;
  const int tid = threadIdx.x;
  int bad = 0;
  if (tid == 0) bad |= (offs[0] != 0) | (offs[batch] != total);
  for (int64_t b = tid; b < batch; b += kThreads) bad |= offs[b + 1] < offs[b];
  if (__syncthreads_or(bad)) {
    if (tid == 0) out[0] = -1;
    return;
  }
  if (tid == 0) carry_sh = 0;
  __syncthreads();
  for (int64_t base = 0; base < batch; base += kThreads) {
    const int64_t b = base + tid;
    const int64_t len = b < batch ? offs[b + 1] - offs[b] : 0;
    const int64_t cnt = (len + block - 1) / block;
    const int64_t first = carry_sh + cta_inclusive_scan(cnt, warp_tot) - cnt;
    for (int64_t c = 0; c < cnt; ++c) out[first + c] = offs[b] + c * block;
    __syncthreads();
    if (tid == kThreads - 1) carry_sh = first + cnt;
    __syncthreads();
  }
  for (int64_t i = carry_sh + tid; i <= n_out; i += kThreads) out[i] = total;
}

// (cos, sin) of the rotary angle p * base^(-2i/dim) for p < npos and i < dim/2
__global__ void rope_table_kernel(float2* __restrict__ table, int npos, int half, double base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= npos * half) return;
  const int p = idx / half, i = idx % half;
  const double theta = (double)p * pow(base, -2.0 * (double)i / (double)(2 * half));
  table[idx] = make_float2((float)cos(theta), (float)sin(theta));
}

}  // namespace

cudaError_t launch_rope_table(float2* table, int npos, int dim, double base, cudaStream_t s) {
  const int n = npos * (dim / 2);
  rope_table_kernel<<<(n + 255) / 256, 256, 0, s>>>(table, npos, dim / 2, base);
  return cudaGetLastError();
}

cudaError_t launch_block_offsets(const int64_t* offs, int64_t batch, int64_t total, int block,
                                 int64_t* out, int64_t n_out, cudaStream_t s) {
  block_offsets_kernel<<<1, kThreads, 0, s>>>(offs, batch, total, block, out, n_out);
  return cudaGetLastError();
}

}  // namespace jfa
