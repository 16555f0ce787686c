// Jagged tile scheduler: offsets -> heavy-first work lists, built on the device.
//
// Meta GEM MFU write-up (piletech.kr/articles/112134), details section: the
// Generalized Dot-Product Attention bullet names software tile scheduling for
// jagged tensors, the Jagged Flash Attention bullet persistent-kernel
// scheduling, and the Base Batch Shuffling bullet pairs heavy and light work.
// Here every (sequence, head, tile) becomes one work item with an integer
// cost (inner-loop steps); items are ordered by cost, heaviest first (the
// longest-processing-time rule), ties by (sequence, tile) ascending, heads
// adjacent.  Persistent CTAs then take items i, i + grid, i + 2*grid, ...
//
// The whole list is built by one CTA from the offsets in device memory, so a
// call never synchronises with the host and can be captured in a CUDA graph.
// The same kernel validates the offsets and writes the status word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 128;  // costs >= kBuckets-1 share the heaviest bucket

__device__ __forceinline__ int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Inclusive block-wide scan of one int per thread.
__device__ int block_inclusive_scan(int x, int* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int res = x + (warp > 0 ? warp_tot[warp - 1] : 0);
  __syncthreads();
  return res;
}

struct ListSpec {
  bool key_major;  // false: q-tiles, true: k-tiles
  int tile;        // rows (q-list) or keys (k-list) per item
  int step;        // keys (q-list) or rows (k-list) per inner step
};

// Number of tiles of sequence b and the cost of tile t.
__device__ __forceinline__ int tiles_of(const ListSpec& L, int64_t lq, int64_t lk) {
  return (int)cdiv64(L.key_major ? lk : lq, L.tile);
}

__device__ __forceinline__ int cost_of(const ListSpec& L, int causal, int64_t lq, int64_t lk,
                                       int t) {
  int64_t c;
  if (!L.key_major) {
    int64_t keys = causal ? min(lk, (int64_t)(t + 1) * L.tile) : lk;
    c = cdiv64(keys, L.step);
  } else if (!causal) {
    c = cdiv64(lq, L.step);
  } else {
    // rows >= the first key of this tile, counted in whole inner steps
    int64_t first = ((int64_t)t * L.tile) / L.step;
    c = cdiv64(lq, L.step) - first;
    if (c < 0) c = 0;
  }
  return (int)c;
}

// Sequence owning unit u: the largest b with prefix[b] <= u.
__device__ __forceinline__ int find_seq(const int* prefix, int64_t B, int u) {
  int64_t lo = 0, hi = B;  // prefix[lo] <= u < prefix[hi]
  while (hi - lo > 1) {
    int64_t mid = (lo + hi) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid;
  }
  return (int)lo;
}

__device__ void build_list(const Problem& p, const ListSpec& L, int* prefix, WorkItem* list,
                           int* n_out, int* warp_tot, int* hist, int* start, int* run,
                           int (*wcount)[kBuckets]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t B = p.batch;
  // 1. tiles per sequence -> exclusive prefix sums in prefix[0..B]
  int carry = 0;
  for (int64_t base = 0; base < B; base += kThreads) {
    int64_t b = base + tid;
    int cnt = 0;
    if (b < B) {
      int64_t lq = p.offs_q[b + 1] - p.offs_q[b];
      int64_t lk = p.offs_k[b + 1] - p.offs_k[b];
      cnt = tiles_of(L, lq, lk);
    }
    int inc = block_inclusive_scan(cnt, warp_tot);
    if (b < B) prefix[b] = carry + inc - cnt;
    // the last thread's inclusive value is this round's total
    if (tid == kThreads - 1) warp_tot[0] = inc;
    __syncthreads();
    carry += warp_tot[0];
    __syncthreads();
  }
  if (tid == 0) prefix[B] = carry;
  const int U = carry;
  for (int c = tid; c < kBuckets; c += kThreads) { hist[c] = 0; run[c] = 0; }
  for (int i = tid; i < kWarps * kBuckets; i += kThreads) (&wcount[0][0])[i] = 0;
  __syncthreads();

  // 2. histogram of buckets
  for (int u = tid; u < U; u += kThreads) {
    int b = find_seq(prefix, B, u);
    int t = u - prefix[b];
    int64_t lq = p.offs_q[b + 1] - p.offs_q[b];
    int64_t lk = p.offs_k[b + 1] - p.offs_k[b];
    int c = min(cost_of(L, p.causal, lq, lk, t), kBuckets - 1);
    atomicAdd(&hist[c], 1);
  }
  __syncthreads();
  // 3. bucket starts, heaviest bucket first
  if (tid == 0) {
    int acc = 0;
    for (int c = kBuckets - 1; c >= 0; --c) { start[c] = acc; acc += hist[c]; }
  }
  __syncthreads();

  // 4. stable placement, kThreads units per round
  for (int base = 0; base < U; base += kThreads) {
    int u = base + tid;
    bool valid = u < U;
    int b = 0, t = 0, cost = 0, c = -1;
    if (valid) {
      b = find_seq(prefix, B, u);
      t = u - prefix[b];
      int64_t lq = p.offs_q[b + 1] - p.offs_q[b];
      int64_t lk = p.offs_k[b + 1] - p.offs_k[b];
      cost = cost_of(L, p.causal, lq, lk, t);
      c = min(cost, kBuckets - 1);
    }
    unsigned peers = __match_any_sync(0xffffffffu, c);
    int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wcount[warp][c] = __popc(peers);
    __syncthreads();
    for (int cc = tid; cc < kBuckets; cc += kThreads) {
      int acc = run[cc];
      for (int w = 0; w < kWarps; ++w) {
        int x = wcount[w][cc];
        wcount[w][cc] = acc;
        acc += x;
      }
      run[cc] = acc;
    }
    __syncthreads();
    if (valid) {
      int64_t pos = (int64_t)start[c] + wcount[warp][c] + rank;
      for (int h = 0; h < p.heads; ++h) list[pos * p.heads + h] = make_int4(b, h, t, cost);
    }
    __syncthreads();
    for (int i = tid; i < kWarps * kBuckets; i += kThreads) (&wcount[0][0])[i] = 0;
    __syncthreads();
  }
  if (tid == 0) *n_out = U * p.heads;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_kernel(Problem p, Workspace ws, ListSpec lq_spec, ListSpec lk_spec, int build_q,
                int build_k, int self_attention) {
  __shared__ int warp_tot[32];
  __shared__ int hist[kBuckets], start[kBuckets], run[kBuckets];
  __shared__ int wcount[kWarps][kBuckets];
  const int tid = threadIdx.x;
  const int64_t B = p.batch;

  // Validate: offs[0] == 0, non-decreasing, offs[B] == total; equal lengths
  // for self-attention.
  int bad = 0;
  if (tid == 0) {
    bad |= (p.offs_q[0] != 0) | (p.offs_k[0] != 0);
    bad |= (p.offs_q[B] != p.total_q) | (p.offs_k[B] != p.total_k);
  }
  for (int64_t b = tid; b < B; b += kThreads) {
    int64_t lq = p.offs_q[b + 1] - p.offs_q[b];
    int64_t lk = p.offs_k[b + 1] - p.offs_k[b];
    bad |= (lq < 0) | (lk < 0);
    bad |= (lq > 0x3fffffffLL) | (lk > 0x3fffffffLL);
    if (self_attention) bad |= (lq != lk);
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) {
      ws.hdr->status = JFA_ERR_BAD_OFFSETS;
      ws.hdr->n_q = 0;
      ws.hdr->n_k = 0;
    }
    return;
  }
  if (build_q)
    build_list(p, lq_spec, ws.q_prefix, ws.list_q, &ws.hdr->n_q, warp_tot, hist, start, run,
               wcount);
  else if (tid == 0)
    ws.hdr->n_q = 0;
  if (build_k)
    build_list(p, lk_spec, ws.k_prefix, ws.list_k, &ws.hdr->n_k, warp_tot, hist, start, run,
               wcount);
  else if (tid == 0)
    ws.hdr->n_k = 0;
  if (tid == 0) ws.hdr->status = JFA_OK;
}

}  // namespace

cudaError_t launch_schedule(const Problem& p, const Workspace& ws, const SchedConfig& c,
                            cudaStream_t s) {
  ListSpec lq{false, c.q_rows, c.q_keys_step};
  ListSpec lk{true, c.k_keys, c.k_rows_step};
  schedule_kernel<<<1, kThreads, 0, s>>>(p, ws, lq, lk, c.build_q, c.build_k, c.self_attention);
  return cudaGetLastError();
}

}  // namespace jfa
