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
// Each item also carries its sequence's first rows and lengths, so a kernel
// needs one 32-byte load per item and no dependent offset lookups.
//
// The whole list is built by one CTA from the offsets in device memory, so a
// call never synchronises with the host and can be captured in a CUDA graph.
// The same kernel validates the offsets and writes the status word.  Per-
// sequence data and prefix sums live in shared memory for batches of up to
// kCacheB sequences and in the workspace beyond that.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 128;  // costs >= kBuckets-1 share the heaviest bucket
constexpr int kCacheB = 4096;  // sequences cached in shared memory

struct SchedShared {
  int warp_tot[32];
  int hist[kBuckets], start[kBuckets], run[kBuckets];
  int wcount[kWarps][kBuckets];
  int4 seq[kCacheB];        // (q0, k0, lq, lk)
  int pref[kCacheB + 1];    // tile prefix sums of the list being built
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

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

__device__ __forceinline__ int tiles_of(const ListSpec& L, int lq, int lk) {
  return cdiv(L.key_major ? lk : lq, L.tile);
}

// Inner steps the kernel runs for tile t of a sequence with lengths (lq, lk).
__device__ __forceinline__ int cost_of(const ListSpec& L, int causal, int lq, int lk, int t) {
  if (!L.key_major) {
    const int keys = causal ? min(lk, (t + 1) * L.tile) : lk;
    return cdiv(keys, L.step);
  }
  if (!causal) return cdiv(lq, L.step);
  // rows >= the first key of this tile, counted in whole inner steps
  return max(0, cdiv(lq, L.step) - (t * L.tile) / L.step);
}

// Sequence owning unit u: the largest b with pref[b] <= u.
__device__ __forceinline__ int find_seq(const int* pref, int B, int u) {
  int lo = 0, hi = B;  // pref[lo] <= u < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ void build_list(const Problem& p, const ListSpec& L, const int4* seq, int* pref,
                           WorkItem* list, int* n_out, SchedShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = (int)p.batch;
  // 1. tiles per sequence -> exclusive prefix sums in pref[0..B]
  int carry = 0;
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int cnt = 0;
    if (b < B) cnt = tiles_of(L, seq[b].z, seq[b].w);
    const int inc = block_inclusive_scan(cnt, sh.warp_tot);
    if (b < B) pref[b] = carry + inc - cnt;
    if (tid == kThreads - 1) sh.warp_tot[0] = inc;  // this round's total
    __syncthreads();
    carry += sh.warp_tot[0];
    __syncthreads();
  }
  if (tid == 0) pref[B] = carry;
  const int U = carry;
  for (int c = tid; c < kBuckets; c += kThreads) { sh.hist[c] = 0; sh.run[c] = 0; }
  for (int i = tid; i < kWarps * kBuckets; i += kThreads) (&sh.wcount[0][0])[i] = 0;
  __syncthreads();

  // 2. histogram of buckets
  for (int u = tid; u < U; u += kThreads) {
    const int b = find_seq(pref, B, u);
    const int4 s = seq[b];
    atomicAdd(&sh.hist[min(cost_of(L, p.causal, s.z, s.w, u - pref[b]), kBuckets - 1)], 1);
  }
  __syncthreads();
  // 3. bucket starts, heaviest bucket first
  if (warp == 0) {
    // descending exclusive scan over kBuckets counts, 4 buckets per lane
    int v[4], sum = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) { v[t] = sh.hist[kBuckets - 1 - (lane * 4 + t)]; sum += v[t]; }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    int acc = inc - sum;
#pragma unroll
    for (int t = 0; t < 4; ++t) { sh.start[kBuckets - 1 - (lane * 4 + t)] = acc; acc += v[t]; }
  }
  __syncthreads();

  // 4. stable placement, kThreads units per round
  for (int base = 0; base < U; base += kThreads) {
    const int u = base + tid;
    const bool valid = u < U;
    int b = 0, t = 0, cost = 0, c = -1;
    int4 s = make_int4(0, 0, 0, 0);
    if (valid) {
      b = find_seq(pref, B, u);
      t = u - pref[b];
      s = seq[b];
      cost = cost_of(L, p.causal, s.z, s.w, t);
      c = min(cost, kBuckets - 1);
    }
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) sh.wcount[warp][c] = __popc(peers);
    __syncthreads();
    for (int cc = tid; cc < kBuckets; cc += kThreads) {
      int acc = sh.run[cc];
      for (int w = 0; w < kWarps; ++w) {
        const int x = sh.wcount[w][cc];
        sh.wcount[w][cc] = acc;
        acc += x;
      }
      sh.run[cc] = acc;
    }
    __syncthreads();
    if (valid) {
      const int64_t pos = (int64_t)sh.start[c] + sh.wcount[warp][c] + rank;
      for (int h = 0; h < p.heads; ++h) {
        WorkItem w;
        w.b = b; w.h = h; w.tile = t; w.cost = cost;
        w.q0 = s.x; w.k0 = s.y; w.lq = s.z; w.lk = s.w;
        list[pos * p.heads + h] = w;
      }
    }
    __syncthreads();
    for (int i = tid; i < kWarps * kBuckets; i += kThreads) (&sh.wcount[0][0])[i] = 0;
    __syncthreads();
  }
  if (tid == 0) *n_out = U * p.heads;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_kernel(Problem p, Workspace ws, ListSpec lq_spec, ListSpec lk_spec, int build_q,
                int build_k, int self_attention) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SchedShared& sh = *reinterpret_cast<SchedShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int B = (int)p.batch;
  const bool cached = B <= kCacheB;
  int4* seq = cached ? sh.seq : ws.seq;
  int* pref_q = cached ? sh.pref : ws.q_prefix;
  int* pref_k = cached ? sh.pref : ws.k_prefix;

  // Validate: offs[0] == 0, non-decreasing, offs[B] == total; equal lengths
  // for self-attention.  Record (q0, k0, lq, lk) per sequence.
  int bad = 0;
  if (tid == 0) {
    bad |= (p.offs_q[0] != 0) | (p.offs_k[0] != 0);
    bad |= (p.offs_q[B] != p.total_q) | (p.offs_k[B] != p.total_k);
  }
  for (int b = tid; b < B; b += kThreads) {
    const int64_t q0 = p.offs_q[b], q1 = p.offs_q[b + 1];
    const int64_t k0 = p.offs_k[b], k1 = p.offs_k[b + 1];
    const int64_t lq = q1 - q0, lk = k1 - k0;
    int e = (lq < 0) | (lk < 0) | (q1 > p.total_q) | (k1 > p.total_k) | (q0 < 0) | (k0 < 0);
    if (self_attention) e |= (lq != lk);
    bad |= e;
    if (!e) seq[b] = make_int4((int)q0, (int)k0, (int)lq, (int)lk);
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
    build_list(p, lq_spec, seq, pref_q, ws.list_q, &ws.hdr->n_q, sh);
  else if (tid == 0)
    ws.hdr->n_q = 0;
  if (build_k)
    build_list(p, lk_spec, seq, pref_k, ws.list_k, &ws.hdr->n_k, sh);
  else if (tid == 0)
    ws.hdr->n_k = 0;
  if (tid == 0) ws.hdr->status = JFA_OK;
}

}  // namespace

cudaError_t launch_schedule(const Problem& p, const Workspace& ws, const SchedConfig& c,
                            cudaStream_t s) {
  ListSpec lq{false, c.q_rows, c.q_keys_step};
  ListSpec lk{true, c.k_keys, c.k_rows_step};
  const int smem = (int)sizeof(SchedShared);
  cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  schedule_kernel<<<1, kThreads, smem, s>>>(p, ws, lq, lk, c.build_q, c.build_k, c.self_attention);
  return cudaGetLastError();
}

}  // namespace jfa
