// Jagged tile scheduler: offsets -> heavy-first work lists, built on the device.
//
// Meta GEM MFU write-up (piletech.kr/articles/112134), details section: the
// Generalized Dot-Product Attention bullet names software tile scheduling for
// jagged tensors, the Jagged Flash Attention bullet persistent-kernel
// scheduling, and the Base Batch Shuffling bullet pairs heavy and light work.
//
// Rule.  Every (sequence, head, tile) is one work item whose cost is the
// number of inner steps the kernel runs for it.  Sequences are ordered by
// their total cost, heaviest first (the longest-processing-time rule at
// sequence granularity; costs are bucketed into 128 levels relative to the
// heaviest sequence, ties by sequence index).  The tiles of one sequence are
// contiguous, heaviest tile first, and the heads of one tile are adjacent.
// Persistent CTAs take items i, i + grid, i + 2*grid, ..., or, for lists whose
// items average at least kClaimMinMeanCost steps, claim the next item from a
// counter as they become free (the SiLU/L kernels; see feed.cuh).  Either way the
// items that run at the same time belong to few sequences and share their K/V
// tiles through L2, while the heavy sequences start first.
// Each item also carries its sequence's first rows and lengths, so a kernel
// needs one 32-byte load per item and no dependent offset lookups.
//
// The lists are built from the offsets in device memory by one CTA (two when both
// lists are wanted and fit in shared memory, one list each), so a call never
// synchronises with the host and can be captured in a CUDA graph.  The
// same kernel validates the offsets and writes the status word.  Per-sequence
// arrays live in shared memory for up to kCacheB sequences and in the
// workspace beyond that.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace jfa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 128;
constexpr int kCacheB = 6144;  // sequences whose arrays fit in shared memory (32 B each)
static_assert(kWarps == 32, "the per-bucket prefix over warps takes one lane per warp");

struct SchedShared {
  int warp_tot[32];
  int hist[kBuckets], start[kBuckets], run[kBuckets];
  int wcount[kWarps][kBuckets + 1];  // padded: a bucket's column spans all 32 banks
  int red;
  unsigned long long ctot;  // total cost of the list's units
  int4 seq[kCacheB];      // (q0, k0, lq, lk)
  int ntile[kCacheB];     // tiles of the list being built
  int bucket[kCacheB];    // cost bucket of the sequence
  int order[kCacheB];     // sequences in list order
  int first[kCacheB + 1]; // first unit of the r-th sequence in list order
};

static_assert(sizeof(SchedShared) <= 232448, "scheduler arrays within one CTA's shared memory");

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
    int t = lane < kWarps ? warp_tot[lane] : 0;
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

// k-th tile of a sequence in list order (heaviest first): causal q-tiles grow
// in cost with the tile index, so they are taken from the last one.
__device__ __forceinline__ int tile_at(const ListSpec& L, int causal, int n, int k) {
  return (causal && !L.key_major) ? n - 1 - k : k;
}

struct Arrays {
  int4* seq;
  int* ntile;
  int* bucket;
  int* order;
  int* first;
};

// Lists whose items average at least this many steps are taken by the tensor-core
// kernels' CTAs from a counter as they become free; shorter items keep the fixed
// round-robin assignment, whose per-item cost is lower.
constexpr int kClaimMinMeanCost = 6;

__device__ void build_list(const Problem& p, const ListSpec& L, const Arrays& A, WorkItem* list,
                           int* n_out, int* claim0, int* claim1, SchedShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = (int)p.batch;

  // 1. tiles and total cost per sequence; the heaviest total
  long long cmax = 0, csum = 0;
  for (int b = tid; b < B; b += kThreads) {
    const int4 s = A.seq[b];
    const int n = tiles_of(L, s.z, s.w);
    long long c = 0;
    for (int t = 0; t < n; ++t) c += cost_of(L, p.causal, s.z, s.w, t);
    A.ntile[b] = n;
    A.bucket[b] = (int)min(c, (long long)0x7fffffff);  // total cost for now
    cmax = max(cmax, c);
    csum += c;
  }
  if (tid == 0) sh.ctot = 0;
  // block max
  for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  if (tid == 0) sh.red = 0;
  __syncthreads();
  if (lane == 0) atomicMax(&sh.red, (int)min(cmax, (long long)0x7fffffff));
  for (int o = 16; o > 0; o >>= 1) csum += __shfl_xor_sync(0xffffffffu, csum, o);
  if (lane == 0) atomicAdd(&sh.ctot, (unsigned long long)csum);
  for (int c = tid; c < kBuckets; c += kThreads) { sh.hist[c] = 0; sh.run[c] = 0; }
  for (int i = tid; i < kWarps * (kBuckets + 1); i += kThreads) (&sh.wcount[0][0])[i] = 0;
  __syncthreads();
  const long long top = sh.red;

  // 2. cost buckets (relative to the heaviest sequence) and their histogram; one atomic
  //    per bucket and warp (equal costs are common: fixed-size blocks all share one)
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int k = -1;
    if (b < B) {
      const long long c = A.bucket[b];
      k = top > 0 ? (int)(c * (kBuckets - 1) / top) : 0;
      A.bucket[b] = k;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, k);
    if (k >= 0 && lane == __ffs(peers) - 1) atomicAdd(&sh.hist[k], __popc(peers));
  }
  __syncthreads();
  // 3. bucket starts, heaviest bucket first (descending exclusive scan, 4 buckets per lane)
  if (warp == 0) {
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

  // 4. stable counting sort of the sequences by bucket -> order[]
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    const bool valid = b < B;
    const int c = valid ? A.bucket[b] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) sh.wcount[warp][c] = __popc(peers);
    __syncthreads();
    // per bucket, exclusive prefix of the warps' counts: one warp per bucket, lane w
    // holding warp w's count
    for (int cc = warp; cc < kBuckets; cc += kWarps) {
      const int x = sh.wcount[lane][cc];
      const int before = sh.run[cc];
      int inc = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      sh.wcount[lane][cc] = before + inc - x;
      __syncwarp();
      if (lane == 31) sh.run[cc] = before + inc;
    }
    __syncthreads();
    if (valid) A.order[sh.start[c] + sh.wcount[warp][c] + rank] = b;
    __syncthreads();
    for (int i = tid; i < kWarps * (kBuckets + 1); i += kThreads) (&sh.wcount[0][0])[i] = 0;
    __syncthreads();
  }

  // 5. first unit of every sequence in list order
  int carry = 0;
  for (int base = 0; base < B; base += kThreads) {
    const int r = base + tid;
    const int cnt = r < B ? A.ntile[A.order[r]] : 0;
    const int inc = block_inclusive_scan(cnt, sh.warp_tot);
    if (r < B) A.first[r] = carry + inc - cnt;
    if (tid == kThreads - 1) sh.warp_tot[0] = inc;  // this round's total
    __syncthreads();
    carry += sh.warp_tot[0];
    __syncthreads();
  }

  // 6. write the items (unit u = sequence tile, item u * H + h).  A warp takes 32
  //    consecutive units, one per lane: the lane finds its unit's sequence by a binary
  //    search of the units' prefix first[] (sequences without units are skipped) and forms
  //    the unit's fields.  The warp then writes the 32 units' items in order, lane l of a
  //    round writing the round's item l with its unit's fields fetched by shuffles, so the
  //    warp's 32-byte stores are consecutive and each unit costs one search, not H.
  //    Item counts stay below 2^31 (checked on the host), so the indices are 32-bit.
  const int n_units = carry, H = p.heads;
  for (int u0 = warp * 32; u0 < n_units; u0 += kThreads) {
    const int u = u0 + lane;
    int fb = 0, ft = 0, fc = 0;
    int4 fs = make_int4(0, 0, 0, 0);
    if (u < n_units) {
      int lo = 0, hi = B - 1;  // the last r with first[r] <= u
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (A.first[mid] <= u) lo = mid; else hi = mid - 1;
      }
      fb = A.order[lo];
      fs = A.seq[fb];
      ft = tile_at(L, p.causal, A.ntile[fb], u - A.first[lo]);
      fc = cost_of(L, p.causal, fs.z, fs.w, ft);
    }
    const int n = min(32, n_units - u0) * H;  // items of this warp's units
    WorkItem* dst = list + (int64_t)u0 * H;
    for (int e0 = 0; e0 < n; e0 += 32) {  // uniform over the warp: every lane shuffles
      const int e = e0 + lane, src = min(e, n - 1) / H;
      WorkItem w;
      w.b = __shfl_sync(0xffffffffu, fb, src);
      w.h = e - src * H;
      w.tile = __shfl_sync(0xffffffffu, ft, src);
      w.cost = __shfl_sync(0xffffffffu, fc, src);
      w.q0 = __shfl_sync(0xffffffffu, fs.x, src);
      w.k0 = __shfl_sync(0xffffffffu, fs.y, src);
      w.lq = __shfl_sync(0xffffffffu, fs.z, src);
      w.lk = __shfl_sync(0xffffffffu, fs.w, src);
      if (e < n) dst[e] = w;
    }
  }
  const int n_items = n_units * H;
  if (tid == 0) {
    *n_out = n_items;
    // claim counters of the kernels that walk this list: 0 (taken from), or -1 (fixed
    // assignment)
    const int init = sh.ctot >= (unsigned long long)kClaimMinMeanCost * (unsigned long long)carry ? 0 : -1;
    *claim0 = init;
    if (claim1) *claim1 = init;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_kernel(Problem p, Workspace ws, ListSpec lq_spec, ListSpec lk_spec, int build_q,
                int build_k, int self_attention) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SchedShared& sh = *reinterpret_cast<SchedShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int B = (int)p.batch;
  Arrays A;
  if (B <= kCacheB) {
    A = Arrays{sh.seq, sh.ntile, sh.bucket, sh.order, sh.first};
  } else {
    A = Arrays{ws.seq, ws.seq_ints, ws.seq_ints + (B + 1), ws.seq_ints + 2 * (B + 1),
               ws.seq_ints + 3 * (B + 1)};
  }

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
    if (!e) A.seq[b] = make_int4((int)q0, (int)k0, (int)lq, (int)lk);
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) {
      ws.hdr->status = JFA_ERR_BAD_OFFSETS;
      ws.hdr->n_q = 0;
      ws.hdr->n_k = 0;
      for (int c = 0; c < 3; ++c) ws.hdr->claim[c] = 0;
    }
    return;
  }
  // With two CTAs (both lists wanted, per-sequence arrays in each CTA's shared memory),
  // CTA 0 builds the q-list and CTA 1 the k-list; both validated the same offsets.
  const bool split = gridDim.x == 2;
  if (!split || blockIdx.x == 0) {
    if (build_q)
      build_list(p, lq_spec, A, ws.list_q, &ws.hdr->n_q, &ws.hdr->claim[kClaimFwd], &ws.hdr->claim[kClaimDq], sh);
    else if (tid == 0)
      ws.hdr->n_q = 0;
  }
  if (!split || blockIdx.x == 1) {
    if (build_k)
      build_list(p, lk_spec, A, ws.list_k, &ws.hdr->n_k, &ws.hdr->claim[kClaimDkdv], nullptr, sh);
    else if (tid == 0)
      ws.hdr->n_k = 0;
  }
  if (tid == 0) ws.hdr->status = JFA_OK;
}

}  // namespace

cudaError_t launch_schedule(const Problem& p, const Workspace& ws, const SchedConfig& c,
                            cudaStream_t s) {
  ListSpec lq{false, c.q_rows, c.q_keys_step};
  ListSpec lk{true, c.k_keys, c.k_rows_step};
  const int smem = (int)sizeof(SchedShared);
  cudaError_t e = kernel_setup((const void*)schedule_kernel, kThreads, smem);
  if (e != cudaSuccess) return e;
  // both lists from two CTAs at once when each CTA can keep its own per-sequence arrays
  const int grid = (c.build_q && c.build_k && p.batch <= kCacheB) ? 2 : 1;
  schedule_kernel<<<grid, kThreads, smem, s>>>(p, ws, lq, lk, c.build_q, c.build_k, c.self_attention);
  return cudaGetLastError();
}

}  // namespace jfa
