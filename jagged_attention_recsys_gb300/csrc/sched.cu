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
// The lists are built from the offsets in device memory, so a call never
// synchronises with the host and can be captured in a CUDA graph.  The same kernel
// validates the offsets and writes the status word.  Per-sequence arrays live in
// shared memory for up to kCacheB sequences (sized to the batch, so that a small batch
// asks for little) and in the workspace beyond that.  Each CTA computes a list's whole
// order and prefix, which takes a few thousand cycles and no communication; one SM then
// stores only about 16 bytes a cycle, so a large list is written by several CTAs, each
// taking a share of the units ("slices"), and both lists, when both are wanted and the
// arrays fit in shared memory, by separate CTAs.  Past kCacheB sequences one CTA builds
// everything, in the workspace.
#include <cuda_runtime.h>

#include <algorithm>
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
  int wmax[kWarps];                  // per warp: the heaviest sequence's cost
  unsigned long long wsum[kWarps];   // per warp: the summed cost of its sequences
};

// Per-sequence arrays in shared memory, after SchedShared, for up to `cap` sequences:
// seq (q0, k0, lq, lk) int4 [cap], then int ntile [cap] (tiles of the list being built),
// bucket [cap] (cost bucket), order [cap] (sequences in list order) and first [cap + 1]
// (first unit of the r-th sequence in list order).  A launch reserves them for its own
// batch only, so that a small batch asks for little shared memory.
constexpr size_t kSeqArraysOff = (sizeof(SchedShared) + 15) / 16 * 16;
__host__ __device__ constexpr size_t sched_smem_bytes(int cap) {
  return kSeqArraysOff + 16 * (size_t)cap + 4 * (4 * (size_t)cap + 1);
}
static_assert(sched_smem_bytes(kCacheB) <= 232448, "scheduler arrays within one CTA's shared memory");

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

// Tiles and steps are powers of two (checked on the host), so the scheduler divides by
// shifting.
struct ListSpec {
  bool key_major;  // false: q-tiles, true: k-tiles
  int tile;        // rows (q-list) or keys (k-list) per item
  int step;        // keys (q-list) or rows (k-list) per inner step
  int tile_shift, step_shift;  // log2 of tile and step
};

__device__ __forceinline__ int cdiv_shift(int a, int sh) { return (a + (1 << sh) - 1) >> sh; }

__device__ __forceinline__ int tiles_of(const ListSpec& L, int lq, int lk) {
  return cdiv_shift(L.key_major ? lk : lq, L.tile_shift);
}

// Inner steps the kernel runs for tile t of a sequence with lengths (lq, lk).
__device__ __forceinline__ int cost_of(const ListSpec& L, int causal, int lq, int lk, int t) {
  if (!L.key_major) {
    const int keys = causal ? min(lk, (t + 1) * L.tile) : lk;
    return cdiv_shift(keys, L.step_shift);
  }
  if (!causal) return cdiv_shift(lq, L.step_shift);
  // rows >= the first key of this tile, counted in whole inner steps
  return max(0, cdiv_shift(lq, L.step_shift) - ((t * L.tile) >> L.step_shift));
}

// Total cost of a sequence's n tiles: closed form where every tile costs the same.
__device__ __forceinline__ long long total_cost(const ListSpec& L, int causal, int lq, int lk, int n) {
  if (!causal) return (long long)n * cost_of(L, 0, lq, lk, 0);
  long long c = 0;
  for (int t = 0; t < n; ++t) c += cost_of(L, causal, lq, lk, t);
  return c;
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

// Builds one list.  Slice `slice` of `slices` CTAs building the same list: every CTA
// computes the whole order and prefix (steps 1-5, a few thousand cycles) and writes the
// items of its own share of the units only, so large lists are written by many SMs
// without any CTA waiting for another.  Slice 0 writes the list's count and counters.
__device__ void build_list(const Problem& p, const ListSpec& L, const Arrays& A, WorkItem* list,
                           int* n_out, int* claim0, int* claim1, SchedShared& sh, int slice,
                           int slices) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = (int)p.batch;

  // 1. tiles and total cost per sequence; the heaviest total (per-warp partials, then
  //    every thread reads the 32 warps' maxima)
  int cmax = 0;
  unsigned long long csum = 0;
  for (int b = tid; b < B; b += kThreads) {
    const int4 s = A.seq[b];
    const int n = tiles_of(L, s.z, s.w);
    const long long c = total_cost(L, p.causal, s.z, s.w, n);
    A.ntile[b] = n;
    const int ci = (int)min(c, (long long)0x7fffffff);
    A.bucket[b] = ci;  // total cost for now
    cmax = max(cmax, ci);
    csum += (unsigned long long)c;
  }
  for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
  for (int o = 16; o > 0; o >>= 1) csum += __shfl_xor_sync(0xffffffffu, csum, o);
  if (lane == 0) {
    sh.wmax[warp] = cmax;
    sh.wsum[warp] = csum;
  }
  for (int c = tid; c < kBuckets; c += kThreads) { sh.hist[c] = 0; sh.run[c] = 0; }
  for (int i = tid; i < kWarps * (kBuckets + 1); i += kThreads) (&sh.wcount[0][0])[i] = 0;
  __syncthreads();
  int top = 0;
  for (int w = 0; w < kWarps; ++w) top = max(top, sh.wmax[w]);

  // 2. cost buckets (relative to the heaviest sequence) and their histogram; one atomic
  //    per bucket and warp (equal costs are common: fixed-size blocks all share one)
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int k = -1;
    if (b < B) {
      const int c = A.bucket[b];  // 0 <= c <= top
      if (top <= 0)
        k = 0;
      else if (top < (1 << 24))  // c (kBuckets - 1) fits 32 bits
        k = (int)((unsigned)c * (unsigned)(kBuckets - 1) / (unsigned)top);
      else
        k = (int)((long long)c * (kBuckets - 1) / top);
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
  if (B <= kThreads) {
    // one round: a sequence's place in its bucket is the number of same-bucket sequences
    // in earlier lanes of its warp plus those in earlier warps, summed directly from the
    // per-warp counts (zeroed in step 1)
    const int b = tid;
    const bool valid = b < B;
    const int c = valid ? A.bucket[b] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) sh.wcount[warp][c] = __popc(peers);
    __syncthreads();
    if (valid) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += sh.wcount[w][c];
      A.order[sh.start[c] + before + rank] = b;
    }
    __syncthreads();
  }
  for (int base = 0; B > kThreads && base < B; base += kThreads) {
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

  // 6. write the items (unit u = sequence tile, item u * H + h) of this slice's units.  A
  //    warp takes 32 consecutive units, one per lane: the lane finds its unit's sequence by
  //    a binary search of the units' prefix first[] (sequences without units are skipped)
  //    and forms the unit's two 16-byte halves.  The warp then writes the units' items in
  //    order, 16 per store instruction: lane l stores half l & 1 of item l >> 1 with the
  //    fields fetched from the unit's lane by shuffles, so each instruction fills 512
  //    contiguous bytes.  One search per unit, not per item.
  //    Item counts stay below 2^31 (checked on the host), so the indices are 32-bit.
  const int n_units = carry, H = p.heads;
  const int u_lo = (int)((long long)n_units * slice / slices);
  const int u_hi = (int)((long long)n_units * (slice + 1) / slices);
  const int half = lane & 1;
  for (int u0 = u_lo + warp * 32; u0 < u_hi; u0 += kThreads) {
    const int u = u0 + lane;
    int4 fa = make_int4(0, 0, 0, 0);  // (b, -, tile, cost)
    int4 fs = make_int4(0, 0, 0, 0);  // (q0, k0, lq, lk)
    if (u < u_hi) {
      int lo = 0, hi = B - 1;  // the last r with first[r] <= u
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (A.first[mid] <= u) lo = mid; else hi = mid - 1;
      }
      const int b = A.order[lo];
      fs = A.seq[b];
      const int t = tile_at(L, p.causal, A.ntile[b], u - A.first[lo]);
      fa = make_int4(b, 0, t, cost_of(L, p.causal, fs.z, fs.w, t));
    }
    const int n = min(32, u_hi - u0) * H;  // items of this warp's units
    int4* dst = reinterpret_cast<int4*>(list + (int64_t)u0 * H);
    for (int e0 = 0; e0 < n; e0 += 16) {  // uniform over the warp: every lane shuffles
      const int e = e0 + (lane >> 1), src = min(e, n - 1) / H;
      const int a0 = __shfl_sync(0xffffffffu, fa.x, src), a2 = __shfl_sync(0xffffffffu, fa.z, src);
      const int a3 = __shfl_sync(0xffffffffu, fa.w, src), s0 = __shfl_sync(0xffffffffu, fs.x, src);
      const int s1 = __shfl_sync(0xffffffffu, fs.y, src), s2 = __shfl_sync(0xffffffffu, fs.z, src);
      const int s3 = __shfl_sync(0xffffffffu, fs.w, src);
      const int4 v = half ? make_int4(s0, s1, s2, s3) : make_int4(a0, e - src * H, a2, a3);
      if (e < n) dst[2 * e + half] = v;
    }
  }
  const int n_items = n_units * H;
  if (tid == 0 && slice == 0) {
    *n_out = n_items;
    // claim counters of the kernels that walk this list: 0 (taken from), or -1 (fixed
    // assignment)
    unsigned long long ctot = 0;  // total cost of the list's units
    for (int w = 0; w < kWarps; ++w) ctot += sh.wsum[w];
    const int init = ctot >= (unsigned long long)kClaimMinMeanCost * (unsigned long long)carry ? 0 : -1;
    *claim0 = init;
    if (claim1) *claim1 = init;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
schedule_kernel(Problem p, Workspace ws, ListSpec lq_spec, ListSpec lk_spec, int build_q,
                int build_k, int self_attention, int split, int slices) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SchedShared& sh = *reinterpret_cast<SchedShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int B = (int)p.batch;
  Arrays A;
  if (B <= kCacheB) {
    int4* seq = reinterpret_cast<int4*>(smem_raw + kSeqArraysOff);
    int* ints = reinterpret_cast<int*>(seq + B);
    A = Arrays{seq, ints, ints + B, ints + 2 * B, ints + 3 * B};
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
    if (tid == 0 && blockIdx.x == 0) {
      ws.hdr->status = JFA_ERR_BAD_OFFSETS;
      ws.hdr->n_q = 0;
      ws.hdr->n_k = 0;
      for (int c = 0; c < 3; ++c) ws.hdr->claim[c] = 0;
    }
    return;
  }
  // With split (both lists wanted, per-sequence arrays in each CTA's shared memory),
  // even CTAs build the q-list and odd ones the k-list; both validated the same offsets.
  // The CTAs of one list are its slices.
  const int which = split ? (int)(blockIdx.x & 1) : -1;
  const int slice = split ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  if (which != 1) {
    if (build_q)
      build_list(p, lq_spec, A, ws.list_q, &ws.hdr->n_q, &ws.hdr->claim[kClaimFwd], &ws.hdr->claim[kClaimDq], sh,
                 slice, slices);
    else if (tid == 0 && slice == 0)
      ws.hdr->n_q = 0;
  }
  if (which != 0) {
    if (build_k)
      build_list(p, lk_spec, A, ws.list_k, &ws.hdr->n_k, &ws.hdr->claim[kClaimDkdv], nullptr, sh, slice, slices);
    else if (tid == 0 && slice == 0)
      ws.hdr->n_k = 0;
  }
  if (tid == 0 && blockIdx.x == 0) ws.hdr->status = JFA_OK;
}

}  // namespace

int log2_exact(int x) {  // log2 of a power of two, else -1
  if (x <= 0 || (x & (x - 1)) != 0) return -1;
  int k = 0;
  while ((1 << k) < x) ++k;
  return k;
}

// Items one CTA writes when a list is cut into slices: fewer would leave most of the
// launch to the steps every slice repeats.
constexpr int64_t kItemsPerSlice = 1024;
constexpr int kMaxSlices = 32;

cudaError_t launch_schedule(const Problem& p, const Workspace& ws, const SchedConfig& c,
                            cudaStream_t s) {
  ListSpec lq{false, c.q_rows, c.q_keys_step, log2_exact(c.q_rows), log2_exact(c.q_keys_step)};
  ListSpec lk{true, c.k_keys, c.k_rows_step, log2_exact(c.k_keys), log2_exact(c.k_rows_step)};
  if (lq.tile_shift < 0 || lq.step_shift < 0 || lk.tile_shift < 0 || lk.step_shift < 0)
    return cudaErrorInvalidValue;  // every kernel family's tiles and steps are powers of two
  cudaError_t e = kernel_setup((const void*)schedule_kernel, kThreads, sched_smem_bytes(kCacheB));
  if (e != cudaSuccess) return e;
  const bool in_smem = p.batch <= kCacheB;  // else the arrays live in the workspace, one CTA
  const size_t smem = sched_smem_bytes(in_smem ? (int)p.batch : 0);
  // both lists from two CTAs at once when each CTA can keep its own per-sequence arrays
  const int split = (c.build_q && c.build_k && in_smem) ? 1 : 0;
  // slices: from a bound on the larger list's items, H (rows / tile + B)
  int slices = 1;
  if (in_smem) {
    int64_t units = 0;
    if (c.build_q) units = std::max<int64_t>(units, p.total_q / c.q_rows + p.batch);
    if (c.build_k) units = std::max<int64_t>(units, p.total_k / c.k_keys + p.batch);
    const int64_t items = units * p.heads;
    slices = (int)std::min<int64_t>(kMaxSlices, std::max<int64_t>(1, items / kItemsPerSlice));
  }
  const int grid = (split ? 2 : 1) * slices;
  schedule_kernel<<<grid, kThreads, smem, s>>>(p, ws, lq, lk, c.build_q, c.build_k, c.self_attention, split,
                                               slices);
  return cudaGetLastError();
}

}  // namespace jfa
