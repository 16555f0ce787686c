// Internal declarations shared by the libjfa translation units (host and device).
// Nothing here is part of the public ABI (include/jfa.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "jfa.h"

namespace jfa {

constexpr int kActSoftmax = 0;
constexpr int kActSiluOverLen = 1;

// Masked scores are moved down by this amount (in the log2-scaled score
// domain) instead of being replaced by -inf: exp2 of a masked score then
// underflows to exactly 0 once the running row maximum comes from a valid
// key, no inf - inf can arise, and no -inf fill is needed on partial tiles
// (the "subtraction instead of -inf masking" of the Jagged Flash Attention
// bullet, Meta GEM MFU write-up, piletech.kr/articles/112134, details).
// The same shift drives SiLU(u - shift) to (-)0 for the non-softmax variant.
constexpr float kMaskShift = 1048576.0f;  // 2^20

// One unit of work produced by the jagged tile scheduler: (sequence b, head h,
// tile index inside the sequence, cost = number of inner steps the kernel will
// run for it) plus the sequence's first query / key rows and its query / key
// lengths, so that a kernel needs a single 32-byte load per item.
// Query-major lists hold q-tiles, key-major lists hold k-tiles.
struct __align__(16) WorkItem {
  int b, h, tile, cost;
  int q0, k0, lq, lk;
};

__device__ __forceinline__ WorkItem load_item(const WorkItem* list, int i) {
  const int4* p = reinterpret_cast<const int4*>(list + i);
  const int4 a = __ldg(p), c = __ldg(p + 1);
  WorkItem w;
  w.b = a.x; w.h = a.y; w.tile = a.z; w.cost = a.w;
  w.q0 = c.x; w.k0 = c.y; w.lq = c.z; w.lk = c.w;
  return w;
}

// Device workspace header; lives at offset 0 of the caller's workspace.
struct WsHeader {
  int status;    // jfa_status of the last call (device-detected errors only)
  int n_q;       // items in the query-major list
  int n_k;       // items in the key-major list
  int claim[3];  // next list item to take: forward, dK/dV, dQ (0 or -1, set by the
                 // scheduler; a kernel that takes items rewinds its counter to 0)
  int pad[58];
};
static_assert(sizeof(WsHeader) == 256, "workspace header");
enum : int { kClaimFwd = 0, kClaimDkdv = 1, kClaimDq = 2 };

// Everything a kernel needs to know about one request.
struct Problem {
  const int64_t* offs_q;
  const int64_t* offs_k;
  int64_t batch, total_q, total_k;
  int heads, dim_qk, dim_v;
  float scale;
  int causal;
  int act;
  // Rotary position embedding of q and k (BlockAttention), or nullptr: (cos, sin) of the
  // angle of position p and pair i at rope[p * (dim_qk/2) + i], for p < rope_npos.  Rows
  // are at the position of their index inside their sequence.
  const float2* rope;
  int rope_npos;
  // BlockAttention with two blocks per tile: a row attends only keys of its own
  // block_mask-row block, counted from its sequence's first row (a power of two that the
  // compute warpgroups' column spans divide; 0: whole sequences).
  int block_mask;
  // When set, the tensor-core dQ pass writes its rows in fp32 here instead of bf16 into
  // its dq argument (pooled attention's per-sequence query gradients, summed afterwards).
  float* dq_f32;
};

// Carve-up of the caller's workspace.
struct Workspace {
  WsHeader* hdr;
  int4* seq;            // [B] (q0, k0, lq, lk) per sequence (scheduler scratch, large batches)
  int* seq_ints;        // [4 (B+1)] per-sequence scheduler arrays (scratch, large batches)
  WorkItem* list_q;     // [max_items_q]
  WorkItem* list_k;     // [max_items_k]
  float* drow;          // [2 * T_q * H] backward row terms (layout chosen by the kernel family)
  int64_t max_items_q, max_items_k;
};

// Smallest tile any kernel uses; bounds the number of work items.
constexpr int kMinTile = 32;

size_t workspace_layout(int64_t batch, int64_t total_q, int64_t total_k, int heads, void* base,
                        Workspace* out);

// Scheduler: validates offsets, writes the status word and builds the lists
// requested (a q-list of tiles of q_rows rows whose inner loop steps over keys
// in blocks of q_keys_step, and/or a k-list of tiles of k_keys keys whose
// inner loop steps over rows in blocks of k_rows_step).
struct SchedConfig {
  int q_rows, q_keys_step;
  int k_keys, k_rows_step;
  int build_q, build_k;
  int self_attention;  // causal or GDPA self: Lq_b must equal Lk_b
};
cudaError_t launch_schedule(const Problem& p, const Workspace& ws, const SchedConfig& c,
                            cudaStream_t s);

// CUDA-core kernels (fp32 arithmetic; inputs fp32 or bf16).
extern const SchedConfig kSimtSched;
cudaError_t launch_simt_fwd(const Problem& p, int dtype, const void* q, const void* k,
                            const void* v, void* o, float* lse, const Workspace& ws,
                            cudaStream_t s);
cudaError_t launch_bwd_rowterm(const Problem& p, int dtype, const void* o, const void* dout,
                               const Workspace& ws, cudaStream_t s);
cudaError_t launch_simt_dkdv(const Problem& p, int dtype, const void* q, const void* k,
                             const void* v, const float* lse, const void* dout, void* dk,
                             void* dv, const Workspace& ws, cudaStream_t s);
cudaError_t launch_simt_dq(const Problem& p, int dtype, const void* q, const void* k,
                           const void* v, const float* lse, const void* dout, void* dq,
                           const Workspace& ws, cudaStream_t s);

// Pooled multi-head attention: broadcast of the m shared query rows into B blocks of
// m rows with offsets b*m, and the fixed-order sum of the B per-block query gradients.
cudaError_t launch_pooled_broadcast(int64_t batch, int32_t m, int64_t row_bytes, const void* q,
                                    void* q_rep, int64_t* offs_q, cudaStream_t s);
cudaError_t launch_pooled_reduce(int dtype, bool rep_f32, int64_t batch, int64_t per_seq_elems,
                                 const void* dq_rep, void* dq, cudaStream_t s);

// The rotary embedding's (cos, sin) table: npos positions by dim/2 pairs, angle
// p * base^(-2i/dim), computed in double precision.
cudaError_t launch_rope_table(float2* table, int npos, int dim, double base, cudaStream_t s);

// BlockAttention: the offsets of the fixed `block`-row blocks of every sequence, then empty
// sequences up to n_out (n_out + 1 entries); out[0] = -1 for offsets that are not valid.
cudaError_t launch_block_offsets(const int64_t* offs, int64_t batch, int64_t total, int block,
                                 int64_t* out, int64_t n_out, cudaStream_t s);

int num_sms();

// Identity of the CUDA context current on the calling host thread, or 0 when none is
// current (or the driver cannot say).  Per-context state the library caches (kernel
// attributes, the no-allocation scratch address, the side stream) is keyed on it, so
// that state set up under one context is never used under another: after
// cudaDeviceReset the primary context is a new one, and a driver-API context on the
// same device loads its own copy of the module.
unsigned long long current_context_id();

// Sets a kernel's dynamic shared-memory limit, and returns its resident CTAs per SM at
// (threads, smem), once per kernel and context; later calls answer from a cache.  These
// are not stream operations, so launches that follow stay capturable in a CUDA graph.
cudaError_t kernel_setup(const void* func, int threads, size_t smem, int* per_sm = nullptr);

}  // namespace jfa
