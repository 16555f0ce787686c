// C ABI of libjfa: argument validation, workspace carve-up, kernel dispatch,
// status reporting and optional per-kernel event timing.  See include/jfa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "tc.h"

namespace jfa {

int num_sms() {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The driver's context queries, looked up once.
namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
template <class F>
F driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return (F)ptr;
  return nullptr;
}
}  // namespace

unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // never 0 for a real context
}

cudaError_t kernel_setup(const void* func, int threads, size_t smem, int* per_sm) {
  // Kernel attributes belong to the context's copy of the module: the cache is keyed on
  // the context, so a reset device (a new primary context) or another context on the
  // same device sets them up again.
  struct Entry { unsigned long long ctx; const void* func; int threads; size_t smem; int per_sm; };
  static std::mutex mu;
  static std::vector<Entry> cache;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx != 0)
    for (const Entry& x : cache)
      if (x.ctx == ctx && x.func == func && x.threads == threads && x.smem == smem) {
        if (per_sm) *per_sm = x.per_sm;
        return cudaSuccess;
      }
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem);
  if (e != cudaSuccess) return e;
  const unsigned long long now = current_context_id();  // set once the runtime made one current
  if (now != 0) cache.push_back({now, func, threads, smem, n});
  if (per_sm) *per_sm = n;
  return cudaSuccess;
}

size_t workspace_layout(int64_t batch, int64_t total_q, int64_t total_k, int heads, void* base,
                        Workspace* out) {
  char* b = (char*)base;
  size_t off = 0;
  Workspace w{};
  w.hdr = (WsHeader*)(b + off);
  off = align_up(off + sizeof(WsHeader), 256);
  w.seq = (int4*)(b + off);
  off = align_up(off + sizeof(int4) * (size_t)batch, 256);
  w.seq_ints = (int*)(b + off);
  off = align_up(off + 4 * sizeof(int) * (size_t)(batch + 1), 256);
  w.max_items_q = (int64_t)heads * (total_q / kMinTile + batch + 1);
  w.list_q = (WorkItem*)(b + off);
  off = align_up(off + sizeof(WorkItem) * (size_t)w.max_items_q, 256);
  w.max_items_k = (int64_t)heads * (total_k / kMinTile + batch + 1);
  w.list_k = (WorkItem*)(b + off);
  off = align_up(off + sizeof(WorkItem) * (size_t)w.max_items_k, 256);
  w.drow = (float*)(b + off);
  off = align_up(off + 2 * sizeof(float) * (size_t)total_q * (size_t)heads, 256);
  if (out) *out = w;
  return off;
}

// ---------------------------------------------------------------------------
// Kernel timing (benchmarks only)
// ---------------------------------------------------------------------------
namespace {
struct Prof {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  struct Pending { int kind; cudaEvent_t a, b; };
  std::vector<Pending> pending;
  int64_t launches[JFA_KERNEL_KINDS] = {0};
  double ms[JFA_KERNEL_KINDS] = {0};
};
Prof& prof() {
  static Prof p;
  return p;
}
cudaEvent_t take_event() {
  Prof& P = prof();
  if (!P.pool.empty()) {
    cudaEvent_t e = P.pool.back();
    P.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
jfa_status drain() {
  Prof& P = prof();
  jfa_status st = JFA_OK;
  for (auto& x : P.pending) {
    float t = 0.f;
    if (cudaEventSynchronize(x.b) != cudaSuccess || cudaEventElapsedTime(&t, x.a, x.b) != cudaSuccess)
      st = JFA_ERR_CUDA;
    P.launches[x.kind] += 1;
    P.ms[x.kind] += t;
    P.pool.push_back(x.a);
    P.pool.push_back(x.b);
  }
  P.pending.clear();
  return st;
}

// Records events around one launch when profiling is on.
struct Timed {
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  Timed(int k, cudaStream_t st) : kind(k), s(st) {
    if (!prof().on) return;
    if (prof().pending.size() > 65536) drain();
    a = take_event();
    b = take_event();
    if (!a || !b) {  // no timing for this launch; keep whichever event was made
      if (a) prof().pool.push_back(a);
      if (b) prof().pool.push_back(b);
      a = b = nullptr;
      return;
    }
    cudaEventRecord(a, s);
  }
  ~Timed() {
    if (!a || !b) return;
    cudaEventRecord(b, s);
    prof().pending.push_back({kind, a, b});
  }
};

inline jfa_status cu(cudaError_t e) { return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA; }

// A second stream per device and host thread, with a fork and a join event, for
// independent work that may overlap the caller's stream (the backward row terms
// run beside the scheduler).  Created on first use and kept for the thread's life;
// nullptr when it cannot be created (the work then runs on the caller's stream).
struct SideStream {
  unsigned long long ctx = 0;  // the context the stream and events belong to
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream() {
  constexpr int kMaxDevices = 64;
  thread_local SideStream sides[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  if (ctx == 0) return nullptr;
  SideStream& sd = sides[dev];
  if (!sd.s || sd.ctx != ctx) {  // first use, or a new context (the old handles died with it)
    cudaStream_t st = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
      if (a) cudaEventDestroy(a);
      cudaStreamDestroy(st);
      return nullptr;
    }
    sd.ctx = ctx;
    sd.s = st;
    sd.fork = a;
    sd.join = b;
  }
  return &sd;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

enum class Kind { Self, Cross, Gdpa };

jfa_status check_params(const jfa_params* p, Kind kind) {
  if (!p) return JFA_ERR_INVALID_ARG;
  if (p->batch < 0 || p->total_q < 0 || p->total_k < 0 || p->heads < 1) return JFA_ERR_INVALID_ARG;
  if (p->dim_qk < 1 || p->dim_v < 1) return JFA_ERR_INVALID_ARG;
  if (p->dtype != JFA_F32 && p->dtype != JFA_BF16) return JFA_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || p->scale == INFINITY) return JFA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return JFA_ERR_INVALID_ARG;
  if ((p->flags & ~JFA_PLANNED) != 0) return JFA_ERR_INVALID_ARG;
  if (p->batch == 0 && (p->total_q != 0 || p->total_k != 0)) return JFA_ERR_INVALID_ARG;
  if (p->total_q > INT32_MAX || p->total_k > INT32_MAX) return JFA_ERR_UNSUPPORTED;
  // the work lists' item counts (and item indices) are 32-bit
  const int64_t rows = p->total_q > p->total_k ? p->total_q : p->total_k;
  if ((int64_t)p->heads * (rows / kMinTile + p->batch + 1) > INT32_MAX) return JFA_ERR_UNSUPPORTED;
  if (kind == Kind::Self && p->total_k != p->total_q) return JFA_ERR_INVALID_ARG;
  if (kind == Kind::Cross && p->causal) return JFA_ERR_UNSUPPORTED;
  if (kind == Kind::Gdpa && p->causal && p->total_k != p->total_q) return JFA_ERR_INVALID_ARG;
  if (jfa_path_for(p) < 0) return JFA_ERR_UNSUPPORTED;
  return JFA_OK;
}

jfa_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

jfa_status prepare(const jfa_params* p, void* ws, size_t ws_bytes, Workspace* w) {
  if (!ws || ((uintptr_t)ws & 255u) != 0) return JFA_ERR_WORKSPACE;
  size_t need = workspace_layout(p->batch, p->total_q, p->total_k, p->heads, ws, w);
  if (ws_bytes < need) return JFA_ERR_WORKSPACE;
  return JFA_OK;
}

Problem make_problem(const jfa_params* p, const int64_t* oq, const int64_t* ok, int act) {
  Problem r;
  r.offs_q = oq;
  r.offs_k = ok;
  r.batch = p->batch;
  r.total_q = p->total_q;
  r.total_k = p->total_k;
  r.heads = p->heads;
  r.dim_qk = p->dim_qk;
  r.dim_v = p->dim_v;
  r.scale = p->scale;
  r.causal = p->causal;
  r.act = act;
  r.rope = nullptr;
  r.rope_npos = 0;
  r.block_mask = 0;
  r.dq_f32 = nullptr;
  return r;
}

// An empty batch still resets the status word so jfa_status_check reports it.
jfa_status empty_call(const Workspace& w, cudaStream_t s) {
  return cu(cudaMemsetAsync(w.hdr, 0, sizeof(WsHeader), s));
}

jfa_status run_fwd(const jfa_params* p, Kind kind, int act, const void* q, const void* k,
                   const void* v, const int64_t* oq, const int64_t* ok, void* o, float* lse,
                   void* ws, size_t ws_bytes, cudaStream_t s, const float2* rope = nullptr,
                   int rope_npos = 0, int block_mask = 0) {
  jfa_status st = check_params(p, kind);
  if (st != JFA_OK) return st;
  if ((st = check_ptrs({oq, ok})) != JFA_OK) return st;
  if (p->batch > 0 && p->total_q > 0) {
    if ((st = check_ptrs({q, o})) != JFA_OK) return st;
    if (act == kActSoftmax && (st = check_ptrs({lse})) != JFA_OK) return st;
  }
  if (p->total_k > 0 && (st = check_ptrs({k, v})) != JFA_OK) return st;
  Workspace w;
  if ((st = prepare(p, ws, ws_bytes, &w)) != JFA_OK) return st;
  if (p->batch == 0) return empty_call(w, s);
  Problem pr = make_problem(p, oq, ok, act);
  pr.rope = rope;
  pr.rope_npos = rope_npos;
  pr.block_mask = block_mask;
  const int path = jfa_path_for(p);
  if (!(p->flags & JFA_PLANNED)) {
    SchedConfig sc = path == 1 ? tc_fwd_sched(pr) : kSimtSched;
    sc.build_q = 1;
    sc.build_k = 0;
    sc.self_attention = (kind == Kind::Self) || p->causal;
    Timed t(JFA_KERNEL_SCHEDULE, s);
    if ((st = cu(launch_schedule(pr, w, sc, s))) != JFA_OK) return st;
  }
  Timed t(JFA_KERNEL_FWD, s);
  if (path == 1) return cu(launch_tc_fwd(pr, q, k, v, o, lse, w, s));
  return cu(launch_simt_fwd(pr, p->dtype, q, k, v, o, lse, w, s));
}

jfa_status run_bwd(const jfa_params* p, Kind kind, int act, const void* q, const void* k,
                   const void* v, const void* o, const float* lse, const void* dout,
                   const int64_t* oq, const int64_t* ok, void* dq, void* dk, void* dv, void* ws,
                   size_t ws_bytes, cudaStream_t s, const float2* rope = nullptr,
                   int rope_npos = 0, int block_mask = 0, float* dq_f32 = nullptr) {
  jfa_status st = check_params(p, kind);
  if (st != JFA_OK) return st;
  if ((st = check_ptrs({oq, ok})) != JFA_OK) return st;
  if (p->batch > 0 && p->total_q > 0) {
    if ((st = check_ptrs({q, dout, dq})) != JFA_OK) return st;
    if (act == kActSoftmax && (st = check_ptrs({o, lse})) != JFA_OK) return st;
  }
  if (p->total_k > 0 && (st = check_ptrs({k, v, dk, dv})) != JFA_OK) return st;
  Workspace w;
  if ((st = prepare(p, ws, ws_bytes, &w)) != JFA_OK) return st;
  if (p->batch == 0) return empty_call(w, s);
  Problem pr = make_problem(p, oq, ok, act);
  pr.rope = rope;
  pr.rope_npos = rope_npos;
  pr.block_mask = block_mask;
  pr.dq_f32 = jfa_path_for(p) == 1 ? dq_f32 : nullptr;
  const int path = jfa_path_for(p);
  const bool planned = (p->flags & JFA_PLANNED) != 0;
  // The row terms (softmax only) depend on o, dout and lse alone: they run on a side
  // stream while the scheduler builds the lists, and the caller's stream waits for
  // them before the dK/dV pass.  A planned call builds no lists and runs them in line.
  SideStream* sd = act == kActSoftmax && !planned ? side_stream() : nullptr;
  if (sd && (cudaEventRecord(sd->fork, s) != cudaSuccess ||
             cudaStreamWaitEvent(sd->s, sd->fork, 0) != cudaSuccess))
    return JFA_ERR_CUDA;
  if (!planned) {
    SchedConfig sc = path == 1 ? tc_bwd_sched(pr) : kSimtSched;
    sc.build_q = 1;
    sc.build_k = 1;
    sc.self_attention = (kind == Kind::Self) || p->causal;
    Timed t(JFA_KERNEL_SCHEDULE, s);
    if ((st = cu(launch_schedule(pr, w, sc, s))) != JFA_OK) return st;
  }
  if (act == kActSoftmax) {
    cudaStream_t rs = sd ? sd->s : s;
    {
      Timed t(JFA_KERNEL_BWD_D, rs);
      st = path == 1 ? cu(launch_tc_rowstat(pr, o, dout, lse, w, rs))
                     : cu(launch_bwd_rowterm(pr, p->dtype, o, dout, w, rs));
    }
    if (sd && (cudaEventRecord(sd->join, rs) != cudaSuccess ||
               cudaStreamWaitEvent(s, sd->join, 0) != cudaSuccess))
      return JFA_ERR_CUDA;
    if (st != JFA_OK) return st;
  }
  {
    Timed t(JFA_KERNEL_BWD_DKDV, s);
    if (path == 1)
      st = cu(launch_tc_dkdv(pr, q, k, v, lse, dout, dk, dv, w, s));
    else
      st = cu(launch_simt_dkdv(pr, p->dtype, q, k, v, lse, dout, dk, dv, w, s));
    if (st != JFA_OK) return st;
  }
  Timed t(JFA_KERNEL_BWD_DQ, s);
  if (path == 1) return cu(launch_tc_dq(pr, q, k, v, lse, dout, dq, w, s));
  return cu(launch_simt_dq(pr, p->dtype, q, k, v, lse, dout, dq, w, s));
}

// Both lists, for the forward and backward calls of these params: the backward's q-list
// is the forward's (same tiles and steps on each path), so one build serves the three
// passes.  self_attention: Lq_b must equal Lk_b.
jfa_status run_plan(const jfa_params* p, const int64_t* oq, const int64_t* ok, bool self_attention,
                    void* ws, size_t ws_bytes, cudaStream_t s) {
  Workspace w;
  jfa_status st = prepare(p, ws, ws_bytes, &w);
  if (st != JFA_OK) return st;
  if (p->batch == 0) return empty_call(w, s);
  Problem pr = make_problem(p, oq, ok, kActSoftmax);
  const int path = jfa_path_for(p);
  SchedConfig sc = path == 1 ? tc_bwd_sched(pr) : kSimtSched;
  if (path == 1) {
    const SchedConfig f = tc_fwd_sched(pr);
    if (f.q_rows != sc.q_rows || f.q_keys_step != sc.q_keys_step) return JFA_ERR_UNSUPPORTED;
  }
  sc.build_q = 1;
  sc.build_k = 1;
  sc.self_attention = self_attention || p->causal;
  Timed t(JFA_KERNEL_SCHEDULE, s);
  return cu(launch_schedule(pr, w, sc, s));
}

// Pooled multi-head attention: the cross-attention workspace, then the query-row offsets
// b*m, the broadcast query rows and their per-sequence gradients.
struct PooledWs {
  size_t base, offs, q_rep, dq_rep, total;
};
PooledWs pooled_layout(const jfa_params* p, int32_t m) {
  PooledWs r;
  const size_t e = p->dtype == JFA_BF16 ? 2 : 4;
  const size_t elems = (size_t)p->batch * (size_t)m * (size_t)p->heads * (size_t)p->dim_qk;
  r.base = workspace_layout(p->batch, p->total_q, p->total_k, p->heads, nullptr, nullptr);
  r.offs = align_up(r.base, 256);
  r.q_rep = align_up(r.offs + 8 * (size_t)(p->batch + 1), 256);
  // the per-sequence query gradients stay in fp32 until they are summed
  r.dq_rep = align_up(r.q_rep + elems * e, 256);
  r.total = align_up(r.dq_rep + elems * 4, 256);
  return r;
}

jfa_status check_pooled(const jfa_params* p, int32_t m, void* ws, size_t ws_bytes, PooledWs* lay) {
  if (!p || m < 1) return JFA_ERR_INVALID_ARG;
  if (p->total_q != p->batch * (int64_t)m) return JFA_ERR_INVALID_ARG;
  if (p->causal) return JFA_ERR_UNSUPPORTED;
  const size_t e = p->dtype == JFA_BF16 ? 2 : 4;
  if (((size_t)p->heads * (size_t)p->dim_qk * e) % 4 != 0) return JFA_ERR_UNSUPPORTED;
  jfa_status st = check_params(p, Kind::Cross);
  if (st != JFA_OK) return st;
  if (!ws || ((uintptr_t)ws & 255u) != 0) return JFA_ERR_WORKSPACE;
  *lay = pooled_layout(p, m);
  if (ws_bytes < lay->total) return JFA_ERR_WORKSPACE;
  return JFA_OK;
}

// BlockAttention: the self-attention workspace for B + ceil(T/64) block sequences, then the
// block offsets.
constexpr int kBlock = 64;
// The tensor-core path runs two blocks per 128-row tile: the offsets are cut into pieces
// of two blocks, and the kernels mask each row to its own block's keys (Problem's
// block_mask), which halves the tiles and items against one block per tile.  The fp32
// path keeps one block per sequence.
constexpr int kPiece = 2 * kBlock;
int piece_rows(const jfa_params* p) { return jfa_path_for(p) == 1 ? kPiece : kBlock; }
int64_t piece_count(const jfa_params* p, int rows) { return p->batch + (p->total_q + rows - 1) / rows; }
// the workspace is laid out for the larger count, so that its size does not depend on the path
int64_t block_count(const jfa_params* p) { return piece_count(p, kBlock); }
constexpr double kRopeBase = 10000.0;  // the rotary embedding's frequency base
struct BlockWs {
  size_t offs, rope, total;
};
BlockWs block_layout(const jfa_params* p) {
  BlockWs r;
  const int64_t nb = block_count(p);
  r.offs = align_up(workspace_layout(nb, p->total_q, p->total_k, p->heads, nullptr, nullptr), 256);
  // then the rotary embedding's (cos, sin) table: the positions of a piece by dim_qk/2 pairs
  r.rope = align_up(r.offs + 8 * (size_t)(nb + 1), 256);
  r.total = align_up(r.rope + sizeof(float2) * kPiece * (size_t)(p->dim_qk > 0 ? p->dim_qk / 2 : 0), 256);
  return r;
}

// params of the block sequences, after the checks a block call makes before any launch
jfa_status check_block(const jfa_params* p, void* ws, size_t ws_bytes, jfa_params* pb, BlockWs* lay) {
  jfa_status st = check_params(p, Kind::Self);
  if (st != JFA_OK) return st;
  if (!ws || ((uintptr_t)ws & 255u) != 0) return JFA_ERR_WORKSPACE;
  *lay = block_layout(p);
  if (ws_bytes < lay->total) return JFA_ERR_WORKSPACE;
  *pb = *p;
  pb->batch = piece_count(p, piece_rows(p));
  return JFA_OK;
}

}  // namespace
}  // namespace jfa

namespace jfa {
namespace {
// The rotary embedding needs the tensor-core path with Dqk = Dv (its kernels rotate the
// Q and K tiles in shared memory).
jfa_status check_rope(const jfa_params* p) {
  if (jfa_path_for(p) != 1 || p->dim_qk != p->dim_v) return JFA_ERR_UNSUPPORTED;
  return JFA_OK;
}

jfa_status block_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                     const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                     cudaStream_t s, bool rope) {
  jfa_params pb;
  BlockWs lay;
  jfa_status st = check_block(p, ws, ws_bytes, &pb, &lay);
  if (st != JFA_OK) return st;
  if (rope && (st = check_rope(p)) != JFA_OK) return st;
  if ((st = check_ptrs({offs})) != JFA_OK) return st;
  if (p->total_q > 0 && (st = check_ptrs({q, k, v, o, lse})) != JFA_OK) return st;
  int64_t* boffs = (int64_t*)((char*)ws + lay.offs);
  float2* table = (float2*)((char*)ws + lay.rope);
  const int rows = piece_rows(p);
  // a planned call finds the block offsets and the rotary table in the workspace
  if (p->batch > 0 && !(p->flags & JFA_PLANNED)) {
    Timed t(JFA_KERNEL_AUX, s);
    if ((st = cu(launch_block_offsets(offs, p->batch, p->total_q, rows, boffs, pb.batch, s))) != JFA_OK)
      return st;
    if (rope && (st = cu(launch_rope_table(table, rows, p->dim_qk, kRopeBase, s))) != JFA_OK) return st;
  }
  return run_fwd(&pb, Kind::Self, kActSoftmax, q, k, v, boffs, boffs, o, lse, ws, ws_bytes, s,
                 rope ? table : nullptr, rope ? rows : 0, rows == kPiece ? kBlock : 0);
}

jfa_status block_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                     const void* o, const float* lse, const void* dout, const int64_t* offs,
                     void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, cudaStream_t s,
                     bool rope) {
  jfa_params pb;
  BlockWs lay;
  jfa_status st = check_block(p, ws, ws_bytes, &pb, &lay);
  if (st != JFA_OK) return st;
  if (rope && (st = check_rope(p)) != JFA_OK) return st;
  if ((st = check_ptrs({offs})) != JFA_OK) return st;
  if (p->total_q > 0 && (st = check_ptrs({q, k, v, o, lse, dout, dq, dk, dv})) != JFA_OK) return st;
  int64_t* boffs = (int64_t*)((char*)ws + lay.offs);
  float2* table = (float2*)((char*)ws + lay.rope);
  const int rows = piece_rows(p);
  // a planned call finds the block offsets and the rotary table in the workspace
  if (p->batch > 0 && !(p->flags & JFA_PLANNED)) {
    Timed t(JFA_KERNEL_AUX, s);
    if ((st = cu(launch_block_offsets(offs, p->batch, p->total_q, rows, boffs, pb.batch, s))) != JFA_OK)
      return st;
    if (rope && (st = cu(launch_rope_table(table, rows, p->dim_qk, kRopeBase, s))) != JFA_OK) return st;
  }
  return run_bwd(&pb, Kind::Self, kActSoftmax, q, k, v, o, lse, dout, boffs, boffs, dq, dk, dv, ws,
                 ws_bytes, s, rope ? table : nullptr, rope ? rows : 0, rows == kPiece ? kBlock : 0);
}

// The block offsets, the rotary table (where the rotary calls are supported) and the
// lists of the block sequences.
jfa_status block_plan(const jfa_params* p, const int64_t* offs, void* ws, size_t ws_bytes, cudaStream_t s) {
  jfa_params pb;
  BlockWs lay;
  jfa_status st = check_block(p, ws, ws_bytes, &pb, &lay);
  if (st != JFA_OK) return st;
  if ((st = check_ptrs({offs})) != JFA_OK) return st;
  int64_t* boffs = (int64_t*)((char*)ws + lay.offs);
  float2* table = (float2*)((char*)ws + lay.rope);
  const int rows = piece_rows(p);
  if (p->batch > 0) {
    Timed t(JFA_KERNEL_AUX, s);
    if ((st = cu(launch_block_offsets(offs, p->batch, p->total_q, rows, boffs, pb.batch, s))) != JFA_OK)
      return st;
    if (check_rope(p) == JFA_OK && (st = cu(launch_rope_table(table, rows, p->dim_qk, kRopeBase, s))) != JFA_OK)
      return st;
  }
  return run_plan(&pb, boffs, boffs, true, ws, ws_bytes, s);
}
}  // namespace
}  // namespace jfa

using namespace jfa;

extern "C" {

size_t jfa_workspace_size(const jfa_params* p) {
  if (!p || p->batch < 0 || p->total_q < 0 || p->total_k < 0 || p->heads < 1) return 0;
  return workspace_layout(p->batch, p->total_q, p->total_k, p->heads, nullptr, nullptr);
}

int jfa_path_for(const jfa_params* p) {
  if (!p) return -1;
  if (p->dim_qk < 1 || p->dim_v < 1 || p->dim_qk > 128 || p->dim_v > 128) return -1;
  if (p->dtype == JFA_BF16 && tc_supports(p->dim_qk, p->dim_v)) return 1;
  if (p->dtype == JFA_F32 || p->dtype == JFA_BF16) return 0;
  return -1;
}

jfa_status jfa_plan(const jfa_params* p, const int64_t* offs_q, const int64_t* offs_k, void* ws,
                    size_t ws_bytes, jfa_stream_t stream) {
  jfa_status st = check_params(p, Kind::Gdpa);
  if (st != JFA_OK) return st;
  if ((st = check_ptrs({offs_q, offs_k})) != JFA_OK) return st;
  return run_plan(p, offs_q, offs_k, offs_q == offs_k, ws, ws_bytes, (cudaStream_t)stream);
}

jfa_status jfa_block_plan(const jfa_params* p, const int64_t* offs, void* ws, size_t ws_bytes,
                          jfa_stream_t stream) {
  return block_plan(p, offs, ws, ws_bytes, (cudaStream_t)stream);
}

jfa_status jfa_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                   const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                   jfa_stream_t stream) {
  return run_fwd(p, Kind::Self, kActSoftmax, q, k, v, offs, offs, o, lse, ws, ws_bytes,
                 (cudaStream_t)stream);
}

jfa_status jfa_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                   const void* o, const float* lse, const void* dout, const int64_t* offs,
                   void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                   jfa_stream_t stream) {
  return run_bwd(p, Kind::Self, kActSoftmax, q, k, v, o, lse, dout, offs, offs, dq, dk, dv, ws,
                 ws_bytes, (cudaStream_t)stream);
}

jfa_status jfa_cross_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const int64_t* offs_q, const int64_t* offs_k, void* o, float* lse,
                         void* ws, size_t ws_bytes, jfa_stream_t stream) {
  return run_fwd(p, Kind::Cross, kActSoftmax, q, k, v, offs_q, offs_k, o, lse, ws, ws_bytes,
                 (cudaStream_t)stream);
}

jfa_status jfa_cross_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         const int64_t* offs_q, const int64_t* offs_k, void* dq, void* dk,
                         void* dv, void* ws, size_t ws_bytes, jfa_stream_t stream) {
  return run_bwd(p, Kind::Cross, kActSoftmax, q, k, v, o, lse, dout, offs_q, offs_k, dq, dk, dv,
                 ws, ws_bytes, (cudaStream_t)stream);
}

jfa_status jfa_gdpa_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                        const int64_t* offs_q, const int64_t* offs_k, void* o, void* ws,
                        size_t ws_bytes, jfa_stream_t stream) {
  return run_fwd(p, Kind::Gdpa, kActSiluOverLen, q, k, v, offs_q, offs_k, o, nullptr, ws,
                 ws_bytes, (cudaStream_t)stream);
}

jfa_status jfa_gdpa_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                        const void* dout, const int64_t* offs_q, const int64_t* offs_k,
                        void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        jfa_stream_t stream) {
  return run_bwd(p, Kind::Gdpa, kActSiluOverLen, q, k, v, nullptr, nullptr, dout, offs_q, offs_k,
                 dq, dk, dv, ws, ws_bytes, (cudaStream_t)stream);
}

size_t jfa_pooled_workspace_size(const jfa_params* p, int32_t m) {
  if (!p || m < 1 || p->batch < 0 || p->total_k < 0 || p->heads < 1 || p->dim_qk < 1) return 0;
  if (p->total_q != p->batch * (int64_t)m) return 0;
  return pooled_layout(p, m).total;
}

jfa_status jfa_pooled_fwd(const jfa_params* p, int32_t m, const void* q, const void* k,
                          const void* v, const int64_t* offs_k, void* o, float* lse, void* ws,
                          size_t ws_bytes, jfa_stream_t stream) {
  PooledWs lay;
  jfa_status st = check_pooled(p, m, ws, ws_bytes, &lay);
  if (st != JFA_OK) return st;
  if (p->flags & JFA_PLANNED) return JFA_ERR_UNSUPPORTED;
  // every argument is checked before the broadcast kernel is launched
  if ((st = check_ptrs({offs_k})) != JFA_OK) return st;
  if (p->batch > 0 && (st = check_ptrs({q, o, lse})) != JFA_OK) return st;
  if (p->total_k > 0 && (st = check_ptrs({k, v})) != JFA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  int64_t* offs_q = (int64_t*)(base + lay.offs);
  void* q_rep = base + lay.q_rep;
  if (p->batch > 0) {
    const size_t e = p->dtype == JFA_BF16 ? 2 : 4;
    Timed t(JFA_KERNEL_AUX, s);
    if ((st = cu(launch_pooled_broadcast(p->batch, m, (int64_t)p->heads * p->dim_qk * (int64_t)e, q,
                                         q_rep, offs_q, s))) != JFA_OK)
      return st;
  }
  return run_fwd(p, Kind::Cross, kActSoftmax, q_rep, k, v, offs_q, offs_k, o, lse, ws, ws_bytes, s);
}

jfa_status jfa_pooled_bwd(const jfa_params* p, int32_t m, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          const int64_t* offs_k, void* dq, void* dk, void* dv, void* ws,
                          size_t ws_bytes, jfa_stream_t stream) {
  PooledWs lay;
  jfa_status st = check_pooled(p, m, ws, ws_bytes, &lay);
  if (st != JFA_OK) return st;
  if (p->flags & JFA_PLANNED) return JFA_ERR_UNSUPPORTED;
  // every argument is checked before the broadcast kernel is launched
  if ((st = check_ptrs({offs_k})) != JFA_OK) return st;
  if (p->batch > 0 && (st = check_ptrs({q, dq, o, lse, dout})) != JFA_OK) return st;
  if (p->total_k > 0 && (st = check_ptrs({k, v, dk, dv})) != JFA_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  char* base = (char*)ws;
  int64_t* offs_q = (int64_t*)(base + lay.offs);
  void* q_rep = base + lay.q_rep;
  void* dq_rep = base + lay.dq_rep;
  const size_t e = p->dtype == JFA_BF16 ? 2 : 4;
  if (p->batch > 0) {
    Timed t(JFA_KERNEL_AUX, s);
    if ((st = cu(launch_pooled_broadcast(p->batch, m, (int64_t)p->heads * p->dim_qk * (int64_t)e, q,
                                         q_rep, offs_q, s))) != JFA_OK)
      return st;
  }
  // the tensor-core dQ pass leaves the per-sequence gradients in fp32 (no bf16 rounding
  // before the sum); the fp32 path computes in fp32 anyway
  const bool rep_f32 = p->dtype == JFA_BF16 && jfa_path_for(p) == 1;
  st = run_bwd(p, Kind::Cross, kActSoftmax, q_rep, k, v, o, lse, dout, offs_q, offs_k, dq_rep, dk,
               dv, ws, ws_bytes, s, nullptr, 0, 0, rep_f32 ? (float*)dq_rep : nullptr);
  if (st != JFA_OK || p->batch == 0) return st;
  Timed t(JFA_KERNEL_AUX, s);
  return cu(launch_pooled_reduce(p->dtype, rep_f32, p->batch, (int64_t)m * p->heads * p->dim_qk, dq_rep, dq,
                                 s));
}

size_t jfa_block_workspace_size(const jfa_params* p) {
  if (!p || p->batch < 0 || p->total_q < 0 || p->total_k < 0 || p->heads < 1) return 0;
  return block_layout(p).total;
}

jfa_status jfa_block_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                         jfa_stream_t stream) {
  return block_fwd(p, q, k, v, offs, o, lse, ws, ws_bytes, (cudaStream_t)stream, false);
}

jfa_status jfa_block_rope_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                              const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                              jfa_stream_t stream) {
  return block_fwd(p, q, k, v, offs, o, lse, ws, ws_bytes, (cudaStream_t)stream, true);
}

jfa_status jfa_block_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, const int64_t* offs,
                         void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                         jfa_stream_t stream) {
  return block_bwd(p, q, k, v, o, lse, dout, offs, dq, dk, dv, ws, ws_bytes, (cudaStream_t)stream, false);
}

jfa_status jfa_block_rope_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                              const void* o, const float* lse, const void* dout, const int64_t* offs,
                              void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                              jfa_stream_t stream) {
  return block_bwd(p, q, k, v, o, lse, dout, offs, dq, dk, dv, ws, ws_bytes, (cudaStream_t)stream, true);
}

jfa_status jfa_status_check(const void* ws, jfa_stream_t stream) {
  if (!ws || ((uintptr_t)ws & 255u) != 0) return JFA_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return JFA_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
  if (st < 0 || st > JFA_ERR_CUDA) return JFA_ERR_CUDA;
  return (jfa_status)st;
}

const char* jfa_status_string(jfa_status s) {
  switch (s) {
    case JFA_OK: return "ok";
    case JFA_ERR_INVALID_ARG: return "invalid argument";
    case JFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case JFA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case JFA_ERR_BAD_OFFSETS: return "offsets are not a valid jagged layout";
    case JFA_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    case JFA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

jfa_status jfa_test_hold(int on) { return cu(tc_set_test_hold(on)); }

jfa_status jfa_profile_enable(int on) {
  prof().on = on != 0;
  return JFA_OK;
}

jfa_status jfa_profile_reset(void) {
  jfa_status st = drain();
  for (int i = 0; i < JFA_KERNEL_KINDS; ++i) {
    prof().launches[i] = 0;
    prof().ms[i] = 0;
  }
  return st;
}

jfa_status jfa_profile_read(int kind, int64_t* launches, double* total_ms) {
  if (kind < 0 || kind >= JFA_KERNEL_KINDS || !launches || !total_ms) return JFA_ERR_INVALID_ARG;
  jfa_status st = drain();
  *launches = prof().launches[kind];
  *total_ms = prof().ms[kind];
  return st;
}

}  // extern "C"
