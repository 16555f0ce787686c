/*
 * jfa.h -- C ABI of libjfa, Jagged Flash Attention for one NVIDIA GB300 (sm_103a).
 *
 * Source of the method.  Meta GEM MFU co-design write-up
 * (piletech.kr/articles/112134), "상세 정리" (details) section:
 *   - jagged-input bullet: per-request sequences have different lengths, and
 *     padding them wastes up to half of the attention compute; the attention
 *     patterns are self, cross, pooled multi-head and asymmetric QKV;
 *   - Jagged Flash Attention bullet: attention that works directly on the
 *     variable-length tensors, masks by subtraction instead of -inf fill, and
 *     parallelises the backward pass without atomic operations;
 *   - Generalized Dot-Product Attention bullet: the same pipeline for
 *     non-softmax activations, with software tile scheduling over jagged
 *     tensors.
 * The pages give no formulas; the ones below are the plain definitions.
 *
 * Jagged tensors.  B sequences are concatenated without padding.  Sequence b
 * owns query rows offs_q[b] .. offs_q[b+1]-1 and key/value rows
 * offs_k[b] .. offs_k[b+1]-1.  Offsets are int64 [B+1] in DEVICE memory,
 * offs[0] == 0, non-decreasing, offs[B] == total rows.
 *
 * Layouts (row-major, contiguous, every pointer 16-byte aligned):
 *   Q  [T_q, H, Dqk]   K [T_k, H, Dqk]   V [T_k, H, Dv]
 *   O  [T_q, H, Dv]    dO [T_q, H, Dv]   lse [T_q, H] fp32 (natural log)
 *   dQ/dK/dV have the shapes of Q/K/V.  Values are fp32 or bf16 (params.dtype),
 *   lse is always fp32.
 *
 * Math, per sequence b and head h (i < Lq_b query rows, j < Lk_b key rows):
 *   s_ij = scale * <q_i, k_j>; valid pairs: j < Lk_b, and j <= i when causal.
 *   softmax:  P_ij = exp(s_ij - lse_i) over the valid j, o_i = sum_j P_ij v_j,
 *             lse_i = log sum_{valid j} exp(s_ij).  A row with no valid key
 *             (cross-attention with Lk_b == 0) gets o_i = 0, lse_i = -inf.
 *   SiLU/L:   P_ij = SiLU(s_ij) / Lq_b over the valid j, o_i = sum_j P_ij v_j.
 *   Backward: the analytic gradients of a loss whose gradient w.r.t. O is dO.
 *
 * Ownership and threading.  The caller owns every buffer.  The library never
 * allocates device memory on these paths and keeps no per-call state; its
 * only scratch is the caller's workspace (size from jfa_workspace_size).
 * One workspace must not be used by two calls that may run concurrently.
 * The one exception is jfa_fwd_noalloc below, whose scratch is a fixed array
 * inside the library shared by all of its calls.
 *
 * Asynchrony and errors.  Every compute call only enqueues work on `stream`
 * (NULL = the legacy default stream) and returns.  Argument errors are
 * detected on the host before anything is launched, and returned.  Errors
 * found on the device are written to a status word inside the workspace:
 * offsets that are not a valid jagged layout (the call then computes nothing
 * and leaves its outputs untouched), or a bounded wait inside a kernel that
 * gave up (the outputs are then incomplete).  jfa_status_check()
 * synchronises the stream and returns that word.  The library never aborts,
 * traps or prints.
 */
#ifndef JFA_H_
#define JFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st* jfa_stream_t;

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  JFA_ERR_UNSUPPORTED = 2, /* valid request the library does not implement */
  JFA_ERR_WORKSPACE = 3,   /* workspace missing, misaligned or too small */
  JFA_ERR_BAD_OFFSETS = 4, /* (device) offsets are not a jagged layout of the given totals */
  JFA_ERR_TIMEOUT = 5,     /* (device) a bounded wait inside a kernel gave up */
  JFA_ERR_CUDA = 6         /* a CUDA runtime or driver call failed */
} jfa_status;

typedef enum { JFA_F32 = 0, JFA_BF16 = 1 } jfa_dtype;

typedef struct {
  int64_t batch;   /* B >= 0 */
  int64_t total_q; /* T_q = offs_q[B] <= 2^31 - 1 */
  int64_t total_k; /* T_k = offs_k[B] <= 2^31 - 1; equal to total_q for self-attention */
  int32_t heads;   /* H >= 1; H * (max(T_q, T_k) / 32 + B + 1) <= 2^31 - 1 (work-list
                      items), else JFA_ERR_UNSUPPORTED */
  int32_t dim_qk;  /* Dqk: bf16 supports 64 and 128; fp32 supports 1..128 */
  int32_t dim_v;   /* Dv:  bf16 supports 64 and 128; fp32 supports 1..128 */
  float scale;     /* score scale > 0, normally 1/sqrt(Dqk) */
  int32_t causal;  /* 1: key j visible to query i only if j <= i (self-attention only) */
  int32_t dtype;   /* jfa_dtype of Q, K, V, O, dO, dQ, dK, dV */
  int32_t flags;   /* 0, or JFA_PLANNED (see jfa_plan); other bits: JFA_ERR_INVALID_ARG */
} jfa_params;

#define JFA_PLANNED 1

/*
 * Bytes of device workspace the calls below need for these params (work lists
 * of the jagged tile scheduler, the backward row term D, the status word).
 * Any call may be given a larger workspace.  Depends on batch, total_q,
 * total_k and heads only.  Returns 0 for a null pointer.
 */
size_t jfa_workspace_size(const jfa_params* p);

/*
 * Work lists built once for several calls (the jagged tile scheduler of the
 * Generalized Dot-Product Attention bullet, run once per batch instead of once
 * per call).  Every compute call starts by validating its offsets and building
 * its heavy-first work lists in the workspace.  jfa_plan does that once, for
 * the forward and the backward calls of these params: the same offsets serve
 * every call of a training step, and the plan serves every layer whose params
 * differ from the plan's only in scale, dim_qk, dim_v or dtype, as long as
 * jfa_path_for gives the same kernel family (and, for jfa_block_rope_*, dim_qk
 * is the plan's: the rotary table depends on it).
 *
 * A later call then passes params with flags = JFA_PLANNED, the same offsets
 * (the same pointers, their contents unchanged) and the same workspace; it
 * launches no scheduler and reads the planned lists.  Calls ordered after the
 * plan on the GPU (the same stream, or an event) may use it any number of
 * times, one at a time; it stays valid until the workspace is used by a call
 * without JFA_PLANNED or by another plan.  A planned call does not reset the
 * status word: it keeps the plan's status (JFA_ERR_BAD_OFFSETS makes every
 * planned call compute nothing), and after JFA_ERR_TIMEOUT the lists must be
 * planned again.  Nothing checks that a planned call's offsets are the plan's:
 * other offsets with the same totals produce wrong results, within the
 * buffers' bounds.
 *
 * jfa_plan serves jfa_fwd, jfa_bwd, jfa_cross_fwd, jfa_cross_bwd, jfa_gdpa_fwd
 * and jfa_gdpa_bwd (pass offs_q == offs_k for self-attention; causal needs
 * Lq_b == Lk_b, checked on the device); jfa_block_plan serves the four
 * BlockAttention calls (it also writes their block offsets and, where
 * jfa_block_rope_* is supported, the rotary table).  The pooled calls and
 * jfa_fwd_noalloc return JFA_ERR_UNSUPPORTED for JFA_PLANNED.  Argument errors
 * are those of the calls served; p->flags may be 0 or JFA_PLANNED and does not
 * change what is built.
 */
jfa_status jfa_plan(const jfa_params* p, const int64_t* offs_q, const int64_t* offs_k, void* ws,
                    size_t ws_bytes, jfa_stream_t stream);
jfa_status jfa_block_plan(const jfa_params* p, const int64_t* offs, void* ws, size_t ws_bytes,
                          jfa_stream_t stream);

/*
 * Softmax self-attention forward (Jagged Flash Attention bullet).  One offsets
 * array serves queries and keys (total_k must equal total_q).  Writes O and lse.
 * Causal masking is allowed.
 */
jfa_status jfa_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                   const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                   jfa_stream_t stream);

/*
 * Softmax self-attention backward, without atomics (Jagged Flash Attention
 * bullet): a key-tile-major pass writes dK and dV, a query-tile-major pass
 * writes dQ, each output element is written exactly once.  o and lse are the
 * outputs of jfa_fwd on the same inputs; dout is dL/dO.
 */
jfa_status jfa_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                   const void* o, const float* lse, const void* dout, const int64_t* offs,
                   void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                   jfa_stream_t stream);

/*
 * Softmax cross-attention forward with independent query and key offsets and
 * possibly Dv != Dqk (jagged-input bullet: cross and asymmetric-QKV patterns).
 * Causal must be 0.  A sequence with Lk_b == 0 yields o = 0 and lse = -inf.
 */
jfa_status jfa_cross_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const int64_t* offs_q, const int64_t* offs_k, void* o, float* lse,
                         void* ws, size_t ws_bytes, jfa_stream_t stream);

/* Backward of jfa_cross_fwd; same passes as jfa_bwd. */
jfa_status jfa_cross_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout,
                         const int64_t* offs_q, const int64_t* offs_k, void* dq, void* dk,
                         void* dv, void* ws, size_t ws_bytes, jfa_stream_t stream);

/*
 * Non-softmax (Generalized Dot-Product Attention bullet) forward:
 * P_ij = SiLU(s_ij) / Lq_b on the valid pairs, O = P V.  No lse is produced.
 * Pass the same pointer as offs_q and offs_k for self-attention; causal is
 * allowed only then (Lq_b == Lk_b is checked on the device).
 */
jfa_status jfa_gdpa_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                        const int64_t* offs_q, const int64_t* offs_k, void* o, void* ws,
                        size_t ws_bytes, jfa_stream_t stream);

/* Backward of jfa_gdpa_fwd (no D term, no lse); same two atomic-free passes. */
jfa_status jfa_gdpa_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                        const void* dout, const int64_t* offs_q, const int64_t* offs_k,
                        void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                        jfa_stream_t stream);

/*
 * Allocation-free variant of jfa_fwd.  The pages describe no such call; it
 * exists for callers that cannot allocate device memory at all -- for example
 * a plugin running inside a host application that owns the device allocator
 * and forbids other allocations, or a serving process that must not allocate
 * once it has started -- and so cannot provide the workspace jfa_fwd needs.
 *
 * Same arguments, layouts and results as jfa_fwd, minus the workspace: the
 * scratch (work lists and status word) lives in one 64 MiB array compiled
 * into the library, which every GPU that loads the library holds until the
 * process exits.  Requests whose workspace (jfa_workspace_size) would exceed
 * 64 MiB are rejected with JFA_ERR_WORKSPACE before anything is launched.
 * The call itself never allocates: no cudaMalloc, no cudaFree, no allocating
 * library routine.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current) and caches it;
 * make that first call before any stream capture.  The cache is keyed on the
 * CUDA context, not the device number: after cudaDeviceReset, or under another
 * context on the same device, the first call looks the address up again (and
 * that call, too, should come before any capture).  All calls share the one
 * array, which keeps the last call's contents, so calls that may overlap on
 * the GPU (different streams, or different host threads) race and must be
 * serialised by the caller.  Errors found on the device are silent here:
 * offsets that are not a valid jagged layout make the call compute nothing,
 * as in jfa_fwd, and a bounded wait inside a kernel that gives up leaves the
 * outputs incomplete; the status word that jfa_fwd's caller reads with
 * jfa_status_check lives in the shared array, which this variant's caller
 * cannot name.
 */
jfa_status jfa_fwd_noalloc(const jfa_params* p, const void* q, const void* k, const void* v,
                           const int64_t* offs, void* o, float* lse, jfa_stream_t stream);

/*
 * Pooled multi-head attention (Meta GEM MFU write-up,
 * piletech.kr/articles/112134, details section, jagged-input bullet: pooled
 * multi-head attention is one of the attention patterns over jagged
 * sequences).  m learned query rows per head, q [m, H, Dqk], are shared by
 * every sequence: sequence b's m outputs are the softmax attention of those
 * rows over its own keys and values, k/v rows offs_k[b] .. offs_k[b+1]-1
 * (non-causal, scale = p->scale).
 *   o   [B*m, H, Dv], lse [B*m, H]: sequence b's rows are b*m .. b*m+m-1;
 *       a sequence without keys gets o = 0, lse = -inf.
 *   dq  [m, H, Dqk]: the sum over sequences of each sequence's gradient of the
 *       shared rows (fixed order, bitwise reproducible); dk, dv as in
 *       jfa_cross_bwd.
 * p->batch = B, p->total_q = B*m (the rows of o), p->total_k = offs_k[B],
 * p->causal = 0.  The workspace (size from jfa_pooled_workspace_size, 256-byte
 * aligned) also holds the query rows broadcast to every sequence and their
 * per-sequence gradients, kept in fp32 until they are summed; it is used as by
 * jfa_cross_fwd / jfa_cross_bwd otherwise, and errors are reported the same
 * way.  Runs on the cross-attention kernels.
 */
size_t jfa_pooled_workspace_size(const jfa_params* p, int32_t m);
jfa_status jfa_pooled_fwd(const jfa_params* p, int32_t m, const void* q, const void* k,
                          const void* v, const int64_t* offs_k, void* o, float* lse, void* ws,
                          size_t ws_bytes, jfa_stream_t stream);
jfa_status jfa_pooled_bwd(const jfa_params* p, int32_t m, const void* q, const void* k,
                          const void* v, const void* o, const float* lse, const void* dout,
                          const int64_t* offs_k, void* dq, void* dk, void* dv, void* ws,
                          size_t ws_bytes, jfa_stream_t stream);

/*
 * BlockAttention (Meta GEM MFU write-up, piletech.kr/articles/112134, details
 * section, BlockAttention bullet: fixed 64-token blocks make attention linear
 * in the sequence length).  Softmax self-attention in which row i of a
 * sequence sees only the keys of its own block, rows 64*floor(i/64) ..
 * 64*floor(i/64)+63 of the same sequence (the last block may be shorter), and
 * with p->causal = 1 only those not after it.  Arguments and outputs as for
 * jfa_fwd / jfa_bwd.  The offsets are cut into blocks on the device and the
 * self-attention kernels run on the blocks as sequences of their own; the
 * workspace (jfa_block_workspace_size) holds the block offsets and room for up
 * to B + ceil(T/64) block sequences.  The pages combine the blocks with a fused
 * rotary position embedding: see jfa_block_rope_fwd / jfa_block_rope_bwd below.
 */
size_t jfa_block_workspace_size(const jfa_params* p);
jfa_status jfa_block_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                         jfa_stream_t stream);
jfa_status jfa_block_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                         const void* o, const float* lse, const void* dout, const int64_t* offs,
                         void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                         jfa_stream_t stream);

/*
 * BlockAttention with the fused rotary position embedding (same bullet: the 64-token
 * blocks are combined with a fused rotary position embedding).  The page gives none of
 * the embedding's parameters; this library follows RoFormer's definition: columns
 * (2i, 2i+1) of every q and k row, at position p, turn by the angle p * 10000^(-2i/D)
 * (D = dim_qk), with p the row's index inside its sequence.  Inside one block the scores
 * depend only on the difference of positions, so this equals counting positions from
 * each block's first row, which is how the kernels do it.  q and k are the unrotated
 * inputs; dq and dk are the gradients with respect to them.  The rotation is applied to
 * the Q and K tiles in shared memory between their load and the MMAs (no extra pass over
 * HBM), and its transpose to dQ and dK before they are stored.  Arguments, outputs,
 * workspace (jfa_block_workspace_size) and errors as for jfa_block_fwd / jfa_block_bwd;
 * bf16 with dim_qk == dim_v (64 or 128) only, else JFA_ERR_UNSUPPORTED.
 */
jfa_status jfa_block_rope_fwd(const jfa_params* p, const void* q, const void* k, const void* v,
                              const int64_t* offs, void* o, float* lse, void* ws, size_t ws_bytes,
                              jfa_stream_t stream);
jfa_status jfa_block_rope_bwd(const jfa_params* p, const void* q, const void* k, const void* v,
                              const void* o, const float* lse, const void* dout, const int64_t* offs,
                              void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                              jfa_stream_t stream);

/*
 * Synchronises `stream`, then returns the device status word of the last
 * call that used `ws` (JFA_OK, JFA_ERR_BAD_OFFSETS or JFA_ERR_TIMEOUT), or
 * JFA_ERR_CUDA if the synchronisation itself failed.
 */
jfa_status jfa_status_check(const void* ws, jfa_stream_t stream);

/* Static, human-readable name of a status code. */
const char* jfa_status_string(jfa_status s);

/*
 * Kernel timing, for benchmarks.  While enabled, every kernel the library
 * launches is bracketed by CUDA events recorded on its launch stream.
 * jfa_profile_read synchronises those events and returns, for kernel kind
 * `kind` (a JFA_KERNEL_* value), the number of launches and their summed
 * device time in milliseconds since the last reset.  Not thread-safe.
 */
enum {
  JFA_KERNEL_SCHEDULE = 0, /* jagged tile scheduler: offsets -> heavy-first work lists */
  JFA_KERNEL_FWD = 1,      /* forward tile loop */
  JFA_KERNEL_BWD_D = 2,    /* backward row term D = rowsum(dO * O) */
  JFA_KERNEL_BWD_DKDV = 3, /* key-tile-major dK/dV pass */
  JFA_KERNEL_BWD_DQ = 4,   /* query-tile-major dQ pass */
  JFA_KERNEL_AUX = 5,      /* pooled query broadcast and gradient sum; block offsets */
  JFA_KERNEL_KINDS = 6
};
jfa_status jfa_profile_enable(int on);
jfa_status jfa_profile_reset(void);
jfa_status jfa_profile_read(int kind, int64_t* launches, double* total_ms);

/*
 * Test hook for the bounded waits inside the tensor-core kernels.  Every wait on
 * an mbarrier in those kernels gives up after about two seconds, records
 * JFA_ERR_TIMEOUT in the workspace's status word, lets the CTA's other roles
 * leave, waits for the CTA's own copies and MMAs in flight and frees its
 * tensor memory, so the context stays usable.  While `on` is nonzero, every
 * bf16 forward launch in the calling thread's current context (jfa_fwd,
 * jfa_cross_fwd, jfa_gdpa_fwd and the calls built on them) starts with its MMA
 * issuer waiting on a barrier that nothing arrives on, before any MMA is
 * issued; the call then reports JFA_ERR_TIMEOUT through jfa_status_check and
 * leaves its outputs incomplete.  Off by default; turn it off again before
 * normal use.  Synchronises the device.
 */
jfa_status jfa_test_hold(int on);

/*
 * Which kernel family serves a request with these params: 1 = tcgen05/TMA
 * tensor-core kernels (bf16), 0 = CUDA-core fp32 kernels, -1 = unsupported.
 */
int jfa_path_for(const jfa_params* p);

/*
 * Base Batch Shuffling: a plan that spreads a global batch over `ranks`
 * data-parallel ranks with balanced attention work and no data exchanged
 * between ranks (Meta GEM MFU write-up, piletech.kr/articles/112134, details
 * section, Base Batch Shuffling bullet: sub-batches of 128 samples sorted by
 * sequence length, the heaviest merged with the lightest in turn).  Host
 * function; touches no GPU.  Every rank calls it with the same per-sample
 * costs and gets the same plan, then loads only the sub-batches assigned to
 * it.
 *
 * Plan (readings where the pages are silent):
 *   - sub-batch s holds samples s*sub .. min((s+1)*sub, n_samples)-1, and costs
 *     the sum of their `cost` (the caller's measure, e.g. useful attention
 *     FLOPs: Lq*Lk, or L(L+1)/2 when causal);
 *   - sub-batches are sorted by cost, heaviest first, ties by index;
 *   - pair i merges the i-th heaviest with the i-th lightest (the middle one of
 *     an odd count stays single);
 *   - pairs go to ranks in serpentine order 0, 1, .., R-1, R-1, .., 0, 0, ..,
 *     so ranks receive equally many pairs, within one.
 *
 * cost       host int64 [n_samples], every value >= 0
 * sub        samples per sub-batch (the pages use 128), >= 1
 * ranks      number of ranks, >= 1
 * sub_rank   host int32 [ceil(n_samples/sub)], out: rank of each sub-batch
 * sub_slot   host int32 [ceil(n_samples/sub)], out: its position in that
 *            rank's list (heavy member of a pair first)
 * rank_cost  host int64 [ranks] or NULL, out: each rank's total cost
 * Returns JFA_ERR_INVALID_ARG (and writes nothing) for n_samples < 0, sub < 1,
 * ranks < 1, a negative cost, or a NULL array with n_samples > 0.
 */
jfa_status jfa_bbs_plan(const int64_t* cost, int64_t n_samples, int32_t sub, int32_t ranks,
                        int32_t* sub_rank, int32_t* sub_slot, int64_t* rank_cost);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H_ */
