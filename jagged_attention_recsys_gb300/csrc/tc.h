// Tensor-core (tcgen05 + TMA) jagged attention kernels for sm_103a, bf16 in, fp32 accumulate.
#pragma once

#include "internal.h"

namespace jfa {

bool tc_supports(int dim_qk, int dim_v);
// Test hook of the forward kernel's bounded waits (jfa_test_hold); synchronous.
cudaError_t tc_set_test_hold(int on);
SchedConfig tc_fwd_sched(const Problem& p);
SchedConfig tc_bwd_sched(const Problem& p);
cudaError_t launch_tc_fwd(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, const Workspace& ws, cudaStream_t s);
// Backward row pass: head-major (lse * log2 e, D = <dO, O>) pairs in the workspace.
cudaError_t launch_tc_rowstat(const Problem& p, const void* o, const void* dout, const float* lse,
                              const Workspace& ws, cudaStream_t s);
cudaError_t launch_tc_dkdv(const Problem& p, const void* q, const void* k, const void* v,
                           const float* lse, const void* dout, void* dk, void* dv,
                           const Workspace& ws, cudaStream_t s);
cudaError_t launch_tc_dq(const Problem& p, const void* q, const void* k, const void* v,
                         const float* lse, const void* dout, void* dq, const Workspace& ws,
                         cudaStream_t s);

}  // namespace jfa
