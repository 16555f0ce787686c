// Tensor-core backward (placeholder wiring: forwards to the CUDA-core passes until the
// tcgen05 dK/dV and dQ kernels land).
#include "tc.h"

namespace jfa {

SchedConfig tc_bwd_sched(const Problem&) { return kSimtSched; }

cudaError_t launch_tc_dkdv(const Problem& p, const void* q, const void* k, const void* v,
                           const float* lse, const void* dout, void* dk, void* dv,
                           const Workspace& ws, cudaStream_t s) {
  return launch_simt_dkdv(p, JFA_BF16, q, k, v, lse, dout, dk, dv, ws, s);
}

cudaError_t launch_tc_dq(const Problem& p, const void* q, const void* k, const void* v,
                         const float* lse, const void* dout, void* dq, const Workspace& ws,
                         cudaStream_t s) {
  return launch_simt_dq(p, JFA_BF16, q, k, v, lse, dout, dq, ws, s);
}

}  // namespace jfa
