#include "tc.h"
namespace jfa {
bool tc_supports(int, int) { return false; }
SchedConfig tc_fwd_sched(const Problem&) { return kSimtSched; }
SchedConfig tc_bwd_sched(const Problem&) { return kSimtSched; }
cudaError_t launch_tc_fwd(const Problem&, const void*, const void*, const void*, void*, float*,
                          const Workspace&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_dkdv(const Problem&, const void*, const void*, const void*, const float*,
                           const void*, void*, void*, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_tc_dq(const Problem&, const void*, const void*, const void*, const float*,
                         const void*, void*, const Workspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace jfa
