// jfa_fwd_noalloc: the softmax self-attention forward with its scratch in a
// fixed device array compiled into the library, for callers that cannot
// allocate device memory (see include/jfa.h).
//
// The scratch (scheduler work lists and status word) normally lives in the
// caller's workspace.  Here it lives in `g_scratch`, a file-scope __device__
// array of kNoallocScratchBytes that every GPU loading this library keeps
// until the process exits.  In host code `g_scratch` names only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress (with
// the device current) at set-up and cached; the kernels are given that address.
//
// The address belongs to one CUDA context's copy of the module, so the cache is
// keyed on the context, not on the device number: after cudaDeviceReset the
// primary context is a new one with its own copy of the array, and a driver-API
// context on the same device loads a separate copy.  Either way the first call
// under the new context looks the address up again.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)64 << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_scratch[kNoallocScratchBytes];

struct ScratchAddr {
  unsigned long long ctx;
  void* ptr;
};
std::mutex g_mutex;
std::vector<ScratchAddr> g_scratch_addr;  // one entry per context seen

// Device address of g_scratch in the current context; nullptr on failure.
void* scratch_in_current_context() {
  std::lock_guard<std::mutex> lock(g_mutex);
  const unsigned long long ctx = jfa::current_context_id();
  if (ctx != 0)
    for (const ScratchAddr& a : g_scratch_addr)
      if (a.ctx == ctx) return a.ptr;
  // set-up: the device that is current (and its context, which the runtime makes
  // current here if none was)
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();  // clear this (non-sticky) error so later calls do not see it
    return nullptr;
  }
  const unsigned long long now = jfa::current_context_id();
  if (now != 0) g_scratch_addr.push_back({now, ptr});
  return ptr;
}

}  // namespace

extern "C" jfa_status jfa_fwd_noalloc(const jfa_params* p, const void* q, const void* k,
                                      const void* v, const int64_t* offs, void* o, float* lse,
                                      jfa_stream_t stream) {
  if (p == nullptr) return JFA_ERR_INVALID_ARG;
  // its scratch is shared by every call, so it cannot hold a plan for later calls
  if (p->flags != 0) return (p->flags & ~JFA_PLANNED) ? JFA_ERR_INVALID_ARG : JFA_ERR_UNSUPPORTED;
  const size_t need = jfa_workspace_size(p);
  if (need == 0) return JFA_ERR_INVALID_ARG;
  if (need > kNoallocScratchBytes) return JFA_ERR_WORKSPACE;
  void* scratch = scratch_in_current_context();
  if (scratch == nullptr) return JFA_ERR_CUDA;
  return jfa_fwd(p, q, k, v, offs, o, lse, scratch, kNoallocScratchBytes, stream);
}
