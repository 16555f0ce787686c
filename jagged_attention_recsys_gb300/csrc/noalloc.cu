// jfa_fwd_noalloc: the softmax self-attention forward with its scratch in a
// fixed device array compiled into the library, for callers that cannot
// allocate device memory (see include/jfa.h).
//
// The scratch (scheduler work lists and status word) normally lives in the
// caller's workspace.  Here it lives in `g_scratch`, a file-scope __device__
// array of kNoallocScratchBytes that every GPU loading this library keeps
// until the process exits.  In host code `g_scratch` names only a host-side
// stand-in, so its device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached; the kernels are
// given that address.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)64 << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_scratch on the current device; nullptr on failure.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();  // clear this (non-sticky) error so later calls do not see it
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" jfa_status jfa_fwd_noalloc(const jfa_params* p, const void* q, const void* k,
                                      const void* v, const int64_t* offs, void* o, float* lse,
                                      jfa_stream_t stream) {
  if (p == nullptr) return JFA_ERR_INVALID_ARG;
  const size_t need = jfa_workspace_size(p);
  if (need == 0) return JFA_ERR_INVALID_ARG;
  if (need > kNoallocScratchBytes) return JFA_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return JFA_ERR_CUDA;
  return jfa_fwd(p, q, k, v, offs, o, lse, scratch, kNoallocScratchBytes, stream);
}
