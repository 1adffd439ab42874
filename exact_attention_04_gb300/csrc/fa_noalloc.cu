// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory.
//
// fa_bwd needs a caller-provided workspace.  Some callers have no way to get
// one: code that runs where a device allocation is not allowed (an allocator
// hook or a custom memory pool that must not re-enter itself, a plugin
// handed only its tensors by a host framework, a real-time loop that forbids
// cudaMalloc's implicit synchronisation).  For them this file keeps the
// workspace in a fixed array in device memory that belongs to the library.
//
// The array is FA_BWD_NOALLOC_MAX_SCRATCH_BYTES long.  Every GPU that loads
// this part of the library keeps it until the process exits.  Its device
// address is looked up per device, with that device current, by the first
// call that gets past the argument checks; make that first call before any
// stream capture.  A lookup that fails is not remembered: the call returns
// FA_ERR_CUDA, clears the error it left in the thread's last-error slot, and
// the next call tries again.  All calls share the one array: two calls whose
// kernels overlap on the GPU (different streams, or threads without
// ordering) race on it.  Nothing in it has to start at zero: the first of the
// three backward launches rewrites every region it later reads (D, the
// scaled LSE, and the zeroed dQ accumulator), so whatever the previous call
// left behind does not matter.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_MAX_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];   // device address per device, nullptr until found

// Device address of g_bwd_scratch on the current device (host code sees only
// a host-side stand-in for the array's name, never usable as a pointer), or
// nullptr if the lookup failed.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) == cudaSuccess) {
      g_scratch_ptr[dev] = ptr;
    } else {
      cudaGetLastError();   // leave no stale error for the launches of a later call
      return nullptr;
    }
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" fa_status_t fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                      const void* dO, const float* lse, void* dq, void* dk,
                                      void* dv, int B, int H, int N, int d, float scale,
                                      int causal, const int* kv_len, void* stream) {
  // fa_bwd's own checks first, so that every bad argument gets fa_bwd's code;
  // "workspace too small" becomes "scratch too small" (FA_ERR_INVALID_ARG).
  const size_t limit = static_cast<size_t>(FA_BWD_NOALLOC_MAX_SCRATCH_BYTES);
  const fa_status_t st = fa::bwd_check_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale,
                                            causal, kv_len, limit);
  if (st != FA_OK) return st;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len, scratch,
                limit, stream);
}
