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
// address is looked up once per device, on the first call made while that
// device is current; make that first call before any stream capture.  All
// calls share the one array: two calls whose kernels overlap on the GPU
// (different streams, or threads without ordering) race on it.  Nothing in
// it has to start at zero: the first of the three backward launches rewrites
// every region it later reads (D, the scaled LSE, and the zeroed dQ
// accumulator), so whatever the previous call left behind does not matter.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_MAX_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  std::once_flag once;
  cudaError_t err = cudaErrorUnknown;
  void* ptr = nullptr;
};

ScratchAddress g_scratch[kMaxDevices];

// Device address of g_bwd_scratch on the current device (host code sees only
// a host-side stand-in for the array's name, never usable as a pointer).
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  ScratchAddress& s = g_scratch[dev];
  std::call_once(s.once, [&s] {
    s.err = cudaGetSymbolAddress(&s.ptr, g_bwd_scratch);
    if (s.err != cudaSuccess) s.ptr = nullptr;
  });
  return s.err == cudaSuccess ? s.ptr : nullptr;
}

}  // namespace

extern "C" fa_status_t fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                      const void* dO, const float* lse, void* dq, void* dk,
                                      void* dv, int B, int H, int N, int d, float scale,
                                      int causal, const int* kv_len, void* stream) {
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > static_cast<size_t>(FA_BWD_NOALLOC_MAX_SCRATCH_BYTES)) return FA_ERR_INVALID_ARG;
  void* scratch = scratch_for_current_device();
  if (!scratch) return FA_ERR_CUDA;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len, scratch,
                static_cast<size_t>(FA_BWD_NOALLOC_MAX_SCRATCH_BYTES), stream);
}
