// Self-test of the bounded waits that every kernel in the library relies on.
//
// One thread initialises an mbarrier that nothing will ever arrive at and
// waits on it with the same bounded wait the attention kernels use, with a
// short limit.  The wait must give up, and the kernel must record the
// timeout in the device status word and return, so that fa_check() reports
// FA_ERR_TIMEOUT and the context stays usable.  Nothing faults or hangs: the
// wait ends at its limit by construction.
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kSiteSelfTest = 98;

__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(int* status,
                                                             unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  // parity 0 is the phase that is never completed: nobody arrives
  if (!ptx::mbar_wait(&bar, 0, &abort_flag, timeout_ns))
    atomicCAS(status, 0, status_code(kSiteSelfTest));
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, unsigned long long timeout_ns, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
