// Failure-detection self test: a wait on an mbarrier that nothing arrives on.
//
// The kernel exercises the same bounded wait every pipeline of the library
// uses: it gives up after the limit, records BEA_STATUS_TIMEOUT in the device
// status word and returns normally, leaving the context usable.
#include "common.cuh"
#include "ptx.cuh"

namespace bea {
namespace {

__global__ void selftest_wait_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // phase 0 never completes: no thread arrives
    wait_parity(&bar, 0, &abort_flag, status, limit_ns);
  }
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(uint32_t* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_timeout_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace bea
