// Self-test of the bounded-wait error path: a kernel waits on an mbarrier
// that nothing ever arrives at.  The wait gives up after the library's limit
// (tc::kTimeoutCycles), the kernel records the timeout in the device error
// word and returns normally, so the context stays usable.
#include "q4k_internal.h"
#include "tc_ptx.cuh"

namespace q4k {
namespace {

__global__ void wait_timeout_selftest_kernel(int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (!tc::mbar_wait_sleep(&bar, 0)) atomicOr(err, 4);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace q4k
