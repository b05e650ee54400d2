// selftest.cu -- moe_fp8_selftest_wait: exercises the bounded device wait that every
// kernel of the library uses, without faulting or hanging the GPU.
//
// One thread waits on an mbarrier phase that nothing will complete (no copy, no MMA and no
// other thread is ever going to arrive on it), with a caller-given limit of microseconds.
// The wait gives up, the kernel sets MOE_STATUS_WAIT_TIMEOUT in the workspace's status word
// and returns, and the context stays usable -- the same path a kernel takes when one of its
// own waits runs out.
#include "launch.h"
#include "tc.cuh"

namespace moe {

__global__ void wait_selftest_kernel(Header* hdr, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, limit_ns)) set_status(hdr, MOE_STATUS_WAIT_TIMEOUT);
}

cudaError_t launch_wait_selftest(Header* hdr, uint32_t limit_us, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(hdr, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError();
}

}  // namespace moe
