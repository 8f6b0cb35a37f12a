// selftest.cu -- the failure-detection self-test: a bounded wait that runs out.
//
// Every wait of this library's kernels on an mbarrier is bounded (device.cuh,
// mbar_wait_bounded: 1 s of the global timer or 2^24 polls); a wait that runs
// out records PKV_ETIMEOUT in the pool's status word and the kernel returns
// instead of spinning.  This kernel drives exactly that path without a fault:
// one warp waits, through the same helper, on a barrier that nothing arrives
// on, then records the timeout and exits.  The context stays usable.
#include <cuda_runtime.h>

#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);                         // one arrival expected; none comes
    fence_mbar_init();
  }
  __syncwarp();
  const bool got = mbar_wait_bounded(&bar, 0);
  if (!__any_sync(0xffffffffu, got) && threadIdx.x == 0) record_error(status, PKV_ETIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
