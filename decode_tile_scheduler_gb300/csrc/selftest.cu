// selftest.cu -- fia_selftest_bounded_wait: the bounded barrier wait that
// every pipeline of the library uses, run against a barrier that nothing ever
// completes, so that its time-out path (error word 1, the kernel returns and
// the context stays usable) can be tested without a broken pipeline.
#include "common.cuh"
#include "internal.h"
#include "../../include/fia.h"

namespace fia {
namespace {

__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none ever comes
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    status[0] = 0;
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait_ns(&bar, 0, status, limit_ns);
    status[1] = (int32_t)((globaltimer_ns() - t0) / 1000);  // microseconds waited
    status[2] = ok ? 1 : 0;
  }
}

}  // namespace
}  // namespace fia

extern "C" fia_status fia_selftest_bounded_wait(int32_t* status, uint64_t limit_ns, void* stream) {
  if (!status) return FIA_ERR_NULL_ARG;
  if (limit_ns < 1000000ull || limit_ns > 1000000000ull) return FIA_ERR_BAD_SHAPE;
  fia::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? FIA_OK : FIA_ERR_CUDA;
}
