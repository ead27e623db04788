// Self-test of the bounded-wait path: one CTA waits on a barrier that nothing
// signals; the wait must give up after the limit and record a timeout.
#include "bsa_internal.h"
#include "bsa_ptx.cuh"

namespace bsa {

__global__ void bsa_wait_selftest_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, status, limit_ns};
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, ctl, kSiteSelftest);
  __syncthreads();
}

cudaError_t launch_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  bsa_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace bsa
