// Self-test of the bounded device waits that every pipelined kernel here uses.
//
// One CTA initialises an mbarrier that nothing will ever arrive on and waits
// for it with the same helper the grouped GEMMs use, under a caller-chosen
// limit.  The wait must give up, raise the CTA's abort flag and report
// MOE_DEVERR_TIMEOUT through the status word; the kernel then returns
// normally, so the context stays usable.  Nothing traps or spins forever.

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

__global__ void wait_timeout_kernel(int* status, unsigned long long limit_ns,
                                    unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_timer_ns();
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns);
    if (waited_ns) *waited_ns = global_timer_ns() - t0;
    if (!ok) report(status, MOE_DEVERR_TIMEOUT);
  }
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status moe_selftest_wait_timeout(int32_t* status, int64_t limit_ns,
                                                uint64_t* waited_ns, moe_stream_t stream) {
  if (!status || limit_ns <= 0 || limit_ns > 1000000000LL)
    return set_last_error(MOE_ERR_INVALID_ARG,
                          "moe_selftest_wait_timeout: needs a status word and 0 < limit_ns <= 1e9");
  const moe_status st = moe_device_check();
  if (st != MOE_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, stream>>>(status, static_cast<unsigned long long>(limit_ns),
                                            reinterpret_cast<unsigned long long*>(waited_ns));
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return set_last_error(MOE_ERR_CUDA, cudaGetErrorString(err));
  return MOE_OK;
}
