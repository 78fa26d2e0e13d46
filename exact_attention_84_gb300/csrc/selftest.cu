// selftest.cu -- exercises the timeout path of the bounded waits.
//
// One thread block initialises an mbarrier that nothing will ever complete
// and waits on it with the same bounded wait every kernel of the library
// uses, here with a caller-chosen limit.  When the limit runs out the wait
// records the timeout in this file's device status word and the block exits
// normally: no trap, no fault, the context stays usable.  The host then sees
// FA_ERR_TIMEOUT from fa_get_device_status, exactly as it would if a real
// kernel's wait had run out.
#include "fa_device.cuh"
#include "fa_internal.h"

namespace fa {
namespace {

__device__ int g_status_selftest;

__global__ void selftest_timeout_kernel(uint64_t limit_ns, int* waited) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait_limit(smem_u32(&bar), 0, &abort_flag, &g_status_selftest, limit_ns);
    if (waited != nullptr) *waited = ok ? 0 : 1;
  }
}

}  // namespace

cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, nullptr);
  return cudaGetLastError();
}

int status_selftest(bool clear) {
  int s = 0;
  cudaMemcpyFromSymbol(&s, g_status_selftest, sizeof(int));
  if (clear && s != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_status_selftest, &zero, sizeof(int));
  }
  return s;
}

}  // namespace fa
