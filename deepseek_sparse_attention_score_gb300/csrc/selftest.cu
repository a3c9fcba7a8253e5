// Self-test of the bounded-wait path every pipeline kernel relies on: a wait
// on an mbarrier that nothing arrives on runs out after the given number of
// clocks, sets the abort flag and reports DSA_STATUS_TIMEOUT in the status
// word, and the kernel returns normally (no trap, the context stays usable).
#include "common.cuh"

namespace dsa {

namespace {
__global__ void wait_timeout_kernel(long long limit_clocks, int32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  if (!mbar_wait_limit(&bar, 0, &abort_flag, limit_clocks)) set_status(dev_status, DSA_STATUS_TIMEOUT);
}
}  // namespace

int run_wait_timeout_selftest(cudaStream_t stream, long long limit_clocks, int32_t* dev_status) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_clocks, dev_status);
  DSA_CHECK_LAUNCH();
  return DSA_OK;
}

}  // namespace dsa
