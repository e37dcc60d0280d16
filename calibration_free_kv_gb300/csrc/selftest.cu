// Self-test of the bounded waits every kernel uses on its mbarriers (copies and MMAs): one
// thread waits on a barrier that nothing will ever complete; the wait gives up after ~2 s,
// sets KVARN_DEV_WAIT_TIMEOUT and the kernel returns, leaving the context usable.  No fault,
// trap or endless loop is involved.
#include "common.cuh"

namespace kvarn {

__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait(&bar, 0)) flag_error(status, KVARN_DEV_WAIT_TIMEOUT);
}

}  // namespace kvarn

extern "C" int kvarn_selftest_wait_timeout(int32_t* dev_status, void* stream) {
  if (dev_status == nullptr) return KVARN_ERR_INVALID_ARG;
  kvarn::wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? KVARN_OK : KVARN_ERR_CUDA;
}
