// selftest.cu — attn_selftest_wait_timeout: runs the library's bounded mbarrier wait on a
// barrier that nothing ever arrives at, so a test can watch the wait give up, the timeout bit
// reach the device status word and the context stay usable, without faulting or hanging a GPU.
#include "common.cuh"

namespace attn {
namespace {

// One warp; the barrier expects one arrival that never comes.  Every lane waits through the same
// helper the attention kernels use (with the caller's short limit), then the kernel returns.
__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned int* status,
                                                          unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, status, limit_ns);
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" ATTN_API attn_status_t attn_selftest_wait_timeout(unsigned int timeout_us,
                                                             attn_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 2000000u) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  unsigned int* status = device_status_ptr();
  if (!status) return ATTN_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      status, static_cast<unsigned long long>(timeout_us) * 1000ull);
  return launch_status();
}
