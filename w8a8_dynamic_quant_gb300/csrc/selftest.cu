// selftest.cu -- w8a8_selftest_bounded_wait: makes the library's bounded
// mbarrier wait run out on purpose, so that its error path (the status word
// receives W8A8_ERR_DEVICE_TIMEOUT, the kernel returns, the context stays
// usable) can be checked on a GPU without any fault or hang.
//
// Failure reporting follows the spirit of the failure table at the end of
// page "Qwen3.8-FP8 on Ascend 950: Why Weights Become MXFP8 at Load Time"
// ("Where It Breaks or Falls Back"): a condition the operation cannot meet
// is reported as an error code, never as a crash.  Here the condition is a
// wait whose event never comes: one CTA initialises one mbarrier that no
// thread arrives on and no copy completes on, and waits on it with the same
// helper (tc::mbar_wait) every tensor-core kernel uses, with a short limit.
// Nothing is in flight when the wait gives up, so the kernel simply returns.
#include "kernels.cuh"
#include "tc_common.cuh"

namespace w8a8 {
namespace {

__global__ void __launch_bounds__(32, 1) bounded_wait_kernel(DeviceStatus* st, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    tc::mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    // nobody arrives: phase 0 never completes, so the wait gives up after limit_ns
    if (tc::mbar_wait(smem_u32(&bar), 0u, &s_abort, st, 99u, limit_ns)) set_status(st, W8A8_ERR_CUDA, 98u);
  }
  __syncwarp();
}

}  // namespace
}  // namespace w8a8

using namespace w8a8;

extern "C" W8A8_API w8a8_status w8a8_selftest_bounded_wait(void* ws, uint32_t limit_us, w8a8_stream_t stream) {
  if (!ws) return W8A8_ERR_WORKSPACE;
  if (limit_us == 0 || limit_us > 2000000u) return W8A8_ERR_SHAPE;
  bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<DeviceStatus*>(ws),
                                                                           uint64_t(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}
