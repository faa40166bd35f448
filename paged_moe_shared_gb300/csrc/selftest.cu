// Self-test of the kernels' failure path: a wait that can never be satisfied
// must give up after its limit, report RIMURU_DEV_TIMEOUT through a device
// status word and return, leaving the CUDA context usable.  The same bounded
// mbarrier wait guards every pipeline stage of the GEMM kernels.
#include <cuda_runtime.h>

#include <string>

#include "device.cuh"
#include "internal.h"

namespace rimuru {
namespace {

// One CTA: thread 0 initialises an mbarrier that expects one arrival, nobody
// arrives, and every thread of warp 0 waits for it with the given limit.
__global__ void bounded_wait_selftest_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);
    abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  const bool got = dev::mbar_wait(&bar, 0, &abort_flag, timeout_ns);
  if (!__all_sync(0xffffffffu, got) && threadIdx.x == 0) dev::set_error(status, RIMURU_DEV_TIMEOUT);
}

}  // namespace
}  // namespace rimuru

extern "C" int rimuru_selftest_bounded_wait(uint32_t timeout_us, int* status_out) {
  rimuru::clear_error();
  if (!status_out) return rimuru::fail(RIMURU_ERR_ARG, "null status pointer");
  if (timeout_us == 0 || timeout_us > 2000000u)
    return rimuru::fail(RIMURU_ERR_ARG, "timeout must be in (0, 2 s]");
  int* d_status = nullptr;
  cudaError_t e = cudaMalloc(&d_status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(d_status, 0, sizeof(int));
  if (e == cudaSuccess) {
    rimuru::bounded_wait_selftest_kernel<<<1, 32>>>(static_cast<uint64_t>(timeout_us) * 1000u,
                                                    d_status);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  int h = -1;
  if (e == cudaSuccess) e = cudaMemcpy(&h, d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (d_status) cudaFree(d_status);
  if (e != cudaSuccess)
    return rimuru::fail(RIMURU_ERR_CUDA, std::string("self-test: ") + cudaGetErrorString(e));
  *status_out = h;
  return RIMURU_OK;
}
