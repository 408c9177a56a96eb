// selftest.cu -- a device check of the failure path every pipeline wait in
// this library shares: a wait that nothing completes gives up after its time
// limit, reports SA_DEV_TIMEOUT in the caller's status word and lets the
// kernel return, so the context stays usable. Nothing here faults, traps or
// hangs: the wait is the library's own bounded mbarrier wait.
#include "ptx.cuh"
#include "sa_internal.cuh"

namespace sa {
namespace {

// One CTA of one warp: an mbarrier that expects one arrival nobody makes.
__global__ void __launch_bounds__(32) wait_never_kernel(int32_t* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const volatile int never = 0;
  const bool done = mbar_wait_warp(b, 0, AbortSignal{&never, nullptr});
  if (!done && threadIdx.x == 0 && dev_status) atomicOr(dev_status, SA_DEV_TIMEOUT);
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_check_wait_timeout(int32_t* dev_status, void* stream) {
  if (!dev_status) return SA_ERR_INVALID_ARG;
  sa::wait_never_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}
