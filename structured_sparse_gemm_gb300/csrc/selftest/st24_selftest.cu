// st24_selftest.cu -- self-test of the failure-detection path: one CTA waits,
// with the library's bounded wait, on an mbarrier that nothing arrives at.
// The wait gives up after its limit (about a second), records the timeout in
// the device status word and the kernel returns: no trap, no hang, no copy in
// flight, and the context stays usable.  Not on the product path.
#include "st24_device.cuh"
#include "st24_selftest.h"

namespace st24 {
namespace {

__global__ void wait_for_nothing(unsigned* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0u, status);   // phase 0 never completes
}

}  // namespace
}  // namespace st24

extern "C" st24_status st24_selftest_wait_timeout(void* stream) {
  const st24::DeviceInfo* dev = st24::current_device_info();
  if (!dev) return ST24_ERR_CUDA;
  st24::wait_for_nothing<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status);
  return cudaGetLastError() == cudaSuccess ? ST24_OK : ST24_ERR_CUDA;
}
