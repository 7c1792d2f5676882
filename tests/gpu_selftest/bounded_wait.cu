// Test kernel for the library's bounded mbarrier wait (ptx.cuh): one thread
// waits on a barrier that nothing ever arrives on. The wait must give up after
// the limit and report it; the CUDA context must stay usable afterwards.
#include <cstdint>

#include "ptx.cuh"

__global__ void wait_on_silent_barrier(uint64_t limit_ns, int* status, unsigned long long* waited_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = mla::ptx::smem_addr(&bar);
  if (threadIdx.x == 0) mla::ptx::mbar_init(b, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = mla::ptx::globaltimer_ns();
    const bool ok = mla::ptx::mbar_wait_bounded(b, 0, limit_ns);
    *waited_ns = mla::ptx::globaltimer_ns() - t0;
    *status = ok ? 0 : -5;  // -5 = MLA_ERR_TIMEOUT
  }
}

extern "C" int run_wait_on_silent_barrier(uint64_t limit_ns, int* status_dev, unsigned long long* waited_dev) {
  wait_on_silent_barrier<<<1, 32>>>(limit_ns, status_dev, waited_dev);
  return (int)cudaDeviceSynchronize();
}
