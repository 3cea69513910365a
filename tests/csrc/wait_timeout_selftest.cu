// Test-only kernel for the bounded pipeline waits of the library (sm103.cuh, mbar_wait).
//
// One CTA, two warps.  Warp 0 lane 0 waits on an mbarrier that nothing ever arrives on; after
// `timeout_ns` the wait gives up, sets the CTA's abort flag and records the timeout code in the
// status word.  Warp 1 lane 0 waits on a second, equally dead mbarrier with a limit 1000x longer;
// it must give up because it sees the abort flag, not because of its own limit.  Both return
// normally: no trap, no fault, the context stays usable.
#include <cstdint>
#include <cuda_runtime.h>

#include "sm103.cuh"

namespace {

__global__ void dead_wait_kernel(int* status, uint64_t timeout_ns, unsigned long long* elapsed) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(&bars[0], 1);
    fa::mbar_init(&bars[1], 1);
    fa::fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = fa::globaltimer_ns();
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    fa::Ctl ctl{&abort_flag, status, warp == 0 ? timeout_ns : timeout_ns * 1000};
    const bool ok = fa::mbar_wait(&bars[warp], 0, ctl);  // phase 0 never completes
    elapsed[warp] = ok ? 0ull : (fa::globaltimer_ns() - t0);
  }
  __syncthreads();
}

}  // namespace

extern "C" int wait_timeout_selftest(int timeout_ms, unsigned long long* elapsed_ns_host) {
  int* status = nullptr;
  unsigned long long* elapsed = nullptr;
  if (cudaMalloc(&status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMalloc(&elapsed, 2 * sizeof(unsigned long long)) != cudaSuccess) return -1;
  cudaMemset(status, 0, sizeof(int));
  cudaMemset(elapsed, 0, 2 * sizeof(unsigned long long));
  dead_wait_kernel<<<1, 64>>>(status, static_cast<uint64_t>(timeout_ms) * 1000000ull, elapsed);
  if (cudaDeviceSynchronize() != cudaSuccess) return -2;
  int st = 0;
  cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
  cudaMemcpy(elapsed_ns_host, elapsed, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  cudaFree(status);
  cudaFree(elapsed);
  return st;
}
