// Microbenchmark (not part of the library): GPU-wide throughput of fp32 additions into
// L2-resident memory, the operation the dK/dV kernel uses to accumulate dQ partials.  16-byte
// red.global.add.v4.f32 from every thread, against cp.reduce.async.bulk of 16 KB from shared
// memory issued by one thread per CTA.  Each CTA adds into its own 64 KB region of a 16 MB
// buffer; CUDA events around each launch; prints GB/s of additions (bytes of fp32 operands).
#include <cstdio>
#include <cstdlib>
#include <cstdint>
#include "sm103.cuh"
using namespace fa;

__global__ void __launch_bounds__(256, 1) red_v4_kernel(float* buf, int iters) {
  float* region = buf + (blockIdx.x & 255) * 16384;  // 64 KB
  for (int i = 0; i < iters; ++i) {
    // the CTA covers its 64 KB region once per iteration: 256 threads x 16 x 16 B
#pragma unroll
    for (int k = 0; k < 16; ++k)
      red_add_v4(region + (k * 256 + threadIdx.x) * 4, 1.f, 1.f, 1.f, 1.f);
  }
}

template <int INFLIGHT>
__global__ void __launch_bounds__(256, 1) red_bulk_kernel(float* buf, int iters) {
  extern __shared__ __align__(1024) uint8_t sm[];
  for (int e = threadIdx.x; e < 16384 / 4; e += blockDim.x) reinterpret_cast<float*>(sm)[e] = 1.f;
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    float* region = buf + (blockIdx.x & 255) * 16384;
    const uint32_t src = smem_u32(sm);
    for (int i = 0; i < iters; ++i) {
      for (int q = 0; q < 4; ++q) {  // the 64 KB region in four 16 KB bulk reductions
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                     :: "l"(region + q * 4096), "r"(src), "r"(16384) : "memory");
        bulk_commit();
        asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(INFLIGHT) : "memory");
      }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  __syncthreads();
}

int main() {
  float* buf;
  cudaMalloc(&buf, 16 << 20);
  cudaMemset(buf, 0, 16 << 20);
  cudaEvent_t a, b;
  cudaEventCreate(&a); cudaEventCreate(&b);
  const int iters = 200, ctas = 148;
  const double bytes = double(ctas) * iters * 65536;
  for (int rep = 0; rep < 2; ++rep) {
    red_v4_kernel<<<ctas, 256>>>(buf, 5);
    cudaEventRecord(a);
    red_v4_kernel<<<ctas, 256>>>(buf, iters);
    cudaEventRecord(b);
    cudaError_t e = cudaEventSynchronize(b);
    if (e != cudaSuccess) { printf("red.v4: %s\n", cudaGetErrorString(e)); return 1; }
    float ms; cudaEventElapsedTime(&ms, a, b);
    printf("red.global.add.v4.f32, 148 CTAs x 256 threads: %.0f GB/s of fp32 additions\n", bytes / ms / 1e6);
    cudaFuncSetAttribute(red_bulk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384);
    cudaFuncSetAttribute(red_bulk_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384);
    red_bulk_kernel<1><<<ctas, 256, 16384>>>(buf, 5);
    cudaEventRecord(a);
    red_bulk_kernel<1><<<ctas, 256, 16384>>>(buf, iters);
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    if (e != cudaSuccess) { printf("bulk: %s\n", cudaGetErrorString(e)); return 1; }
    cudaEventElapsedTime(&ms, a, b);
    printf("cp.reduce.async.bulk 16 KB, 2 in flight per CTA: %.0f GB/s\n", bytes / ms / 1e6);
    red_bulk_kernel<0><<<ctas, 256, 16384>>>(buf, 5);
    cudaEventRecord(a);
    red_bulk_kernel<0><<<ctas, 256, 16384>>>(buf, iters);
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    if (e != cudaSuccess) { printf("bulk0: %s\n", cudaGetErrorString(e)); return 1; }
    cudaEventElapsedTime(&ms, a, b);
    printf("cp.reduce.async.bulk 16 KB, 1 in flight per CTA: %.0f GB/s\n", bytes / ms / 1e6);
  }
  return 0;
}
