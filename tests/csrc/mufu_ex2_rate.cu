// Microbenchmark (not part of the library): throughput of the MUFU exponential, the one
// transcendental of the online softmax (exp2 with log2 e folded into the scale).  One CTA per SM,
// every thread running 8 independent chains x -> ex2(x) - 1 (the subtraction keeps x in
// [-1/2, 0] and runs on the FMA pipe), in two forms: ex2.approx.ftz.f32 (one exponential per
// lane and instruction, the form the kernels use) and ex2.approx.ftz.bf16x2 (two per lane).
// The rate per SM comes from clock64 around each CTA's loop; the GPU-wide rate from CUDA events.
#include <cuda_bf16.h>
#include <cstdio>
#include <cstdint>

constexpr int kChains = 8;

template <bool kPacked>
__global__ void ex2_kernel(float* sink, unsigned long long* cycles, int iters) {
  __syncthreads();
  const unsigned long long t0 = clock64();
  float r = 0.f;
  if constexpr (!kPacked) {
    float x[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) x[c] = -0.001f * (threadIdx.x % 97 + c);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) {
        float y;
        asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x[c]));
        x[c] = y - 1.0f;
      }
    }
#pragma unroll
    for (int c = 0; c < kChains; ++c) r += x[c];
  } else {
    uint32_t x[kChains];
    const uint32_t one = 0x3f803f80u;  // (1.0, 1.0) in bf16
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      __nv_bfloat162 v = __floats2bfloat162_rn(-0.001f * (threadIdx.x % 97 + c), -0.002f * c);
      x[c] = *reinterpret_cast<uint32_t*>(&v);
    }
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) {
        uint32_t y;
        asm volatile("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x[c]));
        asm volatile("sub.rn.bf16x2 %0, %1, %2;" : "=r"(x[c]) : "r"(y), "r"(one));
      }
    }
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
      __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x[c]);
      r += __low2float(v) + __high2float(v);
    }
  }
  __syncthreads();
  const unsigned long long t1 = clock64();
  if (r == 12345.f) sink[threadIdx.x] = r;  // keeps the chains live; never true
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <bool kPacked>
static int run(const char* name, int sms, int threads, float* sink, unsigned long long* cyc) {
  const int iters = 2048;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  ex2_kernel<kPacked><<<sms, threads>>>(sink, cyc, 64);
  cudaEventRecord(a);
  ex2_kernel<kPacked><<<sms, threads>>>(sink, cyc, iters);
  cudaEventRecord(b);
  cudaError_t e = cudaEventSynchronize(b);
  if (e != cudaSuccess) {
    printf("%s: %s\n", name, cudaGetErrorString(e));
    return 1;
  }
  float ms;
  cudaEventElapsedTime(&ms, a, b);
  static unsigned long long h[1024];
  cudaMemcpy(h, cyc, sizeof(unsigned long long) * sms, cudaMemcpyDeviceToHost);
  unsigned long long mx = 0;
  for (int i = 0; i < sms; ++i) mx = h[i] > mx ? h[i] : mx;
  const double per_lane = kPacked ? 2.0 : 1.0;
  const double per_cta = double(threads) * iters * kChains * per_lane;
  printf("%s, %d threads per CTA: %.1f exponentials per cycle per SM, %.2f T exponentials/s\n",
         name, threads, per_cta / double(mx), per_cta * sms / (ms * 1e-3) / 1e12);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return 0;
}

int main() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms > 1024) sms = 1024;
  float* sink;
  unsigned long long* cyc;
  cudaMalloc(&sink, 1024 * sizeof(float));
  cudaMalloc(&cyc, 1024 * sizeof(unsigned long long));
  int rc = 0;
  for (int threads : {128, 256, 512}) rc |= run<false>("ex2.approx.ftz.f32", sms, threads, sink, cyc);
  for (int threads : {128, 256, 512}) rc |= run<true>("ex2.approx.ftz.bf16x2", sms, threads, sink, cyc);
  cudaFree(sink);
  cudaFree(cyc);
  return rc;
}
