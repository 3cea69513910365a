// Microbenchmark (not part of the library): cycles per tcgen05.mma (kind::f16, cta_group::1,
// M = 128, K = 16) for several N, with A from shared memory (SS) or tensor memory (TS), with the
// issuing thread's sub-partition otherwise idle or shared with warps running independent FMA
// chains (or packed FFMA2, MUFU, tensor-memory loads).  One CTA per SM; thread 0 issues `iters`
// MMAs into one accumulator, commits and waits (bounded by the library's mbarrier wait).
// Operands are zero-filled (values are irrelevant).
// Prints one line per case: cycles per MMA at issue and at completion, FLOP/clk/SM, status.
#include <cstdio>
#include <cstdint>
#include "sm103.cuh"
using namespace fa;

// CHAIN: issue the MMAs 8 at a time through the library's one-asm K-step chain (N = 128, SS,
// K-major), as the attention kernels do.  KIND: what the busy warps run (0: four independent
// scalar FFMA chains; 1: four packed FFMA2 chains; 2: MUFU ex2; 3: tensor-memory loads of 32
// columns of their lane quadrant at columns [384, 512), which the MMAs do not touch).
template <int N, bool TS, bool BMN, int BUSY, bool CHAIN = false, int KIND = 0>
__global__ void __launch_bounds__(384, 1) rate_kernel(int iters, long long* out, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* sm = smem_raw + pad;
  for (int i = threadIdx.x; i < 131072 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 131072);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 131072 + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + 131072 + 16);
  if (threadIdx.x == 0) { *abort_flag = 0; mbar_init(bar, 1); fence_mbar_init(); }
  if (threadIdx.x < 32) { tmem_alloc(slot, 512); tmem_relinquish(); }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  const Ctl ctl{abort_flag, status, 2000000000ull};
  // BUSY extra warps per SMSP spin on dependent FMAs while thread 0 issues MMAs (warp w runs on
  // SMSP w % 4; thread 0 is in warp 0, so warps 4 and 8 share its SMSP)
  if (threadIdx.x >= 128 && (threadIdx.x / 128) <= BUSY) {
    float x0 = threadIdx.x * 1e-3f, x1 = x0 + 1.f, x2 = x0 + 2.f, x3 = x0 + 3.f, y = 1.0001f;
    float x4 = x0 + 4.f, x5 = x0 + 5.f, x6 = x0 + 6.f, x7 = x0 + 7.f;
    uint32_t u = 0;
    const uint32_t tq = tmem + (((threadIdx.x / 32u) & 3u) * 32u << 16) + 384u;
    for (int i = 0; i < iters * 8; ++i) {
      if (KIND == 0) {
        x0 = fmaf(x0, y, 1e-7f); x1 = fmaf(x1, y, 1e-7f); x2 = fmaf(x2, y, 1e-7f); x3 = fmaf(x3, y, 1e-7f);
      } else if (KIND == 1) {
        const float2 yy = make_float2(y, y), cc = make_float2(1e-7f, 1e-7f);
        float2 a0 = fma2(make_float2(x0, x1), yy, cc), a1 = fma2(make_float2(x2, x3), yy, cc);
        float2 a2 = fma2(make_float2(x4, x5), yy, cc), a3 = fma2(make_float2(x6, x7), yy, cc);
        x0 = a0.x; x1 = a0.y; x2 = a1.x; x3 = a1.y; x4 = a2.x; x5 = a2.y; x6 = a3.x; x7 = a3.y;
      } else if (KIND == 2) {
        x0 = ex2(x0 * -1e-3f); x1 = ex2(x1 * -1e-3f); x2 = ex2(x2 * -1e-3f); x3 = ex2(x3 * -1e-3f);
      } else if ((i & 3) == 0) {  // KIND 3, a quarter as many iterations: each waits for its load
        uint32_t r[32];
        tmem_ld32(tq + 32u * ((i >> 2) & 3), r);
        tmem_wait_ld();
        reg_fence(r);
        u ^= r[0] ^ r[31];
      }
    }
    if (x0 + x1 + x2 + x3 + x4 + x5 + x6 + x7 == 12345.f || u == 0xdeadbeefu) out[2] = 1;
  }
  if (threadIdx.x == 0) {
    const uint32_t sbase = smem_u32(sm);
    const uint64_t da = sdesc_sw128(sbase, 16384, 1024);           // A: 128 x 16, K-major
    const uint64_t db = sdesc_sw128(sbase + 32768, 16384, 1024);   // B
    constexpr uint32_t id = idesc_bf16(128, N, false, BMN);
    const long long t0 = clock64();
    if (CHAIN) {
      for (int i = 0; i < iters; i += 8) mma_ss_kmajor_k128(tmem + 0, da, db, id, i > 0 ? 1u : 0u);
    } else {
      for (int i = 0; i < iters; ++i) {
        if (TS) mma_ts(tmem + 0, tmem + 256, db, id, i > 0 ? 1u : 0u);
        else mma_ss(tmem + 0, da, db, id, i > 0 ? 1u : 0u);
      }
    }
    const long long t1 = clock64();
    mma_commit(bar);
    mbar_wait(bar, 0, ctl);
    const long long t2 = clock64();
    if (blockIdx.x == 0) { out[0] = t1 - t0; out[1] = t2 - t0; }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

template <int N, bool TS, bool BMN, int BUSY = 0, bool CHAIN = false, int KIND = 0>
void run(const char* name, int iters, long long* d_out, int* d_status) {
  auto k = rate_kernel<N, TS, BMN, BUSY, CHAIN, KIND>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 131072 + 2048);
  k<<<148, 384, 131072 + 2048>>>(iters, d_out, d_status);
  cudaError_t e = cudaDeviceSynchronize();
  long long h[2];
  cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
  int st = 0;
  cudaMemcpy(&st, d_status, sizeof(int), cudaMemcpyDeviceToHost);
  const double flop = 2.0 * 128 * N * 16;
  printf("%-22s N=%3d iters=%d  issue %.1f cyc/mma  complete %.1f cyc/mma  %.0f flop/clk/SM  %s st=%d\n",
         name, N, iters, double(h[0]) / iters, double(h[1]) / iters, flop * iters / double(h[1]),
         cudaGetErrorString(e), st);
}

int main() {
  long long* d_out; int* d_status;
  cudaMalloc(&d_out, 24); cudaMalloc(&d_status, 4); cudaMemset(d_status, 0, 4);
  const int it = 4096;
  run<64, false, false, 0>("SS, B K-major", it, d_out, d_status);
  run<128, false, false, 0>("SS, B K-major", it, d_out, d_status);
  run<256, false, false, 0>("SS, B K-major", it, d_out, d_status);
  run<64, true, true, 0>("TS, B MN-major", it, d_out, d_status);
  run<128, true, true, 0>("TS, B MN-major", it, d_out, d_status);
  run<256, true, true, 0>("TS, B MN-major", it, d_out, d_status);
  run<64, false, true, 0>("SS, B MN-major", it, d_out, d_status);
  run<128, false, true, 0>("SS, B MN-major", it, d_out, d_status);
  run<64, true, true, 1>("TS, +1 busy warp", it, d_out, d_status);
  run<64, true, true, 2>("TS, +2 busy warps", it, d_out, d_status);
  run<128, true, true, 2>("TS, +2 busy warps", it, d_out, d_status);
  run<128, false, false, 2>("SS, +2 busy warps", it, d_out, d_status);
  run<128, false, false, 1>("SS, +1 busy warp", it, d_out, d_status);
  run<256, false, false, 1>("SS, +1 busy warp", it, d_out, d_status);
  run<256, false, false, 2>("SS, +2 busy warps", it, d_out, d_status);
  run<128, false, false, 0, true>("SS chain of 8, idle", it, d_out, d_status);
  run<128, false, false, 2, true>("SS chain of 8, +2 busy", it, d_out, d_status);
  run<128, false, false, 2, false, 1>("SS, +2 busy FFMA2", it, d_out, d_status);
  run<128, false, false, 2, false, 2>("SS, +2 busy MUFU", it, d_out, d_status);
  run<128, false, false, 2, false, 3>("SS, +2 busy TMEM ld", it, d_out, d_status);
  return 0;
}
