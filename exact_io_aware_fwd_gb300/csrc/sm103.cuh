// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA tile copies,
// tensor-memory allocation and access, and tcgen05 MMA with shared-memory descriptors.
//
// Every wrapper here is a direct use of one documented PTX instruction; nothing is taken from a
// vendor library.  Shared-memory tiles are in the 128-byte-swizzled layout that a TMA tile copy
// with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 64 bf16 (128 B), 8-row groups of 1024 B, and
// the 16-byte granule g of row r stored at granule g ^ (r & 7).  Every such tile starts on a
// 1024-byte boundary.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() {
  return __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
}

// ------------------------------------------------------------------------------------------
// Pipeline control shared by all roles of a CTA: an abort flag in shared memory and the
// library's device status word.  A wait that runs past `timeout_ns` sets both; every other wait
// in the CTA then gives up as soon as it sees the flag, so all roles reach the common exit.
struct Ctl {
  volatile int* abort_flag;  // shared memory
  int* status;               // global status word (first error wins)
  uint64_t timeout_ns;
};

enum : int { kErrTimeout = 4, kErrLayout = 1 };

__device__ __forceinline__ void ctl_fail(const Ctl& c, int code) {
  *c.abort_flag = 1;
  atomicCAS(c.status, 0, code);
}

// ------------------------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and leaves the CTA in
// the aborted state) if the wait runs past the limit or another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Ctl& c) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.timeout_ns) {
      ctl_fail(c, kErrTimeout);
      return false;
    }
  }
}

// Wait that ignores the abort flag, used only to drain this CTA's own asynchronous work (the
// copies and MMAs it issued) before it exits: a copy still in flight at exit would land in the
// shared memory of the next CTA on the SM.  Such work completes within microseconds whatever
// happened to the pipeline, so the limit never falls below kDrainLimitNs, however short the
// pipeline limit is; it only ends a wait on a memory system that has stopped answering.
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, const Ctl& c) {
  const uint32_t a = smem_u32(bar);
  const uint64_t limit = c.timeout_ns > kDrainLimitNs ? c.timeout_ns : kDrainLimitNs;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > limit) {
      ctl_fail(c, kErrTimeout);
      return;
    }
  }
}

// Whole-warp variant: every lane waits, and the warp agrees on the outcome so that the
// .sync.aligned instructions that follow are executed by all lanes or by none.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const Ctl& c) {
  bool ok = mbar_wait(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------------------------------
// Proxy fences and named barriers
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------------------------------
// TMA (tensor maps are kernel parameters declared __grid_constant__)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Contiguous bulk copy global -> shared (both addresses 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Element-wise float32 addition of `bytes` of shared memory into global memory by the TMA unit
// (both addresses 16-byte aligned, bytes % 16 == 0), tracked by the thread's bulk async-groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until every bulk async-group of this thread has completed (its writes performed).
__device__ __forceinline__ void bulk_wait0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy accesses to global memory (and those it synchronised with)
// before its later async-proxy ones (TMA), and vice versa.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// Tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// TMEM address: lane in bits 31..16, column in bits 15..0.  A warp may only touch the 32
// lanes of its quadrant (warp_id % 4).
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// 32 lanes x 32 consecutive 32-bit columns: thread (lane) i gets row i, columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}
#undef FA_R8
#undef FA_W8

// After tcgen05.wait::ld the registers are valid; this empty asm ties every register to a
// point after the wait so the compiler cannot hoist a use above it.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulator in tensor memory, one CTA)
//
// Shared-memory matrix descriptor (64 bit): start address >> 4 in bits 0..13, leading-
// dimension byte offset >> 4 in bits 16..29, stride-dimension byte offset >> 4 in bits 32..45,
// descriptor version 1 in bits 46..47, base offset 0, swizzle mode in bits 61..63
// (2 = 128-byte swizzle).
//  K-major operand (rows of the M/N dimension, K contiguous): SBO = 1024 (next 8-row group);
//    LBO unused.  Advance K by 16 elements = +32 bytes inside a 64-element (128 B) panel; the
//    next 64-element panel of K starts a separate [rows x 128 B] block.
//  MN-major operand (M/N contiguous in 64-element panels, K along rows): LBO = byte distance
//    between consecutive 64-element M/N panels, SBO = 1024 (next 8 K-rows); advance K by 16
//    rows = +2048 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16: D = f32 (bits 4..5 = 1), A = B = bf16 (bits 7..9 and
// 10..12 = 1), A/B major-ness in bits 15/16 (1 = MN-major), N >> 3 in bits 17..22,
// M >> 4 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]; A is M x K with row m in lane m, bf16 pairs packed per column.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Whole K-step chains in one asm block.  Step k uses the base descriptors plus constant offsets
// (16-byte units for shared-memory descriptors, columns for a tensor-memory A operand); the first
// step overwrites D unless `accumulate` is nonzero, the others accumulate.  Keeping the issuing
// thread's instructions between MMAs to two adds per step made the forward 3-4% faster on GB300.
// (Measured there: one tcgen05.mma per 64 cycles at N = 128 with the sub-partition otherwise
// idle; ~120 next to two warps issuing a scalar fp32 instruction every cycle, while packed
// FFMA2, MUFU, integer and tensor-memory-load traffic leave the rate at 64.)
#define FA_MMA_SS_STEP(AO, BO)                                                     \
  "add.s64 ra, %1, " #AO ";\n\tadd.s64 rb, %2, " #BO ";\n\t"                    \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, q;\n\t"
#define FA_MMA_TS_STEP(AO, BO)                                                     \
  "add.u32 ta, %1, " #AO ";\n\tadd.s64 rb, %2, " #BO ";\n\t"                    \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], rb, %3, q;\n\t"
#define FA_MMA_HEAD                                                                \
  "{\n\t.reg .pred p, q;\n\t.reg .b64 ra, rb;\n\t.reg .b32 ta;\n\t"          \
  "setp.ne.b32 p, %4, 0;\n\tsetp.ne.b32 q, %5, 0;\n\t"

// K-major A and B (S = Q K^T style), K = 64: steps of 32 bytes inside one 128-byte panel.
__device__ __forceinline__ void mma_ss_kmajor_k64(uint32_t d, uint64_t a, uint64_t b,
                                                  uint32_t id, uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               FA_MMA_SS_STEP(2, 2) FA_MMA_SS_STEP(4, 4) FA_MMA_SS_STEP(6, 6) "}"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}
// K = 128: two 64-element panels 16 KB apart.
__device__ __forceinline__ void mma_ss_kmajor_k128(uint32_t d, uint64_t a, uint64_t b,
                                                   uint32_t id, uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               FA_MMA_SS_STEP(2, 2) FA_MMA_SS_STEP(4, 4) FA_MMA_SS_STEP(6, 6)
               FA_MMA_SS_STEP(1024, 1024) FA_MMA_SS_STEP(1026, 1026)
               FA_MMA_SS_STEP(1028, 1028) FA_MMA_SS_STEP(1030, 1030) "}"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}
template <int D>
__device__ __forceinline__ void mma_ss_kmajor(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                              uint32_t accumulate) {
  static_assert(D == 64 || D == 128, "K = 64 or 128");
  if constexpr (D == 64) mma_ss_kmajor_k64(d, a, b, id, accumulate);
  else mma_ss_kmajor_k128(d, a, b, id, accumulate);
}
// A = bf16 pairs in tensor memory, 8 columns (16 K elements) per step; B MN-major, K = 128 rows
// of 128 bytes: +2048 bytes per step.
__device__ __forceinline__ void mma_ts_k128_step8(uint32_t d, uint32_t a_tmem, uint64_t b,
                                                  uint32_t id, uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               FA_MMA_TS_STEP(8, 128) FA_MMA_TS_STEP(16, 256) FA_MMA_TS_STEP(24, 384)
               FA_MMA_TS_STEP(32, 512) FA_MMA_TS_STEP(40, 640) FA_MMA_TS_STEP(48, 768)
               FA_MMA_TS_STEP(56, 896) "}"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}

// As mma_ts_k128_step8 with A packed per 64-element half: the first 64 K elements in columns
// [0, 32), the next 64 in [64, 96) (the layout of P^T / dS^T written by two elementwise groups).
__device__ __forceinline__ void mma_ts_k128_split(uint32_t d, uint32_t a_tmem, uint64_t b,
                                                  uint32_t id, uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               FA_MMA_TS_STEP(8, 128) FA_MMA_TS_STEP(16, 256) FA_MMA_TS_STEP(24, 384)
               FA_MMA_TS_STEP(64, 512) FA_MMA_TS_STEP(72, 640) FA_MMA_TS_STEP(80, 768)
               FA_MMA_TS_STEP(88, 896) "}"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}
// A and B both MN-major over K = 128 rows of 128 bytes: +2048 bytes per step for both.
__device__ __forceinline__ void mma_ss_mn_k128(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                               uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
               FA_MMA_SS_STEP(128, 128) FA_MMA_SS_STEP(256, 256) FA_MMA_SS_STEP(384, 384)
               FA_MMA_SS_STEP(512, 512) FA_MMA_SS_STEP(640, 640) FA_MMA_SS_STEP(768, 768)
               FA_MMA_SS_STEP(896, 896) "}"
               :: "r"(d), "l"(a), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}

// The mbarrier receives one arrive once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------------------------------
// Numerics helpers
// Packed fp32 pairs (sm_100 family): two correctly rounded operations per instruction.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Byte offset of 16-byte granule g (0..7) of row r inside a 128-byte-swizzled panel.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t g) {
  return r * 128u + ((g ^ (r & 7u)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Number of entries of the ascending list[0, cnt) below lim (whole warp; a sorted list fails the
// test only after its last passing entry).
__device__ __forceinline__ int warp_count_below(const int32_t* list, int cnt, int lim) {
  int total = 0;
  for (int c = 0; c < cnt; c += 32) {
    const int idx = c + static_cast<int>(lane_id());
    const bool ok = idx < cnt && __ldg(list + idx) < lim;
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    total += __popc(m);
    if (m != 0xffffffffu) break;
  }
  return total;
}

// ------------------------------------------------------------------------------------------
// Global-memory synchronisation between CTAs (the dQ accumulation protocol of the dK/dV kernel)
__device__ __forceinline__ uint64_t atom_add_acquire_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acquire.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Orders this thread's earlier memory operations, and those of other threads that it has
// synchronised with (cumulativity), before its later ones, at GPU scope.
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void st_v4(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

__device__ __forceinline__ void red_add_v4(float* gaddr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

}  // namespace fa
