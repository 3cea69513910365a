// Forward kernel: exact attention O = softmax(scale * Q K^T) V and LSE, one CTA per
// (b, h, 256-row query block) holding two 128-row query tiles that alternate on the tensor core.
//
// Method (first page "FlashAttention：不减少一次注意力计算，为什么反而更快", sections 关键设计一
// and 关键设计二; page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section
// "FlashAttention-1：分块与在线 softmax", Fig. 4): for each key tile K_j, V_j the CTA computes
// S_ij = Q_i K_j^T, updates the running row max m and row sum l, and accumulates the
// unnormalised output O~ += P~ V_j; O = O~ / l and LSE = m + log l are written once at the end.
// S_ij and P_ij live only in tensor memory.
//
// GB300 design (the pages' A100 tile rules are prior art, not the blueprint):
//  * warp 0: TMA producer.  Q tiles once, then K_j and V_j through a ring of smem stages with
//    full/empty mbarriers (page two, section "FlashAttention-3", Fig. 7: producer warps load,
//    consumer warps compute).
//  * warp 1: single-thread tcgen05.mma issuer.  S_t = Q_t K_j^T (both operands in smem) and
//    O_t += P_t V_j with P_t read straight from tensor memory, alternating the two tiles so
//    that one tile's softmax overlaps the other tile's MMAs (ping-pong of FlashAttention-3).
//  * dense d = 64 (kHalfSteps): each 128-key K/V stage is consumed as two 64-key half steps,
//    so the two tiles need 256 tensor-memory columns and two CTAs (of 320 threads, softmax in
//    warps 2-9) share an SM: four query tiles in flight per SM.
//  * warps 4-7 / 8-11: one warpgroup per query tile, one thread per query row: tcgen05.ld of
//    the S row, row max, exp2 of (S * scale * log2 e - m), P packed to bf16 and stored back
//    over S in tensor memory, row sum.  O~ is rescaled in tensor memory only when the running
//    max of some row of the warp moved (conditional rescaling, page two, section
//    "FlashAttention-4"); results stay exact because l and O~ always use the same reference.
//  * causal: key tiles past the diagonal are skipped, the diagonal tile is masked element-wise
//    (page two, FlashAttention-1 section, causal paragraph).
//  * epilogue: O~ / l -> bf16 -> swizzled smem (over the Q tile) -> TMA store (rows >= N are
//    clipped by the tensor map); LSE with plain coalesced stores.
//  * variable-length (kVarlen): packed [total, H, d] tensors with per-sequence token offsets;
//    a sequence's tiles are 3-D TMA boxes (d, head, token) that may run into the next
//    sequence: those keys are masked like padding, and the rows of a sequence's last tile are
//    stored one by one instead of by the (sequence-blind) TMA store.  Grouped-query attention
//    reads K and V of head h / (H / Hkv).
//  * block-sparse (kSparse): the K/V stream is the union of the kept key tiles of the CTA's two
//    query tiles (a sorted list from the block index); each query tile runs S, softmax and P V
//    only on its own kept tiles, so skipped tiles cost neither loads nor MMAs (page two,
//    FlashAttention-1 section: the block-sparse extension skips zero blocks).
#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

namespace {

// Rescale when the running max grows by more than this (log2 units).  Measured on GB300:
// 8 (a stale reference, FlashAttention-4 style) is 3.5% faster on the long causal case but the
// row's largest probability is then 2^delta instead of exactly 1 and its bf16 rounding is not
// cancelled by l; with large logits that pushes O past 1e-2.  0 keeps the exact running max
// (the O~ correction is still skipped for a warp whose 32 rows all kept their max).
#ifndef FA_RESCALE_THRESHOLD
#define FA_RESCALE_THRESHOLD 0.0f
#endif
// 1: normalise O~ by the sum of the bf16-rounded P and keep a separate exact sum for LSE
// (the alternative fix for a stale max; 9% slower, so off by default).
#ifndef FA_ROUNDED_SUM
#define FA_ROUNDED_SUM 0
#endif
// Software exp2 (FlashAttention-4's idea of moving part of the exponentials off the MUFU pipe,
// page two, section "FlashAttention-4"): N > 0 sends one pair of every N in the unmasked softmax
// loop through exp2_poly2 on the FMA pipe instead of MUFU ex2.  Off: measured slower on GB300
// (MUFU is not the ceiling; the extra instructions crowd the MMA-issuing thread).
#ifndef FA_SOFT_EXP2
#define FA_SOFT_EXP2 0
#endif
constexpr float kRescaleThreshold = FA_RESCALE_THRESHOLD;

// 2^x for a pair, x <= 0: 2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2].  Adding
// 1.5 * 2^23 rounds x to an integer held in the low mantissa bits of t; 2^f comes from a degree-3
// polynomial (least-squares fit of 2^f on Chebyshev nodes of [-1/2, 1/2], relative error below
// 8e-5, far under the 2^-9 of the bf16 rounding that P gets next), and 2^n is applied by adding
// n << 23 to the polynomial's exponent field (t << 23 is exactly n << 23: the low 9 bits of
// 1.5 * 2^23's pattern are zero).  x is clamped at -126 so that the exponent stays in range.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  x.x = fmaxf(x.x, -126.f);
  x.y = fmaxf(x.y, -126.f);
  const float2 magic = make_float2(12582912.f, 12582912.f);
  const float2 t = add2(x, magic);
  const float2 r = add2(t, make_float2(-12582912.f, -12582912.f));  // round(x), exact
  const float2 f = fma2(r, make_float2(-1.f, -1.f), x);               // x - round(x), exact
  float2 q = fma2(make_float2(0.05508868396282196f, 0.05508868396282196f), f,
                  make_float2(0.24260404706001282f, 0.24260404706001282f));
  q = fma2(q, f, make_float2(0.6932762265205383f, 0.6932762265205383f));
  q = fma2(q, f, make_float2(0.9999289512634277f, 0.9999289512634277f));
  const uint32_t e0 = __float_as_uint(q.x) + __float_as_uint(t.x) * 8388608u;
  const uint32_t e1 = __float_as_uint(q.y) + __float_as_uint(t.y) * 8388608u;
  return make_float2(__uint_as_float(e0), __uint_as_float(e1));
}
constexpr float kLn2 = 0.693147180559945309f;

// O += P V over 64 keys: A = bf16 pairs in tensor memory, 8 columns per 16-key step; B (V)
// MN-major, 16 key rows of 128 bytes = +2048 bytes per step.
__device__ __forceinline__ void mma_ts_k64_step4(uint32_t d, uint32_t a_tmem, uint64_t b,
                                                 uint32_t id, uint32_t accumulate) {
  asm volatile(FA_MMA_HEAD
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               FA_MMA_TS_STEP(8, 128) FA_MMA_TS_STEP(16, 256) FA_MMA_TS_STEP(24, 384) "}"
               :: "r"(d), "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate), "n"(1) : "memory");
}

// Dense d = 64: each 128-key K/V stage is consumed as two 64-key half steps (S of 128 x 64,
// softmax over 64 scores per row, P V over 64 keys), so a CTA's two query tiles need 64 + 64
// tensor-memory columns each and two CTAs share an SM: four query tiles in flight per SM
// instead of two.  At d = 64 the tiles' serial chains (S -> softmax -> P V), not the tensor
// pipe, set the pace; more tiles in flight fill the pipe.
template <int D, bool kSparse, bool kVarlen>
constexpr bool kHalfSteps = (D == 64) && !kSparse && !kVarlen;
// Threads per CTA: warp 0 TMA, warp 1 MMA, then two softmax warpgroups (warps 4-11; with half
// steps warps 2-9, so that two CTAs' 640 threads get 96 registers each: a warp's tensor-memory
// lanes follow warp % 4, so any four consecutive warps cover the 128 rows).
template <int D, bool kSparse, bool kVarlen>
constexpr int kFwdThreads = kHalfSteps<D, kSparse, kVarlen> ? 320 : 384;

template <int D, bool kHalf = false>
struct FwdLayout {
  static constexpr uint32_t kTile = 128u * D * 2u;  // one 128 x D bf16 tile
  static constexpr int kStages = kHalf ? 2 : ((D == 64) ? 4 : 2);
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + 2 * kTile;
  static constexpr uint32_t kV = kK + kStages * kTile;
  static constexpr uint32_t kBar = kV + kStages * kTile;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full[2], o_full[2], done
  static constexpr int kNumBars = 1 + 4 * kStages + 7;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kCnt = kAbort + 4;  // block-sparse counts: positions, n_0, n_1
  static constexpr uint32_t kBytes = kCnt + 12;
  // TMEM columns: S_0, S_1 (128 each, 64 with half steps), O_0, O_1 (D each)
  static constexpr uint32_t kSCols = kHalf ? 64 : 128;
  static constexpr uint32_t kColS0 = 0, kColO0 = 2 * kSCols;
  static constexpr uint32_t kTmemCols = kHalf ? 256 : 512;
};

template <int D, bool kSparse, bool kVarlen>
__global__ void __launch_bounds__((kFwdThreads<D, kSparse, kVarlen>),
                                  (kHalfSteps<D, kSparse, kVarlen> ? 2 : 1))
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const FwdArgs a) {
  constexpr bool kHalf = kHalfSteps<D, kSparse, kVarlen>;
  using L = FwdLayout<D, kHalf>;
  constexpr int S = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* sm = smem_raw + pad;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + S;
  uint64_t* v_full = k_empty + S;
  uint64_t* v_empty = v_full + S;
  uint64_t* s_full = v_empty + S;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* mma_done = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const Ctl ctl{abort_flag, a.status, a.timeout_ns};

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  if (pad + L::kBytes > a.smem_bytes) {  // cannot happen with the host's sizing; never proceed
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kErrLayout);
    return;
  }

  // ---- work item: heads in groups of `head_group` whose K/V fit in about half of L2; within a
  // group block level major (all heads of one level together) and, with a causal mask, the
  // heaviest blocks first, so that every wave holds CTAs of similar length and the light ones
  // fill the tail.  Groups run one after another.
  // (variable-length: the same order with the longest sequence's block count; the blocks past a
  // shorter sequence's end exit at once)
  const int lin = blockIdx.x;
  const int gsz = a.head_group * a.num_qblocks;  // CTAs per full group
  const int grp = lin / gsz;
  const int heads = min(a.head_group, a.BH - grp * a.head_group);  // heads in this group
  const int idx = lin - grp * gsz;
  const int bh = grp * a.head_group + idx % heads;
  const int qb = a.causal ? (a.num_qblocks - 1 - idx / heads) : (idx / heads);
  const int b = bh / a.H;
  const int h = bh - b * a.H;
  const int hk = h / (a.H / a.Hkv);  // key/value head
  int seq_start = 0, N = a.N;        // this sequence's first token and length
  if constexpr (kVarlen) seq_bounds(a.cu_seqlens, b, a.total, seq_start, N);
  const int q0 = qb * 256;
  if (kVarlen && q0 >= N) return;  // past this sequence's end (uniform over the CTA)
  int kv_len = N;
  if (!kVarlen && a.kv_lens != nullptr) kv_len = min(max(__ldg(a.kv_lens + b), 0), N);
  // TMA box coordinates (y, z) of row r: dense (r, head slice), packed (head, token)
  const int q_y0 = kVarlen ? h : 0, q_z0 = kVarlen ? seq_start : bh;
  const int kv_y0 = kVarlen ? hk : 0, kv_z0 = kVarlen ? seq_start : b * a.Hkv + hk;
  auto row_y = [&](int y0, int r) { return kVarlen ? y0 : r; };
  auto row_z = [&](int z0, int r) { return kVarlen ? z0 + r : z0; };
  int nb[2], nh[2];  // key tiles (128 keys) and half steps (64 keys) of each query tile
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt0 = q0 + 128 * t;
    int nkeys = kv_len;
    if (a.causal) nkeys = min(nkeys, qt0 + 128);
    nb[t] = (qt0 < N) ? (nkeys + 127) / 128 : 0;
    nh[t] = (qt0 < N) ? (nkeys + 63) / 64 : 0;
  }
  const int nb_max = max(nb[0], nb[1]);
  const int T = (N + 127) / 128;

  // block-sparse: the CTA's K/V stream (f_list) and each query tile's key tiles (r_list) come
  // from the block index, cut at the causal / key-length limits nb[]
  const int32_t* f_list = nullptr;
  const int32_t* r_list[2] = {nullptr, nullptr};
  int* cnt_smem = reinterpret_cast<int*>(sm + L::kCnt);
  if constexpr (kSparse) {
    const BlockIndex BI = block_index_layout(T);
    const int32_t* base = a.blk + (a.blk_heads == 1 ? 0 : static_cast<int64_t>(bh % a.H) * BI.words);
    f_list = base + BI.fidx + static_cast<int64_t>(qb) * T;
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (2 * qb + t < T) r_list[t] = base + BI.ridx + static_cast<int64_t>(2 * qb + t) * T;
    if (warp == 2) {
      const int np = warp_count_below(f_list, __ldg(base + BI.fcnt + qb), nb_max * 4);
      int nt[2] = {0, 0};
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (r_list[t] != nullptr)
          nt[t] = warp_count_below(r_list[t], __ldg(base + BI.rcnt + 2 * qb + t), nb[t]);
      if (lane == 0) {
        cnt_smem[0] = np;
        cnt_smem[1] = nt[0];
        cnt_smem[2] = nt[1];
      }
    }
  }

  // ---- setup.  Without a block mask the K/V stream's length is known here, and the thread that
  // initialises the barriers also issues the copies that need no wait (the Q tiles and the first
  // S K/V stages, all fresh) before the CTA-wide barrier that the tensor-memory allocation also
  // waits for; the producer loop then starts at the first stage it has to wait for.
  const int ntiles_q = (nb[1] > 0) ? 2 : 1;
  auto issue_k = [&](int j, int kt) {
    const int s = j % S;
    mbar_arrive_expect_tx(&k_full[s], L::kTile);
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sm + L::kK + s * L::kTile + c * 16384, &tmK, &k_full[s], c * 64,
                  row_y(kv_y0, kt * 128), row_z(kv_z0, kt * 128));
  };
  auto issue_v = [&](int j, int kt) {
    const int s = j % S;
    mbar_arrive_expect_tx(&v_full[s], L::kTile);
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sm + L::kV + s * L::kTile + c * 16384, &tmV, &v_full[s], c * 64,
                  row_y(kv_y0, kt * 128), row_z(kv_z0, kt * 128));
  };
  auto issue_q = [&]() {
    mbar_arrive_expect_tx(q_full, ntiles_q * L::kTile);
    for (int t = 0; t < ntiles_q; ++t)
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sm + L::kQ + t * L::kTile + c * 16384, &tmQ, q_full, c * 64,
                    row_y(q_y0, q0 + 128 * t), row_z(q_z0, q0 + 128 * t));
  };
  const int n_pre = kSparse ? 0 : min(nb_max, S);  // K/V stages issued during the setup
  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_full[t], 1);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
    if (n_pre > 0) {
      issue_q();
      for (int j = 0; j < n_pre; ++j) {
        issue_k(j, j);
        issue_v(j, j);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);
  // positions of the K/V stream and key tiles per query tile
  const int npos = kSparse ? cnt_smem[0] : nb_max;
  const int ncnt[2] = {kSparse ? cnt_smem[1] : nb[0], kSparse ? cnt_smem[2] : nb[1]};

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0 && npos > 0) {
      if (n_pre == 0) issue_q();
      int jk = n_pre, jv = n_pre;  // K and V tiles whose copies have been issued
      for (int j = n_pre; j < npos; ++j) {
        const int s = j % S;
        const uint32_t ph = (j / S) & 1;
        const int kt = kSparse ? (__ldg(f_list + j) >> 2) : j;  // key tile at position j
        if (!mbar_wait(&k_empty[s], ph ^ 1, ctl)) break;
        issue_k(j, kt);
        jk = j + 1;
        if (!mbar_wait(&v_empty[s], ph ^ 1, ctl)) break;
        issue_v(j, kt);
        jv = j + 1;
      }
      // No copy into this CTA's shared memory may still be in flight when the CTA exits, whether
      // or not any role has aborted (one may time out after this thread left its loop).  In a
      // normal run the consumers have already waited for these phases.
      drain_wait(q_full, 0, ctl);
      for (int jj = max(0, jk - S); jj < jk; ++jj) drain_wait(&k_full[jj % S], (jj / S) & 1, ctl);
      for (int jj = max(0, jv - S); jj < jv; ++jj) drain_wait(&v_full[jj % S], (jj / S) & 1, ctl);
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (kHalf && lane == 0 && npos > 0) {
      // Half steps hs = 0 .. nh_max: step hs reads half (hs & 1) of K/V stage hs >> 1.  Per
      // step and query tile: P V of the previous half step, then S of this one (S overwrites
      // that tile's P).  A K stage is released after the S MMAs of its last half step, a V
      // stage after the P V MMAs of its last half step.
      constexpr uint32_t idSh = idesc_bf16(128, 64, false, false);  // S half: 64 keys
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);     // O += P V, V is MN-major
      constexpr uint32_t kHalfBytes = 64u * 128u;                   // 64 key rows of 128 bytes
      bool ok = mbar_wait(q_full, 0, ctl);
      const int nhmax = max(nh[0], nh[1]);
      int cnt[2] = {0, 0};  // S MMAs issued per query tile
      for (int hs = 0; ok && hs <= nhmax; ++hs) {
        const int j = hs >> 1, hf = hs & 1;  // stage position and half of this step
        const int s = j % S;
        const int jp = (hs - 1) >> 1, hp = (hs - 1) & 1;  // those of the previous step (hs >= 1)
        const int sp = (hs >= 1) ? jp % S : 0;
        if (hs < nhmax && hf == 0 && !(ok = mbar_wait(&k_full[s], (j / S) & 1, ctl))) break;
        if (hs >= 1 && hp == 0 && !(ok = mbar_wait(&v_full[sp], (jp / S) & 1, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (hs >= 1 && hs - 1 < nh[t]) {
            if (!(ok = mbar_wait(&p_full[t], (cnt[t] - 1) & 1, ctl))) break;
            tc_fence_after();
            mma_ts_k64_step4(tmem + L::kColO0 + D * t, tmem + L::kColS0 + L::kSCols * t,
                             sdesc_sw128(sbase + L::kV + sp * L::kTile + hp * kHalfBytes, 16384,
                                         1024),
                             idO, cnt[t] > 1 ? 1u : 0u);
            if (cnt[t] == nh[t]) mma_commit(&o_full[t]);  // the tile's last P V
          }
          if (hs < nh[t]) {
            mma_ss_kmajor<D>(tmem + L::kColS0 + L::kSCols * t,
                             sdesc_sw128(sbase + L::kQ + t * L::kTile, 16384, 1024),
                             sdesc_sw128(sbase + L::kK + s * L::kTile + hf * kHalfBytes, 16384,
                                         1024),
                             idSh, 0u);
            mma_commit(&s_full[t]);
            ++cnt[t];
          }
        }
        if (!ok) break;
        if (hs < nhmax && (hf == 1 || hs == nhmax - 1)) mma_commit(&k_empty[s]);
        if (hs >= 1 && (hp == 1 || hs - 1 == nhmax - 1)) mma_commit(&v_empty[sp]);
      }
      mma_commit(mma_done);
      drain_wait(mma_done, 0, ctl);
    }
    if (!kHalf && lane == 0 && npos > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);  // S = Q K^T, both K-major
      constexpr uint32_t idO = idesc_bf16(128, D, false, true);     // O += P V, V is MN-major
      bool ok = mbar_wait(q_full, 0, ctl);
      int cnt[2] = {0, 0};     // S MMAs issued per query tile
      uint32_t use_prev = 0;   // bit t: query tile t used the previous position
      for (int j = 0; ok && j <= npos; ++j) {
        const int s = j % S;
        const int sp = (j + S - 1) % S;
        uint32_t use = 0;  // bit t: query tile t uses position j
        if (j < npos) {
          if constexpr (kSparse) {
            const int e = __ldg(f_list + j);
            const int kt = e >> 2;
            use = (((e & 1) && kt < nb[0]) ? 1u : 0u) | (((e & 2) && kt < nb[1]) ? 2u : 0u);
          } else {
            use = (j < nb[0] ? 1u : 0u) | (j < nb[1] ? 2u : 0u);
          }
        }
        if (j < npos && !(ok = mbar_wait(&k_full[s], (j / S) & 1, ctl))) break;
        if (j >= 1 && !(ok = mbar_wait(&v_full[sp], ((j - 1) / S) & 1, ctl))) break;
        tc_fence_after();
        const uint32_t qbs0 = sbase + L::kQ;
        const uint32_t kbs = sbase + L::kK + s * L::kTile;
        auto issue_S = [&](int t) {  // S_t = Q_t K_j^T, all D / 16 K-steps in one chain
          mma_ss_kmajor<D>(tmem + L::kColS0 + 128 * t,
                           sdesc_sw128(qbs0 + t * L::kTile, 16384, 1024),
                           sdesc_sw128(kbs, 16384, 1024), idS, 0u);
          mma_commit(&s_full[t]);
          ++cnt[t];
        };
        // Block-sparse: S of a tile that starts a use here with no P V pending needs no softmax
        // result, so it goes first and the other tile's softmax overlaps it.  (In the dense
        // stream every position after the first continues both tiles: the plain order below.)
        if constexpr (kSparse) {
#pragma unroll
          for (int t = 0; t < 2; ++t)
            if (((use >> t) & 1u) && !((use_prev >> t) & 1u)) issue_S(t);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if ((use_prev >> t) & 1u) {
            if (!(ok = mbar_wait(&p_full[t], (cnt[t] - 1) & 1, ctl))) break;
            tc_fence_after();
            // O_t += P_t V: 128 keys, 16 per MMA, P packed 2 per column, V rows +2 KB per step
            mma_ts_k128_step8(tmem + L::kColO0 + D * t, tmem + L::kColS0 + 128 * t,
                              sdesc_sw128(sbase + L::kV + sp * L::kTile, 16384, 1024), idO,
                              cnt[t] > 1 ? 1u : 0u);
            if (cnt[t] == ncnt[t]) mma_commit(&o_full[t]);  // the tile's last P V
          }
          // S_t overwrites P_t: after the tile's own P V
          if (((use >> t) & 1u) && (!kSparse || ((use_prev >> t) & 1u))) issue_S(t);
        }
        if (!ok) break;
        if (j < npos) mma_commit(&k_empty[s]);
        if (j >= 1) mma_commit(&v_empty[sp]);
        use_prev = use;
      }
      // every MMA issued by this thread has finished before tensor memory is released
      mma_commit(mma_done);
      drain_wait(mma_done, 0, ctl);
    }
  } else if (warp >= (kHalf ? 2u : 4u)) {
    // ================= softmax warpgroups: one per query tile, one thread per query row
    const int t = (warp - (kHalf ? 2 : 4)) >> 2;
    const uint32_t quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qt0 = q0 + 128 * t;
    const int qi = qt0 + row;
    const uint32_t lanes = (quad * 32u) << 16;
    const uint32_t tS = tmem + lanes + L::kColS0 + L::kSCols * t;
    const uint32_t tO = tmem + lanes + L::kColO0 + D * t;
    const float c2 = a.scale_log2;
    const int n = kHalf ? nh[t] : ncnt[t];
    int kt_next = (kSparse && n > 0) ? __ldg(r_list[t]) : 0;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s (log2 units)
    float l_run = 0.f;        // running sum of exp2(. - m_run)
    float lr_run = 0.f;       // the same sum over the bf16-rounded values (normalises O~)
    bool ok = true;
    if constexpr (kHalf) {
      // one 64-key half step per S: the same online softmax over 64 scores per row (a loop of
      // its own, so that the 128-key loop below, which the d = 128 kernels run, is untouched)
      for (int j = 0; j < n; ++j) {
        if (!(ok = mbar_wait_warp(&s_full[t], j & 1, ctl))) break;
        tc_fence_after();
        uint32_t s[64];
        tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_ld();
        reg_fence(s);
        const int k0 = j * 64;
        const bool masked = (k0 + 64 > kv_len) || (a.causal && k0 + 64 > qt0);
        const int klim = a.causal ? min(kv_len, qi + 1) : kv_len;  // keys < klim are visible
        float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (masked) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (k0 + c < klim) mxv[c & 3] = fmaxf(mxv[c & 3], __uint_as_float(s[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 8) {
            mxv[0] = max3(mxv[0], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            mxv[1] = max3(mxv[1], __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
            mxv[2] = max3(mxv[2], __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
            mxv[3] = max3(mxv[3], __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
          }
        }
        const float mx = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3]));
        const float m_tile = mx * c2;
        float alpha = 1.f;
        bool rescale = false;
        if (m_tile > m_run + kRescaleThreshold) {
          rescale = true;
          alpha = ex2(m_run - m_tile);  // 0 on the first step (m_run = -inf)
          l_run *= alpha;
          lr_run *= alpha;
          m_run = m_tile;
        }
        const float2 cc = make_float2(c2, c2);
        const float2 nm = make_float2(-m_run, -m_run);
        float2 sumv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float sum_r = 0.f;
        uint32_t p[32];
        if (masked) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = fma2(
                make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), cc, nm);
            const float x0 = (k0 + 2 * c < klim) ? ex2(x.x) : 0.f;
            const float x1 = (k0 + 2 * c + 1 < klim) ? ex2(x.y) : 0.f;
            p[c] = pack_bf16(x0, x1);
            sumv[c & 1] = add2(sumv[c & 1], make_float2(x0, x1));
            if (FA_ROUNDED_SUM) sum_r += bf16_lo(p[c]) + bf16_hi(p[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = fma2(
                make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), cc, nm);
            float x0, x1;
            if (FA_SOFT_EXP2 > 0 && c % (FA_SOFT_EXP2 > 0 ? FA_SOFT_EXP2 : 1) == FA_SOFT_EXP2 - 1) {
              const float2 e = exp2_poly2(x);
              x0 = e.x;
              x1 = e.y;
            } else {
              x0 = ex2(x.x);
              x1 = ex2(x.y);
            }
            p[c] = pack_bf16(x0, x1);
            sumv[c & 1] = add2(sumv[c & 1], make_float2(x0, x1));
            if (FA_ROUNDED_SUM) sum_r += bf16_lo(p[c]) + bf16_hi(p[c]);
          }
        }
        l_run += (sumv[0].x + sumv[1].x) + (sumv[0].y + sumv[1].y);
        lr_run += sum_r;
        tmem_st32(tS + 0, p);  // P over the first 32 columns of this tile's S
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
            reg_fence(o);
            const float2 aa = make_float2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 v = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])),
                                    aa);
              o[e] = __float_as_uint(v.x);
              o[e + 1] = __float_as_uint(v.y);
            }
            tmem_st32(tO + 32 * c, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
    }
    for (int j = 0; !kHalf && j < n; ++j) {
      const int kt = kSparse ? kt_next : j;  // key tile of this query tile's j-th S
      if (kSparse && j + 1 < n) kt_next = __ldg(r_list[t] + j + 1);
      if (!(ok = mbar_wait_warp(&s_full[t], j & 1, ctl))) break;
      tc_fence_after();
      uint32_t s[128];
      tmem_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
      tmem_wait_ld();
      reg_fence(s);
      const int k0 = kt * 128;
      const bool masked = (k0 + 128 > kv_len) || (a.causal && k0 == qt0);
      const int klim = a.causal ? min(kv_len, qi + 1) : kv_len;  // keys < klim are visible
      // row max: 3-input max over 4 independent chains (a single chain is 128 dependent steps)
      float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (k0 + c < klim) mxv[c & 3] = fmaxf(mxv[c & 3], __uint_as_float(s[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mxv[0] = max3(mxv[0], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
          mxv[1] = max3(mxv[1], __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
          mxv[2] = max3(mxv[2], __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
          mxv[3] = max3(mxv[3], __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
        }
      }
      const float mx = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3]));
      const float m_tile = mx * c2;
      float alpha = 1.f;
      bool rescale = false;
      if (m_tile > m_run + kRescaleThreshold) {
        rescale = true;
        alpha = ex2(m_run - m_tile);  // 0 on the first tile (m_run = -inf)
        l_run *= alpha;
        lr_run *= alpha;
        m_run = m_tile;
      }
      // p = exp2(s * c2 - m) on pairs: one packed FMA, two MUFU ex2, one pack, one packed add
      const float2 cc = make_float2(c2, c2);
      const float2 nm = make_float2(-m_run, -m_run);
      float2 sumv[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      float sum_r = 0.f;
      uint32_t p[64];
      if (masked) {  // diagonal or key-padding tile (separate loop: no per-element branch)
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = fma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                cc, nm);
          const float x0 = (k0 + 2 * c < klim) ? ex2(x.x) : 0.f;
          const float x1 = (k0 + 2 * c + 1 < klim) ? ex2(x.y) : 0.f;
          p[c] = pack_bf16(x0, x1);
          sumv[c & 1] = add2(sumv[c & 1], make_float2(x0, x1));
          if (FA_ROUNDED_SUM) sum_r += bf16_lo(p[c]) + bf16_hi(p[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float2 x = fma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                cc, nm);
          float x0, x1;
          if (FA_SOFT_EXP2 > 0 && c % (FA_SOFT_EXP2 > 0 ? FA_SOFT_EXP2 : 1) == FA_SOFT_EXP2 - 1) {
            const float2 e = exp2_poly2(x);
            x0 = e.x;
            x1 = e.y;
          } else {
            x0 = ex2(x.x);
            x1 = ex2(x.y);
          }
          p[c] = pack_bf16(x0, x1);
          sumv[c & 1] = add2(sumv[c & 1], make_float2(x0, x1));
          if (FA_ROUNDED_SUM) sum_r += bf16_lo(p[c]) + bf16_hi(p[c]);
        }
      }
      const float sum = (sumv[0].x + sumv[1].x) + (sumv[0].y + sumv[1].y);
      l_run += sum;
      lr_run += sum_r;
      // P over the first 64 columns of S (the MMA issuer reads it as the A operand)
      tmem_st32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
      // O~ *= alpha for rows whose max moved (the previous P V has completed: it was issued
      // before the S MMA whose completion this warp just observed)
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          reg_fence(o);
          const float2 aa = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v = mul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), aa);
            o[e] = __float_as_uint(v.x);
            o[e + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }

    // ---- epilogue: O = O~ / l -> bf16 -> swizzled smem over Q_t -> TMA store; LSE
    const bool tile_live = (qt0 < N);
    // variable-length: a tile that runs past its sequence's end would have the TMA store write
    // into the next sequence, so its rows are stored one by one
    const bool direct = kVarlen && (qt0 + 128 > N);
    if (ok && n > 0) ok = mbar_wait_warp(&o_full[t], 0, ctl);
    // block-sparse: a tile with no kept key tile still had its Q copied in (for the other tile's
    // sake); that copy must land before the staging below reuses its shared memory
    if (kSparse && ok && n == 0 && npos > 0) ok = mbar_wait_warp(q_full, 0, ctl);
    if (tile_live) {  // uniform over the warpgroup
      if (ok) {
        tc_fence_after();
        const float l_o = FA_ROUNDED_SUM ? lr_run : l_run;
        const float inv_l = (l_o > 0.f) ? 1.f / l_o : 0.f;
        const uint32_t stage = sbase + L::kQ + t * L::kTile;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (n > 0) {
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
            reg_fence(o);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv_l,
                              __uint_as_float(o[2 * e + 1]) * inv_l);
          if (direct) {
            if (qi < N) {
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<__nv_bfloat16*>(a.o) +
                  (static_cast<size_t>(seq_start + qi) * a.H + h) * D + 32 * c);
#pragma unroll
              for (int g = 0; g < 4; ++g)
                dst[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else {
            const uint32_t panel = stage + ((32 * c) / 64) * 16384;
            const uint32_t g0 = ((32 * c) % 64) / 8;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              st_shared_v4(panel + sw128_offset(row, g0 + g), pk[4 * g], pk[4 * g + 1],
                           pk[4 * g + 2], pk[4 * g + 3]);
          }
        }
        if (qi < N) {
          const float lse = (l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
          const size_t at = kVarlen ? static_cast<size_t>(h) * a.total + seq_start + qi
                                    : static_cast<size_t>(bh) * N + qi;
          a.lse[at] = lse;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + t, 128);  // every warp of the group arrives, aborted or not
      if (!direct && quad == 0 && lane == 0 && !*abort_flag) {
        for (int c = 0; c < D / 64; ++c)
          tma_store_3d(&tmO, sm + L::kQ + t * L::kTile + c * 16384, c * 64, row_y(q_y0, qt0),
                       row_z(q_z0, qt0));
        bulk_commit();
        bulk_wait_read0();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool kSparse, bool kVarlen>
cudaError_t launch_fwd_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, FwdArgs a, cudaStream_t st) {
  using L = FwdLayout<D, kHalfSteps<D, kSparse, kVarlen>>;
  const uint32_t smem = L::kBytes + 1024;
  cudaError_t e = ensure_smem_limit<fwd_kernel<D, kSparse, kVarlen>>(smem);
  if (e != cudaSuccess) return e;
  a.smem_bytes = smem;
  const unsigned grid = static_cast<unsigned>(a.num_qblocks) * static_cast<unsigned>(a.BH);
  fwd_kernel<D, kSparse, kVarlen><<<grid, kFwdThreads<D, kSparse, kVarlen>, smem, st>>>(tq, tk,
                                                                                       tv, to, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& a, cudaStream_t s) {
  if (a.cu_seqlens != nullptr) {  // variable-length (not combined with a block mask)
    if (d == 64) return launch_fwd_d<64, false, true>(tq, tk, tv, to, a, s);
    return launch_fwd_d<128, false, true>(tq, tk, tv, to, a, s);
  }
  if (a.blk != nullptr) {
    if (d == 64) return launch_fwd_d<64, true, false>(tq, tk, tv, to, a, s);
    return launch_fwd_d<128, true, false>(tq, tk, tv, to, a, s);
  }
  if (d == 64) return launch_fwd_d<64, false, false>(tq, tk, tv, to, a, s);
  return launch_fwd_d<128, false, false>(tq, tk, tv, to, a, s);
}

}  // namespace fa
