// Deterministic dQ: one CTA per (b, h, 128-query tile i) accumulates
//   dQ_i = scale * sum_j dS_ij K_j,   dS_ij = P_ij o (dO_i V_j^T - D_i),  P_ij = exp(S_ij - LSE_i)
// over the key tiles j in a fixed order, entirely in tensor memory, and writes it once.  With the
// dK / dV kernel (which accumulates per key tile in tensor memory as well) this gives a backward
// pass whose results do not depend on the order of atomic additions: the deterministic option the
// pages describe for the official repository (page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知
// 注意力", section "反向传播：用重计算代替存储": deterministic=True is slower and uses more
// memory).  The price is recomputing S_ij and dP_ij once more (3 extra GEMM-steps of 5 per tile
// pair instead of the atomics).
//
// Roles (384 threads): warp 0 TMA producer (Q_i and dO_i once, K_j and V_j through 2 stages),
// warp 1 the MMA issuer, warps 2-3 idle, warps 4-7 / 8-11 two warpgroups, one thread per query
// row, each owning 64 of the 128 keys of a tile:
//   S = Q_i K_j^T      (smem x smem)       -> tensor memory [0, 128)
//   P = exp2(S * scale * log2 e - LSE_i * log2 e), masked, kept in registers as bf16 pairs
//   dP = dO_i V_j^T    (smem x smem)       -> tensor memory, two buffers [128, 256), [256, 384)
//   dS = P o (dP - D_i), packed bf16 over the group's own dP columns
//   dQ += dS K_j       (A = dS from tensor memory, B = K_j MN-major) -> [384, 384 + D)
// Block-sparse (kSparse): the key tiles are the query tile's kept ones (an ascending list from the
// block index, cut at the causal / key-length limit).
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

namespace {

template <int D>
struct DqLayout {
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kDO = kQ + kTile;
  static constexpr uint32_t kK = kDO + kTile;       // 2 stages
  static constexpr uint32_t kV = kK + 2 * kTile;    // 2 stages
  static constexpr uint32_t kBar = kV + 2 * kTile;
  // qdo_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_read, dp_full[2],
  // ds_full[2], dq_full, mma_done
  static constexpr int kNumBars = 17;
  static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kCnt = kAbort + 4;  // block-sparse: key tiles to visit
  static constexpr uint32_t kBytes = kCnt + 4;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;
  static constexpr uint32_t kTmemCols = 512;
};


template <int D, bool kSparse, bool kVarlen>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using L = DqLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* sm = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* qdo_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 9;
  uint64_t* s_read = bars + 10;
  uint64_t* dp_full = bars + 11;
  uint64_t* ds_full = bars + 13;
  uint64_t* dq_full = bars + 15;
  uint64_t* mma_done = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const Ctl ctl{abort_flag, a.status, a.timeout_ns};

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  if (pad + L::kBytes > a.smem_bytes) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kErrLayout);
    return;
  }

  // ---- work item: query tile i of (b, h); causal: the tiles with most key tiles first
  const int nqt_grid = a.num_qtiles;
  const int lin = blockIdx.x;
  const int bh = lin % a.BH;
  const int i = a.causal ? (nqt_grid - 1 - lin / a.BH) : (lin / a.BH);
  const int b = bh / a.H;
  const int h = bh - b * a.H;
  const int hk = h / (a.H / a.Hkv);
  int seq_start = 0, N = a.N;
  if constexpr (kVarlen) seq_bounds(a.cu_seqlens, b, a.total, seq_start, N);
  if (kVarlen && i * 128 >= N) return;  // past this sequence's end (uniform over the CTA)
  const int nqt = kVarlen ? (N + 127) / 128 : nqt_grid;
  int kv_len = N;
  if (!kVarlen && a.kv_lens != nullptr) kv_len = min(max(__ldg(a.kv_lens + b), 0), N);
  int nkeys = kv_len;
  if (a.causal) nkeys = min(nkeys, i * 128 + 128);
  // TMA box coordinates (y, z): dense (row, head slice), packed (head, token)
  const int q_y = kVarlen ? h : i * 128, q_z = kVarlen ? seq_start + i * 128 : bh;
  auto kv_y = [&](int kt) { return kVarlen ? hk : kt * 128; };
  auto kv_z = [&](int kt) { return kVarlen ? seq_start + kt * 128 : b * a.Hkv + hk; };
  // workspace row of query row qi
  const size_t ws_row0 =
      (kVarlen ? (static_cast<size_t>(h) * a.ws_tiles + seq_tile0(seq_start, b) + i)
               : (static_cast<size_t>(bh) * a.ws_tiles + i)) * 128;
  const int nb_dense = (nkeys + 127) / 128;  // key tiles 0 .. nb_dense-1 are visible
  const int32_t* r_list = nullptr;
  int* cnt_smem = reinterpret_cast<int*>(sm + L::kCnt);
  if constexpr (kSparse) {
    const BlockIndex BI = block_index_layout(nqt);
    const int32_t* base = a.blk + (a.blk_heads == 1 ? 0 : static_cast<int64_t>(bh % a.H) * BI.words);
    r_list = base + BI.ridx + static_cast<int64_t>(i) * nqt;
    if (warp == 2) {
      const int c = warp_count_below(r_list, __ldg(base + BI.rcnt + i), nb_dense);
      if (lane == 0) *cnt_smem = c;
    }
  }
  auto ktile = [&](int jj) { return kSparse ? __ldg(r_list + jj) : jj; };

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int k = 0; k < L::kNumBars; ++k) {
      const bool per_warp = (&bars[k] == s_read) || (&bars[k] == ds_full) || (&bars[k] == ds_full + 1);
      mbar_init(&bars[k], per_warp ? 8 : 1);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdQ);
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
  const int nb = kSparse ? *cnt_smem : nb_dense;  // key tiles this query tile visits

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0 && nb > 0) {
      mbar_arrive_expect_tx(qdo_full, 2 * L::kTile);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sm + L::kQ + c * 16384, &tmQ, qdo_full, c * 64, q_y, q_z);
        tma_load_3d(sm + L::kDO + c * 16384, &tmdO, qdo_full, c * 64, q_y, q_z);
      }
      int nk = 0, nv = 0;
      for (int jj = 0; jj < nb; ++jj) {
        const int s = jj & 1;
        const uint32_t ph = (jj >> 1) & 1;
        const int kt = ktile(jj);
        if (!mbar_wait(&k_empty[s], ph ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&k_full[s], L::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm + L::kK + s * L::kTile + c * 16384, &tmK, &k_full[s], c * 64, kv_y(kt),
                      kv_z(kt));
        nk = jj + 1;
        if (!mbar_wait(&v_empty[s], ph ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&v_full[s], L::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm + L::kV + s * L::kTile + c * 16384, &tmV, &v_full[s], c * 64, kv_y(kt),
                      kv_z(kt));
        nv = jj + 1;
      }
      // no copy may still be in flight when the CTA exits, aborted or not
      drain_wait(qdo_full, 0, ctl);
      for (int jj = max(0, nk - 2); jj < nk; ++jj) drain_wait(&k_full[jj & 1], (jj >> 1) & 1, ctl);
      for (int jj = max(0, nv - 2); jj < nv; ++jj) drain_wait(&v_full[jj & 1], (jj >> 1) & 1, ctl);
    }
  } else if (warp == 1) {
    // ================= MMA issuer: S(0), dP(0), then per key tile j:
    //   S(j+1) (once S(j) was read), dP(j+1) (other dP buffer), dQ += dS(j) K_j
    if (lane == 0 && nb > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);  // S, dP: K-major operands
      constexpr uint32_t idQ = idesc_bf16(128, D, false, true);     // dQ: A = dS in TMEM, B = K MN-major
      const uint64_t desc_q = sdesc_sw128(sbase + L::kQ, 16384, 1024);
      const uint64_t desc_do = sdesc_sw128(sbase + L::kDO, 16384, 1024);
      auto desc_k = [&](int jj) { return sdesc_sw128(sbase + L::kK + (jj & 1) * L::kTile, 16384, 1024); };
      auto desc_v = [&](int jj) { return sdesc_sw128(sbase + L::kV + (jj & 1) * L::kTile, 16384, 1024); };
      auto issue_S = [&](int jj) {  // S = Q_i K_j^T (one chain of K-steps, sm103.cuh)
        mma_ss_kmajor<D>(tmem + L::kColS, desc_q, desc_k(jj), idS, 0u);
        mma_commit(s_full);
      };
      auto issue_dP = [&](int jj) {  // dP = dO_i V_j^T into buffer jj % 2
        mma_ss_kmajor<D>(tmem + L::kColDP + 128 * (jj & 1), desc_do, desc_v(jj), idS, 0u);
        mma_commit(&dp_full[jj & 1]);
        mma_commit(&v_empty[jj & 1]);
      };
      auto issue_dQ = [&](int jj) {  // dQ += dS_j K_j  (128 keys, 16 per MMA; dS halves split)
        mma_ts_k128_split(tmem + L::kColDQ, tmem + L::kColDP + 128 * (jj & 1), desc_k(jj), idQ,
                          jj > 0 ? 1u : 0u);
        mma_commit(&k_empty[jj & 1]);
      };
      auto wait_k = [&](int jj) { return mbar_wait(&k_full[jj & 1], (jj >> 1) & 1, ctl); };
      auto wait_v = [&](int jj) { return mbar_wait(&v_full[jj & 1], (jj >> 1) & 1, ctl); };

      bool ok = mbar_wait(qdo_full, 0, ctl) && wait_k(0);
      if (ok) {
        tc_fence_after();
        issue_S(0);
        ok = wait_v(0);
      }
      if (ok) {
        tc_fence_after();
        issue_dP(0);
      }
      for (int jj = 0; ok && jj < nb; ++jj) {
        if (jj + 1 < nb) {
          if (!(ok = mbar_wait(s_read, jj & 1, ctl) && wait_k(jj + 1))) break;
          tc_fence_after();
          issue_S(jj + 1);
          if (!(ok = wait_v(jj + 1))) break;
          tc_fence_after();
          issue_dP(jj + 1);
        }
        if (!(ok = mbar_wait(&ds_full[jj & 1], (jj >> 1) & 1, ctl))) break;
        tc_fence_after();
        issue_dQ(jj);
      }
      if (ok) mma_commit(dq_full);
      mma_commit(mma_done);
      drain_wait(mma_done, 0, ctl);
    }
  } else if (warp >= 4) {
    // ================= P and dS: one thread per query row, one warpgroup per 64 keys
    const uint32_t quad = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int r = quad * 32 + lane;
    const int qi = i * 128 + r;
    const uint32_t lanes = (quad * 32u) << 16;
    const uint32_t tS = tmem + lanes + L::kColS + 64 * grp;
    const float c2 = a.scale_log2;
    const size_t srow = ws_row0 + r;  // padded rows of the tile hold -inf / 0
    const float nl2 = a.neg_lse2[srow];   // -LSE * log2(e) (-inf on padded rows: P = 0)
    const float ndl = a.neg_delta[srow];  // -D
    const float2 cc = make_float2(c2, c2);
    const float2 nl = make_float2(nl2, nl2);
    const float2 nd = make_float2(ndl, ndl);
    bool ok = true;
    for (int jj = 0; jj < nb; ++jj) {
      const int kt = ktile(jj);
      if (!(ok = mbar_wait_warp(s_full, jj & 1, ctl))) break;
      tc_fence_after();
      const int k0 = kt * 128 + 64 * grp;  // first key of this group's columns
      // keys >= klim are masked (causal: key > query; padding: key >= kv_len)
      const int klim = a.causal ? min(kv_len, qi + 1) : kv_len;
      // element masks only where some row of the warp needs them (the causal diagonal, the
      // key-length tail); the test is uniform over the warp, so the loop is chosen once
      const bool masked = __any_sync(0xffffffffu, k0 + 64 > klim);
      uint32_t p[32];
      auto p_from_s = [&](auto kMask) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t sv[32];
          tmem_ld32(tS + 32 * c, sv);
          tmem_wait_ld();
          reg_fence(sv);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 y = fma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                                  cc, nl);
            float x0 = ex2(y.x), x1 = ex2(y.y);
            if constexpr (decltype(kMask)::value) {
              const int kk = k0 + 32 * c + 2 * e;
              x0 = (kk < klim) ? x0 : 0.f;
              x1 = (kk + 1 < klim) ? x1 : 0.f;
            }
            p[16 * c + e] = pack_bf16(x0, x1);
          }
        }
      };
      if (masked) p_from_s(std::true_type{});
      else p_from_s(std::false_type{});
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_read);  // S(j) fully read: S(j+1) may overwrite it

      if (!(ok = mbar_wait_warp(&dp_full[jj & 1], (jj >> 1) & 1, ctl))) break;
      tc_fence_after();
      const uint32_t tDP = tmem + lanes + L::kColDP + 128 * (jj & 1) + 64 * grp;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dv[32];
        tmem_ld32(tDP + 32 * c, dv);
        tmem_wait_ld();
        reg_fence(dv);
        uint32_t ds[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t pe = p[16 * c + e];
          const float2 t = add2(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd);
          const float2 u = mul2(make_float2(bf16_lo(pe), bf16_hi(pe)), t);
          ds[e] = pack_bf16(u.x, u.y);
        }
        tmem_st16(tDP + 16 * c, ds);  // over dP columns this group has already read
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[jj & 1]);
    }

    // ---- epilogue: dQ * scale -> bf16 -> swizzled smem over Q_i -> TMA store (rows >= N are
    // clipped).  d = 128: one 64-column panel per group; d = 64: the first group alone.
    if (ok && nb > 0) ok = mbar_wait_warp(dq_full, 0, ctl);
    const bool writer = (D == 128) || grp == 0;
    // variable-length: a tile that runs past its sequence's end is stored row by row
    const bool direct = kVarlen && (i * 128 + 128 > N);
    if (writer) {
      const int c0 = (D == 128) ? 64 * grp : 0;  // first dQ column of this group
      if (ok) {
        if (nb > 0) tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          if (nb > 0) {
            tmem_ld32(tmem + lanes + L::kColDQ + c0 + 32 * c, v);
            tmem_wait_ld();
            reg_fence(v);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale);
          if (direct) {
            if (qi < N) {
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<__nv_bfloat16*>(a.dq) +
                  (static_cast<size_t>(seq_start + qi) * a.H + h) * D + c0 + 32 * c);
#pragma unroll
              for (int g = 0; g < 4; ++g)
                dst[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else {
            const uint32_t panel = sbase + L::kQ + (c0 / 64) * 16384;
#pragma unroll
            for (int g = 0; g < 4; ++g)
              st_shared_v4(panel + sw128_offset(r, 4 * c + g), pk[4 * g], pk[4 * g + 1],
                           pk[4 * g + 2], pk[4 * g + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + grp, 128);  // every warp of the group arrives, aborted or not
      if (!direct && quad == 0 && lane == 0 && !*abort_flag) {
        tma_store_3d(&tmdQ, sm + L::kQ + (c0 / 64) * 16384, c0, q_y, q_z);
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
cudaError_t launch_dq_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const CUtensorMap& tdq, BwdArgs a,
                        cudaStream_t st) {
  using L = DqLayout<D>;
  // The kernel allocates all 512 tensor-memory columns, so a second resident CTA would only sit in
  // tcgen05.alloc: ask for enough shared memory (d = 64 needs less than half an SM's) that one
  // CTA fills the SM.
  const uint32_t smem = L::kBytes + 1024 < 120u * 1024u ? 120u * 1024u : L::kBytes + 1024;
  cudaError_t e = ensure_smem_limit<bwd_dq_kernel<D, kSparse, kVarlen>>(smem);
  if (e != cudaSuccess) return e;
  a.smem_bytes = smem;
  const unsigned grid = static_cast<unsigned>(a.num_qtiles) * static_cast<unsigned>(a.BH);
  bwd_dq_kernel<D, kSparse, kVarlen><<<grid, 384, smem, st>>>(tq, tk, tv, tdo, tdq, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& a, cudaStream_t s) {
  if (a.cu_seqlens != nullptr) {
    if (d == 64) return launch_dq_d<64, false, true>(tq, tk, tv, tdo, tdq, a, s);
    return launch_dq_d<128, false, true>(tq, tk, tv, tdo, tdq, a, s);
  }
  if (a.blk != nullptr) {
    if (d == 64) return launch_dq_d<64, true, false>(tq, tk, tv, tdo, tdq, a, s);
    return launch_dq_d<128, true, false>(tq, tk, tv, tdo, tdq, a, s);
  }
  if (d == 64) return launch_dq_d<64, false, false>(tq, tk, tv, tdo, tdq, a, s);
  return launch_dq_d<128, false, false>(tq, tk, tv, tdo, tdq, a, s);
}

}  // namespace fa
