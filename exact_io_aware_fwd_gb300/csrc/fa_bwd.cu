// Backward pass kernels.
//
// Method (page "FlashAttention：不减少一次注意力计算，为什么反而更快", section 关键设计三):
// the forward pass saved only O and the per-row log-sum-exp; the backward pass recomputes each
// score tile S_ij = Q_i K_j^T and P_ij = exp(S_ij - LSE_i) on chip, and uses
//   D_i = dO_i . O_i,  dP = dO V^T,  dS = P o (dP - D),
//   dV_j += P_ij^T dO_i,  dK_j += dS_ij^T Q_i,  dQ_i += dS_ij K_j
// (with the softmax scale applied to dK and dQ by the chain rule through S = scale * Q K^T).
//
// Kernels:
//  bwd_preprocess  -D = -rowsum(dO o O) and -LSE * log2(e) into the workspace (negated so that
//                  P and dP - D are single packed FMA / add instructions; padded rows get 0 and
//                  -inf, which makes their recomputed P exactly 0), and resets the record of
//                  every query tile of fa_bwd's dQ accumulation.
//  bwd_dkdv        one CTA per (b, h, 128-key tile j); dK_j and dV_j accumulate in tensor memory
//                  over the query tiles i (causal: i >= j only).  Warps: TMA producer, MMA
//                  issuer, the dQ claim warp, one idle, and kGroups warpgroups that each handle
//                  128 / kGroups of the 128 query columns of every key row for P and dS, drain
//                  their share of dQ_{i-1} between P_i and dS_i (while dP_i runs), and write
//                  their share of the dV and dK panels at the end.  Per query tile:
//                    S^T = K_j Q_i^T and dP^T = V_j dO_i^T   (tcgen05, both operands in smem)
//                    P^T = exp2(S^T * scale * log2 e - LSE_i * log2 e), written back over S^T
//                    dS^T = P^T o (dP^T - D_i), written back over dP^T and to smem
//                    dV += P^T dO_i, dK += dS^T Q_i          (A operand read from tensor memory)
//                    dQ_i = dS K_j                            (A = dS from smem, MN-major)
//  bwd_dq_convert  dQ = bf16(scale * accumulator), or 0 for a query tile nobody claimed.
//
// dQ across key tiles.  dQ_i = sum_j dS_ij K_j gets one partial per key tile j that visits query
// tile i, from different CTAs in no fixed order.  The partials meet in a float32 accumulator in
// the workspace, which is never zeroed:
//   * the first key tile to claim the query tile (an atomic increment of the tile's record,
//     made about a tile period before its partial is drained) stores its partial, in whole
//     128-byte lines, so the accumulator's lines need no read from device memory;
//   * every other one adds its partial with vector reductions (red.global.add.v4.f32) once the
//     record shows that the first one's stores are visible.
// The additions make dQ non-deterministic in the last bits, as the pages note for the default
// backward (page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section
// "反向传播：用重计算代替存储"); dK and dV are accumulated in a fixed order.  Without a causal mask
// key tile j visits the query tiles starting at tile j (j, j + 1, ..., wrapping around), so that
// the claims of a query tile arrive a tile period apart, as they do under the causal order.
//
// dQ accumulator layout ("tile-major"): for (b, h), query tile i, column group g (4 floats)
// and row r of the tile, element (r, 4g + e) is at float index
//   (((bh * num_qtiles + i) * (d / 4) + g) * 128 + r) * 4 + e,
// so that 32 consecutive rows of one column group are 512 contiguous bytes and a warp's
// vector reduction (or store) covers four whole 128-byte lines.
#include <type_traits>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

Workspace workspace_layout(int BH, int N, int d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t npad = static_cast<size_t>((N + kTileRows - 1) / kTileRows) * kTileRows;
  Workspace w;
  w.dq_acc_off = 0;
  w.neg_lse2_off = up(static_cast<size_t>(BH) * npad * d * sizeof(float));
  w.neg_delta_off = w.neg_lse2_off + up(static_cast<size_t>(BH) * npad * sizeof(float));
  w.dq_cnt_off = w.neg_delta_off + up(static_cast<size_t>(BH) * npad * sizeof(float));
  w.total = w.dq_cnt_off + up(static_cast<size_t>(BH) * (npad / kTileRows) * sizeof(DqTileCount));
  return w;
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Row geometry of the preprocess and dQ-conversion kernels.  Dense: block (i, bh) is query tile i
// of head slice bh of [B*H, N, d].  Variable-length: block (i, b*H + h) is tile i of sequence b,
// head h of the packed [total, H, d] tensors, whose workspace tile is h * ws_tiles + tile0 + i.
struct RowGeo {
  const int32_t* cu;  // token offsets [B + 1] (variable-length only)
  int H, total, ws_tiles;
};

template <bool kVarlen>
struct TileRows {
  int n;                // rows of this sequence (dense: N)
  size_t ws_tile;       // workspace tile (stats rows ws_tile * 128 + r, dQ accumulator tile)
  size_t tok0;          // dense: bh * N; variable-length: first token of the sequence
  int heads, h;         // variable-length: row stride in heads and this head
  __device__ TileRows(int i, int bh, int N, int nqt, const RowGeo& g) {
    if constexpr (kVarlen) {
      const int b = bh / g.H;
      h = bh - b * g.H;
      heads = g.H;
      int start;
      seq_bounds(g.cu, b, g.total, start, n);
      tok0 = static_cast<size_t>(start);
      ws_tile = static_cast<size_t>(h) * g.ws_tiles + seq_tile0(start, b) + i;
    } else {
      n = N;
      h = 0;
      heads = 1;
      tok0 = static_cast<size_t>(bh) * N;
      ws_tile = static_cast<size_t>(bh) * nqt + i;
    }
  }
  __device__ size_t row(int q) const {  // element offset / D of row q ([.., d] rows)
    return kVarlen ? (tok0 + q) * heads + h : tok0 + q;
  }
  __device__ size_t lse(int q, int total) const {  // LSE index of row q
    return kVarlen ? static_cast<size_t>(h) * total + tok0 + q : tok0 + q;
  }
};

// ------------------------------------------------------------------------------------------
// Preprocess: one block per (head slice, query tile), tph tiles per head slice, query tile
// fastest (a 1-D grid: B*H may exceed the 65,535 limit of a grid's y dimension); 256 threads.
template <int D, bool kVarlen>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ O,
                                                             const __nv_bfloat16* __restrict__ dO,
                                                             const float* __restrict__ lse, int N,
                                                             int nqt, float* __restrict__ neg_lse2,
                                                             float* __restrict__ neg_delta,
                                                             DqTileCount* __restrict__ recs,
                                                             int tph, RowGeo geo) {
  constexpr int G = D / 8;     // lanes per row (8 bf16 = 16 bytes each)
  constexpr int RPW = 32 / G;  // rows per warp per pass
  const int i = static_cast<int>(blockIdx.x % tph);
  const TileRows<kVarlen> tr(i, static_cast<int>(blockIdx.x / tph), N, nqt, geo);
  if (kVarlen && i * 128 >= tr.n) return;  // past this sequence's end
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / G, cl = lane % G;
  for (int rr = warp * RPW + sub; rr < 128; rr += 8 * RPW) {
    const int q = i * 128 + rr;
    float acc = 0.f;
    if (q < tr.n) {
      const size_t off = tr.row(q) * D + cl * 8;
      const uint4 o = __ldg(reinterpret_cast<const uint4*>(O + off));
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(dO + off));
      const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc += bf16_lo(ov[e]) * bf16_lo(gv[e]) + bf16_hi(ov[e]) * bf16_hi(gv[e]);
    }
#pragma unroll
    for (int m = G / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (cl == 0) {
      const size_t idx = tr.ws_tile * 128 + rr;
      float l2 = INFINITY;
      if (q < tr.n) {
        const float l = __ldg(lse + tr.lse(q, geo.total));
        l2 = (l == -INFINITY) ? INFINITY : l * kLog2e;  // a row with no key: P must be 0
      }
      neg_lse2[idx] = -l2;
      neg_delta[idx] = (q < tr.n) ? -acc : 0.f;
    }
  }
  if (recs != nullptr && threadIdx.x == 0) recs[tr.ws_tile].word = 0ull;  // nobody claimed it yet
}

// ------------------------------------------------------------------------------------------
// dQ convert: the preprocess kernel's 1-D grid, 256 threads; thread = (row r, pair of column
// groups).  A tile that no key tile claimed has no partial in the accumulator: its dQ is 0.
template <int D, bool kVarlen>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                             const DqTileCount* __restrict__ recs,
                                                             __nv_bfloat16* __restrict__ dQ, int N,
                                                             int nqt, float scale, int tph,
                                                             RowGeo geo) {
  const int i = static_cast<int>(blockIdx.x % tph);
  const TileRows<kVarlen> tr(i, static_cast<int>(blockIdx.x / tph), N, nqt, geo);
  const int r = threadIdx.x & 127;
  const int q = i * 128 + r;
  if (q >= tr.n) return;
  const float* tile = acc + tr.ws_tile * 128 * D;
  // (the accumulator is read either way, so that its loads need not wait for the record's)
  const bool claimed = static_cast<uint32_t>(__ldg(&recs[tr.ws_tile].word)) != 0u;
  // 16 columns of row r per step: four 16-byte loads (a warp reads 32 consecutive rows of one
  // 4-column group, 512 contiguous bytes each), then the whole 32-byte sector of bf16 output
  // written by this thread (two 16-byte stores back to back), so no output sector is assembled
  // from the partial writes of two threads
  const float2 sc = make_float2(scale, scale);
  for (int ch = threadIdx.x >> 7; ch < D / 16; ch += 2) {
    float4 a[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      a[g] = __ldg(reinterpret_cast<const float4*>(tile + ((4 * ch + g) * 128 + r) * 4));
      if (!claimed) a[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    uint32_t w[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float2 lo = mul2(make_float2(a[g].x, a[g].y), sc);
      const float2 hi = mul2(make_float2(a[g].z, a[g].w), sc);
      w[2 * g] = pack_bf16(lo.x, lo.y);
      w[2 * g + 1] = pack_bf16(hi.x, hi.y);
    }
    uint4* dst = reinterpret_cast<uint4*>(dQ + tr.row(q) * D + ch * 16);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// ------------------------------------------------------------------------------------------
// dK / dV kernel
template <int D>
struct BwdLayout {
  static constexpr uint32_t kTile = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;       // 2 stages
  static constexpr uint32_t kDO = kQ + 2 * kTile;  // 2 stages
  static constexpr uint32_t kDS = kDO + 2 * kTile; // 128 keys x 128 queries bf16
  static constexpr uint32_t kLse = kDS + 32768;    // 2 stages x 128 floats
  static constexpr uint32_t kDelta = kLse + 1024;  // 2 stages x 128 floats
  // d = 64: two slots of one dQ partial (128 rows x D fp32, the accumulator tile's layout) that
  // the TMA unit adds into the accumulator (there is no room for them at d = 128)
  static constexpr bool kBulkDQ = (D == 64);
  static constexpr uint32_t kPart = 128u * D * 4u;
  static constexpr uint32_t kStage = kDelta + 1024;
  static constexpr uint32_t kBar = kStage + (kBulkDQ ? 2u * kPart : 0u);
  // kv_full, q_full[2], q_empty[2], do_full[2], do_empty[2], s_full, p_full, dp_full, ds_full,
  // dq_full, dq_empty, dkdv_full, mma_done, then the dQ claims' mode_full[2], mode_empty[2],
  // first_stored[2], then (d = 64) staged[2], stage_empty[2], the second dq_empty
  static constexpr int kNumBars = 28;
  static constexpr uint32_t kMode = kBar + kNumBars * 8;  // 2 slots: how a drain writes
  static constexpr uint32_t kKind = kMode + 8;            // 2 slots: the mode of a staged partial
  static constexpr uint32_t kTmemSlot = kKind + 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kBytes = kAbort + 4;
  // TMEM columns.  S^T (fp32) in [0, 128); P^T packed as bf16 pairs over the first half of each
  // 64-query half's own columns: queries 64h..64h+63 -> columns [64h, 64h + 32).  dP^T (fp32) in
  // [128, 256), dS^T packed the same way at 128 + [64h, 64h + 32); dQ_i (fp32, D columns) is
  // accumulated over [128, 128 + D) once dK += dS^T Q has consumed dS^T.  At d = 64 there are two
  // such dP regions, [128, 256) for even and [256, 384) for odd query iterations, so that dP(i+1)
  // need not wait for dQ(i) to be drained; dV and dK follow them.
  static constexpr bool kDP2 = (D == 64);
  static constexpr uint32_t kColS = 0, kColDP = 128;
  static constexpr uint32_t kColDV = kDP2 ? 384 : 256, kColDK = kColDV + D;
  static constexpr uint32_t kTmemCols = 512;
};

// Warpgroups sharing the elementwise work (P, dS, the dQ drain, the epilogue); each owns
// 128 / kGroups query columns of every key row.  Measured on GB300: 4 groups are no faster
// than 2 at d = 128 and 6% slower at d = 64 (the kernel is bound by moving the fp32 dQ
// partials to L2 and by shared-memory traffic, not by the latency of these phases).
#ifndef FA_BWD_GROUPS
#define FA_BWD_GROUPS 2
#endif
constexpr int kGroups = FA_BWD_GROUPS;
constexpr int kQG = 128 / kGroups;  // query columns per group
static_assert(kGroups == 2 || kGroups == 4, "two or four elementwise warpgroups");

// Packed bf16 column of the 16-query k-step kk (0..7) inside the S^T or dP^T region: a group
// writes its packed values over the first half of its own columns.
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return (16 * kk / kQG) * kQG + ((16 * kk) % kQG) / 2;
}

constexpr int kBwdThreads = 128 * (1 + kGroups);

// How the drain warps write one partial dQ tile (see "dQ across key tiles" above).
enum : int { kModeAdd = 0, kModeFirst = 1 };

// Waits until the first claimant of a query tile has stored its partial (bit 63 of the tile's
// word).  Bounded like every pipeline wait.
__device__ __forceinline__ bool wait_first_stored(const uint64_t* word, const Ctl& c) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_u64(word) & kDqStored) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.timeout_ns) {
      ctl_fail(c, kErrTimeout);
      return false;
    }
  }
}

// kWithDQ = false: the deterministic variant, dQ is computed by bwd_dq_kernel instead (no dQ
// GEMM, no drain, no atomics, no dS copy in shared memory).
// kSparse: block-sparse; the key tile visits only the query tiles its mask column keeps (a
// descending list from the block index, whose prefix of tiles >= the key tile is the causal part).
// kVarlen: packed variable-length batch (see the forward kernel); grouped-query attention (Hkv <
// H) makes the CTA of key/value head hk walk the query tiles of all H / Hkv heads of its group,
// so dK and dV sum over the group in tensor memory.
template <int D, bool kWithDQ, bool kSparse, bool kVarlen>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdK,
                    const __grid_constant__ CUtensorMap tmdV, const BwdArgs a) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* sm = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = bars + 3;
  uint64_t* do_full = bars + 5;
  uint64_t* do_empty = bars + 7;
  uint64_t* s_full = bars + 9;
  uint64_t* p_full = bars + 10;
  uint64_t* dp_full = bars + 11;
  uint64_t* ds_full = bars + 12;
  uint64_t* dq_full = bars + 13;
  uint64_t* dq_empty = bars + 14;
  uint64_t* dkdv_full = bars + 15;
  uint64_t* mma_done = bars + 16;
  uint64_t* mode_full = bars + 17;     // [2] the claim warp published how a drain writes
  uint64_t* mode_empty = bars + 19;    // [2] every drain warp took it (its drain has begun)
  uint64_t* first_stored = bars + 21;  // [2] every drain warp issued its stores of a first partial
  uint64_t* staged = bars + 23;        // [2] (d = 64) every drain warp wrote its share of a slot
  uint64_t* stage_empty = bars + 25;   // [2] (d = 64) the TMA unit has read the slot
  // the drain of iteration it releases dq_empty_of(it): at d = 64 one barrier per dP region
  auto dq_empty_of = [&](int it) { return (L::kDP2 && (it & 1)) ? bars + 27 : dq_empty; };
  auto dp_col = [&](int it) { return L::kColDP + ((L::kDP2 && (it & 1)) ? 128u : 0u); };
  volatile int* mode_slot = reinterpret_cast<volatile int*>(sm + L::kMode);
  volatile int* stage_kind = reinterpret_cast<volatile int*>(sm + L::kKind);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kAbort);
  const Ctl ctl{abort_flag, a.status, a.timeout_ns};

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  if (pad + L::kBytes > a.smem_bytes) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kErrLayout);
    return;
  }

  // ---- work item: head-major (one or two heads' Q, dO and dQ accumulator live in L2 at a
  // time); within a head key tile 0 first (with a causal mask the lowest tiles have most work)
  const int lin = blockIdx.x;
  const int bkv = lin / a.num_qtiles;  // (b, key/value head)
  const int j = lin % a.num_qtiles;
  const int b = bkv / a.Hkv;
  const int hk = bkv - b * a.Hkv;
  const int G = a.H / a.Hkv;  // query heads per key/value head
  int seq_start = 0, N = a.N;
  if constexpr (kVarlen) seq_bounds(a.cu_seqlens, b, a.total, seq_start, N);
  if (kVarlen && j * 128 >= N) return;  // past this sequence's end (uniform over the CTA)
  const int nqt = kVarlen ? (N + 127) / 128 : a.num_qtiles;  // this sequence's query tiles
  int kv_len = N;
  if (!kVarlen && a.kv_lens != nullptr) kv_len = min(max(__ldg(a.kv_lens + b), 0), N);
  const int i0 = a.causal ? j : 0;
  int nI = (j * 128 < kv_len) ? (nqt - i0) : 0;  // query tiles this key tile visits per head
  // workspace rows / dQ accumulator tiles of query head h: (ws_head(h) * ws_tiles + tile0 + i)
  const int ws_tile0 = kVarlen ? seq_tile0(seq_start, b) : 0;
  auto ws_head = [&](int h) { return kVarlen ? h : b * a.H + h; };
  // TMA box coordinates (y, z) of row r: dense (r, head slice), packed (head, token)
  auto q_y = [&](int h, int r) { return kVarlen ? h : r; };
  auto q_z = [&](int h, int r) { return kVarlen ? seq_start + r : b * a.H + h; };
  const int kv_y = kVarlen ? hk : j * 128;
  const int kv_z = kVarlen ? seq_start + j * 128 : bkv;
  const int32_t* c_list = nullptr;
  if constexpr (kSparse) {
    const BlockIndex BI = block_index_layout(nqt);
    // (block-sparse calls have Hkv == H: bkv is the query head slice)
    const int32_t* base = a.blk + (a.blk_heads == 1 ? 0 : static_cast<int64_t>(bkv % a.H) * BI.words);
    c_list = base + BI.cidx + static_cast<int64_t>(j) * nqt;
    nI = (j * 128 < kv_len) ? __ldg(base + (a.causal ? BI.cccnt : BI.ccnt) + j) : 0;
  }
  // without a causal mask key tile j starts at query tile j and wraps around, so the key tiles of
  // a head reach any one query tile a tile period apart (dQ accumulation, see above)
  auto qtile = [&](int it) {
    if constexpr (kSparse) return __ldg(c_list + it);
    return a.causal ? i0 + it : (j + it < nqt ? j + it : j + it - nqt);
  };
  // iteration it -> (query head of the group, query tile); G == 1 without grouped queries
  auto head_of = [&](int it) { return hk * G + (G == 1 ? 0 : it / nI); };
  auto tile_of = [&](int it) { return qtile(G == 1 ? it : it % nI); };
  const int nIt = nI * G;  // iterations of the CTA
  // workspace tile (record, accumulator tile) of query head qh, query tile qt
  auto ws_tile_of = [&](int qh, int qt) {
    return static_cast<size_t>(ws_head(qh)) * a.ws_tiles + ws_tile0 + qt;
  };

  if (warp == 0 && lane == 0) {
    *abort_flag = 0;
    for (int k = 0; k < L::kNumBars; ++k) {
      // P, dS, the release of dQ_i's tensor memory and the drain barriers are signalled by every
      // warp of the elementwise warpgroups
      uint32_t count = 1;
      if (&bars[k] == p_full || &bars[k] == ds_full || &bars[k] == dq_empty || k == 27 ||
          &bars[k] == &mode_empty[0] || &bars[k] == &mode_empty[1] ||
          &bars[k] == &first_stored[0] || &bars[k] == &first_stored[1] ||
          &bars[k] == &staged[0] || &bars[k] == &staged[1])
        count = 4 * kGroups;
      mbar_init(&bars[k], count);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdK);
    tma_prefetch_desc(&tmdV);
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

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0 && nIt > 0) {
      mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sm + L::kK + c * 16384, &tmK, kv_full, c * 64, kv_y, kv_z);
        tma_load_3d(sm + L::kV + c * 16384, &tmV, kv_full, c * 64, kv_y, kv_z);
      }
      int nq = 0, ndo = 0;
      for (int it = 0; it < nIt; ++it) {
        const int h = head_of(it), i = tile_of(it), s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        if (!mbar_wait(&q_empty[s], ph ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&q_full[s], L::kTile + 1024);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm + L::kQ + s * L::kTile + c * 16384, &tmQ, &q_full[s], c * 64,
                      q_y(h, i * 128), q_z(h, i * 128));
        const size_t srow =
            (static_cast<size_t>(ws_head(h)) * a.ws_tiles + ws_tile0 + i) * 128;
        bulk_load(sm + L::kLse + s * 512, a.neg_lse2 + srow, 512, &q_full[s]);
        bulk_load(sm + L::kDelta + s * 512, a.neg_delta + srow, 512, &q_full[s]);
        nq = it + 1;
        if (!mbar_wait(&do_empty[s], ph ^ 1, ctl)) break;
        mbar_arrive_expect_tx(&do_full[s], L::kTile);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sm + L::kDO + s * L::kTile + c * 16384, &tmdO, &do_full[s], c * 64,
                      q_y(h, i * 128), q_z(h, i * 128));
        ndo = it + 1;
      }
      // no copy may still be in flight when the CTA exits, aborted or not
      drain_wait(kv_full, 0, ctl);
      for (int it = max(0, nq - 2); it < nq; ++it) drain_wait(&q_full[it & 1], (it >> 1) & 1, ctl);
      for (int it = max(0, ndo - 2); it < ndo; ++it)
        drain_wait(&do_full[it & 1], (it >> 1) & 1, ctl);
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0 && nIt > 0) {
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);  // S^T, dP^T: K-major operands
      constexpr uint32_t idKV = idesc_bf16(128, D, false, true);    // dV, dK: A in TMEM, B MN-major
      constexpr uint32_t idQ = idesc_bf16(128, D, true, true);      // dQ: A = dS MN-major, B MN-major
      const uint32_t kb = sbase + L::kK, vb = sbase + L::kV, dsb = sbase + L::kDS;
      // Issue order (software-pipelined over query tiles): S(0), dP(0), dV(0), S(1), then per
      // tile i: dK(i), dQ(i) | dV(i+1), dP(i+1) | S(i+2).  The tensor pipe always has the next
      // tile's work queued while the P/dS warpgroups compute, and dV(i+1) covers the drain of
      // dQ(i) that dP(i+1) waits for.  Every MMA waits for the copies of its own operands (dV(i+1)
      // for dO(i+1), although P(i+1) alone is what it follows), and a stage is released only after
      // the last MMA that reads it: Q_i after dK(i), dO_i after the later of dP(i) and dV(i).
      // descriptors of each operand buffer; a k-step adds its byte offset to the start address
      const uint64_t desc_k = sdesc_sw128(kb, 16384, 1024), desc_v = sdesc_sw128(vb, 16384, 1024);
      const uint64_t desc_ds = sdesc_sw128(dsb, 16384, 1024);
      auto desc_q = [&](int it) {
        return sdesc_sw128(sbase + L::kQ + (it & 1) * L::kTile, 16384, 1024);
      };
      auto desc_do = [&](int it) {
        return sdesc_sw128(sbase + L::kDO + (it & 1) * L::kTile, 16384, 1024);
      };
      // Each product is one chain of K-steps (sm103.cuh); with two elementwise groups the
      // packed P^T / dS^T halves sit at columns [0, 32) and [64, 96) (packed_col).
      auto ts_chain = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
        if constexpr (kQG == 64) {
          mma_ts_k128_split(d, a, b, idKV, acc);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(d, a + packed_col(kk), b + kk * 128, idKV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_S = [&](int it) {  // S^T = K_j Q_i^T
        mma_ss_kmajor<D>(tmem + L::kColS, desc_k, desc_q(it), idS, 0u);
        mma_commit(s_full);
      };
      auto issue_dP = [&](int it) {  // dP^T = V_j dO_i^T
        mma_ss_kmajor<D>(tmem + dp_col(it), desc_v, desc_do(it), idS, 0u);
        mma_commit(dp_full);
      };
      auto issue_dV = [&](int it) {  // dV += P^T dO_i   (128 queries, 16 per MMA: +2 KB rows)
        ts_chain(tmem + L::kColDV, tmem + L::kColS, desc_do(it), it > 0 ? 1u : 0u);
      };
      // dO_i is read by dP(i) and dV(i): its stage is released after whichever is issued last
      auto release_do = [&](int it) { mma_commit(&do_empty[it & 1]); };
      auto issue_dK_dQ = [&](int it) {
        ts_chain(tmem + L::kColDK, tmem + dp_col(it), desc_q(it), it > 0 ? 1u : 0u);  // dK += dS^T Q_i
        mma_commit(&q_empty[it & 1]);
        if (kWithDQ) {  // dQ_i = dS K_j  (128 keys, 16 per MMA) over dP^T
          mma_ss_mn_k128(tmem + dp_col(it), desc_ds, desc_k, idQ, 0u);
          mma_commit(dq_full);
        }
      };
      auto wait_q = [&](int it) { return mbar_wait(&q_full[it & 1], (it >> 1) & 1, ctl); };
      auto wait_do = [&](int it) { return mbar_wait(&do_full[it & 1], (it >> 1) & 1, ctl); };

      bool ok = mbar_wait(kv_full, 0, ctl) && wait_q(0);
      if (ok) {
        tc_fence_after();
        issue_S(0);
        ok = wait_do(0);
      }
      if (ok) {
        tc_fence_after();
        issue_dP(0);
        ok = mbar_wait(p_full, 0, ctl);
      }
      if (ok) {
        tc_fence_after();
        issue_dV(0);
        release_do(0);  // dP(0) went first
        if (nIt > 1 && (ok = wait_q(1))) {
          tc_fence_after();
          issue_S(1);
        }
      }
      for (int it = 0; ok && it < nIt; ++it) {
        if (!(ok = mbar_wait(ds_full, it & 1, ctl))) break;
        tc_fence_after();
        issue_dK_dQ(it);
        if (it + 1 < nIt && L::kDP2) {
          // d = 64: dP(i+1) has a region of its own (dQ(i - 1)'s, drained before dS(i)), so it
          // goes first, ahead of the P(i+1) that dV(i+1) waits for
          if (!(ok = wait_do(it + 1))) break;
          if (kWithDQ && it >= 1 && !(ok = mbar_wait(dq_empty_of(it - 1), ((it - 1) >> 1) & 1, ctl)))
            break;
          tc_fence_after();
          issue_dP(it + 1);
          if (!(ok = mbar_wait(p_full, (it + 1) & 1, ctl))) break;
          tc_fence_after();
          issue_dV(it + 1);
          release_do(it + 1);
          if (it + 2 < nIt) {
            if (!(ok = wait_q(it + 2))) break;
            tc_fence_after();
            issue_S(it + 2);
          }
        } else if (it + 1 < nIt) {
          // dV(i+1) reads dO(i+1): its copy must have landed (P(i+1) does not depend on it)
          if (!(ok = mbar_wait(p_full, (it + 1) & 1, ctl) && wait_do(it + 1))) break;
          tc_fence_after();
          issue_dV(it + 1);
          if (kWithDQ && !(ok = mbar_wait(dq_empty, it & 1, ctl))) break;
          tc_fence_after();
          issue_dP(it + 1);
          release_do(it + 1);
          if (it + 2 < nIt) {
            if (!(ok = wait_q(it + 2))) break;
            tc_fence_after();
            issue_S(it + 2);
          }
        }
      }
      if (ok) mma_commit(dkdv_full);
      mma_commit(mma_done);
      drain_wait(mma_done, 0, ctl);
    }
  } else if (warp == 2 || warp == 3) {
    // ================= dQ claims (at d = 128 one thread of each warp, warp 2 the even iterations
    // and warp 3 the odd ones; at d = 64 warp 2 alone).  Claims each query tile and tells the
    // drain warps whether to store its partial (the tile's first claimant) or add it (any later
    // one, once the first one's stores are visible).  A claim is an acquiring atomic add on the
    // tile's word, whose old value also says whether the first partial is stored yet.  An atomic
    // from this SM waits behind the SM's own dQ additions in flight (thousands of cycles, about a
    // tile period) and an acquiring one holds back its thread's later memory operations meanwhile,
    // so claims are made two drains ahead: iteration it at the start of the drain of it - 2
    // (iteration 0 at the start, iteration 1 at the drain of 0), at d = 128 by two threads taking
    // turns.  Claims thus follow the order of the drains, and under the causal order (and the
    // rotated non-causal one) the first claimant of a tile is the key tile that drains it first.
    // After the drain warps have issued a first partial's stores, a fence orders them before the
    // record's bit 63.
    constexpr int kClaimThreads = L::kBulkDQ ? 1 : 2;
    const int par = static_cast<int>(warp) - 2;
    if (kWithDQ && lane == 0 && par < kClaimThreads && nIt > par) {
      auto rec = [&](int it) { return &a.dq_cnt[ws_tile_of(head_of(it), tile_of(it))].word; };
      int firsts0 = 0, firsts1 = 0;  // first partials of this thread per first_stored slot
      int prev_first = -1;  // this thread's previous iteration, if it stored a first partial
      auto first_done = [&](int it) -> bool {  // the drain of `it` stores a first partial
        int& f = (it & 1) ? firsts1 : firsts0;
        if (!mbar_wait(&first_stored[it & 1], f & 1, ctl)) return false;
        ++f;
        fence_acq_rel_gpu();  // the drain warps' stores (seen through first_stored) go first
        red_add_relaxed_u64(rec(it), kDqStored);
        return true;
      };
      bool ok = true;
      for (int it = par; ok && it < nIt; it += kClaimThreads) {
        // claim time: the start of the drain of it - 2 (of 0 for iteration 1)
        if (it >= 1 && !(ok = mbar_wait(&mode_empty[it < 2 ? 0 : it & 1],
                                        it < 2 ? 0u : ((it - 2) >> 1) & 1, ctl)))
          break;
        if (prev_first >= 0) {
          if (!(ok = first_done(prev_first))) break;
          prev_first = -1;
        }
        const uint64_t old = atom_add_acquire_u64(rec(it), 1ull);
        const bool first = static_cast<uint32_t>(old) == 0u;
        if (!first && !(old & kDqStored) && !(ok = wait_first_stored(rec(it), ctl))) break;
        mode_slot[it & 1] = first ? kModeFirst : kModeAdd;
        mbar_arrive(&mode_full[it & 1]);
        if (first) prev_first = it;
      }
      if (ok && prev_first >= 0) first_done(prev_first);  // this thread's last iteration's
    } else if (L::kBulkDQ && kWithDQ && lane == 0 && par == 1 && nIt > 0) {
      // ================= dQ additions at d = 64 (warp 3): hands each staged partial to the TMA
      // unit, which adds it into the accumulator (cp.reduce.async.bulk), so the drain warps never
      // wait for the L2 to take their additions; a slot is released once the unit has read it.
      // Every iteration but the last (whose partial the drain warps add themselves)
      bool ok = true;
      int prev_kind = -1;
      for (int it = 0; it < nIt - 1; ++it) {
        const int s = it & 1;
        if (!(ok = mbar_wait(&staged[s], (it >> 1) & 1, ctl))) break;
        const int kind = stage_kind[s];
        if (kind == kModeAdd) {
          // the acquire of the first partial's bit (generic proxy) precedes these additions
          fence_proxy_async_global();
          bulk_reduce_add_f32(a.dq_acc + ws_tile_of(head_of(it), tile_of(it)) * 128 * D,
                              sm + L::kStage + s * L::kPart, L::kPart);
          bulk_commit();
        }
        if (it >= 1) {  // the previous slot, once read
          if (prev_kind == kModeAdd) {
            if (kind == kModeAdd) bulk_wait_read1();
            else bulk_wait_read0();
          }
          mbar_arrive(&stage_empty[(it - 1) & 1]);
        }
        prev_kind = kind;
      }
      bulk_wait0();  // every addition performed before the CTA exits (aborted or not)
    }
  } else if (warp >= 4) {
    // ================= P, dS, the dQ drain and the epilogue: one thread per row of the tile,
    // one warpgroup per kQG query columns of P / dS and D / kGroups columns of dQ
    const uint32_t quad = warp & 3;
    const int grp = (warp - 4) >> 2;
    const int q0 = kQG * grp;  // first query column of this group
    const int r = quad * 32 + lane;
    const int key = j * 128 + r;
    const bool row_live = key < kv_len;
    const uint32_t lanes = (quad * 32u) << 16;
    const uint32_t tS = tmem + lanes + L::kColS + q0;
    constexpr int kDC = D / kGroups;  // dQ columns drained by this group
    // dP^T / dS^T and dQ columns of iteration it (two alternating regions at d = 64)
    auto tDP_of = [&](int it) { return tmem + lanes + dp_col(it) + q0; };
    auto tDQ_of = [&](int it) { return tmem + lanes + dp_col(it) + kDC * grp; };
    const float c2 = a.scale_log2;

    // dQ_i (query row r of the tile, this group's columns) into the fp32 accumulator: load,
    // release the tensor memory (dP_{i+1} waits for it), then the atomics, which overlap dP_{i+1}
    // The atomics of the second half of this thread's dQ columns wait until dS has been handed
    // to the MMA thread (after ds_full), so that they overlap dK += dS^T Q and dQ = dS K instead
    // of delaying dS; the values wait in registers (dQ must leave tensor memory before dP(i+1)
    // overwrites it, but the additions can come later).
    constexpr int kGroups4 = kDC / 4;       // 4-column groups of this thread's dQ columns
#ifndef FA_DQ_LATE64
#define FA_DQ_LATE64 0
#endif
#ifndef FA_DQ_LATE128
#define FA_DQ_LATE128 8
#endif
    // of which issued after dS.  Measured on GB300 (dK/dV kernel): d = 128 with 0 / 4 / 8 / 12 of
    // 16 deferred: 4.90 / 4.28 / 4.27 / 4.88 ms on long-causal 1x32x16384, 2.98 / 2.45 / 2.38 /
    // 2.74 ms on causal 16x16x4096 (12 needs 163 registers); d = 64 with 0 / 4 / 8 of 8: 0.932 /
    // 0.977 / 1.047 ms on 64x16x1024 (there the atomics are a smaller share than the MMA issue).
    constexpr int kLate = (D == 128) ? FA_DQ_LATE128 : FA_DQ_LATE64;
    uint32_t dq_late[4 * (kLate > 0 ? kLate : 1)];
    float* late_tile = nullptr;
    auto drain = [&](int it, int qh, int qt) -> bool {  // (qh, qt): query head, tile of it
      if (!mbar_wait_warp(&mode_full[it & 1], (it >> 1) & 1, ctl)) return false;
      const int mode = mode_slot[it & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(&mode_empty[it & 1]);
      if (!mbar_wait_warp(dq_full, it & 1, ctl)) return false;
      tc_fence_after();
      float* tile = a.dq_acc + ws_tile_of(qh, qt) * 128 * D;
      const int g0 = kGroups4 * grp;  // first 4-column group of this group's columns
      const uint32_t tDQ = tDQ_of(it);
      uint32_t v[kDC];
      if constexpr (kDC == 64) {
        tmem_ld32(tDQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      } else if constexpr (kDC == 32) {
        tmem_ld32(tDQ, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      } else {
        tmem_ld16(tDQ, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
      }
      tmem_wait_ld();
      reg_fence(v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_empty_of(it));
      if (L::kBulkDQ && it + 1 < nIt) {
        // d = 64: a first partial is stored directly; any other goes to a shared-memory slot (the
        // accumulator tile's layout) whose addition the TMA unit performs.  Not the CTA's last
        // drain: the dV and dK stores that follow it go through the TMA unit too and would wait
        // behind that addition (measured on GB300: dK/dV 0.926 -> 0.916 ms on 64x16x1024x64 with
        // the last partial added by the drain warps, below)
        const int ss = it & 1;
        if (!mbar_wait_warp(&stage_empty[ss], ((it >> 1) & 1) ^ 1, ctl)) return false;
        if (mode == kModeFirst) {
#pragma unroll
          for (int g = 0; g < kGroups4; ++g)
            st_v4(tile + ((g0 + g) * 128 + r) * 4, __uint_as_float(v[4 * g]),
                  __uint_as_float(v[4 * g + 1]), __uint_as_float(v[4 * g + 2]),
                  __uint_as_float(v[4 * g + 3]));
          __syncwarp();
          if (lane == 0) mbar_arrive(&first_stored[it & 1]);
        } else {
          const uint32_t slot = sbase + L::kStage + ss * L::kPart;
#pragma unroll
          for (int g = 0; g < kGroups4; ++g)
            st_shared_v4(slot + (((g0 + g) * 128 + r) * 4) * 4, v[4 * g], v[4 * g + 1],
                         v[4 * g + 2], v[4 * g + 3]);
          fence_proxy_async_smem();  // the TMA unit reads the slot
        }
        __syncwarp();
        if (lane == 0) {
          stage_kind[ss] = mode;
          mbar_arrive(&staged[ss]);
        }
        return true;
      }
      if (mode == kModeFirst) {  // the tile's first partial: stored, whole lines per warp
#pragma unroll
        for (int g = 0; g < kGroups4; ++g)
          st_v4(tile + ((g0 + g) * 128 + r) * 4, __uint_as_float(v[4 * g]),
                __uint_as_float(v[4 * g + 1]), __uint_as_float(v[4 * g + 2]),
                __uint_as_float(v[4 * g + 3]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&first_stored[it & 1]);
        return true;
      }
#pragma unroll
      for (int g = 0; g < kGroups4 - kLate; ++g)
        red_add_v4(tile + ((g0 + g) * 128 + r) * 4, __uint_as_float(v[4 * g]),
                   __uint_as_float(v[4 * g + 1]), __uint_as_float(v[4 * g + 2]),
                   __uint_as_float(v[4 * g + 3]));
#pragma unroll
      for (int e = 0; e < 4 * kLate; ++e) dq_late[e] = v[4 * (kGroups4 - kLate) + e];
      late_tile = tile + (g0 + kGroups4 - kLate) * 128 * 4;
      return true;
    };
    auto drain_late = [&]() {  // the deferred additions of the last drain, if any
      if (late_tile == nullptr) return;
#pragma unroll
      for (int g = 0; g < kLate; ++g)
        red_add_v4(late_tile + (g * 128 + r) * 4, __uint_as_float(dq_late[4 * g]),
                   __uint_as_float(dq_late[4 * g + 1]), __uint_as_float(dq_late[4 * g + 2]),
                   __uint_as_float(dq_late[4 * g + 3]));
      late_tile = nullptr;
    };

    bool ok = true;
    int h_prev = 0, i_prev = 0;  // previous iteration's query head and tile (drained in this one)
    for (int it = 0; it < nIt; ++it) {
      const int h = head_of(it), i = tile_of(it), s = it & 1;
      const uint32_t ph = (it >> 1) & 1;
      if (!(ok = mbar_wait_warp(&q_full[s], ph, ctl))) break;  // LSE and D are in smem
      if (!(ok = mbar_wait_warp(s_full, it & 1, ctl))) break;
      tc_fence_after();
      const float* nl2 = reinterpret_cast<const float*>(sm + L::kLse + s * 512) + q0;
      const float* nd = reinterpret_cast<const float*>(sm + L::kDelta + s * 512) + q0;
      const float2 cc = make_float2(c2, c2);
      const bool diag = a.causal && (i == j);
      // only the causal diagonal tile and a key tile running past the key length need element
      // masks; every other tile (the test is uniform over the CTA) skips them
      const bool masked = diag || (j * 128 + 128 > kv_len);
      uint32_t p[kQG / 2];
      // d = 64 has the registers to keep P in fp32 for dS (no unpacking of the bf16 pairs; dS
      // then uses the unrounded P): measured on GB300, dK/dV 0.915 -> 0.892 ms at 64x16x1024x64
      constexpr bool kPf = (D == 64);
      float pf[kPf ? kQG : 1];
      auto p_from_s = [&](auto kMask) {
#pragma unroll
        for (int c = 0; c < kQG / 32; ++c) {
          uint32_t sv[32];
          tmem_ld32(tS + 32 * c, sv);
          tmem_wait_ld();
          reg_fence(sv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int ql = 32 * c + 4 * e;  // query within this group
            const float4 l4 = *reinterpret_cast<const float4*>(nl2 + ql);  // -LSE * log2(e)
            const float2 y0 = fma2(make_float2(__uint_as_float(sv[4 * e]), __uint_as_float(sv[4 * e + 1])),
                                   cc, make_float2(l4.x, l4.y));
            const float2 y1 = fma2(make_float2(__uint_as_float(sv[4 * e + 2]), __uint_as_float(sv[4 * e + 3])),
                                   cc, make_float2(l4.z, l4.w));
            float x[4] = {ex2(y0.x), ex2(y0.y), ex2(y1.x), ex2(y1.y)};
            if constexpr (decltype(kMask)::value) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                if (diag) x[u] = (r <= q0 + ql + u) ? x[u] : 0.f;  // key > query: masked
                if (!row_live) x[u] = 0.f;
              }
            }
            p[16 * c + 2 * e] = pack_bf16(x[0], x[1]);
            p[16 * c + 2 * e + 1] = pack_bf16(x[2], x[3]);
            if constexpr (kPf) {
#pragma unroll
              for (int u = 0; u < 4; ++u) pf[ql + u] = x[u];
            }
          }
        }
      };
      if (masked) p_from_s(std::true_type{});
      else p_from_s(std::false_type{});
      // P^T over the first half of this group's columns (all of its S^T was read)
      if (kQG == 64) tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      else tmem_st16(tS, *reinterpret_cast<uint32_t(*)[16]>(&p[0]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);

      if (kWithDQ && it > 0 && !(ok = drain(it - 1, h_prev, i_prev))) break;

      if (!(ok = mbar_wait_warp(dp_full, it & 1, ctl))) break;
      tc_fence_after();
      const uint32_t tDP = tDP_of(it);
#pragma unroll
      for (int c = 0; c < kQG / 32; ++c) {
        uint32_t dv[32];
        tmem_ld32(tDP + 32 * c, dv);
        tmem_wait_ld();
        reg_fence(dv);
        uint32_t ds[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int ql = 32 * c + 4 * e;
          const float4 d4 = *reinterpret_cast<const float4*>(nd + ql);  // -D
          const uint32_t pa = p[16 * c + 2 * e], pb = p[16 * c + 2 * e + 1];
          const float2 t0 = add2(make_float2(__uint_as_float(dv[4 * e]), __uint_as_float(dv[4 * e + 1])),
                                 make_float2(d4.x, d4.y));
          const float2 t1 = add2(make_float2(__uint_as_float(dv[4 * e + 2]), __uint_as_float(dv[4 * e + 3])),
                                 make_float2(d4.z, d4.w));
          const float2 p0 = kPf ? make_float2(pf[ql], pf[ql + 1]) : make_float2(bf16_lo(pa), bf16_hi(pa));
          const float2 p1 = kPf ? make_float2(pf[ql + 2], pf[ql + 3]) : make_float2(bf16_lo(pb), bf16_hi(pb));
          const float2 u0 = mul2(p0, t0);
          const float2 u1 = mul2(p1, t1);
          ds[2 * e] = pack_bf16(u0.x, u0.y);
          ds[2 * e + 1] = pack_bf16(u1.x, u1.y);
        }
        // dS^T packed over dP^T columns this group has already read (A operand of dK += dS^T Q)
        tmem_st16(tDP + 16 * c, ds);
        if (kWithDQ) {  // and to smem as [key row][query], 128-byte swizzled (A of dQ = dS K)
          const int qa = q0 + 32 * c;  // absolute first query of this chunk
          const uint32_t panel = sbase + L::kDS + (qa >> 6) * 16384;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            st_shared_v4(panel + sw128_offset(r, ((qa & 63) >> 3) + g), ds[4 * g], ds[4 * g + 1],
                         ds[4 * g + 2], ds[4 * g + 3]);
        }
      }
      tmem_wait_st();
      if (kWithDQ) fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);
      if (kWithDQ) drain_late();  // dQ(it - 1)'s deferred additions overlap dK / dQ(it)
      h_prev = h;
      i_prev = i;
    }
    if (kWithDQ) drain_late();  // (an aborted loop may leave one pending)
    if (kWithDQ && ok && nIt > 0) {
      ok = drain(nIt - 1, h_prev, i_prev);
      if (ok) drain_late();
    }

    // ---- epilogue: the 64-column panels of dV and scale * dK (bf16, swizzled, over the V or K
    // tile in smem, which no MMA reads any more) are shared out over the groups; one TMA store
    // per panel
    if (ok && nIt > 0) ok = mbar_wait_warp(dkdv_full, 0, ctl);
    constexpr int kPanels = 2 * (D / 64);  // dV panels, then dK panels
    if (ok && nIt > 0) tc_fence_after();
    // variable-length: a key tile that runs past its sequence's end is stored row by row
    const bool direct = kVarlen && (j * 128 + 128 > N);
    for (int pn = grp; pn < kPanels; pn += kGroups) {
      const bool is_dk = pn >= D / 64;
      const int cp = pn % (D / 64);  // column panel within the matrix
      const uint32_t col = (is_dk ? L::kColDK : L::kColDV) + 64 * cp;
      const float mul = is_dk ? a.scale : 1.f;
      const uint32_t panel = sbase + (is_dk ? L::kK : L::kV) + cp * 16384;
      if (ok) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          if (nIt > 0) {
            tmem_ld32(tmem + lanes + col + 32 * c, v);
            tmem_wait_ld();
            reg_fence(v);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul);
          if (direct) {
            if (key < N) {
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<__nv_bfloat16*>(is_dk ? a.dk : a.dv) +
                  (static_cast<size_t>(seq_start + key) * a.Hkv + hk) * D + 64 * cp + 32 * c);
#pragma unroll
              for (int g = 0; g < 4; ++g)
                dst[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
            }
          } else {
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
        tma_store_3d(is_dk ? &tmdK : &tmdV, sm + (is_dk ? L::kK : L::kV) + cp * 16384, cp * 64,
                     kv_y, kv_z);
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

}  // namespace

namespace {
// Blocks of a 1-D grid of `tiles` per head slice times `heads` slices; 0 when that exceeds the
// grid's x limit (2^31 - 1) or is empty.
unsigned flat_grid(long long tiles, long long heads) {
  const long long n = tiles * heads;
  return (tiles <= 0 || heads <= 0 || n > 0x7fffffffLL) ? 0u : static_cast<unsigned>(n);
}
}  // namespace

cudaError_t launch_bwd_preprocess(int d, const void* O, const void* dO, const float* lse, int BH,
                                  int N, float* neg_lse2, float* neg_delta, DqTileCount* recs,
                                  cudaStream_t s) {
  const int nqt = (N + 127) / 128;
  const unsigned grid = flat_grid(nqt, BH);
  if (grid == 0) return cudaErrorInvalidConfiguration;
  auto o = static_cast<const __nv_bfloat16*>(O);
  auto g = static_cast<const __nv_bfloat16*>(dO);
  const RowGeo geo{nullptr, 1, 0, 0};
  if (d == 64)
    bwd_preprocess_kernel<64, false><<<grid, 256, 0, s>>>(o, g, lse, N, nqt, neg_lse2, neg_delta,
                                                           recs, nqt, geo);
  else
    bwd_preprocess_kernel<128, false><<<grid, 256, 0, s>>>(o, g, lse, N, nqt, neg_lse2,
                                                            neg_delta, recs, nqt, geo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess_varlen(int d, const void* O, const void* dO, const float* lse,
                                         const int32_t* cu, int B, int H, int max_tiles,
                                         int total, int ws_tiles, float* neg_lse2,
                                         float* neg_delta, DqTileCount* recs, cudaStream_t s) {
  const unsigned grid = flat_grid(max_tiles, static_cast<long long>(B) * H);
  if (grid == 0) return cudaErrorInvalidConfiguration;
  auto o = static_cast<const __nv_bfloat16*>(O);
  auto g = static_cast<const __nv_bfloat16*>(dO);
  const RowGeo geo{cu, H, total, ws_tiles};
  if (d == 64)
    bwd_preprocess_kernel<64, true><<<grid, 256, 0, s>>>(o, g, lse, 0, 0, neg_lse2, neg_delta,
                                                          recs, max_tiles, geo);
  else
    bwd_preprocess_kernel<128, true><<<grid, 256, 0, s>>>(o, g, lse, 0, 0, neg_lse2, neg_delta,
                                                           recs, max_tiles, geo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(int d, const float* dq_acc, const DqTileCount* recs, void* dQ,
                                  int BH, int N, float scale, cudaStream_t s) {
  const int nqt = (N + 127) / 128;
  const unsigned grid = flat_grid(nqt, BH);
  if (grid == 0) return cudaErrorInvalidConfiguration;
  auto out = static_cast<__nv_bfloat16*>(dQ);
  const RowGeo geo{nullptr, 1, 0, 0};
  if (d == 64)
    bwd_dq_convert_kernel<64, false><<<grid, 256, 0, s>>>(dq_acc, recs, out, N, nqt, scale, nqt,
                                                           geo);
  else
    bwd_dq_convert_kernel<128, false><<<grid, 256, 0, s>>>(dq_acc, recs, out, N, nqt, scale, nqt,
                                                            geo);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert_varlen(int d, const float* dq_acc, const DqTileCount* recs,
                                         void* dQ, const int32_t* cu, int B, int H,
                                         int max_tiles, int total, int ws_tiles, float scale,
                                         cudaStream_t s) {
  const unsigned grid = flat_grid(max_tiles, static_cast<long long>(B) * H);
  if (grid == 0) return cudaErrorInvalidConfiguration;
  auto out = static_cast<__nv_bfloat16*>(dQ);
  const RowGeo geo{cu, H, total, ws_tiles};
  if (d == 64)
    bwd_dq_convert_kernel<64, true><<<grid, 256, 0, s>>>(dq_acc, recs, out, 0, 0, scale, max_tiles,
                                                          geo);
  else
    bwd_dq_convert_kernel<128, true><<<grid, 256, 0, s>>>(dq_acc, recs, out, 0, 0, scale,
                                                           max_tiles, geo);
  return cudaGetLastError();
}

namespace {
template <int D, bool kWithDQ, bool kSparse, bool kVarlen>
cudaError_t launch_dkdv_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                          BwdArgs a, cudaStream_t st) {
  using L = BwdLayout<D>;
  constexpr uint32_t kMaxSmem = 232448;  // 227 KB, the per-block opt-in limit of sm_100-family GPUs
  const uint32_t smem = (L::kBytes + 1024 <= kMaxSmem) ? L::kBytes + 1024 : kMaxSmem;
  cudaError_t e = ensure_smem_limit<bwd_dkdv_kernel<D, kWithDQ, kSparse, kVarlen>>(smem);
  if (e != cudaSuccess) return e;
  a.smem_bytes = smem;
  // one CTA per (b, key/value head, key tile)
  const unsigned grid = static_cast<unsigned>(a.num_qtiles) *
                        static_cast<unsigned>(a.BH / a.H * a.Hkv);
  bwd_dkdv_kernel<D, kWithDQ, kSparse, kVarlen><<<grid, kBwdThreads, smem, st>>>(
      tq, tk, tv, tdo, tdk, tdv, a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_dkdv(int d, bool with_dq, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdArgs& a, cudaStream_t s) {
#define FA_DKDV(DD, WQ, SP, VL) launch_dkdv_d<DD, WQ, SP, VL>(tq, tk, tv, tdo, tdk, tdv, a, s)
  if (a.cu_seqlens != nullptr) {  // variable-length (not combined with a block mask)
    if (d == 64) return with_dq ? FA_DKDV(64, true, false, true) : FA_DKDV(64, false, false, true);
    return with_dq ? FA_DKDV(128, true, false, true) : FA_DKDV(128, false, false, true);
  }
  if (a.blk != nullptr) {
    if (d == 64) return with_dq ? FA_DKDV(64, true, true, false) : FA_DKDV(64, false, true, false);
    return with_dq ? FA_DKDV(128, true, true, false) : FA_DKDV(128, false, true, false);
  }
  if (d == 64) return with_dq ? FA_DKDV(64, true, false, false) : FA_DKDV(64, false, false, false);
  return with_dq ? FA_DKDV(128, true, false, false) : FA_DKDV(128, false, false, false);
#undef FA_DKDV
}

}  // namespace fa
