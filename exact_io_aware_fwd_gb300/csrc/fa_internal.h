// Internal interface between the C-ABI layer (fa_api.cu) and the kernel translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

constexpr int kTileRows = 128;  // query rows per Q tile and keys per K/V tile

// Block-sparse index: the lists of kept 128 x 128 tiles that the kernels walk, built on the
// device from a uint8 block mask [T][T] (T = ceil(N / 128)).  int32 words per mask head:
//   fcnt[Tb]     positions of the shared K/V stream of each 256-row query block (Tb = ceil(T/2))
//   fidx[Tb][T]  key tile * 4 + 1 (kept by the block's first query tile) + 2 (by its second)
//   rcnt[T]      kept key tiles of each query tile;  ridx[T][T]  those key tiles, ascending
//   ccnt[T]      kept query tiles of each key tile;  cccnt[T]  how many of them are >= the key
//                tile (the causal prefix);  cidx[T][T]  those query tiles, descending
// Sorted lists let a kernel cut them at a key-length or causal limit by counting a prefix.
struct BlockIndex {
  int64_t fcnt, fidx, rcnt, ridx, ccnt, cccnt, cidx, words;
};
__host__ __device__ inline BlockIndex block_index_layout(int T) {
  BlockIndex L;
  const int64_t t = T, tb = (T + 1) / 2;
  L.fcnt = 0;
  L.fidx = L.fcnt + tb;
  L.rcnt = L.fidx + tb * t;
  L.ridx = L.rcnt + t;
  L.ccnt = L.ridx + t * t;
  L.cccnt = L.ccnt + t;
  L.cidx = L.cccnt + t;
  L.words = L.cidx + t * t;
  return L;
}

// Rows of one sequence in the packed variable-length layout [total, heads, d]: sequence b holds
// tokens [cu[b], cu[b+1]) (clamped to [0, total], so any offsets stay in bounds).
__host__ __device__ inline void seq_bounds(const int32_t* cu, int b, int total, int& start,
                                           int& len) {
  int s0 = cu[b], s1 = cu[b + 1];
  s0 = s0 < 0 ? 0 : (s0 > total ? total : s0);
  s1 = s1 < s0 ? s0 : (s1 > total ? total : s1);
  start = s0;
  len = s1 - s0;
}
// First 128-row tile of sequence b in the per-head variable-length workspace: ceil(start / 128)
// + b never overlaps sequence b - 1's tiles and stays below ceil(total / 128) + B.
__host__ __device__ inline int seq_tile0(int start, int b) { return (start + 127) / 128 + b; }

// Forward kernel arguments (tensor maps travel separately as __grid_constant__ parameters).
// Dense layout: [B, H, N, d] (K, V: [B, Hkv, N, d]).  Variable-length layout (cu_seqlens set):
// packed [total, H, d] (K, V: [total, Hkv, d]), N is the longest sequence.
struct FwdArgs {
  int H, N, BH;
  int Hkv;                // key/value heads: H, or a divisor of H (grouped-query attention)
  int num_qblocks;        // 256-row query blocks per (b, h)
  int head_group;         // heads scheduled together (their K/V stay resident in L2)
  int causal;
  float scale_log2;       // scale * log2(e)
  const int32_t* kv_lens; // device int32[B] or nullptr
  float* lse;             // [B, H, N] fp32 (variable-length: [H, total])
  void* o;                // O itself (variable-length: rows of a sequence's last tile)
  const int32_t* cu_seqlens;  // variable-length token offsets [B + 1], or nullptr
  int total;              // variable-length: tokens in the packed tensors
  const int32_t* blk;     // block-sparse index (BlockIndex layout) or nullptr for dense
  int blk_heads;          // mask heads in blk: 1 (shared by every head) or H
  int* status;            // library status word (device)
  uint64_t timeout_ns;    // limit of a single pipeline wait
  uint32_t smem_bytes;    // dynamic shared memory actually granted
};

// Record of one 128-row query tile of one head in fa_bwd's dQ accumulation (16 bytes, in the
// workspace; reset by the preprocess).  The key tiles that contribute a partial dQ to the tile
// coordinate through one 64-bit word: each adds 1 to it to claim the tile (the low 32 bits count
// the claims), and the first claimant, once its partial is stored into the accumulator, sets bit
// 63, after which the others add theirs.  One atomic thus tells a claimant both whether it is
// the first and whether the first one's stores are visible.  A tile nobody claimed (no key tile
// contributes) is converted as zeros.
struct DqTileCount {
  uint64_t word;
  uint64_t spare;
};
constexpr uint64_t kDqStored = 1ull << 63;  // the first claimant's partial is in the accumulator

struct BwdArgs {
  int H, N, BH;
  int Hkv;                // key/value heads (grouped-query attention when < H)
  int num_qtiles;         // ceil(N / 128) = padded rows / 128
  int ws_tiles;           // 128-row tiles per head in the workspace: num_qtiles (dense), or
                          // ceil(total / 128) + B (variable-length, see seq_tile0)
  const int32_t* cu_seqlens;  // variable-length token offsets [B + 1], or nullptr
  int total;
  void* dq;               // dQ, dK, dV themselves (variable-length: rows of a last tile)
  void* dk;
  void* dv;
  int causal;
  float scale;            // softmax scale (dK is scaled by it at the end)
  float scale_log2;       // scale * log2(e)
  const int32_t* kv_lens;
  const float* neg_lse2;  // workspace: -LSE * log2(e), [BH][Npad], -inf on padded rows
  const float* neg_delta; // workspace: -D = -rowsum(dO o O), [BH][Npad], 0 on padded rows
  float* dq_acc;          // workspace: dQ accumulator, tile-major (see fa_bwd.cu)
  DqTileCount* dq_cnt;    // workspace: per query tile records of the dQ accumulation
  const int32_t* blk;     // block-sparse index or nullptr (as in FwdArgs)
  int blk_heads;
  int* status;
  uint64_t timeout_ns;
  uint32_t smem_bytes;
};

// Workspace layout (all offsets 256-byte aligned): dq_acc | -LSE*log2(e) | -D | tile records.
// BH heads of N rows padded to 128; the variable-length workspace is
// workspace_layout(H, ws_tiles * 128, d).
struct Workspace {
  size_t dq_acc_off, neg_lse2_off, neg_delta_off, dq_cnt_off, total;
};
Workspace workspace_layout(int BH, int N, int d);

// Raises kernel K's dynamic shared-memory limit once per device (the attribute persists; setting
// it on every launch would also be a non-stream call inside a captured CUDA graph).
template <auto K>
cudaError_t ensure_smem_limit(uint32_t bytes) {
  static std::atomic<uint64_t> done{0};  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Launchers return cudaSuccess or the launch error.
cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, const FwdArgs& a, cudaStream_t s);
// recs: reset the tile records of fa_bwd's dQ accumulation, or nullptr (deterministic path)
cudaError_t launch_bwd_preprocess(int d, const void* O, const void* dO, const float* lse,
                                  int BH, int N, float* neg_lse2, float* neg_delta,
                                  DqTileCount* recs, cudaStream_t s);
// variable-length preprocess / dQ conversion: grid over (tile, b, h) of a packed batch
cudaError_t launch_bwd_preprocess_varlen(int d, const void* O, const void* dO, const float* lse,
                                         const int32_t* cu, int B, int H, int max_tiles,
                                         int total, int ws_tiles, float* neg_lse2,
                                         float* neg_delta, DqTileCount* recs, cudaStream_t s);
cudaError_t launch_bwd_dq_convert_varlen(int d, const float* dq_acc, const DqTileCount* recs,
                                         void* dQ, const int32_t* cu, int B, int H,
                                         int max_tiles, int total, int ws_tiles, float scale,
                                         cudaStream_t s);
// with_dq: also accumulate dQ in the workspace (fa_bwd); without: dK, dV only (deterministic path)
cudaError_t launch_bwd_dkdv(int d, bool with_dq, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo,
                            const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdArgs& a,
                            cudaStream_t s);
// dQ by query tile, accumulated in tensor memory in a fixed order and stored as bf16
cudaError_t launch_bwd_dq(int d, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& a, cudaStream_t s);
// block-sparse index of mask_heads masks [T][T] into `index` (mask_heads * words int32)
cudaError_t launch_block_index(const uint8_t* mask, int T, int mask_heads, int32_t* index,
                               cudaStream_t s);
cudaError_t launch_bwd_dq_convert(int d, const float* dq_acc, const DqTileCount* recs, void* dQ,
                                  int BH, int N, float scale, cudaStream_t s);

}  // namespace fa
