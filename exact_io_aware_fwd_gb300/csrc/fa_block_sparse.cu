// Block-sparse index builder: turns a uint8 block mask over 128 x 128 tiles into the sorted tile
// lists the attention kernels walk (layout: BlockIndex in fa_internal.h).  Block-sparse
// attention skips the tiles whose mask block is zero and stays exact inside the kept ones
// (page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section "FlashAttention-1：分块与在线
// softmax"; first page, section "IO 复杂度、内存复杂度与 exactness 的边界": HBM traffic
// Theta(Nd + N^2 d^2 s / M) for a fraction s of kept blocks).
//
// One warp per list: lanes test 32 tiles at a time and a ballot gives each kept tile its slot,
// so every list comes out sorted without a separate sort.
#include "fa_internal.h"

namespace fa {

namespace {

__global__ void __launch_bounds__(32) block_index_kernel(const uint8_t* __restrict__ mask, int T,
                                                         BlockIndex L, int32_t* __restrict__ index) {
  const int lane = threadIdx.x;
  const unsigned below = (1u << lane) - 1u;
  const uint8_t* m = mask + static_cast<size_t>(blockIdx.y) * T * T;
  int32_t* out = index + static_cast<size_t>(blockIdx.y) * L.words;
  const int Tb = (T + 1) / 2;
  int x = blockIdx.x;
  if (x < Tb) {
    // shared K/V stream of the 256-row query block x: union of its two query tiles' rows
    const int r0 = 2 * x, r1 = 2 * x + 1;
    int n = 0;
    for (int c = 0; c < T; c += 32) {
      const int kt = c + lane;
      const bool u0 = kt < T && m[static_cast<size_t>(r0) * T + kt] != 0;
      const bool u1 = kt < T && r1 < T && m[static_cast<size_t>(r1) * T + kt] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, u0 || u1);
      if (u0 || u1)
        out[L.fidx + static_cast<int64_t>(x) * T + n + __popc(bal & below)] =
            kt * 4 + (u0 ? 1 : 0) + (u1 ? 2 : 0);
      n += __popc(bal);
    }
    if (lane == 0) out[L.fcnt + x] = n;
    return;
  }
  x -= Tb;
  if (x < T) {
    // key tiles of query tile x, ascending
    int n = 0;
    for (int c = 0; c < T; c += 32) {
      const int kt = c + lane;
      const bool u = kt < T && m[static_cast<size_t>(x) * T + kt] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, u);
      if (u) out[L.ridx + static_cast<int64_t>(x) * T + n + __popc(bal & below)] = kt;
      n += __popc(bal);
    }
    if (lane == 0) out[L.rcnt + x] = n;
    return;
  }
  x -= T;
  // query tiles of key tile x, descending (so that "query tile >= x" is a prefix)
  int n = 0, nc = 0;
  for (int c = 0; c < T; c += 32) {
    const int i = T - 1 - (c + lane);
    const bool u = i >= 0 && m[static_cast<size_t>(i) * T + x] != 0;
    const unsigned bal = __ballot_sync(0xffffffffu, u);
    if (u) out[L.cidx + static_cast<int64_t>(x) * T + n + __popc(bal & below)] = i;
    n += __popc(bal);
    nc += __popc(__ballot_sync(0xffffffffu, u && i >= x));
  }
  if (lane == 0) {
    out[L.ccnt + x] = n;
    out[L.cccnt + x] = nc;
  }
}

}  // namespace

cudaError_t launch_block_index(const uint8_t* mask, int T, int mask_heads, int32_t* index,
                               cudaStream_t s) {
  const BlockIndex L = block_index_layout(T);
  const dim3 grid(static_cast<unsigned>((T + 1) / 2 + 2 * T), static_cast<unsigned>(mask_heads));
  block_index_kernel<<<grid, 32, 0, s>>>(mask, T, L, index);
  return cudaGetLastError();
}

}  // namespace fa
