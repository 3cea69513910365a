// C-ABI entry points (declared in include/fa.h): argument validation, TMA tensor-map encoding,
// kernel launches and the device status word.  Nothing here allocates device memory.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"

namespace {

__device__ int g_fa_status = 0;  // first device-side error since the last fa_get_error()

constexpr int kMaxDevices = 64;

// Per-device address of the status word (looked up once per device; calls from several host
// threads may race to look it up, and all of them store the same value).
int* status_ptr() {
  static std::atomic<int*> ptrs[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* cached = ptrs[dev].load(std::memory_order_acquire);
  if (cached != nullptr) return cached;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
  ptrs[dev].store(static_cast<int*>(p), std::memory_order_release);
  return static_cast<int*>(p);
}

// Limit of a single pipeline wait in the kernels, read at every call so that a process can
// change it between calls: FA_WAIT_TIMEOUT_US (microseconds) if set to a positive value, else
// FA_WAIT_TIMEOUT_MS (milliseconds), else 2 s.  A wait is normally a few microseconds; a limit
// below that makes a normal launch give up with FA_ERR_TIMEOUT, which is how the kernels' timeout
// paths are exercised without a fault.  (The waits a CTA makes for its own copies and MMAs before
// it exits keep a limit of at least 1 s, whatever this is.)
uint64_t wait_timeout_ns() {
  if (const char* e = std::getenv("FA_WAIT_TIMEOUT_US")) {
    const long long v = std::strtoll(e, nullptr, 10);
    if (v > 0) return static_cast<uint64_t>(v) * 1000ull;
  }
  if (const char* e = std::getenv("FA_WAIT_TIMEOUT_MS")) {
    const long long v = std::strtoll(e, nullptr, 10);
    if (v > 0) return static_cast<uint64_t>(v) * 1000000ull;
  }
  return 2000ull * 1000000ull;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {  // looked up once, thread-safely
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// [B*H][N][d] bf16 viewed as a 3-D tensor (d, N, B*H); boxes of 64 x 128 x 1 elements with the
// 128-byte swizzle.  Rows past N are out of bounds: zero-filled on load, dropped on store.
bool make_tile_map(CUtensorMap* m, const void* base, int BH, int N, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed variable-length [total][heads][d] bf16 viewed as a 3-D tensor (d, heads, total); boxes
// of 64 x 1 x 128 elements (128 consecutive tokens of one head), same smem image as a tile map's
// box.  Tokens past `total` are zero-filled on load and dropped on store.
bool make_packed_map(CUtensorMap* m, const void* base, int total, int heads, int d) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(total)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_sizes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  // 128-row tiles of every (b, h) must be addressable with 32-bit coordinates, and one block per
  // (b, h, 128-row tile) must fit a 1-D grid (at most 2^31 - 1 blocks)
  if (N > (1 << 30)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>((N + 127) / 128) * B * H > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

float resolve_scale(float scale, int d) {
  return (scale < 0.f) ? 1.0f / std::sqrt(static_cast<float>(d)) : scale;
}

constexpr float kLog2e = 1.4426950408889634f;

// The kernels are built for sm_103a only (compute capability 10.3); on any other GPU no image
// would load, so the call is refused before any launch.
fa_status check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  return (major == 10 && minor == 3) ? FA_OK : FA_ERR_UNSUPPORTED;
}

fa_status check_workspace(void* ws, size_t bytes, size_t need) {
  if (ws == nullptr) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return FA_ERR_INVALID_ARG;
  if (bytes < need) return FA_ERR_WORKSPACE;
  return FA_OK;
}

// One attention problem as every entry point describes it.
struct Problem {
  int B, H, Hkv, N, d;  // N: sequence length (variable-length: the longest sequence)
  int causal;
  float scale;
  const int32_t* kv_lens;     // dense key lengths [B] or nullptr
  const int32_t* cu_seqlens;  // variable-length token offsets [B + 1] or nullptr
  int total;                  // variable-length: tokens in the packed tensors
  const int32_t* blk;         // block-sparse index or nullptr
  int blk_heads;
  bool varlen() const { return cu_seqlens != nullptr; }
  int ws_tiles() const {  // 128-row workspace tiles per workspace head
    return varlen() ? (total + 127) / 128 + B : (N + 127) / 128;
  }
  fa::Workspace workspace() const {
    return varlen() ? fa::workspace_layout(H, ws_tiles() * 128, d)
                    : fa::workspace_layout(B * H, N, d);
  }
};

fa_status check_problem(const Problem& p) {
  fa_status st = check_sizes(p.B, p.H, p.N, p.d);
  if (st != FA_OK) return st;
  if (p.Hkv <= 0 || p.H % p.Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(p.scale)) return FA_ERR_INVALID_ARG;
  if (p.varlen()) {
    if (p.total < 0 || p.kv_lens != nullptr || p.blk != nullptr) return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(p.total) + 128LL * (p.B + 1) > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    if (static_cast<long long>(p.H) * p.ws_tiles() * 128 > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    // (N here is the longest sequence; check_sizes bounded its tiles x B x H)
  }
  if (p.blk != nullptr && p.Hkv != p.H) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Tensor map of a [.., rows, d] tensor with `heads` heads: dense [B][heads][N][d] or packed
// [total][heads][d].
bool map_of(CUtensorMap* m, const void* base, const Problem& p, int heads) {
  return p.varlen() ? make_packed_map(m, base, p.total, heads, p.d)
                    : make_tile_map(m, base, p.B * heads, p.N, p.d);
}

fa_status fwd_impl(const Problem& p, const void* Q, const void* K, const void* V, void* O,
                   float* LSE, void* stream) {
  fa_status st = check_problem(p);
  if (st != FA_OK) return st;
  if (p.varlen() && p.total == 0) return FA_OK;  // no tokens (empty tensors may be NULL)
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  int* status = status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  const int BH = p.B * p.H, d = p.d, N = p.N;
  CUtensorMap tq, tk, tv, to;
  if (!map_of(&tq, Q, p, p.H) || !map_of(&tk, K, p, p.Hkv) || !map_of(&tv, V, p, p.Hkv) ||
      !map_of(&to, O, p, p.H))
    return FA_ERR_CUDA;
  fa::FwdArgs a{};
  a.H = p.H;
  a.N = N;
  a.BH = BH;
  a.Hkv = p.Hkv;
  a.num_qblocks = (N + 255) / 256;
  {
    // heads whose K and V (2 * N * d bf16 each) fit in 64 MB, about half of the 129 MB L2
    const long long kv_bytes = 4LL * N * d;
    const long long g = (64LL << 20) / (kv_bytes > 0 ? kv_bytes : 1);
    a.head_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  }
  a.causal = p.causal ? 1 : 0;
  a.scale_log2 = resolve_scale(p.scale, d) * kLog2e;
  a.kv_lens = p.kv_lens;
  a.lse = LSE;
  a.o = O;
  a.cu_seqlens = p.cu_seqlens;
  a.total = p.total;
  a.blk = p.blk;
  a.blk_heads = p.blk_heads;
  a.status = status;
  a.timeout_ns = wait_timeout_ns();
  if (static_cast<long long>(a.num_qblocks) * BH > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  cudaError_t e = fa::launch_fwd(d, tq, tk, tv, to, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status check_block_index(const void* index, int mask_heads, int H) {
  if (index == nullptr || (reinterpret_cast<uintptr_t>(index) & 15u) != 0) return FA_ERR_INVALID_ARG;
  if (mask_heads != 1 && mask_heads != H) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Validation, tensor maps and arguments shared by the backward kernels.
struct BwdSetup {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
  fa::BwdArgs a{};
};

fa_status bwd_setup(BwdSetup& st, const Problem& p, const void* Q, const void* K, const void* V,
                    const void* dO, void* dK, void* dV, void* dQ, void* workspace,
                    size_t workspace_bytes) {
  fa_status rc = check_problem(p);
  if (rc != FA_OK) return rc;
  if (!Q || !K || !V || !dO || !dK || !dV) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dK) ||
      !aligned16(dV) || (dQ && !aligned16(dQ)))
    return FA_ERR_INVALID_ARG;
  const fa::Workspace w = p.workspace();
  if ((rc = check_workspace(workspace, workspace_bytes, w.total)) != FA_OK) return rc;
  if ((rc = check_device()) != FA_OK) return rc;
  int* status = status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  if (!map_of(&st.tq, Q, p, p.H) || !map_of(&st.tk, K, p, p.Hkv) ||
      !map_of(&st.tv, V, p, p.Hkv) || !map_of(&st.tdo, dO, p, p.H) ||
      !map_of(&st.tdk, dK, p, p.Hkv) || !map_of(&st.tdv, dV, p, p.Hkv) ||
      (dQ && !map_of(&st.tdq, dQ, p, p.H)))
    return FA_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  fa::BwdArgs& a = st.a;
  a.H = p.H;
  a.N = p.N;
  a.BH = p.B * p.H;
  a.Hkv = p.Hkv;
  a.num_qtiles = (p.N + 127) / 128;
  a.ws_tiles = p.ws_tiles();
  a.cu_seqlens = p.cu_seqlens;
  a.total = p.total;
  a.dq = dQ;
  a.dk = dK;
  a.dv = dV;
  a.causal = p.causal ? 1 : 0;
  a.scale = resolve_scale(p.scale, p.d);
  a.scale_log2 = a.scale * kLog2e;
  a.kv_lens = p.kv_lens;
  a.neg_lse2 = reinterpret_cast<const float*>(ws + w.neg_lse2_off);
  a.neg_delta = reinterpret_cast<const float*>(ws + w.neg_delta_off);
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc_off);
  a.dq_cnt = reinterpret_cast<fa::DqTileCount*>(ws + w.dq_cnt_off);
  a.blk = p.blk;
  a.blk_heads = p.blk_heads;
  a.status = status;
  a.timeout_ns = wait_timeout_ns();
  if (static_cast<long long>(a.num_qtiles) * a.BH > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Every fused backward entry point: preprocess, then either the dK/dV kernel with the dQ
// accumulation and the dQ conversion, or (deterministic) the dK/dV kernel without dQ and the
// per-query-tile dQ kernel.
fa_status bwd_impl(const Problem& p, const void* Q, const void* K, const void* V, const void* O,
                   const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                   void* workspace, size_t workspace_bytes, bool deterministic, void* stream) {
  fa_status rc = check_problem(p);
  if (rc != FA_OK) return rc;
  if (p.varlen() && p.total == 0) return FA_OK;  // no tokens (empty tensors may be NULL)
  if (!O || !LSE || !dQ || !aligned16(O)) return FA_ERR_INVALID_ARG;
  BwdSetup st;
  rc = bwd_setup(st, p, Q, K, V, dO, dK, dV, dQ, workspace, workspace_bytes);
  if (rc != FA_OK) return rc;
  const fa::Workspace w = p.workspace();
  char* ws = static_cast<char*>(workspace);
  float* neg_lse2 = reinterpret_cast<float*>(ws + w.neg_lse2_off);
  float* neg_delta = reinterpret_cast<float*>(ws + w.neg_delta_off);
  float* acc = reinterpret_cast<float*>(ws + w.dq_acc_off);
  fa::DqTileCount* recs = reinterpret_cast<fa::DqTileCount*>(ws + w.dq_cnt_off);
  fa::DqTileCount* reset = deterministic ? nullptr : recs;  // the deterministic path has none
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int max_tiles = (p.N + 127) / 128;
  cudaError_t e =
      p.varlen() ? fa::launch_bwd_preprocess_varlen(p.d, O, dO, LSE, p.cu_seqlens, p.B, p.H,
                                                    max_tiles, p.total, p.ws_tiles(), neg_lse2,
                                                    neg_delta, reset, s)
                 : fa::launch_bwd_preprocess(p.d, O, dO, LSE, p.B * p.H, p.N, neg_lse2, neg_delta,
                                             reset, s);
  if (e == cudaSuccess)
    e = fa::launch_bwd_dkdv(p.d, /*with_dq=*/!deterministic, st.tq, st.tk, st.tv, st.tdo, st.tdk,
                            st.tdv, st.a, s);
  if (e == cudaSuccess) {
    if (deterministic)
      e = fa::launch_bwd_dq(p.d, st.tq, st.tk, st.tv, st.tdo, st.tdq, st.a, s);
    else if (p.varlen())
      e = fa::launch_bwd_dq_convert_varlen(p.d, acc, recs, dQ, p.cu_seqlens, p.B, p.H,
                                           max_tiles, p.total, p.ws_tiles(), st.a.scale, s);
    else
      e = fa::launch_bwd_dq_convert(p.d, acc, recs, dQ, p.B * p.H, p.N, st.a.scale, s);
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

Problem dense_problem(int B, int H, int Hkv, int N, int d, int causal, float scale,
                      const int32_t* kv_lens) {
  Problem p{};
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.N = N;
  p.d = d;
  p.causal = causal;
  p.scale = scale;
  p.kv_lens = kv_lens;
  p.blk_heads = 1;
  return p;
}

Problem varlen_problem(const int32_t* cu_seqlens, int B, int max_seqlen, int total, int H,
                       int Hkv, int d, int causal, float scale) {
  Problem p = dense_problem(B, H, Hkv, max_seqlen, d, causal, scale, nullptr);
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  return p;
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK) return 0;
  return fa::workspace_layout(B * H, N, d).total;
}

fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int N, int d, int causal, float scale, const int32_t* kv_lens, void* stream) {
  return fwd_impl(dense_problem(B, H, H, N, d, causal, scale, kv_lens), Q, K, V, O, LSE, stream);
}

fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                     int H, int Hkv, int N, int d, int causal, float scale,
                     const int32_t* kv_lens, void* stream) {
  return fwd_impl(dense_problem(B, H, Hkv, N, d, causal, scale, kv_lens), Q, K, V, O, LSE,
                  stream);
}

fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const int32_t* cu_seqlens, int B, int max_seqlen, int total, int H,
                        int Hkv, int d, int causal, float scale, void* stream) {
  if (cu_seqlens == nullptr) return FA_ERR_INVALID_ARG;
  return fwd_impl(varlen_problem(cu_seqlens, B, max_seqlen, total, H, Hkv, d, causal, scale), Q,
                  K, V, O, LSE, stream);
}

size_t fa_block_index_size(int N, int mask_heads) {
  if (N <= 0 || N > (1 << 30) || mask_heads <= 0 || mask_heads > 65535) return 0;
  return static_cast<size_t>(mask_heads) *
         static_cast<size_t>(fa::block_index_layout((N + 127) / 128).words) * sizeof(int32_t);
}

fa_status fa_block_index_build(const uint8_t* block_mask, int N, int mask_heads, void* index,
                               size_t index_bytes, void* stream) {
  if (block_mask == nullptr || index == nullptr) return FA_ERR_INVALID_ARG;
  const size_t need = fa_block_index_size(N, mask_heads);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(index) & 15u) != 0) return FA_ERR_INVALID_ARG;
  if (index_bytes < need) return FA_ERR_WORKSPACE;
  fa_status st = check_device();
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_block_index(block_mask, (N + 127) / 128, mask_heads,
                                         static_cast<int32_t*>(index),
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_block_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              int B, int H, int N, int d, int causal, float scale,
                              const int32_t* kv_lens, const void* block_index, int mask_heads,
                              void* stream) {
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_block_index(block_index, mask_heads, H)) != FA_OK) return st;
  Problem p = dense_problem(B, H, H, N, d, causal, scale, kv_lens);
  p.blk = static_cast<const int32_t*>(block_index);
  p.blk_heads = mask_heads;
  return fwd_impl(p, Q, K, V, O, LSE, stream);
}

fa_status fa_bwd_preprocess(const void* O, const void* dO, const float* LSE, int B, int H, int N,
                            int d, void* workspace, size_t workspace_bytes, void* stream) {
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if (!O || !dO || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(O) || !aligned16(dO)) return FA_ERR_INVALID_ARG;
  const int BH = B * H;
  const fa::Workspace w = fa::workspace_layout(BH, N, d);
  if ((st = check_workspace(workspace, workspace_bytes, w.total)) != FA_OK) return st;
  if ((st = check_device()) != FA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = fa::launch_bwd_preprocess(
      d, O, dO, LSE, BH, N, reinterpret_cast<float*>(ws + w.neg_lse2_off),
      reinterpret_cast<float*>(ws + w.neg_delta_off),
      reinterpret_cast<fa::DqTileCount*>(ws + w.dq_cnt_off), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                      void* dV, int B, int H, int N, int d, int causal, float scale,
                      const int32_t* kv_lens, void* workspace, size_t workspace_bytes,
                      void* stream) {
  BwdSetup st;
  fa_status rc = bwd_setup(st, dense_problem(B, H, H, N, d, causal, scale, kv_lens), Q, K, V, dO,
                           dK, dV, nullptr, workspace, workspace_bytes);
  if (rc != FA_OK) return rc;
  cudaError_t e = fa::launch_bwd_dkdv(d, /*with_dq=*/true, st.tq, st.tk, st.tv, st.tdo, st.tdk,
                                      st.tdv, st.a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd_dq_convert(void* dQ, int B, int H, int N, int d, float scale, void* workspace,
                            size_t workspace_bytes, void* stream) {
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if (!dQ || !aligned16(dQ)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const int BH = B * H;
  const fa::Workspace w = fa::workspace_layout(BH, N, d);
  if ((st = check_workspace(workspace, workspace_bytes, w.total)) != FA_OK) return st;
  if ((st = check_device()) != FA_OK) return st;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = fa::launch_bwd_dq_convert(
      d, reinterpret_cast<const float*>(ws + w.dq_acc_off),
      reinterpret_cast<const fa::DqTileCount*>(ws + w.dq_cnt_off), dQ, BH, N,
      resolve_scale(scale, d), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int d,
                 int causal, float scale, const int32_t* kv_lens, void* workspace,
                 size_t workspace_bytes, void* stream) {
  // every argument is checked before the first of the three launches
  return bwd_impl(dense_problem(B, H, H, N, d, causal, scale, kv_lens), Q, K, V, O, dO, LSE, dQ,
                  dK, dV, workspace, workspace_bytes, /*deterministic=*/false, stream);
}

fa_status fa_bwd_deterministic(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                               int B, int H, int N, int d, int causal, float scale,
                               const int32_t* kv_lens, void* workspace, size_t workspace_bytes,
                               void* stream) {
  return bwd_impl(dense_problem(B, H, H, N, d, causal, scale, kv_lens), Q, K, V, O, dO, LSE, dQ,
                  dK, dV, workspace, workspace_bytes, /*deterministic=*/true, stream);
}

fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Hkv, int N,
                     int d, int causal, float scale, const int32_t* kv_lens, int deterministic,
                     void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(dense_problem(B, H, Hkv, N, d, causal, scale, kv_lens), Q, K, V, O, dO, LSE,
                  dQ, dK, dV, workspace, workspace_bytes, deterministic != 0, stream);
}

size_t fa_bwd_varlen_workspace_size(int B, int total, int H, int d) {
  if (B <= 0 || H <= 0 || total < 0 || (d != 64 && d != 128)) return 0;
  const long long rows = (static_cast<long long>(total + 127) / 128 + B) * 128;  // per head
  if (static_cast<long long>(H) * rows > 0x7fffffffLL) return 0;
  return fa::workspace_layout(H, static_cast<int>(rows), d).total;
}

fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                        const int32_t* cu_seqlens, int B, int max_seqlen, int total, int H,
                        int Hkv, int d, int causal, float scale, int deterministic,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (cu_seqlens == nullptr) return FA_ERR_INVALID_ARG;
  return bwd_impl(varlen_problem(cu_seqlens, B, max_seqlen, total, H, Hkv, d, causal, scale), Q,
                  K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes, deterministic != 0,
                  stream);
}

fa_status fa_bwd_block_sparse(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                              int B, int H, int N, int d, int causal, float scale,
                              const int32_t* kv_lens, const void* block_index, int mask_heads,
                              int deterministic, void* workspace, size_t workspace_bytes,
                              void* stream) {
  fa_status rc = check_sizes(B, H, N, d);
  if (rc != FA_OK) return rc;
  if ((rc = check_block_index(block_index, mask_heads, H)) != FA_OK) return rc;
  Problem p = dense_problem(B, H, H, N, d, causal, scale, kv_lens);
  p.blk = static_cast<const int32_t*>(block_index);
  p.blk_heads = mask_heads;
  return bwd_impl(p, Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, workspace_bytes,
                  deterministic != 0, stream);
}

fa_status fa_get_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  int* status = status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  switch (v) {
    case 0: return FA_OK;
    case 4: return FA_ERR_TIMEOUT;
    default: return FA_ERR_CUDA;
  }
}

}  // extern "C"
