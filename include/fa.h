/*
 * Exact IO-aware attention (forward and backward) for one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation is exact scaled-dot-product attention, O = softmax(scale * Q K^T) V, computed
 * tile by tile with online-softmax running statistics so that the N x N score and probability
 * matrices never reach device memory, and its backward pass, which recomputes P from the
 * log-sum-exp saved by the forward pass.
 *   Definition:  "FlashAttention：不减少一次注意力计算，为什么反而更快", section 关键设计一
 *                (S = QK^T/sqrt(d), P = softmax(S), O = PV);
 *   recurrence:  "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section
 *                "FlashAttention-1：分块与在线 softmax", Fig. 4;
 *   backward:    first page, section 关键设计三 (D_i = dO_i . O_i, dS = P o (dP - D)).
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous [B, H, N, d] bfloat16 (the layout of torch.bfloat16 tensors of
 *     that shape), row statistics are contiguous [B, H, N] float32.  Every pointer is DEVICE
 *     memory owned by the caller and must be 16-byte aligned.  The library allocates no
 *     device memory; the backward pass takes a caller-provided workspace.
 *   - d (head dimension) is 64 or 128; N >= 1 is any length (no tile multiple needed);
 *     ceil(N / 128) * B * H <= 2^31 - 1 (one thread block per 128-row tile of every head).
 *   - scale < 0 selects the default 1/sqrt(d) (softmax_scale=None in the pages' interface,
 *     first page, section 使用契约); scale == 0 is allowed.
 *   - causal != 0 masks key j > query i.  kv_lens (DEVICE int32[B], or NULL for "all N") masks
 *     keys j >= kv_lens[b] of batch b; values are clamped to [0, N].  A query row with no
 *     unmasked key gets O = 0, LSE = -inf and zero gradients.
 *   - stream is a cudaStream_t passed as void*; NULL is the legacy default stream.  Calls are
 *     asynchronous with respect to the host.
 *   - Argument errors are returned synchronously before anything is launched.  A launch
 *     failure returns FA_ERR_CUDA.  A device-side pipeline wait that exceeds its time limit
 *     ends the kernel cleanly and records FA_ERR_TIMEOUT in a library-owned device status
 *     word, which fa_get_error() reports.
 *   - Outputs are fully overwritten; inputs are never modified.
 */
#ifndef EXACT_IO_AWARE_FA_H
#define EXACT_IO_AWARE_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, non-positive size, bad workspace size */
  FA_ERR_UNSUPPORTED = 2,  /* head dimension other than 64/128, or the GPU is not sm_103 */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a kernel launch failed */
  FA_ERR_TIMEOUT = 4,      /* a device pipeline wait ran past its limit (see fa_get_error) */
  FA_ERR_WORKSPACE = 5     /* workspace pointer NULL or smaller than fa_bwd_workspace_size() */
} fa_status;

/*
 * Forward pass.  Computes, for every (b, h):
 *   O[b,h]   = softmax(scale * Q[b,h] K[b,h]^T, masked) V[b,h]            [N, d] bf16
 *   LSE[b,h] = log sum_j exp(scale * q_i . k_j)  (natural log, masked)     [N]    fp32
 * Q, K, V: inputs [B,H,N,d] bf16.  O: output [B,H,N,d] bf16.  LSE: output [B,H,N] fp32.
 * Cite: first page, 关键设计一/二 (tiling, online softmax, L = m + log l saved for backward).
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                 int B, int H, int N, int d, int causal, float scale,
                 const int32_t* kv_lens, void* stream);

/*
 * Bytes of workspace fa_bwd needs for these sizes: a float32 dQ accumulator, the per-row
 * statistics -D = -rowsum(dO o O) and -LSE * log2(e), each padded to a multiple of 128 rows per
 * (b, h), and a 16-byte record per 128-row query tile.  Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass: dQ, dK, dV (all [B,H,N,d] bf16 outputs) of L with dL/dO = dO, given the
 * forward inputs Q, K, V, its outputs O and LSE, and the same B, H, N, d, causal, scale and
 * kv_lens.  Checks every argument, then runs the work of fa_bwd_preprocess, fa_bwd_dkdv and
 * fa_bwd_dq_convert in that order on `stream` (nothing is launched when a check fails).
 * workspace: DEVICE memory of at least fa_bwd_workspace_size() bytes, 256-byte
 * aligned, owned by the caller, contents on entry irrelevant.
 * Cite: first page, 关键设计三 (recomputation of S_ij, P_ij from the saved statistic;
 * dV += P^T dO, dQ += dS K, dK += dS^T Q).
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV,
                 int B, int H, int N, int d, int causal, float scale,
                 const int32_t* kv_lens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages of fa_bwd, exported so that each can be launched (and timed) on its own.
 * They must run in this order on one stream with the same arguments and workspace.
 *  fa_bwd_preprocess: -D_i = -sum_k dO_ik O_ik, -LSE_i * log2(e) into the workspace, and
 *                     resets every query tile's record (first page, 关键设计三,
 *                     D_i = dO_i^T O_i).  The dQ accumulator itself is not touched.
 *  fa_bwd_dkdv:       one pass over the query tiles per key tile: recomputes P^T from LSE,
 *                     writes dK, dV, and puts each key tile's partial dS K into the dQ
 *                     accumulator: the first key tile to claim a query tile (through its record)
 *                     stores its partial, the others add theirs with float32 atomics once it has
 *                     (non-deterministic in the last bits).
 *  fa_bwd_dq_convert: dQ = bf16(scale * accumulator); 0 for a query tile that no key tile
 *                     claimed (every key masked).
 */
fa_status fa_bwd_preprocess(const void* O, const void* dO, const float* LSE,
                            int B, int H, int N, int d,
                            void* workspace, size_t workspace_bytes, void* stream);
fa_status fa_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO,
                      void* dK, void* dV, int B, int H, int N, int d, int causal, float scale,
                      const int32_t* kv_lens, void* workspace, size_t workspace_bytes,
                      void* stream);
fa_status fa_bwd_dq_convert(void* dQ, int B, int H, int N, int d, float scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Deterministic backward pass: the arguments and results of fa_bwd, bit-for-bit reproducible from
 * run to run.  dK and dV accumulate per key tile in tensor memory (as in fa_bwd); dQ is computed
 * per query tile by a second kernel that recomputes S and dP and accumulates dQ over the key
 * tiles in a fixed order, instead of fp32 atomics.  More work than fa_bwd (the deterministic
 * option the pages describe for the official repository is likewise slower: page
 * "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section "反向传播：用重计算代替存储").
 * workspace: as for fa_bwd (its dQ accumulator is not used).
 */
fa_status fa_bwd_deterministic(const void* Q, const void* K, const void* V, const void* O,
                               const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                               int B, int H, int N, int d, int causal, float scale,
                               const int32_t* kv_lens, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Grouped-query attention (multi-query when Hkv == 1): H query heads share Hkv key/value heads,
 * query head h reading K and V of head h / (H / Hkv).  Q, O, dO, dQ: [B, H, N, d]; K, V, dK,
 * dV: [B, Hkv, N, d]; LSE [B, H, N]; H % Hkv == 0.  dK and dV of a key/value head sum the
 * gradients of all its query heads (accumulated in tensor memory, no atomics).  Otherwise the
 * arguments, results and workspace (fa_bwd_workspace_size(B, H, N, d)) of fa_fwd / fa_bwd;
 * deterministic != 0 as fa_bwd_deterministic.  GQA/MQA is a feature of the official library the
 * pages list (page "FlashAttention 入门：从 FA1 到 FA4 的 IO 感知注意力", section "独立 flash-attn
 * 与 PyTorch SDPA 的区别").
 */
fa_status fa_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int H, int Hkv, int N, int d, int causal, float scale,
                     const int32_t* kv_lens, void* stream);
fa_status fa_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Hkv,
                     int N, int d, int causal, float scale, const int32_t* kv_lens,
                     int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Variable-length (packed, un-padded) batches: B sequences of different lengths stored back to
 * back, as the official library's varlen interface does (same section of the same page; the
 * un-padded layout is also a headline of FlashAttention-4, section "硬件、数据类型、确定性与填充
 * 注意事项").  Sequence b is tokens [cu_seqlens[b], cu_seqlens[b + 1]) of
 *   Q, O, dO, dQ: [total, H, d] bf16;  K, V, dK, dV: [total, Hkv, d] bf16;  LSE: [H, total] fp32,
 * and attends only to itself (self-attention; the causal mask is per sequence).
 * cu_seqlens: DEVICE int32[B + 1], non-decreasing, cu_seqlens[0] = 0, cu_seqlens[B] = total
 * (offsets are clamped to [0, total]).  max_seqlen: at least the longest sequence (sizes the
 * grid; tokens beyond it are not computed).  H % Hkv == 0 (grouped-query as above).
 * Workspace: fa_bwd_varlen_workspace_size(B, total, H, d) bytes, 256-byte aligned.
 * A sequence of length 0 produces nothing; total == 0 launches nothing.
 */
fa_status fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const int32_t* cu_seqlens, int B, int max_seqlen, int total, int H,
                        int Hkv, int d, int causal, float scale, void* stream);
size_t fa_bwd_varlen_workspace_size(int B, int total, int H, int d);
fa_status fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                        const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                        const int32_t* cu_seqlens, int B, int max_seqlen, int total, int H,
                        int Hkv, int d, int causal, float scale, int deterministic,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Block-sparse attention.  A block mask over tiles of 128 queries x 128 keys keeps or drops
 * whole tiles: the scores of query i and key j count only where
 * block_mask[i / 128][j / 128] != 0 (and the causal and key-length masks keep them too); the
 * kernels skip dropped tiles entirely, so work and HBM traffic scale with the kept fraction s,
 * and the result is exact attention under that mask.  Cite: page "FlashAttention 入门：从 FA1 到
 * FA4 的 IO 感知注意力", section "FlashAttention-1：分块与在线 softmax" (the block-sparse
 * extension skips zero blocks, exact within the kept ones); first page, section "IO 复杂度、
 * 内存复杂度与 exactness 的边界" (HBM accesses Theta(Nd + N^2 d^2 s / M)).
 *
 * Use: build the block index once per mask with fa_block_index_build, then pass it to any
 * number of fa_fwd_block_sparse / fa_bwd_block_sparse calls with the same N.
 *
 * fa_block_index_size: bytes of the index for sequence length N and mask_heads masks
 *   (4 * (2 * T^2 + 3 * T + Tb * (T + 1)) bytes per mask, about 10 * T^2, with T = ceil(N / 128)
 *   and Tb = ceil(T / 2)); 0 for invalid sizes.
 * fa_block_index_build: block_mask is DEVICE uint8 [mask_heads][T][T], row = query tile,
 *   column = key tile, nonzero = kept.  index: DEVICE memory of at least
 *   fa_block_index_size(N, mask_heads) bytes, 16-byte aligned, owned by the caller; it holds the
 *   sorted lists of kept tiles the kernels walk.  Asynchronous on `stream`; the mask may be
 *   freed or changed once the build has run.  FA_ERR_WORKSPACE if index_bytes is too small.
 * fa_fwd_block_sparse / fa_bwd_block_sparse: the arguments and results of fa_fwd / fa_bwd (the
 *   backward with the same workspace) plus block_index (built for this N) and mask_heads: 1
 *   (one mask shared by every batch and head) or H (mask h for head h of every batch).
 *   deterministic != 0 makes the backward bit-reproducible as fa_bwd_deterministic does.  A
 *   query row that keeps no visible key gets O = 0, LSE = -inf and zero gradients.
 */
size_t fa_block_index_size(int N, int mask_heads);
fa_status fa_block_index_build(const uint8_t* block_mask, int N, int mask_heads, void* index,
                               size_t index_bytes, void* stream);
fa_status fa_fwd_block_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              int B, int H, int N, int d, int causal, float scale,
                              const int32_t* kv_lens, const void* block_index, int mask_heads,
                              void* stream);
fa_status fa_bwd_block_sparse(const void* Q, const void* K, const void* V, const void* O,
                              const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                              int B, int H, int N, int d, int causal, float scale,
                              const int32_t* kv_lens, const void* block_index, int mask_heads,
                              int deterministic, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * fa_bwd for callers that cannot allocate device memory.  The pages have no counterpart: this
 * entry point exists for callers with no device allocator to take the backward workspace from
 * (code running where cudaMalloc is forbidden or unsafe, such as host callbacks or allocator
 * hooks, plugins whose host framework owns every allocation, or C callers without one).
 * Arguments and results are those of fa_bwd without the workspace: the workspace is a 64 MiB
 * static device array inside the library, held by every GPU that loads the library until the
 * process exits.  Sizes with fa_bwd_workspace_size(B, H, N, d) > 64 MiB return
 * FA_ERR_WORKSPACE before anything is launched (at d = 128 that is about 129,000 padded rows
 * B * H * roundup(N, 128); at d = 64 about 254,000).  Nothing is allocated.  The first call on
 * each device looks up the array's device address with that device current; make it before
 * any stream capture.  All calls share the array: calls that overlap on the GPU race and must
 * be serialised by the caller.  Every part of the array a call reads is first written by the
 * same call (the statistics and tile records by its first stage, each accumulator tile by the
 * first key tile that contributes to it), so earlier contents never affect a result.
 */
fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                         int B, int H, int N, int d, int causal, float scale,
                         const int32_t* kv_lens, void* stream);

/*
 * Synchronises `stream`, returns the first device-side error recorded since the previous call
 * (FA_OK if none) and clears it.  A pending CUDA error on the stream gives FA_ERR_CUDA.
 */
fa_status fa_get_error(void* stream);

/* Static, NUL-terminated description of a status code. */
const char* fa_status_string(fa_status status);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_IO_AWARE_FA_H */
