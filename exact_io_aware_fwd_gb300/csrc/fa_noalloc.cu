// fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.
//
// Some callers have no allocator to draw the backward workspace from: code that runs where
// cudaMalloc is forbidden or unsafe (inside a host callback or an allocator hook, a plugin whose
// host framework owns every device allocation, a real-time loop that must not stall on the
// allocator), or a C caller with no device allocator at all.  For them this entry point takes the
// workspace from a fixed device array compiled into the library instead of from the caller.
//
// The array is a file-scope static __device__ buffer of kNoAllocScratchBytes.  Every GPU that
// loads the library holds it until the process exits.  In host code its name is only a host-side
// stand-in, so its device address is obtained once per device with cudaGetSymbolAddress (on the
// first call made with that device current) and handed to the kernels as a plain pointer.
//
// Behaviour:
//  * sizes whose workspace exceeds the array are rejected with FA_ERR_WORKSPACE before anything
//    is launched;
//  * no cudaMalloc, cudaFree or other allocating routine is called;
//  * every call shares the one array and it keeps the previous call's contents; the backward's
//    first stage rewrites all of it that is read later (it zeroes the dQ accumulator and rewrites
//    every per-row statistic), so stale contents never leak into a result;
//  * calls whose execution overlaps on the GPU (different streams without ordering, or several
//    host threads) race on the array and must be serialised by the caller;
//  * the first call on each device performs the address lookup; make it before any stream capture.
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device

static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The library's kernels are built for compute capability 10.3 only; on any other GPU the array
// has no device image either, so the call is refused before the address lookup.
fa_status check_device_cc() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  return (major == 10 && minor == 3) ? FA_OK : FA_ERR_UNSUPPORTED;
}

// Device address of g_bwd_scratch on the current device, looked up once per device.  A failed
// lookup is cleared from the runtime's last-error state, so that it is not reported again by a
// later, unrelated call.
void* scratch_address() {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

fa_status fa_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                         int H, int N, int d, int causal, float scale, const int32_t* kv_lens,
                         void* stream) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;  // larger than the static array
  const fa_status dev_ok = check_device_cc();
  if (dev_ok != FA_OK) return dev_ok;
  void* ws = scratch_address();
  if (ws == nullptr) return FA_ERR_CUDA;
  return fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, causal, scale, kv_lens, ws,
                kNoAllocScratchBytes, stream);
}

}  // extern "C"
