// attn_bwd_noalloc: the backward for callers that cannot allocate device
// memory themselves.
//
// attn_bwd needs a caller-provided fp32 workspace of B*Hq*Sq floats (the row
// terms Delta_i). Some callers have no way to get one: code inside a framework
// that owns every device allocation and forbids raw cudaMalloc, or a plug-in
// that is handed tensors but no allocator. This entry point uses a fixed
// workspace that lives in the library itself: a file-scope __device__ array of
// kMaxRows floats (8 MiB), which every GPU that loads the library keeps until
// the process exits. It calls no cudaMalloc, cudaFree or any other allocating
// routine.
//
// Set-up: the first call on a device looks up the device address of the array
// (cudaGetSymbolAddress, with that device current) and caches it; make that
// first call before any stream capture. The cached address belongs to the
// device's primary context: after cudaDeviceReset the entry point must not be
// called again in that process. All calls share the one array and it
// keeps the last call's contents; nothing in it has to start at zero (every
// call writes each Delta entry before reading it). Calls that overlap on the
// GPU (for example on two streams at once) race on the array.
#include <mutex>

#include "launch.h"

#define MATTN_API extern "C" __attribute__((visibility("default")))

namespace mattn {
namespace {

constexpr size_t kMaxRows = size_t(1) << 21;  // B*Hq*Sq <= 2,097,152 (8 MiB of fp32)

static __device__ __align__(256) float g_bwd_workspace[kMaxRows];

// Device address of the array on the current device (nullptr on failure).
float* workspace_address() {
  static float* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cuda_status(cudaGetDevice(&dev)) != ATTN_OK || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    if (cuda_status(cudaGetSymbolAddress(&ptr, g_bwd_workspace)) != ATTN_OK) return nullptr;
    addr[dev] = static_cast<float*>(ptr);
  }
  return addr[dev];
}

}  // namespace
}  // namespace mattn

MATTN_API attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                       const void* o, const float* lse, const void* dO,
                                       void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                       int Sq, int Skv, int D, unsigned variant,
                                       const attn_params* p, struct CUstream_st* stream) {
  // every argument check first: an invalid call fails without any CUDA call
  mattn::BwdProblem bp;
  const attn_status st = mattn::bwd_check_args(bp, q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv,
                                               Sq, Skv, D, variant, p);
  if (st != ATTN_OK) return st;
  if ((size_t)B * (size_t)Hq * (size_t)Sq > mattn::kMaxRows) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  float* ws = mattn::workspace_address();
  if (!ws) return ATTN_ERR_CUDA;
  // the array holds the row terms only (the exact size: never the fp16 path,
  // whose copies it has no room for)
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, ws, attn_bwd_workspace_bytes(B, Hq, Sq), B,
                  Hq, Hkv, Sq, Skv, D, variant, p, stream);
}
