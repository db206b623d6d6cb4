// Jagged batches (FlexAttention page, variant list: irregular ("jagged")
// tensors next to document masking): n sequences packed back to back with no
// padding, described by cumulative lengths cu_seqlens[0..n] (cu[0] = 0,
// nondecreasing, cu[n] = total). Attention within each sequence and not
// across them is the document mask over the packed positions, so this file
// only turns cu_seqlens into per-position document ids; the forward,
// backward and block mask then run unchanged with B = 1 and S = total.
#include <cuda_runtime.h>

#include "mattn.h"
#include "status.h"

#define MATTN_API extern "C" __attribute__((visibility("default")))

namespace mattn {
namespace {

// doc_id[p] = the s with cu[s] <= p < cu[s + 1] (binary search over cu).
__global__ void seqlens_to_doc_kernel(const int* __restrict__ cu, int n, int total,
                                      int* __restrict__ doc_id) {
  for (int pos = blockIdx.x * blockDim.x + threadIdx.x; pos < total;
       pos += gridDim.x * blockDim.x) {
    int lo = 0, hi = n - 1;  // find the last s with cu[s] <= pos
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= pos) lo = mid;
      else hi = mid - 1;
    }
    doc_id[pos] = lo;
  }
}

}  // namespace
}  // namespace mattn

MATTN_API attn_status attn_doc_ids_from_seqlens(const int* cu_seqlens, int n, int total,
                                                int* doc_id, struct CUstream_st* stream) {
  if (n < 1 || total < 0) return ATTN_ERR_INVALID_ARG;
  if (total == 0) return ATTN_OK;
  if (!cu_seqlens || !doc_id) return ATTN_ERR_INVALID_ARG;
  const int threads = 256;
  int blocks = (total + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  mattn::seqlens_to_doc_kernel<<<blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      cu_seqlens, n, total, doc_id);
  return mattn::cuda_status(cudaGetLastError());
}
