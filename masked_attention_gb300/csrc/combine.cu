// Merge of partial attention results over disjoint key sets, such as the
// key/value shards of context-parallel attention (FlexAttention page, variant
// list: sliding window + document masking + causal + context parallel). The
// rule is the merge step of the online softmax (Online-Softmax/FlashAttention
// page, 2-pass online softmax: partial maxima and sums combine with
// exponential weights) applied to whole results, each normalised by its own
// sum:  LSE = ln sum_k exp(LSE_k),  O = sum_k exp(LSE_k - LSE) O_k.
//
// Bound by HBM: per row it reads the parts' O rows and LSE values and writes
// one O row and one LSE. One warp per row; lane l holds D/32 consecutive
// elements, so each part's row is one coalesced warp access. A part whose LSE
// is -inf (no kept key there) has weight 0 and its row is not read.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "mattn.h"
#include "status.h"

#define MATTN_API extern "C" __attribute__((visibility("default")))

namespace mattn {
namespace {

constexpr int kCombineThreads = 256;

template <int E, bool kBf16>
struct RowIo;

template <int E>
struct RowIo<E, true> {  // bf16: E elements = E * 2 bytes per lane
  static __device__ __forceinline__ void load(const void* base, size_t off, float* x) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(
        static_cast<const __nv_bfloat16*>(base) + off);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float2 f = __bfloat1622float2(p[e]);
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(void* base, size_t off, const float* x) {
    __nv_bfloat162* p =
        reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int e = 0; e < E / 2; ++e) p[e] = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
  }
};

template <int E>
struct RowIo<E, false> {  // fp32
  static __device__ __forceinline__ void load(const void* base, size_t off, float* x) {
    const float* p = static_cast<const float*>(base) + off;
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = p[e];
  }
  static __device__ __forceinline__ void store(void* base, size_t off, const float* x) {
    float* p = static_cast<float*>(base) + off;
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = x[e];
  }
};

template <int D, bool kBf16>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const void* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                   long long rows, void* __restrict__ o, float* __restrict__ lse) {
  constexpr int E = D / 32;
  using Io = RowIo<E, kBf16>;
  const int lane = threadIdx.x & 31;
  const long long wpb = kCombineThreads / 32;
  const long long step = (long long)gridDim.x * wpb;
  for (long long r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += step) {
    // the largest part LSE, then the sum of the weights relative to it
    float m = -INFINITY;
    for (int k = lane; k < n; k += 32) m = fmaxf(m, lse_parts[(size_t)k * rows + r]);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.0f;
    float out_lse = -INFINITY;
    if (m != -INFINITY) {
      float tot = 0.0f;
      for (int k = lane; k < n; k += 32) {
        const float lk = lse_parts[(size_t)k * rows + r];
        tot += lk == -INFINITY ? 0.0f : expf(lk - m);
      }
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
      const float inv = 1.0f / tot;
      for (int k = 0; k < n; ++k) {
        const float lk = lse_parts[(size_t)k * rows + r];  // one address: a broadcast
        if (lk == -INFINITY) continue;
        const float w = expf(lk - m) * inv;
        float x[E];
        Io::load(o_parts, ((size_t)k * rows + r) * D + lane * E, x);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, x[e], acc[e]);
      }
      out_lse = m + logf(tot);
    }
    Io::store(o, (size_t)r * D + lane * E, acc);
    if (lane == 0) lse[r] = out_lse;
  }
}

template <int D, bool kBf16>
cudaError_t launch_combine(const void* o_parts, const float* lse_parts, int n, long long rows,
                           void* o, float* lse, cudaStream_t s) {
  const long long wpb = kCombineThreads / 32;
  long long blocks = (rows + wpb - 1) / wpb;
  if (blocks > 152 * 8) blocks = 152 * 8;  // grid-stride over the rows
  combine_kernel<D, kBf16><<<(unsigned)blocks, kCombineThreads, 0, s>>>(o_parts, lse_parts, n,
                                                                       rows, o, lse);
  return cudaGetLastError();
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace
}  // namespace mattn

MATTN_API attn_status attn_combine(const void* o_parts, const float* lse_parts, int n_parts,
                                   long long rows, int D, int dtype, void* o, float* lse,
                                   struct CUstream_st* stream) {
  using namespace mattn;
  if (n_parts < 1 || rows < 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_UNSUPPORTED;
  if (rows == 0) return ATTN_OK;
  if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(o_parts) | reinterpret_cast<uintptr_t>(o);
  const uintptr_t a4 = reinterpret_cast<uintptr_t>(lse_parts) | reinterpret_cast<uintptr_t>(lse);
  if ((a16 & 15) || (a4 & 3)) return ATTN_ERR_MISALIGNED;
  const size_t elem = dtype == ATTN_F32 ? 4 : 2;
  const size_t row_bytes = elem * (size_t)D;
  if (overlaps(o, row_bytes * rows, o_parts, row_bytes * rows * n_parts) ||
      overlaps(lse, 4 * (size_t)rows, lse_parts, 4 * (size_t)rows * n_parts) ||
      overlaps(o, row_bytes * rows, lse_parts, 4 * (size_t)rows * n_parts) ||
      overlaps(lse, 4 * (size_t)rows, o_parts, row_bytes * rows * n_parts))
    return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == ATTN_BF16)
    e = D == 64 ? launch_combine<64, true>(o_parts, lse_parts, n_parts, rows, o, lse, s)
                : launch_combine<128, true>(o_parts, lse_parts, n_parts, rows, o, lse, s);
  else
    e = D == 64 ? launch_combine<64, false>(o_parts, lse_parts, n_parts, rows, o, lse, s)
                : launch_combine<128, false>(o_parts, lse_parts, n_parts, rows, o, lse, s);
  return mattn::cuda_status(e);
}
