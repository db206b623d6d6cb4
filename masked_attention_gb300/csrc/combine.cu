// Merge of partial attention results over disjoint key sets, such as the
// key/value shards of context-parallel attention (FlexAttention page, variant
// list: sliding window + document masking + causal + context parallel). The
// rule is the merge step of the online softmax (Online-Softmax/FlashAttention
// page, 2-pass online softmax: partial maxima and sums combine with
// exponential weights) applied to whole results, each normalised by its own
// sum:  LSE = ln sum_k exp(LSE_k),  O = sum_k exp(LSE_k - LSE) O_k.
//
// Bound by HBM: per row it reads the parts' O rows and LSE values and writes
// one O row and one LSE. Each lane moves 16 bytes of a row (a row of D
// elements takes D * size / 16 lanes, so a warp merges 1 to 4 rows at once),
// and the loads of up to eight parts are issued before any of them is used,
// so many loads per lane are in flight. A part whose weight is 0 (LSE_k =
// -inf: no kept key there) is not read. The grid is one resident wave
// (occupancy times the SM count), striding over the rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "host_util.h"
#include "launch.h"

#define MATTN_API extern "C" __attribute__((visibility("default")))

namespace mattn {
namespace {

constexpr int kCombineThreads = 256;

// 16 bytes of a row: 8 bf16 or 4 fp32 elements.
template <bool kBf16>
__device__ __forceinline__ void unpack16(const uint4& v, float* x) {
  if constexpr (kBf16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] = __uint_as_float(w[e] << 16);
      x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
  } else {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
}

template <bool kBf16>
__device__ __forceinline__ uint4 pack16(const float* x) {
  if constexpr (kBf16) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
}

// NP: parts the kernel is built for (2, 4 or 8, n <= NP; 0: any n, in
// chunks of 8). A lane keeps 8 loads of 16 bytes in flight (4 for two
// parts): G = 8 / NP row groups of the warp (2 for two parts), each with its
// NP parts, per pass. (Measured on the merge of 2 to 8 parts of 262,144 rows
// at D = 128: 8 loads per lane beat 4 at 3 and 4 parts by 15-25 % and lost
// to it by 5 % at 2 parts; loading the first pass's part rows before their
// LSEs are known was 10-40 % slower.)
template <int D, bool kBf16, int NP, bool kOutBf16 = kBf16>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const void* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                   long long rows, void* __restrict__ o, float* __restrict__ lse) {
  constexpr int kElem = kBf16 ? 2 : 4;
  constexpr int kLanesPerRow = D * kElem / 16;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  constexpr int kVec = 16 / kElem;  // elements per lane
  constexpr int P = NP == 0 ? 8 : NP;
  constexpr int G = P == 2 ? 2 : 8 / P;  // row groups per pass
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, sl = lane % kLanesPerRow;
  const long long nwarps = (long long)gridDim.x * (kCombineThreads / 32);
  const long long w0 = ((long long)blockIdx.x * kCombineThreads + threadIdx.x) >> 5;
  const uint4* parts = static_cast<const uint4*>(o_parts);
  const size_t vec_per_row = (size_t)kLanesPerRow;
  const long long stride = nwarps * kRowsPerWarp * G;
  // merged row g of a pass: normalise, store the row and its LSE
  auto finish = [&](const long long (&r)[G], const float (&m)[G], const float (&tot)[G],
                    float (&acc)[G][kVec]) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (r[g] >= rows || !MATTN_IN_BOUNDS(kSiteCombineOut, r[g], rows)) continue;
      const bool any = tot[g] > 0.0f;
      const float inv = any ? 1.0f / tot[g] : 0.0f;
#pragma unroll
      for (int e = 0; e < kVec; ++e) acc[g][e] *= inv;
      if constexpr (kOutBf16 && !kBf16) {  // fp32 parts, bf16 output: 4 elements, 8 bytes
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[g][0], acc[g][1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[g][2], acc[g][3]);
        static_cast<uint2*>(o)[(size_t)r[g] * vec_per_row + sl] =
            make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
      } else {
        static_cast<uint4*>(o)[(size_t)r[g] * vec_per_row + sl] = pack16<kBf16>(acc[g]);
      }
      if (sl == 0) lse[r[g]] = any ? m[g] + logf(tot[g]) : -INFINITY;
    }
  };

  if constexpr (NP != 0) {
    // n <= NP: one round of loads per pass. The LSEs of the next pass are
    // loaded while this pass's part rows are in flight, so the part loads
    // (issued only for parts of nonzero weight) wait on no LSE round trip.
    float lnext[G][P];
    auto load_lse = [&](long long base) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int u = 0; u < P; ++u) {
          const long long rr = base + (long long)g * kRowsPerWarp + sub;
          lnext[g][u] = (u < n && rr < rows &&
                         MATTN_IN_BOUNDS(kSiteCombineIn, (long long)u * rows + rr, (long long)n * rows))
                            ? __ldg(lse_parts + (size_t)u * rows + rr)
                            : -INFINITY;
        }
    };
    long long rb = w0 * kRowsPerWarp * G;
    if (rb < rows) load_lse(rb);
    for (; rb < rows; rb += stride) {
      long long r[G];
      float m[G], tot[G], acc[G][kVec], w[G][P];
      uint4 raw[G][P];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        r[g] = rb + (long long)g * kRowsPerWarp + sub;
        m[g] = -INFINITY;
#pragma unroll
        for (int u = 0; u < P; ++u) m[g] = fmaxf(m[g], lnext[g][u]);
#pragma unroll
        for (int u = 0; u < P; ++u) {
          w[g][u] = (lnext[g][u] == -INFINITY) ? 0.0f : expf(lnext[g][u] - m[g]);
          raw[g][u] = w[g][u] > 0.0f && MATTN_IN_BOUNDS(kSiteCombineIn,
                                                         (long long)u * rows + r[g],
                                                         (long long)n * rows)
                          ? __ldcs(parts + ((size_t)u * rows + r[g]) * vec_per_row + sl)
                          : make_uint4(0, 0, 0, 0);
        }
      }
      if (rb + stride < rows) load_lse(rb + stride);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        tot[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[g][e] = 0.0f;
#pragma unroll
        for (int u = 0; u < P; ++u) {
          tot[g] += w[g][u];
          float x[kVec];
          unpack16<kBf16>(raw[g][u], x);
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc[g][e] = fmaf(w[g][u], x[e], acc[g][e]);
        }
      }
      finish(r, m, tot, acc);
    }
  } else {
    // any n: the parts in chunks of 8, the largest LSE of each row first
    for (long long rb = w0 * kRowsPerWarp * G; rb < rows; rb += stride) {
      long long r[G];
      float m[G], tot[G], acc[G][kVec];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        r[g] = rb + (long long)g * kRowsPerWarp + sub;
        m[g] = -INFINITY;
        tot[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < kVec; ++e) acc[g][e] = 0.0f;
      }
      for (int k = 0; k < n; ++k)
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (r[g] < rows && MATTN_IN_BOUNDS(kSiteCombineIn, (long long)k * rows + r[g],
                                             (long long)n * rows))
            m[g] = fmaxf(m[g], lse_parts[(size_t)k * rows + r[g]]);
      for (int k0 = 0; k0 < n; k0 += P) {
        float w[G][P];
        uint4 raw[G][P];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int u = 0; u < P; ++u) {
            const int k = k0 + u;
            const float lk = (k < n && r[g] < rows &&
                              MATTN_IN_BOUNDS(kSiteCombineIn, (long long)k * rows + r[g],
                                              (long long)n * rows))
                                 ? lse_parts[(size_t)k * rows + r[g]]
                                 : -INFINITY;
            w[g][u] = (lk == -INFINITY || m[g] == -INFINITY) ? 0.0f : expf(lk - m[g]);
            raw[g][u] = w[g][u] > 0.0f ? parts[((size_t)k * rows + r[g]) * vec_per_row + sl]
                                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int u = 0; u < P; ++u) {
            tot[g] += w[g][u];
            float x[kVec];
            unpack16<kBf16>(raw[g][u], x);
#pragma unroll
            for (int e = 0; e < kVec; ++e) acc[g][e] = fmaf(w[g][u], x[e], acc[g][e]);
          }
      }
      finish(r, m, tot, acc);
    }
  }
}

template <int D, bool kBf16, int NP, bool kOutBf16 = kBf16>
cudaError_t launch_np(const void* o_parts, const float* lse_parts, int n, long long rows,
                      void* o, float* lse, cudaStream_t s) {
  constexpr int kRowsPerWarp = 32 / (D * (kBf16 ? 2 : 4) / 16);
  constexpr int G = NP == 2 ? 2 : 8 / (NP == 0 ? 8 : NP);
  const long long rows_per_block = (long long)(kCombineThreads / 32) * kRowsPerWarp * G;
  long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  static int per_sm = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<D, kBf16, NP, kOutBf16>,
                                                      kCombineThreads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  });
  const long long resident = (long long)sm_count() * per_sm;
  if (blocks > resident) blocks = resident;  // one resident wave, grid-stride over the rows
  combine_kernel<D, kBf16, NP, kOutBf16><<<(unsigned)blocks, kCombineThreads, 0, s>>>(
      o_parts, lse_parts, n, rows, o, lse);
  return cudaGetLastError();
}

template <int D, bool kBf16>
cudaError_t launch_combine(const void* o_parts, const float* lse_parts, int n, long long rows,
                           void* o, float* lse, cudaStream_t s) {
  if (n <= 2) return launch_np<D, kBf16, 2>(o_parts, lse_parts, n, rows, o, lse, s);
  if (n <= 4) return launch_np<D, kBf16, 4>(o_parts, lse_parts, n, rows, o, lse, s);
  if (n <= 8) return launch_np<D, kBf16, 8>(o_parts, lse_parts, n, rows, o, lse, s);
  return launch_np<D, kBf16, 0>(o_parts, lse_parts, n, rows, o, lse, s);
}

template <int D>
cudaError_t launch_f32_bf16(const float* o_parts, const float* lse_parts, int n, long long rows,
                            void* o, float* lse, cudaStream_t s) {
  if (n <= 2) return launch_np<D, false, 2, true>(o_parts, lse_parts, n, rows, o, lse, s);
  if (n <= 4) return launch_np<D, false, 4, true>(o_parts, lse_parts, n, rows, o, lse, s);
  if (n <= 8) return launch_np<D, false, 8, true>(o_parts, lse_parts, n, rows, o, lse, s);
  return launch_np<D, false, 0, true>(o_parts, lse_parts, n, rows, o, lse, s);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

cudaError_t launch_combine_f32_bf16(const float* o_parts, const float* lse_parts, int n_parts,
                                    long long rows, int D, void* o, float* lse,
                                    cudaStream_t stream) {
  return D == 64 ? launch_f32_bf16<64>(o_parts, lse_parts, n_parts, rows, o, lse, stream)
                 : launch_f32_bf16<128>(o_parts, lse_parts, n_parts, rows, o, lse, stream);
}

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

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(combine)
}  // namespace mattn
