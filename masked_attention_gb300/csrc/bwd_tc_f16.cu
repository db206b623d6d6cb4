// The backward's fp16 path: Q, K, V and dO converted to fp16 copies in the
// caller's workspace (recording the largest |x| of each), and the fp16
// instantiation of the dQ and dK/dV kernels (bwd_tc_kernel.cuh, F16). Whole
// tiles at position offset 0 only; bwd_tc.cu launches these before the bf16
// kernels of the same call.
#include "bwd_tc_kernel.cuh"

namespace mattn {
namespace {

struct F16Convert {
  const uint4* src[4];  // Q, K, V, dO (bf16, 8 per uint4)
  uint4* dst[4];        // their fp16 copies
  size_t n8[4];         // uint4 count of each
  unsigned* mx;         // [4] largest |x| (float bits; the record starts at 0)
};

// blockIdx.y picks the tensor; a grid-stride loop converts 8 values per step
// (bf16 -> fp32 -> fp16, round to nearest) and the block's largest |x| goes
// to the record with one atomicMax (non-negative floats order as their bits).
__global__ void to_f16_kernel(const F16Convert c) {
  const int t = blockIdx.y;
  const uint4* __restrict__ src = c.src[t];
  uint4* __restrict__ dst = c.dst[t];
  const size_t n = c.n8[t];
  float m = 0.0f;
  bool nan = false;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
      m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
      nan |= (lo != lo) | (hi != hi);
      o[e] = pack_f16x2(lo, hi);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (nan) m = INFINITY;  // a NaN input fails the range test like an infinite one
  __shared__ float wmax[32];
  for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? wmax[threadIdx.x] : 0.0f;
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    if (threadIdx.x == 0) atomicMax(c.mx + t, __float_as_uint(m));
  }
}

template <int D>
cudaError_t launch_f16_mode(const BwdProblem& bp, int mode, int score, cudaStream_t stream) {
  switch (score) {
    case 0: return launch_mode<D, 0, false, true>(bp, mode, bp.f16_max, stream);
    case 1: return launch_mode<D, 1, false, true>(bp, mode, bp.f16_max, stream);
    case 2: return launch_mode<D, 2, false, true>(bp, mode, bp.f16_max, stream);
    default: return launch_mode<D, 3, false, true>(bp, mode, bp.f16_max, stream);
  }
}

}  // namespace

cudaError_t launch_bwd_f16_prepare(const BwdProblem& bp, cudaStream_t stream) {
  const FwdProblem& f = bp.f;
  cudaError_t e = cudaMemsetAsync(bp.f16_max, 0, 4 * sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const size_t nq = (size_t)f.B * f.Hq * f.Sq * f.D / 8, nk = (size_t)f.B * f.Hkv * f.Skv * f.D / 8;
  F16Convert c;
  c.src[0] = static_cast<const uint4*>(f.q);
  c.src[1] = static_cast<const uint4*>(f.k);
  c.src[2] = static_cast<const uint4*>(f.v);
  c.src[3] = static_cast<const uint4*>(bp.dO);
  c.dst[0] = static_cast<uint4*>(bp.q16);
  c.dst[1] = static_cast<uint4*>(bp.k16);
  c.dst[2] = static_cast<uint4*>(bp.v16);
  c.dst[3] = static_cast<uint4*>(bp.do16);
  c.n8[0] = nq;
  c.n8[1] = nk;
  c.n8[2] = nk;
  c.n8[3] = nq;
  c.mx = bp.f16_max;
  to_f16_kernel<<<dim3(4 * sm_count(), 4), 256, 0, stream>>>(c);
  return cudaGetLastError();
}

cudaError_t launch_bwd_f16_mode(const BwdProblem& bp, int mode, cudaStream_t stream) {
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  return bp.f.D == 64 ? launch_f16_mode<64>(bp, mode, score, stream)
                      : launch_f16_mode<128>(bp, mode, score, stream);
}

MATTN_DEBUG_RECORD_ACCESSORS(bwd_tc_f16)

}  // namespace mattn
