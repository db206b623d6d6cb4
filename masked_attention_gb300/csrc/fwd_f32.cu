// fp32 forward on the FFMA pipes, for fp32 inputs at fp32 accuracy (tf32
// tensor-core products would miss a 1e-4 bound). One pass over the key tiles
// with the online softmax of the Online-Softmax/FlashAttention page (running
// max m, running sum l, accumulator rescaled when m grows), score_mod applied
// per element before the softmax (FlexAttention page, "FlexAttention").
//
// CTA = 64 query rows of one (b, h); two threads per row, each holding half of
// the head dimension. Keys and values stream through shared memory 32 rows at
// a time. Any Sq, Skv >= 1 is accepted (ragged tiles are bounds-checked).
#include <cmath>

#include "launch.h"

namespace mattn {
namespace {

constexpr int kRows = 64;   // query rows per CTA
constexpr int kChunk = 32;  // keys per shared-memory chunk

template <int D>
__global__ void __launch_bounds__(128) fwd_f32_kernel(FwdProblem p) {
  constexpr int DH = D / 2;
  __shared__ float sK[kChunk][D];
  __shared__ float sV[kChunk][D];

  const int bh = blockIdx.y;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int hk = h / (p.Hq / p.Hkv);
  const int q0 = blockIdx.x * kRows;
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int i = q0 + r;
  const bool row_ok = i < p.Sq;

  const float* Q = static_cast<const float*>(p.q) + ((size_t)(b * p.Hq + h) * p.Sq) * D;
  const float* K = static_cast<const float*>(p.k) + ((size_t)(b * p.Hkv + hk) * p.Skv) * D;
  const float* V = static_cast<const float*>(p.v) + ((size_t)(b * p.Hkv + hk) * p.Skv) * D;

  float q[DH], acc[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    q[d] = row_ok ? Q[(size_t)i * D + half * DH + d] : 0.0f;
    acc[d] = 0.0f;
  }
  const float slope = (p.variant & ATTN_SCORE_ALIBI) ? alibi_slope(p.score, h) : 0.0f;
  // distance-indexed bias of this head (relative position encoding), or nullptr
  const float* rb = p.score.rel_bias ? p.score.rel_bias + (size_t)h * p.score.rb_len : nullptr;
  float m = -INFINITY, l = 0.0f;

  // Which key tiles to visit: the block-mask lists of this 128-row tile, or
  // every tile up to the causal bound.
  const int qt = q0 / kTile;
  const int nkv = (p.Skv + kTile - 1) / kTile;
  int n_full, n_part;
  const int *lf = nullptr, *lp = nullptr;
  if (p.lists.full_cnt) {
    const int row = b * p.lists.nq + qt;
    n_full = p.lists.full_cnt[row];
    n_part = p.lists.part_cnt[row];
    if (!MATTN_IN_BOUNDS(kSiteF32, n_full, min(nkv, p.lists.nkv) + 1)) n_full = 0;
    if (!MATTN_IN_BOUNDS(kSiteF32, n_part, min(nkv, p.lists.nkv) + 1 - n_full)) n_part = 0;
    lf = p.lists.full_idx + (size_t)row * p.lists.nkv;
    lp = p.lists.part_idx + (size_t)row * p.lists.nkv;
  } else {
    int last = nkv;
    if ((p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX))
      last = causal_tiles(p.mask, min(q0 + kRows, p.Sq) - 1, nkv);
    n_full = (p.variant & ATTN_MASK_BITS) ? 0 : last;
    n_part = (p.variant & ATTN_MASK_BITS) ? last : 0;
  }

  for (int t = 0; t < n_full + n_part; ++t) {
    const bool partial = t >= n_full;
    int kt = partial ? (lp ? lp[t - n_full] : t - n_full) : (lf ? lf[t] : t);
    if (!MATTN_IN_BOUNDS(kSiteF32, kt, nkv)) kt = 0;
    for (int j0 = kt * kTile; j0 < min((kt + 1) * kTile, p.Skv); j0 += kChunk) {
      __syncthreads();
      for (int e = threadIdx.x; e < kChunk * D; e += 128) {
        const int jj = e / D, d = e % D;
        const bool ok = j0 + jj < p.Skv;
        sK[jj][d] = ok ? K[(size_t)(j0 + jj) * D + d] : 0.0f;
        sV[jj][d] = ok ? V[(size_t)(j0 + jj) * D + d] : 0.0f;
      }
      __syncthreads();
      float s[kChunk];
      float cmax = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kChunk; ++jj) {
        float part = 0.0f;
#pragma unroll
        for (int d = 0; d < DH; ++d) part = fmaf(q[d], sK[jj][half * DH + d], part);
        float x = (part + __shfl_xor_sync(0xffffffffu, part, 1)) * p.score.scale;
        const int j = j0 + jj;
        if (p.variant & ATTN_SCORE_ALIBI) x -= slope * float(i - j + p.mask.q_off - p.mask.kv_off);
        bool keep = row_ok && j < p.Skv;
        if (rb && keep && MATTN_IN_BOUNDS(kSiteF32, i - j + p.score.rb_zero, p.score.rb_len))
          x += rb[i - j + p.score.rb_zero];
        if (p.variant & ATTN_SCORE_SOFTCAP) x = p.score.softcap * tanhf(x / p.score.softcap);
        if (partial && keep) keep = mask_keep(p.mask, b, i, j);
        s[jj] = keep ? x : -INFINITY;
        cmax = fmaxf(cmax, s[jj]);
      }
      const float m_new = fmaxf(m, cmax);
      if (m_new == -INFINITY) continue;  // nothing kept so far
      const float corr = expf(m - m_new);  // m = -inf -> 0
      l *= corr;
#pragma unroll
      for (int d = 0; d < DH; ++d) acc[d] *= corr;
#pragma unroll
      for (int jj = 0; jj < kChunk; ++jj) {
        const float w = expf(s[jj] - m_new);
        l += w;
#pragma unroll
        for (int d = 0; d < DH; ++d) acc[d] = fmaf(w, sV[jj][half * DH + d], acc[d]);
      }
      m = m_new;
    }
  }

  if (!row_ok) return;
  float* O = static_cast<float*>(p.o) + ((size_t)(b * p.Hq + h) * p.Sq + i) * D + half * DH;
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
  for (int d = 0; d < DH; ++d) O[d] = acc[d] * inv;
  if (half == 0) p.lse[(size_t)(b * p.Hq + h) * p.Sq + i] = l > 0.0f ? m + logf(l) : -INFINITY;
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdProblem& p, cudaStream_t stream) {
  dim3 grid((p.Sq + kRows - 1) / kRows, p.B * p.Hq);
  if (p.D == 64) fwd_f32_kernel<64><<<grid, 128, 0, stream>>>(p);
  else fwd_f32_kernel<128><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(fwd_f32)
}  // namespace mattn
