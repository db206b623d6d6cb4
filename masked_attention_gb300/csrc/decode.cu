// Decode against a key/value cache (FlexAttention page, variant list:
// PagedAttention, alone and with a sliding window): a few new query rows per
// sequence attend to a long cache of keys and values, contiguous or paged.
// The work is bound by HBM: every key and value row has to be read once,
// and per key there are only 2 * D products per query row.
//
// A CTA takes one (batch element, key/value head) and one split of the key
// range. The query rows of all query heads of the GQA group that share the
// key/value head (group * Sq <= 16 rows) form one 16-row tile, so each key
// and value row is read once for all of them. Four warps stream blocks of 16
// keys through per-warp double-buffered shared memory (cp.async, rows padded
// to D * 2 + 16 bytes so the fragment loads hit distinct banks) and run the
// products on the warp-level tensor-core instruction (mma.sync m16n8k16,
// bf16 in, fp32 accumulate): S = Q K^T, then the online softmax of the
// Online-Softmax/FlashAttention page on S (running maximum and sum per row,
// accumulator rescaled when the maximum grows), then O += P V with P taken
// from the S accumulators as the next product's A operand. Every mask term
// and score modification is evaluated per element (FlexAttention page,
// score_mod applied before the softmax). The four warps' partial states
// merge in shared memory; across splits, fp32 partial results in the
// caller's workspace are merged by the online-softmax merge
// (LSE = ln sum e^LSE_k, O = sum e^(LSE_k - LSE) O_k).
#include <cmath>
#include <mutex>

#include "host_util.h"
#include "launch.h"

namespace mattn {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = 4;
constexpr int kBlk = 16;    // keys per warp step
constexpr int kStages = 2;  // per-warp K/V double buffer

template <int D>
struct DecCfg {
  static constexpr int kRowBytes = D * 2 + 16;        // padded shared-memory row
  static constexpr int kBlkBytes = kBlk * kRowBytes;  // a block of 16 K or V rows
  static constexpr int kWarpBytes = kStages * 2 * kBlkBytes;
  // after the key loop a warp's area holds its m, l (16 each) and O (16 x D) in fp32
  static_assert(kWarpBytes >= (2 * 16 + 16 * D) * 4, "merge state fits the warp area");
  static constexpr int kSmem = kDecWarps * kWarpBytes;
};

// 16-byte asynchronous copy; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16) B (16x8 bf16)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Per-row constants of a thread's two rows (r = lane / 4 and r + 8).
struct DecRow {
  bool valid;      // r < group * Sq
  int i;           // query row of the call
  int pos;         // absolute position q_offset + i
  int doc;         // document id at pos
  float slope2;    // ALiBi slope of the row's head, log2 units
  const float* rb; // relative-bias table of the row's head, or nullptr
};

template <int D, int SCORE>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeProblem dp) {
  using C = DecCfg<D>;
  const FwdProblem& p = dp.f;
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int b = blockIdx.y / p.Hkv, hkv = blockIdx.y % p.Hkv;
  const int group = p.Hq / p.Hkv;
  const int R = group * p.Sq;                                // rows of this CTA (<= 16)
  const size_t row0 = (size_t)(b * p.Hq + hkv * group) * p.Sq;  // first Q / O / LSE row
  const unsigned mbits = p.variant & ATTN_MASK_BITS;
  const int* docb = (mbits & ATTN_MASK_DOCUMENT) ? p.mask.doc_id + (size_t)b * p.mask.doc_len
                                                 : nullptr;
  const int P = (mbits & ATTN_MASK_PREFIX) ? p.mask.prefix_len[b] : INT_MIN;

  // key range of this split, narrowed by the causal and window bounds when
  // no prefix term can keep keys outside them
  const int split_lo = dp.k_begin + split * dp.chunk;
  const int split_hi = min(dp.k_end, split_lo + dp.chunk);
  int k_lo = split_lo, k_hi = split_hi;
  if (!(mbits & ATTN_MASK_PREFIX)) {
    if (mbits & ATTN_MASK_CAUSAL) k_hi = min(k_hi, p.mask.q_off + p.Sq - p.mask.kv_off);
    if (mbits & ATTN_MASK_WINDOW)
      k_lo = max(k_lo, p.mask.q_off - p.mask.window + 1 - p.mask.kv_off);
  }
  k_lo = max(k_lo, 0) & ~(kBlk - 1);

  // the thread's rows
  DecRow rw[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = (lane >> 2) + 8 * h2;
    DecRow& d = rw[h2];
    d.valid = r < R;
    const int g = d.valid ? r / p.Sq : 0;
    d.i = d.valid ? r % p.Sq : 0;
    d.pos = p.mask.q_off + d.i;
    const int h = hkv * group + g;
    d.doc = (docb && MATTN_IN_BOUNDS(kSiteDecSide, d.pos, p.mask.doc_len)) ? docb[d.pos] : 0;
    d.slope2 = (SCORE & 1) ? alibi_slope(p.score, h) * kLog2e : 0.0f;
    d.rb = (SCORE & 4) ? p.score.rel_bias + (size_t)h * p.score.rb_len : nullptr;
  }

  // Q fragments (A operand, 16 rows x D), rows past R are 0
  const __nv_bfloat16* Q = static_cast<const __nv_bfloat16*>(p.q) + row0 * D;
  const size_t total_rows = (size_t)p.B * p.Hq * p.Sq;
  uint32_t qa[D / 16][4];
  {
    const int r0 = lane >> 2, c0 = 2 * (lane & 3);
    auto qpair = [&](int r, int c) -> uint32_t {  // Q[r][c], Q[r][c + 1] of this CTA's rows
      if (r >= R || !MATTN_IN_BOUNDS(kSiteDecQ, (row0 + r) * D + c, total_rows * D)) return 0u;
      return *reinterpret_cast<const uint32_t*>(Q + (size_t)r * D + c);
    };
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c = 16 * kk + c0;
      qa[kk][0] = qpair(r0, c);
      qa[kk][1] = qpair(r0 + 8, c);
      qa[kk][2] = qpair(r0, c + 8);
      qa[kk][3] = qpair(r0 + 8, c + 8);
    }
  }

  // key and value rows: contiguous [B][Hkv][Skv][D] or page pools
  // [num_pages][Hkv][page][D]. A 16-key block lies within one page (pages
  // hold a multiple of 16 keys), so a block takes one page-table entry; the
  // entry of the block a warp loads next is read one step ahead, off the
  // copy's critical path. Rows past Skv repeat the last key (masked); a page
  // index outside [0, num_pages) reads as zeros (nothing is read).
  const __nv_bfloat16* Kb = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* Vb = static_cast<const __nv_bfloat16*>(p.v);
  const int kb_first = k_lo / kBlk + warp, kb_end = (k_hi + kBlk - 1) / kBlk;
  auto page_of = [&](int kb) -> int {  // physical page of key block kb (< kb_end), or -1
    if (!p.page_table || kb >= kb_end) return 0;
    const int lp = (kb * kBlk) / p.page_size;
    if (!MATTN_IN_BOUNDS(kSiteDecTable, lp, p.pages_per_seq)) return -1;
    const int pg = p.page_table[(size_t)b * p.pages_per_seq + lp];
    return (pg >= 0 && pg < p.num_pages) ? pg : -1;
  };
  const size_t kv_elems = p.page_table ? (size_t)p.num_pages * p.Hkv * p.page_size * D
                                       : (size_t)p.B * p.Hkv * p.Skv * D;
  (void)kv_elems;
  const uint32_t warea = static_cast<uint32_t>(__cvta_generic_to_shared(smem)) + warp * C::kWarpBytes;
  auto load_block = [&](int kb, int stage, int pg) {
    const uint32_t kdst = warea + stage * 2 * C::kBlkBytes;
    const uint32_t vdst = kdst + C::kBlkBytes;
    constexpr int kChunks = kBlk * D / 8;  // 16-byte pieces per block
#pragma unroll
    for (int c = lane; c < kChunks; c += 32) {
      const int kr = c / (D / 8), kc = c % (D / 8);
      const int j = min(kb * kBlk + kr, p.Skv - 1);
      size_t off;
      bool ok = true;
      if (p.page_table) {
        ok = pg >= 0;
        off = ok ? (((size_t)pg * p.Hkv + hkv) * p.page_size + (j & (p.page_size - 1))) * D : 0;
      } else {
        off = (((size_t)b * p.Hkv + hkv) * p.Skv + j) * D;
      }
      off += kc * 8;
      if (!MATTN_IN_BOUNDS(kSiteDecKV, off / 8, kv_elems / 8)) {
        ok = false;
        off = 0;
      }
      cp_async16(kdst + kr * C::kRowBytes + kc * 16, Kb + off, ok ? 16u : 0u);
      cp_async16(vdst + kr * C::kRowBytes + kc * 16, Vb + off, ok ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
  const float sl2 = p.score.scale * kLog2e;

  if (kb_first < kb_end) load_block(kb_first, 0, page_of(kb_first));
  if (kb_first + kDecWarps < kb_end) load_block(kb_first + kDecWarps, 1, page_of(kb_first + kDecWarps));
  int stage = 0;
  for (int kb = kb_first; kb < kb_end; kb += kDecWarps, stage ^= 1) {
    const int pg_next = page_of(kb + 2 * kDecWarps);
    if (kb + kDecWarps < kb_end) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncwarp();
    const uint32_t kbuf = warea + stage * 2 * C::kBlkBytes, vbuf = kbuf + C::kBlkBytes;
    // S = Q K^T for 16 keys: two 8-key n-tiles
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int key = ((lane >> 4) << 3) + (lane & 7);
      const int col = 16 * kk + (((lane >> 3) & 1) << 3);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbuf + key * C::kRowBytes + col * 2, b0, b1, b2, b3);
      mma16816(s[0], qa[kk], b0, b1);
      mma16816(s[1], qa[kk], b2, b3);
    }
    // score_mod and mask per element, in log2 units; masked -> -inf
    const int j0 = kb * kBlk;
    float t[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const DecRow& rr = rw[e >> 1];
        const int j = j0 + 8 * nt + 2 * (lane & 3) + (e & 1);
        const int pk = p.mask.kv_off + j;
        float x = s[nt][e] * sl2;
        if constexpr ((SCORE & 1) != 0) x -= rr.slope2 * float(rr.pos - pk);
        if constexpr ((SCORE & 4) != 0) {
          if (rr.valid && j < p.Skv &&
              MATTN_IN_BOUNDS(kSiteDecSide, rr.i - j + p.score.rb_zero, p.score.rb_len))
            x += rr.rb[rr.i - j + p.score.rb_zero] * kLog2e;
        }
        if constexpr ((SCORE & 2) != 0)
          x = p.score.softcap * kLog2e * tanhf(x / (p.score.softcap * kLog2e));
        bool keep = rr.valid && j >= split_lo && j < split_hi;
        bool and_terms = true;
        if (mbits & ATTN_MASK_CAUSAL) and_terms = and_terms && pk <= rr.pos;
        if (mbits & ATTN_MASK_WINDOW) and_terms = and_terms && rr.pos - pk < p.mask.window;
        if (docb)
          and_terms = and_terms && (j < p.Skv && MATTN_IN_BOUNDS(kSiteDecSide, pk, p.mask.doc_len)
                                        ? docb[pk] == rr.doc
                                        : false);
        keep = keep && (and_terms || pk < P);
        t[nt][e] = keep ? x : -INFINITY;
      }
    // online softmax per row (a row's 16 scores sit in one quad of lanes)
    float corr[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float mx = fmaxf(fmaxf(t[0][2 * h2], t[0][2 * h2 + 1]), fmaxf(t[1][2 * h2], t[1][2 * h2 + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m[h2], mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      corr[h2] = ex2_approx(m[h2] - m_use);  // -inf -> 0
      m[h2] = m_new;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        t[nt][2 * h2] = ex2_approx(t[nt][2 * h2] - m_use);
        t[nt][2 * h2 + 1] = ex2_approx(t[nt][2 * h2 + 1] - m_use);
      }
      l[h2] = l[h2] * corr[h2] + t[0][2 * h2] + t[0][2 * h2 + 1] + t[1][2 * h2] + t[1][2 * h2 + 1];
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= corr[0];
      o[n][1] *= corr[0];
      o[n][2] *= corr[1];
      o[n][3] *= corr[1];
    }
    // P (bf16) as the A operand: the S accumulator layout is the A layout
    const uint32_t pa[4] = {pack_bf16x2(t[0][0], t[0][1]), pack_bf16x2(t[0][2], t[0][3]),
                            pack_bf16x2(t[1][0], t[1][1]), pack_bf16x2(t[1][2], t[1][3])};
    // O += P V: V rows (keys) as the k dimension, transposed fragment loads
#pragma unroll
    for (int n = 0; n < D / 8; n += 2) {
      const int key = (((lane >> 3) & 1) << 3) + (lane & 7);
      const int col = 8 * (n + (lane >> 4));
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbuf + key * C::kRowBytes + col * 2, b0, b1, b2, b3);
      mma16816(o[n], pa, b0, b1);
      mma16816(o[n + 1], pa, b2, b3);
    }
    __syncwarp();
    if (kb + 2 * kDecWarps < kb_end) load_block(kb + 2 * kDecWarps, stage, pg_next);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncwarp();

  // row sums over the quad, then the four warps' states meet in shared memory
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 1);
    l[h2] += __shfl_xor_sync(0xffffffffu, l[h2], 2);
  }
  float* wm = reinterpret_cast<float*>(smem + warp * C::kWarpBytes);
  float* wl = wm + 16;
  float* wo = wm + 32;  // [16][D]
  if ((lane & 3) == 0) {
    wm[lane >> 2] = m[0];
    wm[(lane >> 2) + 8] = m[1];
    wl[lane >> 2] = l[0];
    wl[(lane >> 2) + 8] = l[1];
  }
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    const int c = 8 * n + 2 * (lane & 3), r = lane >> 2;
    wo[r * D + c] = o[n][0];
    wo[r * D + c + 1] = o[n][1];
    wo[(r + 8) * D + c] = o[n][2];
    wo[(r + 8) * D + c + 1] = o[n][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 16 * D; idx += kDecThreads) {
    const int r = idx / D, c = idx % D;
    if (r >= R) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(smem + w * C::kWarpBytes)[r]);
    float L = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float* a = reinterpret_cast<const float*>(smem + w * C::kWarpBytes);
        const float wt = ex2_approx(a[r] - M);  // -inf -> 0
        L += wt * a[16 + r];
        acc += wt * a[32 + r * D + c];
      }
    }
    const float out = L > 0.0f ? acc / L : 0.0f;
    const float lse = L > 0.0f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    if (!MATTN_IN_BOUNDS(kSiteDecOut, row0 + r, total_rows)) continue;
    if (dp.ws_o) {  // a split's partial result, fp32
      if (!MATTN_IN_BOUNDS(kSiteDecOut, split, dp.splits)) continue;
      dp.ws_o[((size_t)split * total_rows + row0 + r) * D + c] = out;
      if (c == 0) dp.ws_lse[(size_t)split * total_rows + row0 + r] = lse;
    } else {
      static_cast<__nv_bfloat16*>(p.o)[(row0 + r) * D + c] = __float2bfloat16_rn(out);
      if (c == 0) p.lse[row0 + r] = lse;
    }
  }
}

template <int D, int SCORE>
cudaError_t launch_typed(const DecodeProblem& dp, cudaStream_t stream) {
  using C = DecCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_kernel<D, SCORE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const dim3 grid(dp.splits, dp.f.B * dp.f.Hkv);
  decode_kernel<D, SCORE><<<grid, kDecThreads, C::kSmem, stream>>>(dp);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecodeProblem& dp, cudaStream_t s) {
  const unsigned v = dp.f.variant;
  const int score = ((v & ATTN_SCORE_ALIBI) ? 1 : 0) | ((v & ATTN_SCORE_SOFTCAP) ? 2 : 0) |
                    ((v & ATTN_SCORE_RELBIAS) ? 4 : 0);
  switch (score) {
    case 0: return launch_typed<D, 0>(dp, s);
    case 1: return launch_typed<D, 1>(dp, s);
    case 2: return launch_typed<D, 2>(dp, s);
    case 3: return launch_typed<D, 3>(dp, s);
    case 4: return launch_typed<D, 4>(dp, s);
    case 5: return launch_typed<D, 5>(dp, s);
    case 6: return launch_typed<D, 6>(dp, s);
    default: return launch_typed<D, 7>(dp, s);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem& dp, cudaStream_t stream) {
  return dp.f.D == 64 ? launch_d<64>(dp, stream) : launch_d<128>(dp, stream);
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(decode)
}  // namespace mattn
