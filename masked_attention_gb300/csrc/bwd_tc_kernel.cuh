// Backward on the tensor cores (tcgen05, TMEM, TMA).
//
// The FlexAttention page ("Performance" section) describes a deterministic
// backward that recomputes intermediates rather than storing them; this one
// recomputes the probabilities from the forward's LSE and uses no atomics, so
// reruns are bitwise identical:
//
//   delta_kernel   an estimate Dhat_i = <dO_i, O_i> from the bf16 output O
//   bwd_kernel<dQ> per (b, h, query tile), over its key tiles:
//                  S = Q K^T, P = exp(score_mod(S) - LSE), dP = dO V^T, and
//                  the exact Delta_i = sum_j P dP (it equals <dO_i, O_i> for
//                  the exact O; the bf16 O is off by up to an ulp, which on
//                  rows with few keys moves dQ by ~1e-2), accumulated on the fly:
//                  A += (P g (dP - Dhat)) K, B += bf16(P g) K,
//                  dQ = scale (A - (Delta - Dhat) B), g = score_mod'.
//                  A carries the well-conditioned bulk (like dS itself), the
//                  correction term is small. Delta goes to the workspace.
//   bwd_kernel<dKV> per (b, kv head, key tile), over the query heads of its
//                  group and the query tiles of the transposed block mask:
//                  S^T = K Q^T, P^T, dV += P^T dO, dP^T = V dO^T,
//                  dS^T = P^T (dP^T - Delta) score_mod', dK += dS^T Q (x scale)
//
// Precision. The products P^T dO, dS^T Q and (P g (dP - Dhat)) K take their
// first operand from TMEM in bf16. Rounding it once costs up to 2^-9 of each
// term, which on rows and keys with few dominant terms moves a gradient of
// magnitude 2..4 by several 1e-3: together with the final rounding of the
// output to bf16 (up to 0.0078 there) that exceeds 1e-2. Each of these
// operands is therefore split into a bf16 part and the bf16 rounding of its
// remainder, x = hi + lo, and both parts are multiplied (two products into
// the same accumulator): the error of hi + lo is about 2^-17 of x. The soft-
// cap's tanh is evaluated to fp32 accuracy for the same reason (an odd
// polynomial for small arguments, tanhf otherwise).
//
// Both kernels share one structure (384 threads):
//   warps 0-7  compute, two warpgroups: thread t of warpgroup g owns row
//              t % 128 of the fixed tile (TMEM lane) and columns
//              [64 g, 64 g + 64) of each streamed tile
//   warp  8    TMA producer: the fixed tiles once per unit, then the streamed
//              tiles (plus LSE, Delta and document ids of the dKV stream) into
//              a ring
//   warp  9    MMA issuer and TMEM owner
//   warps 10-11 idle (the rest of the third warpgroup)
// Tensor memory: S [0,128), dP [128,256), accumulators from 256 (dQ: A, B;
// dKV: dV, dK). The bf16 operands of the TS products are written over the
// S and dP columns their warpgroup has read: warpgroup g's 64 columns hold
// its 32 columns of hi parts, then its 32 columns of lo parts (dQ: P g over
// S, the lo part of A beside it, the hi part of A over dP).
//
// Product order per streamed tile j (the tensor pipe runs them in order):
//   dKV: dV += P_j^T dO (hi, lo) | S_{j+1} | dK += dS_j^T Q (hi, lo) | dP_{j+1}
//   dQ:  B += (P g)_j K, A += lo_j K | S_{j+1} | A += hi_j K | dP_{j+1}
// so the next tile's S is computed while the compute warps still work on the
// current tile's dS (dKV). In dQ's bf16 path the lo part of A sits over S, so
// B waits for dS too; with fp16 operands (no lo part) B follows P g at once:
//   dQ fp16: B += (P g)_j K | S_{j+1} | A += dS_j K | dP_{j+1}
#pragma once

#include <cmath>
#include <cuda_fp16.h>
#include <mutex>

#include "host_util.h"
#include "launch.h"

namespace mattn {
namespace {

constexpr int kThreads = 384;
constexpr int kComputeWarps = 8;
// Registers: the CTA is launched with 168 per thread (384 x 168 = 64512 of the
// SM's 65536); the third warpgroup (producer, MMA, two idle warps) gives up
// most of its share to the compute warps, which hold 64 scores, their P g and
// the packed operands of a tile half: 256 x 208 + 128 x 88 = 64512.
constexpr int kRegsCompute = 208;
constexpr int kRegsOther = 88;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
enum Mode { kDQ = 0, kDKV = 1 };

template <int D, int MODE>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kSlots = D == 128 ? 2 : 4;
  // extra bytes per slot: doc ids, LSE and Delta of the streamed rows (the
  // last two for dKV), 1024-aligned so the next slot's tiles stay aligned
  static constexpr int kSlotExtra = 2048;
  static constexpr int kSlotBytes = 2 * kTileBytes + kSlotExtra;
  static constexpr int kOffFix = 0;
  static constexpr int kOffSlots = 2 * kTileBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kSlotBytes;
  // fix_full, fix_empty, s_full, dp_full, p_full, ds_full, acc_done, acc_free,
  // drain, dx_full, then per slot and half (0: Q or K with the extras, 1: dO
  // or V) full[2][kSlots] and empty[2][kSlots]
  static constexpr int kNumBars = 10 + 4 * kSlots;
  // per-row partial sums of Delta of the two warpgroups, double-buffered
  static constexpr int kOffDx = (kOffBars + kNumBars * 8 + 15) & ~15;
  static constexpr int kOffMisc = kOffDx + 2 * 2 * kTile * 4;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr uint32_t kColAcc = 256;
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
};

struct BwdArgs {
  FwdProblem f;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  const float* delta;  // Delta, read by the dKV kernel
  float* delta_out;    // Delta, written by the dQ kernel (same buffer)
  BlockLists lists;    // forward lists (dQ) or transposed lists (dKV)
  // fp16 path: the largest |x| of Q, K, V, dO (float bits; written by the
  // conversion to fp16) decides between the fp16 kernels and the bf16 ones,
  // which are both launched and of which one returns at once; nullptr: no
  // fp16 copies, the bf16 kernels run
  const unsigned* f16_max;
};

// One unit of work and its iteration list.
struct BUnit {
  int b, h;      // dQ: query head; dKV: kv head
  int tile;      // dQ: query tile; dKV: key tile
  int n_full, n_part, group;  // per head of the group (dKV) or total (dQ)
  const int* lf;
  const int* lp;
  int n_inner;  // tiles of the streamed dimension (the debug build checks list entries)
  __device__ __forceinline__ int n() const { return (n_full + n_part) * group; }
  // iteration -> (head offset within group, streamed tile index, partial?)
  __device__ __forceinline__ void at(int it, int& hoff, int& t, bool& partial) const {
    const int m = n_full + n_part;
    hoff = it / m;
    const int j = it % m;
    partial = j >= n_full;
    t = j < n_full ? (lf ? lf[j] : j) : (lp ? lp[j - n_full] : j - n_full);
    if (!MATTN_IN_BOUNDS(kSiteBwdList, t, n_inner)) t = 0;
  }
};

template <int MODE, bool GENERAL>
__device__ __forceinline__ BUnit decode_bwd(const BwdArgs& a, int u) {
  const FwdProblem& p = a.f;
  const int nq = GENERAL ? (p.Sq + kTile - 1) / kTile : p.Sq / kTile;
  const int nkv = GENERAL ? (p.Skv + kTile - 1) / kTile : p.Skv / kTile;
  // without a block mask the causal tile bound holds only at offset 0 (else
  // every tile is visited and masked element by element)
  const bool at_zero = !GENERAL || (p.mask.q_off == 0 && p.mask.kv_off == 0);
  const int heads = MODE == kDQ ? p.Hq : p.Hkv;
  const int rank = u / heads, h = u % heads;
  const int n_outer = MODE == kDQ ? nq : nkv;
  const int n_inner = MODE == kDQ ? nkv : nq;
  const bool causal_bound =
      (p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX) && at_zero;
  int row;
  if (a.lists.full_cnt) {
    row = a.lists.order[rank];
    if (!MATTN_IN_BOUNDS(kSiteBwdList, row, p.B * n_outer)) row = 0;
  } else if (causal_bound)  // longest first: dQ large query tiles first, dKV small key tiles first
    row = MODE == kDQ ? (rank % p.B) * nq + (nq - 1 - rank / p.B) : rank;  // dKV by batch element
  else row = rank;
  BUnit U;
  U.b = row / n_outer;
  U.tile = row % n_outer;
  U.h = h;
  U.group = MODE == kDQ ? 1 : p.Hq / p.Hkv;
  if (a.lists.full_cnt) {
    U.n_full = a.lists.full_cnt[row];
    U.n_part = a.lists.part_cnt[row];
    U.lf = a.lists.full_idx + (size_t)row * n_inner;
    U.lp = a.lists.part_idx + (size_t)row * n_inner;
    if (!MATTN_IN_BOUNDS(kSiteBwdList, U.n_full, n_inner + 1)) U.n_full = 0;
    if (!MATTN_IN_BOUNDS(kSiteBwdList, U.n_part, n_inner + 1 - U.n_full)) U.n_part = 0;
  } else {
    int first = 0, last = n_inner;
    if (causal_bound) {
      if (MODE == kDQ) last = min(n_inner, U.tile + 1);
      else first = min(U.tile, n_inner);
    }
    const bool masked = (p.variant & ATTN_MASK_BITS) != 0;
    U.n_full = masked ? 0 : last - first;
    U.n_part = masked ? last - first : 0;
    U.lf = U.lp = nullptr;  // dense: tiles first .. last-1 (first > 0 only for the causal dKV bound)
  }
  U.n_inner = n_inner;
  return U;
}

template <int MODE, bool GENERAL>
__device__ __forceinline__ int dense_first(const BwdArgs& a, const BUnit& U) {
  const FwdProblem& p = a.f;
  const bool at_zero = !GENERAL || (p.mask.q_off == 0 && p.mask.kv_off == 0);
  const bool causal_bound =
      (p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX) && at_zero;
  return (!a.lists.full_cnt && MODE == kDKV && causal_bound) ? U.tile : 0;
}

__global__ void delta_kernel(const __nv_bfloat16* __restrict__ o,
                             const __nv_bfloat16* __restrict__ dO, float* __restrict__ delta,
                             size_t rows, int D) {
  const size_t row = (size_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat16* a = o + row * D;
  const __nv_bfloat16* b = dO + row * D;
  float acc = 0.0f;
  for (int d = 2 * lane; d < D; d += 64) {
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(a + d));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(b + d));
    acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) delta[row] = acc;
}

// tanh of 16 values in place to fp32 accuracy: the odd Taylor series of
// tanh at 0 through y^9 where every |y| of the warp's group is at most 1/4
// (the first omitted term, 1382 y^11 / 155925, is below 9e-9 of tanh y
// there), tanhf otherwise. The choice is uniform over the warp.
__device__ __forceinline__ void tanh16(float (&y)[16]) {
  float m = 0.0f;
#pragma unroll
  for (int c = 0; c < 16; c += 2) m = fmax3(m, fabsf(y[c]), fabsf(y[c + 1]));
  if (__all_sync(0xffffffffu, m <= 0.25f)) {
    const float2 c3 = make_float2(-1.0f / 3.0f, -1.0f / 3.0f);
    const float2 c5 = make_float2(2.0f / 15.0f, 2.0f / 15.0f);
    const float2 c7 = make_float2(-17.0f / 315.0f, -17.0f / 315.0f);
    const float2 c9 = make_float2(62.0f / 2835.0f, 62.0f / 2835.0f);
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const float2 v = make_float2(y[c], y[c + 1]);
      const float2 v2 = fmul2(v, v);
      float2 u = ffma2(v2, c9, c7);
      u = ffma2(v2, u, c5);
      u = ffma2(v2, u, c3);
      u = fmul2(u, v2);
      const float2 t = ffma2(v, u, v);
      y[c] = t.x;
      y[c + 1] = t.y;
    }
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) y[c] = tanhf(y[c]);
  }
}

// tcgen05 instruction descriptor with fp16 A and B (format fields 0; the
// bf16 one sets them to 1).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major) {
  return idesc_bf16(M, N, b_mn_major) & ~((1u << 7) | (1u << 10));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

// The bf16 pair of (a, b) and the bf16 pair of their rounding remainders:
// hi + lo represents a and b to about 2^-17 of their magnitude.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  const float2 h = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
  const float2 r = ffma2(h, make_float2(-1.0f, -1.0f), make_float2(a, b));
  lo = pack_bf16x2(r.x, r.y);
}

// TMEM column (within a 128-column S or dP block) of the 8 packed columns
// that hold K-step kk (16 streamed rows) of a split operand: warpgroup kk / 4
// wrote its hi parts at 64 (kk / 4) and its lo parts 32 columns further.
__device__ __forceinline__ uint32_t hi_col(int kk) { return 64u * (kk >> 2) + 8u * (kk & 3); }

// D(tmem) += A(tmem, 8 K-steps at hi_col + extra) * B(smem, MN-major), K = 128.
// b_desc: descriptor of the B tile's first row; K-step kk advances 16 rows =
// 2048 bytes (the start-address field counts 16-byte units). Called by the
// whole (converged) MMA warp; lane 0 issues (mma_ts_warp).
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_base, uint32_t extra,
                                         uint64_t b_desc, uint32_t idesc, bool accumulate) {
  uint32_t a[8];
  uint64_t b[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    a[kk] = a_base + hi_col(kk) + extra;
    b[kk] = b_desc + (uint64_t)(kk * 128);
  }
  mma_ts_warp<8>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// D(tmem) = A(smem) * B(smem)^T over D (both K-major): K-step kk advances 32
// bytes inside a 64-column box and moves to the next box every 4 steps.
// Called by the whole MMA warp.
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc) {
  constexpr int K = D / 16;
  uint64_t a[K], b[K];
#pragma unroll
  for (int kk = 0; kk < K; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * kTile * 128 + (kk % 4) * 32) >> 4);
    a[kk] = a_desc + off;
    b[kk] = b_desc + off;
  }
  mma_ss_warp<K>(d_tmem, a, b, idesc, 0u);
}

// Whether the fp16 copies of Q, K, V and dO hold the inputs exactly enough
// and the fp16 operands of the TS products stay in range: every |x| at most
// 60000 (fp16's largest finite value is 65504), and |dS| <= 2 D max|dO|
// max|V| at most 60000 (|dP| <= D max|dO| max|V|, and |Delta| too; P and the
// soft-cap's derivative are at most 1). A NaN fails every test.
__device__ __forceinline__ bool f16_in_range(const unsigned* mx, int D) {
  const float q = __uint_as_float(mx[0]), k = __uint_as_float(mx[1]),
              v = __uint_as_float(mx[2]), d = __uint_as_float(mx[3]);
  const float lim = 60000.0f;
  return q <= lim && k <= lim && v <= lim && d <= lim && 2.0f * float(D) * d * v <= lim;
}

// GENERAL: Sq or Skv is not a multiple of 128, or the call's queries and
// keys sit at position offsets (a separate instantiation, so the kernel for
// whole tiles at offset 0 keeps its code unchanged). 3-D tensor maps read
// zeros past the sequence, the extras of a tile that runs past it are loaded
// by the producer's lanes with bounds, padding keys are masked in dQ, padding
// query rows get LSE +inf in dK/dV (their P is 0), rows past the sequence are
// not stored; every mask term, ALiBi and the document ids use the absolute
// positions q_offset + i and kv_offset + j.
// F16: Q, K, V, dO come from fp16 copies and every product takes fp16
// operands: P, P g and dS rounded once to fp16 (2^-11 relative, against bf16's
// 2^-8) meet the flat bound without a second, lo part, so each TS product is
// one product instead of two (dQ: 4 per tile pair, dK/dV: 4, against 5 and 6).
template <int D, int SCORE, int MODE, bool GENERAL, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdArgs a) {
  using C = BwdCfg<D, MODE>;
  const FwdProblem& p = a.f;
  // the fp16 and bf16 kernels of an fp16-path call: one of them returns here
  if (a.f16_max != nullptr && f16_in_range(a.f16_max, D) != F16) return;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sFix = smem + C::kOffFix;      // dQ: Q, dO    dKV: K, V
  uint8_t* sSlots = smem + C::kOffSlots;  // dQ: K, V, doc    dKV: Q, dO, doc, LSE, Delta
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* fix_full = bars + 0;
  uint64_t* fix_empty = bars + 1;
  uint64_t* s_full = bars + 2;
  uint64_t* dp_full = bars + 3;
  uint64_t* p_full = bars + 4;
  uint64_t* ds_full = bars + 5;
  uint64_t* acc_done = bars + 6;
  uint64_t* acc_free = bars + 7;
  uint64_t* drain = bars + 8;
  uint64_t* dx_full = bars + 9;
  // A slot's two halves are filled and released separately: the second
  // (dO for dKV, V for dQ) is free once dV, or dP, has read it, well before
  // the first, so its next load starts early. full0/empty0: first half.
  uint64_t* slot_full0 = bars + 10;
  uint64_t* slot_full1 = bars + 10 + C::kSlots;
  uint64_t* slot_empty0 = bars + 10 + 2 * C::kSlots;
  uint64_t* slot_empty1 = bars + 10 + 3 * C::kSlots;
  float* sdx = reinterpret_cast<float*>(smem + C::kOffDx);  // [2 units][2 groups][128 rows]
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const bool has_doc = (p.variant & ATTN_MASK_DOCUMENT) != 0;

  if (threadIdx.x == 0) {
    mbar_init(fix_full, 1);
    mbar_init(fix_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, kComputeWarps);  // one arrive per compute warp
    mbar_init(ds_full, kComputeWarps);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, kComputeWarps);
    mbar_init(drain, 1);
    mbar_init(dx_full, kComputeWarps);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(slot_full0 + s, 1);
      mbar_init(slot_full1 + s, 1);
      mbar_init(slot_empty0 + s, 1);
      mbar_init(slot_empty1 + s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_base_smem, 512);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_smem;

  const int nq = GENERAL ? (p.Sq + kTile - 1) / kTile : p.Sq / kTile;
  const int nkv = GENERAL ? (p.Skv + kTile - 1) / kTile : p.Skv / kTile;
  const int num_units = MODE == kDQ ? p.B * nq * p.Hq : p.B * nkv * p.Hkv;
  const int group = p.Hq / p.Hkv;

  if (warp >= kComputeWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  }
  if (warp == kWarpProducer) {
    // ------------------------------------------------------------- producer
    // With ATTN_FAULT_NO_LOADS nothing is issued and the consumers' waits run out.
    const bool issue = !(p.fault_inject & ATTN_FAULT_NO_LOADS);
    const bool leader = lane == 0 && issue;
    // GENERAL: the streamed rows' extras start 16-byte aligned for every tile
    // when the row lengths are multiples of 4 (bulk copies need that)
    const bool rows_al = (p.Sq & 3) == 0;
    const int doc_off = MODE == kDQ ? p.mask.kv_off : p.mask.q_off;  // streamed rows' offset
    const bool doc_al = (p.mask.doc_len & 3) == 0 && (doc_off & 3) == 0;
    const int len = MODE == kDQ ? p.Skv : p.Sq;
    (void)rows_al;
    (void)doc_al;
    (void)len;
    (void)issue;
    uint32_t slot_it = 0, fix_it = 0;
    bool ok = true, pending1 = false;  // pending1: tile slot_it's second half issued alone
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const BUnit U = decode_bwd<MODE, GENERAL>(a, u);
      const int n = U.n();
      if (n == 0) continue;
      const int first = dense_first<MODE, GENERAL>(a, U);
      ok = __all_sync(0xffffffffu, wait_bounded(fix_empty, (fix_it & 1) ^ 1, wd));
      if (!ok) break;
      if (leader) {
        mbar_arrive_expect_tx(fix_full, 2 * C::kTileBytes);
        // dQ: Q and dO rows of (b, h, tile); dKV: K and V rows of (b, hk, tile)
        const CUtensorMap* m0 = MODE == kDQ ? &tm_q : &tm_k;
        const CUtensorMap* m1 = MODE == kDQ ? &tm_do : &tm_v;
        if constexpr (GENERAL) {
          const int slice = MODE == kDQ ? U.b * p.Hq + U.h : U.b * p.Hkv + U.h;
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            tma_load_3d(sFix + bx * C::kBoxBytes, m0, fix_full, bx * 64, U.tile * kTile, slice);
            tma_load_3d(sFix + C::kTileBytes + bx * C::kBoxBytes, m1, fix_full, bx * 64,
                        U.tile * kTile, slice);
          }
        } else {
          const int row = MODE == kDQ ? (U.b * p.Hq + U.h) * p.Sq + U.tile * kTile
                                      : (U.b * p.Hkv + U.h) * p.Skv + U.tile * kTile;
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            tma_load_2d(sFix + bx * C::kBoxBytes, m0, fix_full, bx * 64, row);
            tma_load_2d(sFix + C::kTileBytes + bx * C::kBoxBytes, m1, fix_full, bx * 64, row);
          }
        }
      }
      __syncwarp();
      ++fix_it;
      for (int it = 0; it < n && ok; ++it) {
        int hoff, t;
        bool partial;
        U.at(it, hoff, t, partial);
        t += first;
        const int slot = slot_it % C::kSlots;
        const uint32_t ph = ((slot_it / C::kSlots) & 1) ^ 1;
        uint8_t* base = sSlots + slot * C::kSlotBytes;
        // second half first: it is released earlier
        ok = __all_sync(0xffffffffu, wait_bounded(slot_empty1 + slot, ph, wd));
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(slot_full1 + slot, C::kTileBytes);
          if constexpr (GENERAL) {  // V rows of (b, hk, t) or dO rows of (b, h, t)
            const int slice =
                MODE == kDQ ? U.b * p.Hkv + U.h / group : U.b * p.Hq + U.h * group + hoff;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_3d(base + C::kTileBytes + bx * C::kBoxBytes, MODE == kDQ ? &tm_v : &tm_do,
                          slot_full1 + slot, bx * 64, t * kTile, slice);
          } else if (MODE == kDQ) {  // V rows of (b, hk, t)
            const int row = (U.b * p.Hkv + U.h / group) * p.Skv + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_2d(base + C::kTileBytes + bx * C::kBoxBytes, &tm_v, slot_full1 + slot,
                          bx * 64, row);
          } else {            // dO rows of (b, h, t)
            const int h = U.h * group + hoff;
            const int qrow = (U.b * p.Hq + h) * p.Sq + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_2d(base + C::kTileBytes + bx * C::kBoxBytes, &tm_do, slot_full1 + slot,
                          bx * 64, qrow);
          }
        }
        __syncwarp();
        pending1 = true;
        ok = __all_sync(0xffffffffu, wait_bounded(slot_empty0 + slot, ph, wd));
        if (!ok) break;
        if constexpr (GENERAL) {
          // The streamed rows' document ids (keys for dQ, queries for dKV)
          // and, for dKV, their LSE and Delta go to the slot's extras: by
          // asynchronous bulk copies when the tile lies inside the sequence
          // and the source rows start 16-byte aligned, else from the 32 lanes,
          // bounded by the sequence (a position past it gets document id -1,
          // LSE +inf, so its P is 0, and Delta 0); the leader's arrive below
          // releases these stores with the slot.
          const bool whole = (t + 1) * kTile <= len;
          const size_t doc0 =
              has_doc ? (size_t)U.b * p.mask.doc_len + doc_off + t * kTile : 0;
          const bool bulk_doc =
              has_doc && doc_al && whole && doc_off + (t + 1) * kTile <= p.mask.doc_len;
          const size_t qrow0 =
              MODE == kDKV ? (size_t)(U.b * p.Hq + U.h * group + hoff) * p.Sq + t * kTile : 0;
          const bool bulk_rows = MODE == kDKV && rows_al && whole;
          int* xdoc = reinterpret_cast<int*>(base + 2 * C::kTileBytes);
          float* xlse = reinterpret_cast<float*>(base + 2 * C::kTileBytes + 512);
          float* xdel = reinterpret_cast<float*>(base + 2 * C::kTileBytes + 1024);
          if (issue && ((has_doc && !bulk_doc) || (MODE == kDKV && !bulk_rows))) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = lane + 32 * k, pos = t * kTile + c;
              const bool in = pos < len;
              if (has_doc && !bulk_doc)
                xdoc[c] = (in && doc_off + pos < p.mask.doc_len) ? p.mask.doc_id[doc0 + c] : -1;
              if (MODE == kDKV && !bulk_rows) {
                xlse[c] = in ? p.lse[qrow0 + c] : INFINITY;
                xdel[c] = in ? a.delta[qrow0 + c] : 0.0f;
              }
            }
            __syncwarp();
          }
          uint32_t bytes = C::kTileBytes;
          if (bulk_doc) bytes += 512;
          if (bulk_rows) bytes += 1024;
          if (leader) mbar_arrive_expect_tx(slot_full0 + slot, bytes);
          if (leader) {  // K rows of (b, hk, t) or Q rows of (b, h, t)
            const int slice =
                MODE == kDQ ? U.b * p.Hkv + U.h / group : U.b * p.Hq + U.h * group + hoff;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_3d(base + bx * C::kBoxBytes, MODE == kDQ ? &tm_k : &tm_q, slot_full0 + slot,
                          bx * 64, t * kTile, slice);
            if (bulk_rows) {
              bulk_load(xlse, p.lse + qrow0, 512, slot_full0 + slot);
              bulk_load(xdel, a.delta + qrow0, 512, slot_full0 + slot);
            }
            if (bulk_doc) bulk_load(xdoc, p.mask.doc_id + doc0, 512, slot_full0 + slot);
          }
        } else {
          uint32_t bytes = C::kTileBytes;
          if (has_doc) bytes += 512;
          if (MODE == kDKV) bytes += 1024;
          if (leader) mbar_arrive_expect_tx(slot_full0 + slot, bytes);
          if (leader && MODE == kDQ) {  // K rows and the keys' document ids
            const int row = (U.b * p.Hkv + U.h / group) * p.Skv + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_2d(base + bx * C::kBoxBytes, &tm_k, slot_full0 + slot, bx * 64, row);
            if (has_doc)
              bulk_load(base + 2 * C::kTileBytes,
                        p.mask.doc_id + (size_t)U.b * p.mask.doc_len + t * kTile, 512,
                        slot_full0 + slot);
          } else if (leader) {  // Q rows and the queries' document ids, LSE and Delta
            const int h = U.h * group + hoff;
            const size_t qrow = (size_t)(U.b * p.Hq + h) * p.Sq + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_2d(base + bx * C::kBoxBytes, &tm_q, slot_full0 + slot, bx * 64, (int)qrow);
            if (has_doc)
              bulk_load(base + 2 * C::kTileBytes,
                        p.mask.doc_id + (size_t)U.b * p.mask.doc_len + t * kTile, 512,
                        slot_full0 + slot);
            bulk_load(base + 2 * C::kTileBytes + 512, p.lse + qrow, 512, slot_full0 + slot);
            bulk_load(base + 2 * C::kTileBytes + 1024, a.delta + qrow, 512, slot_full0 + slot);
          }
        }
        __syncwarp();
        ++slot_it;
        pending1 = false;
      }
    }
    if (!ok && !(p.fault_inject & ATTN_FAULT_NO_LOADS)) {  // let copies in flight land
      // (slot_it counts tiles whose loads were all issued; the tile after
      // them may have its second half in flight)
      if (pending1) wait_drain(slot_full1 + slot_it % C::kSlots, (slot_it / C::kSlots) & 1);
      for (uint32_t k = 1; k <= C::kSlots && k <= slot_it; ++k) {
        const uint32_t it = slot_it - k;
        wait_drain(slot_full0 + it % C::kSlots, (it / C::kSlots) & 1);
        wait_drain(slot_full1 + it % C::kSlots, (it / C::kSlots) & 1);
      }
      if (fix_it > 0) wait_drain(fix_full, (fix_it - 1) & 1);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (waits stay converged) and issues each
    // product as one block (issue_ss, issue_ts); lane 0 issues.
    constexpr uint32_t kIdescSS = F16 ? idesc_f16(128, 128, false) : idesc_bf16(128, 128, false);
    constexpr uint32_t kIdescTS = F16 ? idesc_f16(128, D, true) : idesc_bf16(128, D, true);
    // shared-memory descriptors: K-major (SS operands) and MN-major (B of the
    // TS products) views of the fixed tiles and of ring slot 0; other slots
    // and tiles add their byte offset >> 4
    const uint64_t dFixK = sdesc_sw128(smem_u32(sFix), 16, 1024);
    const uint64_t dSlotK = sdesc_sw128(smem_u32(sSlots), 16, 1024);
    const uint64_t dSlotMN = sdesc_sw128(smem_u32(sSlots), C::kBoxBytes, 1024);
    constexpr uint64_t kTileOff = C::kTileBytes >> 4;
    const uint32_t colS = tmem, colP = tmem + 128, acc0 = tmem + C::kColAcc,
                   acc1 = tmem + C::kColAcc + D;
    uint32_t slot_it = 0, fix_it = 0, p_it = 0, ds_it = 0, acc_it = 0;
    bool ok = true;
    auto slot_off = [&](uint32_t seq) {
      return (uint64_t)(((seq % C::kSlots) * C::kSlotBytes) >> 4);
    };
    // S = fix0 . slot0^T into S, dP = fix1 . slot1^T into dP
    auto issue_s = [&](uint32_t seq) {
      issue_ss<D>(colS, dFixK, dSlotK + slot_off(seq), kIdescSS);
      mma_commit_warp(s_full);
    };
    auto issue_dp = [&](uint32_t seq) {
      issue_ss<D>(colP, dFixK + kTileOff, dSlotK + slot_off(seq) + kTileOff, kIdescSS);
      mma_commit_warp(dp_full);
    };
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const BUnit U = decode_bwd<MODE, GENERAL>(a, u);
      const int n = U.n();
      if (n == 0) continue;
      ok = __all_sync(0xffffffffu, wait_bounded(fix_full, fix_it & 1, wd));
      if (!ok) break;
      ++fix_it;
      ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + slot_it % C::kSlots,
                                                (slot_it / C::kSlots) & 1, wd));
      if (!ok) break;
      tc_fence_after();
      issue_s(slot_it);
      ok = __all_sync(0xffffffffu, wait_bounded(slot_full1 + slot_it % C::kSlots,
                                                (slot_it / C::kSlots) & 1, wd));
      if (!ok) break;
      tc_fence_after();
      issue_dp(slot_it);
      if (MODE == kDQ) mma_commit_warp(slot_empty1 + slot_it % C::kSlots);  // V read
      if (n == 1) mma_commit_warp(fix_empty);  // the fixed tiles are read by S and dP only
      __syncwarp();
      for (int it = 0; it < n && ok; ++it) {
        const uint32_t seq = slot_it + it;
        const uint64_t s0 = dSlotMN + slot_off(seq);  // K (dQ) or Q (dKV), as B
        const uint64_t s1 = s0 + kTileOff;             // V (dQ) or dO (dKV), as B
        if (it == 0) {  // the accumulators of the previous unit have been read
          ok = __all_sync(0xffffffffu, wait_bounded(acc_free, (acc_it & 1) ^ 1, wd));
          if (!ok) break;
        }
        const bool acc = it > 0;
        if constexpr (MODE == kDKV) {
          // dV += P^T dO (hi, lo parts over S)
          ok = __all_sync(0xffffffffu, wait_bounded(p_full, p_it & 1, wd));
          if (!ok) break;
          ++p_it;
          tc_fence_after();
          issue_ts(acc0, colS, 0, s1, kIdescTS, acc);
          if constexpr (!F16) issue_ts(acc0, colS, 32, s1, kIdescTS, true);
          mma_commit_warp(slot_empty1 + seq % C::kSlots);  // dO read
        } else if constexpr (F16) {
          // B += (P g) K as soon as P g is stored (over S): with no lo part of
          // A beside it, the next tile's S follows at once and is computed
          // while the compute warps work on dS
          ok = __all_sync(0xffffffffu, wait_bounded(p_full, p_it & 1, wd));
          if (!ok) break;
          ++p_it;
          tc_fence_after();
          issue_ts(acc1, colS, 0, s0, kIdescTS, acc);
        } else {
          // B += (P g) K and A += lo K (operands over S)
          ok = __all_sync(0xffffffffu, wait_bounded(ds_full, ds_it & 1, wd));
          if (!ok) break;
          ++ds_it;
          tc_fence_after();
          issue_ts(acc1, colS, 0, s0, kIdescTS, acc);
          issue_ts(acc0, colS, 32, s0, kIdescTS, acc);
        }
        __syncwarp();
        if (it + 1 < n) {  // S of the next tile (its P/lo operands over S are consumed)
          ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + (seq + 1) % C::kSlots,
                                                    ((seq + 1) / C::kSlots) & 1, wd));
          if (!ok) break;
          tc_fence_after();
          issue_s(seq + 1);
          __syncwarp();
        }
        if constexpr (MODE == kDKV) {
          // dK += dS^T Q (hi, lo parts over dP)
          ok = __all_sync(0xffffffffu, wait_bounded(ds_full, ds_it & 1, wd));
          if (!ok) break;
          ++ds_it;
          tc_fence_after();
          issue_ts(acc1, colP, 0, s0, kIdescTS, acc);
          if constexpr (!F16) issue_ts(acc1, colP, 32, s0, kIdescTS, true);
        } else {
          // A += hi K (operand over dP); with fp16 operands the only part,
          // so it starts the accumulator, once dS is stored
          if constexpr (F16) {
            ok = __all_sync(0xffffffffu, wait_bounded(ds_full, ds_it & 1, wd));
            if (!ok) break;
            ++ds_it;
            tc_fence_after();
          }
          issue_ts(acc0, colP, 0, s0, kIdescTS, F16 ? acc : true);
        }
        mma_commit_warp(slot_empty0 + seq % C::kSlots);  // Q or K read
        __syncwarp();
        if (it + 1 < n) {  // dP of the next tile (the operands over dP are consumed)
          ok = __all_sync(0xffffffffu, wait_bounded(slot_full1 + (seq + 1) % C::kSlots,
                                                    ((seq + 1) / C::kSlots) & 1, wd));
          if (!ok) break;
          tc_fence_after();
          issue_dp(seq + 1);
          if (MODE == kDQ) mma_commit_warp(slot_empty1 + (seq + 1) % C::kSlots);  // V read
          if (it + 2 == n) mma_commit_warp(fix_empty);
          __syncwarp();
        }
      }
      if (!ok) break;
      ++acc_it;
      mma_commit_warp(acc_done);
      __syncwarp();
      slot_it += n;
    }
    mma_commit_warp(drain);
    __syncwarp();
    wait_drain(drain, 0);
  } else if (warp < kComputeWarps) {
    // ------------------------------------------------------------- compute
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsCompute));
    const int g = warp >> 2;           // column half of the streamed tile
    const int t = threadIdx.x & 127;   // row of the fixed tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t colS = tmem + lane_base + 64 * g;
    const uint32_t colP = tmem + lane_base + 128 + 64 * g;
    const uint32_t colAcc = tmem + lane_base + C::kColAcc;
    const float scale = p.score.scale;
    const float cap = p.score.softcap, inv_cap = 1.0f / p.score.softcap;
    uint32_t slot_it = 0, s_it = 0, acc_it = 0, dx_it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const BUnit U = decode_bwd<MODE, GENERAL>(a, u);
      const int n = U.n();
      const int first = dense_first<MODE, GENERAL>(a, U);
      // the thread's own row: a query row (dQ) or a key row (dKV)
      const int r = U.tile * kTile + t;
      constexpr int kHalfD = D / 2;  // accumulator columns stored by each warpgroup
      if (n == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (MODE == kDQ) {
          const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
          if ((GENERAL && r >= p.Sq) || !MATTN_IN_BOUNDS(kSiteBwdGrad, qrow, (size_t)p.B * p.Hq * p.Sq))
            continue;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + qrow * D +
                                                g * kHalfD);
          for (int c = 0; c < kHalfD / 8; ++c) dst[c] = z;
          if (g == 0) a.delta_out[qrow] = 0.0f;
        } else {
          const size_t off = ((size_t)(U.b * p.Hkv + U.h) * p.Skv + r) * D + g * kHalfD;
          if ((GENERAL && r >= p.Skv) ||
              !MATTN_IN_BOUNDS(kSiteBwdGrad, off / D, (size_t)p.B * p.Hkv * p.Skv))
            continue;
          uint4* dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk) + off);
          uint4* dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv) + off);
          for (int c = 0; c < kHalfD / 8; ++c) dk[c] = z, dv[c] = z;
        }
        continue;
      }
      const int* docb = has_doc ? p.mask.doc_id + (size_t)U.b * p.mask.doc_len : nullptr;
      // GENERAL: this row's absolute position (query rows: q_offset + r; key rows: kv_offset + r)
      const int r_abs = GENERAL ? r + (MODE == kDQ ? p.mask.q_off : p.mask.kv_off) : r;
      const int my_doc = (docb && (!GENERAL || r_abs < p.mask.doc_len) &&
                          MATTN_IN_BOUNDS(kSiteBwdDoc, r_abs, p.mask.doc_len))
                             ? docb[r_abs]
                             : 0;
      const int dqk = GENERAL ? p.mask.q_off - p.mask.kv_off : 0;  // absolute i - j = (i - j) + dqk
      (void)dqk;
      const int P = (p.variant & ATTN_MASK_PREFIX) ? p.mask.prefix_len[U.b] : INT_MIN;
      float row_lse2 = 0.0f, row_delta = 0.0f, row_dhat = 0.0f;
      if (MODE == kDQ) {
        const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
        // GENERAL: a row past Sq (the last tile's padding) gets LSE +inf: its P is 0
        const bool in =
            (!GENERAL || r < p.Sq) && MATTN_IN_BOUNDS(kSiteBwdRow, qrow, (size_t)p.B * p.Hq * p.Sq);
        const float l = in ? p.lse[qrow] : (GENERAL ? INFINITY : 0.0f);
        row_lse2 = l == -INFINITY ? INFINITY : l * kLog2e;  // empty row: every p is 0
        row_dhat = in ? a.delta[qrow] : 0.0f;  // estimate from the bf16 O (delta_kernel)
      }
      for (int it = 0; it < n; ++it) {
        int hoff, tt;
        bool partial;
        U.at(it, hoff, tt, partial);
        tt += first;
        // GENERAL, dQ: a key tile that runs past Skv is masked element by element
        if (GENERAL && MODE == kDQ && (tt + 1) * kTile > p.Skv) partial = true;
        const int h = MODE == kDQ ? U.h : U.h * group + hoff;
        const uint32_t seq = slot_it + it;
        const uint8_t* base = sSlots + (seq % C::kSlots) * C::kSlotBytes;
        const int* sdoc = reinterpret_cast<const int*>(base + 2 * C::kTileBytes) + 64 * g;
        const float* slse = reinterpret_cast<const float*>(base + 2 * C::kTileBytes + 512) + 64 * g;
        const float* sdel = reinterpret_cast<const float*>(base + 2 * C::kTileBytes + 1024) + 64 * g;
        // the slot's shared-memory extras (doc ids, LSE, Delta) are read directly
        ok = __all_sync(0xffffffffu,
                        wait_bounded(slot_full0 + seq % C::kSlots, (seq / C::kSlots) & 1, wd));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_bounded(s_full, s_it & 1, wd));
        if (!ok) break;
        tc_fence_after();
        const int c0 = tt * kTile + 64 * g;  // position of this warpgroup's first column
        const float slope = (SCORE & 1) ? alibi_slope(p.score, h) : 0.0f;
        // mask bounds on the column c of this warpgroup's 64 (see below)
        int lo = INT_MIN, hi = INT_MAX, pre = INT_MIN;
        if (partial) {
          if constexpr (GENERAL) {  // absolute positions; keys past Skv: none kept
            if (MODE == kDQ) {  // row i = r, column j = c0 + c
              if (p.variant & ATTN_MASK_CAUSAL) hi = r - c0 + dqk + 1;
              if (p.variant & ATTN_MASK_WINDOW) lo = r - c0 + dqk - p.mask.window + 1;
              hi = min(hi, p.Skv - c0);
              if (P != INT_MIN) pre = min(P - p.mask.kv_off, p.Skv) - c0;
            } else {            // row j = r, column i = c0 + c
              if (p.variant & ATTN_MASK_CAUSAL) lo = r - c0 - dqk;
              if (p.variant & ATTN_MASK_WINDOW) hi = r - c0 - dqk + p.mask.window;
              if (P != INT_MIN && r_abs < P) pre = INT_MAX;
            }
          } else if (MODE == kDQ) {  // row i = r, column j = c0 + c
            if (p.variant & ATTN_MASK_CAUSAL) hi = r - c0 + 1;
            if (p.variant & ATTN_MASK_WINDOW) lo = r - c0 - p.mask.window + 1;
            if (P != INT_MIN) pre = P - c0;
          } else {            // row j = r, column i = c0 + c
            if (p.variant & ATTN_MASK_CAUSAL) lo = r - c0;
            if (p.variant & ATTN_MASK_WINDOW) hi = r - c0 + p.mask.window;
            if (P != INT_MIN && r < P) pre = INT_MAX;
          }
        }
        // (j - i) = base_ji + sgn * c for the column c of this warpgroup's 64
        // (absolute positions: minus dqk)
        const int base_ji = (MODE == kDQ ? c0 - r : r - c0) - (GENERAL ? dqk : 0);
        // relative-position bias (SCORE bit 4, general instantiation only, no
        // offsets): the table entry of distance i - j is rb0 + rbs * c,
        // clamped to the table (the clamped entries belong to padding rows or
        // keys, which are masked or have P = 0)
        const float* rbt =
            (SCORE & 4) ? p.score.rel_bias + (size_t)h * p.score.rb_len : nullptr;
        const int rb0 = -base_ji + p.score.rb_zero;
        const int rbs = MODE == kDQ ? -1 : 1;
        (void)rbt;
        (void)rb0;
        (void)rbs;
        const float sgn = MODE == kDQ ? 1.0f : -1.0f;
        // P (and P g) from S, 16 columns at a time, two columns per packed
        // instruction; v keeps P g for dS. An empty row (LSE = -inf) occurs
        // only in partial tiles, where the mask zeroes all of it, so LSE needs
        // no special case here.
        constexpr bool kKeepP = MODE == kDQ && (SCORE & 2) != 0;  // Delta needs P itself
        float v[64];
        float pf[kKeepP ? 64 : 1];
        {
          uint32_t rr[64];
          tmem_ld32(colS, *reinterpret_cast<uint32_t(*)[32]>(rr));
          tmem_ld32(colS + 32, *reinterpret_cast<uint32_t(*)[32]>(rr + 32));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(rr));
          tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(rr + 32));
#pragma unroll
          for (int e = 0; e < 64; ++e) v[e] = __uint_as_float(rr[e]);
        }
        // ALiBi in log2 units: slope2 (base_ji + sgn c) = a0 + a1 c
        const float slope2 = slope * kLog2e;
        const float a0 = slope2 * float(base_ji), a1 = slope2 * sgn;
        const float sl2 = scale * kLog2e;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {  // 32 columns: 16 packed TMEM columns per part
          uint32_t hi16[16], lo16[16];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const int q = 2 * h2 + q2;
            // minus the LSE of each column in log2 units (dKV: the column's
            // own row of the stream; dQ: this thread's row)
            float2 nl[8];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              if constexpr (MODE == kDKV) {
                const float4 l4 = *reinterpret_cast<const float4*>(slse + 16 * q + 2 * e);
                const float2 m2 = make_float2(-kLog2e, -kLog2e);
                nl[e] = fmul2(make_float2(l4.x, l4.y), m2);
                nl[e + 1] = fmul2(make_float2(l4.z, l4.w), m2);
              } else {
                nl[e] = nl[e + 1] = make_float2(-row_lse2, -row_lse2);
              }
            }
            float2 pr[8], gg[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int c = 16 * q + 2 * e;
              const float2 sv = make_float2(v[c], v[c + 1]);
              float2 rbv = make_float2(0.0f, 0.0f);
              if constexpr ((SCORE & 4) != 0) {
                const int last = p.score.rb_len - 1;
                const int i0 = min(max(rb0 + rbs * c, 0), last);
                const int i1 = min(max(rb0 + rbs * (c + 1), 0), last);
                rbv = make_float2(__ldg(rbt + i0), __ldg(rbt + i1));
              }
              float2 arg;
              if constexpr ((SCORE & 2) == 0) {
                // log2-unit score: s sl2 (+ ALiBi) (+ bias) - LSE2, one packed FMA each
                float2 bias = nl[e];
                if constexpr ((SCORE & 1) != 0)
                  bias = ffma2(make_float2(a1, a1), make_float2(float(c), float(c + 1)),
                               fadd2(bias, make_float2(a0, a0)));
                if constexpr ((SCORE & 4) != 0)
                  bias = ffma2(rbv, make_float2(kLog2e, kLog2e), bias);
                arg = ffma2(sv, make_float2(sl2, sl2), bias);
                gg[e] = make_float2(1.0f, 1.0f);
              } else {
                float2 x = fmul2(sv, make_float2(scale, scale));
                if constexpr ((SCORE & 1) != 0)
                  x = ffma2(make_float2(slope * sgn, slope * sgn),
                            make_float2(float(c), float(c + 1)),
                            fadd2(x, make_float2(slope * float(base_ji), slope * float(base_ji))));
                if constexpr ((SCORE & 4) != 0) x = fadd2(x, rbv);  // the bias enters before the cap
                pr[e] = fmul2(x, make_float2(inv_cap, inv_cap));  // tanh argument
              }
              if constexpr ((SCORE & 2) == 0) pr[e] = arg;
            }
            if constexpr ((SCORE & 2) != 0) {
              float th[16];
#pragma unroll
              for (int e = 0; e < 8; ++e) th[2 * e] = pr[e].x, th[2 * e + 1] = pr[e].y;
              tanh16(th);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float2 t2 = make_float2(th[2 * e], th[2 * e + 1]);
                gg[e] = ffma2(fmul2(t2, make_float2(-1.0f, -1.0f)), t2, make_float2(1.0f, 1.0f));
                // cap tanh in log2 units minus LSE2
                pr[e] = ffma2(t2, make_float2(cap * kLog2e, cap * kLog2e), nl[e]);
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int c = 16 * q + 2 * e;
              float p0 = ex2_approx(pr[e].x), p1 = ex2_approx(pr[e].y);
              if (partial) {
                // bitwise terms, document id read on a warp-uniform condition:
                // no divergent branch per element
                const bool same0 = docb ? (sdoc[c] == my_doc) : true;
                const bool same1 = docb ? (sdoc[c + 1] == my_doc) : true;
                const bool keep0 = ((c >= lo) & (c < hi) & same0) | (c < pre);
                const bool keep1 = ((c + 1 >= lo) & (c + 1 < hi) & same1) | (c + 1 < pre);
                p0 = keep0 ? p0 : 0.0f;
                p1 = keep1 ? p1 : 0.0f;
              }
              const float2 p2 = make_float2(p0, p1);
              float2 vg = p2;
              if constexpr ((SCORE & 2) != 0) vg = fmul2(p2, gg[e]);
              v[c] = vg.x;
              v[c + 1] = vg.y;
              if constexpr (kKeepP) pf[c] = p0, pf[c + 1] = p1;
              if constexpr (F16) {  // P^T for dV += P^T dO, or P g for B += (P g) K
                hi16[8 * q2 + e] = MODE == kDKV ? pack_f16x2(p0, p1) : pack_f16x2(vg.x, vg.y);
              } else if constexpr (MODE == kDKV) {  // P^T, split, for dV += P^T dO
                split_bf16x2(p0, p1, hi16[8 * q2 + e], lo16[8 * q2 + e]);
              } else {  // P g in bf16, for B += (P g) K
                hi16[8 * q2 + e] = pack_bf16x2(vg.x, vg.y);
              }
            }
          }
          tmem_st16(colS + 16 * h2, hi16);
          if constexpr (MODE == kDKV && !F16) tmem_st16(colS + 32 + 16 * h2, lo16);
        }
        if constexpr (MODE == kDKV || F16) {  // P (dKV) or P g (dQ, fp16) is stored
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_full);
        }
        ok = __all_sync(0xffffffffu, wait_bounded(dp_full, s_it & 1, wd));
        if (!ok) break;
        ++s_it;
        tc_fence_after();
        // dKV: dS = P g (dP - Delta);  dQ: P g (dP - Dhat) and Delta += P dP.
        // Split into hi and lo parts, 32 columns at a time; every part goes
        // over columns this warpgroup has already read (the dKV lo parts of
        // the first 32 columns wait for the second half's load).
        uint32_t dl0[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t rr[32];
          tmem_ld32(colP + 32 * hh, rr);
          tmem_ld_wait_regs(rr);
          uint32_t dh[16], dl[16];
          float2 dacc = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int c = 32 * hh + e;
            float4 d4;
            if constexpr (MODE == kDKV) d4 = *reinterpret_cast<const float4*>(sdel + c);
            else d4 = make_float4(row_dhat, row_dhat, row_dhat, row_dhat);
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              const float2 dp = make_float2(__uint_as_float(rr[e + 2 * z]),
                                            __uint_as_float(rr[e + 2 * z + 1]));
              const float2 dl2 = z ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
              const float2 vv = make_float2(v[c + 2 * z], v[c + 2 * z + 1]);
              // dKV: dS = P g (dP - Delta);  dQ: P g (dP - Dhat)
              const float2 ds = fmul2(vv, ffma2(dl2, make_float2(-1.0f, -1.0f), dp));
              if constexpr (MODE == kDQ) {  // Delta += P dP
                if constexpr (kKeepP)
                  dacc = ffma2(make_float2(pf[c + 2 * z], pf[c + 2 * z + 1]), dp, dacc);
                else  // identity or ALiBi score_mod: P g = P
                  dacc = ffma2(vv, dp, dacc);
              }
              if constexpr (F16) dh[e / 2 + z] = pack_f16x2(ds.x, ds.y);
              else split_bf16x2(ds.x, ds.y, dh[e / 2 + z], dl[e / 2 + z]);
            }
          }
          if constexpr (MODE == kDQ) row_delta += dacc.x + dacc.y;
          tmem_st16(colP + 16 * hh, dh);
          if constexpr (F16) {
            // no lo parts
          } else if constexpr (MODE == kDKV) {
            if (hh == 0) {
#pragma unroll
              for (int e = 0; e < 16; ++e) dl0[e] = dl[e];
            } else {
              tmem_st16(colP + 32, dl0);
              tmem_st16(colP + 48, dl);
            }
          } else {
            tmem_st16(colS + 32 + 16 * hh, dl);  // beside P g over S
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
      if (!ok) break;
      slot_it += n;
      // epilogue: each warpgroup stores half of the accumulator columns
      ok = __all_sync(0xffffffffu, wait_bounded(acc_done, acc_it & 1, wd));
      if (!ok) break;
      ++acc_it;
      tc_fence_after();
      auto store_half = [&](uint32_t col, __nv_bfloat16* dst, float mul, bool in) {
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(col + 32 * c, rr);
          tmem_ld_wait_regs(rr);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * mul,
                                __uint_as_float(rr[2 * e + 1]) * mul);
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (in) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      };
      if (MODE == kDQ) {  // dQ = scale (A - (Delta - Dhat) B); Delta to the workspace
        // the two warpgroups' partial sums of Delta meet in shared memory
        float* dx = sdx + (dx_it & 1) * 2 * kTile;
        dx[g * kTile + t] = row_delta;
        __syncwarp();
        if (lane == 0) mbar_arrive(dx_full);
        ok = __all_sync(0xffffffffu, wait_bounded(dx_full, dx_it & 1, wd));
        if (!ok) break;
        ++dx_it;
        const float delta = dx[t] + dx[kTile + t];
        const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
        const bool in =
            (!GENERAL || r < p.Sq) && MATTN_IN_BOUNDS(kSiteBwdGrad, qrow, (size_t)p.B * p.Hq * p.Sq);
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + (in ? qrow : 0) * D + g * kHalfD;
        const float corr = delta - row_dhat;
#pragma unroll
        for (int c = 0; c < kHalfD / 32; ++c) {
          uint32_t ra[32], rb[32];
          tmem_ld32(colAcc + g * kHalfD + 32 * c, ra);
          tmem_ld32(colAcc + D + g * kHalfD + 32 * c, rb);
          tmem_ld_wait_regs(ra);
          tmem_ld_wait_regs(rb);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x0 = scale * fmaf(-corr, __uint_as_float(rb[2 * e]), __uint_as_float(ra[2 * e]));
            const float x1 = scale * fmaf(-corr, __uint_as_float(rb[2 * e + 1]), __uint_as_float(ra[2 * e + 1]));
            pk[e] = pack_bf16x2(x0, x1);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (in) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
        if (g == 0 && in) a.delta_out[qrow] = delta;
      } else {
        const size_t off = ((size_t)(U.b * p.Hkv + U.h) * p.Skv + r) * D + g * kHalfD;
        // every thread loads its accumulator (a warp-wide TMEM load); the
        // debug build skips the stores of a row outside dK / dV
        const bool in = (!GENERAL || r < p.Skv) &&
                        MATTN_IN_BOUNDS(kSiteBwdGrad, off / D, (size_t)p.B * p.Hkv * p.Skv);
        store_half(colAcc + g * kHalfD, static_cast<__nv_bfloat16*>(a.dv) + off, 1.0f, in);
        store_half(colAcc + D + g * kHalfD, static_cast<__nv_bfloat16*>(a.dk) + off, scale, in);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int SCORE, int MODE, bool GENERAL, bool F16>
cudaError_t launch_one(const BwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, int units,
                       cudaStream_t stream) {
  using C = BwdCfg<D, MODE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_kernel<D, SCORE, MODE, GENERAL, F16>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  });
  if (attr_err != cudaSuccess) return attr_err;
  // setmaxnreg.inc draws on the registers the launch holds: refuse to launch
  // if the compiled register count cannot cover the split (the increase
  // would wait forever)
  static int regs = -1;
  static std::once_flag regs_once;
  std::call_once(regs_once, [] {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, bwd_kernel<D, SCORE, MODE, GENERAL, F16>) == cudaSuccess)
      regs = fa.numRegs;
  });
  if (regs < 0 || 256LL * kRegsCompute + 128LL * kRegsOther > (long long)regs * kThreads)
    return cudaErrorInvalidConfiguration;
  const int grid = units < sm_count() ? units : sm_count();
  if (grid == 0) return cudaSuccess;
  bwd_kernel<D, SCORE, MODE, GENERAL, F16>
      <<<grid, kThreads, C::kSmemAlloc, stream>>>(mq, mk, mv, mdo, a);
  return cudaGetLastError();
}

// Delta-hat from the bf16 O and dO (both paths).
inline cudaError_t launch_delta(const BwdProblem& bp, cudaStream_t stream) {
  const FwdProblem& f = bp.f;
  const size_t rows = (size_t)f.B * f.Hq * f.Sq;
  delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(f.o), static_cast<const __nv_bfloat16*>(bp.dO),
      bp.delta, rows, f.D);
  return cudaGetLastError();
}

// One of the two kernels (MODE) of the backward. F16: over the fp16 copies of
// Q, K, V, dO (whole tiles only). guard: the fp16 path's range record, or
// nullptr when the call has no fp16 copies.
template <int D, int SCORE, bool GENERAL, bool F16>
cudaError_t launch_mode(const BwdProblem& bp, int mode, const unsigned* guard,
                        cudaStream_t stream) {
  static_assert(!(F16 && GENERAL), "fp16 copies serve whole tiles at offset 0 only");
  const FwdProblem& f = bp.f;
  CUtensorMap mq, mk, mv, mdo;
  if constexpr (GENERAL) {  // 3-D views [B*H][S][D]: a tile past the sequence reads zeros
    if (!make_map_bf16_3d(&mq, f.q, (long long)f.B * f.Hq, f.Sq, D) ||
        !make_map_bf16_3d(&mk, f.k, (long long)f.B * f.Hkv, f.Skv, D) ||
        !make_map_bf16_3d(&mv, f.v, (long long)f.B * f.Hkv, f.Skv, D) ||
        !make_map_bf16_3d(&mdo, bp.dO, (long long)f.B * f.Hq, f.Sq, D))
      return cudaErrorInvalidValue;
  } else {
    const CUtensorMapDataType dt =
        F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map_bf16(&mq, F16 ? bp.q16 : f.q, (long long)f.B * f.Hq * f.Sq, D, dt) ||
        !make_map_bf16(&mk, F16 ? bp.k16 : f.k, (long long)f.B * f.Hkv * f.Skv, D, dt) ||
        !make_map_bf16(&mv, F16 ? bp.v16 : f.v, (long long)f.B * f.Hkv * f.Skv, D, dt) ||
        !make_map_bf16(&mdo, F16 ? bp.do16 : bp.dO, (long long)f.B * f.Hq * f.Sq, D, dt))
      return cudaErrorInvalidValue;
  }
  BwdArgs a{f, bp.dO, bp.dq, bp.dk, bp.dv, bp.delta, bp.delta, f.lists, guard};
  const int nq = (f.Sq + kTile - 1) / kTile, nkv = (f.Skv + kTile - 1) / kTile;
  if (mode == kDQ) return launch_one<D, SCORE, kDQ, GENERAL, F16>(a, mq, mk, mv, mdo,
                                                                   f.B * nq * f.Hq, stream);
  a.lists = bp.t_lists;
  return launch_one<D, SCORE, kDKV, GENERAL, F16>(a, mq, mk, mv, mdo, f.B * nkv * f.Hkv, stream);
}

// The whole bf16 backward: Delta-hat, then the dQ and dK/dV kernels.
template <int D, int SCORE, bool GENERAL>
cudaError_t launch_typed(const BwdProblem& bp, cudaStream_t stream) {
  cudaError_t e = launch_delta(bp, stream);
  if (e != cudaSuccess) return e;
  e = launch_mode<D, SCORE, GENERAL, false>(bp, kDQ, nullptr, stream);
  if (e != cudaSuccess) return e;
  return launch_mode<D, SCORE, GENERAL, false>(bp, kDKV, nullptr, stream);
}

}  // namespace
}  // namespace mattn
