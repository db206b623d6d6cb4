// bf16 forward on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Algorithm: the 1-pass FlashAttention recurrence named on the
// Online-Softmax/FlashAttention page (online softmax: running max m, running
// sum l, accumulator rescaled when m grows), with score_mod applied per element
// before the softmax and the mask applied only on partial tiles (FlexAttention
// page: "FlexAttention" section, the variant list, and the item on exploiting
// mask sparsity). The score matrix never leaves the SM.
//
// Work unit: two 128-row query tiles ("rows" A and B) that read the same K/V
// tiles: one query tile of two query heads (2h, 2h+1) of one batch element,
// which see the same key-tile list because the mask does not depend on the
// head, or, for multi-head attention without block-mask lists, the query
// tiles 2q and 2q+1 of one head. Units are taken longest-first (block-mask
// `order`) by a persistent grid of one CTA per SM.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax for row A (thread t owns query row t: TMEM lane t)
//   warps 4-7  softmax for row B
//   warp  8    TMA producer: Q tiles once per unit, then K/V tiles into a ring
//   warp  9    MMA issuer (one thread) and TMEM owner
//   warp  10   second MMA issuer at D = 64 (row B), idle at D = 128
//   warp  11   idle
// The third warpgroup hands registers to the softmax warpgroups (setmaxnreg).
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A, O_B (D columns
// each) from 256. P (bf16) overwrites the first 64 columns of its S tile and
// is the A operand of the P.V product, read straight from TMEM.
//
// Per key tile j and row X:  S_X = Q_X K_j^T (SS MMA) -> softmax warps read
// S_X, write P_X -> O_X += P_X V_j (TS MMA). The MMA warp alternates rows so
// one row's softmax overlaps the other row's products.
#pragma once

#include <cmath>
#include <mutex>
#include <type_traits>

#include "host_util.h"
#include "launch.h"

namespace mattn {
namespace {

constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 208;  // 2 x 128 x 208 + 128 x 88 = 64512 = 384 x 168
constexpr int kRegsOther = 88;
constexpr int kSoftmaxThreads = 128;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpMma2 = 10;  // second MMA issuer (separate-P kernels: head B)

template <int D>
struct Cfg {
  static constexpr int kTileBytes = kTile * D * 2;  // one 128-row bf16 tile
  static constexpr int kBoxes = D / 64;             // 64-column (128-byte) TMA boxes
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kSlots = D == 128 ? 4 : 8;   // K/V ring
  static constexpr int kOffQ = 0;
  static constexpr int kOffSlots = 2 * kTileBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kTileBytes;
  // barriers: q_full, q_empty, drain, s_full[2], p_full[2], o_done[2], o_free[2],
  // s_free[2], pv_done[2], drain2, slot_full[kSlots], slot_empty[kSlots]
  static constexpr int kNumBars = 16 + 2 * kSlots;
  // per-warp document ids, read as int4: 16-byte aligned
  static constexpr int kOffDoc = (kOffBars + kNumBars * 8 + 15) & ~15;
  // Per-warp area of kWarpArea bytes, used in the key-tile loop for the two
  // windows of the relative-position bias (float [2][kRbWindow], double-
  // buffered by tile) and in the epilogue to stage 32 rows x 32 bf16 columns
  // of the output.
  static constexpr int kRbWindow = 160;
  static constexpr int kStageBytes = 32 * 32 * 2;
  static constexpr int kWarpArea = kStageBytes;
  static_assert(2 * kRbWindow * 4 <= kWarpArea, "bias windows fit the per-warp area");
  static constexpr int kOffArea = kOffDoc + 8 * kTile * 4;
  static constexpr int kOffMisc = kOffArea + 8 * kWarpArea;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;     // slack for 1024-byte alignment
  static constexpr uint32_t kColO0 = 256;
  // D = 64 leaves TMEM room for P apart from S (columns 384 + 64x): the
  // softmax frees S as soon as it has read it and the next Q.K^T overlaps the
  // rest of its work. At D = 128 the 512 columns hold S_A, S_B, O_A, O_B and P
  // overwrites S, so the next Q.K^T waits for the P.V product.
  static constexpr bool kSepP = D == 64;
  // One MMA warp per head at D = 64: the tensor pipe queues about one product,
  // so a single issuer leaves it idle whenever it waits or commits; with two,
  // one head's products run while the other's issuer waits. At D = 128 (P
  // over S) a single issuer alternating heads keeps the two heads' softmax
  // phases apart, which matters more there: with two issuers they align and
  // contend for the special-function unit (soft-cap: 1.38 -> 1.84 ms measured).
  static constexpr bool kDualMma = kSepP;
  static constexpr uint32_t kColP = 384;
  static_assert(!kSepP || kColP + 128 <= 512, "tensor memory columns");
  static_assert(kOffDoc % 16 == 0 && (kTile * 4) % 16 == 0, "int4 reads of document ids");
  static_assert(kOffArea % 16 == 0, "uint4 staging of the output");
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
};

struct Unit {
  // Row slot x (softmax warpgroup x) is query tile qt[x] of query head h[x];
  // h[1] < 0: a single-row unit.
  int b, qt[2], h[2];
  // Row slot x's fields. kRegs: by selection, which keeps the unit in
  // registers; otherwise by indexing with x, which is not a compile-time
  // constant and so puts the unit in local memory, read from there where a
  // field is used. Which is faster depends on the instantiation's register
  // pressure (measured; see kUnitRegs in the kernel).
  template <bool kRegs>
  __device__ __forceinline__ int head(int x) const {
    if constexpr (kRegs) return x ? h[1] : h[0];
    else return h[x];
  }
  template <bool kRegs>
  __device__ __forceinline__ int qtile(int x) const {
    if constexpr (kRegs) return x ? qt[1] : qt[0];
    else return qt[x];
  }
  int n_full, n_part;
  const int* lf;
  const int* lp;
  int nkv;  // key tiles of the problem (the debug build checks list entries against it)
  __device__ __forceinline__ int n() const { return n_full + n_part; }
  // Visiting order: partial tiles, then full tiles, each from the largest key
  // index down. Keys near the query usually carry the largest scores (causal
  // diagonal, ALiBi), so the running maximum settles early and the
  // accumulator is rarely rescaled. The softmax result does not depend on it.
  __device__ __forceinline__ bool partial(int j) const { return j < n_part; }
  __device__ __forceinline__ int kt(int j) const {
    int t;
    if (j < n_part) {
      const int a = n_part - 1 - j;
      t = lp ? lp[a] : a;
    } else {
      const int a = n_full - 1 - (j - n_part);
      t = lf ? lf[a] : a;
    }
    return MATTN_IN_BOUNDS(kSiteFwdList, t, nkv) ? t : 0;
  }
};

// Static schedule of a persistent CTA: round r takes unit r*G + c for even r
// and r*G + (G-1-c) for odd r (G CTAs, c = blockIdx.x). On a longest-first
// unit order this zigzag evens out the total work per CTA.
__device__ __forceinline__ int zigzag_unit(int r) {
  const int c = (r & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
  return r * (int)gridDim.x + c;
}

// Two kinds of unit. Multi-head attention without block-mask lists (or with a
// causal mask alone, whose lists it does not need) pairs the
// query tiles 2q and 2q + 1 of one head: both rows read the same K/V tiles,
// so each tile is loaded into shared memory once for two products, as the
// heads of a GQA group share theirs. The pair visits the union of its rows'
// key tiles (the later row's causal range); the earlier row masks the tile
// past its own range element by element like any other masked column.
// Otherwise a unit is one query tile of the query heads 2h and 2h + 1, which
// see the same key-tile list because the mask does not depend on the head.
// Pairs only at D = 128: at D = 64 (separate P, one MMA warp per row) they
// measured slower than head pairs (causal ALiBi B4 H16 S2048: 91 against 81 us).
// A causal mask alone needs no lists (a tile is full below the diagonal,
// partial on it, empty above), so on contiguous K/V pairs serve it with or
// without them (causal B8 H16 S4096 with lists: 0.535 -> 0.520 ms); the paged
// kernel keeps head pairs there (0.570 against 0.579 ms with 64-token pages).
template <int D, bool PAGED>
__host__ __device__ __forceinline__ bool pair_tiles(const FwdProblem& p) {
  return D == 128 && p.Hq == p.Hkv &&
         (p.lists.full_cnt == nullptr ||
          (!PAGED && (p.variant & ATTN_MASK_BITS) == ATTN_MASK_CAUSAL));
}

template <int D, bool PAGED>
__host__ __device__ __forceinline__ int count_units(const FwdProblem& p) {
  const int nq = (p.Sq + kTile - 1) / kTile;
  return pair_tiles<D, PAGED>(p) ? p.B * ((nq + 1) / 2) * p.Hq : p.B * nq * ((p.Hq + 1) / 2);
}

template <int D, bool PAGED>
__device__ __forceinline__ Unit decode_unit(const FwdProblem& p, int u) {
  const int nq = (p.Sq + kTile - 1) / kTile, nkv = (p.Skv + kTile - 1) / kTile;
  const bool causal_bound = (p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX);
  Unit U;
  if (pair_tiles<D, PAGED>(p)) {
    const int npair = (nq + 1) / 2;
    const int rank = u / p.Hq, h = u % p.Hq;
    const int qp = causal_bound ? npair - 1 - rank / p.B : rank % npair;  // longest first
    U.b = causal_bound ? rank % p.B : rank / npair;
    U.qt[0] = 2 * qp;
    U.qt[1] = 2 * qp + 1;
    U.h[0] = h;
    U.h[1] = U.qt[1] < nq ? h : -1;
    const int rows_end = min((U.qtile<true>(U.h[1] >= 0) + 1) * kTile, p.Sq);
    const int last = causal_bound ? causal_tiles(p.mask, rows_end - 1, nkv) : nkv;
    const bool masked = (p.variant & ATTN_MASK_BITS) != 0;
    U.n_full = masked ? 0 : last;
    U.n_part = masked ? last : 0;
    U.lf = U.lp = nullptr;
    U.nkv = nkv;
    return U;
  }
  const int nhp = (p.Hq + 1) / 2;
  const int rank = u / nhp, hp = u % nhp;
  int row;
  if (p.lists.full_cnt) {
    row = p.lists.order[rank];
    if (!MATTN_IN_BOUNDS(kSiteFwdList, row, p.B * nq)) row = 0;
  } else if (causal_bound) {
    row = (rank % p.B) * nq + (nq - 1 - rank / p.B);  // longest first
  } else {
    row = rank;
  }
  U.b = row / nq;
  U.qt[0] = U.qt[1] = row % nq;
  U.h[0] = 2 * hp;
  U.h[1] = 2 * hp + 1 < p.Hq ? 2 * hp + 1 : -1;
  if (p.lists.full_cnt) {
    U.n_full = p.lists.full_cnt[row];
    U.n_part = p.lists.part_cnt[row];
    U.lf = p.lists.full_idx + (size_t)row * p.lists.nkv;
    U.lp = p.lists.part_idx + (size_t)row * p.lists.nkv;
    if (!MATTN_IN_BOUNDS(kSiteFwdList, U.n_full, min(nkv, p.lists.nkv) + 1)) U.n_full = 0;
    if (!MATTN_IN_BOUNDS(kSiteFwdList, U.n_part, min(nkv, p.lists.nkv) + 1 - U.n_full))
      U.n_part = 0;
  } else {
    const int last =
        causal_bound ? causal_tiles(p.mask, min((U.qt[0] + 1) * kTile, p.Sq) - 1, nkv) : nkv;
    const bool masked = (p.variant & ATTN_MASK_BITS) != 0;
    U.n_full = masked ? 0 : last;
    U.n_part = masked ? last : 0;
    U.lf = U.lp = nullptr;
  }
  U.nkv = nkv;
  return U;
}

// Document id of key j, or -1 past the end of the keys (those columns are
// masked by the key-length bound anyway). lim: entries of docb from key 0 on.
__device__ __forceinline__ int doc_at(const int* docb, int j, int Skv, int lim) {
  return (j < Skv && MATTN_IN_BOUNDS(kSiteFwdDoc, j, lim)) ? docb[j] : -1;
}

// A key tile is masked element by element when the lists call it partial or
// it runs past Skv (its columns from Skv - j0 on hold zero-filled keys).
__device__ __forceinline__ bool elementwise_tile(const Unit& U, int j, int kt, int Skv) {
  return U.partial(j) || (kt + 1) * kTile > Skv;
}

// TMA loads of one 128-row K or V tile of (b, kv head hk) at key tile kt,
// called by the whole producer warp (issue: whether copies are issued at
// all): one box per 64 columns, issued by lane 0, or, from a paged cache, one
// box per page and 64 columns (pages past the last one holding keys repeat
// it: their rows are masked), lane q reading page q's table entry and
// issuing its boxes, so the table reads of a tile overlap instead of each
// waiting for the previous one. The boxes of page q land q * page_size rows
// into the tile, a multiple of the 8-row swizzle period.
template <int kBoxes, int kBoxBytes, bool kPaged>
__device__ __forceinline__ void load_kv_tile(uint8_t* dst, const CUtensorMap* map,
                                             uint64_t* bar, const int* page_table, int ps,
                                             int pages_per_seq, int Skv, int Hkv, int b, int hk,
                                             int kt, int lane, bool issue) {
  if constexpr (!kPaged) {
    if (issue && lane == 0) {
#pragma unroll
      for (int bx = 0; bx < kBoxes; ++bx)
        tma_load_3d(dst + bx * kBoxBytes, map, bar, bx * 64, kt * kTile, b * Hkv + hk);
    }
    return;
  }
  const int per = kTile / ps;  // <= 8 pages per tile (page size >= 16)
  const int last = (Skv + ps - 1) / ps - 1;
  if (issue && lane < per) {
    const int q = lane;
    const int lp = min(kt * per + q, last);
    const int phys = MATTN_IN_BOUNDS(kSiteFwdPage, lp, pages_per_seq)
                         ? page_table[(size_t)b * pages_per_seq + lp]
                         : 0;
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_load_3d(dst + bx * kBoxBytes + q * ps * 128, map, bar, bx * 64, 0, phys * Hkv + hk);
  }
}

// Per-row, per-tile constants of the score transform.
struct TileCtx {
  float sl2, sc, cl2, slope, slope2, scale, inv_cap;
  float base;        // j0 - i: (j - i) = base + c
  int hi, lo, pre;   // mask bounds on the column c (see transform_tile)
  const int* wdoc;   // document ids of the key tile (shared memory), or nullptr
  int doc_i;
  uint32_t modes;    // per 32-column chunk of a partial tile (chunk_modes)
  // Relative-position bias window of this warp's 32 rows (shared memory), or
  // nullptr: row i = (first row of the warp) + lane and column c read entry
  // 127 + lane - c, the table value for distance i - j.
  const float* rb;
  // Soft-cap without the bias terms: |s| <= plim (|s / cap| <= 1) allows the
  // polynomial form s * Q(s^2) of cap * log2(e) * tanh(s / cap) (tanh_poly).
  float plim;
  float pa[4];
};

// Odd polynomial for tanh on [-1, 1]: tanh(y) ~ y * sum_k c_k * y^(2k),
// a least-squares fit of tanh(y) / y in y^2 on Chebyshev nodes of [0, 1],
// reweighted toward the minimax relative error: at most 8.2e-5 relative
// (fp32 Horner evaluation included), below the 2^-10.9 of tanh.approx.

// Coefficients of s * Q(s^2) = cap * log2(e) * tanh(s * sc) for |s * sc| <= 1,
// with sc = scale / cap: a_k = c_k * sc^(2k+1) * cap * log2(e).
__device__ __forceinline__ void tanh_poly_coeffs(float sc, float cl2, float* a) {
  const float sc2 = sc * sc;
  const float f0 = sc * cl2, f1 = f0 * sc2, f2 = f1 * sc2, f3 = f2 * sc2;
  a[0] = 0.99991864f * f0;
  a[1] = -0.3306548f * f1;
  a[2] = 0.11889856f * f2;
  a[3] = -0.02663025f * f3;
}

__device__ __forceinline__ float rb_at(const TileCtx& t, int c) {
  return t.rb[127 + (int)(threadIdx.x & 31) - c];
}

// Starts the copy of a warp's bias window: dst[k] = tab[first + k] for
// k < kRbWindow (indices clamped to the table; the clamped entries belong to
// rows or keys past the sequence ends, which are masked or not stored), as
// one cp.async group.
template <int W>
__device__ __forceinline__ void rb_fill(float* dst, const float* tab, int len, int first) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < W / 32; ++m) {
    const int k = lane + 32 * m;
    int idx = first + k;
    idx = idx < 0 ? 0 : (idx >= len ? len - 1 : idx);
    cp_async4(dst + k, tab + idx);
  }
  cp_async_commit();
}

constexpr uint32_t kChunkKept = 0, kChunkMasked = 1, kChunkMixed = 2;

// Whole-warp bounded wait (every lane polls; the result is the same for all).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, wd));
}

// S = Q K^T over D (K-major operands, 128-byte swizzle): K-step kk advances
// 32 bytes inside a 64-column box and moves to the next box every 4 steps.
// Called by the whole (converged) MMA warp; lane 0 issues (mma_ss_warp).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
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

// O += P V: P (bf16, 8 TMEM columns per 16 keys) times V (MN-major); K-step kk
// advances 16 key rows = 2048 bytes. Called by the whole MMA warp.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
  uint32_t a[8];
  uint64_t b[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    a[kk] = p_tmem + kk * 8;
    b[kk] = b_desc + (uint64_t)((kk * 16 * 128) >> 4);
  }
  mma_ts_warp<8>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// Loads n32 x 32 columns of this thread's TMEM lane into s (one wait for all).
__device__ __forceinline__ void load_cols(uint32_t col, float* s, int n32) {
  uint32_t* r = reinterpret_cast<uint32_t*>(s);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < n32) tmem_ld32(col + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < n32) tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(r + 32 * c));
}

// s[0..N) <- score_mod(s) in log2 units minus `shift` for the columns
// c0 .. c0+N-1 of the tile; masked entries -inf.
template <int SCORE, int N>
__device__ __forceinline__ void transform_cols(float* s, int c0, const TileCtx& t, float shift,
                                               bool partial) {
  constexpr bool kRB = (SCORE & 4) != 0;  // relative-position bias
  if constexpr ((SCORE & 3) == 0) {
    const float2 m2 = make_float2(t.sl2, t.sl2), sh2 = make_float2(-shift, -shift);
#pragma unroll
    for (int c = 0; c < N; c += 2) {
      const float2 e = ffma2(make_float2(s[c], s[c + 1]), m2, sh2);
      s[c] = e.x;
      s[c + 1] = e.y;
    }
    if constexpr (kRB) {
#pragma unroll
      for (int c = 0; c < N; ++c) s[c] = fmaf(rb_at(t, c0 + c), kLog2e, s[c]);
    }
  } else if constexpr ((SCORE & 3) == 1) {
    const float b0 = fmaf(t.slope2, t.base + float(c0), -shift);
#pragma unroll
    for (int c = 0; c < N; ++c) s[c] = fmaf(s[c], t.sl2, fmaf(t.slope2, float(c), b0));
    if constexpr (kRB) {
#pragma unroll
      for (int c = 0; c < N; ++c) s[c] = fmaf(rb_at(t, c0 + c), kLog2e, s[c]);
    }
  } else {
    bool poly = false;
    if constexpr (SCORE == 2) {
      // Soft-cap alone: where every |s| of the warp's columns is in the
      // polynomial's range, tanh is evaluated as s * Q(s^2) with packed FMAs
      // instead of on the special-function unit, which the exponentiation
      // also needs (tanh.approx takes twice the issue time of ex2.approx
      // there); otherwise the whole call takes the tanh.approx path below.
      float mx = 0.0f;
#pragma unroll
      for (int c = 0; c < N; ++c) mx = fmaxf(mx, fabsf(s[c]));
      if (__all_sync(0xffffffffu, mx <= t.plim)) {
        const float2 a0 = make_float2(t.pa[0], t.pa[0]), a1 = make_float2(t.pa[1], t.pa[1]),
                     a2 = make_float2(t.pa[2], t.pa[2]), a3 = make_float2(t.pa[3], t.pa[3]);
        const float2 sh2 = make_float2(-shift, -shift);
#pragma unroll
        for (int c = 0; c < N; c += 2) {
          const float2 x = make_float2(s[c], s[c + 1]);
          const float2 u = fmul2(x, x);
          float2 q = ffma2(a3, u, a2);
          q = ffma2(q, u, a1);
          q = ffma2(q, u, a0);
          const float2 e = ffma2(q, x, sh2);
          s[c] = e.x;
          s[c + 1] = e.y;
        }
        poly = true;
      }
    }
    if (!poly) {
      const float b0 = t.slope * (t.base + float(c0));
      const float2 cl = make_float2(t.cl2, t.cl2), sh2 = make_float2(-shift, -shift);
#pragma unroll
      for (int c = 0; c < N; c += 2) {
        float2 y;
        if constexpr ((SCORE & 3) == 2) {
          y = fmul2(make_float2(s[c], s[c + 1]), make_float2(t.sc, t.sc));
        } else {
          y.x = fmaf(s[c], t.scale, fmaf(t.slope, float(c), b0)) * t.inv_cap;
          y.y = fmaf(s[c + 1], t.scale, fmaf(t.slope, float(c + 1), b0)) * t.inv_cap;
        }
        if constexpr (kRB) {  // the bias enters before the cap
          y.x = fmaf(rb_at(t, c0 + c), t.inv_cap, y.x);
          y.y = fmaf(rb_at(t, c0 + c + 1), t.inv_cap, y.y);
        }
        const float2 e = ffma2(make_float2(tanh_approx(y.x), tanh_approx(y.y)), cl, sh2);
        s[c] = e.x;
        s[c + 1] = e.y;
      }
    }
  }
  // mask_mod on a partial tile: keep (lo < c <= hi and same document) or
  // c < pre. Chunks of 32 columns that every row of the warp keeps need no
  // work and chunks no row keeps become -inf (t.modes, see chunk_modes); only
  // mixed chunks are masked element by element. There the terms are combined
  // with bitwise operators and the document ids are read unconditionally, four
  // at a time: a short-circuit form would make every element a divergent
  // branch around a load.
  if (partial) {
#pragma unroll
    for (int q = 0; q < N / 32; ++q) {
      const int a = c0 + 32 * q;  // first column of the chunk
      const uint32_t mode = (t.modes >> (2 * (a >> 5))) & 3u;
      if (mode == kChunkKept) continue;
      float* sq = s + 32 * q;
      if (mode == kChunkMasked) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sq[c] = -INFINITY;
        continue;
      }
      if (t.wdoc) {
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const int4 dv = *reinterpret_cast<const int4*>(t.wdoc + a + c);
          const int d4[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int cc = a + c + e;
            const bool keep =
                ((cc <= t.hi) & (cc > t.lo) & (d4[e] == t.doc_i)) | (cc < t.pre);
            sq[c + e] = keep ? sq[c + e] : -INFINITY;
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int cc = a + c;
          const bool keep = ((cc <= t.hi) & (cc > t.lo)) | (cc < t.pre);
          sq[c] = keep ? sq[c] : -INFINITY;
        }
      }
    }
  }
}

// Warp-uniform mode of each 32-column chunk of a partial tile, two bits per
// chunk: kept by every row of the warp, masked for every row, or mixed. From
// the rows' column bounds and the min/max document id of the chunk's keys;
// exact for "kept" and "masked", conservative ("mixed") otherwise. Integer
// compares run at half rate, so deciding whole chunks saves most of the
// per-element mask work on diagonal, window-edge and document-edge tiles.
__device__ __forceinline__ uint32_t chunk_modes(const TileCtx& t) {
  const int lane = threadIdx.x & 31;
  uint32_t modes = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int a = 32 * q;
    const bool pre_all = a + 31 < t.pre, pre_none = a >= t.pre;
    bool all = ((a + 31 <= t.hi) & (a > t.lo)) | pre_all;
    bool none = ((a > t.hi) | (a + 31 <= t.lo)) & pre_none;
    if (t.wdoc) {
      const int dl = t.wdoc[a + lane];
      const int dmin = __reduce_min_sync(0xffffffffu, dl);
      const int dmax = __reduce_max_sync(0xffffffffu, dl);
      const bool d_all = (dmin == t.doc_i) & (dmax == t.doc_i);
      const bool d_none = (t.doc_i < dmin) | (t.doc_i > dmax);
      all = (all & d_all) | pre_all;
      none = none | (d_none & pre_none);
    }
    const uint32_t m = __all_sync(0xffffffffu, all)    ? kChunkKept
                       : __all_sync(0xffffffffu, none) ? kChunkMasked
                                                       : kChunkMixed;
    modes |= m << (2 * q);
  }
  return modes;
}

// pk[0..N/2) <- bf16 pairs of 2^s; returns the fp32 sum.
template <int N>
__device__ __forceinline__ float exp2_pack(const float* s, uint32_t* pk) {
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
#pragma unroll
  for (int c = 0; c < N; c += 2) {
    const float2 pr = make_float2(ex2_approx(s[c]), ex2_approx(s[c + 1]));
    acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], pr);
    pk[c >> 1] = pack_bf16x2(pr.x, pr.y);
  }
  const float2 a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
  return a.x + a.y;
}

// PAGED: K/V come from a paged cache (a separate instantiation: the page-table
// code in the load warp measurably slowed the contiguous kernel).
template <int D, int SCORE, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdProblem p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sSlots = smem + C::kOffSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* drain = bars + 2;
  uint64_t* s_full = bars + 3;   // [2]
  uint64_t* p_full = bars + 5;   // [2]
  uint64_t* o_done = bars + 7;   // [2]
  uint64_t* o_free = bars + 9;   // [2]
  uint64_t* s_free = bars + 11;  // [2] (separate P only) S read by the softmax
  uint64_t* pv_done = bars + 13; // [2] (separate P only) P.V product complete
  uint64_t* drain2 = bars + 15;  // (separate P only) second MMA warp's products
  uint64_t* slot_full = bars + 16;
  uint64_t* slot_empty = bars + 16 + C::kSlots;
  int* sdoc = reinterpret_cast<int*>(smem + C::kOffDoc);
  uint8_t* sarea = smem + C::kOffArea;  // per-warp bias windows / output staging
  uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};

  if (threadIdx.x == 0) {
    // With separate P each head has its own MMA warp and every Q tile and
    // ring slot is released by two commits (one per warp, or two by the one
    // warp that used it).
    mbar_init(q_full, 1);
    mbar_init(q_empty, C::kDualMma ? 2 : 1);
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full + x, 1);
      mbar_init(p_full + x, kSoftmaxThreads / 32);  // one arrive per softmax warp
      mbar_init(o_done + x, 1);
      mbar_init(o_free + x, kSoftmaxThreads / 32);
      mbar_init(s_free + x, kSoftmaxThreads / 32);
      mbar_init(pv_done + x, 1);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(slot_full + s, 1);
      mbar_init(slot_empty + s, C::kDualMma ? 2 : 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_smem;

  const int num_units = count_units<D, PAGED>(p);
  // Unit fields in registers or local memory (Unit::head), as measured per
  // instantiation: registers gained 2-5 % on the contiguous kernels without
  // the bias; local memory was faster for the paged kernel without soft-cap
  // (causal B8 H16 S4096, 16-token pages: 0.71 against 0.80 ms) and for soft-
  // cap + bias (GQA prefix B2 Hq32 S8192: 1.61 against 1.82 ms), registers
  // for the paged soft-cap and the ALiBi + bias kernels (1-2 %).
  constexpr bool kUnitRegs = PAGED ? (SCORE & 2) != 0 : (SCORE & 6) != 6;
  const int group = p.Hq / p.Hkv;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  }
  if (warp == kWarpProducer) {
    // ------------------------------------------------------------- producer
    // The whole warp runs the loop (waits stay converged); lane 0 issues.
    // With ATTN_FAULT_NO_LOADS nothing is issued and the consumers' waits run out.
    const bool issue = !(p.fault_inject & ATTN_FAULT_NO_LOADS);
    const bool leader = lane == 0 && issue;
    uint32_t slot_it = 0, q_it = 0;
    bool ok = true;
    for (int r = 0; r * (int)gridDim.x < num_units && ok; ++r) {
      const int u = zigzag_unit(r);
      if (u >= num_units) continue;
      const Unit U = decode_unit<D, PAGED>(p, u);
      const int n = U.n();
      if (n == 0) continue;
      const bool two = U.h[1] >= 0;
      const int hk0 = U.h[0] / group, hk1 = two ? U.h[1] / group : hk0;
      const bool shared = !two || hk0 == hk1;
      const int hks[2] = {hk0, hk1};
      auto hk_of = [&](int x) {
        if constexpr (kUnitRegs) return x ? hk1 : hk0;
        else return hks[x];
      };
      ok = __all_sync(0xffffffffu, wait_bounded(q_empty, (q_it & 1) ^ 1, wd));
      if (!ok) break;
      if (leader) {
        mbar_arrive_expect_tx(q_full, (two ? 2 : 1) * C::kTileBytes);
        for (int x = 0; x < (two ? 2 : 1); ++x) {
          const int slice = U.b * p.Hq + U.head<kUnitRegs>(x);
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_3d(sQ + x * C::kTileBytes + bx * C::kBoxBytes, &tm_q, q_full, bx * 64,
                        U.qtile<kUnitRegs>(x) * kTile, slice);
        }
      }
      __syncwarp();
      ++q_it;
      for (int j = 0; j < n && ok; ++j) {
        const int kt = U.kt(j);
        // order: K_A, [K_B], V_A, [V_B]
        for (int t = 0; t < (shared ? 2 : 4) && ok; ++t) {
          const int per = shared ? 1 : 2;
          const bool is_v = t >= per;
          const int x = shared ? 0 : (t % 2);
          const int slot = slot_it % C::kSlots;
          ok = __all_sync(0xffffffffu,
                          wait_bounded(slot_empty + slot, ((slot_it / C::kSlots) & 1) ^ 1, wd));
          if (!ok) break;
          if (leader) mbar_arrive_expect_tx(slot_full + slot, C::kTileBytes);
          __syncwarp();
          load_kv_tile<C::kBoxes, C::kBoxBytes, PAGED>(sSlots + slot * C::kTileBytes,
                                                is_v ? &tm_v : &tm_k, slot_full + slot,
                                                p.page_table, p.page_size, p.pages_per_seq,
                                                p.Skv, p.Hkv, U.b, hk_of(x), kt, lane, issue);
          __syncwarp();
          ++slot_it;
        }
      }
    }
    if (!ok && !(p.fault_inject & ATTN_FAULT_NO_LOADS)) {  // let copies in flight land
      for (uint32_t k = 0; k < C::kSlots && k < slot_it; ++k) {
        const uint32_t it = slot_it - 1 - k;
        wait_drain(slot_full + it % C::kSlots, (it / C::kSlots) & 1);
      }
      if (q_it > 0) wait_drain(q_full, (q_it - 1) & 1);
    }
  } else if (warp == kWarpMma || (C::kDualMma && warp == kWarpMma2)) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (waits stay converged); lane 0 issues the
    // products and the commits, each product's K-steps as one block
    // (mma_ss_warp, mma_ts_warp). Loop state stays in registers and the
    // shared-memory descriptors are precomputed: the start-address field is
    // in 16-byte units, so an offset is added as (bytes >> 4).
    constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false);
    constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
    const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = sdesc_sw128(smem_u32(sSlots), 16, 1024);
    const uint64_t dV0 = sdesc_sw128(smem_u32(sSlots), C::kBoxBytes, 1024);
    if constexpr (!C::kDualMma) {
      uint32_t slot_it = 0, q_it = 0, p_it0 = 0, p_it1 = 0, o_it0 = 0, o_it1 = 0;
      bool ok = true;
      for (int r = 0; r * (int)gridDim.x < num_units && ok; ++r) {
        const int u = zigzag_unit(r);
        if (u >= num_units) continue;
        const Unit U = decode_unit<D, PAGED>(p, u);
        const int n = U.n();
        if (n == 0) continue;
        const int nx = U.h[1] >= 0 ? 2 : 1;
        const bool shared = nx == 1 || (U.h[0] / group == U.h[1] / group);
        const uint32_t T = shared ? 2u : 4u;  // ring slots per key tile
        ok = wait_warp(q_full, q_it & 1, wd);
        if (!ok) break;
        ++q_it;
        tc_fence_after();
        // S_x(0) for both heads
        for (int x = 0; x < nx && ok; ++x) {
          const uint32_t seq = slot_it + (shared ? 0u : (uint32_t)x);
          const uint32_t slot = seq % C::kSlots;
          if (x == 0 || !shared) {
            ok = wait_warp(slot_full + slot, (seq / C::kSlots) & 1, wd);
            if (!ok) break;
            tc_fence_after();
          }
          issue_qk<D>(tmem + 128u * x, dQ0 + ((x * C::kTileBytes) >> 4),
                      dK0 + ((slot * C::kTileBytes) >> 4), kIdescQK);
          mma_commit_warp(s_full + x);
          if (!shared || x == nx - 1) mma_commit_warp(slot_empty + slot);
          __syncwarp();
        }
        if (ok && n == 1) mma_commit_warp(q_empty);
        // The tile loop, compiled once for units whose two heads share the
        // K/V tiles (kSh: two ring slots per key tile) and once for units
        // whose heads have their own (four slots). With shared tiles the
        // slots of V_j and K_{j+1} are waited for before P_x(j): K_{j+1} is
        // loaded a whole tile ahead, so nothing but the P wait stands between
        // the softmax's hand-over and the two products (GQA prefix-LM
        // workload 5 % faster). With four slots per tile K_{j+1} arrives only
        // after V_j's successors and the waits stay after the P wait (waiting
        // early there, or the early-wait code in the same loop, was 2-4 %
        // slower on the multi-head workloads).
        auto tile_loop = [&](auto sh_tag) {
          constexpr bool kSh = decltype(sh_tag)::value;
          for (int j = 0; j < n && ok; ++j) {
            for (int x = 0; x < nx && ok; ++x) {
              const uint32_t vseq = slot_it + j * T + (kSh ? 1u : 2u + x);
              const uint32_t vslot = vseq % C::kSlots;
              const uint32_t kseq = slot_it + (j + 1) * T + (kSh ? 0u : (uint32_t)x);
              const uint32_t kslot = kseq % C::kSlots;
              if (kSh && x == 0) {
                ok = wait_warp(slot_full + vslot, (vseq / C::kSlots) & 1, wd);
                if (!ok) break;
                if (j + 1 < n) {
                  ok = wait_warp(slot_full + kslot, (kseq / C::kSlots) & 1, wd);
                  if (!ok) break;
                }
              }
              // O_x += P_x V_j
              ok = wait_warp(p_full + x, (x ? p_it1 : p_it0) & 1, wd);
              if (!ok) break;
              if (x) ++p_it1; else ++p_it0;
              if (j == 0) {
                ok = wait_warp(o_free + x, ((x ? o_it1 : o_it0) & 1) ^ 1, wd);
                if (!ok) break;
                if (x) ++o_it1; else ++o_it0;
              }
              if (!kSh) {
                ok = wait_warp(slot_full + vslot, (vseq / C::kSlots) & 1, wd);
                if (!ok) break;
              }
              tc_fence_after();
              issue_pv<D>(tmem + C::kColO0 + D * x, tmem + 128u * x,
                          dV0 + ((vslot * C::kTileBytes) >> 4), kIdescPV, j > 0);
              if (!kSh || x == nx - 1) mma_commit_warp(slot_empty + vslot);
              __syncwarp();
              if (j + 1 < n) {  // S_x(j+1)
                if (!kSh) {
                  ok = wait_warp(slot_full + kslot, (kseq / C::kSlots) & 1, wd);
                  if (!ok) break;
                  tc_fence_after();
                }
                issue_qk<D>(tmem + 128u * x, dQ0 + ((x * C::kTileBytes) >> 4),
                            dK0 + ((kslot * C::kTileBytes) >> 4), kIdescQK);
                mma_commit_warp(s_full + x);
                if (!kSh || x == nx - 1) mma_commit_warp(slot_empty + kslot);
                __syncwarp();
              } else {
                mma_commit_warp(o_done + x);
              }
            }
            if (ok && j + 1 == n - 1) mma_commit_warp(q_empty);
          }
        };
        if (shared) tile_loop(std::true_type{});
        else tile_loop(std::false_type{});
        __syncwarp();
        slot_it += n * T;
      }
    } else {
      // Separate P, one MMA warp per head: warp kWarpMma serves head A and
      // kWarpMma2 head B, so neither head's products wait behind the other's.
      // S_x(j+1) = Q_x K_{j+1}^T is issued as soon as the softmax has read
      // S_x(j) (s_free), before P_x(j) exists; O_x += P_x(j) V_j follows when
      // P_x(j) is ready. kq counts this head's Q.K^T products (tile k waits
      // for s_free phase k-1), kp its P.V products. Every Q tile and ring slot
      // gets exactly two release commits: one from each warp when both heads
      // read it, else two from the warp that did.
      const int x = warp == kWarpMma ? 0 : 1;
      uint32_t slot_it = 0, q_it = 0, kq = 0, kp = 0, o_it = 0;
      bool ok = true;
      for (int r = 0; r * (int)gridDim.x < num_units && ok; ++r) {
        const int u = zigzag_unit(r);
        if (u >= num_units) continue;
        const Unit U = decode_unit<D, PAGED>(p, u);
        const int n = U.n();
        if (n == 0) continue;
        const int nx = U.h[1] >= 0 ? 2 : 1;
        const bool shared = nx == 1 || (U.h[0] / group == U.h[1] / group);
        const uint32_t T = shared ? 2u : 4u;  // ring slots per key tile
        const uint32_t base = slot_it;
        slot_it += n * T;
        ++q_it;
        if (x >= nx) continue;  // single-head unit: head B's warp has nothing to do
        const bool both = nx == 2 && shared;  // the other warp releases the same slots
        ok = wait_warp(q_full, (q_it - 1) & 1, wd);
        if (!ok) break;
        // S_x(jj) = Q_x K_jj^T
        auto do_qk = [&](int jj) -> bool {
          if constexpr (C::kSepP) {
            if (kq > 0 && !wait_warp(s_free + x, (kq - 1) & 1, wd)) return false;
          }
          const uint32_t kseq = base + jj * T + (shared ? 0u : (uint32_t)x);
          const uint32_t kslot = kseq % C::kSlots;
          if (!wait_warp(slot_full + kslot, (kseq / C::kSlots) & 1, wd)) return false;
          tc_fence_after();
          issue_qk<D>(tmem + 128u * x, dQ0 + ((x * C::kTileBytes) >> 4),
                      dK0 + ((kslot * C::kTileBytes) >> 4), kIdescQK);
          mma_commit_warp(s_full + x);
          mma_commit_warp(slot_empty + kslot);
          if (!both) mma_commit_warp(slot_empty + kslot);
          if (jj + 1 == n) {  // the unit's last Q.K^T for this head
            mma_commit_warp(q_empty);
            if (nx == 1) mma_commit_warp(q_empty);
          }
          __syncwarp();
          ++kq;
          return true;
        };
        // O_x += P_x(jj) V_jj
        auto do_pv = [&](int jj) -> bool {
          if (!wait_warp(p_full + x, kp & 1, wd)) return false;
          if (jj == 0) {
            if (!wait_warp(o_free + x, (o_it & 1) ^ 1, wd)) return false;
            ++o_it;
          }
          const uint32_t vseq = base + jj * T + (shared ? 1u : 2u + x);
          const uint32_t vslot = vseq % C::kSlots;
          if (!wait_warp(slot_full + vslot, (vseq / C::kSlots) & 1, wd)) return false;
          tc_fence_after();
          const uint32_t pcol = C::kSepP ? C::kColP + 64u * x : 128u * x;
          issue_pv<D>(tmem + C::kColO0 + D * x, tmem + pcol,
                      dV0 + ((vslot * C::kTileBytes) >> 4), kIdescPV, jj > 0);
          if (C::kSepP) mma_commit_warp(pv_done + x);
          mma_commit_warp(slot_empty + vslot);
          if (!both) mma_commit_warp(slot_empty + vslot);
          if (jj + 1 == n) mma_commit_warp(o_done + x);
          __syncwarp();
          ++kp;
          return true;
        };
        if constexpr (C::kSepP) {
          // separate P: S_x(j+1) as soon as S_x(j) is read, then P_x(j) V_j
          for (int j = -1; j < n && ok; ++j) {
            if (j + 1 < n) ok = do_qk(j + 1);
            if (ok && j >= 0) ok = do_pv(j);
          }
        } else {
          // P overwrites S: S_x(j+1) only after P_x(j) V_j has been issued
          ok = do_qk(0);
          for (int j = 0; j < n && ok; ++j) {
            ok = do_pv(j);
            if (ok && j + 1 < n) ok = do_qk(j + 1);
          }
        }
      }
      // all products issued by this warp are complete before TMEM is freed
      uint64_t* dr = x ? drain2 : drain;
      mma_commit_warp(dr);
      __syncwarp();
      wait_drain(dr, 0);
    }
    if constexpr (!C::kDualMma) {
      // all products issued by this warp are complete before TMEM is freed
      mma_commit_warp(drain);
      __syncwarp();
      wait_drain(drain, 0);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int x = warp / 4;            // head slot 0 or 1
    const int t = threadIdx.x & 127;   // query row within the tile == TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t colS = tmem + lane_base + 128u * x;
    const uint32_t colO = tmem + lane_base + C::kColO0 + D * x;
    int* wdoc = sdoc + warp * kTile;   // this warp's copy of the key tile's document ids
    float* wrb = reinterpret_cast<float*>(sarea + warp * C::kWarpArea);  // two bias windows
    const float sl2 = p.score.scale * kLog2e;              // raw score -> log2 units
    const float sc = p.score.scale / p.score.softcap;      // raw score -> tanh argument
    const float cl2 = p.score.softcap * kLog2e;            // tanh -> log2 units
    float pa[4];
    tanh_poly_coeffs(sc, cl2, pa);
    const float plim = p.score.softcap / p.score.scale;    // |s| <= plim: |s / cap| <= 1
    uint32_t s_it = 0, o_it = 0;
    bool ok = true;
    for (int rr = 0; rr * (int)gridDim.x < num_units && ok; ++rr) {
      const int u = zigzag_unit(rr);
      if (u >= num_units) continue;
      const Unit U = decode_unit<D, PAGED>(p, u);
      const int h = U.head<kUnitRegs>(x);
      if (h < 0) continue;
      const int n = U.n();
      const int i = U.qtile<kUnitRegs>(x) * kTile + t;
      const bool row_in = i < p.Sq;  // a last query tile may run past Sq
      const size_t orow = ((size_t)(U.b * p.Hq + h) * p.Sq + i);
      __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o) + orow * D;
      const size_t total_rows = (size_t)p.B * p.Hq * p.Sq;
      (void)total_rows;
      if (n == 0) {
        if (row_in && MATTN_IN_BOUNDS(kSiteFwdO, orow, total_rows)) {
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(O)[c] = z;
          p.lse[orow] = -INFINITY;
        }
        continue;
      }
      const float slope = (SCORE & 1) ? alibi_slope(p.score, h) : 0.0f;
      const float slope2 = slope * kLog2e;
      // document ids by key column and query row of this call (the row of
      // doc_id is indexed by absolute position)
      const int* docb = (p.variant & ATTN_MASK_DOCUMENT)
                            ? p.mask.doc_id + (size_t)U.b * p.mask.doc_len + p.mask.kv_off
                            : nullptr;
      const int doc_lim = p.mask.doc_len - p.mask.kv_off;
      (void)doc_lim;
      const int doc_i =
          (docb && row_in && MATTN_IN_BOUNDS(kSiteFwdDoc, p.mask.q_off + i, p.mask.doc_len))
              ? p.mask.doc_id[(size_t)U.b * p.mask.doc_len + p.mask.q_off + i]
              : 0;
      const int dqk = p.mask.q_off - p.mask.kv_off;  // absolute i - j = (i - j) + dqk
      const int P = (p.variant & ATTN_MASK_PREFIX) ? p.mask.prefix_len[U.b] : INT_MIN;
      float m_ref = -INFINITY, l = 0.0f;
      // Key-tile indices are read two tiles ahead and the document ids of a
      // partial tile one tile ahead, so neither global read waits on the
      // critical path (lane l holds ids l, l+32, l+64, l+96).
      int kt_cur = U.kt(0), kt_n1 = n > 1 ? U.kt(1) : 0;
      // relative-position bias of this head: windows copied one tile ahead
      const float* rtab =
          (SCORE & 4) ? p.score.rel_bias + (size_t)h * p.score.rb_len : nullptr;
      const int rb_first = U.qtile<kUnitRegs>(x) * kTile + (warp & 3) * 32 - 127 + p.score.rb_zero;  // minus j0
      if (rtab) rb_fill<C::kRbWindow>(wrb, rtab, p.score.rb_len, rb_first - kt_cur * kTile);
      int dcur[4] = {0, 0, 0, 0};
      if (docb && elementwise_tile(U, 0, kt_cur, p.Skv)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) dcur[c] = doc_at(docb, kt_cur * kTile + lane + 32 * c, p.Skv, doc_lim);
      }

      for (int j = 0; j < n; ++j) {
        const int kt = kt_cur;
        const int kt_n2 = j + 2 < n ? U.kt(j + 2) : 0;
        int dnext[4] = {0, 0, 0, 0};
        if (docb && j + 1 < n && elementwise_tile(U, j + 1, kt_n1, p.Skv)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) dnext[c] = doc_at(docb, kt_n1 * kTile + lane + 32 * c, p.Skv, doc_lim);
        }
        const int j0 = kt * kTile;
        const bool partial = elementwise_tile(U, j, kt, p.Skv);
        if (partial && docb) {
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 4; ++c) wdoc[lane + 32 * c] = dcur[c];
          __syncwarp();
        }
        const float* rb_win = nullptr;
        if (rtab) {
          // the next tile's window goes to the other buffer (read two tiles
          // ago: every lane is past it), then this tile's must have landed
          __syncwarp();
          if (j + 1 < n)
            rb_fill<C::kRbWindow>(wrb + ((j + 1) & 1) * C::kRbWindow, rtab, p.score.rb_len,
                                  rb_first - kt_n1 * kTile);
          else
            cp_async_commit();  // empty group: the wait below still covers this tile
          cp_async_wait<1>();
          __syncwarp();
          rb_win = wrb + (j & 1) * C::kRbWindow;
        }
        kt_cur = kt_n1;
        kt_n1 = kt_n2;
#pragma unroll
        for (int c = 0; c < 4; ++c) dcur[c] = dnext[c];
        TileCtx tc{sl2, sc, cl2, slope, slope2, p.score.scale, 1.0f / p.score.softcap,
                   float(j0 - i - dqk),
                   min((p.variant & ATTN_MASK_CAUSAL) ? i + dqk - j0 : INT_MAX, p.Skv - 1 - j0),
                   (p.variant & ATTN_MASK_WINDOW) ? i + dqk - j0 - p.mask.window : INT_MIN,
                   P == INT_MIN ? INT_MIN : min(P - p.mask.kv_off, p.Skv) - j0,
                   docb ? wdoc : nullptr, doc_i, 0u, rb_win, plim,
                   {pa[0], pa[1], pa[2], pa[3]}};
        if (partial) tc.modes = chunk_modes(tc);  // before the wait: off the critical path
        ok = __all_sync(0xffffffffu, wait_bounded(s_full + x, s_it & 1, wd));
        if (!ok) break;
        ++s_it;
        tc_fence_after();
        // Steady state: exponentiate against the current reference max with no
        // max pass, 64 columns at a time, keeping P as packed bf16. A tile whose
        // sum is not finite or exceeds 2^64 (the first tile, or a tile whose
        // scores outgrow the reference) is redone from S (still in TMEM) with
        // its true maximum, rescaling l and O.
        uint32_t pk[64];
        float tsum = 0.0f;
        bool redo;
        {
          // the second half's load is in flight while the first half is processed
          float v0[64], v1[64];
          load_cols(colS, v0, 2);
          tmem_ld32(colS + 64, *reinterpret_cast<uint32_t(*)[32]>(v1));
          tmem_ld32(colS + 96, *reinterpret_cast<uint32_t(*)[32]>(v1 + 32));
          if (__all_sync(0xffffffffu, m_ref == -INFINITY)) {
            // No row of the warp has a reference yet (a unit's first tile,
            // or every earlier tile was masked for all of them): both halves
            // are transformed first and the tile's own row maximum becomes
            // the reference, so the largest weight is exactly 1 as in the max
            // pass below. A row masked in the whole tile keeps no reference
            // (its weights are 0 here); where some rows of a warp have one
            // and others not, the others' sums come out infinite or NaN and
            // the redo below sets their reference from the tile's maximum.
            transform_cols<SCORE, 64>(v0, 0, tc, 0.0f, partial);
            tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(v1));
            tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(v1 + 32));
            transform_cols<SCORE, 64>(v1, 64, tc, 0.0f, partial);
            const float mt = fmaxf(row_max<64>(v0), row_max<64>(v1));
            m_ref = mt;
            const float m_use = mt == -INFINITY ? 0.0f : mt;
            const float2 sh = make_float2(-m_use, -m_use);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              const float2 e0 = fadd2(make_float2(v0[c], v0[c + 1]), sh);
              v0[c] = e0.x;
              v0[c + 1] = e0.y;
              const float2 e1 = fadd2(make_float2(v1[c], v1[c + 1]), sh);
              v1[c] = e1.x;
              v1[c + 1] = e1.y;
            }
            tsum = exp2_pack<64>(v0, pk);
            tsum += exp2_pack<64>(v1, pk + 32);
          } else {
            transform_cols<SCORE, 64>(v0, 0, tc, m_ref, partial);
            tsum = exp2_pack<64>(v0, pk);
            tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(v1));
            tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(v1 + 32));
            transform_cols<SCORE, 64>(v1, 64, tc, m_ref, partial);
            tsum += exp2_pack<64>(v1, pk + 32);
          }
          redo = !(tsum <= 18446744073709551616.0f);
        }
        if (__any_sync(0xffffffffu, redo)) {
          // pass 1: the tile's maximum, 32 columns at a time
          float mt = -INFINITY;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float v[32];
            load_cols(colS + 32 * qq, v, 1);
            transform_cols<SCORE, 32>(v, 32 * qq, tc, 0.0f, partial);
            mt = fmaxf(mt, row_max<32>(v));
          }
          const float m_new = redo ? fmaxf(m_ref, mt) : m_ref;
          const float alpha = ex2_approx(m_ref - m_new);  // m_ref = -inf gives 0
          const bool need_o = redo && j > 0 && m_ref != -INFINITY && m_new > m_ref;
          if (redo && m_new > m_ref) l *= alpha;
          if (__any_sync(0xffffffffu, need_o)) {
            if constexpr (C::kSepP) {
              // S(j) was computed before the previous tile's P.V: let it land in O
              ok = __all_sync(0xffffffffu, wait_bounded(pv_done + x, s_it & 1, wd));
              if (!ok) break;
              tc_fence_after();
            }
            const float a = need_o ? alpha : 1.0f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(colO + 32 * c, r);
              tmem_ld_wait_regs(r);
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a);
              tmem_st32(colO + 32 * c, r);
            }
          }
          m_ref = m_new;
          // pass 2: exponentiate against the new reference
          const float m_use = m_ref == -INFINITY ? 0.0f : m_ref;
          tsum = 0.0f;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            float v[32];
            load_cols(colS + 32 * qq, v, 1);
            transform_cols<SCORE, 32>(v, 32 * qq, tc, m_use, partial);
            tsum += exp2_pack<32>(v, pk + 16 * qq);
          }
        }
        l += tsum;
        uint32_t colP = colS;  // P overwrites S
        if constexpr (C::kSepP) {
          // S(j) is read: the next Q.K^T may overwrite it. P goes to its own
          // columns once the previous tile's P.V product has consumed them.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(s_free + x);
          if (s_it > 1) {
            ok = __all_sync(0xffffffffu, wait_bounded(pv_done + x, s_it & 1, wd));
            if (!ok) break;
            tc_fence_after();
          }
          colP = tmem + lane_base + C::kColP + 64u * x;
        }
        tmem_st32(colP, *reinterpret_cast<uint32_t(*)[32]>(pk));
        tmem_st32(colP + 32, *reinterpret_cast<uint32_t(*)[32]>(pk + 32));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + x);
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, LSE = ln(sum exp); the LSE store goes first
      // so that it does not queue behind the output's
      if (row_in && MATTN_IN_BOUNDS(kSiteFwdLse, orow, total_rows))
        p.lse[orow] = l > 0.0f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      ok = __all_sync(0xffffffffu, wait_bounded(o_done + x, o_it & 1, wd));
      if (!ok) break;
      ++o_it;
      tc_fence_after();
      // O is written through shared memory so that the global stores are
      // coalesced: per 32 columns, each thread puts its row's 64 bytes in the
      // warp's staging area (16-byte units swizzled by (row >> 1) & 3: no bank
      // conflicts either way), then a store instruction covers 8 whole
      // 64-byte row segments instead of one 16-byte piece of 32 rows.
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      uint4* stg = reinterpret_cast<uint4*>(sarea + warp * C::kWarpArea);
      const int row0 = U.qtile<kUnitRegs>(x) * kTile + (warp & 3) * 32;  // the warp's first row
      __nv_bfloat16* Oh = static_cast<__nv_bfloat16*>(p.o) + (size_t)(U.b * p.Hq + h) * p.Sq * D;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t r[64];
        tmem_ld32(colO + 64 * cc, *reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld32(colO + 64 * cc + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(r));
        tmem_ld_wait_regs(*reinterpret_cast<uint32_t(*)[32]>(r + 32));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = 2 * cc + hh;  // 32-column chunk
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(r[32 * hh + 2 * e]) * inv,
                                __uint_as_float(r[32 * hh + 2 * e + 1]) * inv);
          __syncwarp();  // the previous chunk's reads of the staging area are done
#pragma unroll
          for (int e = 0; e < 4; ++e)
            stg[lane * 4 + (e ^ ((lane >> 1) & 3))] =
                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int rr = 8 * k + (lane >> 2), e = lane & 3;
            const uint4 v = stg[rr * 4 + (e ^ ((rr >> 1) & 3))];
            if (row0 + rr < p.Sq &&
                MATTN_IN_BOUNDS(kSiteFwdO, (size_t)(U.b * p.Hq + h) * p.Sq + row0 + rr, total_rows))
              *reinterpret_cast<uint4*>(Oh + (size_t)(row0 + rr) * D + 32 * c + 8 * e) = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free + x);
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

// ----------------------------------------------------------------- host side
template <int D, int SCORE, bool PAGED = false>
cudaError_t launch_typed(const FwdProblem& p, cudaStream_t stream) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv;
  const bool paged = PAGED;
  const long long kv_slices = paged ? (long long)p.num_pages * p.Hkv : (long long)p.B * p.Hkv;
  const int kv_rows = paged ? p.page_size : p.Skv;
  if (!make_map_bf16_3d(&mq, p.q, (long long)p.B * p.Hq, p.Sq, D) ||
      !make_map_bf16_3d(&mk, p.k, kv_slices, kv_rows, D, paged ? p.page_size : kTile) ||
      !make_map_bf16_3d(&mv, p.v, kv_slices, kv_rows, D, paged ? p.page_size : kTile))
    return cudaErrorInvalidValue;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fwd_tc_kernel<D, SCORE, PAGED>,
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
    if (cudaFuncGetAttributes(&fa, fwd_tc_kernel<D, SCORE, PAGED>) == cudaSuccess)
      regs = fa.numRegs;
  });
  if (regs < 0 || 2LL * kSoftmaxThreads * kRegsSoftmax + 128LL * kRegsOther >
                      (long long)regs * kThreads)
    return cudaErrorInvalidConfiguration;
  const int units = count_units<D, PAGED>(p);
  const int grid = units < sm_count() ? units : sm_count();
  if (grid == 0) return cudaSuccess;
  fwd_tc_kernel<D, SCORE, PAGED><<<grid, kThreads, C::kSmemAlloc, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace
}  // namespace mattn
