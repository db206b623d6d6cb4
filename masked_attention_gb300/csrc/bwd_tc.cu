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
//                  A += bf16(P g (dP - Dhat)) K, B += bf16(P g) K,
//                  dQ = scale (A - (Delta - Dhat) B), g = score_mod'.
//                  A carries the well-conditioned bulk (like dS itself), the
//                  correction term is small. Delta goes to the workspace.
//   bwd_kernel<dKV> per (b, kv head, key tile), over the query heads of its
//                  group and the query tiles of the transposed block mask:
//                  S^T = K Q^T, P^T, dV += P^T dO, dP^T = V dO^T,
//                  dS^T = P^T (dP^T - Delta) score_mod', dK += dS^T Q (x scale)
//
// Both kernels share one structure (192 threads):
//   warps 0-3  compute: thread t owns row t of the fixed tile (TMEM lane t)
//   warp  4    TMA producer: the fixed tiles once per unit, then the streamed
//              tiles (plus LSE, Delta and document ids of the dKV stream) into
//              a ring
//   warp  5    MMA issuer and TMEM owner
// Tensor memory: S [0,128), dP [128,256), accumulators from 256 (dQ: A, B;
// dKV: dV, dK). The bf16 A operands of the TS products (dQ: P g and P g dP;
// dKV: P and dS) overwrite the first 64 columns of S and dP.
#include <cmath>
#include <mutex>

#include "host_util.h"
#include "launch.h"

namespace mattn {
namespace {

constexpr int kThreads = 192;
constexpr int kWarpProducer = 4;
constexpr int kWarpMma = 5;
enum Mode { kDQ = 0, kDKV = 1 };

template <int D, int MODE>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxes = D / 64;
  static constexpr int kBoxBytes = kTile * 128;
  static constexpr int kSlots = D == 128 ? 2 : 4;
  // extra bytes per slot: doc ids (both modes) + LSE + Delta (dKV), 1024-aligned
  static constexpr int kSlotExtra = MODE == kDKV ? 2048 : 1024;
  static constexpr int kSlotBytes = 2 * kTileBytes + kSlotExtra;
  static constexpr int kOffFix = 0;
  static constexpr int kOffSlots = 2 * kTileBytes;
  static constexpr int kOffBars = kOffSlots + kSlots * kSlotBytes;
  // fix_full, fix_empty, s_full, dp_full, p_full, ds_full, acc_done, acc_free, drain,
  // slot_full[kSlots], slot_empty[kSlots]
  static constexpr int kNumBars = 9 + 2 * kSlots;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr uint32_t kColAcc = 256;
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
};

// One unit of work and its iteration list.
struct BUnit {
  int b, h;      // dQ: query head; dKV: kv head
  int tile;      // dQ: query tile; dKV: key tile
  int n_full, n_part, group;  // per head of the group (dKV) or total (dQ)
  const int* lf;
  const int* lp;
  __device__ __forceinline__ int n() const { return (n_full + n_part) * group; }
  // iteration -> (head offset within group, streamed tile index, partial?)
  __device__ __forceinline__ void at(int it, int& hoff, int& t, bool& partial) const {
    const int m = n_full + n_part;
    hoff = it / m;
    const int j = it % m;
    partial = j >= n_full;
    t = j < n_full ? (lf ? lf[j] : j) : (lp ? lp[j - n_full] : j - n_full);
  }
};

template <int MODE>
__device__ __forceinline__ BUnit decode_bwd(const BwdArgs& a, int u) {
  const FwdProblem& p = a.f;
  const int nq = p.Sq / kTile, nkv = p.Skv / kTile;
  const int heads = MODE == kDQ ? p.Hq : p.Hkv;
  const int rank = u / heads, h = u % heads;
  const int n_outer = MODE == kDQ ? nq : nkv;
  const int n_inner = MODE == kDQ ? nkv : nq;
  const bool causal_bound = (p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX);
  int row;
  if (a.lists.full_cnt) row = a.lists.order[rank];
  else if (causal_bound)  // longest first: dQ large query tiles first, dKV small key tiles first
    row = MODE == kDQ ? (rank % p.B) * nq + (nq - 1 - rank / p.B) : (rank % p.B) * nkv + rank / p.B;
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
  return U;
}

template <int MODE>
__device__ __forceinline__ int dense_first(const BwdArgs& a, const BUnit& U) {
  const FwdProblem& p = a.f;
  const bool causal_bound = (p.variant & ATTN_MASK_CAUSAL) && !(p.variant & ATTN_MASK_PREFIX);
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

template <int D, int SCORE, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdArgs a) {
  using C = BwdCfg<D, MODE>;
  const FwdProblem& p = a.f;
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
  uint64_t* slot_full = bars + 9;
  uint64_t* slot_empty = bars + 9 + C::kSlots;
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
    mbar_init(p_full, 128);
    mbar_init(ds_full, 128);
    mbar_init(acc_done, 1);
    mbar_init(acc_free, 128);
    mbar_init(drain, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(slot_full + s, 1);
      mbar_init(slot_empty + s, 1);
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

  const int nq = p.Sq / kTile, nkv = p.Skv / kTile;
  const int num_units = MODE == kDQ ? p.B * nq * p.Hq : p.B * nkv * p.Hkv;
  const int group = p.Hq / p.Hkv;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------- producer
    {
      // With ATTN_FAULT_NO_LOADS nothing is issued and the consumers' waits run out.
      const bool leader = lane == 0 && !(p.fault_inject & ATTN_FAULT_NO_LOADS);
      uint32_t slot_it = 0, fix_it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const BUnit U = decode_bwd<MODE>(a, u);
        const int n = U.n();
        if (n == 0) continue;
        const int first = dense_first<MODE>(a, U);
        ok = __all_sync(0xffffffffu, wait_bounded(fix_empty, (fix_it & 1) ^ 1, wd));
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(fix_full, 2 * C::kTileBytes);
          // dQ: Q and dO rows of (b, h, tile); dKV: K and V rows of (b, hk, tile)
          const int row = MODE == kDQ ? (U.b * p.Hq + U.h) * p.Sq + U.tile * kTile
                                      : (U.b * p.Hkv + U.h) * p.Skv + U.tile * kTile;
          const CUtensorMap* m0 = MODE == kDQ ? &tm_q : &tm_k;
          const CUtensorMap* m1 = MODE == kDQ ? &tm_do : &tm_v;
          for (int bx = 0; bx < C::kBoxes; ++bx) {
            tma_load_2d(sFix + bx * C::kBoxBytes, m0, fix_full, bx * 64, row);
            tma_load_2d(sFix + C::kTileBytes + bx * C::kBoxBytes, m1, fix_full, bx * 64, row);
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
          ok = __all_sync(0xffffffffu,
                          wait_bounded(slot_empty + slot, ((slot_it / C::kSlots) & 1) ^ 1, wd));
          if (!ok) break;
          uint8_t* base = sSlots + slot * C::kSlotBytes;
          uint32_t bytes = 2 * C::kTileBytes;
          if (has_doc) bytes += 512;
          if (MODE == kDKV) bytes += 1024;
          if (leader) mbar_arrive_expect_tx(slot_full + slot, bytes);
          if (leader && MODE == kDQ) {
            const int row = (U.b * p.Hkv + U.h / group) * p.Skv + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx) {
              tma_load_2d(base + bx * C::kBoxBytes, &tm_k, slot_full + slot, bx * 64, row);
              tma_load_2d(base + C::kTileBytes + bx * C::kBoxBytes, &tm_v, slot_full + slot,
                          bx * 64, row);
            }
            if (has_doc)
              bulk_load(base + 2 * C::kTileBytes,
                        p.mask.doc_id + (size_t)U.b * p.mask.doc_len + t * kTile, 512,
                        slot_full + slot);
          } else if (leader) {
            const int h = U.h * group + hoff;
            const size_t qrow = (size_t)(U.b * p.Hq + h) * p.Sq + t * kTile;
            for (int bx = 0; bx < C::kBoxes; ++bx) {
              tma_load_2d(base + bx * C::kBoxBytes, &tm_q, slot_full + slot, bx * 64, (int)qrow);
              tma_load_2d(base + C::kTileBytes + bx * C::kBoxBytes, &tm_do, slot_full + slot,
                          bx * 64, (int)qrow);
            }
            if (has_doc)
              bulk_load(base + 2 * C::kTileBytes,
                        p.mask.doc_id + (size_t)U.b * p.mask.doc_len + t * kTile, 512,
                        slot_full + slot);
            bulk_load(base + 2 * C::kTileBytes + 512, p.lse + qrow, 512, slot_full + slot);
            bulk_load(base + 2 * C::kTileBytes + 1024, a.delta + qrow, 512, slot_full + slot);
          }
          __syncwarp();
          ++slot_it;
        }
      }
      if (!ok && !(p.fault_inject & ATTN_FAULT_NO_LOADS)) {  // let copies in flight land
        for (uint32_t k = 0; k < C::kSlots && k < slot_it; ++k) {
          const uint32_t it = slot_it - 1 - k;
          wait_drain(slot_full + it % C::kSlots, (it / C::kSlots) & 1);
        }
        if (fix_it > 0) wait_drain(fix_full, (fix_it - 1) & 1);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    {
      const bool leader = lane == 0;
      constexpr uint32_t kIdescSS = idesc_bf16(128, 128, false);
      constexpr uint32_t kIdescTS = idesc_bf16(128, D, true);
      const uint32_t fix_addr = smem_u32(sFix);
      const uint32_t slots_addr = smem_u32(sSlots);
      uint32_t slot_it = 0, fix_it = 0, p_it = 0, ds_it = 0, acc_it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const BUnit U = decode_bwd<MODE>(a, u);
        const int n = U.n();
        if (n == 0) continue;
        ok = __all_sync(0xffffffffu, wait_bounded(fix_full, fix_it & 1, wd));
        if (!ok) break;
        ++fix_it;
        tc_fence_after();
        for (int it = 0; it < n && ok; ++it) {
          const uint32_t seq = slot_it + it;
          const uint32_t slot = seq % C::kSlots;
          ok = __all_sync(0xffffffffu, wait_bounded(slot_full + slot, (seq / C::kSlots) & 1, wd));
          if (!ok) break;
          tc_fence_after();
          const uint32_t s0 = slots_addr + slot * C::kSlotBytes;  // K (dQ) or Q (dKV)
          const uint32_t s1 = s0 + C::kTileBytes;                 // V (dQ) or dO (dKV)
          // S = fix0 . slot0^T and dP = fix1 . slot1^T (K-major operands)
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * C::kBoxBytes + (kk % 4) * 32;
              mma_bf16_ss(tmem, sdesc_sw128(fix_addr + off, 16, 1024),
                          sdesc_sw128(s0 + off, 16, 1024), kIdescSS, kk > 0);
            }
            mma_commit(s_full);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk / 4) * C::kBoxBytes + (kk % 4) * 32;
              mma_bf16_ss(tmem + 128, sdesc_sw128(fix_addr + C::kTileBytes + off, 16, 1024),
                          sdesc_sw128(s1 + off, 16, 1024), kIdescSS, kk > 0);
            }
            mma_commit(dp_full);
          }
          __syncwarp();
          if (it == 0) {
            ok = __all_sync(0xffffffffu, wait_bounded(acc_free, (acc_it & 1) ^ 1, wd));
            if (!ok) break;
          }
          if (MODE == kDKV) {  // dV += P^T dO (B = dO tile, MN-major)
            ok = __all_sync(0xffffffffu, wait_bounded(p_full, p_it & 1, wd));
            if (!ok) break;
            ++p_it;
            tc_fence_after();
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_bf16_ts(tmem + C::kColAcc, tmem + kk * 8,
                            sdesc_sw128(s1 + kk * 16 * 128, C::kBoxBytes, 1024), kIdescTS,
                            (it > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
          ok = __all_sync(0xffffffffu, wait_bounded(ds_full, ds_it & 1, wd));
          if (!ok) break;
          ++ds_it;
          tc_fence_after();
          // dQ: A += (P g dP) K, B += (P g) K;   dKV: dK += dS^T Q   (B = slot0, MN-major)
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_bf16_ts(tmem + C::kColAcc + D, tmem + 128 + kk * 8,
                          sdesc_sw128(s0 + kk * 16 * 128, C::kBoxBytes, 1024), kIdescTS,
                          (it > 0 || kk > 0) ? 1u : 0u);
            if (MODE == kDQ) {
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)
                mma_bf16_ts(tmem + C::kColAcc, tmem + kk * 8,
                            sdesc_sw128(s0 + kk * 16 * 128, C::kBoxBytes, 1024), kIdescTS,
                            (it > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(slot_empty + slot);
          }
          __syncwarp();
        }
        if (!ok) break;
        ++acc_it;
        if (leader) {
          mma_commit(acc_done);
          mma_commit(fix_empty);
        }
        __syncwarp();
        slot_it += n;
      }
      if (leader) mma_commit(drain);
      __syncwarp();
      wait_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------- compute
    const int t = threadIdx.x;  // row of the fixed tile == TMEM lane
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t colS = tmem + lane_base;
    const uint32_t colP = tmem + lane_base + 128;
    const uint32_t colAcc = tmem + lane_base + C::kColAcc;
    const float scale = p.score.scale;
    uint32_t slot_it = 0, s_it = 0, acc_it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const BUnit U = decode_bwd<MODE>(a, u);
      const int n = U.n();
      const int first = dense_first<MODE>(a, U);
      // the thread's own row: a query row (dQ) or a key row (dKV)
      const int r = U.tile * kTile + t;
      if (n == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (MODE == kDQ) {
          const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + qrow * D);
          for (int c = 0; c < D / 8; ++c) dst[c] = z;
          a.delta_out[qrow] = 0.0f;
        } else {
          const size_t off = ((size_t)(U.b * p.Hkv + U.h) * p.Skv + r) * D;
          uint4* dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk) + off);
          uint4* dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv) + off);
          for (int c = 0; c < D / 8; ++c) dk[c] = z, dv[c] = z;
        }
        continue;
      }
      const int* docb = has_doc ? p.mask.doc_id + (size_t)U.b * p.mask.doc_len : nullptr;
      const int my_doc = docb ? docb[r] : 0;
      const int P = (p.variant & ATTN_MASK_PREFIX) ? p.mask.prefix_len[U.b] : INT_MIN;
      float row_lse2 = 0.0f, row_delta = 0.0f, row_dhat = 0.0f;
      if (MODE == kDQ) {
        const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
        const float l = p.lse[qrow];
        row_lse2 = l == -INFINITY ? INFINITY : l * kLog2e;  // empty row: every p is 0
        row_dhat = a.delta[qrow];  // estimate from the bf16 O (delta_kernel)
        row_delta = 0.0f;          // exact: sum_j P dP, accumulated below
      }
      for (int it = 0; it < n; ++it) {
        int hoff, tt;
        bool partial;
        U.at(it, hoff, tt, partial);
        tt += first;
        const int h = MODE == kDQ ? U.h : U.h * group + hoff;
        const uint32_t seq = slot_it + it;
        const uint32_t slot = seq % C::kSlots;
        const uint8_t* base = sSlots + slot * C::kSlotBytes;
        const int* sdoc = reinterpret_cast<const int*>(base + 2 * C::kTileBytes);
        const float* slse = reinterpret_cast<const float*>(base + 2 * C::kTileBytes + 512);
        const float* sdelta = reinterpret_cast<const float*>(base + 2 * C::kTileBytes + 1024);
        // the slot's shared-memory extras (doc ids, LSE, Delta) are read directly
        ok = __all_sync(0xffffffffu, wait_bounded(slot_full + slot, (seq / C::kSlots) & 1, wd));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_bounded(s_full, s_it & 1, wd));
        if (!ok) break;
        const int c0 = tt * kTile;  // first column position (key for dQ, query for dKV)
        if constexpr (MODE == kDQ) {
          // Wait for S and dP; 32 columns at a time: P g -> S columns, P g dP -> dP
          // columns (bf16, packed below the columns still to be read), Delta += P dP.
          ok = __all_sync(0xffffffffu, wait_bounded(dp_full, s_it & 1, wd));
          if (!ok) break;
          ++s_it;
          tc_fence_after();
          const float slope = (SCORE & 1) ? alibi_slope(p.score, h) : 0.0f;
          int lo = INT_MIN, hi = INT_MAX, pre = INT_MIN;  // row i = r, column j = c0 + c
          if (partial) {
            if (p.variant & ATTN_MASK_CAUSAL) hi = r - c0 + 1;
            if (p.variant & ATTN_MASK_WINDOW) lo = r - c0 - p.mask.window + 1;
            if (P != INT_MIN) pre = P - c0;
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            uint32_t rs[32], rp[32];
            tmem_ld32(colS + 32 * qq, rs);
            tmem_ld32(colP + 32 * qq, rp);
            tmem_ld_wait_regs(rs);
            tmem_ld_wait_regs(rp);
            uint32_t pg_pk[16], pd_pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float pg2[2], pd2[2];
#pragma unroll
              for (int z = 0; z < 2; ++z) {
                const int c = 32 * qq + e + z;
                float x = __uint_as_float(rs[e + z]) * scale, g = 1.0f;
                if constexpr ((SCORE & 1) != 0) x = fmaf(slope, float(c0 - r + c), x);
                if constexpr ((SCORE & 2) != 0) {
                  const float th = tanh_approx(x * (1.0f / p.score.softcap));
                  x = p.score.softcap * th;
                  g = 1.0f - th * th;
                }
                float pr = ex2_approx(fmaf(x, kLog2e, -row_lse2));
                if (partial) {
                  // bitwise terms, document id read on a warp-uniform condition:
                  // no divergent branch per element
                  const bool same = docb ? (sdoc[c] == my_doc) : true;
                  const bool keep = ((c >= lo) & (c < hi) & same) | (c < pre);
                  pr = keep ? pr : 0.0f;
                }
                const float dp = __uint_as_float(rp[e + z]);
                row_delta = fmaf(pr, dp, row_delta);
                pg2[z] = pr * g;
                pd2[z] = pg2[z] * (dp - row_dhat);
              }
              pg_pk[e >> 1] = pack_bf16x2(pg2[0], pg2[1]);
              pd_pk[e >> 1] = pack_bf16x2(pd2[0], pd2[1]);
            }
            tmem_st16(colS + 16 * qq, pg_pk);
            tmem_st16(colP + 16 * qq, pd_pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(ds_full);
          continue;
        }
        tc_fence_after();
        float v[kTile];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(colS + 32 * c, rr);
          tmem_ld_wait_regs(rr);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[32 * c + e] = __uint_as_float(rr[e]);
        }
        const float slope = (SCORE & 1) ? alibi_slope(p.score, h) : 0.0f;
        // (j - i) = base_ji + sgn * c
        const int base_ji = MODE == kDQ ? c0 - r : r - c0;
        const float sgn = MODE == kDQ ? 1.0f : -1.0f;
        int lo = INT_MIN, hi = INT_MAX, pre = INT_MIN;
        if (partial) {
          if (MODE == kDQ) {  // row i = r, column j = c0 + c
            if (p.variant & ATTN_MASK_CAUSAL) hi = r - c0 + 1;
            if (p.variant & ATTN_MASK_WINDOW) lo = r - c0 - p.mask.window + 1;
            if (P != INT_MIN) pre = P - c0;
          } else {            // row j = r, column i = c0 + c
            if (p.variant & ATTN_MASK_CAUSAL) lo = r - c0;
            if (p.variant & ATTN_MASK_WINDOW) hi = r - c0 + p.mask.window;
            if (P != INT_MIN && r < P) pre = INT_MAX;
          }
        }
        // v <- P * score_mod'(s), the factor dS needs; for dKV, P itself (bf16)
        // goes to TMEM as the A operand of dV += P^T dO, 64 columns at a time.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
          float prev = 0.0f;
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int c = 64 * half + e;
            float x = v[c] * scale, g = 1.0f;
            if constexpr ((SCORE & 1) != 0) x = fmaf(slope, float(base_ji) + sgn * float(c), x);
            if constexpr ((SCORE & 2) != 0) {
              const float th = tanh_approx(x * (1.0f / p.score.softcap));
              x = p.score.softcap * th;
              g = 1.0f - th * th;
            }
            float lse2 = row_lse2;
            if constexpr (MODE == kDKV) lse2 = slse[c] == -INFINITY ? INFINITY : slse[c] * kLog2e;
            float pr = ex2_approx(fmaf(x, kLog2e, -lse2));
            if (partial) {
              // bitwise terms, document id read on a warp-uniform condition:
              // no divergent branch per element
              const bool same = docb ? (sdoc[c] == my_doc) : true;
              const bool keep = ((c >= lo) & (c < hi) & same) | (c < pre);
              pr = keep ? pr : 0.0f;
            }
            if constexpr (MODE == kDKV) {
              if (e & 1) pk[e >> 1] = pack_bf16x2(prev, pr);
              else prev = pr;
            }
            v[c] = pr * g;
          }
          if constexpr (MODE == kDKV) tmem_st32(colS + 32 * half, pk);
        }
        if constexpr (MODE == kDKV) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(p_full);
        }
        ok = __all_sync(0xffffffffu, wait_bounded(dp_full, s_it & 1, wd));
        if (!ok) break;
        ++s_it;
        tc_fence_after();
        // dS = p g (dP - Delta) -> bf16 into the first 64 columns of dP
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(colP + 32 * c, rr);
          tmem_ld_wait_regs(rr);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int cc = 32 * c + e;
            const float dl = MODE == kDQ ? row_delta : sdelta[cc];
            v[cc] = v[cc] * (__uint_as_float(rr[e]) - dl);
          }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t rr[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = pack_bf16x2(v[64 * c + 2 * e], v[64 * c + 2 * e + 1]);
          tmem_st32(colP + 32 * c, rr);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_full);
      }
      if (!ok) break;
      slot_it += n;
      // epilogue
      ok = __all_sync(0xffffffffu, wait_bounded(acc_done, acc_it & 1, wd));
      if (!ok) break;
      ++acc_it;
      tc_fence_after();
      auto store_row = [&](uint32_t col, __nv_bfloat16* dst, float mul) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(col + 32 * c, rr);
          tmem_ld_wait_regs(rr);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * mul, __uint_as_float(rr[2 * e + 1]) * mul);
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      };
      if (MODE == kDQ) {  // dQ = scale (A - (Delta - Dhat) B); Delta to the workspace
        const size_t qrow = (size_t)(U.b * p.Hq + U.h) * p.Sq + r;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + qrow * D;
        const float corr = row_delta - row_dhat;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ra[32], rb[32];
          tmem_ld32(colAcc + D + 32 * c, ra);
          tmem_ld32(colAcc + 32 * c, rb);
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
          for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
        a.delta_out[qrow] = row_delta;
      } else {
        const size_t off = ((size_t)(U.b * p.Hkv + U.h) * p.Skv + r) * D;
        store_row(colAcc, static_cast<__nv_bfloat16*>(a.dv) + off, 1.0f);
        store_row(colAcc + D, static_cast<__nv_bfloat16*>(a.dk) + off, scale);
      }
      tc_fence_before();
      mbar_arrive(acc_free);
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

template <int D, int SCORE, int MODE>
cudaError_t launch_one(const BwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, int units,
                       cudaStream_t stream) {
  using C = BwdCfg<D, MODE>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(bwd_kernel<D, SCORE, MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int grid = units < sm_count() ? units : sm_count();
  if (grid == 0) return cudaSuccess;
  bwd_kernel<D, SCORE, MODE><<<grid, kThreads, C::kSmemAlloc, stream>>>(mq, mk, mv, mdo, a);
  return cudaGetLastError();
}

template <int D, int SCORE>
cudaError_t launch_typed(const BwdProblem& bp, cudaStream_t stream) {
  const FwdProblem& f = bp.f;
  const size_t rows = (size_t)f.B * f.Hq * f.Sq;
  delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(f.o), static_cast<const __nv_bfloat16*>(bp.dO),
      bp.delta, rows, D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_bf16(&mq, f.q, (long long)f.B * f.Hq * f.Sq, D) ||
      !make_map_bf16(&mk, f.k, (long long)f.B * f.Hkv * f.Skv, D) ||
      !make_map_bf16(&mv, f.v, (long long)f.B * f.Hkv * f.Skv, D) ||
      !make_map_bf16(&mdo, bp.dO, (long long)f.B * f.Hq * f.Sq, D))
    return cudaErrorInvalidValue;
  BwdArgs a{f, bp.dO, bp.dq, bp.dk, bp.dv, bp.delta, bp.delta, f.lists};
  e = launch_one<D, SCORE, kDQ>(a, mq, mk, mv, mdo, f.B * (f.Sq / kTile) * f.Hq, stream);
  if (e != cudaSuccess) return e;
  a.lists = bp.t_lists;
  return launch_one<D, SCORE, kDKV>(a, mq, mk, mv, mdo, f.B * (f.Skv / kTile) * f.Hkv, stream);
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdProblem& bp, cudaStream_t stream) {
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (bp.f.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0>(bp, stream);
      case 1: return launch_typed<64, 1>(bp, stream);
      case 2: return launch_typed<64, 2>(bp, stream);
      default: return launch_typed<64, 3>(bp, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0>(bp, stream);
    case 1: return launch_typed<128, 1>(bp, stream);
    case 2: return launch_typed<128, 2>(bp, stream);
    default: return launch_typed<128, 3>(bp, stream);
  }
}

}  // namespace mattn
