// Device-side building blocks shared by the attention kernels: the mask and
// score modifications (FlexAttention page: score_mod applied element-wise
// before the softmax, and the mask variants it lists), bounded waits, and thin
// inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda.h>

#include "debug.cuh"
#include "mattn.h"  // include/ is on the include path

namespace mattn {

constexpr int kTile = ATTN_TILE;  // 128 query rows x 128 key columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Arguments common to the kernels (plain data, passed by value).
// ---------------------------------------------------------------------------
struct MaskArgs {
  unsigned variant;       // mask bits (ATTN_MASK_*)
  int window;
  const int* doc_id;      // [B][doc_len], indexed by absolute position
  int doc_len;            // max(q_off + Sq, kv_off + Skv)
  const int* prefix_len;  // [B]
  int q_off, kv_off;      // absolute position of query row 0 / key 0
};

struct ScoreArgs {
  float scale;
  float softcap;
  const float* slopes;    // [Hq] or nullptr -> 2^(-8(h+1)/Hq)
  int Hq;
  const float* rel_bias;  // [Hq][rb_len] distance-indexed bias, or nullptr
  int rb_len;             // Sq + Skv - 1
  int rb_zero;            // index of distance 0: Skv - 1
};

struct BlockLists {       // device view of attn_block_mask (nullptr full_cnt = none)
  const int* full_cnt;
  const int* part_cnt;
  const int* full_idx;
  const int* part_idx;
  const int* order;
  int nq, nkv;
};

__device__ __forceinline__ float alibi_slope(const ScoreArgs& s, int h) {
  return s.slopes ? s.slopes[h] : exp2f(-8.0f * float(h + 1) / float(s.Hq));
}

// Number of leading key tiles the causal term allows for query rows up to
// `last_row` (rows and key columns of the call; absolute positions add the
// offsets): tiles past the one holding absolute key position q_off+last_row.
__device__ __forceinline__ int causal_tiles(const MaskArgs& m, int last_row, int nkv) {
  const int jmax = last_row + m.q_off - m.kv_off;  // last key column with j <= i
  return jmax < 0 ? 0 : min(nkv, jmax / kTile + 1);
}

// keep(b, i, j) exactly as the mask bits define it, for query row i and key
// column j of the call (their absolute positions add the offsets). Used by
// the fp32 kernel.
__device__ __forceinline__ bool mask_keep(const MaskArgs& m, int b, int i, int j) {
  i += m.q_off;
  j += m.kv_off;
  bool keep = true;
  if (m.variant & ATTN_MASK_CAUSAL) keep = keep && (j <= i);
  if (m.variant & ATTN_MASK_WINDOW) keep = keep && (i - j < m.window);
  if (m.variant & ATTN_MASK_DOCUMENT) {
    const int* d = m.doc_id + (size_t)b * m.doc_len;
    const bool in = MATTN_IN_BOUNDS(kSiteF32, i, m.doc_len) && MATTN_IN_BOUNDS(kSiteF32, j, m.doc_len);
    keep = keep && in && (d[i] == d[j]);
  }
  if (m.variant & ATTN_MASK_PREFIX) keep = keep || (j < m.prefix_len[b]);
  return keep;
}

// ---------------------------------------------------------------------------
// Status word and bounded waits.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Per-CTA watchdog: every wait gives up after `timeout_ns`, raises the CTA's
// abort flag (so the other roles stop waiting too) and records
// ATTN_ERR_TIMEOUT in the status word. Returns false when the wait failed.
struct Watchdog {
  volatile int* abort_flag;  // shared memory
  int* status;               // global memory
  uint64_t timeout_ns;
};

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` nanoseconds pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const Watchdog& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  const uint32_t hint = w.timeout_ns < 1000000ull ? (uint32_t)w.timeout_ns : 1000000u;
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (*w.abort_flag) return false;
    if (global_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1;
      report_status(w.status, ATTN_ERR_TIMEOUT);
      return false;
    }
  }
}

// Wait used on the abort path to let work in flight finish: ignores the abort
// flag and gives up after 200 ms.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 200000000ull) return;
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) and fences.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tile load: x = column, y = row within one (b, h) slice, z = slice. Rows
// past the slice's end (y beyond S) are filled with zeros.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 4-byte asynchronous copy global -> shared (cp.async), its group commit and
// the wait for all groups but the newest `n` (n = 0 or 1).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads/stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA and commit wrappers carry no "memory" clobber: they touch no memory
// the compiler manages, and asm volatile keeps them in order with the mbarrier
// waits (which do clobber memory) around them.
// D(tmem) (+)= A(smem) * B(smem)^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D(tmem) (+)= A(tmem) * B(smem), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Products issued by a whole, converged warp: lane 0 issues all K-steps of
// one product in a single block, the other lanes skip them by predicate.
// On this GPU the tensor pipe then accepts M128 N128 K16 products at its
// full rate (64 cycles each); issued one at a time from a divergent single
// thread, each product costs about 3.5 times that. `first` is the enable
// input of the first K-step (0: overwrite D); the others accumulate.
template <int K>
__device__ __forceinline__ void mma_ss_warp(uint32_t d, const uint64_t (&a)[K],
                                            const uint64_t (&b)[K], uint32_t idesc,
                                            uint32_t first) {
  static_assert(K == 4 || K == 8, "4 or 8 K-steps");
  if constexpr (K == 8) {
    asm volatile(
      "{\n\t.reg .pred pl, pa, pt;\n\t.reg .b32 ln;\n\t"
      "mov.u32 ln, %laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      "setp.ne.b32 pa, %2, 0;\n\t"
      "setp.eq.b32 pt, 0, 0;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, pa;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %11, %12, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %13, %14, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %15, %16, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %17, %18, %1, pt;\n\t"
      "}" ::"r"(d), "r"(idesc), "r"(first), "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]), "l"(a[4]), "l"(b[4]), "l"(a[5]), "l"(b[5]), "l"(a[6]), "l"(b[6]), "l"(a[7]), "l"(b[7]));
  } else {
    asm volatile(
      "{\n\t.reg .pred pl, pa, pt;\n\t.reg .b32 ln;\n\t"
      "mov.u32 ln, %laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      "setp.ne.b32 pa, %2, 0;\n\t"
      "setp.eq.b32 pt, 0, 0;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %4, %1, pa;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %1, pt;\n\t"
      "}" ::"r"(d), "r"(idesc), "r"(first), "l"(a[0]), "l"(b[0]), "l"(a[1]), "l"(b[1]), "l"(a[2]), "l"(b[2]), "l"(a[3]), "l"(b[3]));
  }
}

// The same with A read from tensor memory (a[k]: TMEM address of K-step k).
template <int K>
__device__ __forceinline__ void mma_ts_warp(uint32_t d, const uint32_t (&a)[K],
                                            const uint64_t (&b)[K], uint32_t idesc,
                                            uint32_t first) {
  static_assert(K == 8, "8 K-steps");
  asm volatile(
      "{\n\t.reg .pred pl, pa, pt;\n\t.reg .b32 ln;\n\t"
      "mov.u32 ln, %laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      "setp.ne.b32 pa, %2, 0;\n\t"
      "setp.eq.b32 pt, 0, 0;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %4, %1, pa;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%11], %12, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%13], %14, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%15], %16, %1, pt;\n\t"
      "@pl tcgen05.mma.cta_group::1.kind::f16 [%0], [%17], %18, %1, pt;\n\t"
      "}" ::"r"(d), "r"(idesc), "r"(first), "r"(a[0]), "l"(b[0]), "r"(a[1]), "l"(b[1]), "r"(a[2]), "l"(b[2]), "r"(a[3]), "l"(b[3]), "r"(a[4]), "l"(b[4]), "r"(a[5]), "l"(b[5]), "r"(a[6]), "l"(b[6]), "r"(a[7]), "l"(b[7]));
}

// tcgen05.commit from a converged warp (issued by lane 0, the lane that
// issued the products it tracks).
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred pl;\n\t.reg .b32 ln;\n\t"
      "mov.u32 ln, %laneid;\n\t"
      "setp.eq.u32 pl, ln, 0;\n\t"
      "@pl tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar)));
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar)));
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N tile.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format
// (1 = bf16), 15 A major (0 = K), 16 B major (1 = MN), [17,23) N >> 3,
// [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 form), 128-byte swizzle.
// [0,14) start >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
// offset >> 4, [46,48) = 1, [61,64) layout (2 = 128B swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// tcgen05.wait::ld that also names the 32 registers a prior tcgen05.ld fills,
// so the compiler cannot move their uses above the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
        "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
        "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
        "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
        "+r"(r[31])
      :
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Hardware approximations (MUFU): 2^x and tanh(x).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100 family): two lanes of fp32 arithmetic per instruction.
union F2 {
  float2 f;
  unsigned long long u;
};

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  F2 x, y, z, d;
  x.f = a;
  y.f = b;
  z.f = c;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.u) : "l"(x.u), "l"(y.u), "l"(z.u));
  return d.f;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  F2 x, y, d;
  x.f = a;
  y.f = b;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(x.u), "l"(y.u));
  return d.f;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  F2 x, y, d;
  x.f = a;
  y.f = b;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(x.u), "l"(y.u));
  return d.f;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of n (a multiple of 16) values with 8 independent chains.
template <int N>
__device__ __forceinline__ float row_max(const float* v) {
  float m[8];
#pragma unroll
  for (int a = 0; a < 8; ++a) m[a] = fmaxf(v[a], v[a + 8]);
#pragma unroll
  for (int c = 16; c < N; c += 16) {
#pragma unroll
    for (int a = 0; a < 8; ++a) m[a] = fmax3(m[a], v[c + a], v[c + 8 + a]);
  }
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace mattn
