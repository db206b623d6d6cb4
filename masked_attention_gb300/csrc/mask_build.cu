// Block-mask builder (FlexAttention page, item on exploiting the sparsity of
// the attention mask): for every (query tile, key tile) pair decide whether all,
// some or none of its pairs are kept, then write ascending lists of the full
// and partial tiles, plus a longest-first order of the list rows.
//
// Classification is exact. Interval bounds decide most tiles without looking
// at single pairs (causal, window and prefix terms from the tile corners, the
// document term from the min/max document id of each range); a tile whose
// bounds decide nothing is classified by evaluating the mask on its pairs.
#include "launch.h"

namespace mattn {
namespace {

constexpr int kEmpty = 0, kPartial = 1, kFull = 2;

struct Range {
  int lo, hi;  // inclusive
};

// lim: entries of doc from position 0 on (the debug build checks against it).
__device__ __forceinline__ void warp_doc_minmax(const int* doc, Range r, int lim, int& mn,
                                                int& mx) {
  const int lane = threadIdx.x & 31;
  mn = INT_MAX;
  mx = INT_MIN;
  for (int p = r.lo + lane; p <= r.hi; p += 32) {
    const int d = MATTN_IN_BOUNDS(kSiteMaskBuild, p, lim) ? doc[p] : 0;
    mn = min(mn, d);
    mx = max(mx, d);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
}

// Sound tri-state per term: 2 = every pair kept, 0 = no pair kept, 1 = unknown.
__device__ __forceinline__ int bounds_state(const MaskArgs& m, int b, Range ri, Range rj,
                                            int qmin, int qmax, int kmin, int kmax) {
  bool and_all = true, and_none = false;
  if (m.variant & ATTN_MASK_CAUSAL) {  // j <= i
    and_all = and_all && (rj.hi <= ri.lo);
    and_none = and_none || (rj.lo > ri.hi);
  }
  if (m.variant & ATTN_MASK_WINDOW) {  // i - j < W
    and_all = and_all && (ri.hi - rj.lo < m.window);
    and_none = and_none || (ri.lo - rj.hi >= m.window);
  }
  if (m.variant & ATTN_MASK_DOCUMENT) {  // doc[i] == doc[j]
    and_all = and_all && (qmin == qmax && kmin == kmax && qmin == kmin);
    and_none = and_none || (qmax < kmin || kmax < qmin);
  }
  if (m.variant & ATTN_MASK_PREFIX) {  // OR j < P
    const int P = m.prefix_len[b];
    if (rj.hi < P) return kFull;
    const bool pre_none = rj.lo >= P;
    if (and_none && pre_none) return kEmpty;
    if (and_all) return kFull;
    return kPartial + 8;  // undecided
  }
  if (and_none) return kEmpty;
  if (and_all) return kFull;
  return kPartial + 8;  // undecided
}

constexpr int kClassifyThreads = 512;  // 16 warps, one key tile per warp at a time

__global__ void __launch_bounds__(kClassifyThreads) classify_kernel(MaskArgs m, int Sq, int Skv,
                                                       int transposed, int* cnt_full,
                                                       int* cnt_part, int* idx_full,
                                                       int* idx_part) {
  extern __shared__ signed char sstate[];
  const int b = blockIdx.y;
  const int outer = blockIdx.x;
  const int nq = (Sq + kTile - 1) / kTile;
  const int nkv = (Skv + kTile - 1) / kTile;
  const int n_outer = transposed ? nkv : nq;
  const int n_inner = transposed ? nq : nkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Tile ranges are in the call's rows and columns; the mask terms and the
  // document ids use absolute positions (row + q_off, column + kv_off).
  const int* doc = (m.variant & ATTN_MASK_DOCUMENT) ? m.doc_id + (size_t)b * m.doc_len : nullptr;
  const int* docq = doc ? doc + m.q_off : nullptr;   // by query row
  const int* dock = doc ? doc + m.kv_off : nullptr;  // by key column
  const int limq = m.doc_len - m.q_off, limk = m.doc_len - m.kv_off;
  (void)limq;
  (void)limk;

  const int outer_len = transposed ? Skv : Sq;
  const Range ro{outer * kTile, min((outer + 1) * kTile, outer_len) - 1};
  int omin = 0, omax = 0;
  if (doc) warp_doc_minmax(transposed ? dock : docq, ro, transposed ? limk : limq, omin, omax);  // every warp computes it

  for (int inner = warp; inner < n_inner; inner += kClassifyThreads / 32) {
    const int inner_len = transposed ? Sq : Skv;
    const Range rn{inner * kTile, min((inner + 1) * kTile, inner_len) - 1};
    const Range ri = transposed ? rn : ro;
    const Range rj = transposed ? ro : rn;
    const Range ria{ri.lo + m.q_off, ri.hi + m.q_off};    // absolute
    const Range rja{rj.lo + m.kv_off, rj.hi + m.kv_off};
    // The document term can only remove pairs: a tile the other terms already
    // leave empty is empty, and its document ids need not be read.
    MaskArgs m_nodoc = m;
    m_nodoc.variant &= ~ATTN_MASK_DOCUMENT;
    int st = bounds_state(m_nodoc, b, ria, rja, 0, 0, 0, 0);
    bool doc_uniform = true;  // one document id over the tile's rows and columns
    if (st != kEmpty && doc) {
      int nmin = 0, nmax = 0;
      warp_doc_minmax(transposed ? docq : dock, rn, transposed ? limq : limk, nmin, nmax);
      const int qmin = transposed ? nmin : omin, qmax = transposed ? nmax : omax;
      const int kmin = transposed ? omin : nmin, kmax = transposed ? omax : nmax;
      doc_uniform = qmin == qmax && kmin == kmax && qmin == kmin;
      st = bounds_state(m, b, ria, rja, qmin, qmax, kmin, kmax);
    }
    if (st >= 8) {  // undecided: look at the pairs
      // Lane l owns columns l, l+32, l+64, l+96 of the tile; their document
      // ids stay in registers and each row reads its own id once. The terms
      // are combined bitwise, so no lane branches around a load.
      const int ncols = rj.hi - rj.lo + 1;
      int dj[4];
      bool valid[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = lane + 32 * k;
        valid[k] = c < ncols;
        dj[k] = (doc && valid[k] && MATTN_IN_BOUNDS(kSiteMaskBuild, rj.lo + c, limk))
                    ? dock[rj.lo + c]
                    : 0;
      }
      // The rows' document ids too: lane l holds rows l, l+32, l+64, l+96 and
      // each row's id is shuffled out, so the row loop never waits on memory.
      int qd[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = ri.lo + lane + 32 * k;
        qd[k] = (doc && i <= ri.hi && MATTN_IN_BOUNDS(kSiteMaskBuild, i, limq)) ? docq[i] : 0;
      }
      const bool causal = m.variant & ATTN_MASK_CAUSAL, window = m.variant & ATTN_MASK_WINDOW;
      const int P = (m.variant & ATTN_MASK_PREFIX) ? m.prefix_len[b] : INT_MIN;
      // Where the causal and window terms keep every pair and the prefix none,
      // a tile whose rows and columns do not all share one document certainly
      // drops a pair: only a kept pair has to be found, and the scan stops at
      // the first one instead of looking for a dropped row far down the tile.
      const bool range_all =
          (!causal || rja.hi <= ria.lo) && (!window || ria.hi - rja.lo < m.window);
      const bool prefix_none = rja.lo >= P;
      bool any_keep = false, any_drop = range_all && prefix_none && !doc_uniform;
      for (int i = ri.lo; i <= ri.hi; ++i) {
        const int r = i - ri.lo, k = r >> 5;
        const int mine = k == 0 ? qd[0] : k == 1 ? qd[1] : k == 2 ? qd[2] : qd[3];
        const int di = __shfl_sync(0xffffffffu, mine, r & 31);
        const int ia = i + m.q_off;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = rja.lo + lane + 32 * k;
          const bool keep =
              ((!causal | (j <= ia)) & (!window | (ia - j < m.window)) & (dj[k] == di)) | (j < P);
          any_keep |= valid[k] & keep;
          any_drop |= valid[k] & !keep;
        }
        if (__any_sync(0xffffffffu, any_keep) && __any_sync(0xffffffffu, any_drop)) break;
      }
      const bool wk = __any_sync(0xffffffffu, any_keep);
      const bool wd = __any_sync(0xffffffffu, any_drop);
      st = wk ? (wd ? kPartial : kFull) : kEmpty;
    }
    if (lane == 0) sstate[inner] = static_cast<signed char>(st);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const size_t row = (size_t)b * n_outer + outer;
    int nf = 0, np = 0;
    for (int inner = 0; inner < n_inner; ++inner) {
      const int st = sstate[inner];
      if (st == kFull) idx_full[row * n_inner + nf++] = inner;
      else if (st == kPartial) idx_part[row * n_inner + np++] = inner;
    }
    cnt_full[row] = nf;
    cnt_part[row] = np;
  }
}

// Longest-first order of the B * n_outer list rows, by the number of visited
// tiles (full + partial), descending, ties by row index. Each thread ranks its
// rows against all others (costs staged in shared memory); large inputs that
// do not fit fall back to one thread's counting sort over global memory.
// by_batch (the transposed lists, which only the dK/dV kernel reads): batch
// element by batch element, longest first within each, so the kernel streams
// one batch element's queries and dO at a time and they stay in the L2.
constexpr int kOrderSmemRows = 12288;

__global__ void order_kernel(const int* cnt_full, const int* cnt_part, int n_rows, int n_outer,
                             int n_inner, int by_batch, int* order) {
  extern __shared__ int cost[];
  // rows ranked among themselves: all rows, or those of one batch element
  const int group = by_batch ? n_outer : n_rows;
  if (n_rows <= kOrderSmemRows) {
    for (int r = threadIdx.x; r < n_rows; r += blockDim.x) cost[r] = cnt_full[r] + cnt_part[r];
    __syncthreads();
    for (int r = threadIdx.x; r < n_rows; r += blockDim.x) {
      const int c = cost[r];
      const int first = (r / group) * group;
      int rank = first;
      for (int k = first; k < first + group; ++k) {
        const int ck = cost[k];
        rank += (ck > c) || (ck == c && k < r);
      }
      if (MATTN_IN_BOUNDS(kSiteMaskBuild, rank, n_rows)) order[rank] = r;
    }
    return;
  }
  if (threadIdx.x != 0) return;
  int* hist = cost;  // n_inner + 2 buckets
  for (int first = 0; first < n_rows; first += group) {
    for (int c = 0; c < n_inner + 2; ++c) hist[c] = 0;
    for (int r = first; r < first + group; ++r) {
      const int c = cnt_full[r] + cnt_part[r];
      if (MATTN_IN_BOUNDS(kSiteMaskBuild, c, n_inner + 1)) ++hist[c];
    }
    int pos = first;
    for (int c = n_inner; c >= 0; --c) {
      const int n = hist[c];
      hist[c] = pos;
      pos += n;
    }
    for (int r = first; r < first + group; ++r) {
      const int c = cnt_full[r] + cnt_part[r];
      if (!MATTN_IN_BOUNDS(kSiteMaskBuild, c, n_inner + 1)) continue;
      const int at = hist[c]++;
      if (MATTN_IN_BOUNDS(kSiteMaskBuild, at, n_rows)) order[at] = r;
    }
  }
}

}  // namespace

cudaError_t launch_block_mask(const MaskArgs& m, int B, int Sq, int Skv, int transposed,
                              int* cnt_full, int* cnt_part, int* idx_full, int* idx_part,
                              int* order, cudaStream_t stream) {
  const int nq = (Sq + kTile - 1) / kTile;
  const int nkv = (Skv + kTile - 1) / kTile;
  const int n_outer = transposed ? nkv : nq;
  const int n_inner = transposed ? nq : nkv;
  dim3 grid(n_outer, B);
  classify_kernel<<<grid, kClassifyThreads, n_inner, stream>>>(m, Sq, Skv, transposed, cnt_full, cnt_part,
                                                  idx_full, idx_part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n_rows = B * n_outer;
  const size_t smem = sizeof(int) * (size_t)(n_rows <= kOrderSmemRows ? n_rows : n_inner + 2);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  order_kernel<<<1, 1024, smem, stream>>>(cnt_full, cnt_part, n_rows, n_outer, n_inner,
                                          transposed, order);
  return cudaGetLastError();
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(mask_build)
}  // namespace mattn
