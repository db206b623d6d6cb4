// The exported C ABI (include/mattn.h): argument checks, block-mask buffer
// layout, and dispatch to the kernels. Every check returns before anything
// is launched; nothing here allocates device memory.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "host_util.h"
#include "launch.h"

#define MATTN_API extern "C" __attribute__((visibility("default")))

namespace mattn {

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

attn_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  t_last_cuda_error = e;
  return ATTN_ERR_CUDA;
}

namespace {

__device__ int g_status;  // status word used when the caller passes none

int* default_status() {
  // one address per device (a module variable has a separate copy per device)
  static int* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cuda_status(cudaGetDevice(&dev)) != ATTN_OK || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cuda_status(cudaGetSymbolAddress(&p, g_status)) != ATTN_OK) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

__global__ void fill_empty_rows(void* o, float* lse, size_t rows, int D, int elem_bytes) {
  const size_t n = rows * (size_t)D;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    if (elem_bytes == 4) static_cast<float*>(o)[e] = 0.0f;
    else static_cast<uint16_t*>(o)[e] = 0;
    if (e % D == 0) lse[e / D] = -INFINITY;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr unsigned kKnownBits = ATTN_MASK_BITS | ATTN_SCORE_BITS;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct MaskLayout {
  size_t full_cnt, part_cnt, full_idx, part_idx, order;
  size_t t_full_cnt, t_part_cnt, t_full_idx, t_part_idx, t_order;
  size_t total;
};

MaskLayout mask_layout(int B, int Sq, int Skv, int transposed) {
  const size_t nq = (size_t)(Sq + kTile - 1) / kTile, nkv = (size_t)(Skv + kTile - 1) / kTile;
  const size_t I = sizeof(int);
  MaskLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.full_cnt = take(I * B * nq);
  L.part_cnt = take(I * B * nq);
  L.full_idx = take(I * B * nq * nkv);
  L.part_idx = take(I * B * nq * nkv);
  L.order = take(I * B * nq);
  if (transposed) {
    L.t_full_cnt = take(I * B * nkv);
    L.t_part_cnt = take(I * B * nkv);
    L.t_full_idx = take(I * B * nkv * nq);
    L.t_part_idx = take(I * B * nkv * nq);
    L.t_order = take(I * B * nkv);
  }
  L.total = off;
  return L;
}

attn_status check_mask_params(unsigned variant, const attn_params* p, int B, int Sq, int Skv) {
  if (variant & ~kKnownBits) return ATTN_ERR_INVALID_ARG;
  if ((variant & ATTN_MASK_WINDOW) && p->window < 1) return ATTN_ERR_INVALID_ARG;
  if ((variant & ATTN_MASK_DOCUMENT) && !p->doc_id) return ATTN_ERR_INVALID_ARG;
  if ((variant & ATTN_MASK_PREFIX) && !p->prefix_len) return ATTN_ERR_INVALID_ARG;
  if ((variant & ATTN_SCORE_SOFTCAP) && !(p->softcap > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if ((variant & ATTN_SCORE_RELBIAS) &&
      (!p->rel_bias || (reinterpret_cast<uintptr_t>(p->rel_bias) & 3)))
    return ATTN_ERR_INVALID_ARG;
  if (p->q_offset < 0 || p->kv_offset < 0) return ATTN_ERR_INVALID_ARG;
  if ((long long)p->q_offset + Sq > INT_MAX || (long long)p->kv_offset + Skv > INT_MAX)
    return ATTN_ERR_INVALID_ARG;  // absolute positions are int
  if ((variant & ATTN_SCORE_RELBIAS) && (p->q_offset || p->kv_offset))
    return ATTN_ERR_UNSUPPORTED;
  const long long need = std::max((long long)p->q_offset + Sq, (long long)p->kv_offset + Skv);
  if (p->doc_len != 0 && p->doc_len < need) return ATTN_ERR_INVALID_ARG;
  (void)B;
  return ATTN_OK;
}

MaskArgs mask_args(unsigned variant, const attn_params* p, int Sq, int Skv) {
  MaskArgs m;
  m.variant = variant & ATTN_MASK_BITS;
  m.window = p->window;
  m.doc_id = p->doc_id;
  m.q_off = p->q_offset;
  m.kv_off = p->kv_offset;
  const long long lq = (long long)p->q_offset + Sq, lk = (long long)p->kv_offset + Skv;
  m.doc_len = p->doc_len ? p->doc_len : (int)(lq > lk ? lq : lk);
  m.prefix_len = p->prefix_len;
  return m;
}

// The block mask must describe the same mask and shape as the call.
attn_status check_block_mask(const attn_block_mask* bm, unsigned variant, const attn_params* p,
                             int B, int Sq, int Skv, bool need_transposed) {
  if (!bm) return ATTN_OK;
  const unsigned mbits = variant & ATTN_MASK_BITS;
  if (bm->B != B || bm->Sq != Sq || bm->Skv != Skv || bm->variant != mbits)
    return ATTN_ERR_INVALID_ARG;
  if ((mbits & ATTN_MASK_WINDOW) && bm->window != p->window) return ATTN_ERR_INVALID_ARG;
  if ((mbits & ATTN_MASK_DOCUMENT) && bm->doc_id != p->doc_id) return ATTN_ERR_INVALID_ARG;
  if ((mbits & ATTN_MASK_PREFIX) && bm->prefix_len != p->prefix_len) return ATTN_ERR_INVALID_ARG;
  if (bm->q_offset != p->q_offset || bm->kv_offset != p->kv_offset) return ATTN_ERR_INVALID_ARG;
  if ((mbits & ATTN_MASK_DOCUMENT) && bm->doc_len != mask_args(variant, p, Sq, Skv).doc_len)
    return ATTN_ERR_INVALID_ARG;
  if (!bm->full_cnt || !bm->part_cnt || !bm->full_idx || !bm->part_idx || !bm->order)
    return ATTN_ERR_INVALID_ARG;
  if (need_transposed && (!bm->t_full_cnt || !bm->t_part_cnt || !bm->t_full_idx ||
                          !bm->t_part_idx || !bm->t_order))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status fill_problem(FwdProblem& f, const void* q, const void* k, const void* v, void* o,
                         float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                         unsigned variant, const attn_params* p) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || Hkv < 1 || Sq < 0 || Skv < 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->dtype != ATTN_BF16 && p->dtype != ATTN_F32) return ATTN_ERR_UNSUPPORTED;
  attn_status st = check_mask_params(variant, p, B, Sq, Skv);
  if (st != ATTN_OK) return st;
  if (!std::isfinite(p->scale) || p->scale < 0.0f) return ATTN_ERR_INVALID_ARG;
  f = FwdProblem{};
  f.q = q;
  f.k = k;
  f.v = v;
  f.o = o;
  f.lse = lse;
  f.B = B;
  f.Hq = Hq;
  f.Hkv = Hkv;
  f.Sq = Sq;
  f.Skv = Skv;
  f.D = D;
  f.variant = variant;
  f.mask = mask_args(variant, p, Sq, Skv);
  f.score.scale = p->scale != 0.0f ? p->scale : 1.0f / std::sqrt((float)D);
  f.score.softcap = p->softcap;
  f.score.slopes = p->alibi_slopes;
  f.score.Hq = Hq;
  f.score.rel_bias = (variant & ATTN_SCORE_RELBIAS) ? p->rel_bias : nullptr;
  f.score.rb_len = Sq + Skv - 1;
  f.score.rb_zero = Skv - 1;
  if (p->block_mask) {
    const attn_block_mask* bm = p->block_mask;
    f.lists = BlockLists{bm->full_cnt, bm->part_cnt, bm->full_idx, bm->part_idx, bm->order,
                         bm->nq, bm->nkv};
  } else {
    f.lists = BlockLists{nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0};
  }
  f.status = p->status;  // resolved by resolve_status() once every check has passed
  f.timeout_ns = p->timeout_ns ? p->timeout_ns : 4000000000ull;
  f.fault_inject = p->fault_inject;
  f.page_table = p->page_table;
  f.page_size = p->page_size;
  f.pages_per_seq = p->pages_per_seq;
  f.num_pages = p->num_pages;
  return ATTN_OK;
}

attn_status resolve_status(FwdProblem& f) {
  if (!f.status) f.status = default_status();
  return f.status ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace mattn

using namespace mattn;

MATTN_API const char* attn_status_str(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "tensor base pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE_TOO_SMALL: return "buffer too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

MATTN_API size_t attn_block_mask_bytes(int B, int Sq, int Skv, int transposed) {
  if (B < 0 || Sq < 0 || Skv < 0) return 0;
  return mask_layout(B, Sq, Skv, transposed).total;
}

MATTN_API attn_status build_block_mask(unsigned variant, const attn_params* p, int B, int Sq,
                                       int Skv, void* buf, size_t bytes, int transposed,
                                       attn_block_mask* out, struct CUstream_st* stream) {
  if (!p || !out || B < 1 || Sq < 1 || Skv < 1) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_mask_params(variant, p, B, Sq, Skv);
  if (st != ATTN_OK) return st;
  if (!buf) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(buf) & 255u) return ATTN_ERR_MISALIGNED;
  const MaskLayout L = mask_layout(B, Sq, Skv, transposed);
  if (bytes < L.total) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  const MaskArgs m = mask_args(variant, p, Sq, Skv);
  char* base = static_cast<char*>(buf);
  auto at = [&](size_t off) { return reinterpret_cast<int*>(base + off); };
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = cuda_status(launch_block_mask(m, B, Sq, Skv, 0, at(L.full_cnt), at(L.part_cnt),
                                     at(L.full_idx), at(L.part_idx), at(L.order), s));
  if (st != ATTN_OK) return st;
  attn_block_mask r{};
  r.B = B;
  r.Sq = Sq;
  r.Skv = Skv;
  r.nq = (Sq + kTile - 1) / kTile;
  r.nkv = (Skv + kTile - 1) / kTile;
  r.variant = variant & ATTN_MASK_BITS;
  r.window = p->window;
  r.doc_id = (variant & ATTN_MASK_DOCUMENT) ? p->doc_id : nullptr;
  r.prefix_len = (variant & ATTN_MASK_PREFIX) ? p->prefix_len : nullptr;
  r.q_offset = p->q_offset;
  r.kv_offset = p->kv_offset;
  r.doc_len = m.doc_len;
  r.full_cnt = at(L.full_cnt);
  r.part_cnt = at(L.part_cnt);
  r.full_idx = at(L.full_idx);
  r.part_idx = at(L.part_idx);
  r.order = at(L.order);
  if (transposed) {
    st = cuda_status(launch_block_mask(m, B, Sq, Skv, 1, at(L.t_full_cnt), at(L.t_part_cnt),
                                       at(L.t_full_idx), at(L.t_part_idx), at(L.t_order), s));
    if (st != ATTN_OK) return st;
    r.t_full_cnt = at(L.t_full_cnt);
    r.t_part_cnt = at(L.t_part_cnt);
    r.t_full_idx = at(L.t_full_idx);
    r.t_part_idx = at(L.t_part_idx);
    r.t_order = at(L.t_order);
  }
  *out = r;
  return ATTN_OK;
}

MATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int Hq, int Hkv, int Sq, int Skv, int D, unsigned variant,
                               const attn_params* p, struct CUstream_st* stream) {
  FwdProblem f;
  attn_status st = fill_problem(f, q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, variant, p);
  if (st != ATTN_OK) return st;
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !o || !lse || (Skv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return ATTN_ERR_MISALIGNED;
  st = check_block_mask(p->block_mask, variant, p, B, Sq, Skv, false);
  if (st != ATTN_OK) return st;
  if (p->page_table) {  // paged K/V cache: bf16 tensor-core forward only
    if (p->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
    if (variant & ATTN_SCORE_RELBIAS) return ATTN_ERR_UNSUPPORTED;
    const int ps = p->page_size;
    if (ps != 16 && ps != 32 && ps != 64 && ps != 128) return ATTN_ERR_UNSUPPORTED;
    if (p->num_pages < 1 || p->pages_per_seq < 1 ||
        (long long)p->pages_per_seq * ps < (long long)Skv)
      return ATTN_ERR_INVALID_ARG;
    if (!aligned16(p->page_table) && (reinterpret_cast<uintptr_t>(p->page_table) & 3))
      return ATTN_ERR_MISALIGNED;
  }
  st = resolve_status(f);
  if (st != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int elem = p->dtype == ATTN_F32 ? 4 : 2;
  if (Skv == 0) {  // every row is empty: O = 0, LSE = -inf
    fill_empty_rows<<<256, 256, 0, s>>>(o, lse, (size_t)B * Hq * Sq, D, elem);
    return cuda_status(cudaGetLastError());
  }
  cudaError_t e;
  if (p->dtype == ATTN_F32) {
    e = launch_fwd_f32(f, s);
  } else {
    e = launch_fwd_tc(f, s);
  }
  return cuda_status(e);
}

namespace mattn {
namespace {

constexpr int kDecodeMaxRows = 16;  // query heads per key/value head times Sq

// Splits of the keys for decode: enough CTAs for about eight per SM (more
// loads in flight: on 16 sequences x 8 key/value heads x 32768 keys, 10
// splits ran at 0.87 of the measured HBM bandwidth against 0.82-0.85 with 3),
// at least 128 keys per split, at most 64 splits; chunk = keys per split
// (multiple of 16). Returns the split count.
int decode_splits(int B, int Hkv, int Skv, int& chunk) {
  const long long ctas = (long long)B * Hkv;
  long long want = ctas > 0 ? (8LL * sm_count() + ctas - 1) / ctas : 1;
  long long cap = (Skv + 127) / 128;
  if (want > cap) want = cap;
  if (want > 64) want = 64;
  if (want < 1) want = 1;
  chunk = (int)(((Skv + want - 1) / want + 15) / 16 * 16);
  if (chunk < 16) chunk = 16;
  return (int)((Skv + chunk - 1) / chunk);
}

size_t decode_ws_per_split(int B, int Hq, int Sq, int D) {
  const size_t rows = (size_t)B * Hq * Sq;
  return align256(rows * D * sizeof(float)) + align256(rows * sizeof(float));
}

}  // namespace
}  // namespace mattn

MATTN_API size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1 || (D != 64 && D != 128)) return 0;
  int chunk = 0;
  const int splits = decode_splits(B, Hkv, Skv, chunk);
  return splits > 1 ? (size_t)splits * decode_ws_per_split(B, Hq, Sq, D) : 0;
}

MATTN_API attn_status attn_decode(const void* q, const void* k, const void* v, void* o,
                                  float* lse, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                  unsigned variant, const attn_params* p, void* workspace,
                                  size_t workspace_bytes, struct CUstream_st* stream) {
  DecodeProblem dp;
  attn_status st = fill_problem(dp.f, q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, variant, p);
  if (st != ATTN_OK) return st;
  if (p->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if ((long long)(Hq / Hkv) * Sq > kDecodeMaxRows) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hkv > 65535) return ATTN_ERR_UNSUPPORTED;  // one grid row per (b, hkv)
  if (B == 0 || Sq == 0) return ATTN_OK;
  if (!q || !o || !lse || (Skv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3))
    return ATTN_ERR_MISALIGNED;
  if (p->page_table) {
    const int ps = p->page_size;
    if (ps != 16 && ps != 32 && ps != 64 && ps != 128) return ATTN_ERR_UNSUPPORTED;
    if (p->num_pages < 1 || p->pages_per_seq < 1 ||
        (long long)p->pages_per_seq * ps < (long long)Skv)
      return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(p->page_table) & 3) return ATTN_ERR_MISALIGNED;
  }
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_MISALIGNED;
  st = resolve_status(dp.f);
  if (st != ATTN_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Skv == 0) {  // every row is empty: O = 0, LSE = -inf
    fill_empty_rows<<<256, 256, 0, s>>>(o, lse, (size_t)B * Hq * Sq, D, 2);
    return cuda_status(cudaGetLastError());
  }
  // keys that some row can keep: without a prefix term, the causal bound of
  // the last row and the window bound of the first one limit them
  long long k_begin = 0, k_end = Skv;
  if (!(variant & ATTN_MASK_PREFIX)) {
    const long long qo = p->q_offset, ko = p->kv_offset;
    if (variant & ATTN_MASK_CAUSAL) k_end = std::min<long long>(k_end, qo + Sq - ko);
    if (variant & ATTN_MASK_WINDOW) k_begin = std::max<long long>(0, qo - p->window + 1 - ko);
  }
  k_begin &= ~15LL;
  if (k_end <= k_begin) {  // no row keeps a key: O = 0, LSE = -inf
    fill_empty_rows<<<256, 256, 0, s>>>(o, lse, (size_t)B * Hq * Sq, D, 2);
    return cuda_status(cudaGetLastError());
  }
  const int span = (int)(k_end - k_begin);
  int chunk = 0;
  int splits = decode_splits(B, Hkv, span, chunk);
  const size_t per = decode_ws_per_split(B, Hq, Sq, D);
  const size_t fit = workspace ? workspace_bytes / per : 0;
  if ((size_t)splits > fit) {  // as many splits as the workspace holds
    splits = fit >= 2 ? (int)fit : 1;
    chunk = (int)(((span + splits - 1) / splits + 15) / 16 * 16);
    splits = (span + chunk - 1) / chunk;
  }
  if (splits <= 1) {
    chunk = (span + 15) / 16 * 16;
    splits = 1;
  }
  dp.splits = splits;
  dp.chunk = chunk;
  dp.k_begin = (int)k_begin;
  dp.k_end = (int)k_end;
  const size_t rows = (size_t)B * Hq * Sq;
  dp.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  dp.ws_lse = splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                    align256(rows * D * sizeof(float)) * splits)
                         : nullptr;
  st = cuda_status(launch_decode(dp, s));
  if (st != ATTN_OK || splits == 1) return st;
  return cuda_status(launch_combine_f32_bf16(dp.ws_o, dp.ws_lse, splits, (long long)rows, D, o,
                                             lse, s));
}

MATTN_API size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq) {
  if (B < 0 || Hq < 0 || Sq < 0) return 0;
  return sizeof(float) * (size_t)B * Hq * Sq;
}

namespace mattn {
namespace {

// Byte offsets in the workspace of the backward's fp16 path: the Delta row
// terms, the range record, then the fp16 copies of Q, K, V, dO, each 256-byte
// aligned. Returns the total.
struct BwdF16Layout {
  size_t rec, q16, k16, v16, do16, total;
};

BwdF16Layout bwd_f16_layout(int B, int Hq, int Hkv, int Sq, int Skv, int D) {
  BwdF16Layout l;
  l.rec = align256(sizeof(float) * (size_t)B * Hq * Sq);
  l.q16 = l.rec + 256;
  const size_t nq = align256((size_t)B * Hq * Sq * D * 2), nk = align256((size_t)B * Hkv * Skv * D * 2);
  l.k16 = l.q16 + nq;
  l.v16 = l.k16 + nk;
  l.do16 = l.v16 + nk;
  l.total = l.do16 + nq;
  return l;
}

}  // namespace
}  // namespace mattn

MATTN_API size_t attn_bwd_workspace_bytes_f16(int B, int Hq, int Hkv, int Sq, int Skv, int D) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Skv < 0 || D < 0) return 0;
  return mattn::bwd_f16_layout(B, Hq, Hkv, Sq, Skv, D).total;
}

namespace mattn {

// Every check of attn_bwd's arguments except those on the workspace; makes no
// CUDA call. Fills bp.f on success.
attn_status bwd_check_args(BwdProblem& bp, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                           unsigned variant, const attn_params* p) {
  attn_status st = fill_problem(bp.f, q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B,
                                Hq, Hkv, Sq, Skv, D, variant, p);
  if (st != ATTN_OK) return st;
  if (p->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (p->page_table) return ATTN_ERR_UNSUPPORTED;                 // forward only
  if (B == 0 || Sq == 0 || Skv == 0) return ATTN_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse) ||
      ((variant & ATTN_MASK_DOCUMENT) && !aligned16(p->doc_id)))
    return ATTN_ERR_MISALIGNED;
  return check_block_mask(p->block_mask, variant, p, B, Sq, Skv, true);
}

}  // namespace mattn

MATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dO, void* dq, void* dk, void* dv,
                               void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                               int Sq, int Skv, int D, unsigned variant, const attn_params* p,
                               struct CUstream_st* stream) {
  BwdProblem bp;
  attn_status st = bwd_check_args(bp, q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D,
                                  variant, p);
  if (st != ATTN_OK) return st;
  if (!workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, Hq, Sq)) return ATTN_ERR_WORKSPACE_TOO_SMALL;
  st = resolve_status(bp.f);
  if (st != ATTN_OK) return st;
  bp.dO = dO;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  bp.delta = static_cast<float*>(workspace);
  // fp16 path: whole tiles at offset 0 without the bias table, and room for
  // the copies
  const BwdF16Layout fl = bwd_f16_layout(B, Hq, Hkv, Sq, Skv, D);
  if (workspace_bytes >= fl.total && Sq % 128 == 0 && Skv % 128 == 0 && p->q_offset == 0 &&
      p->kv_offset == 0 && !(variant & ATTN_SCORE_RELBIAS)) {
    char* w = static_cast<char*>(workspace);
    bp.f16_max = reinterpret_cast<unsigned*>(w + fl.rec);
    bp.q16 = w + fl.q16;
    bp.k16 = w + fl.k16;
    bp.v16 = w + fl.v16;
    bp.do16 = w + fl.do16;
  }
  if (p->block_mask) {
    const attn_block_mask* bm = p->block_mask;
    bp.t_lists = BlockLists{bm->t_full_cnt, bm->t_part_cnt, bm->t_full_idx, bm->t_part_idx,
                            bm->t_order, bm->nkv, bm->nq};
  } else {
    bp.t_lists = BlockLists{nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0};
  }
  const cudaError_t e = launch_bwd_tc(bp, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
  return cuda_status(e);
}

MATTN_API attn_status attn_check_status(int* status_dev, struct CUstream_st* stream) {
  int* addr = status_dev ? status_dev : default_status();
  if (!addr) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  attn_status st = cuda_status(cudaStreamSynchronize(s));
  if (st != ATTN_OK) return st;
  int h = 0;
  st = cuda_status(cudaMemcpy(&h, addr, sizeof(int), cudaMemcpyDeviceToHost));
  if (st != ATTN_OK) return st;
  if (h != 0) {
    st = cuda_status(cudaMemset(addr, 0, sizeof(int)));
    if (st != ATTN_OK) return st;
  }
  return static_cast<attn_status>(h);
}

MATTN_API const char* attn_last_cuda_error(void) {
  return cudaGetErrorName(t_last_cuda_error);
}

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(api)
}  // namespace mattn

#ifdef MATTN_DEBUG
// ---------------------------------------------------------------------------
// Debug build only: the bounds-check records (debug.cuh) of every kernel
// translation unit, and a self-test of the check.
// ---------------------------------------------------------------------------
#include "mattn_debug.h"

namespace mattn {
namespace {

__global__ void debug_selftest_kernel(int* buf, int n) {
  const int t = threadIdx.x;
  const long long idx = t == 0 ? (long long)n + 3 : t;  // thread 0: planted past the end
  if (MATTN_IN_BOUNDS(kSiteSelfTest, idx, n)) buf[idx] += 1;
}

struct DebugTu {
  cudaError_t (*fetch)(DebugRecord*);
  cudaError_t (*clear)();
};

const DebugTu kDebugTus[] = {
    {debug_fetch_api, debug_clear_api},
    {debug_fetch_fwd_f32, debug_clear_fwd_f32},
    {debug_fetch_fwd_tc, debug_clear_fwd_tc},
    {debug_fetch_fwd_tc_rb, debug_clear_fwd_tc_rb},
    {debug_fetch_fwd_tc_paged, debug_clear_fwd_tc_paged},
    {debug_fetch_bwd_tc, debug_clear_bwd_tc},
    {debug_fetch_bwd_tc_ragged, debug_clear_bwd_tc_ragged},
    {debug_fetch_bwd_tc_f16, debug_clear_bwd_tc_f16},
    {debug_fetch_decode, debug_clear_decode},
    {debug_fetch_combine, debug_clear_combine},
    {debug_fetch_mask_build, debug_clear_mask_build},
};

}  // namespace
}  // namespace mattn

MATTN_API attn_status attn_debug_record(attn_debug_info* out, int clear) {
  using namespace mattn;
  if (!out) return ATTN_ERR_INVALID_ARG;
  *out = attn_debug_info{};
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  for (const DebugTu& tu : kDebugTus) {
    DebugRecord r{};
    e = tu.fetch(&r);
    if (e != cudaSuccess) return cuda_status(e);
    if (r.count && !out->count) {
      out->site = r.site;
      out->index = r.index;
      out->bound = r.bound;
    }
    out->count += r.count;
    if (clear && r.count) {
      e = tu.clear();
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  return ATTN_OK;
}

MATTN_API const char* attn_debug_site_name(int site) {
  using namespace mattn;
  switch (site) {
    case kSiteNone: return "none";
    case kSiteFwdList: return "forward: block-mask list entry";
    case kSiteFwdPage: return "forward: page-table entry";
    case kSiteFwdDoc: return "forward: document id";
    case kSiteFwdO: return "forward: O row store";
    case kSiteFwdLse: return "forward: LSE store";
    case kSiteBwdList: return "backward: block-mask list entry";
    case kSiteBwdRow: return "backward: LSE / Delta row term";
    case kSiteBwdDoc: return "backward: document id";
    case kSiteBwdGrad: return "backward: dQ / dK / dV row store";
    case kSiteDecQ: return "decode: query row";
    case kSiteDecKV: return "decode: key / value row";
    case kSiteDecTable: return "decode: page-table entry";
    case kSiteDecSide: return "decode: document id or relative-bias entry";
    case kSiteDecOut: return "decode: output or split partial store";
    case kSiteCombineIn: return "merge: part row or LSE";
    case kSiteCombineOut: return "merge: merged row store";
    case kSiteF32: return "fp32 forward: list entry, document id or bias entry";
    case kSiteMaskBuild: return "block-mask builder: document id or order entry";
    case kSiteSelfTest: return "self-test: planted index";
  }
  return "unknown";
}

MATTN_API attn_status attn_debug_selftest(struct CUstream_st* stream) {
  using namespace mattn;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  constexpr int n = 16;
  DebugRecord r{};
  cudaError_t e = debug_clear_api();
  int* buf = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&buf, n * sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(buf, 0, n * sizeof(int), s);
  if (e == cudaSuccess) {
    debug_selftest_kernel<<<1, n, 0, s>>>(buf, n);
    e = cudaGetLastError();
  }
  int host[n] = {};
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, buf, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = debug_fetch_api(&r);
  if (buf) cudaFree(buf);
  if (e != cudaSuccess) return cuda_status(e);
  bool good = r.count == 1 && r.site == kSiteSelfTest && r.index == n + 3 && r.bound == n &&
              host[0] == 0;
  for (int t = 1; t < n; ++t) good = good && host[t] == 1;
  e = debug_clear_api();
  if (e != cudaSuccess) return cuda_status(e);
  return good ? ATTN_OK : ATTN_ERR_UNSUPPORTED;
}
#endif  // MATTN_DEBUG
