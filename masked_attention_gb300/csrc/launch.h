// Internal interface between the C ABI (api.cu) and the kernel translation
// units. Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "status.h"

namespace mattn {

struct FwdProblem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Sq, Skv, D;
  unsigned variant;
  MaskArgs mask;
  ScoreArgs score;
  BlockLists lists;  // lists.full_cnt == nullptr: visit every tile the causal bound allows
  int* status;
  uint64_t timeout_ns;
  unsigned fault_inject;  // ATTN_FAULT_NO_LOADS: the load warp issues nothing
  const int* page_table;  // paged K/V cache [B][pages_per_seq], or nullptr (contiguous)
  int page_size, pages_per_seq, num_pages;
};

struct BwdProblem {
  FwdProblem f;        // q, k, v, o (read), lse (read)
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* delta;        // workspace [B, Hq, Sq]
  BlockLists t_lists;  // transposed lists (per key tile), or full_cnt == nullptr
  // fp16 path (whole tiles at offset 0, workspace large enough): fp16 copies
  // of Q, K, V, dO in the workspace and the record of their largest |x|;
  // nullptr otherwise
  void* q16 = nullptr;
  void* k16 = nullptr;
  void* v16 = nullptr;
  void* do16 = nullptr;
  unsigned* f16_max = nullptr;
};

// Decode (few query rows against a long cache): one CTA per (batch element,
// key/value head, split of the keys); a split's partial result goes to the
// fp32 workspace when splits > 1, else straight to o and lse.
struct DecodeProblem {
  FwdProblem f;
  int splits;
  int chunk;     // keys per split, a multiple of 16
  int k_begin;   // keys [k_begin, k_end) can be kept (k_begin a multiple of 16);
  int k_end;     // split s covers [k_begin + s * chunk, ...) within them
  float* ws_o;   // [splits][B*Hq*Sq][D] fp32, or nullptr (splits == 1)
  float* ws_lse; // [splits][B*Hq*Sq]
};

cudaError_t launch_decode(const DecodeProblem& dp, cudaStream_t stream);

#ifdef MATTN_DEBUG
// Debug build: each kernel translation unit's bounds-check record (copy out
// and clear; see debug.cuh).
#define MATTN_DECLARE_DEBUG_RECORD(name)             \
  cudaError_t debug_fetch_##name(DebugRecord* out); \
  cudaError_t debug_clear_##name();
MATTN_DECLARE_DEBUG_RECORD(api)
MATTN_DECLARE_DEBUG_RECORD(fwd_f32)
MATTN_DECLARE_DEBUG_RECORD(fwd_tc)
MATTN_DECLARE_DEBUG_RECORD(fwd_tc_rb)
MATTN_DECLARE_DEBUG_RECORD(fwd_tc_paged)
MATTN_DECLARE_DEBUG_RECORD(bwd_tc)
MATTN_DECLARE_DEBUG_RECORD(bwd_tc_ragged)
MATTN_DECLARE_DEBUG_RECORD(bwd_tc_f16)
MATTN_DECLARE_DEBUG_RECORD(decode)
MATTN_DECLARE_DEBUG_RECORD(combine)
MATTN_DECLARE_DEBUG_RECORD(mask_build)
#undef MATTN_DECLARE_DEBUG_RECORD
#endif

// Merge of fp32 partial results into bf16 O (and fp32 LSE): the
// online-softmax merge of attn_combine with fp32 parts and a bf16 output.
cudaError_t launch_combine_f32_bf16(const float* o_parts, const float* lse_parts, int n_parts,
                                    long long rows, int D, void* o, float* lse,
                                    cudaStream_t stream);

// Block-mask builder: writes counts, ascending index lists and the
// longest-first order for the per-query-tile (transposed = 0) or per-key-tile
// (transposed = 1) view.
cudaError_t launch_block_mask(const MaskArgs& m, int B, int Sq, int Skv, int transposed,
                              int* cnt_full, int* cnt_part, int* idx_full, int* idx_part,
                              int* order, cudaStream_t stream);

cudaError_t launch_fwd_f32(const FwdProblem& p, cudaStream_t stream);
cudaError_t launch_fwd_tc(const FwdProblem& p, cudaStream_t stream);
cudaError_t launch_fwd_tc_rb(const FwdProblem& p, cudaStream_t stream);     // relative bias
cudaError_t launch_fwd_tc_paged(const FwdProblem& p, cudaStream_t stream);  // paged K/V
cudaError_t launch_bwd_tc(const BwdProblem& p, cudaStream_t stream);
// Sq or Skv not a multiple of 128, or position offsets (bwd_tc_ragged.cu).
cudaError_t launch_bwd_tc_ragged(const BwdProblem& p, cudaStream_t stream);
// fp16 path of the backward (bwd_tc_f16.cu): zero the range record and
// convert Q, K, V, dO to the fp16 copies; one fp16 kernel (mode: 0 dQ, 1 dK/dV)
cudaError_t launch_bwd_f16_prepare(const BwdProblem& p, cudaStream_t stream);
cudaError_t launch_bwd_f16_mode(const BwdProblem& p, int mode, cudaStream_t stream);

// The checks attn_bwd makes on everything but its workspace (no CUDA call);
// fills bp.f when they pass.
attn_status bwd_check_args(BwdProblem& bp, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                           unsigned variant, const attn_params* p);

}  // namespace mattn
