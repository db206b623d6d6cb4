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
};

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

// The checks attn_bwd makes on everything but its workspace (no CUDA call);
// fills bp.f when they pass.
attn_status bwd_check_args(BwdProblem& bp, const void* q, const void* k, const void* v,
                           const void* o, const float* lse, const void* dO, void* dq, void* dk,
                           void* dv, int B, int Hq, int Hkv, int Sq, int Skv, int D,
                           unsigned variant, const attn_params* p);

}  // namespace mattn
