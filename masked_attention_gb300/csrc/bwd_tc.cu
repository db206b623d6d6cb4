// Launches of the backward (kernel in bwd_tc_kernel.cuh) for sequence
// lengths that are multiples of the 128-row tile at position offset 0 without
// the relative-position bias; other calls go to the GENERAL instantiation
// compiled in bwd_tc_ragged.cu. With fp16 copies in the workspace the fp16
// kernels (compiled in bwd_tc_f16.cu) run, each followed by its bf16
// counterpart, of which the one the inputs' range does not select returns at
// once.
#include "bwd_tc_kernel.cuh"

namespace mattn {

namespace {

template <int D, int SCORE>
cudaError_t launch_bf16(const BwdProblem& bp, cudaStream_t stream) {
  if (!bp.f16_max) return launch_typed<D, SCORE, false>(bp, stream);
  cudaError_t e = launch_bwd_f16_prepare(bp, stream);
  if (e != cudaSuccess) return e;
  e = launch_delta(bp, stream);
  if (e != cudaSuccess) return e;
  for (int mode : {int(kDQ), int(kDKV)}) {
    e = launch_bwd_f16_mode(bp, mode, stream);
    if (e != cudaSuccess) return e;
    e = launch_mode<D, SCORE, false, false>(bp, mode, bp.f16_max, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdProblem& bp, cudaStream_t stream) {
  if (bp.f.Sq % kTile != 0 || bp.f.Skv % kTile != 0 || bp.f.mask.q_off != 0 ||
      bp.f.mask.kv_off != 0 || (bp.f.variant & ATTN_SCORE_RELBIAS))
    return launch_bwd_tc_ragged(bp, stream);
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (bp.f.D == 64) {
    switch (score) {
      case 0: return launch_bf16<64, 0>(bp, stream);
      case 1: return launch_bf16<64, 1>(bp, stream);
      case 2: return launch_bf16<64, 2>(bp, stream);
      default: return launch_bf16<64, 3>(bp, stream);
    }
  }
  switch (score) {
    case 0: return launch_bf16<128, 0>(bp, stream);
    case 1: return launch_bf16<128, 1>(bp, stream);
    case 2: return launch_bf16<128, 2>(bp, stream);
    default: return launch_bf16<128, 3>(bp, stream);
  }
}

MATTN_DEBUG_RECORD_ACCESSORS(bwd_tc)

}  // namespace mattn
