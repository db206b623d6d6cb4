// Launches of the backward (kernel in bwd_tc_kernel.cuh) for sequence
// lengths that are multiples of the 128-row tile at position offset 0 without
// the relative-position bias; other calls go to the GENERAL instantiation
// compiled in bwd_tc_ragged.cu.
#include "bwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_bwd_tc(const BwdProblem& bp, cudaStream_t stream) {
  if (bp.f.Sq % kTile != 0 || bp.f.Skv % kTile != 0 || bp.f.mask.q_off != 0 ||
      bp.f.mask.kv_off != 0 || (bp.f.variant & ATTN_SCORE_RELBIAS))
    return launch_bwd_tc_ragged(bp, stream);
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (bp.f.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0, false>(bp, stream);
      case 1: return launch_typed<64, 1, false>(bp, stream);
      case 2: return launch_typed<64, 2, false>(bp, stream);
      default: return launch_typed<64, 3, false>(bp, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0, false>(bp, stream);
    case 1: return launch_typed<128, 1, false>(bp, stream);
    case 2: return launch_typed<128, 2, false>(bp, stream);
    default: return launch_typed<128, 3, false>(bp, stream);
  }
}

MATTN_DEBUG_RECORD_ACCESSORS(bwd_tc)

}  // namespace mattn
