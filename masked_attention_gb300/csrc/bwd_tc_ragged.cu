// Launches of the backward (kernel in bwd_tc_kernel.cuh) for sequence
// lengths that are not multiples of the 128-row tile or calls at position
// offsets (the GENERAL instantiation; compiled in its own file, so the
// builds run in parallel).
#include "bwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_bwd_tc_ragged(const BwdProblem& bp, cudaStream_t stream) {
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (bp.f.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0, true>(bp, stream);
      case 1: return launch_typed<64, 1, true>(bp, stream);
      case 2: return launch_typed<64, 2, true>(bp, stream);
      default: return launch_typed<64, 3, true>(bp, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0, true>(bp, stream);
    case 1: return launch_typed<128, 1, true>(bp, stream);
    case 2: return launch_typed<128, 2, true>(bp, stream);
    default: return launch_typed<128, 3, true>(bp, stream);
  }
}

MATTN_DEBUG_RECORD_ACCESSORS(bwd_tc_ragged)

}  // namespace mattn
