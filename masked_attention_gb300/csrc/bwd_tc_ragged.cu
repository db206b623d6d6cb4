// Launches of the backward (kernel in bwd_tc_kernel.cuh) for sequence
// lengths that are not multiples of the 128-row tile, calls at position
// offsets and calls with the relative-position bias (the GENERAL
// instantiation; compiled in its own file, so the builds run in parallel).
#include "bwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_bwd_tc_ragged(const BwdProblem& bp, cudaStream_t stream) {
  const int score = ((bp.f.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((bp.f.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0) |
                    ((bp.f.variant & ATTN_SCORE_RELBIAS) ? 4 : 0);
  if (bp.f.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0, true>(bp, stream);
      case 1: return launch_typed<64, 1, true>(bp, stream);
      case 2: return launch_typed<64, 2, true>(bp, stream);
      case 3: return launch_typed<64, 3, true>(bp, stream);
      case 4: return launch_typed<64, 4, true>(bp, stream);
      case 5: return launch_typed<64, 5, true>(bp, stream);
      case 6: return launch_typed<64, 6, true>(bp, stream);
      default: return launch_typed<64, 7, true>(bp, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0, true>(bp, stream);
    case 1: return launch_typed<128, 1, true>(bp, stream);
    case 2: return launch_typed<128, 2, true>(bp, stream);
    case 3: return launch_typed<128, 3, true>(bp, stream);
    case 4: return launch_typed<128, 4, true>(bp, stream);
    case 5: return launch_typed<128, 5, true>(bp, stream);
    case 6: return launch_typed<128, 6, true>(bp, stream);
    default: return launch_typed<128, 7, true>(bp, stream);
  }
}

MATTN_DEBUG_RECORD_ACCESSORS(bwd_tc_ragged)

}  // namespace mattn
