// Launches of the bf16 tensor-core forward (kernel in fwd_tc_kernel.cuh) that
// read K and V from a paged cache, for the score_mod variants without the
// relative-position bias.
#include "fwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_fwd_tc_paged(const FwdProblem& p, cudaStream_t stream) {
  const int score = ((p.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((p.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (p.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0, true>(p, stream);
      case 1: return launch_typed<64, 1, true>(p, stream);
      case 2: return launch_typed<64, 2, true>(p, stream);
      default: return launch_typed<64, 3, true>(p, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0, true>(p, stream);
    case 1: return launch_typed<128, 1, true>(p, stream);
    case 2: return launch_typed<128, 2, true>(p, stream);
    default: return launch_typed<128, 3, true>(p, stream);
  }
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(fwd_tc_paged)
}  // namespace mattn
