// Launches of the bf16 tensor-core forward (kernel in fwd_tc_kernel.cuh) for
// the score_mod variants with the relative-position bias (SCORE bit 4).
#include "fwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_fwd_tc_rb(const FwdProblem& p, cudaStream_t stream) {
  const int score = ((p.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((p.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (p.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 4>(p, stream);
      case 1: return launch_typed<64, 5>(p, stream);
      case 2: return launch_typed<64, 6>(p, stream);
      default: return launch_typed<64, 7>(p, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 4>(p, stream);
    case 1: return launch_typed<128, 5>(p, stream);
    case 2: return launch_typed<128, 6>(p, stream);
    default: return launch_typed<128, 7>(p, stream);
  }
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(fwd_tc_rb)
}  // namespace mattn
