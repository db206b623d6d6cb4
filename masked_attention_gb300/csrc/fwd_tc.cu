// Launches of the bf16 tensor-core forward (kernel in fwd_tc_kernel.cuh) for
// the score_mod variants without the relative-position bias over contiguous
// K/V; the variants with the bias (fwd_tc_rb.cu) and over a paged cache
// (fwd_tc_paged.cu) are compiled in their own files, so the builds run in
// parallel.
#include "fwd_tc_kernel.cuh"

namespace mattn {

cudaError_t launch_fwd_tc(const FwdProblem& p, cudaStream_t stream) {
  if (p.page_table) return launch_fwd_tc_paged(p, stream);
  if (p.variant & ATTN_SCORE_RELBIAS) return launch_fwd_tc_rb(p, stream);
  const int score = ((p.variant & ATTN_SCORE_ALIBI) ? 1 : 0) |
                    ((p.variant & ATTN_SCORE_SOFTCAP) ? 2 : 0);
  if (p.D == 64) {
    switch (score) {
      case 0: return launch_typed<64, 0>(p, stream);
      case 1: return launch_typed<64, 1>(p, stream);
      case 2: return launch_typed<64, 2>(p, stream);
      default: return launch_typed<64, 3>(p, stream);
    }
  }
  switch (score) {
    case 0: return launch_typed<128, 0>(p, stream);
    case 1: return launch_typed<128, 1>(p, stream);
    case 2: return launch_typed<128, 2>(p, stream);
    default: return launch_typed<128, 3>(p, stream);
  }
}

}  // namespace mattn

namespace mattn {
MATTN_DEBUG_RECORD_ACCESSORS(fwd_tc)
}  // namespace mattn
