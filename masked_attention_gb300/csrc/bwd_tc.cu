// Backward kernels (built in a later step).
#include "launch.h"

namespace mattn {

cudaError_t launch_bwd_tc(const BwdProblem&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace mattn
