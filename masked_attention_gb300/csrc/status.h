// Mapping of CUDA runtime results onto the library's status codes, shared by
// every translation unit that returns one (the definition is in api.cu).
#pragma once

#include <cuda_runtime.h>

#include "mattn.h"

namespace mattn {

// ATTN_OK for cudaSuccess; otherwise ATTN_ERR_CUDA, remembering the error
// for attn_last_cuda_error() (per calling thread).
attn_status cuda_status(cudaError_t e);

}  // namespace mattn
