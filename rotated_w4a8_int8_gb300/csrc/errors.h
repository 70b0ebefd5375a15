// Recording of the CUDA error behind a CONVROT_ERR_CUDA status (per thread).
#pragma once
#include <cuda_runtime_api.h>

namespace convrot {
// Records "<what>: <CUDA error text>" and returns CONVROT_ERR_CUDA.
int record_cuda_error(const char* what, cudaError_t e);
// Records `what` verbatim and returns CONVROT_ERR_CUDA.
int record_error(const char* what);
}  // namespace convrot
