// Host-only helpers of the ConvRot C ABI.
#include <cstdio>

#include "../../include/convrot.h"
#include "errors.h"

static thread_local char g_last_error[256] = "";

namespace convrot {
int record_cuda_error(const char* what, cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorString(e),
                cudaGetErrorName(e));
  return CONVROT_ERR_CUDA;
}
int record_error(const char* what) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return CONVROT_ERR_CUDA;
}
}  // namespace convrot

extern "C" const char* convrot_last_error(void) { return g_last_error; }

extern "C" int convrot_padded_k(int K) {
  if (K <= 0) return 0;
  return static_cast<int>(((static_cast<long long>(K) + CONVROT_BLOCK - 1) / CONVROT_BLOCK) * CONVROT_BLOCK);
}

extern "C" const char* convrot_status_string(int status) {
  switch (status) {
    case CONVROT_OK: return "ok";
    case CONVROT_ERR_INVALID_ARG: return "invalid argument";
    case CONVROT_ERR_MISALIGNED: return "misaligned pointer or pitch";
    case CONVROT_ERR_UNSUPPORTED: return "unsupported dtype, code format or size";
    case CONVROT_ERR_CUDA: return "CUDA launch or runtime error";
    case CONVROT_ERR_DEVICE_TIMEOUT: return "a kernel timed out waiting on the device";
    default: return "unknown status";
  }
}
