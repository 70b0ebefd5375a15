// Host-only helpers of the ConvRot C ABI.
#include "../../include/convrot.h"

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
