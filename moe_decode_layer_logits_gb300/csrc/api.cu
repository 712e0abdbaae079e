// Status strings and the per-device attribute cache of the C ABI.
#include "host_util.h"

namespace moe {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};  // 0 = not queried yet (a benign race: every writer stores the same value)
}  // namespace

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

}  // namespace moe

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null pointer or argument out of range";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: size not handled by the kernels";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: pointer breaks the alignment rule";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: the CUDA runtime reported a launch error";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX: an expanded-index map entry was out of range";
    default: return "unknown moe status";
  }
}
