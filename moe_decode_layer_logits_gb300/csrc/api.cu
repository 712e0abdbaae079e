// Status strings, the per-device attribute cache and the launch-error test
// hook of the C ABI.
#include <atomic>

#include "host_util.h"

namespace moe {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};  // 0 = not queried yet (a benign race: every writer stores the same value)
std::atomic<int> g_fail_next_launch{0};
}  // namespace

bool take_injected_launch_failure() {
  return g_fail_next_launch.load(std::memory_order_relaxed) != 0 && g_fail_next_launch.exchange(0) != 0;
}

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

extern "C" int moe_debug_fail_next_launch(int32_t on) {
  if (on != 0 && on != 1) return MOE_ERR_INVALID_ARG;
  moe::g_fail_next_launch.store(on);
  return MOE_OK;
}
