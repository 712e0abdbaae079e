// Host-side helpers of the C ABI: argument checks, the per-device SM-count
// cache and the mapping of CUDA launch errors to status codes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>

#include "moe_tail.h"  // include/ is on the include path

namespace moe {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Number of SMs of the current device, queried once per device.
int sm_count();

// Status of the launch just made on this thread.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Test hook of the launch-error path (moe_debug_fail_next_launch): true once
// after a request, taken by the next launch of any entry point.
bool take_injected_launch_failure();

// Dynamic shared memory of a launch: `bytes`, or, when a launch failure was
// requested, more than any block may have, so that the runtime refuses the
// launch before anything runs and the entry point returns MOE_ERR_CUDA.
inline size_t launch_smem(size_t bytes) {
  return take_injected_launch_failure() ? (static_cast<size_t>(1) << 22) : bytes;
}

// Launch attribute that lets a kernel start while the previous kernel on the
// stream finishes (the kernels wait on the dependency before touching memory).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Largest number of tokens put on grid.y by one launch; the entry points loop
// over larger T in chunks of this size.
constexpr int64_t kMaxGridY = 65535;

}  // namespace moe
