// Tensor-memory (tcgen05) router GEMM for large batches; see router_tc.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Batches of at least this many tokens (with H >= 64) take the tcgen05 kernel
// (measured at H = 6144, E = 256: 11.4 against 19.8 us at T = 256).
constexpr int64_t kRouterTcMinT = 256;

bool router_tc_supported(int64_t T, int64_t H);

// logits[T, E] = x[T, H] . W[E, H]^T on the tcgen05 tensor cores (one launch).
cudaError_t launch_router_tc(const void* x, const void* w, float* logits, int T, int H, int E, int nsm,
                             cudaStream_t stream);

}  // namespace moe
