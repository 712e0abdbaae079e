// Tensor-memory (tcgen05) router GEMM for large batches; see router_tc.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Batches of more than 64 tokens (with H >= 64) take the tcgen05 kernel
// (measured at H = 6144, E = 256: T = 96 / 128 / 224 in 8.5 / 8.4 / 8.7 us
// against 10.4 / 10.3 / 10.7 us for the register-fed mma.sync kernel with
// 32-token tiles and 9.5 / 9.9 / 14.2 us with 16-token tiles; at T = 64 the
// mma.sync kernel takes 4.8 against 8.3 us).
constexpr int64_t kRouterTcMinT = 65;

bool router_tc_supported(int64_t T, int64_t H);

// logits[T, E] = x[T, H] . W[E, H]^T on the tcgen05 tensor cores (one launch);
// a bounded wait that runs out raises MOE_FLAG_TIMEOUT in err_flag (if given).
cudaError_t launch_router_tc(const void* x, const void* w, float* logits, int T, int H, int E, int32_t* err_flag,
                             int nsm, cudaStream_t stream);

}  // namespace moe
