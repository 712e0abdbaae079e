// moe_topk_route: one warp per token selects the top-k experts from the FP32
// router logits and writes their ids and scaled softmax weights.
#include "host_util.h"
#include "route.cuh"

namespace moe {

constexpr int kRouteWarps = 4;  // tokens per CTA (4 measured faster than 8 at T = 64)

template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
topk_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ wts,
                  int T, int E, int k, float scale) {
  __shared__ __align__(16) uint64_t route_scr[kRouteWarps][kRouteScratch];  // each warp's candidate list
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + warp;
  allow_dependent_launch();
  grid_dependency_wait();
  if (t >= T) return;  // whole warp leaves together; the kernel has no block barrier
  int id;
  float w;
  warp_route<EPL>(logits + static_cast<int64_t>(t) * E, E, k, scale, id, w, route_scr[warp]);
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = id;
    wts[static_cast<int64_t>(t) * k + lane] = w;
  }
}

template <int EPL>
static cudaError_t launch_route(const float* logits, int32_t* ids, float* w, int T, int E, int k, float scale,
                         cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + kRouteWarps - 1) / kRouteWarps), 1, 1);
  cfg.blockDim = dim3(kRouteWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = launch_smem(0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_route_kernel<EPL>, logits, ids, w, T, E, k, scale);
}

}  // namespace moe

extern "C" int moe_topk_route(const float* logits, int32_t* topk_ids, float* topk_w,
                              int64_t T, int64_t E, int32_t k, float routed_scale,
                              cudaStream_t stream) {
  using namespace moe;
  if (T < 0 || E < 1 || k < 1 || k > E || k > MOE_MAX_K || !isfinite(routed_scale))
    return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_E) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_ERR_MISALIGNED;
  const int64_t per_launch = static_cast<int64_t>(1) << 30;  // keeps grid.x in range
  for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
    const int Tc = static_cast<int>(T - t0 < per_launch ? T - t0 : per_launch);
    const float* lg = logits + t0 * E;
    int32_t* ip = topk_ids + t0 * k;
    float* wp = topk_w + t0 * k;
    const int Ei = static_cast<int>(E);
    cudaError_t e;
    if (E <= 32) e = launch_route<1>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    else if (E <= 64) e = launch_route<2>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    else if (E <= 128) e = launch_route<4>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    else if (E <= 256) e = launch_route<8>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    else if (E <= 512) e = launch_route<16>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    else e = launch_route<32>(lg, ip, wp, Tc, Ei, k, routed_scale, stream);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    const int st = launch_status();
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}
