// moe_topk_route: one warp per token selects the top-k experts from the FP32
// router logits and writes their ids and scaled softmax weights.
#include "host_util.h"
#include "route.cuh"

namespace moe {

constexpr int kRouteWarps = 8;  // tokens per CTA

__global__ void __launch_bounds__(kRouteWarps * 32)
topk_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids,
                  float* __restrict__ wts, int T, int E, int k, float scale) {
  extern __shared__ float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* row = smem + warp * E;
  int* sel_id = reinterpret_cast<int*>(smem + kRouteWarps * E) + warp * 2 * MOE_MAX_K;
  float* sel_w = reinterpret_cast<float*>(sel_id + MOE_MAX_K);
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;  // whole warp leaves together; no block-wide barrier below
  const float* src = logits + static_cast<int64_t>(t) * E;
  for (int i = lane; i < E; i += 32) row[i] = src[i];
  __syncwarp();
  warp_route(row, E, k, scale, sel_id, sel_w);
  __syncwarp();
  if (lane < k) {
    ids[static_cast<int64_t>(t) * k + lane] = sel_id[lane];
    wts[static_cast<int64_t>(t) * k + lane] = sel_w[lane];
  }
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
  const size_t smem = sizeof(float) * kRouteWarps * (E + 2 * MOE_MAX_K);
  const int64_t per_launch = kMaxGridY * kRouteWarps * 1024;  // grid.x limit is far away
  for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
    const int Tc = static_cast<int>(T - t0 < per_launch ? T - t0 : per_launch);
    const unsigned grid = static_cast<unsigned>((Tc + kRouteWarps - 1) / kRouteWarps);
    topk_route_kernel<<<grid, kRouteWarps * 32, smem, stream>>>(
        logits + t0 * E, topk_ids + t0 * k, topk_w + t0 * k, Tc, static_cast<int>(E), k, routed_scale);
    const int st = launch_status();
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}
