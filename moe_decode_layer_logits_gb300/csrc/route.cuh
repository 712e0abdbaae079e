// Top-k routing of one token by one warp: selection by logit (descending,
// equal logits in ascending expert order) and the routing weights
// scale * softmax over the selected logits (vllm-project/vllm pull 62174,
// Details: the router folds the routed scaling factor into the weights).
#pragma once

#include "common.cuh"

namespace moe {

// Orders (value, index) pairs: larger value first, then lower index.
__device__ __forceinline__ bool route_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// `row` points at the E logits of one token in shared memory.  Writes the k
// selected expert ids and their weights to sel_id[0..k) / sel_w[0..k) (shared
// memory).  Called by all 32 lanes of one warp; k <= 32, E <= 1024.
__device__ __forceinline__ void warp_route(const float* row, int E, int k, float scale,
                                           int* sel_id, float* sel_w) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit s: element lane + 32 s already selected
  float my_val = 0.f;  // lane j keeps the logit selected in round j
  for (int round = 0; round < k; ++round) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int i = lane, s = 0; i < E; i += 32, ++s) {
      if ((taken >> s) & 1u) continue;
      const float v = row[i];
      if (route_better(v, i, bv, bi)) { bv = v; bi = i; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (route_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == round) my_val = bv;
    if (lane == 0) sel_id[round] = bi;
  }
  // weights: exp relative to the largest selected logit, summed over lanes
  const float top = __shfl_sync(0xFFFFFFFFu, my_val, 0);
  const float e = lane < k ? expf(my_val - top) : 0.f;
  const float sum = warp_sum(e);
  if (lane < k) sel_w[lane] = (scale * e) / sum;
}

}  // namespace moe
