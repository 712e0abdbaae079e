// Top-k routing of one token by one warp: selection by logit (descending,
// equal logits in ascending expert order) and the routing weights
// scale * softmax over the selected logits (vllm-project/vllm pull 62174,
// Details: the router folds the routed scaling factor into the weights).
//
// Lane l holds the logits of experts l, l + 32, ... as order-preserving
// integer keys in registers.  Two selection schemes give the same result:
//  - rounds (any k): each of the k rounds scans the lane's keys (the first
//    maximum wins, i.e. the lowest expert of the lane), then two warp
//    reductions pick the largest key and, among lanes holding it, the lowest
//    expert index; the winner clears its key;
//  - a merge network (k <= 8, at most 8 keys per lane): each lane sorts its
//    candidates, packed as (key, inverted expert index) so that one 64-bit
//    order ranks by logit and then by lower expert, and five butterfly steps
//    merge the lanes' sorted top-8 lists until every lane holds the warp's.
// The rounds issue fewer instructions (better where many warps share an SM);
// the network has the shorter dependency chain (better when one token's
// routing is on the critical path).  Key 0 marks a taken or padding slot:
// every finite logit has a key >= 1.
#pragma once

#include "common.cuh"

namespace moe {

// Monotone map float -> uint32 (a < b  <=>  key(a) < key(b)); -0 and +0 share
// the key of +0, so they tie like equal floats.
__device__ __forceinline__ uint32_t route_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float route_unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Load a token's logits row (global memory, E <= 32 * EPL); lane l gets
// experts l, l + 32, ...  The raw bits are loaded where this is called (the
// loads are not moved towards their first use) and turned into keys by
// route_select, so a caller can issue them early and keep working while they
// fly.  Slots past E hold a marker that route_select turns into key 0.
template <int EPL>
__device__ __forceinline__ void route_load_keys(const float* __restrict__ row, int E, uint32_t (&key)[EPL]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < EPL; ++s) {
    const int i = lane + 32 * s;
    if (i < E) {
      asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(key[s]) : "l"(row + i));
    } else {
      key[s] = 0xFFFFFFFFu;  // a NaN pattern no finite logit has
    }
  }
}

// Raw logit bits (route_load_keys) -> order-preserving keys; the past-E
// marker becomes 0.
template <int EPL>
__device__ __forceinline__ void route_bits_to_keys(uint32_t (&key)[EPL]) {
#pragma unroll
  for (int s = 0; s < EPL; ++s) key[s] = key[s] == 0xFFFFFFFFu ? 0u : route_key(__uint_as_float(key[s]));
}

// Compare-exchange leaving the larger value in `a`.
__device__ __forceinline__ void cx_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b;
  b = a > b ? b : a;
  a = hi;
}

// The warp's 8 largest packed candidates, sorted descending, in every lane.
// Lane l contributes experts l + 32 s (s < EPL <= 8).
template <int EPL>
__device__ __forceinline__ void route_top8(const uint32_t (&key)[EPL], uint64_t (&v)[8]) {
  static_assert(EPL >= 1 && EPL <= 8, "the merge network holds 8 candidates per lane");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 8; ++s)
    v[s] = s < EPL ? (static_cast<uint64_t>(key[s < EPL ? s : 0]) << 32) |
                         static_cast<uint32_t>(~(lane + 32 * s))
                   : 0ull;
  // bitonic sort of the lane's 8 candidates, descending
#pragma unroll
  for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          if ((i & size) == 0) cx_desc(v[i], v[j]);
          else cx_desc(v[j], v[i]);
        }
      }
    }
  }
  // merge with the partner lane's list: the top 8 of two descending lists a,
  // b are max(a[i], b[7 - i]) (a bitonic sequence), sorted by three steps
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint64_t m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v[7 - i], d);
      m[i] = v[i] > o ? v[i] : o;
    }
#pragma unroll
    for (int stride = 4; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((i & stride) == 0) cx_desc(m[i], m[i + stride]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = m[i];
  }
}

// Select the top k (1 <= k <= min(E, 32)) of the logits loaded by
// route_load_keys and weight them.  All 32 lanes call this; lane j < k
// receives the j-th selected expert in `id` and its weight in `w`.  Consumes
// `key`.  NETWORK
// picks the merge network where it applies (k <= 8, EPL <= 8).
template <int EPL, bool NETWORK>
__device__ __forceinline__ void route_select(uint32_t (&key)[EPL], int k, float scale, int& id, float& w) {
  const int lane = threadIdx.x & 31;
  route_bits_to_keys<EPL>(key);
  uint32_t my_key = 0u;
  int my_id = 0;
  int rounds = k;
  if constexpr (NETWORK && EPL <= 8) {
    if (k <= 8) {
      uint64_t v[8];
      route_top8<EPL>(key, v);
      uint64_t mine = 0ull;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i == lane) mine = v[i];
      my_key = static_cast<uint32_t>(mine >> 32);
      my_id = static_cast<int>(~static_cast<uint32_t>(mine));
      rounds = 0;
    }
  }
  for (int round = 0; round < rounds; ++round) {
    uint32_t bk = 0u;
    int bs = 0;
#pragma unroll
    for (int s = 0; s < EPL; ++s) {
      if (key[s] > bk) { bk = key[s]; bs = s; }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t cand = bk == m ? static_cast<uint32_t>(lane + 32 * bs) : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (static_cast<int>(win & 31u) == lane) {
      const int ws = static_cast<int>(win >> 5);
#pragma unroll
      for (int s = 0; s < EPL; ++s) {
        if (s == ws) key[s] = 0u;
      }
    }
    if (lane == round) { my_key = m; my_id = static_cast<int>(win); }
  }
  // weights: exp relative to the largest selected logit, summed over lanes
  const float val = route_unkey(my_key);
  const float top = __shfl_sync(0xFFFFFFFFu, val, 0);
  const float e = lane < k ? expf(val - top) : 0.f;
  const float sum = warp_sum(e);
  id = my_id;
  w = (scale * e) / sum;
}

// Both phases for one token row.
template <int EPL, bool NETWORK>
__device__ __forceinline__ void warp_route(const float* __restrict__ row, int E, int k, float scale,
                                           int& id, float& w) {
  uint32_t key[EPL];
  route_load_keys<EPL>(row, E, key);
  route_select<EPL, NETWORK>(key, k, scale, id, w);
}

}  // namespace moe
