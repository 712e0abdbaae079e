// Top-k routing of one token by one warp: selection by logit (descending,
// equal logits in ascending expert order) and the routing weights
// scale * softmax over the selected logits (vllm-project/vllm pull 62174,
// Details: the router folds the routed scaling factor into the weights).
//
// Lane l holds the logits of experts l, l + 32, ... as order-preserving
// integer keys in registers.  With at most 8 keys per lane (E <= 256) and
// k <= 16 the selection first bounds the k-th largest key from below: the
// lanes form G >= k groups, and the smallest of the G group maxima, tau, is
// exceeded or met by at least G >= k distinct keys, so every one of the top k
// is >= tau, and so is every key that beats one of them.  The keys >= tau
// (about 20 of 256 for k = 8 on Gaussian logits) are the candidates: ballots
// give each its place in a shared-memory list, each candidate counts the
// candidates that beat it (its rank), and the k best write themselves to
// their rank's slot.  No chain of k dependent warp reductions is left.  For
// larger k, or when more than kCandidateCap keys meet tau (heavy ties), the
// selection takes sorted heads: each lane sorts its keys, and each of k rounds
// takes one warp max over the lanes' heads, a ballot of the lanes holding it
// (a second reduction picks the lowest expert only when several lanes tie),
// and the winner pops its head.  Wider rows (E > 256) scan the lane's keys
// each round, then two reductions pick the largest key and the lowest expert
// holding it, and the winner clears its key.  Key 0 marks a taken or padding
// slot: every finite logit has a key >= 1.
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

// Candidate list of one routing warp: kCandidateCap entries, then the k
// selected ones (shared memory, 16-byte aligned).
constexpr int kCandidateCap = 64;
constexpr int kRouteScratch = kCandidateCap + 32;

// (key, expert) as one 64-bit value; a larger value is the better choice
// (larger key, then lower expert).
__device__ __forceinline__ uint64_t route_rank_value(uint32_t key, int expert) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(expert));
}

// Select the top k (1 <= k <= min(E, 32)) of the logits loaded by
// route_load_keys and weight them.  All 32 lanes call this; lane j < k
// receives the j-th selected expert in `id` and its weight in `w`.  Consumes
// `key`.  `scratch` holds kRouteScratch entries of shared memory that only
// this warp uses (for E <= 256, k <= 16), across calls; 16-byte aligned.
template <int EPL>
__device__ __forceinline__ void route_select(uint32_t (&key)[EPL], int k, float scale, int& id, float& w,
                                             uint64_t* scratch) {
  const int lane = threadIdx.x & 31;
  route_bits_to_keys<EPL>(key);
  uint32_t my_key = 0u;
  int my_id = 0;
  int rounds = k;
  if constexpr (EPL <= 8) {
    if (k <= 16) {
      // tau: the smallest of G group maxima, G = 8 or 16 >= k groups of 4 or
      // 2 lanes (larger k leaves too many candidates: sorted heads below)
      uint32_t gm = key[0];
#pragma unroll
      for (int s = 1; s < EPL; ++s) gm = key[s] > gm ? key[s] : gm;
      for (int d = 1; d < 32 && (32 / (2 * d)) >= k; d <<= 1) {
        const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, gm, d);
        gm = o > gm ? o : gm;
      }
      const uint32_t tau = __reduce_min_sync(0xFFFFFFFFu, gm);
      // the candidates' places in the list: slot-major, lanes in order
      // (ascending expert); places past the cap are not written, and a list
      // that would overflow is not used
      uint32_t below;
      asm("mov.u32 %0, %%lanemask_lt;" : "=r"(below));
      uint32_t bal[EPL];
#pragma unroll
      for (int s = 0; s < EPL; ++s) bal[s] = __ballot_sync(0xFFFFFFFFu, key[s] >= tau);
      __syncwarp();  // an earlier call's accesses to the list are complete
      int n = 0;
#pragma unroll
      for (int s = 0; s < EPL; ++s) {
        const int at = n + __popc(bal[s] & below);
        if (key[s] >= tau && at < kCandidateCap) scratch[at] = route_rank_value(key[s], lane + 32 * s);
        n += __popc(bal[s]);
      }
      if (n <= kCandidateCap) {
        // rank = how many candidates beat this one; the values are distinct
        // (one per expert), so the ranks are 0 .. n-1, each once.  The list
        // is padded with 0 (below every candidate) to whole blocks of 8, and
        // each lane ranks candidates lane and lane + 32 in one pass.
        const int nb = (n + 7) >> 3;
        __syncwarp();
        if (n + lane < 8 * nb) scratch[n + lane] = 0ull;
        __syncwarp();
        const ulonglong2* list = reinterpret_cast<const ulonglong2*>(scratch);
        const uint64_t v0 = lane < n ? scratch[lane] : ~0ull;
        const uint64_t v1 = lane + 32 < n ? scratch[lane + 32] : ~0ull;
        int r0 = 0, r1 = 0;
        for (int b = 0; b < nb; ++b) {
          ulonglong2 c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) c[i] = list[4 * b + i];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            r0 += (c[i].x > v0 ? 1 : 0) + (c[i].y > v0 ? 1 : 0);
            r1 += (c[i].x > v1 ? 1 : 0) + (c[i].y > v1 ? 1 : 0);
          }
        }
        uint64_t* chosen = scratch + kCandidateCap;
        if (lane < n && r0 < k) chosen[r0] = v0;
        if (lane + 32 < n && r1 < k) chosen[r1] = v1;
        __syncwarp();
        if (lane < k) {
          const uint64_t v = chosen[lane];
          my_key = static_cast<uint32_t>(v >> 32);
          my_id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(v));
        }
        rounds = 0;
      }
    }
    if (rounds > 0) {
      // Sorted heads: each lane sorts its keys once (descending key,
      // ascending slot among equal keys), then every round needs one warp
      // max over the lanes' heads and a ballot; only when several lanes tie
      // on that key does a second reduction pick the lowest expert.
      uint64_t v[EPL];
#pragma unroll
      for (int s = 0; s < EPL; ++s)
        v[s] = (static_cast<uint64_t>(key[s]) << 32) | static_cast<uint32_t>(0xFFFF - s);
#pragma unroll
      for (int size = 2; size <= EPL; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const int j = i ^ stride;
            if (j > i) {
              if ((i & size) == 0) cx_desc(v[i], v[j]);
              else cx_desc(v[j], v[i]);
            }
          }
        }
      }
      for (int round = 0; round < rounds; ++round) {
        const uint32_t head = static_cast<uint32_t>(v[0] >> 32);
        const uint32_t hexp = static_cast<uint32_t>(lane + 32 * (0xFFFF - static_cast<int>(v[0] & 0xFFFFu)));
        const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, head);
        const uint32_t tied = __ballot_sync(0xFFFFFFFFu, head == m);
        const uint32_t win = (tied & (tied - 1u)) == 0u
                                 ? __shfl_sync(0xFFFFFFFFu, hexp, __ffs(tied) - 1)
                                 : __reduce_min_sync(0xFFFFFFFFu, head == m ? hexp : 0xFFFFFFFFu);
        if (static_cast<int>(win & 31u) == lane) {  // the winner pops its head
#pragma unroll
          for (int i = 0; i + 1 < EPL; ++i) v[i] = v[i + 1];
          v[EPL - 1] = 0ull;
        }
        if (lane == round) { my_key = m; my_id = static_cast<int>(win); }
      }
      rounds = 0;
    }
  }
  for (int round = 0; round < rounds; ++round) {  // wider rows: scan the lane's keys each round
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
template <int EPL>
__device__ __forceinline__ void warp_route(const float* __restrict__ row, int E, int k, float scale,
                                           int& id, float& w, uint64_t* scratch) {
  uint32_t key[EPL];
  route_load_keys<EPL>(row, E, key);
  route_select<EPL>(key, k, scale, id, w, scratch);
}

}  // namespace moe
