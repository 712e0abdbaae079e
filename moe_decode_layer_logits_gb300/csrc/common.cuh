// Device helpers shared by the tail kernels: BF16 packing, streaming 16-byte
// loads and the warp / block / cluster sum reductions with a fixed order.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cooperative_groups.h>
#include <stdint.h>

namespace moe {

namespace cg = cooperative_groups;

// Two BF16 values in one 32-bit word, low half first.
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Round two floats to BF16 (nearest even) and pack them, `a` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 16-byte load through the read-only path that does not allocate in L1: the
// data is read once per launch (expert rows, activations).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load of data that several CTAs re-read (gamma, the router input x).
__device__ __forceinline__ uint4 ld_keep16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Unpack 8 BF16 values of a 16-byte vector into floats.
// The same 8 values as FP32 pairs (element 2i in .x, 2i + 1 in .y).
__device__ __forceinline__ void unpack8x2(const uint4& v, float2 f[4]) {
  f[0] = make_float2(bf16lo(v.x), bf16hi(v.x));
  f[1] = make_float2(bf16lo(v.y), bf16hi(v.y));
  f[2] = make_float2(bf16lo(v.z), bf16hi(v.z));
  f[3] = make_float2(bf16lo(v.w), bf16hi(v.w));
}

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialisation, so it may start while the previous
// kernel on the stream is still running.  It lets its own dependent start
// early (launch_dependents), and it reads or writes no global memory before
// grid_dependency_wait(), which returns once the previous grid has finished
// and its writes are visible.  Without a programmatic predecessor both are
// no-ops.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

// Sum of one float per thread over the block.  Warp partials go to
// scratch[warp]; thread 0 adds them in warp order, so every launch adds in
// the same order.  Every thread gets the total.  `scratch` holds >= 33 floats.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += scratch[w];
    scratch[32] = s;
  }
  __syncthreads();
  return scratch[32];
}

// Split cluster barrier.  A CTA arrives (relaxed) early, e.g. at kernel start,
// and waits just before its first access to a peer's shared memory, which is
// then known to be live; a release-arrive / acquire-wait pair publishes
// shared-memory stores to the peers.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace moe

namespace moe {

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA) primitives for shared-memory pipelines.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One probe of phase `parity`.  It carries no suspend-time hint: with a 1 us
// hint, waits on stage rings and exchanges came back measurably later (the
// tcgen05 router's stage ring: +1.4 us on a 128-CTA launch at T = 8192; the
// persistent tail at T = 512: +0.18 us; the decode layer: +0.05 us).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared::cluster address of `p` (this CTA's shared memory) in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// Store one float into a cluster peer's shared memory; the store counts 4
// bytes on that peer's mbarrier (both given as shared::cluster addresses), so
// the peer learns of it by waiting on its own barrier -- no cluster barrier.
__device__ __forceinline__ void st_async_f32(uint32_t remote, float v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote), "f"(v),
               "r"(remote_bar)
               : "memory");
}

// Probes of phase `parity` of `bar` until it completes; false after
// `max_probes` probes.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int max_probes) {
  for (int it = 0; it < max_probes; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Sum of one float per thread over the whole thread-block cluster, delivered
// by asynchronous remote stores: every warp sends its sum to slot
// [rank * nwarps + warp] of every CTA of the cluster, each store counted on
// the receiving CTA's barrier `bar` (initialised with count 1 and made
// visible to the cluster before the caller's first cluster_arrive_relaxed),
// and each thread adds the cluster size x nwarps slots in that fixed order
// once its own barrier has seen them all, so all CTAs get the same total, bit
// for bit.  A CTA leaves only after every store into its shared memory has
// landed.  Every thread of every CTA calls this once per launch; false (and
// an unspecified total) if the wait ran out.
__device__ __forceinline__ bool cluster_block_sum_async(float& v, float* slots, uint64_t* bar) {
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned n = cluster.num_blocks();
  const unsigned rank = cluster.block_rank();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n * nwarps * 4));
  cluster_wait_acquire();  // every peer has started: its shared memory and barrier are live
  if (static_cast<unsigned>(lane) < n)
    st_async_f32(cluster_addr(slots + rank * nwarps + warp, lane), v, cluster_addr(bar, lane));
  const bool ok = mbar_wait_bounded(bar, 0, 1 << 21);
  float s = 0.f;
  for (int i = 0; i < static_cast<int>(n) * nwarps; ++i) s += slots[i];
  v = s;
  return ok;
}

// L2 policy for data read exactly once (expert rows, activations).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) at `src` into the
// L2.  Only a hint -- later loads still observe every write made before them
// -- so it may be issued before grid_dependency_wait().
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// L2 prefetch hint for the whole 16-byte blocks inside the n floats at `row`
// (no byte outside the row is named).
__device__ __forceinline__ void prefetch_row_l2(const float* row, int n) {
  const uintptr_t b = (reinterpret_cast<uintptr_t>(row) + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t e = (reinterpret_cast<uintptr_t>(row + n)) & ~static_cast<uintptr_t>(15);
  if (e > b) prefetch_l2(reinterpret_cast<const void*>(b), static_cast<uint32_t>(e - b));
}

// Relaxed load used only to choose prefetch addresses before the dependency
// wait (the value may be stale; it is never used for results).
__device__ __forceinline__ int ld_relaxed_s32(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 lds16(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// Barrier among `nthreads` threads (a multiple of 32) on named barrier `id`.
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace moe
