// moe_router_logits_fp32: logits[T, E] = x[T, H] . W[E, H]^T with BF16 inputs,
// FP32 accumulation and FP32 output (lmdeploy pull 4853, Summary; the
// small-token router GEMM).
//
// At decode sizes (T <= 64) the 3 MB gate weight is the whole cost, so the
// kernel is organised to stream W once across as many SMs as possible:
//  - a CTA owns 16*MT experts x 8*NT tokens and a slice of the hidden
//    dimension; its warps split that slice again.  Up to 32 tokens: 32-expert
//    tiles of 8 or 16 tokens (half as many CTAs, each gate-weight fragment
//    staged once per CTA); up to 64 tokens: 16-expert x 16-token tiles;
//  - the first round of each lane's gate-weight fragments is copied into
//    shared memory (cp.async) before the dependency wait: W is a model
//    parameter, so only x waits for the previous kernel;
//  - the CTAs that share an (expert, token) tile form a thread-block cluster
//    (split-K over H) and add their partial tiles through distributed shared
//    memory (remote stores counted on the owner's mbarrier) in ascending rank
//    order -- deterministic, no atomics, no global scratch;
//  - each lane loads 16 contiguous bytes of a W row and of an x row per
//    32-wide chunk of H and feeds them straight from registers into
//    mma.m16n8k16 (W rows as the M side, tokens as the N side).  Within a
//    chunk, hidden index h = 32c + 8q + 4s + {0,1,2,3} plays the role of
//    k-index {2q, 2q+1, 2q+8, 2q+9} of k-step s on both operands, so each
//    product W[e,h] * x[t,h] still meets its own pair: only the summation
//    order inside the tensor core changes.
#include "host_util.h"
#include "common.cuh"
#include "router_tc.h"

namespace moe {

constexpr size_t kRouterStaticSmem = 48 * 1024;  // larger router CTAs take dynamic shared memory



__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Partial tiles are kept in accumulator-fragment order: element
// i = ((mt * NT + nt) * 4 + reg) * 32 + lane holds expert 16 mt + g +
// 8 (reg >> 1) and token 8 nt + 2 q + (reg & 1) of the tile (g = lane / 4,
// q = lane % 4), so that every shared-memory access below is conflict-free.
template <int NT, int MT>
__device__ __forceinline__ void frag_to_tile(int i, int& e, int& t) {
  const int lane = i & 31, reg = (i >> 5) & 3, f = i >> 7;
  const int nt = f % NT, mt = f / NT;
  e = 16 * mt + (lane >> 2) + 8 * (reg >> 1);
  t = 8 * nt + 2 * (lane & 3) + (reg & 1);
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); `full`
// false copies nothing and zero-fills the 16 bytes.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool full) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Shared memory of one router CTA (16 MT experts x 8 NT tokens, WARPS warps,
// U 32-wide chunks of H per warp and round).
template <int NT, int WARPS, int MT, int U>
struct RouterSmem {
  static constexpr int kTile = 16 * MT * 8 * NT;  // outputs per tile
  // each lane's gate-weight fragments of its warp's first round, staged before
  // the dependency wait (every thread reads back only its own slots)
  uint4 w_stage[WARPS][U][MT][2][32];
  float red[WARPS][kTile];
  float part[kTile];  // split-K: part[src * per + i] = rank src's partial of output ib + i
  uint64_t xbar;      // split-K: completes when every CTA's partials of this CTA's outputs have landed
};

template <int NT, int WARPS, int MT, int U>
__device__ __forceinline__ void router_body(RouterSmem<NT, WARPS, MT, U>& sm, const uint16_t* __restrict__ x,
                                            const uint16_t* __restrict__ W, float* __restrict__ logits, int T,
                                            int H, int E) {
  constexpr int TILE = RouterSmem<NT, WARPS, MT, U>::kTile;
  constexpr int kRouterUnroll = U;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * 16 * MT, t0 = blockIdx.y * 8 * NT;
  const int S = gridDim.z, z = blockIdx.z;
  const int C = (H + 31) >> 5;
  const int cb = static_cast<int>(static_cast<int64_t>(C) * z / S);
  const int ce = static_cast<int>(static_cast<int64_t>(C) * (z + 1) / S);
  const int wb = cb + (ce - cb) * warp / WARPS;
  const int we = cb + (ce - cb) * (warp + 1) / WARPS;

  if (S > 1) {
    if (tid == 0) {
      mbar_init(&sm.xbar, 1);
      mbar_init_fence();  // visible to the cluster's remote stores after the cluster barrier
    }
    cluster_arrive_relaxed();
  }
  allow_dependent_launch();
  // While the previous kernel finishes: L2 prefetch of this CTA's slice of
  // the gate weight and, from the first expert tile, of the token rows of x
  // (hints; the loads below follow the dependency wait and see the final data
  // whatever the hint fetched).
  if (ce > cb) {
    const int h0 = cb * 32, h1 = min(H, ce * 32);
    if (tid < 16 * MT && e0 + tid < E)
      prefetch_l2(W + static_cast<int64_t>(e0 + tid) * H + h0, static_cast<uint32_t>((h1 - h0) * 2));
    else if (blockIdx.x == 0 && tid >= 32 * MT && tid < 32 * MT + 8 * NT && t0 + tid - 32 * MT < T)
      prefetch_l2(x + static_cast<int64_t>(t0 + tid - 32 * MT) * H + h0, static_cast<uint32_t>((h1 - h0) * 2));
  }
  // this lane's gate-weight rows: expert 16 mt + g (A) and 16 mt + g + 8 (B)
  const uint16_t* pw[MT][2];
  bool okw[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = e0 + 16 * mt + g + 8 * h;
      okw[mt][h] = e < E;
      pw[mt][h] = W + static_cast<int64_t>(okw[mt][h] ? e : 0) * H + 8 * q;
    }
  // The gate weight is a model parameter that no kernel still running on the
  // stream writes, so its first round is copied into shared memory while the
  // previous kernel finishes; only x is read after the dependency wait.
  // Fragments outside W are zero-filled (the dummy source W is never read).
#pragma unroll
  for (int u = 0; u < kRouterUnroll; ++u) {
    const int cc = wb + u;
    const bool ok = cc < we && (cc * 32 + 8 * q) < H;
    const int64_t off = static_cast<int64_t>(cc) * 32;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        cp_async16(&sm.w_stage[warp][u][mt][h][lane],
                   (ok && okw[mt][h]) ? static_cast<const void*>(pw[mt][h] + off) : W, ok && okw[mt][h]);
  }
  cp_async_commit();
  grid_dependency_wait();
  const uint16_t* px[NT];
  bool okx[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tt = t0 + 8 * nt + g;
    okx[nt] = tt < T;
    px[nt] = x + static_cast<int64_t>(okx[nt] ? tt : 0) * H + 8 * q;
  }

  float acc[MT][NT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;

  const uint4 zero = make_uint4(0, 0, 0, 0);
  // one round: kRouterUnroll 32-wide chunks of H starting at chunk c
  auto load_x = [&](int c, uint4 (&b)[kRouterUnroll][NT]) {
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
      const int cc = c + u;
      const bool ok = cc < we && (cc * 32 + 8 * q) < H;
      const int64_t off = static_cast<int64_t>(cc) * 32;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) b[u][nt] = (ok && okx[nt]) ? ld_keep16(px[nt] + off) : zero;
    }
  };
  auto mma_chunk = [&](int mt, const uint4& a0, const uint4& a1, const uint4 (&b)[NT]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_bf16_16816(acc[mt][nt], a0.x, a1.x, a0.y, a1.y, b[nt].x, b[nt].y);
      mma_bf16_16816(acc[mt][nt], a0.z, a1.z, a0.w, a1.w, b[nt].z, b[nt].w);
    }
  };
  {  // first round: the gate weight from the fragments staged before the wait
    uint4 b[kRouterUnroll][NT];
    load_x(wb, b);
    cp_async_wait_all();  // this thread's own staged fragments
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        mma_chunk(mt, sm.w_stage[warp][u][mt][0][lane], sm.w_stage[warp][u][mt][1][lane], b[u]);
  }
  for (int c = wb + kRouterUnroll; c < we; c += kRouterUnroll) {
    uint4 a[kRouterUnroll][MT][2], b[kRouterUnroll][NT];
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
      const int cc = c + u;
      const bool ok = cc < we && (cc * 32 + 8 * q) < H;
      const int64_t off = static_cast<int64_t>(cc) * 32;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) a[u][mt][h] = (ok && okw[mt][h]) ? ld_stream16(pw[mt][h] + off) : zero;
    }
    load_x(c, b);
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) mma_chunk(mt, a[u][mt][0], a[u][mt][1], b[u]);
  }

#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) sm.red[warp][((mt * NT + nt) * 4 + r) * 32 + lane] = acc[mt][nt][r];
  __syncthreads();
  if (S == 1) {
    for (int i = tid; i < TILE; i += WARPS * 32) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < WARPS; ++w) s += sm.red[w][i];
      int e, t;
      frag_to_tile<NT, MT>(i, e, t);
      if (e0 + e < E && t0 + t < T) logits[static_cast<int64_t>(t0 + t) * E + e0 + e] = s;
    }
    return;
  }
  // split-K over the cluster: rank r owns outputs [r * per, (r + 1) * per); every
  // CTA sends its partial of those outputs into the owner's part[] by remote
  // stores counted on the owner's barrier, then the owner adds the S partials
  // in rank order.  A CTA leaves only after every store into its shared
  // memory has landed; if that wait ran out, its logits are written as NaN.
  cg::cluster_group cluster = cg::this_cluster();
  const int me = static_cast<int>(cluster.block_rank());
  const int per = TILE / S;  // S (a power of two <= 8) divides TILE
  if (tid == 0) mbar_arrive_expect_tx(&sm.xbar, static_cast<uint32_t>(TILE * 4));  // S peers x per floats
  cluster_wait_acquire();  // every peer has started: its shared memory and barrier are live
  for (int i = tid; i < TILE; i += WARPS * 32) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) s += sm.red[w][i];
    const int owner = i / per;
    st_async_f32(cluster_addr(sm.part + me * per + (i - owner * per), owner), s, cluster_addr(&sm.xbar, owner));
  }
  const bool ok = mbar_wait_bounded(&sm.xbar, 0, 1 << 21);
  const int ib = me * per, ie = ib + per;
  for (int i = ib + tid; i < ie; i += WARPS * 32) {
    float s = 0.f;
    for (int r = 0; r < S; ++r) s += sm.part[r * per + (i - ib)];
    int e, t;
    frag_to_tile<NT, MT>(i, e, t);
    if (e0 + e < E && t0 + t < T)
      logits[static_cast<int64_t>(t0 + t) * E + e0 + e] = ok ? s : __int_as_float(0x7FC00000);
  }
}

// The kernel: shared memory declared statically where it fits in 48 KB, else
// taken from the dynamic allocation (opted in at launch).
template <int NT, int WARPS, int MT, int U>
__global__ void __launch_bounds__(WARPS * 32, (WARPS == 8 && MT == 1) ? 4 : 1)  // 16-token tiles: 4 CTAs an SM
router_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ W, float* __restrict__ logits,
              int T, int H, int E) {
  using Smem = RouterSmem<NT, WARPS, MT, U>;
  if constexpr (sizeof(Smem) <= kRouterStaticSmem) {
    __shared__ Smem sm;
    router_body<NT, WARPS, MT, U>(sm, x, W, logits, T, H, E);
  } else {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    router_body<NT, WARPS, MT, U>(*reinterpret_cast<Smem*>(smem_raw), x, W, logits, T, H, E);
  }
}

// Decode sizes (T <= 64): tiles of 8 or 16 tokens and 16 MT experts, 8 warps
// splitting each CTA's slice of H so that every warp loads its share in one
// round, and a cluster of up to 8 CTAs along H.  Larger T (only with H < 64):
// 32-token tiles, 4 warps.
template <int NT, int WARPS, int MT, int U>
static cudaError_t launch_router(const uint16_t* x, const uint16_t* W, float* logits, int T, int H, int E,
                                 int nsm, cudaStream_t stream) {
  using Smem = RouterSmem<NT, WARPS, MT, U>;
  constexpr bool kDynamic = sizeof(Smem) > kRouterStaticSmem;
  static bool smem_opt_in[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (kDynamic && dev >= 0 && dev < 64 && !smem_opt_in[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(router_kernel<NT, WARPS, MT, U>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(sizeof(Smem)));
    if (e != cudaSuccess) return e;
    smem_opt_in[dev] = true;
  }
  const int t_tiles = (T + 8 * NT - 1) / (8 * NT);
  const int e_tiles = (E + 16 * MT - 1) / (16 * MT);
  const int C = (H + 31) / 32;
  int S = 1;
  // split H over a cluster until the grid covers every SM four times (or each
  // warp would get fewer than one 32-wide chunk per slice)
  while (S < 8 && static_cast<int64_t>(e_tiles) * t_tiles * S < 4 * nsm && C / (2 * S) >= WARPS) S *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(e_tiles, t_tiles, S);
  cfg.blockDim = dim3(WARPS * 32, 1, 1);
  cfg.dynamicSmemBytes = launch_smem(kDynamic ? sizeof(Smem) : 0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0] = pdl_attribute();
  cfg.numAttrs = 1;
  if (S > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = S;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, router_kernel<NT, WARPS, MT, U>, x, W, logits, T, H, E);
}

}  // namespace moe

// err_flag is raised by the tensor-memory kernel (T > 64); the decode-size
// kernel marks a timed-out split-K exchange in its logits (NaN) only: a flag
// store there, even one never executed, cost the decode layer about 0.05 us.
extern "C" int moe_router_logits_fp32(const void* x_bf16, const void* w_gate_bf16, float* logits_out,
                                      int64_t T, int64_t H, int64_t E, int32_t* err_flag, cudaStream_t stream) {
  using namespace moe;
  if (T < 0 || H < 8 || E < 1) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || E > MOE_MAX_E || H > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !w_gate_bf16 || !logits_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(w_gate_bf16, 16) || !aligned(logits_out, 4) || (err_flag && !aligned(err_flag, 4)))
    return MOE_ERR_MISALIGNED;
  const int nsm = sm_count();
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  const uint16_t* W = static_cast<const uint16_t*>(w_gate_bf16);
  if (router_tc_supported(T, H)) {
    // prefill sizes: the tensor-memory kernel, in launches of up to 2^30 tokens
    const int64_t per = static_cast<int64_t>(1) << 30;
    for (int64_t t0 = 0; t0 < T; t0 += per) {
      const int Tc = static_cast<int>(T - t0 < per ? T - t0 : per);
      const cudaError_t e = launch_router_tc(x + t0 * H, W, logits_out + t0 * E, Tc, static_cast<int>(H),
                                             static_cast<int>(E), err_flag, nsm, stream);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      const int st = launch_status();
      if (st != MOE_OK) return st;
    }
    return MOE_OK;
  }
  // decode sizes: 8- or 16-token tiles; more CTAs in flight beat reusing x
  // across a wider tile (measured at T = 64: 16-token tiles 5.3 us, 64-token 7.9 us).
  // Larger batches come here only with H < 64 (32-token tiles).
  const int NT = T <= 8 ? 1 : (T <= 64 ? 2 : 4);
  const int64_t per_launch = static_cast<int64_t>(kMaxGridY) * 8 * NT;
  for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
    const int Tc = static_cast<int>(T - t0 < per_launch ? T - t0 : per_launch);
    const uint16_t* xc = x + t0 * H;
    float* lc = logits_out + t0 * E;
    const int Hi = static_cast<int>(H), Ei = static_cast<int>(E);
    cudaError_t e;
    if (T > 64) e = launch_router<4, 4, 1, 4>(xc, W, lc, Tc, Hi, Ei, nsm, stream);
    else if (NT == 1) e = launch_router<1, 8, 2, 3>(xc, W, lc, Tc, Hi, Ei, nsm, stream);
    else if (T <= 32) e = launch_router<2, 8, 2, 3>(xc, W, lc, Tc, Hi, Ei, nsm, stream);
    else e = launch_router<2, 8, 1, 4>(xc, W, lc, Tc, Hi, Ei, nsm, stream);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    const int st = launch_status();
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}
