// moe_router_logits_fp32: logits[T, E] = x[T, H] . W[E, H]^T with BF16 inputs,
// FP32 accumulation and FP32 output (lmdeploy pull 4853, Summary; the
// small-token router GEMM).
//
// At decode sizes (T <= 64) the 3 MB gate weight is the whole cost, so the
// kernel is organised to stream W once across as many SMs as possible:
//  - a CTA owns 16 experts x (8*NT) tokens and a slice of the hidden dimension;
//    its warps split that slice again;
//  - the CTAs that share an (expert, token) tile form a thread-block cluster
//    (split-K over H) and add their partial tiles through distributed shared
//    memory in ascending rank order -- deterministic, no atomics, no global
//    scratch;
//  - each lane loads 16 contiguous bytes of a W row and of an x row per
//    32-wide chunk of H and feeds them straight from registers into
//    mma.m16n8k16 (W rows as the M side, tokens as the N side).  Within a
//    chunk, hidden index h = 32c + 8q + 4s + {0,1,2,3} plays the role of
//    k-index {2q, 2q+1, 2q+8, 2q+9} of k-step s on both operands, so each
//    product W[e,h] * x[t,h] still meets its own pair: only the summation
//    order inside the tensor core changes.
#include "host_util.h"
#include "common.cuh"

namespace moe {

constexpr int kRouterWarps = 4;
constexpr int kRouterUnroll = 4;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NT>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ W, float* __restrict__ logits,
              int T, int H, int E) {
  constexpr int BT = 8 * NT;  // tokens per tile
  __shared__ float red[kRouterWarps][16][BT];
  __shared__ float part[16 * BT];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * 16, t0 = blockIdx.y * BT;
  const int S = gridDim.z, z = blockIdx.z;
  const int C = (H + 31) >> 5;
  const int cb = static_cast<int>(static_cast<int64_t>(C) * z / S);
  const int ce = static_cast<int>(static_cast<int64_t>(C) * (z + 1) / S);
  const int wb = cb + (ce - cb) * warp / kRouterWarps;
  const int we = cb + (ce - cb) * (warp + 1) / kRouterWarps;

  const int eA = e0 + g, eB = e0 + g + 8;
  const bool okA = eA < E, okB = eB < E;
  const uint16_t* pA = W + static_cast<int64_t>(okA ? eA : 0) * H + 8 * q;
  const uint16_t* pB = W + static_cast<int64_t>(okB ? eB : 0) * H + 8 * q;
  const uint16_t* px[NT];
  bool okx[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tt = t0 + 8 * nt + g;
    okx[nt] = tt < T;
    px[nt] = x + static_cast<int64_t>(okx[nt] ? tt : 0) * H + 8 * q;
  }

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int c = wb; c < we; c += kRouterUnroll) {
    uint4 a[kRouterUnroll][2], b[kRouterUnroll][NT];
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
      const int cc = c + u;
      const bool ok = cc < we && (cc * 32 + 8 * q) < H;
      const int64_t off = static_cast<int64_t>(cc) * 32;
      a[u][0] = (ok && okA) ? ld_stream16(pA + off) : zero;
      a[u][1] = (ok && okB) ? ld_stream16(pB + off) : zero;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) b[u][nt] = (ok && okx[nt]) ? ld_keep16(px[nt] + off) : zero;
    }
#pragma unroll
    for (int u = 0; u < kRouterUnroll; ++u) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_bf16_16816(acc[nt], a[u][0].x, a[u][1].x, a[u][0].y, a[u][1].y, b[u][nt].x, b[u][nt].y);
        mma_bf16_16816(acc[nt], a[u][0].z, a[u][1].z, a[u][0].w, a[u][1].w, b[u][nt].z, b[u][nt].w);
      }
    }
  }

  // accumulator layout: d0,d1 -> (expert g, tokens 2q, 2q+1); d2,d3 -> expert g+8
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][g][8 * nt + 2 * q] = acc[nt][0];
    red[warp][g][8 * nt + 2 * q + 1] = acc[nt][1];
    red[warp][g + 8][8 * nt + 2 * q] = acc[nt][2];
    red[warp][g + 8][8 * nt + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  // output index i = token * 16 + expert: consecutive threads write consecutive experts
  for (int i = tid; i < 16 * BT; i += kRouterWarps * 32) {
    const int e = i & 15, t = i >> 4;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kRouterWarps; ++w) s += red[w][e][t];
    part[i] = s;
  }
  if (S == 1) {
    __syncthreads();
    for (int i = tid; i < 16 * BT; i += kRouterWarps * 32) {
      const int e = e0 + (i & 15), t = t0 + (i >> 4);
      if (e < E && t < T) logits[static_cast<int64_t>(t) * E + e] = part[i];
    }
    return;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int per = (16 * BT + S - 1) / S;
  const int ib = z * per, ie = min(16 * BT, ib + per);
  for (int i = ib + tid; i < ie; i += kRouterWarps * 32) {
    float s = 0.f;
    for (int r = 0; r < S; ++r) s += cluster.map_shared_rank(part, r)[i];
    const int e = e0 + (i & 15), t = t0 + (i >> 4);
    if (e < E && t < T) logits[static_cast<int64_t>(t) * E + e] = s;
  }
  cluster.sync();  // keep this CTA's partial tile alive until every peer has read it
}

template <int NT>
static cudaError_t launch_router(const uint16_t* x, const uint16_t* W, float* logits, int T, int H, int E,
                                 int nsm, cudaStream_t stream) {
  constexpr int BT = 8 * NT;
  const int t_tiles = (T + BT - 1) / BT;
  const int e_tiles = (E + 15) / 16;
  const int C = (H + 31) / 32;
  int S = 1;
  while (S < 8 && static_cast<int64_t>(e_tiles) * t_tiles * S < nsm && C / (2 * S) >= kRouterWarps) S *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(e_tiles, t_tiles, S);
  cfg.blockDim = dim3(kRouterWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (S > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = S;
    cfg.numAttrs = 1;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, router_kernel<NT>, x, W, logits, T, H, E);
}

}  // namespace moe

extern "C" int moe_router_logits_fp32(const void* x_bf16, const void* w_gate_bf16, float* logits_out,
                                      int64_t T, int64_t H, int64_t E, cudaStream_t stream) {
  using namespace moe;
  if (T < 0 || H < 8 || E < 1) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || E > MOE_MAX_E || H > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x_bf16 || !w_gate_bf16 || !logits_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(w_gate_bf16, 16) || !aligned(logits_out, 4)) return MOE_ERR_MISALIGNED;
  const int nsm = sm_count();
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  const uint16_t* W = static_cast<const uint16_t*>(w_gate_bf16);
  const int NT = T <= 8 ? 1 : (T <= 16 ? 2 : 4);
  const int64_t per_launch = static_cast<int64_t>(kMaxGridY) * 8 * NT;
  for (int64_t t0 = 0; t0 < T; t0 += per_launch) {
    const int Tc = static_cast<int>(T - t0 < per_launch ? T - t0 : per_launch);
    const uint16_t* xc = x + t0 * H;
    float* lc = logits_out + t0 * E;
    cudaError_t e;
    if (NT == 1)
      e = launch_router<1>(xc, W, lc, Tc, static_cast<int>(H), static_cast<int>(E), nsm, stream);
    else if (NT == 2)
      e = launch_router<2>(xc, W, lc, Tc, static_cast<int>(H), static_cast<int>(E), nsm, stream);
    else
      e = launch_router<4>(xc, W, lc, Tc, static_cast<int>(H), static_cast<int>(E), nsm, stream);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    const int st = launch_status();
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}
