// The fused MoE tail: finalize (top-k weighted gather through the expanded-
// index map) + shared add + row-parallel partial sum + residual add + RMSNorm,
// FP32 accumulation, one BF16 rounding per output (vllm-project/vllm pull
// 62174, Overview / Claims / Details; milou-sh/vllm pull 3, Ported behavior).
// The router-less variant first routes the token from its FP32 logits
// (moe_tail_fused) while the expert-row gathers are in flight.
//
// Work decomposition: one token row per thread-block cluster; the cluster's
// CTAs split the hidden dimension (split-H) so that small batches still cover
// the GPU, and add their sums of squares through distributed shared memory.
// Each thread owns VPT 16-byte vectors (8 BF16 each) of the row, spaced by the
// block size so that every load instruction of a warp covers 512 contiguous
// bytes.  The k expert rows of a token are gathered KB slots at a time, with
// all of a batch's loads issued before the first FMA.
#include "host_util.h"
#include "route.cuh"

namespace moe {

struct TailParams {
  const uint16_t* rows;
  int64_t n_rows;
  const int32_t* map;
  const float* topk_w;
  int k;
  const uint16_t* shared;
  const uint16_t* partials;
  int R;
  int64_t partial_stride;  // elements between consecutive partial buffers
  const uint16_t* residual;
  const float* gamma;
  float eps;
  uint16_t* residual_out;
  uint16_t* normed_out;
  int H;
  int32_t* err_flag;
  // routing (router-less fused tail only)
  const float* logits;
  int E;
  float scale;
  int32_t* ids_out;
  float* w_out;
};

constexpr int kMaxThreads = 256;  // per CTA; VPT <= 4 covers 1024 vectors (16 KB of a row)

template <int VPT, int KB, bool ROUTE>
__global__ void __launch_bounds__(kMaxThreads)
tail_kernel(const TailParams p) {
  __shared__ int map_s[MOE_MAX_K];
  __shared__ float w_s[MOE_MAX_K];
  __shared__ int id_s[MOE_MAX_K];
  __shared__ float red[33];
  __shared__ float cluster_slot;
  extern __shared__ float logit_s[];  // E floats when ROUTE

  const int t = blockIdx.y;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int cs = gridDim.x;        // CTAs per token (the cluster)
  const int rank = blockIdx.x;     // this CTA's slice of the hidden dimension
  const int nvec = p.H >> 3;
  const int per_cta = (nvec + cs - 1) / cs;
  const int vbeg = rank * per_cta;
  const int vend = min(nvec, vbeg + per_cta);
  const int64_t row_off = static_cast<int64_t>(t) * p.H;
  const int k = p.k;

  // -- slot table: map entries (checked) and, without routing, the weights
  if (tid < k) {
    int m = p.map[static_cast<int64_t>(t) * k + tid];
    if (m < 0 || static_cast<int64_t>(m) >= p.n_rows) {
      if (p.err_flag) atomicOr(p.err_flag, MOE_FLAG_BAD_INDEX);
      m = -1;  // never dereferenced; the row counts as zero
    }
    map_s[tid] = m;
    if (!ROUTE) w_s[tid] = p.topk_w[static_cast<int64_t>(t) * k + tid];
  }
  if (ROUTE) {
    const float* src = p.logits + static_cast<int64_t>(t) * p.E;
    for (int i = tid; i < p.E; i += nthr) logit_s[i] = src[i];
  }
  __syncthreads();

  int vidx[VPT];
  bool vok[VPT];
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    vidx[m] = vbeg + m * nthr + tid;
    vok[m] = vidx[m] < vend;
  }

  // -- shared expert and residual: issued first, consumed last
  uint4 sh[VPT], res[VPT];
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    const int64_t off = row_off + static_cast<int64_t>(vidx[m]) * 8;
    sh[m] = (p.shared && vok[m]) ? ld_stream16(p.shared + off) : make_uint4(0, 0, 0, 0);
    res[m] = vok[m] ? ld_stream16(p.residual + off) : make_uint4(0, 0, 0, 0);
  }

  float acc[VPT][8];
#pragma unroll
  for (int m = 0; m < VPT; ++m)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[m][e] = 0.f;

  // -- top-k weighted sum, KB slots per batch, slots in ascending order
  for (int jb = 0; jb < k; jb += KB) {
    uint4 rv[KB][VPT];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int slot = jb + j;
      const int row = slot < k ? map_s[slot] : -1;
#pragma unroll
      for (int m = 0; m < VPT; ++m) {
        rv[j][m] = (row >= 0 && vok[m])
                       ? ld_stream16(p.rows + static_cast<int64_t>(row) * p.H + static_cast<int64_t>(vidx[m]) * 8)
                       : make_uint4(0, 0, 0, 0);
      }
    }
    if (ROUTE && jb == 0) {
      // route the token while the first batch of rows is in flight
      if (tid < 32) warp_route(logit_s, p.E, k, p.scale, id_s, w_s);
      __syncthreads();
      if (rank == 0 && tid < k) {
        const int64_t o = static_cast<int64_t>(t) * k + tid;
        if (p.ids_out) p.ids_out[o] = id_s[tid];
        if (p.w_out) p.w_out[o] = w_s[tid];
      }
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int slot = jb + j;
      if (slot < k) {
        const float w = w_s[slot];
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
          float f[8];
          unpack8(rv[j][m], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[m][e] = fmaf(w, f[e], acc[m][e]);
        }
      }
    }
  }

  // -- shared expert
  if (p.shared) {
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
      float f[8];
      unpack8(sh[m], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[m][e] += f[e];
    }
  }

  // -- row-parallel partials, r ascending
  for (int rb = 0; rb < p.R; rb += KB) {
    uint4 pv[KB][VPT];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
#pragma unroll
      for (int m = 0; m < VPT; ++m) {
        pv[j][m] = (rb + j < p.R && vok[m])
                       ? ld_stream16(p.partials + static_cast<int64_t>(rb + j) * p.partial_stride + row_off +
                                     static_cast<int64_t>(vidx[m]) * 8)
                       : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      if (rb + j < p.R) {
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
          float f[8];
          unpack8(pv[j][m], f);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[m][e] += f[e];
        }
      }
    }
  }

  // -- residual add, residual_out, sum of squares
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    float f[8];
    unpack8(res[m], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[m][e] = f[e] + acc[m][e];
      ss = fmaf(acc[m][e], acc[m][e], ss);
    }
    if (vok[m]) {
      uint4 o;
      o.x = pack_bf16x2(acc[m][0], acc[m][1]);
      o.y = pack_bf16x2(acc[m][2], acc[m][3]);
      o.z = pack_bf16x2(acc[m][4], acc[m][5]);
      o.w = pack_bf16x2(acc[m][6], acc[m][7]);
      st16(p.residual_out + row_off + static_cast<int64_t>(vidx[m]) * 8, o);
    }
  }

  ss = block_sum(ss, red);
  if (cs > 1) ss = cluster_sum(ss, &cluster_slot);
  const float inv = rsqrtf(ss / static_cast<float>(p.H) + p.eps);

  // -- RMSNorm output
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    if (!vok[m]) continue;
    const float4* g4 = reinterpret_cast<const float4*>(p.gamma + static_cast<int64_t>(vidx[m]) * 8);
    const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1);
    uint4 o;
    o.x = pack_bf16x2(acc[m][0] * inv * g0.x, acc[m][1] * inv * g0.y);
    o.y = pack_bf16x2(acc[m][2] * inv * g0.z, acc[m][3] * inv * g0.w);
    o.z = pack_bf16x2(acc[m][4] * inv * g1.x, acc[m][5] * inv * g1.y);
    o.w = pack_bf16x2(acc[m][6] * inv * g1.z, acc[m][7] * inv * g1.w);
    st16(p.normed_out + row_off + static_cast<int64_t>(vidx[m]) * 8, o);
  }
}

// ---------------------------------------------------------------------------
// Launch configuration: a deterministic function of (T, H, SM count).
// ---------------------------------------------------------------------------

struct TailLaunch {
  int cs;    // CTAs per token (cluster size)
  int vpt;   // 16-byte vectors per thread
  int threads;
};

static TailLaunch choose_tail_launch(int64_t T, int H, int nsm) {
  const int nvec = H / 8;
  // a CTA holds at most 4 * kMaxThreads vectors of the row
  int cs = 1;
  while (cs * 4 * kMaxThreads < nvec) cs *= 2;
  // split the row further while the grid would leave SMs idle and each CTA
  // still gets at least 64 vectors (1 KB of a row)
  while (cs < 8 && T * cs < nsm && (nvec + 2 * cs - 1) / (2 * cs) >= 64) cs *= 2;
  const int per_cta = (nvec + cs - 1) / cs;
  int vpt = (per_cta + kMaxThreads - 1) / kMaxThreads;
  if (vpt < 1) vpt = 1;
  int threads = (per_cta + vpt - 1) / vpt;
  threads = (threads + 31) / 32 * 32;
  return {cs, vpt, threads};
}

template <int VPT, bool ROUTE>
static cudaError_t launch_tail_v(const TailParams& p, int T, const TailLaunch& L, size_t smem,
                                 cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.cs, T, 1);
  cfg.blockDim = dim3(L.threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int nattr = 0;
  if (L.cs > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = L.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    nattr = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, tail_kernel<VPT, 8, ROUTE>, p);
}

template <bool ROUTE>
static int launch_tail(TailParams p, int64_t T, cudaStream_t stream) {
  const int nsm = sm_count();
  const size_t smem = ROUTE ? sizeof(float) * static_cast<size_t>(p.E) : 0;
  for (int64_t t0 = 0; t0 < T; t0 += kMaxGridY) {
    const int Tc = static_cast<int>(T - t0 < kMaxGridY ? T - t0 : kMaxGridY);
    TailParams q = p;
    const int64_t off = t0 * p.H;
    q.residual += off;
    q.residual_out += off;
    q.normed_out += off;
    if (q.shared) q.shared += off;
    if (q.partials) q.partials += off;
    if (q.map) q.map += t0 * p.k;
    if (q.topk_w) q.topk_w += t0 * p.k;
    if (q.logits) q.logits += t0 * p.E;
    if (q.ids_out) q.ids_out += t0 * p.k;
    if (q.w_out) q.w_out += t0 * p.k;
    const TailLaunch L = choose_tail_launch(T, p.H, nsm);
    cudaError_t e;
    switch (L.vpt) {
      case 1: e = launch_tail_v<1, ROUTE>(q, Tc, L, smem, stream); break;
      case 2: e = launch_tail_v<2, ROUTE>(q, Tc, L, smem, stream); break;
      case 3: e = launch_tail_v<3, ROUTE>(q, Tc, L, smem, stream); break;
      default: e = launch_tail_v<4, ROUTE>(q, Tc, L, smem, stream); break;
    }
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    const int st = launch_status();
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

// Checks common to both tail entry points.
static int check_tail_common(const void* rows, int64_t n_rows, const int32_t* map, int32_t k,
                             const void* shared, const void* residual, const float* gamma, float eps,
                             const void* residual_out, const void* normed_out, int64_t T, int64_t H) {
  if (T < 0 || H < 8 || n_rows < 0 || k < 0 || k > MOE_MAX_K || !(eps >= 0.f) || !isfinite(eps))
    return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > 65536) return MOE_ERR_UNSUPPORTED;  // <= 8 CTAs x 1024 vectors
  if (T > 0) {
    if (!residual || !gamma || !residual_out || !normed_out) return MOE_ERR_INVALID_ARG;
    if (k > 0 && (!rows || !map)) return MOE_ERR_INVALID_ARG;
    if (!aligned(residual, 16) || !aligned(gamma, 16) || !aligned(residual_out, 16) ||
        !aligned(normed_out, 16) || (shared && !aligned(shared, 16)) || (rows && !aligned(rows, 16)) ||
        (map && !aligned(map, 4)))
      return MOE_ERR_MISALIGNED;
  }
  return MOE_OK;
}

}  // namespace moe

extern "C" int moe_finalize_add_rmsnorm(const void* rows_bf16, int64_t n_rows, const int32_t* map,
                                        const float* topk_w, int32_t k, const void* shared_bf16,
                                        const void* partials_bf16, int32_t R, const void* residual_bf16,
                                        const float* gamma, float eps, void* residual_out_bf16,
                                        void* normed_out_bf16, int64_t T, int64_t H, int32_t* err_flag,
                                        cudaStream_t stream) {
  using namespace moe;
  int st = check_tail_common(rows_bf16, n_rows, map, k, shared_bf16, residual_bf16, gamma, eps,
                             residual_out_bf16, normed_out_bf16, T, H);
  if (st != MOE_OK) return st;
  if (R < 0 || R > MOE_MAX_R) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (k > 0 && !topk_w) return MOE_ERR_INVALID_ARG;
  if (R > 0 && !partials_bf16) return MOE_ERR_INVALID_ARG;
  if ((topk_w && !aligned(topk_w, 4)) || (R > 0 && !aligned(partials_bf16, 16))) return MOE_ERR_MISALIGNED;
  TailParams p = {};
  p.rows = static_cast<const uint16_t*>(rows_bf16);
  p.n_rows = n_rows;
  p.map = map;
  p.topk_w = topk_w;
  p.k = k;
  p.shared = static_cast<const uint16_t*>(shared_bf16);
  p.partials = R > 0 ? static_cast<const uint16_t*>(partials_bf16) : nullptr;
  p.R = R;
  p.partial_stride = T * H;
  p.residual = static_cast<const uint16_t*>(residual_bf16);
  p.gamma = gamma;
  p.eps = eps;
  p.residual_out = static_cast<uint16_t*>(residual_out_bf16);
  p.normed_out = static_cast<uint16_t*>(normed_out_bf16);
  p.H = static_cast<int>(H);
  p.err_flag = err_flag;
  return launch_tail<false>(p, T, stream);
}

extern "C" int moe_tail_fused(const float* logits, int64_t E, int32_t k, float routed_scale,
                              const void* rows_bf16, int64_t n_rows, const int32_t* map,
                              const void* shared_bf16, const void* residual_bf16, const float* gamma,
                              float eps, void* residual_out_bf16, void* normed_out_bf16,
                              int32_t* topk_ids_out, float* topk_w_out, int64_t T, int64_t H,
                              int32_t* err_flag, cudaStream_t stream) {
  using namespace moe;
  if (E < 1 || k < 1 || k > E || !isfinite(routed_scale)) return MOE_ERR_INVALID_ARG;
  if (E > MOE_MAX_E) return MOE_ERR_UNSUPPORTED;
  int st = check_tail_common(rows_bf16, n_rows, map, k, shared_bf16, residual_bf16, gamma, eps,
                             residual_out_bf16, normed_out_bf16, T, H);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!logits) return MOE_ERR_INVALID_ARG;
  if (!aligned(logits, 4) || (topk_ids_out && !aligned(topk_ids_out, 4)) ||
      (topk_w_out && !aligned(topk_w_out, 4)))
    return MOE_ERR_MISALIGNED;
  TailParams p = {};
  p.rows = static_cast<const uint16_t*>(rows_bf16);
  p.n_rows = n_rows;
  p.map = map;
  p.k = k;
  p.shared = static_cast<const uint16_t*>(shared_bf16);
  p.residual = static_cast<const uint16_t*>(residual_bf16);
  p.gamma = gamma;
  p.eps = eps;
  p.residual_out = static_cast<uint16_t*>(residual_out_bf16);
  p.normed_out = static_cast<uint16_t*>(normed_out_bf16);
  p.H = static_cast<int>(H);
  p.err_flag = err_flag;
  p.logits = logits;
  p.E = static_cast<int>(E);
  p.scale = routed_scale;
  p.ids_out = topk_ids_out;
  p.w_out = topk_w_out;
  return launch_tail<true>(p, T, stream);
}
