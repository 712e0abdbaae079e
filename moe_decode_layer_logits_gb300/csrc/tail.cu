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
#include <atomic>

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

// EPL > 0: route the token from its logits first (E <= 32 * EPL).
template <int VPT, int KB, int EPL>
__global__ void __launch_bounds__(kMaxThreads)
tail_kernel(const TailParams p) {
  constexpr bool ROUTE = EPL > 0;
  __shared__ int map_s[MOE_MAX_K];
  __shared__ float w_s[MOE_MAX_K];
  __shared__ float red[33];
  __shared__ float cluster_slots[8 * (kMaxThreads / 32)];  // [cluster rank][warp]
  __shared__ uint64_t ss_bar;  // split rows: completes when every CTA's warp sums have landed
  __shared__ __align__(16) uint64_t route_scr[EPL > 0 ? kRouteScratch : 1];  // the routing warp's candidate list

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

  if (cs > 1) {
    if (tid == 0) {
      mbar_init(&ss_bar, 1);
      mbar_init_fence();  // visible to the cluster's remote stores after the cluster barrier below
    }
    cluster_arrive_relaxed();
  }
  allow_dependent_launch();
  // While the previous kernel finishes: L2 prefetch of this CTA's slice of the
  // token's rows (hints only; the loads below come after the dependency wait
  // and see the final data whatever the prefetch fetched).
  {
    const int64_t sb = static_cast<int64_t>(vbeg) * 8, slen = static_cast<int64_t>(vend - vbeg) * 16;
    if (slen > 0) {
      if (tid == 0) prefetch_l2(p.residual + row_off + sb, static_cast<uint32_t>(slen));
      if (tid == 1 && p.shared) prefetch_l2(p.shared + row_off + sb, static_cast<uint32_t>(slen));
      if (tid == 2) prefetch_l2(p.gamma + sb, static_cast<uint32_t>(slen * 2));
      if (tid >= 32 && tid < 32 + k) {
        const int m = ld_relaxed_s32(p.map + static_cast<int64_t>(t) * k + (tid - 32));
        if (m >= 0 && static_cast<int64_t>(m) < p.n_rows)
          prefetch_l2(p.rows + static_cast<int64_t>(m) * p.H + sb, static_cast<uint32_t>(slen));
      }
    }
  }
  grid_dependency_wait();

  // router-less variant: warp 0 requests the token's logits first (the
  // selection waits for them, and it overlaps the expert-row gathers)
  constexpr int KEYS = EPL > 0 ? EPL : 1;
  uint32_t keys[KEYS];
  if (ROUTE && tid < 32) route_load_keys<KEYS>(p.logits + static_cast<int64_t>(t) * p.E, p.E, keys);

  // then the slot table's loads (every row gather waits for them), pinned
  // here and consumed at the slot table below
  int map_raw = -1;
  uint32_t w_raw = 0u;
  if (tid < k) {
    const int32_t* mp = p.map + static_cast<int64_t>(t) * k + tid;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(map_raw) : "l"(mp));
    if (!ROUTE) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(w_raw) : "l"(p.topk_w + static_cast<int64_t>(t) * k + tid));
  }

  int vidx[VPT];
  bool vok[VPT];
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    vidx[m] = vbeg + m * nthr + tid;
    vok[m] = vidx[m] < vend;
  }

  // -- shared expert and residual: issued first (they do not depend on the
  //    map), consumed last
  uint4 sh[VPT], res[VPT];
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    const int64_t off = row_off + static_cast<int64_t>(vidx[m]) * 8;
    sh[m] = (p.shared && vok[m]) ? ld_stream16(p.shared + off) : make_uint4(0, 0, 0, 0);
    res[m] = vok[m] ? ld_stream16(p.residual + off) : make_uint4(0, 0, 0, 0);
  }
  // gamma too (up to 2 vectors a thread): otherwise its load would be the
  // last dependent round trip, after the reductions
  constexpr bool kEarlyGamma = VPT <= 2;
  float4 gam[kEarlyGamma ? 2 * VPT : 1];
  if constexpr (kEarlyGamma) {
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
      const float4* g4 = reinterpret_cast<const float4*>(p.gamma + static_cast<int64_t>(vidx[m]) * 8);
      gam[2 * m] = vok[m] ? __ldg(g4) : make_float4(0.f, 0.f, 0.f, 0.f);
      gam[2 * m + 1] = vok[m] ? __ldg(g4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // -- slot table: map entries (checked) and, without routing, the weights
  if (tid < k) {
    int m = map_raw;
    if (m < 0 || static_cast<int64_t>(m) >= p.n_rows) {
      if (p.err_flag) atomicOr(p.err_flag, MOE_FLAG_BAD_INDEX);
      m = -1;  // never dereferenced: the row reads as zeros and its weight is 0
    }
    map_s[tid] = m;
    if (!ROUTE) w_s[tid] = m < 0 ? 0.f : __uint_as_float(w_raw);
  }
  __syncthreads();

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
      if (tid < 32) {
        int id;
        float w;
        route_select<KEYS>(keys, k, p.scale, id, w, route_scr);
        if (tid < k) {
          w_s[tid] = map_s[tid] < 0 ? 0.f : w;  // an unusable slot adds exactly nothing
          if (rank == 0) {
            const int64_t o = static_cast<int64_t>(t) * k + tid;
            if (p.ids_out) p.ids_out[o] = id;
            if (p.w_out) p.w_out[o] = w;
          }
        }
      }
      __syncthreads();
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

  // sum of squares over the token's row: the block, or, when the row is split
  // over a cluster, one exchange of warp sums by remote stores
  if (cs > 1) {
    if (!cluster_block_sum_async(ss, cluster_slots, &ss_bar) && tid == 0 && p.err_flag)
      atomicOr(p.err_flag, MOE_FLAG_TIMEOUT);
  } else {
    ss = block_sum(ss, red);
  }
  const float inv = rsqrtf(ss / static_cast<float>(p.H) + p.eps);

  // -- RMSNorm output
#pragma unroll
  for (int m = 0; m < VPT; ++m) {
    if (!vok[m]) continue;
    float4 g0, g1;
    if constexpr (kEarlyGamma) {
      g0 = gam[2 * m];
      g1 = gam[2 * m + 1];
    } else {
      const float4* g4 = reinterpret_cast<const float4*>(p.gamma + static_cast<int64_t>(vidx[m]) * 8);
      g0 = __ldg(g4);
      g1 = __ldg(g4 + 1);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[m][0] * inv * g0.x, acc[m][1] * inv * g0.y);
    o.y = pack_bf16x2(acc[m][2] * inv * g0.z, acc[m][3] * inv * g0.w);
    o.z = pack_bf16x2(acc[m][4] * inv * g1.x, acc[m][5] * inv * g1.y);
    o.w = pack_bf16x2(acc[m][6] * inv * g1.z, acc[m][7] * inv * g1.w);
    st16(p.normed_out + row_off + static_cast<int64_t>(vidx[m]) * 8, o);
  }
}

// ---------------------------------------------------------------------------
// Large batches: a persistent kernel fed by bulk copies (TMA).
//
// One CTA per SM walks the tokens t = blockIdx.x, + gridDim.x, ...
//  - warp 0 (producer): copies the shared, partial and residual pieces, then
//    (lane j) slot j's expert-row piece, of one chunk of H into a ring of
//    shared-memory stages with cp.async.bulk, counted on the stage's "full"
//    mbarrier; map entries are loaded a token ahead and the next token's rows
//    requested into the L2;
//  - warp 1 (weights): per token, the routing weights -- loaded, or routed
//    from the logits (router-less variant) -- into a ring of token slots, up
//    to kWRing tokens ahead of the consumers; unusable map entries get 0;
//  - warps 2..13 (consumers): FP32 accumulation in the same order as
//    tail_kernel, residual_out stored per chunk, the token's r kept in
//    registers across chunks until the sum of squares is reduced, then the
//    normalised row stored.  Each consumer warp releases a stage ("empty")
//    after reading it and a token slot after the token's last chunk.
// Every wait is bounded: one that runs out sets MOE_FLAG_TIMEOUT and a
// shared abort flag, after which nobody waits any more and the producer only
// drains the copies it has in flight.
// ---------------------------------------------------------------------------

constexpr int kStreamConsumerWarps = 12;
constexpr int kStreamConsumers = 32 * kStreamConsumerWarps;
constexpr int kStreamThreads = 64 + kStreamConsumers;
constexpr int kStreamMaxStages = 8;
constexpr int kMaxAhead = 4;  // tokens whose rows the producer requests into the L2 ahead of their copies
constexpr int kLogitsAhead = 3;  // router-less tail: logits rows requested into the L2 this many tokens ahead
constexpr int kWRing = 4;
constexpr int kStreamSmemBudget = 200 * 1024;
constexpr int kMaxProbes = 1 << 21;  // probes per wait before giving up

struct StreamShape {
  int chunk;        // row elements per stage (multiple of 8)
  int nchunks;      // chunks per row
  int nstages;      // stages in the ring
  int rows;         // row pieces per stage: k slots, shared, R partials, residual
  int stage_bytes;  // rows * chunk * 2 rounded up to 128
  int ahead;        // 0..kMaxAhead: tokens prefetched into the L2 ahead of the one being copied
  int withhold;     // test hook: the stage CTA 0 never copies (its consumers' wait runs out), or -1
};

__device__ __forceinline__ bool stream_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            int32_t* err_flag) {
  for (int it = 0; it < kMaxProbes; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  if (err_flag) atomicOr(err_flag, MOE_FLAG_TIMEOUT);
  return false;
}

// A map entry if it names a row, else -1.
__device__ __forceinline__ int in_rows(int m, int64_t n_rows) {
  return (m >= 0 && static_cast<int64_t>(m) < n_rows) ? m : -1;
}

// A map entry checked for use: -1 (and the error flag raised) if it names no row.
__device__ __forceinline__ int checked_entry(const TailParams& p, int m) {
  if (m < 0 || static_cast<int64_t>(m) >= p.n_rows) {
    if (p.err_flag) atomicOr(p.err_flag, MOE_FLAG_BAD_INDEX);
    return -1;
  }
  return m;
}

// Longest row the stream kernel takes (four 16-byte vectors per consumer thread).
constexpr int kStreamMaxH = 4 * kStreamConsumers * 8;

// Source of the expert-row piece of a slot whose map entry names no row: a
// row of zeros (never written), so with its weight set to 0 the slot adds
// exactly nothing, as in tail_kernel, whatever the other inputs hold.
__device__ __align__(128) uint16_t g_zero_row[kStreamMaxH];

// Source row of piece l of token t's stage: slots 0..k-1 (expert rows through
// the map; an unusable slot reads the zero row and has weight 0), then shared,
// the R partials and the residual.
__device__ __forceinline__ const uint16_t* stream_piece(const TailParams& p, int64_t t, int l, int rows, int slot_row) {
  const int64_t roff = t * p.H;
  if (l < p.k) return slot_row >= 0 ? p.rows + static_cast<int64_t>(slot_row) * p.H : g_zero_row;
  if (p.shared && l == p.k) return p.shared + roff;
  if (l < rows - 1) {
    const int r = l - p.k - (p.shared ? 1 : 0);
    return p.partials + static_cast<int64_t>(r) * p.partial_stride + roff;
  }
  return p.residual + roff;
}

// L2 prefetch hints for every row piece of token t (lane l < k names slot l's
// row).  Hints only: they change no result.
__device__ __forceinline__ void stream_prefetch_token(const TailParams& p, int64_t t, int rows, int slot_row) {
  const int lane = threadIdx.x & 31;
  for (int l = lane; l < rows; l += 32)
    if (l >= p.k || slot_row >= 0) prefetch_l2(stream_piece(p, t, l, rows, slot_row), static_cast<uint32_t>(p.H) * 2u);
}

template <int VPT, int EPL>
__global__ void __launch_bounds__(kStreamThreads, 1)
tail_stream_kernel(const TailParams p, const int T, const StreamShape sh) {
  constexpr bool ROUTE = EPL > 0;
  constexpr int KEYS = EPL > 0 ? EPL : 1;
  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ uint64_t full_bar[kStreamMaxStages];
  __shared__ uint64_t empty_bar[kStreamMaxStages];
  __shared__ uint64_t wfull_bar[kWRing];
  __shared__ uint64_t wempty_bar[kWRing];
  __shared__ float w_ring[kWRing][MOE_MAX_K];
  __shared__ float red[2][kStreamConsumerWarps];
  __shared__ __align__(16) uint64_t route_scr[EPL > 0 ? kRouteScratch : 1];  // the weights warp's candidate list
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = p.k, H = p.H, nvec = H >> 3;
  const int G = static_cast<int>(gridDim.x);
  const int ntok = (T - static_cast<int>(blockIdx.x) + G - 1) / G;
  volatile int* abort_v = &abort_flag;

  if (tid == 0) {
    for (int s = 0; s < sh.nstages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kStreamConsumerWarps);
    }
    for (int s = 0; s < kWRing; ++s) {
      mbar_init(&wfull_bar[s], 1);
      mbar_init(&wempty_bar[s], kStreamConsumerWarps);
    }
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  allow_dependent_launch();
  if (warp == 0) {
    // While the previous kernel finishes: L2 prefetch of this CTA's first
    // tokens, their expert rows named by a relaxed read of the map.  Hints
    // only -- every copy below comes after the dependency wait and sees the
    // final data -- so a stale entry only wastes the hint.
    int pm[kMaxAhead + 1];
#pragma unroll
    for (int q = 0; q <= kMaxAhead; ++q)  // all loads first, then the hints
      pm[q] = (q <= sh.ahead && q < ntok && lane < k)
                  ? ld_relaxed_s32(p.map + (static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(q) * G) * k + lane)
                  : -1;
#pragma unroll
    for (int q = 0; q <= kMaxAhead; ++q) {
      if (q <= sh.ahead && q < ntok)
        stream_prefetch_token(p, static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(q) * G, sh.rows,
                              in_rows(pm[q], p.n_rows));
    }
  } else if (warp == 1) {
    if (lane == 0) prefetch_l2(p.gamma, static_cast<uint32_t>(H) * 4u);
    // router-less tail: the logits rows of the first tokens, which the
    // routing of the first token waits for
    if (ROUTE && lane >= 1 && lane <= kLogitsAhead && lane - 1 < ntok)
      prefetch_row_l2(p.logits + (static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(lane - 1) * G) * p.E, p.E);
  }
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_evict_first_policy();
    const int ahead = sh.ahead;
    // mrow[q]: this lane's raw map entry of token i + q (q <= ahead), loaded
    // a token before it is needed and checked only where it is used, so the
    // producer never waits on a map load it issued itself
    int mrow[kMaxAhead + 1];
#pragma unroll
    for (int q = 0; q <= kMaxAhead; ++q)
      mrow[q] = (q <= ahead && q < ntok && lane < k)
                    ? p.map[(static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(q) * G) * k + lane]
                    : -1;
    int issued = 0;
    const int withheld = blockIdx.x == 0 ? sh.withhold : -1;
    bool stop = false;
    for (int i = 0; i < ntok && !stop; ++i) {
      const int64_t t = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * G;
      int row_cur = -1;
      for (int c = 0; c < sh.nchunks; ++c) {
        const int u = i * sh.nchunks + c, s = u % sh.nstages, n = u / sh.nstages;
        if ((n > 0 && !stream_wait(&empty_bar[s], (n - 1) & 1, abort_v, p.err_flag)) || *abort_v) {
          stop = true;  // no stage is armed after an abort
          break;
        }
        const int c0 = c * sh.chunk;
        const int clen = min(sh.chunk, H - c0);
        if (c == 0 && lane < k) row_cur = checked_entry(p, mrow[0]);
        if (u != withheld) {  // a withheld stage is neither armed nor copied: its full wait runs out
          if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(sh.rows * clen * 2));
          __syncwarp();
          unsigned char* st = stage_mem + static_cast<size_t>(s) * sh.stage_bytes;
          // the pieces that do not depend on the map go first: they fly while
          // the token's first map entries may still be loading
          for (int l = k + lane; l < sh.rows; l += 32)
            bulk_copy_g2s(st + static_cast<size_t>(l) * sh.chunk * 2, stream_piece(p, t, l, sh.rows, -1) + c0,
                          static_cast<uint32_t>(clen * 2), &full_bar[s], pol);
          if (lane < k)
            bulk_copy_g2s(st + static_cast<size_t>(lane) * sh.chunk * 2,
                          stream_piece(p, t, lane, sh.rows, row_cur) + c0, static_cast<uint32_t>(clen * 2),
                          &full_bar[s], pol);
        }
        issued = u + 1;
        if (c == 0) {
          // the L2 prefetch window: tokens i+1..i+ahead are requested once
          // each (all of them after the first token's first stage)
#pragma unroll
          for (int q = 1; q <= kMaxAhead; ++q) {
            if (q <= ahead && i + q < ntok && (i == 0 || q == ahead))
              stream_prefetch_token(p, t + static_cast<int64_t>(q) * G, sh.rows, in_rows(mrow[q], p.n_rows));
          }
          // shift the map ring and request token i+ahead+1's entries
#pragma unroll
          for (int q = 0; q < kMaxAhead; ++q) mrow[q] = mrow[q + 1];
          const int nq = i + ahead + 1;
#pragma unroll
          for (int q = 0; q <= kMaxAhead; ++q) {
            if (q == ahead)
              mrow[q] = (nq < ntok && lane < k) ? p.map[(t + static_cast<int64_t>(ahead + 1) * G) * k + lane] : -1;
          }
        }
      }
    }
    // drain: no copy may land after this CTA exits
    if (lane == 0) {
      for (int u = issued > sh.nstages ? issued - sh.nstages : 0; u < issued; ++u) {
        if (u == withheld) continue;
        for (int it = 0; it < kMaxProbes; ++it)
          if (mbar_try_wait(&full_bar[u % sh.nstages], (u / sh.nstages) & 1)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ weights
    uint32_t keys[KEYS], keys_nxt[KEYS];
    float w_nxt = 0.f;
    int m_nxt = -1;
    // the next token's loads; its map entries are checked only where they are
    // used, a token later, so that no load of the next token stalls the
    // selection of this one
    auto fetch = [&](int64_t t, uint32_t (&kk)[KEYS], float& w, int& m) {
      if (lane < k) {
        m = p.map[t * k + lane];
        if (!ROUTE) w = p.topk_w[t * k + lane];
      }
      if (ROUTE) route_load_keys<KEYS>(p.logits + t * p.E, p.E, kk);
    };
    if (ntok > 0) fetch(blockIdx.x, keys, w_nxt, m_nxt);
    for (int i = 0; i < ntok && !*abort_v; ++i) {
      const int64_t t = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * G;
      float w = w_nxt;
      const int m_raw = m_nxt;
      if (ROUTE) {
#pragma unroll
        for (int e = 0; e < KEYS; ++e) keys_nxt[e] = keys[e];
      }
      if (i + 1 < ntok) fetch(t + G, keys, w_nxt, m_nxt);  // next token's loads in flight
      if (ROUTE && lane == 0 && i + kLogitsAhead < ntok)
        prefetch_row_l2(p.logits + (t + static_cast<int64_t>(kLogitsAhead) * G) * p.E, p.E);
      if (ROUTE) {
        int id;
        route_select<KEYS>(keys_nxt, k, p.scale, id, w, route_scr);  // runs ahead of the consumers
        if (lane < k) {
          if (p.ids_out) p.ids_out[t * k + lane] = id;
          if (p.w_out) p.w_out[t * k + lane] = w;
        }
      }
      const int ok = lane < k && checked_entry(p, m_raw) >= 0;
      const int slot = i % kWRing, n = i / kWRing;
      if (n > 0 && !stream_wait(&wempty_bar[slot], (n - 1) & 1, abort_v, p.err_flag)) break;
      if (lane < k) w_ring[slot][lane] = ok ? w : 0.f;
      __syncwarp();  // the weights are published by lane 0's arrive
      if (lane == 0) mbar_arrive(&wfull_bar[slot]);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ct = tid - 64, cw = warp - 2;
    const int ncv = sh.chunk >> 3;  // vectors per chunk
    float rr[VPT][8];
    // gamma of this thread's vectors, the same for every token: loaded once
    // (up to 2 vectors a thread; wider rows load it per token)
    constexpr bool kGammaRegs = VPT <= 2;
    float4 gam[kGammaRegs ? 2 * VPT : 1];
    if constexpr (kGammaRegs) {
#pragma unroll
      for (int m = 0; m < VPT; ++m) {
        const int v = ct + m * kStreamConsumers;
        const float4* g4 = reinterpret_cast<const float4*>(p.gamma + static_cast<int64_t>(v) * 8);
        gam[2 * m] = v < nvec ? __ldg(g4) : make_float4(0.f, 0.f, 0.f, 0.f);
        gam[2 * m + 1] = v < nvec ? __ldg(g4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    for (int i = 0; i < ntok; ++i) {
      const int64_t t = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * G;
      const int64_t roff = t * H;
      const int slot = i % kWRing;
      if (!*abort_v) stream_wait(&wfull_bar[slot], (i / kWRing) & 1, abort_v, p.err_flag);
      float ss = 0.f;
      for (int c = 0; c < sh.nchunks; ++c) {
        const int u = i * sh.nchunks + c, s = u % sh.nstages, n = u / sh.nstages;
        if (!*abort_v) stream_wait(&full_bar[s], n & 1, abort_v, p.err_flag);
        const unsigned char* st = stage_mem + static_cast<size_t>(s) * sh.stage_bytes;
        const int vb = c * ncv, ve = min(nvec, vb + ncv);
        const int pitch = sh.chunk * 2;
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
          const int v = ct + m * kStreamConsumers;
          if (v < vb || v >= ve) continue;
          const int off = (v - vb) * 16;
          // element pairs in packed FP32 operations: each lane of a pair is
          // one IEEE fma / add, in the same order as the scalar sum
          float2 acc[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
          if (k == 8) {
            // top-8 (the common case): the 8 slots' pieces loaded first, then
            // summed in slot order (the same sum as below; the last chunk of
            // a token takes about 0.2 us less)
            uint4 q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = lds16(st + j * pitch + off);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float w = w_ring[slot][j];
              const float2 w2 = make_float2(w, w);
              float2 f[4];
              unpack8x2(q[j], f);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] = __ffma2_rn(w2, f[e], acc[e]);
            }
          } else {
#pragma unroll 4
            for (int j = 0; j < k; ++j) {
              const float w = w_ring[slot][j];
              const float2 w2 = make_float2(w, w);
              float2 f[4];
              unpack8x2(lds16(st + j * pitch + off), f);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[e] = __ffma2_rn(w2, f[e], acc[e]);
            }
          }
          int l = k;
          if (p.shared) {
            float2 f[4];
            unpack8x2(lds16(st + l * pitch + off), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = __fadd2_rn(acc[e], f[e]);
            ++l;
          }
          for (int r = 0; r < p.R; ++r, ++l) {
            float2 f[4];
            unpack8x2(lds16(st + l * pitch + off), f);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = __fadd2_rn(acc[e], f[e]);
          }
          float2 f[4];
          unpack8x2(lds16(st + (sh.rows - 1) * pitch + off), f);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 r2 = __fadd2_rn(f[e], acc[e]);
            rr[m][2 * e] = r2.x;
            rr[m][2 * e + 1] = r2.y;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(rr[m][e], rr[m][e], ss);
          uint4 o;
          o.x = pack_bf16x2(rr[m][0], rr[m][1]);
          o.y = pack_bf16x2(rr[m][2], rr[m][3]);
          o.z = pack_bf16x2(rr[m][4], rr[m][5]);
          o.w = pack_bf16x2(rr[m][6], rr[m][7]);
          st16(p.residual_out + roff + static_cast<int64_t>(v) * 8, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      if (lane == 0) mbar_arrive(&wempty_bar[slot]);
      // sum of squares over the consumer warps, added in warp order
      ss = warp_sum(ss);
      if (lane == 0) red[i & 1][cw] = ss;
      named_barrier(1, kStreamConsumers);
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kStreamConsumerWarps; ++w) tot += red[i & 1][w];
      const float inv = rsqrtf(tot / static_cast<float>(H) + p.eps);
#pragma unroll
      for (int m = 0; m < VPT; ++m) {
        const int v = ct + m * kStreamConsumers;
        if (v >= nvec) continue;
        float4 g0, g1;
        if constexpr (kGammaRegs) {
          g0 = gam[2 * m];
          g1 = gam[2 * m + 1];
        } else {
          const float4* g4 = reinterpret_cast<const float4*>(p.gamma + static_cast<int64_t>(v) * 8);
          g0 = __ldg(g4);
          g1 = __ldg(g4 + 1);
        }
        uint4 o;
        o.x = pack_bf16x2(rr[m][0] * inv * g0.x, rr[m][1] * inv * g0.y);
        o.y = pack_bf16x2(rr[m][2] * inv * g0.z, rr[m][3] * inv * g0.w);
        o.z = pack_bf16x2(rr[m][4] * inv * g1.x, rr[m][5] * inv * g1.y);
        o.w = pack_bf16x2(rr[m][6] * inv * g1.z, rr[m][7] * inv * g1.w);
        st16(p.normed_out + roff + static_cast<int64_t>(v) * 8, o);
      }
    }
  }
  __syncthreads();
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

template <int VPT, int EPL>
static cudaError_t launch_tail_v(const TailParams& p, int T, const TailLaunch& L, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.cs, T, 1);
  cfg.blockDim = dim3(L.threads, 1, 1);
  cfg.dynamicSmemBytes = launch_smem(0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0] = pdl_attribute();
  int nattr = 1;
  if (L.cs > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = L.cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  // 4 vectors a thread gather 4 slots a batch (16 loads in flight a thread):
  // 8 would not fit the registers beside the routing warp's selection
  return cudaLaunchKernelEx(&cfg, tail_kernel<VPT, (VPT >= 4 ? 4 : 8), EPL>, p);
}

template <int EPL>
static cudaError_t launch_tail_e(const TailParams& q, int Tc, const TailLaunch& L, cudaStream_t stream) {
  switch (L.vpt) {
    case 1: return launch_tail_v<1, EPL>(q, Tc, L, stream);
    case 2: return launch_tail_v<2, EPL>(q, Tc, L, stream);
    case 3: return launch_tail_v<3, EPL>(q, Tc, L, stream);
    default: return launch_tail_v<4, EPL>(q, Tc, L, stream);
  }
}

// Stage geometry of the stream kernel: the fewest chunks per row that leave
// room for at least three stages within the shared-memory budget.
static bool stream_shape(int H, int rows, StreamShape& sh) {
  for (int nch = 1; nch <= 64; ++nch) {
    const int chunk = ((H + nch - 1) / nch + 7) / 8 * 8;
    const int stage = (rows * chunk * 2 + 127) / 128 * 128;
    const int ns = kStreamSmemBudget / stage;
    if (ns >= 3) {
      sh.chunk = chunk;
      sh.nchunks = (H + chunk - 1) / chunk;
      sh.nstages = ns < kStreamMaxStages ? ns : kStreamMaxStages;
      sh.rows = rows;
      sh.stage_bytes = stage;
      sh.ahead = 1;
      sh.withhold = -1;
      return true;
    }
  }
  return false;
}

template <int VPT, int EPL>
static cudaError_t launch_stream_v(const TailParams& p, int T, const StreamShape& sh, int grid,
                                   cudaStream_t stream) {
  static bool smem_opt_in[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev >= 0 && dev < 64 && !smem_opt_in[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(tail_stream_kernel<VPT, EPL>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmemBudget);
    if (e != cudaSuccess) return e;
    smem_opt_in[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = launch_smem(static_cast<size_t>(sh.nstages) * sh.stage_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tail_stream_kernel<VPT, EPL>, p, T, sh);
}

template <int EPL>
static cudaError_t launch_stream_e(const TailParams& p, int T, const StreamShape& sh, int grid, int vpt,
                                   cudaStream_t stream) {
  switch (vpt) {
    case 1: return launch_stream_v<1, EPL>(p, T, sh, grid, stream);
    case 2: return launch_stream_v<2, EPL>(p, T, sh, grid, stream);
    case 3: return launch_stream_v<3, EPL>(p, T, sh, grid, stream);
    default: return launch_stream_v<4, EPL>(p, T, sh, grid, stream);
  }
}

// The stream kernel takes batches of at least two tokens per SM whose rows fit
// four vectors per consumer thread.
static bool use_stream(int64_t T, int H, int rows, int nsm, StreamShape& sh) {
  return T >= 2 * static_cast<int64_t>(nsm) && H <= kStreamMaxH && stream_shape(H, rows, sh);
}

// Test hook of the bounded waits (moe_debug_withhold_stream_stage): a stage
// that the next persistent-kernel launch withholds, taken by that launch.
static std::atomic<int> g_withheld_stage{-1};
static int take_withheld_stage() { return g_withheld_stage.exchange(-1); }

template <bool ROUTE>
static int launch_tail(TailParams p, int64_t T, cudaStream_t stream) {
  const int nsm = sm_count();
  StreamShape sh;
  const int rows = p.k + (p.shared ? 1 : 0) + p.R + 1;
  const bool stream_path = use_stream(T, p.H, rows, nsm, sh);
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
    cudaError_t e;
    if (stream_path) {
      const int grid = Tc < nsm ? Tc : nsm;
      // one token of rows requested into the L2 ahead of its copies
      sh.ahead = 1;
      sh.withhold = t0 == 0 ? take_withheld_stage() : -1;
      const int vpt = (p.H / 8 + kStreamConsumers - 1) / kStreamConsumers;
      if (!ROUTE) e = launch_stream_e<0>(q, Tc, sh, grid, vpt, stream);
      else if (p.E <= 256) e = launch_stream_e<8>(q, Tc, sh, grid, vpt, stream);
      else e = launch_stream_e<32>(q, Tc, sh, grid, vpt, stream);
    } else {
      const TailLaunch L = choose_tail_launch(T, p.H, nsm);
      if (!ROUTE) e = launch_tail_e<0>(q, Tc, L, stream);
      else if (p.E <= 256) e = launch_tail_e<8>(q, Tc, L, stream);
      else e = launch_tail_e<32>(q, Tc, L, stream);
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

extern "C" int moe_debug_withhold_stream_stage(int32_t stage) {
  if (stage < -1) return MOE_ERR_INVALID_ARG;
  moe::g_withheld_stage.store(stage);
  return MOE_OK;
}
