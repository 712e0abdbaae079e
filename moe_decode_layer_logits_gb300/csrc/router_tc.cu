// Router GEMM for batches of more than 64 tokens on the 5th-generation tensor
// cores: logits[T, E] = x[T, H] . W[E, H]^T, BF16 operands, FP32 accumulation
// in tensor memory (lmdeploy pull 4853, Summary: FP32 router logits through a
// BF16 GEMM).  At T in the thousands the router is a dense contraction near
// the tensor-core ridge, and from about a hundred tokens up the deep per-SM
// copy stream below already beats register-fed MMAs, so it is tiled for
// tcgen05:
//  - one CTA per 128-expert x BNT-token tile: the gate weight is the M side
//    (UMMA M = 128) and the tokens the N side (N = BNT, 64..128 in steps of
//    16, chosen per launch so that the grid fills the SMs), so tensor-memory
//    lane i holds expert i of the tile and column j token j;
//  - warp 0 streams 64-wide K blocks of both operands with TMA (128-byte
//    swizzle, out-of-range rows and columns zero-filled) into a 6-stage ring;
//  - warp 1 allocates tensor-memory columns for BNT and one lane issues
//    tcgen05.mma (kind::f16, 4 per K block), releasing each stage with
//    tcgen05.commit when the MMAs that read it complete;
//  - warps 2..5 wait for the final commit and read the accumulator with
//    tcgen05.ld (each warp its 32-lane quarter = 32 experts, 32 tokens per
//    load) into a [token][expert] tile in the CTA's own (now idle) operand
//    ring: for one token the 32 lanes hold 32 consecutive experts, so these
//    writes are free of bank conflicts; the rows then leave as 16-byte
//    stores, 512 contiguous bytes per warp.
// Every wait is bounded; a tile whose pipeline gave up is written as NaN so
// that the failure is visible in the output, and MOE_FLAG_TIMEOUT is raised
// in the caller's error flag if one is given.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "host_util.h"
#include "router_tc.h"

namespace moe {

constexpr int kTcBM = 128;       // experts per tile (UMMA M)
constexpr int kTcBK = 64;        // K elements per stage: one 128-byte swizzle row
constexpr int kTcStages = 6;
constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 epilogue
constexpr int kTcMaxWaits = 1 << 21;

// Tensor-memory columns for an N-wide accumulator: a power of two >= 32.
__host__ __device__ constexpr uint32_t tmem_cols(int n) { return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : 256u; }

template <int BNT>
struct TcSmem {
  uint8_t a[kTcStages][kTcBM * kTcBK * 2];  // gate weight: 16 KB per stage, 1024-byte aligned
  uint8_t b[kTcStages][BNT * kTcBK * 2];    // tokens: BNT * 128 bytes per stage
  uint64_t full[kTcStages];
  uint64_t empty[kTcStages];
  uint64_t tmem_full;
  uint64_t rx_full;  // split-K: the peers' partials of this CTA's tokens have landed
  uint32_t tmem_base;
  int abort_flag;
};

// ---- tcgen05 / TMA primitives --------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms, so the
// stride between 8-row groups is 1024 bytes; the leading offset is not used by
// swizzled K-major layouts.  Bits: start >> 4 [0,14), leading offset >> 4
// [16,30), stride offset >> 4 [32,46), descriptor version 1 [46,48), swizzle
// mode 2 = 128-byte [61,64).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with BF16 A and B, FP32 D, both
// operands K-major: D format [4,6) = 1, A format [7,10) = 1, B format [10,13)
// = 1, N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Bulk copy of `bytes` from this CTA's shared memory into a peer's, completing
// on the peer's mbarrier (both peer addresses from mapa).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Store logits[t, e .. e + 3] (the columns below E), as one 16-byte store
// when `vec` (E a multiple of 4 and a 16-byte aligned base).
__device__ __forceinline__ void store4(float* __restrict__ logits, int t, int e, int E, bool vec, float4 v) {
  float* dst = logits + static_cast<int64_t>(t) * E + e;
  if (vec) {
    if (e < E) *reinterpret_cast<float4*>(dst) = v;
  } else {
    if (e < E) dst[0] = v.x;
    if (e + 1 < E) dst[1] = v.y;
    if (e + 2 < E) dst[2] = v.z;
    if (e + 3 < E) dst[3] = v.w;
  }
}

__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait; gives up early once the CTA's abort flag is raised unless
// `drain` is set (a drain must see the phase, abort or not).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, bool drain) {
  for (int it = 0; it < kTcMaxWaits; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!drain && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}

// withhold_kb (test hook): the K block whose loads the first CTA never
// issues, so that its MMA warp's wait runs out; -1 in normal launches.
template <int BNT>
__global__ void __launch_bounds__(kTcThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                 float* __restrict__ logits, int T, int H, int E, int32_t* err_flag, int withhold_kb) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<BNT>& sm = *reinterpret_cast<TcSmem<BNT>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * BNT, e0 = blockIdx.y * kTcBM;
  const int S = gridDim.z;  // split-K: the cluster's CTAs take consecutive K ranges
  const int nkb_all = (H + kTcBK - 1) / kTcBK;
  const int kb0 = static_cast<int>(static_cast<int64_t>(nkb_all) * blockIdx.z / S);
  const int nkb = static_cast<int>(static_cast<int64_t>(nkb_all) * (blockIdx.z + 1) / S) - kb0;
  volatile int* abort_v = &sm.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.tmem_full, 1);
    mbar_init(&sm.rx_full, 1);
    sm.abort_flag = 0;
    mbar_init_fence();
  }
  static_assert(BNT % 16 == 0 && BNT >= 16 && BNT <= 128, "UMMA N for M = 128");
  if (warp == 1) tmem_alloc(&sm.tmem_base, tmem_cols(BNT));
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = sm.tmem_base;

  allow_dependent_launch();
  grid_dependency_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      const int withheld = (blockIdx.x | blockIdx.y | blockIdx.z) == 0 ? withhold_kb : -1;
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kTcStages, n = kb / kTcStages;
        if (n > 0 && !tc_wait(&sm.empty[s], (n - 1) & 1, abort_v, false)) break;
        issued = kb + 1;
        if (kb == withheld) continue;  // neither armed nor loaded: the MMA warp's wait runs out
        mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>((kTcBM + BNT) * kTcBK * 2));
        tma_load_2d(sm.a[s], &tmap_w, (kb0 + kb) * kTcBK, e0, &sm.full[s]);
        tma_load_2d(sm.b[s], &tmap_x, (kb0 + kb) * kTcBK, t0, &sm.full[s]);
      }
      // drain: no copy may land after this CTA exits
      for (int kb = issued > kTcStages ? issued - kTcStages : 0; kb < issued; ++kb)
        if (kb != withheld) tc_wait(&sm.full[kb % kTcStages], (kb / kTcStages) & 1, abort_v, true);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kTcBM, BNT);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kTcStages, n = kb / kTcStages;
        if (!tc_wait(&sm.full[s], n & 1, abort_v, false)) break;
        tc_fence_after_sync();
        const uint32_t a0 = smem_addr(sm.a[s]), b0 = smem_addr(sm.b[s]);
#pragma unroll
        for (int kk = 0; kk < kTcBK / 16; ++kk) {  // 16 BF16 = 32 bytes of K per MMA
          umma_bf16(tmem_d, umma_desc_sw128(a0 + kk * 32), umma_desc_sw128(b0 + kk * 32), idesc,
                    (kb | kk) != 0);
        }
        umma_commit(&sm.empty[s]);
      }
      umma_commit(&sm.tmem_full);  // also after an abort: it fires once issued MMAs are done
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ epilogue
  // Warps 2..5 own tensor-memory lane quarter q = warp % 4: experts
  // e0 + 32 q + lane.  Each CTA first writes its accumulator as a [token]
  // [expert] tile into its own token ring.  Without split-K the tile is stored
  // as it is.  With split-K tokens [r * BNT/S, (r+1) * BNT/S) of the tile
  // belong to rank r: every CTA sends each peer that peer's rows with one bulk
  // copy into the peer's (idle) weight ring, and each owner adds the S
  // partials in rank order (deterministic) and stores the sums.
  static_assert(BNT * kTcBM * 4 <= sizeof(sm.a) && BNT * kTcBM * 4 <= sizeof(sm.b),
                "the partial tile must fit in either operand ring");
  __syncwarp();  // warps 0 and 1 reconverge after their lane-0 loops
  const bool epi = warp >= 2;
  const int q = warp & 3;
  const int e_t = q * 32 + lane;  // expert within the tile
  const int etid = threadIdx.x - 64;  // 0..127 in the epilogue warps
  float* part = reinterpret_cast<float*>(&sm.b[0][0]);  // [BNT][kTcBM]
  const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  const float nan = __int_as_float(0x7FC00000);
  bool ok = true;
  if (epi) {
    ok = tc_wait(&sm.tmem_full, 0, abort_v, true) && !*abort_v;
    tc_fence_after_sync();
#pragma unroll 1
    for (int c = 0; c < BNT; c += 32) {
      uint32_t v[32];
      tmem_ld_32cols(tmem_d + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c), v);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c + i < BNT) part[(c + i) * kTcBM + e_t] = ok ? __uint_as_float(v[i]) : nan;
    }
  }
  // The 128 epilogue threads store 4 experts each, 4 token rows per pass.
  const int c4 = (etid & 31) * 4;
  if (S == 1) {
    if (epi) {
      named_barrier(1, 128);
#pragma unroll 4
      for (int r = etid >> 5; r < BNT && t0 + r < T; r += 4)
        store4(logits, t0 + r, e0 + c4, E, vec, *reinterpret_cast<const float4*>(part + r * kTcBM + c4));
    }
  } else {
    const int rpo = BNT / S;  // tokens owned per rank
    const int rank = static_cast<int>(cg::this_cluster().block_rank());
    const uint32_t chunk = static_cast<uint32_t>(rpo * kTcBM * 4);
    float* recv = reinterpret_cast<float*>(&sm.a[0][0]);  // [S][rpo][kTcBM]
    if (threadIdx.x == 64) mbar_arrive_expect_tx(&sm.rx_full, static_cast<uint32_t>(S - 1) * chunk);
    if (epi) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tile is read by bulk copies
    cluster_arrive_release();  // every CTA's MMAs are done (rings free) and its tile written
    cluster_wait_acquire();
    if (threadIdx.x == 64) {
      for (int o = 0; o < S; ++o) {
        if (o == rank) continue;
        bulk_copy_to_peer(peer_addr(smem_addr(recv) + static_cast<uint32_t>(rank) * chunk, o),
                          smem_addr(part) + static_cast<uint32_t>(o) * chunk, chunk, peer_addr(smem_addr(&sm.rx_full), o));
      }
    }
    if (epi) ok = tc_wait(&sm.rx_full, 0, abort_v, true) && ok;
    // Arrive once this CTA holds every partial of its tokens; no CTA leaves
    // before all have arrived, so no copy reads the memory of a CTA that exited.
    cluster_arrive_release();
    if (epi) {
      // sum in rank order (a peer's NaN propagates), then store
      for (int r = etid >> 5; r < rpo && t0 + rank * rpo + r < T; r += 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < S) {
            const float* src = j == rank ? part + (rank * rpo + r) * kTcBM : recv + (j * rpo + r) * kTcBM;
            const float4 p = *reinterpret_cast<const float4*>(src + c4);
            acc.x += p.x;
            acc.y += p.y;
            acc.z += p.z;
            acc.w += p.w;
          }
        }
        if (!ok) acc = make_float4(nan, nan, nan, nan);
        store4(logits, t0 + rank * rpo + r, e0 + c4, E, vec, acc);
      }
    }
    cluster_wait_acquire();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && err_flag && *abort_v) atomicOr(err_flag, MOE_FLAG_TIMEOUT);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_d, tmem_cols(BNT));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Row-major BF16 [rows, cols] matrix, boxes of box_rows x 64 with the 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BNT>
static size_t tc_smem_bytes() {
  return sizeof(TcSmem<BNT>) + 1024;  // + alignment slack for the 1024-byte swizzle atoms
}

// Opt the kernel into its dynamic shared memory, once per device.
template <int BNT>
static cudaError_t tc_opt_in(int dev) {
  static std::atomic<bool> done[64];
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev].load()) {
    const cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<BNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(tc_smem_bytes<BNT>()));
    if (e != cudaSuccess) return e;
    done[dev].store(true);
  }
  return cudaSuccess;
}

// How many clusters of S CTAs (S = 2, 4, 8) of this kernel the device holds
// at once (cudaOccupancyMaxActiveClusters, cached per device); 0 if unknown.
template <int BNT>
static int tc_max_clusters(int dev, int S) {
  static std::atomic<int> cache[64][3];  // 0 = not asked yet, else count + 1
  const int si = S == 2 ? 0 : S == 4 ? 1 : 2;
  if (dev < 0 || dev >= 64 || tc_opt_in<BNT>(dev) != cudaSuccess) return 0;
  int c = cache[dev][si].load();
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, S);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = tc_smem_bytes<BNT>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_tc_kernel<BNT>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    c = n + 1;
    cache[dev][si].store(c);
  }
  return c - 1;
}

template <int BNT>
static cudaError_t launch_tc(const CUtensorMap& mx, const CUtensorMap& mw, float* logits, int T, int H, int E,
                             int32_t* err_flag, int withhold_kb, int S, int dev, cudaStream_t stream) {
  const cudaError_t oe = tc_opt_in<BNT>(dev);
  if (oe != cudaSuccess) return oe;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T + BNT - 1) / BNT, (E + kTcBM - 1) / kTcBM, S);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = launch_smem(tc_smem_bytes<BNT>());
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
  return cudaLaunchKernelEx(&cfg, router_tc_kernel<BNT>, mx, mw, logits, T, H, E, err_flag, withhold_kb);
}

static int max_clusters_for(int bnt, int dev, int S) {
  switch (bnt) {
    case 64: return tc_max_clusters<64>(dev, S);
    case 80: return tc_max_clusters<80>(dev, S);
    case 96: return tc_max_clusters<96>(dev, S);
    case 112: return tc_max_clusters<112>(dev, S);
    default: return tc_max_clusters<128>(dev, S);
  }
}

// Launch shape of one router call: token tile and split-K factor.
struct TcShape {
  int bnt, S;
};

// Choose the token tile BNT (64..128, steps of 16) and the split-K cluster
// size S (1, 2, 4, 8) by a small cost model: a CTA's time is its K blocks'
// bytes at the rate one SM streams them (about 120 GB/s, latency-bound), plus
// about 3 us for the split-K exchange, times the number of waves.  Split-K
// grids must fit in one wave of clusters as the device reports it (on GB300
// with ~200 KB of shared memory per CTA: 76 clusters of 2, 36 of 4, 15 of 8;
// sixteen clusters of 8 took two waves, 24 against 13 us), and every rank
// keeps >= 2 K blocks.  Ties go to the larger tile.
// `max_clusters(bnt, S)` gives how many clusters of S CTAs fit at once.
template <class MaxClusters>
static TcShape choose_shape(int T, int H, int E, int nsm, MaxClusters max_clusters) {
  const int nkb = (H + kTcBK - 1) / kTcBK;
  const int ne = (E + kTcBM - 1) / kTcBM;
  TcShape best{128, 1};
  double best_us = 1e30;
  for (int bnt = 128; bnt >= 64; bnt -= 16) {
    const int tiles = ((T + bnt - 1) / bnt) * ne;
    for (int S = 1; S <= 8; S *= 2) {
      const int ctas = tiles * S;
      if (S > 1 && (nkb < 2 * S || ctas > nsm || tiles > max_clusters(bnt, S))) continue;
      const int waves = (ctas + nsm - 1) / nsm;
      const double bytes = static_cast<double>((nkb + S - 1) / S) * (kTcBM + bnt) * kTcBK * 2;
      const double us = waves * (bytes / 120e3 + (S > 1 ? 3.0 : 0.0));
      if (us < best_us * 0.999) {
        best_us = us;
        best = TcShape{bnt, S};
      }
    }
  }
  return best;
}

template <int BNT>
static cudaError_t launch_bnt(const void* x, const void* w, float* logits, int T, int H, int E, int32_t* err_flag,
                              int withhold_kb, int S, int dev, cudaStream_t stream) {
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, T, H, BNT) || !make_map(&mw, w, E, H, kTcBM)) return cudaErrorInvalidValue;
  return launch_tc<BNT>(mx, mw, logits, T, H, E, err_flag, withhold_kb, S, dev, stream);
}

// Test hook of the bounded waits (moe_debug_withhold_router_stage): a K block
// that the next tensor-memory router launch withholds, taken by that launch.
static std::atomic<int> g_withheld_kb{-1};

cudaError_t launch_router_tc(const void* x, const void* w, float* logits, int T, int H, int E, int32_t* err_flag,
                             int nsm, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const TcShape sh = choose_shape(T, H, E, nsm, [dev](int bnt, int S) { return max_clusters_for(bnt, dev, S); });
  const int wk = g_withheld_kb.exchange(-1);
  switch (sh.bnt) {
    case 64: return launch_bnt<64>(x, w, logits, T, H, E, err_flag, wk, sh.S, dev, stream);
    case 80: return launch_bnt<80>(x, w, logits, T, H, E, err_flag, wk, sh.S, dev, stream);
    case 96: return launch_bnt<96>(x, w, logits, T, H, E, err_flag, wk, sh.S, dev, stream);
    case 112: return launch_bnt<112>(x, w, logits, T, H, E, err_flag, wk, sh.S, dev, stream);
    default: return launch_bnt<128>(x, w, logits, T, H, E, err_flag, wk, sh.S, dev, stream);
  }
}

bool router_tc_supported(int64_t T, int64_t H) { return T >= kRouterTcMinT && H >= kTcBK; }

}  // namespace moe

extern "C" int moe_debug_withhold_router_stage(int32_t kb) {
  if (kb < -1) return MOE_ERR_INVALID_ARG;
  moe::g_withheld_kb.store(kb);
  return MOE_OK;
}

// Host-only test hook: the launch shape the tcgen05 router would take for a
// device with `nsm` SMs that holds mc2 / mc4 / mc8 clusters of 2 / 4 / 8 CTAs
// at once (for every token tile).
extern "C" int moe_debug_router_tc_shape(int64_t T, int64_t H, int64_t E, int32_t nsm, int32_t mc2, int32_t mc4,
                                         int32_t mc8, int32_t* bnt, int32_t* split_k) {
  if (T < 1 || T > (int64_t{1} << 30) || H < moe::kTcBK || H > (1 << 20) || E < 1 || E > MOE_MAX_E || nsm < 1 ||
      mc2 < 0 || mc4 < 0 || mc8 < 0 || !bnt || !split_k)
    return MOE_ERR_INVALID_ARG;
  const moe::TcShape sh = moe::choose_shape(static_cast<int>(T), static_cast<int>(H), static_cast<int>(E), nsm,
                                            [=](int, int S) { return S == 2 ? mc2 : S == 4 ? mc4 : mc8; });
  *bnt = sh.bnt;
  *split_k = sh.S;
  return MOE_OK;
}
