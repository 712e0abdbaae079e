/*
 * moe_tail.h -- C ABI of the decode MoE-layer tail on one sm_103a GPU.
 *
 * The tail of a GLM-5.x style MoE decoder layer, from the router to the
 * normalised input of the next layer:
 *
 *   logits = x . W_gate^T                      (BF16 in, FP32 accumulate, FP32 out)
 *   ids, w = top-k(logits), scale * softmax    (routing scale folded into w)
 *   y      = sum_j w[t,j] * rows[map[t,j]]     (MoE finalize, FP32)
 *            + shared + sum_r P[r]             (shared expert, row-parallel partials)
 *   r      = residual + y                      -> residual_out (BF16, rounded once)
 *   out    = r / sqrt(mean(r^2) + eps) * gamma -> normed_out   (BF16, rounded once)
 *
 * Sources: lmdeploy pull 4853 "perf: further optimize GLM-5.2 serving"
 * (Summary: FP32 router logits from BF16 inputs; small-token router GEMM);
 * vllm-project/vllm pull 62174 (Overview, Claims, Details: the deferred
 * top-k reduction is closed by one kernel that does the top-k sum, routed
 * scaling, shared add, reduction, residual add and RMSNorm, accumulating in
 * FP32 and rounding once); milou-sh/vllm pull 3 (Ported behavior: row-parallel
 * partial outputs fused with the reduction, residual add and RMSNorm).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *    every buffer; the library allocates nothing and keeps no state beyond
 *    cached device attributes (SM count) per device and the one-shot request
 *    of the test hook at the end of this header.
 *  - Tensors are row-major with the last dimension contiguous.  BF16 data is
 *    passed as `const void*` holding IEEE bfloat16 bit patterns.
 *  - Work is enqueued on `stream` (which may be 0, the legacy default stream)
 *    on the current device.  No call synchronises or allocates.
 *  - Arguments are checked on the host before anything is launched; a
 *    violation returns a status code and launches nothing.  T == 0 returns
 *    MOE_OK without launching.  A launch error reported by the CUDA runtime
 *    returns MOE_ERR_CUDA.
 *  - BF16 pointers and `gamma` must be 16-byte aligned (16-byte vector
 *    loads); FP32 / int32 pointers 4-byte aligned.
 *  - Results are deterministic: the same inputs and sizes on the same GPU
 *    give bit-identical outputs (fixed summation order, no atomics on data).
 */
#ifndef MOE_TAIL_H
#define MOE_TAIL_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, negative size, k/E/R/eps out of range */
  MOE_ERR_UNSUPPORTED = 2, /* a size the kernels do not handle (H % 8 != 0, E > 1024, ...) */
  MOE_ERR_MISALIGNED = 3,  /* a pointer breaks the alignment rule above */
  MOE_ERR_CUDA = 4,        /* the CUDA runtime reported an error at launch */
  MOE_ERR_BAD_INDEX = 5    /* reserved for callers reading the error flag (see below) */
} moe_status_t;

/* Limits checked on the host. */
#define MOE_MAX_E 1024 /* routed experts per router / route call */
#define MOE_MAX_K 32   /* experts per token */
#define MOE_MAX_R 8    /* row-parallel partial buffers */

/* Bits written (OR-ed) into the optional device error flag. */
#define MOE_FLAG_BAD_INDEX 1 /* some map[t,j] was outside [0, n_rows) */
#define MOE_FLAG_TIMEOUT 2   /* a bounded pipeline wait ran out (outputs of that launch are invalid) */

/* Human-readable name of a status code (static storage, never NULL). */
const char* moe_status_string(int status);

/*
 * Router logits in FP32: logits_out[t, e] = sum_h x[t, h] * w_gate[e, h].
 * lmdeploy pull 4853, Summary: BF16 hidden states times the BF16 gate weight
 * with FP32 accumulation, FP32 logits kept.
 *
 *   x_bf16      [T, H]  BF16, 16-byte aligned
 *   w_gate_bf16 [E, H]  BF16, 16-byte aligned
 *   logits_out  [T, E]  FP32, written
 *   err_flag    device int32 or NULL: MOE_FLAG_TIMEOUT is OR-ed into it when
 *               a bounded wait of the tensor-memory kernel runs out (below)
 *   T >= 0; H >= 8, H % 8 == 0; 1 <= E <= MOE_MAX_E.
 *
 * Products are exact; partial sums are FP32 (tensor-core accumulate), so
 * |logits - exact| is a small multiple of 2^-24 * sum_h |x * w|.
 *
 * w_gate is a model parameter: the kernel starts copying it into shared
 * memory before it waits for the previous kernel on the stream, so it must
 * not be written by a kernel that may still be running on `stream` when this
 * call is made (x may be: it is read only after that wait).
 *
 * Every wait inside the kernels is bounded (2^21 probes, seconds at most):
 * the split-K exchange of the decode-size kernel and the stage pipeline of
 * the tensor-memory kernel that batches of more than 64 tokens (H >= 64)
 * take.  If one runs out, the logits of the affected tile (a split-K owner's
 * outputs, or a 128-expert x token tile) are written as NaN (a quiet NaN in
 * every element) and the call still returns MOE_OK, as the launch was made;
 * the tensor-memory kernel also OR-s MOE_FLAG_TIMEOUT into *err_flag (if
 * err_flag is given), the decode-size kernel reports it in the logits only.
 * NaN logits give unspecified ids downstream.
 */
int moe_router_logits_fp32(const void* x_bf16, const void* w_gate_bf16, float* logits_out,
                           int64_t T, int64_t H, int64_t E, int32_t* err_flag, cudaStream_t stream);

/*
 * Top-k routing: per token the k largest logits (descending; equal logits in
 * ascending expert order) and weights w_j = routed_scale * exp(l_j - l_max) /
 * sum_i exp(l_i - l_max) over the k selected experts.  The routed scaling
 * factor is folded into the weights: vllm pull 62174, Details.
 *
 *   logits     [T, E] FP32 (finite values; NaN/inf give unspecified ids)
 *   topk_ids   [T, k] int32, written
 *   topk_w     [T, k] FP32, written
 *   T >= 0; 1 <= E <= MOE_MAX_E; 1 <= k <= min(E, MOE_MAX_K);
 *   routed_scale finite.
 */
int moe_topk_route(const float* logits, int32_t* topk_ids, float* topk_w,
                   int64_t T, int64_t E, int32_t k, float routed_scale, cudaStream_t stream);

/*
 * MoE finalize + shared add + row-parallel partial sum + residual add + RMSNorm,
 * one kernel, FP32 accumulation, each output rounded to BF16 once (nearest
 * even).  vllm pull 62174, Overview/Claims/Details; milou-sh/vllm pull 3,
 * Ported behavior.  Per token t and element h, in this order:
 *
 *   acc  = sum_{j=0}^{k-1} topk_w[t,j] * rows[map[t,j], h]   (FMA, j ascending)
 *   acc += shared[t, h]                       (if shared_bf16 != NULL)
 *   acc += partials[r, t, h], r = 0..R-1       (if R > 0)
 *   r    = residual[t, h] + acc
 *   residual_out[t, h] = bf16(r)
 *   normed_out[t, h]   = bf16(r * rsqrt(sum_h r^2 / H + eps) * gamma[h])
 *
 *   rows_bf16     [n_rows, H] BF16 unfinalized expert rows (any order)
 *   map           [T, k] int32 expanded-index map, values in [0, n_rows)
 *   topk_w        [T, k] FP32 routing weights (already scaled)
 *   shared_bf16   [T, H] BF16 or NULL
 *   partials_bf16 [R, T, H] BF16, required when R > 0
 *   residual_bf16 [T, H] BF16
 *   gamma         [H] FP32, 16-byte aligned
 *   residual_out  [T, H] BF16, written; may be the same pointer as residual
 *   normed_out    [T, H] BF16, written; must not overlap any input
 *   err_flag      device int32 or NULL.  A map entry outside [0, n_rows) is
 *                 never dereferenced: its row counts as zero and, if err_flag
 *                 is given, MOE_FLAG_BAD_INDEX is OR-ed into *err_flag (the
 *                 caller clears it and reads it after the stream completes).
 *                 MOE_FLAG_TIMEOUT there means a pipeline wait of the
 *                 large-batch kernel ran out and that launch's outputs are
 *                 invalid.
 *   0 <= k <= MOE_MAX_K (k == 0: no routed part; rows/map/topk_w may be NULL);
 *   0 <= R <= MOE_MAX_R; H >= 8, H % 8 == 0, H <= 65536; eps >= 0 and finite.
 */
int moe_finalize_add_rmsnorm(const void* rows_bf16, int64_t n_rows, const int32_t* map,
                             const float* topk_w, int32_t k,
                             const void* shared_bf16, const void* partials_bf16, int32_t R,
                             const void* residual_bf16, const float* gamma, float eps,
                             void* residual_out_bf16, void* normed_out_bf16,
                             int64_t T, int64_t H, int32_t* err_flag, cudaStream_t stream);

/*
 * Router-less fused tail: the top-k routing of moe_topk_route on the given
 * FP32 logits, then the tail of moe_finalize_add_rmsnorm (without partials)
 * with those weights, in one kernel.  vllm pull 62174, Claims: the GEMM2 tail
 * is one kernel instead of three.
 *
 *   logits [T, E] FP32; 1 <= E <= MOE_MAX_E; 1 <= k <= min(E, MOE_MAX_K)
 *   topk_ids_out [T, k] int32 or NULL; topk_w_out [T, k] FP32 or NULL:
 *                 when given, the routing decisions are written there too.
 *   other arguments as in moe_finalize_add_rmsnorm.
 */
int moe_tail_fused(const float* logits, int64_t E, int32_t k, float routed_scale,
                   const void* rows_bf16, int64_t n_rows, const int32_t* map,
                   const void* shared_bf16, const void* residual_bf16, const float* gamma, float eps,
                   void* residual_out_bf16, void* normed_out_bf16,
                   int32_t* topk_ids_out, float* topk_w_out,
                   int64_t T, int64_t H, int32_t* err_flag, cudaStream_t stream);

/*
 * Test hook of the bounded waits; no counterpart on the pages.  The next
 * launch of the persistent tail kernel (the path taken by batches of at
 * least two tokens per SM) leaves stage `stage` of its first CTA unarmed and
 * uncopied, so that CTA's consumers wait for it until their bounded wait
 * runs out (2^21 probes, seconds at most), set MOE_FLAG_TIMEOUT in err_flag and stop
 * waiting; the launch still completes, its outputs are invalid, and the next
 * launch is unaffected.  One launch takes the request (a decode-size launch
 * leaves it for the next persistent one); stage -1 cancels it.  Returns
 * MOE_OK, or MOE_ERR_INVALID_ARG for stage < -1.  Not for production use.
 */
int moe_debug_withhold_stream_stage(int32_t stage);

/*
 * Test hook of the router's bounded waits; no counterpart on the pages.  The
 * next launch of the tensor-memory router kernel (batches of more than 64
 * tokens, H >= 64) issues no loads for K block `kb` (64 columns of H) in its
 * first CTA, so that CTA's MMA warp waits for them until its bounded wait
 * runs out: the first 128-expert x token tile is written as NaN and
 * MOE_FLAG_TIMEOUT is set in err_flag; the other tiles are correct and the
 * next launch is unaffected.  kb -1 cancels the request.  Returns MOE_OK, or
 * MOE_ERR_INVALID_ARG for kb < -1.  Not for production use.
 */
int moe_debug_withhold_router_stage(int32_t kb);

/*
 * Test hook of the launch-error path; no counterpart on the pages.  With
 * on = 1 the next kernel launch made by any entry point asks the CUDA
 * runtime for more dynamic shared memory than a thread block may have; the
 * runtime refuses it before anything runs (a launch-configuration error, not
 * a sticky one), the entry point returns MOE_ERR_CUDA, and later calls run
 * normally.  on = 0 cancels a pending request.  Returns MOE_OK, or
 * MOE_ERR_INVALID_ARG for any other value.  Not for production use.
 */
int moe_debug_fail_next_launch(int32_t on);

/*
 * Test hook of the launch-shape choice of the tensor-memory router (batches
 * of more than 64 tokens); no counterpart on the pages.  Host only, launches
 * nothing.  For a device with `nsm` SMs that holds mc2 / mc4 / mc8 clusters
 * of 2 / 4 / 8 router CTAs at once, writes the token tile the router would
 * take (64, 80, 96, 112 or 128 tokens per CTA, 128 experts each) to *bnt
 * and its split-K cluster size (1, 2, 4 or 8) to *split_k.  Returns MOE_OK,
 * or MOE_ERR_INVALID_ARG for T outside [1, 2^30], H outside [64, 2^20], E outside [1, MOE_MAX_E],
 * nsm < 1, a negative cluster count or a NULL output.
 */
int moe_debug_router_tc_shape(int64_t T, int64_t H, int64_t E, int32_t nsm, int32_t mc2, int32_t mc4,
                              int32_t mc8, int32_t* bnt, int32_t* split_k);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TAIL_H */
