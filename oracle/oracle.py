"""FP64 CPU oracle for the decode MoE-layer tail.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``moe_decode_layer_logits_gb300``) and imports
nothing from it.

Sources (web pages on serving GLM-5.x MoE models):

* lmdeploy pull 4853, "perf: further optimize GLM-5.2 serving", Summary:
  the router GEMM takes BF16 hidden states and the BF16 gate weight and keeps
  FP32 logits.
* vllm-project/vllm pull 62174 (deferred MoE finalize), Overview, Claims,
  Validation and Details: the decode MoE layer leaves its top-k reduction
  open; one fused kernel then does the top-k weighted sum, the routed scaling
  (folded into the routing weights by the router), the shared-expert add, the
  (all-)reduce, the residual add and RMSNorm, accumulating in FP32 and
  rounding once.  The unit test's contract: the fused result equals
  finalize, then shared add, then RMSNorm(all_reduce(.)).
* milou-sh/vllm pull 3, "Port the validated GLM-5.2 H200 production path to
  latest vLLM", Ported behavior: row-parallel partial outputs fused with the
  all-reduce, residual add and RMSNorm; on one GPU the all-reduce becomes a
  sum of R local partial buffers.

Every floating-point step here is done in IEEE double.  BF16 inputs widen to
double exactly; BF16 outputs are rounded from double straight to BF16 (round
to nearest, ties to even) without passing through binary32, so each output is
rounded exactly once.

Readings of points the pages leave open (each one is listed with its reason
in the design notes of the repository):

* routing weights are ``scale * softmax`` over the k selected logits, the
  selection is by raw logit, ties go to the lower expert index and the k ids
  come out in descending logit order;
* RMSNorm is ``r / sqrt(mean(r**2) + eps) * gamma`` with gamma in FP32,
  applied to the unrounded residual sum;
* the accumulated tail is ``residual + (sum_j w_j * row_j + shared + sum_r P_r)``.

Parity status: every function below is pinned by ``tests/test_oracle.py``
(closed forms, a library RMSNorm, exact integer arithmetic, brute force and
exhaustive BF16 rounding).  The scoring-function choice (softmax over the
top-k, scale 2.5 / 1.0) is a reading, not something the pages print, so the
numbers it produces are pinned only against that reading.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "bf16_ulp",
    "router_logits",
    "topk_route",
    "moe_finalize",
    "shared_add",
    "partials_sum",
    "add_rmsnorm",
    "finalize_add_rmsnorm",
    "tail_fused",
]

# ---------------------------------------------------------------------------
# BF16 <-> double.  bfloat16 is the upper half of an IEEE binary32: 1 sign bit,
# 8 exponent bits (bias 127) and 7 stored fraction bits, so 8 significant bits.
# ---------------------------------------------------------------------------

_BF16_MIN_EXP_QUANTUM = -133  # subnormal spacing: 2^-149 * 2^16
_BF16_OVERFLOW = 2.0 ** 128   # values that round to this magnitude become inf


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen BF16 bit patterns (uint16) to double; exact."""
    b = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round doubles to BF16 (nearest, ties to even) directly from double.

    A finite value with binary exponent e (|x| in [2^(e-1), 2^e)) has BF16
    spacing 2^(e-8); below the normal range the spacing stays 2^-133.  The
    value is scaled by a power of two (exact), rounded to an integer with
    ties-to-even, and scaled back (exact).  The result is then a BF16 value,
    which binary32 holds exactly, so its top 16 bits are the BF16 pattern.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q = np.maximum(e - 8, _BF16_MIN_EXP_QUANTUM)
    y = np.ldexp(np.rint(np.ldexp(x, -q)), q)
    out = np.empty(x.shape, dtype=np.uint16)
    finite = np.isfinite(y) & (np.abs(y) < _BF16_OVERFLOW)
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = np.where(finite, y, 0.0).astype(np.float32)
    out[...] = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    big = ~np.isnan(x) & ~finite
    out[big] = np.where(np.signbit(x[big]), 0xFF80, 0x7F80).astype(np.uint16)
    out[np.isnan(x)] = 0x7FC0
    return out


def bf16_ulp(v) -> np.ndarray:
    """Spacing of BF16 values at the magnitude of ``v`` (double in, double out).

    For |v| in [2^(e-1), 2^e) the spacing is 2^(e-8), never below the
    subnormal spacing 2^-133.
    """
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    e = np.where(v == 0.0, _BF16_MIN_EXP_QUANTUM, e - 8)
    return np.ldexp(1.0, np.maximum(e, _BF16_MIN_EXP_QUANTUM))


# ---------------------------------------------------------------------------
# (1) Router logits.  lmdeploy pull 4853, Summary: BF16 inputs, FP32 logits.
#     L[t, e] = sum_h x[t, h] * W[e, h].
# ---------------------------------------------------------------------------

def router_logits(x_bits, w_bits):
    """Return (L, A): L[t,e] = sum_h x[t,h] W[e,h] and A[t,e] = sum_h |x W|.

    Products of two BF16 values are exact in double, and the double sum's
    error is negligible next to any FP32 tolerance.  ``A`` is the magnitude
    against which the GPU's FP32 accumulation error is measured.
    """
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    return x @ w.T, np.abs(x) @ np.abs(w).T


# ---------------------------------------------------------------------------
# (2) Top-k selection and routing weights.  vllm pull 62174, Details: the
#     router folds routed_scaling_factor into the routing weights, so the
#     deferred output carries no scaling of its own.
# ---------------------------------------------------------------------------

def topk_route(logits_f32, k: int, scale: float):
    """Select the k largest logits per row and weight them.

    Selection is by logit value, descending; equal logits keep ascending
    expert order (a stable sort of the negated values).  The weights are
    ``scale * exp(l_j - l_max) / sum_i exp(l_i - l_max)`` over the selected
    experts, evaluated in double and rounded to binary32 once.

    Returns (ids int32 [T,k], w float32 [T,k], w64 float64 [T,k]).
    """
    lg = np.asarray(logits_f32, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(lg, ids, axis=1)
    ex = np.exp(sel - sel[:, :1])
    w64 = float(scale) * ex / ex.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w64.astype(np.float32), w64


# ---------------------------------------------------------------------------
# (3) MoE finalize: the top-k weighted sum through the expanded-index map.
#     vllm pull 62174, Overview and Details ("top-k sum").
# ---------------------------------------------------------------------------

def moe_finalize(rows_bits, row_map, topk_w):
    """routed[t, :] = sum_j w[t, j] * rows[map[t, j], :], in double.

    ``rows_bits`` is the BF16 [N, H] buffer of unfinalized expert rows,
    ``row_map`` the int [T, k] expanded-index map and ``topk_w`` the FP32
    [T, k] routing weights (already scaled).
    """
    rows = bf16_bits_to_f64(rows_bits)
    mp = np.asarray(row_map, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    T, k = mp.shape
    out = np.zeros((T, rows.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * rows[mp[:, j]]
    return out


def shared_add(routed, shared_bits):
    """y = routed + shared (vllm pull 62174, Claims: "shared + routed add")."""
    if shared_bits is None:
        return np.asarray(routed, dtype=np.float64)
    return routed + bf16_bits_to_f64(shared_bits)


def partials_sum(partials_bits):
    """sum_r P[r] over R partial buffers [R, T, H] (milou-sh/vllm pull 3,
    Ported behavior: row-parallel partial outputs summed before the residual
    add and RMSNorm)."""
    p = bf16_bits_to_f64(partials_bits)
    return p.sum(axis=0)


def add_rmsnorm(residual_bits, y, gamma, eps: float):
    """r = residual + y; normed = r / sqrt(mean_h r^2 + eps) * gamma.

    lmdeploy pull 4853 (RMSNorm consumes the pending reduction, fused with the
    residual add) and vllm pull 62174, Details (residual add and RMSNorm after
    the reduction).  The norm uses the unrounded r.
    """
    r = bf16_bits_to_f64(residual_bits) + y
    ms = np.mean(r * r, axis=1, keepdims=True)
    g = np.asarray(gamma, dtype=np.float32).astype(np.float64)
    normed = r / np.sqrt(ms + float(eps)) * g[None, :]
    return r, normed


def finalize_add_rmsnorm(rows_bits, row_map, topk_w, shared_bits, partials_bits,
                         residual_bits, gamma, eps):
    """The whole tail of one decode MoE layer, rounded once at the end.

    y = finalize(rows, map, w) [+ shared] [+ sum_r P_r]; r = residual + y;
    out = RMSNorm(r) * gamma.  ``row_map``/``topk_w`` may have k = 0 columns
    (no routed part); ``shared_bits`` and ``partials_bits`` may be None.

    Returns a dict with the BF16 outputs (``residual_out``, ``normed``), their
    double values (``r``, ``normed64``), and ``abs_terms``: per element the sum
    of the magnitudes of every term that enters r (the yardstick of an FP32
    accumulation's rounding error).
    """
    residual = bf16_bits_to_f64(residual_bits)
    T, H = residual.shape
    mp = np.asarray(row_map, dtype=np.int64).reshape(T, -1)
    w = np.asarray(topk_w, dtype=np.float32).reshape(T, -1)
    if mp.shape[1] > 0:
        y = moe_finalize(rows_bits, mp, w)
        rows = bf16_bits_to_f64(rows_bits)
        absr = np.zeros((T, H))
        for j in range(mp.shape[1]):
            absr += np.abs(w[:, j:j + 1].astype(np.float64)) * np.abs(rows[mp[:, j]])
    else:
        y = np.zeros((T, H))
        absr = np.zeros((T, H))
    y = shared_add(y, shared_bits)
    if shared_bits is not None:
        absr += np.abs(bf16_bits_to_f64(shared_bits))
    if partials_bits is not None:
        y = y + partials_sum(partials_bits)
        absr += np.abs(bf16_bits_to_f64(partials_bits)).sum(axis=0)
    absr += np.abs(residual)
    r, normed = add_rmsnorm(residual_bits, y, gamma, eps)
    return {
        "residual_out": f64_to_bf16_bits(r),
        "normed": f64_to_bf16_bits(normed),
        "r": r,
        "normed64": normed,
        "abs_terms": absr,
    }


def tail_fused(logits_f32, k, scale, rows_bits, row_map, shared_bits,
               residual_bits, gamma, eps):
    """The router-less fused tail: route from FP32 logits, then the tail.

    Returns the ``finalize_add_rmsnorm`` dict plus ``ids``, ``w`` (binary32)
    and ``w64``.
    """
    ids, w, w64 = topk_route(logits_f32, k, scale)
    out = finalize_add_rmsnorm(rows_bits, row_map, w, shared_bits, None,
                               residual_bits, gamma, eps)
    out.update(ids=ids, w=w, w64=w64)
    return out
