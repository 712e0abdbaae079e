"""Tolerances of the GPU-vs-oracle comparisons, derived from the arithmetic.

u = 2^-24 is the unit roundoff of binary32.

* Router logits: |gpu - L| <= 1e-5 * sum_h |x w| (the stated bound).
* Routing weights, GPU formula w_j = (scale * e_j) / sum_i e_i with
  e_j = expf(l_j - l_top) in binary32: the subtraction costs u*|l_j - l_top|,
  expf at most 2 ulp (4u), the 32-lane tree sum 5u plus the largest e error,
  the product and the quotient 2u.  So
  |w_j - w64_j| <= |w64_j| * u * (D_j + D_max + 15), D = |l - l_top|.
* Tail: r is an FMA / add chain of n = k + [shared] + R + 1 binary32 roundings,
  each at most u times a partial sum bounded by S = sum of |terms|, so
  |r32 - r| <= (n + 1) u S  (+ sum_j |dw_j| |row_j| when the weights differ).
  The norm scale inv = rsqrt(ss/H + eps) carries the sum-of-squares error
  (tree depth d <= 128 roundings, plus 2 max|dr| sum|r| / sum r^2 from the
  inputs), rsqrtf's 2 ulp and the two roundings of r * inv * gamma:
  |n32 - n| <= |gamma| inv |dr| + |n| (rel_inv + 2u).
* A BF16 output passes when |bf16(gpu) - bf16(oracle)| <= ulp_bf16 + delta:
  one BF16 ulp as stated, widened by delta only where the FP32 forward error
  bound itself reaches the ulp (cancellation in r, or a near-zero output).
"""

import numpy as np

import oracle as O

U = 2.0 ** -24


def route_weight_tol(logits_f32, ids, w64):
    lg = np.asarray(logits_f32, np.float32).astype(np.float64)
    sel = np.take_along_axis(lg, ids.astype(np.int64), axis=1)
    D = np.abs(sel - sel[:, :1])
    Dmax = D.max(axis=1, keepdims=True)
    return np.abs(w64) * U * (D + Dmax + 15.0) * 1.01 + 1e-45


def tail_deltas(ref, n_ops, gamma, eps, extra_abs_r=None):
    """Per-element error bounds (delta_r, delta_n) for the BF16 outputs."""
    S = ref["abs_terms"]
    dr = (n_ops + 1) * U * S
    if extra_abs_r is not None:
        dr = dr + extra_abs_r
    r = ref["r"]
    H = r.shape[1]
    ss = np.sum(r * r, axis=1, keepdims=True)
    inv = 1.0 / np.sqrt(ss / H + eps)
    rel_ss = 128 * U + 2.0 * dr.max(axis=1, keepdims=True) * np.abs(r).sum(axis=1, keepdims=True) / np.maximum(ss, 1e-300)
    rel_inv = 0.5 * rel_ss + 6 * U
    g = np.abs(np.asarray(gamma, np.float64))[None, :]
    dn = g * inv * dr + np.abs(ref["normed64"]) * (rel_inv + 2 * U)
    return dr * 1.01, dn * 1.01


# Per-case statistics of every BF16 comparison, printed at the end of the run
# (tests/conftest.py, terminal summary): how close each output came and how
# many elements needed the FP32 widening at all.
STATS = []
EXTRA = []  # free-form lines (e.g. rows a chain test could not compare one to one)


def check_bf16(name, gpu_bits, ref_bits, ref_val, delta, max_widened_frac=0.01):
    """Assert |bf16(gpu) - bf16(ref)| <= ulp + delta everywhere; returns stats.

    The stats (also appended to STATS): the largest difference in BF16 ulps,
    the number and fraction of elements more than one ulp away (they passed
    only through delta), the fraction bit-identical to the oracle and the
    fraction of elements whose tolerance was widened at all (delta > ulp/2).
    """
    g = O.bf16_bits_to_f64(gpu_bits)
    o = O.bf16_bits_to_f64(ref_bits)
    ulp = np.maximum(O.bf16_ulp(o), O.bf16_ulp(ref_val))
    diff = np.abs(g - o)
    tol = ulp + delta
    bad = ~(diff <= tol)
    widened = float(np.mean(delta > 0.5 * ulp)) if delta.size else 0.0
    above = int(np.sum(diff > ulp))
    st = {"case": name, "n": int(diff.size),
          "max_ulps": float(np.max(diff / ulp)) if diff.size else 0.0,
          "above_1ulp": above, "above_1ulp_frac": above / max(1, diff.size),
          "exact_frac": float(np.mean(diff == 0)) if diff.size else 1.0,
          "widened_frac": widened, "widened_cap": float(max_widened_frac)}
    STATS.append(st)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{name}: {bad.sum()} of {bad.size} elements beyond 1 BF16 ulp (+FP32 bound); first at {idx.tolist()}: "
            f"gpu {g[tuple(idx[0])]!r} oracle {o[tuple(idx[0])]!r} exact {ref_val[tuple(idx[0])]!r} "
            f"tol {tol[tuple(idx[0])]!r}")
    assert widened <= max_widened_frac, f"{name}: tolerance widened on {widened:.4%} of elements"
    return st
