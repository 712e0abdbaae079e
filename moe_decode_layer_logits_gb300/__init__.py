"""Decode MoE-layer tail for one sm_103a GPU (GLM-5.x style MoE layers).

Python binding of the C ABI in ``include/moe_tail.h``: argument marshalling
only.  Every step runs in the CUDA kernels of ``libmoe_tail.so``; PyTorch
provides device memory and the stream.  Functions take CUDA tensors and
launch on ``stream`` (default: the current torch stream); output tensors are
allocated with torch when not given.

* ``moe_router_logits_fp32(x, w_gate)``      -> FP32 logits [T, E]
* ``moe_topk_route(logits, k, scale)``       -> ids [T, k] int32, weights [T, k] FP32
* ``moe_finalize_add_rmsnorm(...)``          -> (residual_out, normed) BF16 [T, H]
* ``moe_tail_fused(logits, k, scale, ...)``  -> (residual_out, normed, ids, weights)
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import MoeTailError, check, lib

__all__ = [
    "moe_debug_withhold_stream_stage",
    "moe_debug_withhold_router_stage",
    "moe_debug_fail_next_launch",
    "moe_debug_router_tc_shape",
    "moe_router_logits_fp32",
    "moe_topk_route",
    "moe_finalize_add_rmsnorm",
    "moe_tail_fused",
    "MoeTailError",
    "lib",
]


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t, dtype, name, ndim=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    return t.data_ptr()


def moe_router_logits_fp32(x, w_gate, logits_out=None, err_flag=None, stream=None):
    """logits[T, E] = x[T, H] . w_gate[E, H]^T (BF16 in, FP32 accumulate and out).
    err_flag: optional int32 CUDA tensor; MOE_FLAG_TIMEOUT is OR-ed into it
    when a bounded wait of the tensor-memory kernel (T > 64) runs out (the
    affected logits are NaN either way)."""
    T, H = x.shape
    E = w_gate.shape[0]
    if logits_out is None:
        logits_out = torch.empty((T, E), dtype=torch.float32, device=x.device)
    st = lib().moe_router_logits_fp32(_ptr(x, torch.bfloat16, "x", 2), _ptr(w_gate, torch.bfloat16, "w_gate", 2),
                                      _ptr(logits_out, torch.float32, "logits_out", 2), T, H, E,
                                      _ptr(err_flag, torch.int32, "err_flag", optional=True), _stream(stream))
    check(st, "moe_router_logits_fp32")
    return logits_out


def moe_topk_route(logits, k, routed_scale, topk_ids=None, topk_w=None, stream=None):
    """Top-k experts per token (descending, ties to the lower index) and
    routed_scale * softmax over the selected logits."""
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    st = lib().moe_topk_route(_ptr(logits, torch.float32, "logits", 2), _ptr(topk_ids, torch.int32, "topk_ids"),
                              _ptr(topk_w, torch.float32, "topk_w"), T, E, int(k), float(routed_scale),
                              _stream(stream))
    check(st, "moe_topk_route")
    return topk_ids, topk_w


def moe_finalize_add_rmsnorm(rows, row_map, topk_w, shared, residual, gamma, eps, partials=None,
                             residual_out=None, normed_out=None, err_flag=None, stream=None):
    """The fused tail: sum_j w_j rows[map_j] + shared + sum_r partials[r] + residual,
    then RMSNorm * gamma; both outputs rounded to BF16 once."""
    T, H = residual.shape
    k = 0 if row_map is None else int(row_map.shape[1])
    R = 0 if partials is None else int(partials.shape[0])
    n_rows = 0 if rows is None else int(rows.shape[0])
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    if normed_out is None:
        normed_out = torch.empty_like(residual)
    st = lib().moe_finalize_add_rmsnorm(
        _ptr(rows, torch.bfloat16, "rows", 2, optional=True), n_rows,
        _ptr(row_map, torch.int32, "row_map", 2, optional=True),
        _ptr(topk_w, torch.float32, "topk_w", 2, optional=True), k,
        _ptr(shared, torch.bfloat16, "shared", 2, optional=True),
        _ptr(partials, torch.bfloat16, "partials", 3, optional=True), R,
        _ptr(residual, torch.bfloat16, "residual", 2), _ptr(gamma, torch.float32, "gamma", 1), float(eps),
        _ptr(residual_out, torch.bfloat16, "residual_out", 2), _ptr(normed_out, torch.bfloat16, "normed_out", 2),
        T, H, _ptr(err_flag, torch.int32, "err_flag", optional=True), _stream(stream))
    check(st, "moe_finalize_add_rmsnorm")
    return residual_out, normed_out


def moe_tail_fused(logits, k, routed_scale, rows, row_map, shared, residual, gamma, eps,
                   residual_out=None, normed_out=None, topk_ids=None, topk_w=None, want_route=True,
                   err_flag=None, stream=None):
    """Router-less fused tail: route from FP32 logits, then the fused tail."""
    T, H = residual.shape
    E = logits.shape[1]
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    if normed_out is None:
        normed_out = torch.empty_like(residual)
    if want_route and topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=residual.device)
    if want_route and topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=residual.device)
    st = lib().moe_tail_fused(
        _ptr(logits, torch.float32, "logits", 2), E, int(k), float(routed_scale),
        _ptr(rows, torch.bfloat16, "rows", 2), int(rows.shape[0]), _ptr(row_map, torch.int32, "row_map", 2),
        _ptr(shared, torch.bfloat16, "shared", 2, optional=True), _ptr(residual, torch.bfloat16, "residual", 2),
        _ptr(gamma, torch.float32, "gamma", 1), float(eps),
        _ptr(residual_out, torch.bfloat16, "residual_out", 2), _ptr(normed_out, torch.bfloat16, "normed_out", 2),
        _ptr(topk_ids, torch.int32, "topk_ids", optional=True), _ptr(topk_w, torch.float32, "topk_w", optional=True),
        T, H, _ptr(err_flag, torch.int32, "err_flag", optional=True), _stream(stream))
    check(st, "moe_tail_fused")
    return residual_out, normed_out, topk_ids, topk_w


def moe_debug_withhold_stream_stage(stage):
    """Test hook of the bounded waits: the next persistent-kernel launch
    leaves stage `stage` of its first CTA uncopied, so that CTA's wait runs
    out and MOE_FLAG_TIMEOUT is set; -1 cancels the request."""
    check(lib().moe_debug_withhold_stream_stage(int(stage)), "moe_debug_withhold_stream_stage")


def moe_debug_withhold_router_stage(kb):
    """Test hook of the router's bounded waits: the next tensor-memory router
    launch issues no loads for K block `kb` in its first CTA, so that CTA's
    wait runs out, its tile is written as NaN and MOE_FLAG_TIMEOUT is set;
    -1 cancels the request."""
    check(lib().moe_debug_withhold_router_stage(int(kb)), "moe_debug_withhold_router_stage")


def moe_debug_fail_next_launch(on=True):
    """Test hook of the launch-error path: the next kernel launch of any entry
    point is refused by the CUDA runtime (oversized shared-memory request),
    so that call raises MoeTailError with MOE_ERR_CUDA; on=False cancels."""
    check(lib().moe_debug_fail_next_launch(1 if on else 0), "moe_debug_fail_next_launch")


def moe_debug_router_tc_shape(T, H, E, nsm, mc2, mc4, mc8):
    """Test hook (host only): the (token tile, split-K cluster size) the
    tensor-memory router would take for T x H x E on a device with `nsm` SMs
    that holds mc2 / mc4 / mc8 clusters of 2 / 4 / 8 router CTAs at once."""
    bnt, split_k = ctypes.c_int32(), ctypes.c_int32()
    check(lib().moe_debug_router_tc_shape(int(T), int(H), int(E), int(nsm), int(mc2), int(mc4), int(mc8),
                                          ctypes.byref(bnt), ctypes.byref(split_k)), "moe_debug_router_tc_shape")
    return bnt.value, split_k.value
