"""Host side of the C ABI, no GPU needed: the library loads, exports every
symbol include/moe_tail.h declares, and rejects bad arguments before any
launch (every case below fails a host check, so nothing is ever launched and
no fake pointer is ever dereferenced)."""

import ctypes
import os
import re

import pytest

from moe_decode_layer_logits_gb300 import _lib as L
from moe_decode_layer_logits_gb300.build import LIB as LIB_PATH, build_library

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moe_tail.h")

P = 0x10000     # fake, 16-byte aligned, never dereferenced
P2 = 0x10002    # misaligned for BF16 / FP32
NULL = None
S = None        # stream


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB_PATH):
        build_library()
    return L.lib()


@pytest.fixture(autouse=True)
def no_visible_gpu(request):
    # These cases pass fake device addresses; each must fail a host check.  A
    # case that wrongly passed would launch on them, so they only run where no
    # GPU is visible (the failing launch then stays on the host).
    if "lib" in request.fixturenames:
        import torch
        if torch.cuda.is_available():
            pytest.skip("fake-pointer argument checks run only without a visible GPU")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["moe_status_string", "moe_router_logits_fp32", "moe_topk_route",
                 "moe_finalize_add_rmsnorm", "moe_tail_fused"]:
        assert want in names
    # every declared function has a ctypes signature in the binding
    assert set(names) <= set(L.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert L.status_string(code).startswith("MOE_")
    assert "unknown" in L.status_string(99)


# -- moe_router_logits_fp32(x, w, logits, T, H, E, stream)

@pytest.mark.parametrize("args,want", [
    ((P, P, P, -1, 64, 16), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 0, 16), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 64, 0), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 60, 16), L.MOE_ERR_UNSUPPORTED),
    ((P, P, P, 4, 64, 2048), L.MOE_ERR_UNSUPPORTED),
    ((NULL, P, P, 4, 64, 16), L.MOE_ERR_INVALID_ARG),
    ((P, NULL, P, 4, 64, 16), L.MOE_ERR_INVALID_ARG),
    ((P, P, NULL, 4, 64, 16), L.MOE_ERR_INVALID_ARG),
    ((P2, P, P, 4, 64, 16), L.MOE_ERR_MISALIGNED),
    ((P, P2, P, 4, 64, 16), L.MOE_ERR_MISALIGNED),
    ((P, P, P + 1, 4, 64, 16), L.MOE_ERR_MISALIGNED),
    ((NULL, NULL, NULL, 0, 64, 16), L.MOE_OK),  # T == 0: nothing to do
])
def test_router_argument_checks(lib, args, want):
    assert lib.moe_router_logits_fp32(*args, S) == want


# -- moe_topk_route(logits, ids, w, T, E, k, scale, stream)

@pytest.mark.parametrize("args,want", [
    ((P, P, P, -1, 64, 4, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 64, 0, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 4, 5, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 64, 33, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 2048, 8, 1.0), L.MOE_ERR_UNSUPPORTED),
    ((P, P, P, 4, 64, 4, float("nan")), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 64, 4, float("inf")), L.MOE_ERR_INVALID_ARG),
    ((NULL, P, P, 4, 64, 4, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, NULL, P, 4, 64, 4, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P, P, NULL, 4, 64, 4, 1.0), L.MOE_ERR_INVALID_ARG),
    ((P + 2, P, P, 4, 64, 4, 1.0), L.MOE_ERR_MISALIGNED),
    ((NULL, NULL, NULL, 0, 64, 4, 1.0), L.MOE_OK),
])
def test_route_argument_checks(lib, args, want):
    assert lib.moe_topk_route(*args, S) == want


# -- moe_finalize_add_rmsnorm(rows, n_rows, map, w, k, shared, partials, R, residual, gamma, eps,
#                             residual_out, normed_out, T, H, err_flag, stream)

def fin(**kw):
    a = dict(rows=P, n_rows=32, map=P, w=P, k=8, shared=P, partials=NULL, R=0, residual=P, gamma=P,
             eps=1e-6, rout=P, nout=P, T=4, H=64, err=NULL)
    a.update(kw)
    return (a["rows"], a["n_rows"], a["map"], a["w"], a["k"], a["shared"], a["partials"], a["R"],
            a["residual"], a["gamma"], a["eps"], a["rout"], a["nout"], a["T"], a["H"], a["err"])


@pytest.mark.parametrize("kw,want", [
    (dict(T=-1), L.MOE_ERR_INVALID_ARG),
    (dict(H=0), L.MOE_ERR_INVALID_ARG),
    (dict(H=68), L.MOE_ERR_UNSUPPORTED),
    (dict(H=65544), L.MOE_ERR_UNSUPPORTED),
    (dict(k=-1), L.MOE_ERR_INVALID_ARG),
    (dict(k=33), L.MOE_ERR_INVALID_ARG),
    (dict(R=-1), L.MOE_ERR_INVALID_ARG),
    (dict(R=9, partials=P), L.MOE_ERR_INVALID_ARG),
    (dict(R=2), L.MOE_ERR_INVALID_ARG),            # partials missing
    (dict(eps=-1.0), L.MOE_ERR_INVALID_ARG),
    (dict(eps=float("nan")), L.MOE_ERR_INVALID_ARG),
    (dict(eps=float("inf")), L.MOE_ERR_INVALID_ARG),
    (dict(n_rows=-1), L.MOE_ERR_INVALID_ARG),
    (dict(rows=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(map=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(w=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(residual=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(gamma=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(rout=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(nout=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(rows=P2), L.MOE_ERR_MISALIGNED),
    (dict(shared=P + 8), L.MOE_ERR_MISALIGNED),
    (dict(residual=P + 8), L.MOE_ERR_MISALIGNED),
    (dict(gamma=P + 4), L.MOE_ERR_MISALIGNED),
    (dict(rout=P + 8), L.MOE_ERR_MISALIGNED),
    (dict(nout=P2), L.MOE_ERR_MISALIGNED),
    (dict(map=P + 2), L.MOE_ERR_MISALIGNED),
    (dict(w=P + 2), L.MOE_ERR_MISALIGNED),
    (dict(R=1, partials=P + 8), L.MOE_ERR_MISALIGNED),
    (dict(T=0, rows=NULL, map=NULL, w=NULL, residual=NULL, gamma=NULL, rout=NULL, nout=NULL), L.MOE_OK),
])
def test_finalize_argument_checks(lib, kw, want):
    assert lib.moe_finalize_add_rmsnorm(*fin(**kw), S) == want


# -- moe_tail_fused(logits, E, k, scale, rows, n_rows, map, shared, residual, gamma, eps,
#                   residual_out, normed_out, ids_out, w_out, T, H, err_flag, stream)

def fused(**kw):
    a = dict(logits=P, E=256, k=8, scale=2.5, rows=P, n_rows=32, map=P, shared=P, residual=P, gamma=P,
             eps=1e-6, rout=P, nout=P, ids=NULL, w=NULL, T=4, H=64, err=NULL)
    a.update(kw)
    return (a["logits"], a["E"], a["k"], a["scale"], a["rows"], a["n_rows"], a["map"], a["shared"],
            a["residual"], a["gamma"], a["eps"], a["rout"], a["nout"], a["ids"], a["w"], a["T"], a["H"],
            a["err"])


@pytest.mark.parametrize("kw,want", [
    (dict(E=0), L.MOE_ERR_INVALID_ARG),
    (dict(k=0), L.MOE_ERR_INVALID_ARG),
    (dict(k=9, E=8), L.MOE_ERR_INVALID_ARG),
    (dict(E=1025), L.MOE_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), L.MOE_ERR_INVALID_ARG),
    (dict(T=-3), L.MOE_ERR_INVALID_ARG),
    (dict(H=12), L.MOE_ERR_UNSUPPORTED),
    (dict(logits=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(rows=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(map=NULL), L.MOE_ERR_INVALID_ARG),
    (dict(logits=P + 2), L.MOE_ERR_MISALIGNED),
    (dict(ids=P + 2), L.MOE_ERR_MISALIGNED),
    (dict(w=P + 1), L.MOE_ERR_MISALIGNED),
    (dict(residual=P + 2), L.MOE_ERR_MISALIGNED),
    (dict(T=0, logits=NULL, rows=NULL, map=NULL, residual=NULL, gamma=NULL, rout=NULL, nout=NULL), L.MOE_OK),
])
def test_fused_argument_checks(lib, kw, want):
    assert lib.moe_tail_fused(*fused(**kw), S) == want


def test_withhold_hook_argument_check(lib):
    # host-only: the request is stored for the next persistent-kernel launch
    assert lib.moe_debug_withhold_stream_stage(-2) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_withhold_stream_stage(-1) == L.MOE_OK


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import moe_decode_layer_logits_gb300 as M
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.zeros(16, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="CUDA tensor"):
        M.moe_router_logits_fp32(x, w, logits_out=torch.zeros(4, 16), stream=0)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        L.lib()
