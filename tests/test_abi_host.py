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


# -- moe_router_logits_fp32(x, w, logits, T, H, E, err_flag, stream)

@pytest.mark.parametrize("args,want", [
    ((P, P, P, -1, 64, 16, NULL), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 0, 16, NULL), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 64, 0, NULL), L.MOE_ERR_INVALID_ARG),
    ((P, P, P, 4, 60, 16, NULL), L.MOE_ERR_UNSUPPORTED),
    ((P, P, P, 4, 64, 2048, NULL), L.MOE_ERR_UNSUPPORTED),
    ((NULL, P, P, 4, 64, 16, NULL), L.MOE_ERR_INVALID_ARG),
    ((P, NULL, P, 4, 64, 16, NULL), L.MOE_ERR_INVALID_ARG),
    ((P, P, NULL, 4, 64, 16, NULL), L.MOE_ERR_INVALID_ARG),
    ((P2, P, P, 4, 64, 16, NULL), L.MOE_ERR_MISALIGNED),
    ((P, P2, P, 4, 64, 16, NULL), L.MOE_ERR_MISALIGNED),
    ((P, P, P + 1, 4, 64, 16, NULL), L.MOE_ERR_MISALIGNED),
    ((P, P, P, 4, 64, 16, P + 2), L.MOE_ERR_MISALIGNED),
    ((NULL, NULL, NULL, 0, 64, 16, NULL), L.MOE_OK),  # T == 0: nothing to do
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
    # the same for the next tensor-memory router launch
    assert lib.moe_debug_withhold_router_stage(-2) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_withhold_router_stage(-1) == L.MOE_OK


def test_fail_next_launch_hook_argument_check(lib):
    # host-only: a request is stored (and cancelled here) for the next launch
    assert lib.moe_debug_fail_next_launch(2) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_fail_next_launch(-1) == L.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_fail_next_launch(1) == L.MOE_OK
    assert lib.moe_debug_fail_next_launch(0) == L.MOE_OK


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


# ---------------------------------------------------------------------------
# launch shape of the tensor-memory router (host logic, no launch)
# ---------------------------------------------------------------------------

# clusters of 2 / 4 / 8 router CTAs one GB300 (152 SMs) holds at once, as
# cudaOccupancyMaxActiveClusters reports them for ~200 KB of shared memory
GB300_SMS, GB300_CLUSTERS = 152, (76, 36, 15)


def _shape(T, H, E, nsm=GB300_SMS, mc=GB300_CLUSTERS):
    import moe_decode_layer_logits_gb300 as M
    return M.moe_debug_router_tc_shape(T, H, E, nsm, *mc)


def _modelled_us(T, H, E, nsm, bnt, S):
    # the cost model the choice is documented to minimise: a CTA's K-block
    # bytes at ~120 GB/s per SM, ~3 us per split-K exchange, times the waves
    nkb = -(-H // 64)
    ctas = -(-T // bnt) * -(-E // 128) * S
    waves = -(-ctas // nsm)
    return waves * (-(-nkb // S) * (128 + bnt) * 128 / 120e3 + (3.0 if S > 1 else 0.0))


def _feasible(T, H, E, nsm, mc, bnt, S):
    if S == 1:
        return True
    tiles = -(-T // bnt) * -(-E // 128)
    nkb = -(-H // 64)
    return nkb >= 2 * S and tiles * S <= nsm and tiles <= mc[{2: 0, 4: 1, 8: 2}[S]]


def test_router_tc_shape_at_the_measured_sizes(lib):
    # H = 6144, E = 256: the shapes behind the timings in the design notes
    want = {256: (64, 8), 512: (80, 8), 1024: (64, 4), 2048: (128, 4), 4096: (112, 2), 8192: (112, 1)}
    for T, shape in want.items():
        assert _shape(T, 6144, 256) == shape, T


def test_router_tc_shape_is_feasible_and_minimal(lib):
    devices = [(GB300_SMS, GB300_CLUSTERS), (132, (66, 30, 14)), (20, (10, 4, 2)), (GB300_SMS, (0, 0, 0))]
    for T in [65, 100, 128, 255, 256, 300, 513, 777, 1024, 1500, 2048, 3000, 4096, 8192, 16384, 100000]:
        for H in [64, 512, 2056, 6144]:
            for E in [1, 72, 168, 256, 1024]:
                for nsm, mc in devices:
                    bnt, S = _shape(T, H, E, nsm, mc)
                    assert bnt in (64, 80, 96, 112, 128) and S in (1, 2, 4, 8)
                    assert bnt % S == 0  # every rank owns whole token rows
                    assert _feasible(T, H, E, nsm, mc, bnt, S), (T, H, E, nsm, bnt, S)
                    best = min(_modelled_us(T, H, E, nsm, b, s)
                               for b in (64, 80, 96, 112, 128) for s in (1, 2, 4, 8)
                               if _feasible(T, H, E, nsm, mc, b, s))
                    assert _modelled_us(T, H, E, nsm, bnt, S) <= best * 1.001, (T, H, E, nsm, bnt, S)
                    if mc == (0, 0, 0):
                        assert S == 1  # no cluster fits: no split-K


def test_router_tc_shape_argument_checks(lib):
    import ctypes
    b, s = ctypes.c_int32(), ctypes.c_int32()
    ok = dict(T=512, H=6144, E=256, nsm=152, mc2=76, mc4=36, mc8=15)

    def call(**kw):
        a = {**ok, **kw}
        return lib.moe_debug_router_tc_shape(a["T"], a["H"], a["E"], a["nsm"], a["mc2"], a["mc4"], a["mc8"],
                                             kw.get("pb", ctypes.byref(b)), kw.get("ps", ctypes.byref(s)))
    assert call() == L.MOE_OK
    for bad in [dict(T=0), dict(H=32), dict(E=0), dict(E=1025), dict(nsm=0), dict(mc4=-1), dict(pb=None),
                dict(ps=None)]:
        assert call(**bad) == L.MOE_ERR_INVALID_ARG, bad
