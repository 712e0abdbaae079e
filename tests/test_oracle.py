"""Pins for the FP64 oracle: it is checked against things other than itself.

Each check uses a fact the pages or mathematics fix -- hand-derived closed
forms (tests/golden), a library RMSNorm, exact integer arithmetic, brute-force
enumeration and exhaustive BF16 rounding -- and the last group plants
plausible mistakes in a private copy of the oracle to show that some pin
fails for each of them.
"""

import importlib.util
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from moe_decode_layer_logits_gb300.inputs import tail_case, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line)
    return out


def _eval(expr):
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp, "sqrt": math.sqrt}))


# ---------------------------------------------------------------------------
# BF16 rounding
# ---------------------------------------------------------------------------

def check_bf16_golden(o):
    for line in _golden_rows("bf16_rounding_cases.txt"):
        hx, bits = line.split()[:2]
        got = int(o.f64_to_bf16_bits(np.array([float.fromhex(hx)]))[0])
        assert got == int(bits, 16), (hx, hex(got), bits)


def test_bf16_golden_cases():
    check_bf16_golden(O)


def test_bf16_roundtrip_exhaustive():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_bits_to_f64(b)
    keep = ~np.isnan(v)
    assert np.array_equal(O.f64_to_bf16_bits(v[keep]), b[keep])
    assert np.all(np.isnan(O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.array([np.nan])))))


def check_bf16_midpoints(o):
    # every pair of neighbouring finite positive BF16 values, and their mirror
    b = np.arange(0, 0x7F7F, dtype=np.uint16)
    lo = o.bf16_bits_to_f64(b)
    hi = o.bf16_bits_to_f64(b + 1)
    mid = (lo + hi) / 2.0  # exact in double
    even = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(o.f64_to_bf16_bits(mid), even)
    assert np.array_equal(o.f64_to_bf16_bits(np.nextafter(mid, np.inf)), (b + 1).astype(np.uint16))
    assert np.array_equal(o.f64_to_bf16_bits(np.nextafter(mid, -np.inf)), b)
    assert np.array_equal(o.f64_to_bf16_bits(-mid), even | np.uint16(0x8000))


def test_bf16_midpoints_all():
    check_bf16_midpoints(O)


def test_bf16_agrees_with_binary32_bit_rounding():
    # For values that binary32 holds exactly, rounding the binary32 bit
    # pattern with integer arithmetic is an independent definition of RNE.
    rng = np.random.default_rng(7)
    f = (rng.standard_normal(200000) * np.exp(rng.uniform(-60, 60, 200000))).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    low = u & np.uint64(0xFFFF)
    up = u >> np.uint64(16)
    half = np.uint64(0x8000)
    up = np.where((low > half) | ((low == half) & (up & np.uint64(1) == 1)), up + 1, up)
    assert np.array_equal(O.f64_to_bf16_bits(f.astype(np.float64)), up.astype(np.uint16))


def test_bf16_ulp_values():
    assert O.bf16_ulp(1.0) == 2.0 ** -7
    assert O.bf16_ulp(1.99) == 2.0 ** -7
    assert O.bf16_ulp(0.75) == 2.0 ** -8
    assert O.bf16_ulp(-3.0) == 2.0 ** -6
    assert O.bf16_ulp(0.0) == 2.0 ** -133


# ---------------------------------------------------------------------------
# Router logits
# ---------------------------------------------------------------------------

def check_router_integers(o):
    # small integers are exact in BF16; the int64 product is an independent
    # exact result, and the non-square shapes catch a transposed operand.
    rng = np.random.default_rng(11)
    T, E, H = 5, 24, 2048
    xi = rng.integers(-16, 17, size=(T, H))
    wi = rng.integers(-16, 17, size=(E, H))
    L, A = o.router_logits(to_bf16_bits(xi), to_bf16_bits(wi))
    assert L.shape == (T, E)
    assert np.array_equal(L, (xi @ wi.T).astype(np.float64))
    assert np.array_equal(A, (np.abs(xi) @ np.abs(wi).T).astype(np.float64))


def test_router_small_integers_exact():
    check_router_integers(O)


def test_router_one_hot_picks_a_column():
    rng = np.random.default_rng(12)
    E, H = 16, 64
    w = to_bf16_bits(rng.standard_normal((E, H)) * 0.02)
    x = np.zeros((3, H))
    x[0, 5] = 1.0
    x[1, 63] = 1.0
    x[2, 0] = -2.0
    L, _ = O.router_logits(to_bf16_bits(x), w)
    wv = O.bf16_bits_to_f64(w)
    assert np.array_equal(L[0], wv[:, 5])
    assert np.array_equal(L[1], wv[:, 63])
    assert np.array_equal(L[2], -2.0 * wv[:, 0])


# ---------------------------------------------------------------------------
# Top-k routing
# ---------------------------------------------------------------------------

def _brute_topk(row, k):
    E = len(row)
    best = None
    for sub in itertools.combinations(range(E), k):  # ascending tuples
        s = sum(row[i] for i in sub)  # integer-valued: exact
        if best is None or s > best[0]:
            best = (s, sub)
    chosen = best[1]  # first max-sum subset in lexicographic order
    return sorted(chosen, key=lambda i: (-row[i], i))


def _loop_topk(row, k):
    taken = set()
    out = []
    for _ in range(k):
        bi = None
        for i, v in enumerate(row):
            if i in taken:
                continue
            if bi is None or v > row[bi]:
                bi = i
        taken.add(bi)
        out.append(bi)
    return out


def check_topk_bruteforce(o):
    rng = np.random.default_rng(13)
    for E in range(1, 9):
        for _ in range(40):
            row = rng.integers(-3, 4, size=E).astype(np.float32)
            for k in range(1, E + 1):
                ids, _, _ = o.topk_route(row[None, :], k, 1.0)
                want = _brute_topk(list(row), k)
                assert list(ids[0]) == want, (row, k)
                assert list(ids[0]) == _loop_topk(list(row), k)


def test_topk_bruteforce_small():
    check_topk_bruteforce(O)


def check_topk_golden(o):
    for line in _golden_rows("topk_cases.txt"):
        name, lg, k, scale, ids, ws = [p.strip() for p in line.split("|")]
        logits = np.array([[float(v) for v in lg.split()]], dtype=np.float32)
        gi, gw, g64 = o.topk_route(logits, int(k), float(scale))
        assert list(gi[0]) == [int(v) for v in ids.split()], name
        want = np.array([_eval(e) for e in ws.split()])
        assert np.allclose(g64[0], want, rtol=1e-14, atol=0), (name, g64, want)
        assert np.array_equal(gw[0], want.astype(np.float32)), name


def test_topk_golden_cases():
    check_topk_golden(O)


def check_softmax_identities(o):
    rng = np.random.default_rng(14)
    lg = (rng.standard_normal((64, 256)) * 1.6).astype(np.float32)
    for k, scale in [(1, 2.5), (4, 1.0), (8, 2.5), (16, 0.7)]:
        ids, w, w64 = o.topk_route(lg, k, scale)
        assert np.allclose(w64.sum(axis=1), scale, rtol=1e-13)
        sel = np.take_along_axis(lg.astype(np.float64), ids.astype(np.int64), axis=1)
        # ratios w_i / w_0 = exp(l_i - l_0)
        assert np.allclose(w64 / w64[:, :1], np.exp(sel - sel[:, :1]), rtol=1e-13)
        # descending logits, k largest: every unselected logit <= the k-th
        assert np.all(np.diff(sel, axis=1) <= 0)
        mask = np.ones_like(lg, dtype=bool)
        np.put_along_axis(mask, ids.astype(np.int64), False, axis=1)
        rest = np.where(mask, lg.astype(np.float64), -np.inf).max(axis=1)
        assert np.all(rest <= sel[:, -1])
        assert np.array_equal(w, w64.astype(np.float32))
    ids, w, _ = o.topk_route(lg, 1, 2.5)
    assert np.all(w == np.float32(2.5))


def test_softmax_identities():
    check_softmax_identities(O)


# ---------------------------------------------------------------------------
# Finalize + shared add + residual add + RMSNorm
# ---------------------------------------------------------------------------

def _torch_rms_norm(r64, gamma, eps):
    t = torch.from_numpy(np.ascontiguousarray(r64))
    g = torch.from_numpy(gamma.astype(np.float64))
    return torch.nn.functional.rms_norm(t, (t.shape[-1],), g, eps).numpy()


def check_rmsnorm_golden(o):
    for line in _golden_rows("rmsnorm_closed_forms.txt"):
        name, rv, gv, eps, want = [p.strip() for p in line.split("|")]
        r = np.array([[float(v) for v in rv.split()]])
        g = np.array([float(v) for v in gv.split()], dtype=np.float32)
        rr, normed = o.add_rmsnorm(to_bf16_bits(r), np.zeros_like(r), g, float(eps))
        assert np.array_equal(rr, r), name
        wv = np.array([_eval(e) for e in want.split()])
        assert np.allclose(normed[0], wv, rtol=1e-15, atol=0), (name, normed, wv)


def test_rmsnorm_golden_cases():
    check_rmsnorm_golden(O)


def check_single_route_is_library_rmsnorm(o):
    # k = 1, weight 1, no shared expert: the tail is add + RMSNorm of one row
    c = tail_case(6, 512, 16, 1, seed=21, scale=1.0, shared=False, router=False)
    w = np.ones((6, 1), dtype=np.float32)
    out = o.finalize_add_rmsnorm(c["rows"], c["map"], w, None, None, c["residual"], c["gamma"], c["eps"])
    r = O.bf16_bits_to_f64(c["residual"]) + O.bf16_bits_to_f64(c["rows"])[c["map"][:, 0]]
    assert np.array_equal(out["r"], r)
    ref = _torch_rms_norm(r, c["gamma"], c["eps"])
    assert np.allclose(out["normed64"], ref, rtol=1e-13, atol=1e-15)


def test_single_route_reduces_to_add_rmsnorm():
    check_single_route_is_library_rmsnorm(O)


def check_zero_rows_is_plain_add_rmsnorm(o):
    c = tail_case(5, 384, 16, 4, seed=22, shared=True, router=False)
    zero_rows = np.zeros_like(c["rows"])
    out = o.finalize_add_rmsnorm(zero_rows, c["map"], c["topk_w"], c["shared"], None,
                                 c["residual"], c["gamma"], c["eps"])
    r = O.bf16_bits_to_f64(c["residual"]) + O.bf16_bits_to_f64(c["shared"])
    assert np.array_equal(out["r"], r)
    assert np.allclose(out["normed64"], _torch_rms_norm(r, c["gamma"], c["eps"]), rtol=1e-13, atol=1e-15)
    # k = 0 means no routed part at all
    out0 = o.finalize_add_rmsnorm(c["rows"], np.zeros((5, 0), np.int32), np.zeros((5, 0), np.float32),
                                  c["shared"], None, c["residual"], c["gamma"], c["eps"])
    assert np.array_equal(out0["residual_out"], out["residual_out"])
    assert np.array_equal(out0["normed"], out["normed"])


def test_zero_rows_reduce_to_add_rmsnorm():
    check_zero_rows_is_plain_add_rmsnorm(O)


def check_permutation_invariance(o):
    c = tail_case(7, 256, 16, 8, seed=23, router=False)
    base = o.finalize_add_rmsnorm(c["rows"], c["map"], c["topk_w"], c["shared"], None,
                                  c["residual"], c["gamma"], c["eps"])
    rng = np.random.default_rng(5)
    perm = rng.permutation(c["rows"].shape[0])  # new position of each old row
    rows2 = np.empty_like(c["rows"])
    rows2[perm] = c["rows"]
    map2 = perm[c["map"]].astype(np.int32)
    moved = o.finalize_add_rmsnorm(rows2, map2, c["topk_w"], c["shared"], None,
                                   c["residual"], c["gamma"], c["eps"])
    assert np.array_equal(moved["r"], base["r"])
    assert np.array_equal(moved["normed"], base["normed"])


def test_row_buffer_permutation_invariance():
    check_permutation_invariance(O)


def check_constant_rows_closed_form(o):
    # rows[map[t, j]] = c_j everywhere, residual = 0, no shared: r = sum_j w_j c_j
    H, k = 64, 3
    cvals = np.array([0.5, -1.25, 2.0])
    rows = to_bf16_bits(np.repeat(cvals[:, None], H, axis=1))
    mp = np.array([[0, 1, 2], [2, 0, 1]], dtype=np.int32)
    w = np.array([[0.25, 0.5, 1.0], [1.0, 0.125, 0.75]], dtype=np.float32)
    res = np.zeros((2, H), dtype=np.uint16)
    g = np.linspace(0.5, 1.5, H).astype(np.float32)
    eps = 1e-6
    out = o.finalize_add_rmsnorm(rows, mp, w, None, None, res, g, eps)
    for t in range(2):
        cc = float(np.dot(w[t].astype(np.float64), cvals[mp[t]]))
        assert np.all(out["r"][t] == cc)
        assert np.allclose(out["normed64"][t], np.sign(cc) * abs(cc) / math.sqrt(cc * cc + eps) * g.astype(np.float64),
                           rtol=1e-15)


def test_constant_rows_closed_form():
    check_constant_rows_closed_form(O)


def check_rms_invariant(o):
    c = tail_case(9, 1024, 16, 8, seed=24, router=False, s=4.0)
    out = o.finalize_add_rmsnorm(c["rows"], c["map"], c["topk_w"], c["shared"], None,
                                 c["residual"], c["gamma"], 0.0)
    pre = out["normed64"] / c["gamma"].astype(np.float64)[None, :]
    assert np.allclose(np.sqrt(np.mean(pre * pre, axis=1)), 1.0, rtol=1e-12)
    eps = 0.5
    out = o.finalize_add_rmsnorm(c["rows"], c["map"], c["topk_w"], c["shared"], None,
                                 c["residual"], c["gamma"], eps)
    pre = out["normed64"] / c["gamma"].astype(np.float64)[None, :]
    ms = np.mean(out["r"] ** 2, axis=1)
    assert np.allclose(np.sqrt(np.mean(pre * pre, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-12)


def test_rms_invariant():
    check_rms_invariant(O)


def check_partials(o):
    c = tail_case(4, 256, 16, 8, seed=25, router=False, R=1)
    p = c["partials"]
    kz = (np.zeros((4, 0), np.int32), np.zeros((4, 0), np.float32))
    a = o.finalize_add_rmsnorm(c["rows"], *kz, None, p, c["residual"], c["gamma"], c["eps"])
    b = o.finalize_add_rmsnorm(c["rows"], *kz, p[0], None, c["residual"], c["gamma"], c["eps"])
    assert np.array_equal(a["r"], b["r"])
    # R partials sum elementwise; their sum is linear
    c4 = tail_case(3, 128, 16, 8, seed=26, router=False, R=4)
    d = o.finalize_add_rmsnorm(c4["rows"], np.zeros((3, 0), np.int32), np.zeros((3, 0), np.float32),
                               None, c4["partials"], c4["residual"], c4["gamma"], c4["eps"])
    want = O.bf16_bits_to_f64(c4["residual"]) + O.bf16_bits_to_f64(c4["partials"]).sum(axis=0)
    assert np.allclose(d["r"], want, rtol=1e-15, atol=0)


def test_partials_match_shared_and_sum():
    check_partials(O)


def check_composition(o):
    # vllm pull 62174, Validation: fused == finalize, then shared add, then
    # RMSNorm(residual + reduced)
    c = tail_case(6, 512, 32, 8, seed=27, router=False)
    fused = o.finalize_add_rmsnorm(c["rows"], c["map"], c["topk_w"], c["shared"], None,
                                   c["residual"], c["gamma"], c["eps"])
    y = o.shared_add(o.moe_finalize(c["rows"], c["map"], c["topk_w"]), c["shared"])
    r, normed = o.add_rmsnorm(c["residual"], y, c["gamma"], c["eps"])
    assert np.array_equal(fused["r"], r)
    assert np.array_equal(fused["normed64"], normed)
    assert np.array_equal(fused["normed"], o.f64_to_bf16_bits(normed))
    assert np.all(fused["abs_terms"] >= np.abs(fused["r"]) * (1 - 1e-15))


def test_composition_contract():
    check_composition(O)


def test_weighted_sum_linear_in_weights():
    c = tail_case(3, 128, 16, 4, seed=28, router=False)
    a = O.moe_finalize(c["rows"], c["map"], c["topk_w"])
    b = O.moe_finalize(c["rows"], c["map"], (2.0 * c["topk_w"]).astype(np.float32))
    assert np.array_equal(b, 2.0 * a)
    rows = O.bf16_bits_to_f64(c["rows"])
    t, j = 2, 3
    one = np.zeros_like(c["topk_w"])
    one[t, j] = 1.0
    assert np.array_equal(O.moe_finalize(c["rows"], c["map"], one)[t], rows[c["map"][t, j]])


def test_tail_fused_is_route_then_tail():
    c = tail_case(5, 256, 32, 4, seed=29, router=False, logits=True)
    f = O.tail_fused(c["logits"], 4, 2.5, c["rows"], c["map"], c["shared"], c["residual"], c["gamma"], c["eps"])
    ids, w, _ = O.topk_route(c["logits"], 4, 2.5)
    assert np.array_equal(f["ids"], ids)
    t = O.finalize_add_rmsnorm(c["rows"], c["map"], w, c["shared"], None, c["residual"], c["gamma"], c["eps"])
    assert np.array_equal(f["normed"], t["normed"])
    assert np.array_equal(f["residual_out"], t["residual_out"])


# ---------------------------------------------------------------------------
# Planted mistakes: each mutant copy of the oracle must fail at least one pin
# ---------------------------------------------------------------------------

ALL_PINS = [check_bf16_golden, check_bf16_midpoints, check_router_integers, check_topk_bruteforce,
            check_topk_golden, check_softmax_identities, check_rmsnorm_golden,
            check_single_route_is_library_rmsnorm, check_zero_rows_is_plain_add_rmsnorm,
            check_permutation_invariance, check_constant_rows_closed_form, check_rms_invariant,
            check_partials, check_composition]


def _fresh_oracle():
    path = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "oracle.py")
    spec = importlib.util.spec_from_file_location("oracle_mutant", path)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _mut_eps_outside_sqrt(m):
    def add_rmsnorm(residual_bits, y, gamma, eps):
        r = m.bf16_bits_to_f64(residual_bits) + y
        ms = np.mean(r * r, axis=1, keepdims=True)
        return r, r / (np.sqrt(ms) + eps) * np.asarray(gamma, np.float64)[None, :]
    m.add_rmsnorm = add_rmsnorm


def _mut_sum_not_mean(m):
    def add_rmsnorm(residual_bits, y, gamma, eps):
        r = m.bf16_bits_to_f64(residual_bits) + y
        ms = np.sum(r * r, axis=1, keepdims=True)
        return r, r / np.sqrt(ms + eps) * np.asarray(gamma, np.float64)[None, :]
    m.add_rmsnorm = add_rmsnorm


def _mut_drop_shared(m):
    m.shared_add = lambda routed, shared_bits: np.asarray(routed, dtype=np.float64)


def _mut_ignore_map(m):
    def moe_finalize(rows_bits, row_map, topk_w):
        rows = m.bf16_bits_to_f64(rows_bits)
        T, k = np.asarray(row_map).shape
        w = np.asarray(topk_w, np.float64)
        out = np.zeros((T, rows.shape[1]))
        for j in range(k):
            out += w[:, j:j + 1] * rows[np.arange(T) * k + j]
        return out
    m.moe_finalize = moe_finalize


def _mut_softmax_all(m):
    def topk_route(logits_f32, k, scale):
        lg = np.asarray(logits_f32, np.float32).astype(np.float64)
        ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
        ex = np.exp(lg - lg.max(axis=1, keepdims=True))
        w64 = scale * np.take_along_axis(ex, ids, 1) / ex.sum(axis=1, keepdims=True)
        return ids.astype(np.int32), w64.astype(np.float32), w64
    m.topk_route = topk_route


def _mut_ties_high_index(m):
    def topk_route(logits_f32, k, scale):
        lg = np.asarray(logits_f32, np.float32).astype(np.float64)
        E = lg.shape[1]
        rev = np.argsort(-lg[:, ::-1], axis=1, kind="stable")
        ids = (E - 1 - rev)[:, :k]
        sel = np.take_along_axis(lg, ids, 1)
        ex = np.exp(sel - sel[:, :1])
        w64 = scale * ex / ex.sum(axis=1, keepdims=True)
        return ids.astype(np.int32), w64.astype(np.float32), w64
    m.topk_route = topk_route


def _mut_transposed_router(m):
    def router_logits(x_bits, w_bits):
        x = m.bf16_bits_to_f64(x_bits)
        w = m.bf16_bits_to_f64(w_bits)
        H = x.shape[1]
        return x @ w.reshape(H, -1), np.abs(x) @ np.abs(w).reshape(H, -1)
    m.router_logits = router_logits


def _mut_round_via_float(m):
    orig = m.f64_to_bf16_bits

    def f64_to_bf16_bits(x):
        return orig(np.asarray(x, np.float64).astype(np.float32).astype(np.float64))
    m.f64_to_bf16_bits = f64_to_bf16_bits


def _mut_truncate(m):
    def f64_to_bf16_bits(x):
        f = np.asarray(x, np.float64).astype(np.float32)
        return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    m.f64_to_bf16_bits = f64_to_bf16_bits


def _mut_norm_rounded_residual(m):
    def add_rmsnorm(residual_bits, y, gamma, eps):
        r = m.bf16_bits_to_f64(residual_bits) + y
        rq = m.bf16_bits_to_f64(m.f64_to_bf16_bits(r))
        ms = np.mean(rq * rq, axis=1, keepdims=True)
        return r, rq / np.sqrt(ms + eps) * np.asarray(gamma, np.float64)[None, :]
    m.add_rmsnorm = add_rmsnorm


MUTANTS = {
    "eps_outside_sqrt": _mut_eps_outside_sqrt,
    "sum_not_mean": _mut_sum_not_mean,
    "drop_shared": _mut_drop_shared,
    "ignore_map": _mut_ignore_map,
    "softmax_over_all_experts": _mut_softmax_all,
    "ties_to_high_index": _mut_ties_high_index,
    "transposed_router": _mut_transposed_router,
    "double_rounding_via_float": _mut_round_via_float,
    "truncate_not_round": _mut_truncate,
    "norm_of_rounded_residual": _mut_norm_rounded_residual,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = _fresh_oracle()
    MUTANTS[name](m)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(m)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
