"""Host model of the warp top-k selection's candidate bound (no GPU).

The routing warp holds expert l + 32 s in lane l, slot s, as an
order-preserving key.  For E <= 256 and k <= 16 it takes, over G >= k groups
of adjacent lanes (G = 8 for k <= 8, 16 for k <= 16), the smallest of the
group maxima, tau; only the keys >= tau are ranked.  The argument: the G group
maxima are G >= k distinct keys >= tau, so the k-th largest key is >= tau, and
every key that beats a selected one is >= tau too, so ranking only the keys
>= tau gives the same top k as ranking all of them.  This model follows the
same lane, slot, group and list layout (places slot-major, lanes in order) and
checks it against a stable sort of the logits, on Gaussian, tied, all-equal,
signed-zero and narrow rows, every E up to 256 and every k up to 16; rows with
more than 64 candidates are the kernel's fallback and are counted, not ranked.
"""

import struct

import numpy as np
import pytest

CAP = 64


def order_key(f):
    """float -> uint32, monotone; -0 and +0 share the key of +0."""
    u = struct.unpack("<I", struct.pack("<f", float(f)))[0]
    if (u << 1) & 0xFFFFFFFF == 0:
        u = 0
    return (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)


def candidate_select(logits, k):
    """(ids in rank order, candidate count) or (None, count) past the cap."""
    E = len(logits)
    epl = (E + 31) // 32
    key = [[order_key(logits[l + 32 * s]) if l + 32 * s < E else 0 for s in range(epl)] for l in range(32)]
    gm = [max(key[l]) for l in range(32)]
    d = 1
    while d < 32 and 32 // (2 * d) >= k:  # groups of 2d lanes while they number >= k
        gm = [max(gm[l], gm[l ^ d]) for l in range(32)]
        d <<= 1
    groups = 32 // d
    assert groups >= k
    tau = min(gm)
    places = []
    for s in range(epl):  # slot-major, lanes in order: ascending expert
        for l in range(32):
            if key[l][s] >= tau:
                places.append((key[l][s] << 32) | (0xFFFFFFFF - (l + 32 * s)))
    n = len(places)
    assert n >= k
    if n > CAP:
        return None, n
    chosen = [None] * k
    for v in places:
        r = sum(1 for u in places if u > v)  # distinct values: ranks 0 .. n-1
        if r < k:
            assert chosen[r] is None
            chosen[r] = v
    return [0xFFFFFFFF - (v & 0xFFFFFFFF) for v in chosen], n


def reference(logits, k):
    # stable sort by value, descending; -0 == +0; lower expert first among equals
    return sorted(range(len(logits)), key=lambda i: (-(float(logits[i]) + 0.0), i))[:k]


def rows(rng, E):
    yield (rng.standard_normal(E) * 1.57).astype(np.float32)
    yield rng.integers(-2, 3, E).astype(np.float32)
    yield np.full(E, 0.5, np.float32)
    yield np.where(rng.random(E) < 0.5, -0.0, 0.0).astype(np.float32)
    yield (5.0 + 1e-3 * rng.standard_normal(E)).astype(np.float32)
    yield -np.abs(rng.standard_normal(E)).astype(np.float32)


@pytest.mark.parametrize("E", [1, 9, 33, 64, 72, 100, 168, 200, 256])
def test_candidate_bound_matches_a_stable_sort(E):
    rng = np.random.default_rng(E)
    ranked = fallback = 0
    for k in range(1, min(E, 16) + 1):
        for x in rows(rng, E):
            ids, n = candidate_select(x, k)
            if ids is None:
                fallback += 1
                continue
            ranked += 1
            assert ids == reference(x, k), (E, k, x)
    assert ranked > 0
    # Gaussian rows at k = 8, E = 256 rank about 20 candidates: the fallback is for ties
    if E == 256:
        counts = [candidate_select((rng.standard_normal(E) * 1.57).astype(np.float32), 8)[1] for _ in range(200)]
        assert 10 <= np.mean(counts) <= 40 and np.mean(np.array(counts) > CAP) < 0.02


def test_all_equal_rows_overflow_the_list():
    # every key meets tau: more candidates than the list holds, so the kernel
    # takes the sorted heads for such rows
    ids, n = candidate_select(np.zeros(256, np.float32), 8)
    assert ids is None and n == 256
