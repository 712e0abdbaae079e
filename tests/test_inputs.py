"""The seeded input generators (host only): the expert-grouped map layout is
a valid expanded-index map -- every (token, slot) row distinct and inside the
buffer -- with each expert's rows contiguous, tokens ascending, and groups
starting on the padding block."""

import numpy as np
import pytest

from moe_decode_layer_logits_gb300.inputs import expert_sorted_map, tail_case


@pytest.mark.parametrize("T,E,k,block", [(37, 20, 5, 8), (64, 256, 8, 0), (64, 256, 8, 128), (1, 4, 4, 3),
                                         (300, 168, 8, 64)])
def test_expert_sorted_map_layout(T, E, k, block):
    m, n_rows, experts = expert_sorted_map(np.random.default_rng(T * 7 + k), T, E, k, block)
    assert m.shape == (T, k) and m.dtype == np.int32
    assert len(np.unique(m)) == T * k and m.min() >= 0 and m.max() < n_rows
    assert all(len(set(row)) == k for row in experts)  # k distinct experts per token
    end = 0
    for e in range(E):
        tok, slot = np.nonzero(experts == e)
        if tok.size == 0:
            continue
        pos = m[tok, slot]
        order = np.argsort(pos)
        assert np.array_equal(np.diff(pos[order]), np.ones(tok.size - 1))  # contiguous
        assert np.all(np.diff(tok[order]) > 0)  # tokens ascending
        start = pos.min()
        assert start >= end and (block == 0 or start % block == 0)
        end = pos.max() + 1
    assert n_rows == (end if block == 0 else -(-end // block) * block)


def test_tail_case_expert_sorted():
    c = tail_case(64, 256, 256, 8, seed=1, map_layout="expert_sorted", expert_block=8)
    assert c["rows"].shape[0] == c["n_rows"] >= 64 * 8
    assert len(np.unique(c["map"])) == 64 * 8 and c["map"].max() < c["n_rows"]
    with pytest.raises(ValueError):
        tail_case(4, 64, 16, 2, seed=1, map_layout="by-expert")
