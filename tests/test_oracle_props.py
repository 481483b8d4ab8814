"""Property tests of the oracle's pack and acceptance on random tries (CPU only).

Uses hypothesis where installed.  The invariants are the ones the pages fix:
the packed length is the number of distinct prefixes (the trie's node count),
identical beams pack to L nodes, beams with pairwise distinct anchors to W*L,
and every beam position maps back to its own token.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from tests.pins import prefix_tuples  # noqa: E402


@st.composite
def beam_sets(draw):
    W = draw(st.integers(1, 8))
    L = draw(st.integers(1, 6))
    vocab = draw(st.integers(1, 4))
    flat = draw(st.lists(st.integers(0, vocab - 1), min_size=W * L, max_size=W * L))
    return np.array(flat, np.int32).reshape(1, W, L)


@settings(max_examples=150, deadline=None)
@given(beam_sets())
def test_packed_length_is_trie_node_count(beams):
    out = oracle.oracle_pack(beams)
    P = int(out["packed_len"][0])
    assert P == len(prefix_tuples(beams[0]))
    up = out["unpacker"][0]
    assert (out["tokens"][0][up] == beams[0]).all()
    # equal prefixes <=> equal packed index
    W, L = beams.shape[1:]
    for w1 in range(W):
        for w2 in range(W):
            for i in range(L):
                same = (beams[0, w1, : i + 1] == beams[0, w2, : i + 1]).all()
                assert same == (up[w1, i] == up[w2, i])


@settings(max_examples=50, deadline=None)
@given(st.integers(1, 8), st.integers(1, 6), st.integers(0, 1000))
def test_identical_and_distinct_extremes(W, L, seed):
    rng = np.random.default_rng(seed)
    one = rng.integers(0, 50, size=L).astype(np.int32)
    same = np.tile(one, (W, 1))[None]
    assert oracle.oracle_pack(same)["packed_len"][0] == L
    distinct = rng.integers(0, 50, size=(W, L)).astype(np.int32)
    distinct[:, 0] = np.arange(W) + 1000
    assert oracle.oracle_pack(distinct[None])["packed_len"][0] == W * L
