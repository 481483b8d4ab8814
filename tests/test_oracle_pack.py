"""Pins of the oracle's prefix dedup (CPU only).

The pack is pinned by hand-worked examples (tests/golden/pack_examples.json),
closed forms (identical beams pack to L nodes, beams with distinct anchors to
W*L) and a brute-force count of distinct prefix tuples.
"""
import json
import os

import numpy as np
import pytest

import oracle
from tests.pins import prefix_tuples

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pack_examples.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_pack_golden(case):
    beams = np.array(case["beams"], np.int32)
    out = oracle.oracle_pack(beams)
    for key in ("packed_len", "tokens", "packer", "unpacker", "depth"):
        np.testing.assert_array_equal(out[key], np.array(case[key]), err_msg=key)
    np.testing.assert_array_equal(out["mask"], np.array(case["mask"], np.uint32))


def test_identical_beams_pack_to_L():
    beams = np.tile(np.array([[3, 1, 4, 1, 5]], np.int32), (6, 1))[None]
    out = oracle.oracle_pack(beams)
    assert out["packed_len"][0] == 5
    assert (out["unpacker"][0] == np.arange(5)[None, :]).all()


def test_distinct_anchors_pack_to_WL_and_mask_crosses_words():
    # W=2, L=20 with distinct anchors: node (w, i) is packed index w*L+i and its
    # ancestors are w*L .. w*L+i, so row 39 has bits 20..39 (two 32-bit words).
    W, L = 2, 20
    beams = np.stack([np.arange(L), np.arange(L) + 100]).astype(np.int32)[None]
    out = oracle.oracle_pack(beams)
    assert out["packed_len"][0] == W * L
    np.testing.assert_array_equal(out["unpacker"][0], np.arange(W * L).reshape(W, L))
    np.testing.assert_array_equal(out["mask"][0, 39], np.array([0xFFF00000, 0xFF], np.uint32))
    np.testing.assert_array_equal(out["mask"][0, 19], np.array([0x000FFFFF, 0], np.uint32))
    np.testing.assert_array_equal(out["mask"][0, 20], np.array([1 << 20, 0], np.uint32))


def _check_invariants(beams, out):
    B, W, L = beams.shape
    for b in range(B):
        P = int(out["packed_len"][b])
        pref = prefix_tuples(beams[b])
        # P = number of distinct prefixes = trie node count (brute force)
        assert P == len(pref)
        # every packed node is a distinct prefix, in first-occurrence order
        pk = out["packer"][b, :P]
        got = [tuple(int(x) for x in beams[b, f // L, : f % L + 1]) for f in pk]
        assert got == pref
        assert (np.diff(pk) > 0).all()
        up = out["unpacker"][b]
        assert (out["tokens"][b][up] == beams[b]).all()
        assert (up <= np.arange(W * L).reshape(W, L)).all()
        assert (out["depth"][b, :P] == pk % L).all()
        for p in range(P):
            row = out["mask"][b, p]
            bits = [k for k in range(out["mask"].shape[2] * 32) if row[k // 32] >> (k % 32) & 1]
            assert len(bits) == out["depth"][b, p] + 1
            assert p in bits and max(bits) == p
        # mask of a node is contained in the mask of each child
        for w in range(W):
            for i in range(1, L):
                par, ch = out["mask"][b, up[w, i - 1]], out["mask"][b, up[w, i]]
                assert ((par & ch) == par).all()
        assert (out["packer"][b, P:] == -1).all() and (out["mask"][b, P:] == 0).all()


@pytest.mark.parametrize("seed", range(12))
def test_pack_random_tries_invariants(seed):
    rng = np.random.default_rng(seed)
    W, L = int(rng.integers(1, 9)), int(rng.integers(1, 8))
    vocab = int(rng.integers(2, 5))           # small vocab: many shared prefixes
    beams = rng.integers(0, vocab, size=(3, W, L)).astype(np.int32)
    _check_invariants(beams, oracle.oracle_pack(beams))


def test_pack_rejects_too_small_capacity():
    beams = np.arange(8, dtype=np.int32).reshape(1, 2, 4)
    with pytest.raises(ValueError):
        oracle.oracle_pack(beams, P_cap=7)
