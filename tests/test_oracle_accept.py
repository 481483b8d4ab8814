"""Pins of the oracle's greedy verification and unpack (CPU only).

* Hand-worked examples (tests/golden/accept_examples.json) with planted ties.
* The argmax equals numpy's argmax (first maximum) on the widened bf16 rows.
* Acceptance equals plain greedy decoding: stepping along every beam, and the
  greedy walk from the shared anchor, with logits defined per prefix so the
  brute force never sees the oracle's packing.
* Unpack equals the torch.gather of the PyTorch listing in the NVIDIA blog
  "ReDrafter in TensorRT-LLM" (section "Implementing in-Engine Validation and
  Drafting").
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tests.pins import bf16_round, bf16_to_f64, greedy_per_beam, greedy_walk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_accept_golden(case):
    g = _golden()
    V, P = g["vocab"], g["P_max"]
    logits = np.full((1, P, V), -1.0, np.float32)
    for row, entries in case["rows"].items():
        for col, val in entries.items():
            logits[0, int(row), int(col)] = val
    out = oracle.oracle_greedy_accept(bf16_round(logits), np.array(g["beams"], np.int32),
                                      np.array(g["unpacker"], np.int32),
                                      np.array(g["packed_len"], np.int32))
    for key in ("argmax", "accept_len", "best_beam", "n_accepted", "out_tokens"):
        np.testing.assert_array_equal(out[key], np.array(case[key]), err_msg=key)


@pytest.mark.parametrize("seed", range(4))
def test_argmax_matches_numpy_first_maximum(seed):
    rng = np.random.default_rng(seed)
    B, P, V = 2, 5, 3000
    x = (rng.standard_normal((B, P, V)) * 2).astype(np.float32)
    x[0, 1, [7, 2999]] = 50.0                      # planted tie, low and high index
    x[1, 0, [0, 1]] = 50.0
    bits = bf16_round(x)                           # bf16 rounding makes more ties
    beams = np.zeros((B, 1, 1), np.int32)
    up = np.zeros((B, 1, 1), np.int32)
    out = oracle.oracle_greedy_accept(bits, beams, up, np.array([P, 3], np.int32))
    ref = np.argmax(bf16_to_f64(bits), axis=-1)
    np.testing.assert_array_equal(out["argmax"][0], ref[0])
    np.testing.assert_array_equal(out["argmax"][1, :3], ref[1, :3])
    assert (out["argmax"][1, 3:] == -1).all()
    assert out["argmax"][0, 1] == 7 and out["argmax"][1, 0] == 0


@pytest.mark.parametrize("seed", range(10))
def test_accept_equals_greedy_decoding(seed):
    rng = np.random.default_rng(100 + seed)
    B, W, L, V = 3, int(rng.integers(1, 7)), int(rng.integers(1, 6)), 6
    beams = rng.integers(0, 3, size=(B, W, L)).astype(np.int32)
    beams[:, :, 0] = beams[:, :1, 0]                # shared anchor
    P = W * L
    pk = oracle.oracle_pack(beams)
    row_cache = {}

    def row_of(b, pre):                            # logits per prefix, with frequent ties
        key = (b,) + pre
        if key not in row_cache:
            r = np.random.default_rng(hash(key) & 0xFFFFFFFF).integers(0, 3, size=V)
            row_cache[key] = r.astype(np.float32)
        return row_cache[key]

    logits = np.zeros((B, P, V), np.float32)
    for b in range(B):
        for p in range(pk["packed_len"][b]):
            f = pk["packer"][b, p]
            logits[b, p] = row_of(b, tuple(int(x) for x in beams[b, f // L, : f % L + 1]))
    out = oracle.oracle_greedy_accept(bf16_round(logits), beams, pk["unpacker"],
                                      pk["packed_len"])
    for b in range(B):
        def greedy_of(pre):
            return int(np.argmax(row_of(b, pre)))
        acc, best, emitted = greedy_per_beam(beams[b], greedy_of)
        np.testing.assert_array_equal(out["accept_len"][b], acc)
        assert out["best_beam"][b] == best
        a = out["n_accepted"][b]
        assert a == acc[best]
        np.testing.assert_array_equal(out["out_tokens"][b, : a + 1], emitted)
        assert (out["out_tokens"][b, a + 1:] == -1).all()
        assert greedy_walk(beams[b], greedy_of) == emitted


@pytest.mark.parametrize("dtype", [np.uint16, np.float32, np.int32])
def test_unpack_equals_torch_gather(dtype):
    rng = np.random.default_rng(5)
    B, P, W, L, D = 3, 7, 4, 3, 10
    packed = rng.integers(0, 60000, size=(B, P, D)).astype(dtype)
    unpacker = rng.integers(0, P, size=(B, W, L)).astype(np.int32)
    got = oracle.oracle_unpack(packed, unpacker)
    # the PyTorch listing: gather along dim 1 with the unpacker expanded over the last dim
    t = torch.from_numpy(packed.astype(np.int64))
    idx = torch.from_numpy(unpacker.astype(np.int64)).view(B, W * L, 1).expand(-1, -1, D)
    ref = torch.gather(t, 1, idx).reshape(B, W, L, -1).numpy().astype(dtype)
    np.testing.assert_array_equal(got, ref)
