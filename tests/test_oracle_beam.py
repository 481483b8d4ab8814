"""Pins of the oracle's beam-search step (CPU only).

* A single beam reduces to greedy decoding: the best candidate is the argmax
  token and its score is log softmax at that token (closed form).
* Brute force: every candidate's log-probability with numpy's log-sum-exp,
  sorted with lexsort (score descending, flat index ascending), equals the
  oracle's selection.
* From a single live beam (the anchor) the W new beams are the W most likely
  next tokens, in order.
"""
import numpy as np
import pytest

import oracle
from tests.pins import bf16_round, bf16_to_f64


def _logits(rng, B, W, V, ties=False):
    x = (rng.standard_normal((B, W, V)) * 2).astype(np.float32)
    if ties:
        x = np.round(x)          # many exact ties
    return bf16_round(x)


def test_single_beam_is_greedy():
    rng = np.random.default_rng(0)
    lg = _logits(rng, 3, 1, 500)
    s0 = np.array([[0.0], [-1.5], [2.0]])
    out = oracle.oracle_beam_search_step(lg, s0, np.full((3, 1, 2), 7, np.int32))
    x = bf16_to_f64(lg)
    for b in range(3):
        v = int(np.argmax(x[b, 0]))
        lse = np.log(np.exp(x[b, 0] - x[b, 0].max()).sum()) + x[b, 0].max()
        assert out["beams"][b, 0, 2] == v and out["parent"][b, 0] == 0
        assert (out["beams"][b, 0, :2] == 7).all()
        np.testing.assert_allclose(out["scores"][b, 0], s0[b, 0] + x[b, 0, v] - lse, rtol=1e-13)


@pytest.mark.parametrize("seed,W,V,ties", [(1, 4, 300, False), (2, 8, 1000, True),
                                           (3, 5, 64, True), (4, 3, 2000, False)])
def test_brute_force_selection(seed, W, V, ties):
    rng = np.random.default_rng(seed)
    B, t = 4, 3
    lg = _logits(rng, B, W, V, ties)
    scores = rng.standard_normal((B, W)) * 3
    scores[0, 1:] = -np.inf                   # request 0: only beam 0 live
    if ties:
        scores[1, :] = 0.0                    # equal beam scores: ties across beams
    beams = rng.integers(0, 100, size=(B, W, t)).astype(np.int32)
    out = oracle.oracle_beam_search_step(lg, scores, beams)
    x = bf16_to_f64(lg)
    for b in range(B):
        lse = np.log(np.exp(x[b] - x[b].max(1, keepdims=True)).sum(1)) + x[b].max(1)
        cand = (scores[b][:, None] + x[b] - lse[:, None]).reshape(-1)
        idx = np.arange(W * V)
        live = np.isfinite(cand)
        order = np.lexsort((idx[live], -cand[live]))[:W]
        sel = idx[live][order]
        np.testing.assert_array_equal(out["parent"][b], sel // V)
        np.testing.assert_array_equal(out["beams"][b, :, t], sel % V)
        np.testing.assert_array_equal(out["beams"][b, :, :t], beams[b, sel // V])
        np.testing.assert_allclose(out["scores"][b], cand[sel], rtol=1e-12, atol=1e-12)


def test_first_step_from_the_anchor_takes_the_top_tokens():
    rng = np.random.default_rng(9)
    W, V = 6, 400
    lg = _logits(rng, 1, W, V)
    scores = np.full((1, W), -np.inf)
    scores[0, 0] = 0.0
    out = oracle.oracle_beam_search_step(lg, scores, np.full((1, W, 1), 42, np.int32))
    x = bf16_to_f64(lg)[0, 0]
    top = np.lexsort((np.arange(V), -x))[:W]
    np.testing.assert_array_equal(out["beams"][0, :, 1], top)
    assert (out["parent"][0] == 0).all() and (out["beams"][0, :, 0] == 42).all()
