"""Pins of the oracle's stochastic verification (multi-step speculative
sampling over the draft tree), CPU only.

* One child drawn from the drafter's q: the first emitted token is distributed
  as the target p (the speculative-sampling guarantee), and so is the token
  drawn after an accepted child (Monte Carlo, 5 sigma).
* No child: the draw alone follows p (the exponential race is a sampler).
* q = p: every first child is accepted, the walk is beam 0.
* A hand-worked tree where only the residual max(0, p - q) gives the answer.
* A child without target mass is never emitted.
* Temperature -> 0 with a flat drafter reduces to greedy verification
  (oracle_greedy_accept, pinned on its own).
"""
import numpy as np
import pytest

import oracle
import workloads
from tests.pins import bf16_round, bf16_to_f64


def _p(bits, T=1.0):
    x = bf16_to_f64(bits) / T
    e = np.exp(x - x.max())
    return e / e.sum()


def _run(beams, target, draft, T, u_acc, u_smp):
    B, W, L = beams.shape
    pk = oracle.oracle_pack(beams, target.shape[1])
    return pk, oracle.oracle_sample_accept(target, draft, T, beams, pk["packer"], pk["unpacker"],
                                           pk["packed_len"], u_acc, u_smp)


def _freq_close(samples, p, what):
    n = len(samples)
    f = np.bincount(samples, minlength=len(p)) / n
    tol = 5 * np.sqrt(p * (1 - p) / n) + 1e-3
    assert np.all(np.abs(f - p) <= tol), (what, f, p)


def test_one_child_from_q_emits_the_target_distribution():
    rng = np.random.default_rng(0)
    N, V, T = 20000, 6, 1.3
    t0 = bf16_round(rng.normal(0, 1.5, V).astype(np.float32))
    d0 = bf16_round(rng.normal(0, 1.5, V).astype(np.float32))
    t1 = bf16_round(rng.normal(0, 1.5, V).astype(np.float32))
    p0, q0, p1 = _p(t0, T), _p(d0, T), _p(t1, T)
    x = rng.choice(V, size=N, p=q0)
    beams = np.stack([np.zeros(N, np.int32), x.astype(np.int32)], 1)[:, None, :]
    target = np.broadcast_to(np.stack([t0, t1]), (N, 2, V)).copy()
    draft = np.broadcast_to(np.stack([d0, d0]), (N, 2, V)).copy()
    u_acc = rng.random((N, 2), dtype=np.float32)
    u_smp = rng.random((N, V), dtype=np.float32)
    _, out = _run(beams, target, draft, T, u_acc, u_smp)
    _freq_close(out["out_tokens"][:, 0], p0, "first token")
    acc = out["n_accepted"] == 1
    assert 0.2 * N < acc.sum() < N
    np.testing.assert_array_equal(out["out_tokens"][acc, 0], x[acc])
    _freq_close(out["out_tokens"][acc, 1], p1, "token after the accepted child")
    # acceptance rate of one proposal = sum_x min(p, q)
    assert abs(acc.mean() - np.minimum(p0, q0).sum()) < 5 * np.sqrt(0.25 / N)


def test_draw_without_children_follows_the_target():
    rng = np.random.default_rng(1)
    N, V = 20000, 7
    t0 = bf16_round(rng.normal(0, 2.0, V).astype(np.float32))
    beams = np.zeros((N, 1, 1), np.int32)
    target = np.broadcast_to(t0, (N, 1, V)).copy()
    _, out = _run(beams, target, target, 1.0, rng.random((N, 1), dtype=np.float32),
                  rng.random((N, V), dtype=np.float32))
    _freq_close(out["out_tokens"][:, 0], _p(t0), "draw")
    assert np.all(out["n_accepted"] == 0)


def test_draft_equal_to_target_accepts_every_first_child():
    rng = np.random.default_rng(2)
    B, W, L, V = 50, 4, 5, 40
    trees = workloads.draft_trees(B, W, L, V, ("p", 0.5), rng)
    beams = trees.beams
    P = W * L
    target = bf16_round(rng.normal(0, 2, (B, P, V)).astype(np.float32))
    pk, out = _run(beams, target, target, 0.8, rng.random((B, P), dtype=np.float32),
                   rng.random((B, V), dtype=np.float32))
    assert np.all(out["n_accepted"] == L - 1)
    assert np.all(out["best_beam"] == 0)
    np.testing.assert_array_equal(out["out_tokens"][:, :L - 1], beams[:, 0, 1:])
    for b in range(B):
        for w in range(W):
            n = 0
            while n + 1 < L and np.array_equal(beams[b, w, :n + 2], beams[b, 0, :n + 2]):
                n += 1
            assert out["accept_len"][b, w] == n


def test_hand_worked_residual():
    # p = (.5, .3, .2), q = (.2, .5, .3) at the anchor; children 1 (beam 0) and 2 (beam 1).
    # Child 1: 0.7 * q(1) = .35 >= p(1) = .3, rejected; residual (1, 0, 0).
    # Child 2: residual mass 0 at token 2, rejected for any u; residual (1, 0, 0).
    # The draw must be token 0.  (Without the residual, child 2 would pass: .01*.3 < .2.)
    t = bf16_round(np.log(np.array([0.5, 0.3, 0.2], np.float32)))
    d = bf16_round(np.log(np.array([0.2, 0.5, 0.3], np.float32)))
    beams = np.array([[[0, 1], [0, 2]]], np.int32)
    target = np.stack([t, t, t, t])[None]
    draft = np.stack([d, d, d, d])[None]
    for us in (0.05, 0.5, 0.95):
        u_acc = np.array([[0.0, 0.7, 0.01, 0.0]], np.float32)
        pk, out = _run(beams, target, draft, 1.0, u_acc, np.full((1, 3), us, np.float32))
        assert pk["packed_len"][0] == 3
        assert out["n_accepted"][0] == 0
        np.testing.assert_array_equal(out["out_tokens"][0], [0, -1])
        assert out["best_beam"][0] == 0
        np.testing.assert_array_equal(out["accept_len"][0], [0, 0])
    # the same tree with child 1 tested at u = 0.5: .25 < .3, accepted
    u_acc = np.array([[0.0, 0.5, 0.01, 0.0]], np.float32)
    _, out = _run(beams, target, draft, 1.0, u_acc, np.full((1, 3), 0.5, np.float32))
    assert out["n_accepted"][0] == 1 and out["out_tokens"][0, 0] == 1
    np.testing.assert_array_equal(out["accept_len"][0], [1, 0])


def test_child_without_target_mass_is_never_emitted():
    rng = np.random.default_rng(3)
    N, V, x = 3000, 5, 3
    t0 = np.array([0.5, 1.0, -0.5, -100.0, 0.0], np.float32)
    beams = np.tile(np.array([0, x], np.int32), (N, 1))[:, None, :]
    target = np.broadcast_to(bf16_round(t0), (N, 2, V)).copy()
    draft = np.zeros((N, 2, V), np.uint16)
    _, out = _run(beams, target, draft, 1.0, rng.random((N, 2), dtype=np.float32),
                  rng.random((N, V), dtype=np.float32))
    assert np.all(out["n_accepted"] == 0)
    assert not np.any(out["out_tokens"][:, 0] == x)


@pytest.mark.parametrize("seed", [4, 5])
def test_low_temperature_with_flat_drafter_is_greedy(seed):
    rng = np.random.default_rng(seed)
    B, W, L, V = 40, 6, 5, 200
    trees = workloads.draft_trees(B, W, L, V, ("p", 0.6), rng)
    beams = trees.beams
    P = W * L
    pk = oracle.oracle_pack(beams, P)
    # distinct integer logits (exact in bf16, gaps >= 1); plant the first child's token
    # as the argmax at about half of the nodes so that drafts get accepted
    logits = np.zeros((B, P, V), np.float32)
    for b in range(B):
        for n in range(P):
            row = rng.permutation(V).astype(np.float32)
            kids = [c for c in range(n + 1, pk["packed_len"][b])
                    if pk["packer"][b, c] % L > 0 and
                    pk["unpacker"][b].reshape(-1)[pk["packer"][b, c] - 1] == n]
            if kids and rng.random() < 0.6:
                tok = beams[b].reshape(-1)[pk["packer"][b, kids[0]]]
                top = int(np.argmax(row))
                row[top], row[tok] = row[tok], row[top]
            logits[b, n] = row
    target = bf16_round(logits)
    flat = np.zeros_like(target)
    out = oracle.oracle_sample_accept(target, flat, 0.01, beams, pk["packer"], pk["unpacker"],
                                      pk["packed_len"], rng.random((B, P), dtype=np.float32),
                                      rng.random((B, V), dtype=np.float32))
    g = oracle.oracle_greedy_accept(target, beams, pk["unpacker"], pk["packed_len"])
    assert (g["n_accepted"] > 0).sum() > 5
    for k in ("n_accepted", "best_beam", "out_tokens", "accept_len"):
        np.testing.assert_array_equal(out[k], g[k], err_msg=k)
