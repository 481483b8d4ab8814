"""Pins of the oracle's attention (CPU only).

* Tree-masked attention over packed drafts equals independent causal attention
  per beam (brute force, tests/pins.py), with K/V and queries defined per
  prefix so that the brute force never sees the oracle's packing.
* The same tree mask through torch's scaled_dot_product_attention in float64.
* Closed forms: a single visible key returns its value; equal scores return the
  mean of the visible values.
* Causal mode equals torch's causal scaled_dot_product_attention in float64.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.pins import bf16_round, bf16_to_f64, per_beam_attention, prefix_tuples


class PrefixVectors:
    """A fixed random bf16 vector per prefix tuple (as the LLM would compute
    one K/V/q per trie node), independent of any packing."""

    def __init__(self, seed, shape):
        self.seed, self.shape, self.cache = seed, shape, {}

    def bits(self, pre):
        if pre not in self.cache:
            h = hash((self.seed,) + pre) & 0xFFFFFFFF
            x = np.random.default_rng(h).standard_normal(self.shape).astype(np.float32)
            self.cache[pre] = bf16_round(x)
        return self.cache[pre]

    def f64(self, pre):
        return bf16_to_f64(self.bits(pre))


def _tree_case(seed, W, L, vocab, C, Hq, Hkv, D, B=2):
    rng = np.random.default_rng(seed)
    beams = rng.integers(0, vocab, size=(B, W, L)).astype(np.int32)
    beams[:, :, 0] = beams[:, :1, 0]           # shared anchor per request
    P = W * L
    pk = oracle.oracle_pack(beams, P)
    qv, kv, vv = PrefixVectors(seed * 3, (Hq, D)), PrefixVectors(seed * 3 + 1, (Hkv, D)), \
        PrefixVectors(seed * 3 + 2, (Hkv, D))
    q = np.zeros((B, P, Hq, D), np.uint16)
    kn = np.zeros((B, P, Hkv, D), np.uint16)
    vn = np.zeros((B, P, Hkv, D), np.uint16)
    for b in range(B):
        for p in range(pk["packed_len"][b]):
            f = pk["packer"][b, p]
            pre = tuple(int(x) for x in beams[b, f // L, : f % L + 1])
            q[b, p], kn[b, p], vn[b, p] = qv.bits(pre), kv.bits(pre), vv.bits(pre)
    lens = rng.integers(0, C + 1, size=B)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    kc = bf16_round(rng.standard_normal((offs[-1], Hkv, D)).astype(np.float32))
    vc = bf16_round(rng.standard_normal((offs[-1], Hkv, D)).astype(np.float32))
    return beams, pk, q, kn, vn, kc, vc, offs, (qv, kv, vv)


@pytest.mark.parametrize("seed,W,L,vocab,C,Hq,Hkv,D", [
    (0, 3, 4, 3, 5, 2, 1, 8),
    (1, 4, 3, 2, 0, 2, 2, 4),       # no context at all
    (2, 1, 5, 5, 7, 4, 2, 8),       # a single beam: plain causal decode
    (3, 5, 4, 2, 3, 6, 3, 16),
    (4, 2, 6, 4, 9, 1, 1, 8),
])
def test_tree_attention_equals_per_beam_causal(seed, W, L, vocab, C, Hq, Hkv, D):
    beams, pk, q, kn, vn, kc, vc, offs, (qv, kv, vv) = _tree_case(seed, W, L, vocab, C, Hq, Hkv, D)
    o = oracle.oracle_tree_attention(q, kn, vn, kc, vc, offs, pk["packed_len"], pk["mask"],
                                     n_threads=2)
    scale = 1.0 / np.sqrt(D)
    for b in range(beams.shape[0]):
        c0, c1 = offs[b], offs[b + 1]
        ref = per_beam_attention(beams[b], bf16_to_f64(kc[c0:c1]), bf16_to_f64(vc[c0:c1]),
                                 qv.f64, kv.f64, vv.f64, Hq // Hkv, scale)
        for w in range(W):
            for i in range(L):
                pre = tuple(int(x) for x in beams[b, w, : i + 1])
                np.testing.assert_allclose(o[b, pk["unpacker"][b, w, i]], ref[pre],
                                           rtol=1e-12, atol=1e-12)
        assert (o[b, pk["packed_len"][b]:] == 0).all()


def test_tree_attention_matches_torch_sdpa_with_explicit_mask():
    seed, W, L, vocab, C, Hq, Hkv, D = 7, 4, 4, 3, 6, 4, 2, 16
    beams, pk, q, kn, vn, kc, vc, offs, _ = _tree_case(seed, W, L, vocab, C, Hq, Hkv, D, B=1)
    o = oracle.oracle_tree_attention(q, kn, vn, kc, vc, offs, pk["packed_len"], pk["mask"])
    P = int(pk["packed_len"][0])
    pref = prefix_tuples(beams[0])
    # visibility from prefix relations (a key node is visible iff it is a prefix of the query)
    vis = np.zeros((P, P), bool)
    for a in range(P):
        for k in range(P):
            vis[a, k] = pref[a][: len(pref[k])] == pref[k]
    allowed = np.concatenate([np.ones((P, offs[1]), bool), vis], 1)
    G = Hq // Hkv
    for hq in range(Hq):
        h = hq // G
        Q = torch.from_numpy(bf16_to_f64(q[0, :P, hq]))
        K = torch.from_numpy(np.concatenate([bf16_to_f64(kc[:, h]), bf16_to_f64(kn[0, :P, h])]))
        V = torch.from_numpy(np.concatenate([bf16_to_f64(vc[:, h]), bf16_to_f64(vn[0, :P, h])]))
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None], V[None], attn_mask=torch.from_numpy(allowed)[None])[0].numpy()
        np.testing.assert_allclose(o[0, :P, hq], ref, rtol=1e-10, atol=1e-12)


def test_single_visible_key_returns_its_value():
    # no context, root node: the only visible key is the node itself
    beams = np.array([[[1, 2], [3, 4]]], np.int32)          # distinct anchors
    pk = oracle.oracle_pack(beams)
    rng = np.random.default_rng(0)
    D = 8
    q = bf16_round(rng.standard_normal((1, 4, 1, D)).astype(np.float32))
    kn = bf16_round(rng.standard_normal((1, 4, 1, D)).astype(np.float32))
    vn = bf16_round(rng.standard_normal((1, 4, 1, D)).astype(np.float32))
    empty = np.zeros((0, 1, D), np.uint16)
    o = oracle.oracle_tree_attention(q, kn, vn, empty, empty, np.array([0, 0], np.int64),
                                     pk["packed_len"], pk["mask"])
    for p in (0, 2):                                        # the two anchors
        np.testing.assert_array_equal(o[0, p, 0], bf16_to_f64(vn[0, p, 0]))


def test_equal_scores_give_mean_of_visible_values():
    beams = np.array([[[1, 2, 3], [1, 5, 6]]], np.int32)
    pk = oracle.oracle_pack(beams)
    rng = np.random.default_rng(1)
    D, C = 8, 5
    q = np.zeros((1, 6, 1, D), np.uint16)                   # q = 0: every score is 0
    kn = bf16_round(rng.standard_normal((1, 6, 1, D)).astype(np.float32))
    vn = bf16_round(rng.standard_normal((1, 6, 1, D)).astype(np.float32))
    kc = bf16_round(rng.standard_normal((C, 1, D)).astype(np.float32))
    vc = bf16_round(rng.standard_normal((C, 1, D)).astype(np.float32))
    o = oracle.oracle_tree_attention(q, kn, vn, kc, vc, np.array([0, C], np.int64),
                                     pk["packed_len"], pk["mask"])
    # node (1,2)=(1,5,6) is packed index 4; its path is nodes 0, 3, 4
    path = [0, 3, 4]
    mean = (bf16_to_f64(vc[:, 0]).sum(0) + bf16_to_f64(vn[0, path, 0]).sum(0)) / (C + 3)
    np.testing.assert_allclose(o[0, 4, 0], mean, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([5, 1, 9], 4, 2, 8), ([16], 2, 2, 16), ([0, 3], 1, 1, 4)])
def test_causal_attention_matches_torch_sdpa(lens, Hq, Hkv, D):
    rng = np.random.default_rng(sum(lens))
    T = sum(lens)
    q = bf16_round(rng.standard_normal((T, Hq, D)).astype(np.float32))
    k = bf16_round(rng.standard_normal((T, Hkv, D)).astype(np.float32))
    v = bf16_round(rng.standard_normal((T, Hkv, D)).astype(np.float32))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o = oracle.oracle_causal_attention(q, k, v, cu, n_threads=2)
    G = Hq // Hkv
    for b in range(len(lens)):
        s0, s1 = cu[b], cu[b + 1]
        if s1 == s0:
            continue
        for hq in range(Hq):
            Q = torch.from_numpy(bf16_to_f64(q[s0:s1, hq]))
            K = torch.from_numpy(bf16_to_f64(k[s0:s1, hq // G]))
            V = torch.from_numpy(bf16_to_f64(v[s0:s1, hq // G]))
            ref = torch.nn.functional.scaled_dot_product_attention(
                Q[None], K[None], V[None], is_causal=True)[0].numpy()
            np.testing.assert_allclose(o[s0:s1, hq], ref, rtol=1e-10, atol=1e-12)
