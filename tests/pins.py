"""Independent brute-force formulations used to pin the oracle.

None of these share code with ``oracle/``.  They restate what the method must
equal in a different form:

* prefix dedup  == the set of distinct prefix tuples of the beams;
* tree-masked attention over packed drafts == ordinary causal attention run
  separately on every beam (speculative-decoding survey page, SpecInfer
  "Token Tree Verifier": the topology-aware mask computes all sequences in one
  kernel instead of one kernel per sequence);
* greedy verification == plain greedy decoding walked along the beams.
"""
from __future__ import annotations

import numpy as np


def prefix_tuples(beams_b: np.ndarray) -> list:
    """Distinct prefixes of one request's [W, L] beams, in scan order."""
    seen, order = set(), []
    W, L = beams_b.shape
    for w in range(W):
        for i in range(L):
            t = tuple(int(x) for x in beams_b[w, : i + 1])
            if t not in seen:
                seen.add(t)
                order.append(t)
    return order


def bf16_round(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def causal_softmax_attention(q: np.ndarray, keys: np.ndarray, vals: np.ndarray,
                             scale: float) -> np.ndarray:
    """Textbook attention of one query over the given keys (float64)."""
    s = keys @ q * scale
    e = np.exp(s - s.max())
    return (e[:, None] * vals).sum(0) / e.sum()


def per_beam_attention(beams_b, ctx_k, ctx_v, q_of, k_of, v_of, G, scale):
    """Per beam w and position i, attention of the query of prefix (w, 0..i)
    over the context keys plus the keys of prefixes (w, 0..j), j <= i.

    q_of(prefix) -> [Hq, D]; k_of/v_of(prefix) -> [Hkv, D]; ctx_k/ctx_v [C, Hkv, D].
    Returns dict prefix-tuple -> [Hq, D] float64.
    """
    W, L = beams_b.shape
    out = {}
    for w in range(W):
        for i in range(L):
            pre = tuple(int(x) for x in beams_b[w, : i + 1])
            qh = q_of(pre)
            Hq = qh.shape[0]
            ks = [k_of(tuple(int(x) for x in beams_b[w, : j + 1])) for j in range(i + 1)]
            vs = [v_of(tuple(int(x) for x in beams_b[w, : j + 1])) for j in range(i + 1)]
            res = np.zeros_like(qh)
            for hq in range(Hq):
                h = hq // G
                K = np.concatenate([ctx_k[:, h, :], np.stack([k[h] for k in ks])], 0)
                V = np.concatenate([ctx_v[:, h, :], np.stack([v[h] for v in vs])], 0)
                res[hq] = causal_softmax_attention(qh[hq], K, V, scale)
            out[pre] = res
    return out


def greedy_per_beam(beams_b: np.ndarray, greedy_of) -> tuple:
    """Accepted draft count per beam, by stepping along each beam and asking the
    greedy choice (greedy_of(prefix) -> token) at every prefix."""
    W, L = beams_b.shape
    acc = []
    for w in range(W):
        n = 0
        while n < L - 1 and int(beams_b[w, n + 1]) == greedy_of(
                tuple(int(x) for x in beams_b[w, : n + 1])):
            n += 1
        acc.append(n)
    best = int(np.argmax(acc))      # first maximum: lowest beam on ties
    a = acc[best]
    emitted = [int(x) for x in beams_b[best, 1: a + 1]]
    emitted.append(greedy_of(tuple(int(x) for x in beams_b[best, : a + 1])))
    return acc, best, emitted


def greedy_walk(beams_b: np.ndarray, greedy_of) -> list:
    """Plain greedy decoding from the (shared) anchor: take the greedy token; if a
    beam continues the current prefix with it, follow; else emit it and stop."""
    W, L = beams_b.shape
    prefixes = set(prefix_tuples(beams_b))
    cur = (int(beams_b[0, 0]),)
    emitted = []
    while True:
        g = greedy_of(cur)
        emitted.append(g)
        nxt = cur + (g,)
        if len(nxt) <= L and nxt in prefixes:
            cur = nxt
            continue
        return emitted
